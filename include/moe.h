/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE expert-FFN layer library (libmoe_gb300.so).
 *
 * The layer, as the Muse Spark Open explainer ("Muse Spark Open を段階的に分解する") states it:
 *   section 8   a router scores every expert with one FP32 matrix product and keeps the best
 *               k (8 of 256 there) as a set; there is no shared expert;
 *   section 12  the (token, expert) pairs are gathered per expert and each expert computes its
 *               tokens as one batch;
 *   section 9   each chosen expert applies gate, up and down matrices; the expert outputs are
 *               weighted by the router scores and summed;
 *   section 11  expert weights are 4-bit values sharing a block scale; the DGX Spark news item
 *               ("DGX Spark MoE inference optimizations", section 2) names the block-scaled
 *               MXFP4 format: E2M1 elements, one E8M0 scale per 32 consecutive elements.
 *
 * Conventions for every entry point below:
 *   - Tensor pointers are DEVICE pointers owned by the caller (the library never frees or
 *     keeps them).  Shapes are row-major; "[a][b]" means a rows of b elements.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and returns synchronously only argument and launch errors.
 *   - The library allocates no device memory in any entry point.  Scratch space comes from
 *     the caller's workspace `ws` of `ws_bytes` bytes (see moe_workspace_size); it must be
 *     256-byte aligned and initialised once with moe_workspace_init.  Calls that share a
 *     workspace must be ordered on one stream.
 *   - Kernels that wait on hardware barriers give up after a bounded number of polls, record
 *     MOE_ERR_TIMEOUT in the workspace and return; moe_get_device_status reads that word.
 *   - Inputs are assumed finite.
 *   - Shape rules (MOE_ERR_UNSUPPORTED_SHAPE otherwise): 1 <= k <= min(E, 32); E <= 1024;
 *     T >= 0; MOE_ACT_BF16: d % 128 == 0 and I % 32 == 0; MOE_ACT_MXFP4 and MOE_ACT_MXFP8:
 *     d % 256 == 0 and I % 256 == 0 (whole 256-value MMA tiles along both contractions).  NVFP4
 *     expert weights (moe_weight_fmt) are read by MOE_ACT_BF16 and MOE_ACT_MXFP4 (not MXFP8).
 *
 * MXFP4 tensor layout ("canonical"): a [rows][K] matrix is stored as codes q[rows][K/2]
 * (element 2i in the low nibble of byte i, element 2i+1 in the high nibble; bit 3 of a code
 * is the sign) and scales s[rows][K/32] (E8M0: the block's values are code_value * 2^(s-127)).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* moe_stream_t; /* same object as a cudaStream_t */

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null / misaligned pointer, negative size */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* a shape rule above is violated */
    MOE_ERR_WORKSPACE = 3,         /* workspace missing, too small or misaligned */
    MOE_ERR_CUDA = 4,              /* a CUDA runtime call failed (launch error, no device) */
    MOE_ERR_TIMEOUT = 5,           /* device side: a bounded barrier wait ran out */
    MOE_ERR_DEVICE = 6             /* the current device is not an sm_103 GPU */
} moe_status;

/* Activation format of the expert GEMM operands.
 *   MOE_ACT_BF16  -- decode-style path: x is used as bf16, the gate/up output h is rounded to
 *                    bf16 (see moe_layer_forward for its two kernel paths).
 *   MOE_ACT_MXFP4 -- prefill path: x and h are quantised to MXFP4 (same rule as the weight
 *                    packer); tcgen05 block-scaled MMA (kind::mxf4) grouped GEMMs.
 *   MOE_ACT_MXFP8 -- 4-bit weights with 8-bit activations (the baseline configuration of the
 *                    DGX Spark news item, section 2): x and h are quantised to MXFP8, E4M3
 *                    elements (OCP OFP8: bias 7, subnormals, largest finite 448) with one E8M0
 *                    scale per 32 consecutive elements: X = floor(log2(max |v|)) - 8 clamped to
 *                    [-127, 127], scale byte X + 127, each element |v| / 2^X rounded to the
 *                    nearest E4M3 value (ties to even, saturating at 448) with the sign of v
 *                    unless it rounds to zero (stored as +0); an all-zero block gets scale byte 0.
 *                    Needs MXFP4 weights with their tensor-core copies; up to 16 tokens run the
 *                    decode kernels of MOE_ACT_BF16 on the operands' MXFP8 values, more run
 *                    kind::mxf8f6f4 grouped GEMMs (E4M3 tokens x E2M1 weights). */
typedef enum moe_act_fmt { MOE_ACT_BF16 = 0, MOE_ACT_MXFP4 = 1, MOE_ACT_MXFP8 = 2 } moe_act_fmt;

/* Format of the expert weight matrices (moe_expert_weights.wfmt).
 *   MOE_W_MXFP4 -- the canonical MXFP4 layout above.
 *   MOE_W_NVFP4 -- 4-bit values of which 16 share a small scale, about 4.5 bits each (Muse
 *                  Spark Open explainer, section 11): the same E2M1 codes q[rows][K/2], one
 *                  E4M3 scale (OCP OFP8: bias 7, largest finite 448) per 16 consecutive
 *                  elements of a row, s[rows][K/16], and one fp32 global scale per matrix;
 *                  value = E2M1 * E4M3 * global.  Read by the MOE_ACT_BF16 GEMVs and, with
 *                  their tensor-core copies (codes: moe_mxfp4_codes_to_mma; scales:
 *                  moe_mxfp4_scales_to_mma of s read as a [rows][2K] matrix's E8M0 scales, i.e.
 *                  rows x K/16 bytes), by the MOE_ACT_MXFP4 grouped GEMMs (tcgen05
 *                  kind::mxf4nvf4).  There the MXFP4 operands' block scales 2^X are carried as
 *                  UE4M3 powers of two per 16 values relative to one power-of-two factor per row
 *                  (2^(largest X of the row - 8)), which is exact for every block within 17
 *                  binades of the row's largest; a block further below is dropped (its values
 *                  are under 2^-15 of the row's largest block scale). */
typedef enum moe_weight_fmt { MOE_W_MXFP4 = 0, MOE_W_NVFP4 = 1 } moe_weight_fmt;

/* Expert weights of one layer (all device pointers, canonical MXFP4 layout):
 *   gate_q/up_q [E][I][d/2], gate_s/up_s [E][I][d/32]   (gate and up: I rows of d)
 *   down_q      [E][d][I/2], down_s      [E][d][I/32]   (down: d rows of I)
 * The MXFP4 path reads copies re-laid out for the tensor cores (see "tensor-core layouts"):
 *   gate_q_mma, up_q_mma   moe_mxfp4_codes_to_mma(gate_q or up_q, E*I, d)
 *   gate_s_mma, up_s_mma   moe_mxfp4_scales_to_mma(gate_s or up_s, E*I, d)
 *   down_q_mma             moe_mxfp4_codes_to_mma(down_q, E*d, I)
 *   down_s_mma             moe_mxfp4_scales_to_mma(down_s, E*d, I)
 * The BF16 path reads only the canonical tensors (the six copies may be NULL).
 * With wfmt = MOE_W_NVFP4 the scale tensors are E4M3 [E][I][d/16] (gate, up) and [E][d][I/16]
 * (down), 2-byte aligned, and gate_gs / up_gs / down_gs hold the global scale of each expert's
 * matrix ([E] fp32 each); the tensor-core copies are not used.  A zero-initialised struct is
 * MXFP4 (MOE_ERR_INVALID_ARG for any other wfmt). */
typedef struct moe_expert_weights {
    const uint8_t* gate_q;
    const uint8_t* gate_s;
    const uint8_t* up_q;
    const uint8_t* up_s;
    const uint8_t* down_q;
    const uint8_t* down_s;
    const uint8_t* gate_q_mma;
    const uint8_t* gate_s_mma;
    const uint8_t* up_q_mma;
    const uint8_t* up_s_mma;
    const uint8_t* down_q_mma;
    const uint8_t* down_s_mma;
    int32_t wfmt;         /* moe_weight_fmt */
    const float* gate_gs; /* MOE_W_NVFP4 only: [E] */
    const float* up_gs;
    const float* down_gs;
} moe_expert_weights;

/* ---------------------------------------------------------------- library */

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* ABI version of this header (incremented on changes to the entry points or their structs);
 * moe_abi_version() returns the library's, which a caller compares with MOE_ABI_VERSION. */
#define MOE_ABI_VERSION 13
int moe_abi_version(void);

/* Description of the CUDA error behind the calling thread's last MOE_ERR_CUDA (static string). */
const char* moe_last_cuda_error(void);

/* ---------------------------------------------------------------- MXFP4 helpers
 * Block-scaled 4-bit format of the expert weights (DGX Spark news item, section 2; Muse
 * Spark Open explainer, section 11).  Quantisation rule (OCP MX v1.0): per 32-element block,
 * X = floor(log2(max |v|)) - 2 clamped to [-127, 127], scale byte X + 127, each element
 * rounded to nearest on the E2M1 grid {0, .5, 1, 1.5, 2, 3, 4, 6} times 2^X, ties to the
 * even code, saturating at 6 * 2^X; a value that rounds to zero is stored as +0; an
 * all-zero block gets scale byte 0. */

/* Pack fp32 w[rows][K] into q[rows][K/2], s[rows][K/32].  K % 32 == 0, rows >= 0. */
moe_status moe_mxfp4_pack(const float* w, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                          moe_stream_t stream);

/* Dequantise q, s back to fp32 w[rows][K] (exact). */
moe_status moe_mxfp4_unpack(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K, float* w,
                            moe_stream_t stream);

/* ---------------------------------------------------------------- NVFP4 helpers
 * Quantisation rule of the NVFP4 weight format, every step in fp32 with round-to-nearest-even:
 *   global = (largest |w| of the matrix) / 2688 (= 6 * 448), or 1 when that is 0;
 *   for each 16-element block: t = (largest |v| of the block / global) / 6; scale byte = t
 *   rounded to the nearest E4M3 value (ties to even, saturating at 448); D = E4M3 value *
 *   global; each element is |v| / D rounded to the nearest E2M1 magnitude (ties to the even
 *   code, saturating at 6), with the sign of v unless it rounds to 0 (stored as +0); D = 0
 *   gives zero codes. */

/* Pack n_mats fp32 matrices w[n_mats][rows][K] into q[n_mats*rows][K/2], s[n_mats*rows][K/16]
 * and the global scales gs[n_mats] (gs is also the scratch of the per-matrix maximum while the
 * call runs).  K % 32 == 0, rows >= 0, 0 <= n_mats <= 65535; w and q 16-byte aligned, s 2-byte
 * aligned, gs 4-byte aligned. */
moe_status moe_nvfp4_pack(const float* w, int64_t n_mats, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                          float* gs, moe_stream_t stream);

/* Dequantise to fp32: w = (E2M1 value * E4M3 value) * gs[matrix], the exact product of the first
 * two rounded once.  Same shapes and alignment as moe_nvfp4_pack. */
moe_status moe_nvfp4_unpack(const uint8_t* q, const uint8_t* s, const float* gs, int64_t n_mats, int64_t rows,
                            int64_t K, float* w, moe_stream_t stream);

/* Tensor-core layouts of a [rows][K] MXFP4 matrix (rows % 128 == 0, K % 256 == 0), read by the
 * block-scaled MMA path with one contiguous copy per operand tile:
 *   codes   tiles of 128 rows x 256 values (16384 bytes); tile (R, C) = rows 128R..128R+127 x
 *           values 256C..256C+255 sits at tile index R*(K/256) + C.  Inside a tile, the 16-byte
 *           chunk j (values 256C+32j..+31, one 32-element block) of row r is stored at byte
 *           r*128 + (j XOR (r%8))*16 (the 128-byte swizzle the tensor cores read).  Same size
 *           as the canonical codes.
 *   scales  a grid of 512-byte atoms, atom (R, C) = rows 128R..128R+127 x scale columns
 *           4C..4C+3 at atom index R*(K/128) + C; inside an atom, row r and scale column c sit
 *           at byte (r%32)*16 + ((r/32)%4)*4 + (c%4). */

/* Bytes of the tensor-core scale layout of a [rows][K] matrix (rows % 128 == 0, K % 128 == 0;
 * 0 otherwise). */
size_t moe_mxfp4_mma_scale_bytes(int64_t rows, int64_t K);

/* Re-lay canonical scales s[rows][K/32] out into the tensor-core scale layout s_mma. */
moe_status moe_mxfp4_scales_to_mma(const uint8_t* s, int64_t rows, int64_t K, uint8_t* s_mma,
                                   moe_stream_t stream);

/* Re-lay canonical codes q[rows][K/2] out into the tensor-core code tiles q_mma (rows*K/2 bytes;
 * rows % 128 == 0, K % 256 == 0). */
moe_status moe_mxfp4_codes_to_mma(const uint8_t* q, int64_t rows, int64_t K, uint8_t* q_mma,
                                  moe_stream_t stream);

/* ---------------------------------------------------------------- workspace */

/* Bytes of workspace needed by moe_layer_forward (and enough for every step call) at these
 * sizes.  Returns 0 when the shape is unsupported. */
size_t moe_workspace_size(int T, int d, int E, int k, int I, moe_act_fmt fmt);

/* Rows of the padded, expert-grouped activation buffers of the MXFP4 / MXFP8 paths (xa, h): every
 * expert's rows start at a multiple of 128.  An upper bound that depends on sizes only. */
int64_t moe_padded_rows(int T, int k, int E);

/* Zero the workspace control block (status word, counters; the first 8 KB).  Call once per
 * workspace, and again after moe_get_device_status reported MOE_ERR_TIMEOUT (a call that timed
 * out may leave its counters set). */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream);

/* Synchronise `stream`, copy the device status word of `ws` to *out and clear it.
 * *out is MOE_OK or the first device-side error (MOE_ERR_TIMEOUT) recorded since the last
 * call. */
moe_status moe_get_device_status(void* ws, moe_stream_t stream, moe_status* out);

/* Device pointers to the routing buffers inside a layer workspace (ws of ws_bytes bytes, laid out
 * for T, d, E, k, I, fmt as moe_workspace_size sizes it): counts[E], offsets[E+1],
 * perm_token[T*k] and inv_pos[T*k] with the meaning moe_permute gives them (Muse Spark Open
 * explainer, section 12: pairs gathered per expert).  moe_layer_forward and
 * moe_layer_forward_norm write them on every call (on the MOE_ACT_BF16 path with up to eight
 * tokens the one-launch router builds them itself); moe_route on up to eight tokens writes them
 * too.  They hold the last such call's permutation until the next call on ws; reading them is the
 * caller's business (after the call's stream work is done).  No device work, no allocation.
 * MOE_ERR_WORKSPACE when ws is null, misaligned or smaller than the layout. */
moe_status moe_workspace_routing(void* ws, size_t ws_bytes, int T, int d, int E, int k, int I, moe_act_fmt fmt,
                                 int32_t** counts, int32_t** offsets, int32_t** perm_token, int32_t** inv_pos);

/* ---------------------------------------------------------------- layer steps */

/* Router (Muse Spark Open explainer, section 8): logits[t][e] = b[e] + sum_i x[t][i]*W_r[e][i]
 * in fp32 with a fixed reduction order: 32 partial sums, partial c accumulating with fma the
 * elements i with (i/4) % 32 == c in increasing i, combined by an xor butterfly
 * (m = 16, 8, 4, 2, 1), then + b[e].  The k largest logits are kept (ties -> lower e);
 * ids[t][k] is that set in ascending expert order and w[t][k] the softmax of the selected
 * logits (section 9: the weights sum to 1).
 *   x bf16 [T][d]; W_r fp32 [E][d]; b fp32 [E] or NULL (= 0); ids int32 [T][k]; w fp32 [T][k].
 * Uses ws for the T*E logits.  From 256 tokens on (d at most 32768, T*E at most 2^25, x and W_r
 * 16-byte aligned) the logits are first screened on the tensor cores (bf16 parts of W_r, fp32
 * accumulation) with a bound on the screen's error, and the fixed-order logits above are then
 * computed only for the experts that can still be among a token's k largest; every other
 * expert's logit is left as -inf in ws.  ids and w are the same as with every logit computed. */
moe_status moe_route(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                     int32_t* ids, float* w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_route without a workspace and without any allocation (no counterpart in the paper: this
 * serves callers that cannot allocate device memory or own a scratch buffer when they route --
 * code running inside a global-mode CUDA graph capture, where allocation calls are not
 * permitted; hosts whose fixed device memory pool refuses further allocations; foreign-function
 * callers that cannot size and keep a workspace).  Same arguments and results as moe_route.
 * Its scratch (the T*E fp32 logits) is one fixed array of 524288 floats (2 MiB) in the
 * library's device memory, held by every GPU that loads the library until the process exits;
 * T*E > 524288 returns MOE_ERR_UNSUPPORTED_SHAPE.  The first call on a device, with that device
 * current, looks up the array's address (cudaGetSymbolAddress); make that first call before any
 * stream capture.  All calls share the array: every call writes the logits it reads, so nothing
 * carries over, but calls whose work overlaps on the GPU (different streams, or different host
 * threads) race on it and must be serialised by the caller. */
moe_status moe_route_noalloc(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                             int32_t* ids, float* w, moe_stream_t stream);

/* Permutation by expert (section 12).  The T*k pairs (t, j) are ordered by (ids[t][j], t, j):
 *   counts[E]      pairs per expert
 *   offsets[E+1]   exclusive prefix sum of counts
 *   perm_token[P]  token of permuted row r (P = T*k)
 *   inv_pos[P]     permuted row of pair (t, j) at index t*k + j
 * ids as moe_route returns them: each token's k ids distinct and in [0, E).  An id outside
 * [0, E) is not counted and its pair gets no row (its inv_pos entry is not written).
 * For MOE_ACT_MXFP4 and MOE_ACT_MXFP8, unless xa and xa_s are both NULL, it also quantises every
 * token row of x once and writes the activation operand of the [moe_padded_rows][d] matrix of
 * permuted rows in padded expert-grouped order (expert e's rows start at a multiple of 128;
 * padding rows are zero): xa in the tensor-core code tiles and xa_s in the tensor-core scale
 * layout (moe_mxfp4_mma_scale_bytes(moe_padded_rows, d) bytes).  MXFP4 code tiles are those of
 * the weights (moe_padded_rows*d/2 bytes); MXFP8 code tiles (moe_padded_rows*d bytes) hold 128
 * rows x 128 E4M3 bytes each, tile (R, C) at index R*(d/128) + C, the 16-byte chunk j of row r
 * at byte r*128 + (j XOR (r%8))*16.  For MOE_ACT_BF16, xa and xa_s are unused (may be NULL).
 * Writes the per-expert plan (padded offsets, tile table) into ws for the expert calls that
 * follow. */
moe_status moe_permute(const uint16_t* x, const int32_t* ids, int T, int d, int E, int k, moe_act_fmt fmt,
                       int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* inv_pos,
                       uint8_t* xa, uint8_t* xa_s, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Gate/up GEMMs with fused SwiGLU (section 9; SwiGLU h = SiLU(g) * u, g = x W_g^T, u = x W_u^T)
 * for every permuted row, grouped by expert.  Needs the plan that moe_permute wrote into ws.
 *   MOE_ACT_BF16:  reads x bf16 [T][d] through perm_token; writes h bf16 [P][I] (row r =
 *                  permuted row r), h_s unused.
 *   MOE_ACT_MXFP4 / MOE_ACT_MXFP8: reads xa / xa_s; writes the [moe_padded_rows][I] matrix h,
 *                  quantised to the same format, in the same padded order: codes in the
 *                  tensor-core code tiles of the format (moe_padded_rows*I/2 bytes for MXFP4,
 *                  moe_padded_rows*I for MXFP8), scales in the tensor-core scale layout (padding
 *                  rows are zero).  MOE_ACT_MXFP8 reads the weight codes gate_q / up_q (32-byte
 *                  aligned) and the scale copies gate_s_mma / up_s_mma. */
moe_status moe_expert_up_swiglu(const uint16_t* x, const uint8_t* xa, const uint8_t* xa_s, moe_act_fmt fmt,
                                const int32_t* perm_token, const int32_t* offsets, int T, int d, int E, int k,
                                int I, const moe_expert_weights* W, void* h, uint8_t* h_s, void* ws,
                                size_t ws_bytes, moe_stream_t stream);

/* Down GEMM (section 9): y_perm[r] = h[r] W_d[e]^T for every permuted row r of expert e,
 * written as bf16 [P][d] in compact permuted order.  h / h_s as produced by
 * moe_expert_up_swiglu in the same format; perm_token / offsets from moe_permute (perm_token
 * is only read by the MOE_ACT_BF16 path). */
moe_status moe_expert_down(const void* h, const uint8_t* h_s, moe_act_fmt fmt, const int32_t* perm_token,
                           const int32_t* offsets, int T, int d, int E, int k, int I, const moe_expert_weights* W,
                           uint16_t* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Bytes of the pieces operand of moe_decode_pieces: scales = 0 the codes, scales = 1 the scale
 * atoms.  0 when 1 <= T <= 16 and d % 256 == 0 do not hold. */
size_t moe_decode_pieces_bytes(int T, int d, int scales);

/* The token operand of moe_expert_ffn_decode: each row of x bf16 [T][d] (fmt MOE_ACT_BF16), or
 * its MXFP8 values (fmt MOE_ACT_MXFP8, the rule of moe_act_fmt), written as 8 MXFP4 pieces (see
 * moe_layer_forward), rows 8t .. 8t+7 of a 128-row tensor-core tile: codes in xa, scales in xa_s
 * (moe_decode_pieces_bytes(T, d, 0) and (T, d, 1) bytes, xa and x 16-byte aligned; the other
 * rows are not written).  1 <= T <= 16 (T = 0 does nothing) and d % 256 == 0
 * (MOE_ERR_UNSUPPORTED_SHAPE otherwise).  No workspace. */
moe_status moe_decode_pieces(const uint16_t* x, int T, int d, moe_act_fmt fmt, uint8_t* xa, uint8_t* xa_s,
                             moe_stream_t stream);

/* Both expert GEMMs of a small batch on the block-scaled FP4 tensor cores, in one persistent
 * launch (the kernels moe_layer_forward runs for MOE_ACT_BF16 and MOE_ACT_MXFP8 with MXFP4
 * weights carrying their tensor-core copies): gate/up with SwiGLU (section 9) on the token
 * pieces xa / xa_s from moe_decode_pieces (same fmt), h rounded to bf16 (MOE_ACT_BF16) or to
 * MXFP8 (MOE_ACT_MXFP8) and fed to the down GEMM as its own 8 pieces, the expert outputs rounded
 * to bf16 into y_perm [T*k][d] (compact permuted order).  With y != NULL (T <= 4) the weighted
 * sum of moe_combine is fused and written to y bf16 [T][d] (inv_pos and w as moe_combine takes
 * them).  Needs the plan that moe_permute wrote into ws (laid out for the same T, d, E, k, I and
 * fmt).  1 <= T <= 16, d % 256 == 0, I % 256 == 0 and MXFP4 weights with their tensor-core
 * copies (MOE_ERR_UNSUPPORTED_SHAPE otherwise). */
moe_status moe_expert_ffn_decode(const uint8_t* xa, const uint8_t* xa_s, moe_act_fmt fmt, const int32_t* perm_token,
                                 const int32_t* offsets, const int32_t* inv_pos, const float* w, int T, int d,
                                 int E, int k, int I, const moe_expert_weights* W, uint16_t* y_perm, uint16_t* y,
                                 void* ws, size_t ws_bytes, moe_stream_t stream);

/* Weighted sum (section 9): y[t] = sum_j w[t][j] * y_perm[inv_pos[t*k+j]] accumulated in fp32
 * in slot order j = 0..k-1, stored as bf16 [T][d].  inv_pos comes from moe_permute; an entry
 * outside [0, T*k) is not read (that slot contributes nothing), so a bad index cannot make the
 * kernel read outside y_perm. */
moe_status moe_combine(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                       uint16_t* y, moe_stream_t stream);

/* Weighted sum of normalised expert outputs (Muse Spark Open explainer, section 9: each chosen
 * expert's output is normalised before the router-weighted sum; the normalisation is not named
 * there, and this library takes RMSNorm over the d features with no learned scale):
 *   y[t] = sum_j w[t][j] * v_j / sqrt(mean_c(v_j[c]^2) + eps),  v_j = y_perm[inv_pos[t*k+j]],
 * the mean over the d features of the bf16 row, the sum of squares and the weighted sum in
 * fp32 (slot order j = 0..k-1), stored as bf16 [T][d].  Layouts and the inv_pos rule as for
 * moe_combine.
 * eps in (0, 1] (MOE_ERR_INVALID_ARG otherwise); 1e-6 is the reading used by the tests. */
moe_status moe_combine_norm(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                            float eps, uint16_t* y, moe_stream_t stream);

/* The whole layer in one call: route -> permute -> up+SwiGLU -> down -> combine, all on
 * `stream`, with no host synchronisation.  y bf16 [T][d].  ids/w (optional, may be NULL)
 * receive the routing.  The per-expert outputs are rounded to bf16 before the weighted sum,
 * exactly as y_perm would be.  MOE_ACT_BF16 takes one of two kernel paths:
 *   - 1 <= T <= 16, d % 256 == 0, I % 256 == 0 and MXFP4 weights carrying their tensor-core
 *     copies (the *_mma fields): the expert GEMMs run on the block-scaled FP4 tensor cores in one
 *     persistent launch.  Each bf16 activation row (x, and the bf16 SwiGLU output h) is fed as
 *     the exact sum of 8 MXFP4 rows plus a residual: piece p rounds what pieces 0..p-1 left over
 *     onto the E2M1 grid with its own power-of-two block scale, so the residual after 8 pieces
 *     is below 2^-12 of each 32-element block's maximum (about 2^-24 for normal data); products
 *     are exact and accumulate in fp32.  For T <= 4 the weighted sum is fused as well.
 *   - otherwise (NVFP4 weights, no tensor-core copies, other shapes): CUDA-core GEMVs with
 *     exact products (bf16 activations, fp32 accumulation), down GEMV and weighted sum fused.
 * The step entry points (moe_expert_up_swiglu, moe_expert_down with MOE_ACT_BF16) run the
 * GEMVs.  MOE_ACT_MXFP8 runs the first path on the MXFP8 values of x and h for up to 16 tokens,
 * and the kind::mxf8f6f4 grouped GEMMs beyond (moe_expert_up_swiglu, moe_expert_down). */
moe_status moe_layer_forward(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                             int I, const moe_expert_weights* W, moe_act_fmt fmt, uint16_t* y, int32_t* ids,
                             float* w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* moe_layer_forward with the activations in host memory: the copy of x_host (bf16 [T][d]) into the
 * device buffer x_dev, the layer (x_dev -> y_dev, both bf16 [T][d] device buffers of the caller,
 * 16-byte aligned, not overlapping each other or the workspace) and the copy of y_dev back to
 * y_host, all enqueued, without waiting.
 *   in_stream or out_stream NULL: everything in order on `stream`; y_host holds the result once
 *     `stream` has passed that point (for example after cudaStreamSynchronize(stream)).
 *   both given: the copy in runs on in_stream, the layer on `stream`, the copy out on out_stream,
 *     so that a caller alternating two (x_dev, y_dev) pairs over consecutive calls has the copies
 *     of one call overlap the layers of its neighbours (one stream per direction: a copy in never
 *     queues behind a copy out, which waits for its layer).  The library orders the streams with
 *     events it keeps per staging buffer (created on first use, reused; beyond 64 buffers the least
 *     recently used one's events are released after the host has waited for them): the copy into
 *     x_dev waits for the last layer that read x_dev and for the last copy out of it (a buffer may
 *     serve as x_dev in one call and y_dev in another), the layer waits for its input copy and for
 *     the last copy out of and the last layer read of y_dev, the copy out waits for the layer.
 *     y_host holds the result once out_stream has passed that point.  Calls on the same workspace
 *     must share `stream`.
 * x_host and y_host should be page-locked (pinned) for the copies to be asynchronous; pageable
 * memory works, with copies that are synchronous with respect to the host.  The other arguments,
 * the shape rules, the workspace and the errors are moe_layer_forward's; MOE_ERR_INVALID_ARG also
 * for a null host or staging pointer.  A copy or event call that fails returns MOE_ERR_CUDA. */
moe_status moe_layer_forward_host(const uint16_t* x_host, const float* W_r, const float* b, int T, int d, int E,
                                  int k, int I, const moe_expert_weights* W, moe_act_fmt fmt, uint16_t* y_host,
                                  int32_t* ids, float* w, uint16_t* x_dev, uint16_t* y_dev, void* ws,
                                  size_t ws_bytes, moe_stream_t stream, moe_stream_t in_stream,
                                  moe_stream_t out_stream);

/* The layer with each expert's output normalised before the weighted sum (moe_combine_norm's
 * definition; eps in (0, 1]).  Same arguments, workspace and stream rules as moe_layer_forward;
 * the per-expert bf16 outputs go through the workspace (both formats), then the normalised
 * weighted sum produces y. */
moe_status moe_layer_forward_norm(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                  int I, const moe_expert_weights* W, moe_act_fmt fmt, float eps, uint16_t* y,
                                  int32_t* ids, float* w, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- dense MXFP4 linear map
 * The shared latent projections of Muse Spark Open explainer, section 9 (one matrix, shared by
 * all experts, narrows each token from 8192 to 4096 features before the router and the experts;
 * another widens the weighted sum back): y[t][n] = sum_c a(x[t])[c] * W[n][c] for x bf16 [T][K],
 * W MXFP4 [N][K], y bf16 [T][N] (fp32 accumulation, rounded once to bf16).  a(x) is the
 * activation operand of the format: MOE_ACT_BF16 uses the bf16 values (K % 128 == 0,
 * N % 128 == 0, K <= 8192, N <= 8192); MOE_ACT_MXFP4 and MOE_ACT_MXFP8 quantise each row's
 * 32-element blocks like moe_permute does and run the tcgen05 GEMM (K % 256 == 0, N % 256 == 0;
 * MXFP4: W's tensor-core copies q_mma / s_mma required; MXFP8: s_mma and q 32-byte aligned).  A latent layer is moe_dense_linear(W_in) ->
 * moe_layer_forward with d = the latent width -> moe_dense_linear(W_out).
 * ws: moe_dense_workspace_size(T, K, N, fmt) bytes, 256-byte aligned, initialised with
 * moe_workspace_init; device-side timeouts are reported through it (moe_get_device_status). */
typedef struct {
    const uint8_t* q;     /* codes  [N][K/2] */
    const uint8_t* s;     /* scales [N][K/32] */
    const uint8_t* q_mma; /* tensor-core code tiles (moe_mxfp4_codes_to_mma), MOE_ACT_MXFP4 only */
    const uint8_t* s_mma; /* tensor-core scale layout (moe_mxfp4_scales_to_mma), MOE_ACT_MXFP4 only */
} moe_mxfp4_matrix;

size_t moe_dense_workspace_size(int T, int K, int N, moe_act_fmt fmt);  /* 0 for an unsupported shape */
moe_status moe_dense_linear(const uint16_t* x, int T, int K, int N, const moe_mxfp4_matrix* W, moe_act_fmt fmt,
                            uint16_t* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------- failure-detection self-test
 * Not part of the layer.  Every barrier wait in the library's kernels is bounded: when it runs out
 * the kernel records MOE_ERR_TIMEOUT in the workspace status word and finishes, so a lost copy or
 * signal is reported by moe_get_device_status instead of hanging the GPU.  This call runs that
 * path on purpose: one kernel thread waits up to limit_us microseconds (1 .. 1000000) on an
 * mbarrier phase that nothing completes, then records MOE_ERR_TIMEOUT and returns normally.  The
 * CUDA context stays usable.  ws: an initialised workspace (only its control block is used). */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int limit_us, moe_stream_t stream);

/* ---------------------------------------------------------------- synthetic inputs
 * Not part of the layer: the counter-based generator that benchmarks and tests use to create
 * expert weights on the device.  Element n (row-major) of expert `e`'s matrix [rows][K] is
 * float32(2*(u0+u1+u2+u3) - 262140) * c, where u0..u3 are the 16-bit fields (low to high) of
 * SplitMix64(key + (n+1) * 0x9E3779B97F4A7C15) and key = SplitMix64((seed << 32) |
 * (tensor_id << 24) | e).  Writes n_experts consecutive matrices starting at expert_first to
 * out [n_experts][rows][K].  seed < 2^32, tensor_id < 256. */
moe_status moe_synth_weights(uint64_t seed, uint32_t tensor_id, uint32_t expert_first, uint32_t n_experts,
                             int64_t rows, int64_t K, float c, float* out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
