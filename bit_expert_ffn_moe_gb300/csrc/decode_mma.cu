// decode_mma.cu -- the expert GEMMs of small batches (up to 16 tokens) with bf16 or MXFP8
// activations on the block-scaled FP4 tensor cores (tcgen05, kind::mxf4).
//
// At decode sizes every chosen expert sees one or a few tokens and the layer time is the read of
// the 4-bit expert weights (Muse Spark Open explainer, section 13: at one token per expert the
// weight read dominates; DGX Spark news item, section 1: batch-1 generation is bound by weight
// reads).  The tensor cores consume the MXFP4 weights as they are stored, so no CUDA-core work is
// spent per weight: the copy engine streams 16 KB weight tiles into shared memory and one thread
// issues the MMAs.  What remains is to hand the tensor cores the bf16 activations.
//
// Activation pieces.  A bf16 row (x, or the bf16 SwiGLU output h) is written as the exact sum of
// kPieces MXFP4 rows plus a residual: piece p is the block-scaled E2M1 rounding of what the
// earlier pieces left over, r_0 = v, q_p = E2M1(r_p / 2^X_p) * 2^X_p, r_{p+1} = r_p - q_p, with
// the block exponent X_p = floor(log2 max|r_p|) - 2, raised by one when the maximum would
// saturate (so that every element lies within the grid, |r_p| / 2^X_p <= 6).  Rounding to the
// nearest grid value keeps q_p within a factor of two of r_p, so r_p - q_p is exact in fp32, and
// each piece shrinks the block's largest residual at least threefold (typically about eightfold):
// after eight pieces it lies below 2^-12 of the block maximum in the worst case and near 2^-24
// for normal data, far under the bf16 rounding of the layer's outputs.  The MMA of a piece row
// with a weight row is exact in its products and accumulates in fp32, so the piece rows of a
// token sum to its dot products.  A token t's pieces are rows 8t .. 8t+7 of the MMA's A operand
// (M = 128 rows: up to 16 tokens); the epilogue adds the eight lanes of each token.
//
// 8-bit activations (MXFP8: E4M3 elements with one E8M0 scale per 32, the 4-bit-weight /
// 8-bit-activation configuration of the DGX Spark news item, section 2): x and h are first rounded
// to their MXFP8 values, then split into pieces in the same way, so the GEMMs see the 8-bit operand
// to within the same residual.  At these sizes the tensor-core rate is irrelevant (the weight read
// bounds the layer), and pieces keep the weight tiles packed: a kind::mxf8f6f4 MMA would need its
// FP4 operand widened to one byte per value in shared memory, halving the weight bytes in flight.
//
// Kernels (one persistent CTA per SM, the same roles as the grouped prefill GEMMs in umma.cu:
// a producer warp issuing bulk copies into a 4-stage ring, an MMA warp, 8 epilogue warps):
//   up:   tile (active slot u, block p of 128 intermediate rows): A = the token pieces (one
//         128-row tile for every expert), B = 128 gate rows followed by the 128 up rows of the
//         expert, K = d.  Epilogue: per token of the expert, g and u summed over its piece lanes,
//         h = SiLU(g) * u rounded to bf16, and h's own pieces written as the A operand of the down
//         GEMM (slot u's 128-row tile, row 8j + p for the expert's j-th token).
//   down: tile (active slot u, block p of 256 output features): A = slot u's h pieces, B = 256 rows
//         of W_down, K = I.  Epilogue: per token of the expert, the sum over its piece lanes
//         rounded to bf16, stored as that permuted row of y_perm (the weighted sum follows).
// Every barrier wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, stops issuing work,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include "route_common.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kPieces = 8;
constexpr int kDecMaxT = 128 / kPieces;  // tokens whose piece rows fill one 128-row tile
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kTile = kStageTileBytes;
constexpr int kAtom = kScaleAtomBytes;
// Stage ring: every stage holds the A rows that carry data (8 piece rows per token: 1 KB of the
// 128-row tile per token, in its own 1024-byte-aligned region), the two 16 KB weight tiles and the
// six scale atoms; up to kMaxStages stages.  The MMA still reads 128 A rows: the rows past the
// live ones lie in the next region and only reach accumulator lanes that no epilogue reads.
// (Six stages for one token -- 50% more weight bytes in flight per SM -- measured slower on GB300:
// 60.5 against 57.3 us per decode step; five for four tokens: 138.5 against 137.4 us.)
constexpr int kMaxStages = 4;
constexpr int kSmemBudget = 232448;  // 227 KB per CTA
__host__ __device__ constexpr int dec_a_region(int T) { return 1024 * (T < kDecMaxT ? T : kDecMaxT); }
__host__ __device__ constexpr int dec_stage_bytes(int T) { return dec_a_region(T) + 2 * kTile + 6 * kAtom; }
constexpr int kAccCols = 256;
constexpr int kSfBase = kAccCols;
constexpr int kSfCols = 24;
constexpr uint32_t kTmemCols = 512;
constexpr int kBarBytes = 512;
static_assert(kSfBase + kMaxStages * kSfCols <= (int)kTmemCols, "tensor memory budget");

// Shared memory besides the ring: alignment slack, barriers, and the plan as every CTA holds it
// (offsets [E+1], active experts [E], pick counts [E], and per slot the token of each permuted row,
// the permuted row of each slot, the gate weight of each slot and the picked expert).
__host__ __device__ constexpr size_t dec_fixed_smem(int E, int P) {
    return 1024 + kBarBytes + sizeof(int32_t) * (size_t)(3 * E + 1 + 4 * P);
}
// stages of the ring for T tokens, E experts and k picks per token (0: does not fit)
__host__ __device__ constexpr int dec_stages(int T, int E, int k) {
    return (int)(((size_t)kSmemBudget - dec_fixed_smem(E, T * k)) / (size_t)dec_stage_bytes(T)) < kMaxStages
               ? (int)(((size_t)kSmemBudget - dec_fixed_smem(E, T * k)) / (size_t)dec_stage_bytes(T))
               : kMaxStages;
}
static_assert(dec_stages(kDecMaxT, kMaxE, kMaxK) >= 3, "the largest stages fit three deep");
static_assert(dec_stage_bytes(1) % 1024 == 0 && dec_stage_bytes(kDecMaxT) % 1024 == 0, "stage alignment");

// ------------------------------------------------------------------ activation pieces
// Block exponent of a residual block: floor(log2 amax) - 2, plus one when amax > 6 * 2^X, clamped
// to [-127, 127]; amax = 0 gives -127.  Writes 2^-X (exact) to inv.
__device__ __forceinline__ int piece_exponent(float amax, float& inv) {
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // biased exponent; 0 for 0
    int X = ef - 127 - 2;
    if (ef != 0 && amax > __uint_as_float((uint32_t)(X + 127 + 2) << 23) * 1.5f) ++X;  // amax > 6 * 2^X
    X = max(-127, min(127, X));
    inv = __uint_as_float((uint32_t)(127 - X) << 23);
    return X;
}

// Exact values of eight E2M1 codes (one 32-bit word, element 0 in the low nibble).
__device__ __forceinline__ void e2m1x8_values(uint32_t word, float (&v)[8]) {
    uint32_t h[4];
    e2m1x8_to_h2(word, h);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = h2_to_f2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// One piece of eight elements of a block whose maximum residual is amax: the E2M1 codes of
// r / 2^X (returned) and r -= their values * 2^X (exact).  Returns the scale byte in sbyte.
__device__ __forceinline__ uint32_t piece8(float (&r)[8], float amax, uint32_t& sbyte) {
    float inv;
    const int X = piece_exponent(amax, inv);
    sbyte = (uint32_t)(X + 127);
    float s[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i] = r[i] * inv;
    const uint32_t codes = e2m1x8_encode(s);
    float q[8];
    e2m1x8_values(codes, q);
    const float scale = __uint_as_float((uint32_t)(X + 127) << 23);  // 2^X (X >= -126 here or q = 0)
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] -= q[i] * (X == -127 ? __uint_as_float(0x00400000u) : scale);
    return codes;
}

// Four elements: two E2M1 bytes (element 0 in the low nibble), r -= their values * 2^X.
__device__ __forceinline__ uint32_t piece4(float (&r)[4], float amax, uint32_t& sbyte) {
    float inv;
    const int X = piece_exponent(amax, inv);
    sbyte = (uint32_t)(X + 127);
    float s8[8] = {r[0] * inv, r[1] * inv, r[2] * inv, r[3] * inv, 0.f, 0.f, 0.f, 0.f};
    const uint32_t codes = e2m1x8_encode(s8) & 0xFFFFu;
    float q[8];
    e2m1x8_values(codes, q);
    const float scale = X == -127 ? __uint_as_float(0x00400000u) : __uint_as_float((uint32_t)(X + 127) << 23);
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] -= q[i] * scale;
    return codes;
}

__device__ __forceinline__ float absmax8(const float (&r)[8]) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(r[i]));
    return m;
}

// The pieces of item i = (token t, 32-element block b) of x: rows 8t + p of the [128][d] A tile.
// mx8: the block is first rounded to its MXFP8 values (E4M3 elements, one power-of-two scale), so
// the pieces sum to the 8-bit activation operand instead of the bf16 row.
__device__ __forceinline__ void x_pieces_item(const uint16_t* __restrict__ x, int i, int d, int mx8, uint8_t* xa,
                                              uint8_t* xa_s) {
    const int nb = d / 32;
    {
        const int t = i / nb, b = i % nb;
        float r[4][8];
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * d + 32 * b);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint4 u = src[g];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                r[g][2 * m] = bf16_bits_to_f32(w[m] & 0xFFFFu);
                r[g][2 * m + 1] = bf16_bits_to_f32(w[m] >> 16);
            }
        }
        if (mx8) {
            const float amax = fmaxf(fmaxf(absmax8(r[0]), absmax8(r[1])), fmaxf(absmax8(r[2]), absmax8(r[3])));
            float inv;
            const float scale = e8m0_to_f32(mx8_scale_from_amax(amax, inv));
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float q0[4] = {r[g][0], r[g][1], r[g][2], r[g][3]}, q1[4] = {r[g][4], r[g][5], r[g][6], r[g][7]};
                mx8_round4(q0, inv, scale);
                mx8_round4(q1, inv, scale);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    r[g][m] = q0[m];
                    r[g][4 + m] = q1[m];
                }
            }
        }
#pragma unroll 1
        for (int p = 0; p < kPieces; ++p) {
            const float amax = fmaxf(fmaxf(absmax8(r[0]), absmax8(r[1])), fmaxf(absmax8(r[2]), absmax8(r[3])));
            uint32_t sb = 0;
            uint4 c;
            c.x = piece8(r[0], amax, sb);
            c.y = piece8(r[1], amax, sb);
            c.z = piece8(r[2], amax, sb);
            c.w = piece8(r[3], amax, sb);
            const int row = 8 * t + p;
            *reinterpret_cast<uint4*>(xa + mma_tile_offset(row, b, d)) = c;
            xa_s[mma_scale_offset(row, b, d)] = (uint8_t)sb;
        }
    }
}

// x pieces: one thread per (token, 32-element block).
__global__ void __launch_bounds__(256) x_pieces_kernel(const uint16_t* __restrict__ x, int T, int d, int mx8,
                                                       uint8_t* xa, uint8_t* xa_s) {
    // the next kernel (the expert GEMMs) may start its set-up now; it waits for this kernel, and so
    // for the routing, before it reads anything either produced
    pdl_launch_dependents();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < T * (d / 32)) x_pieces_item(x, i, d, mx8, xa, xa_s);
    // the next kernel's dependency wait covers this kernel's predecessors too
    pdl_wait();
}

// ------------------------------------------------------------------ the GEMMs
struct DecArgs {
    const uint8_t* xa;    // token pieces: one 128-row A tile of width d (code tiles, scale atoms)
    const uint8_t* xa_s;
    uint8_t* ha;          // h pieces: one 128-row A tile of width I per active slot (written by the
    uint8_t* ha_s;        //   gate/up epilogue, read by the down tiles of that slot)
    const uint8_t* gq;    // weights, tensor-core layouts: gate / up [E*I][d], down [E*d][I]
    const uint8_t* gs;
    const uint8_t* uq;
    const uint8_t* us;
    const uint8_t* dq;
    const uint8_t* ds;
    PlanView plan;
    const int32_t* offsets;     // [E+1] permuted-row offsets of the experts
    const int32_t* perm_token;  // [T*k]
    int T, E, k, d, I;
    uint16_t* y_perm;           // bf16 [T*k][d]
    const int32_t* inv_pos;     // fused weighted sum: [T*k] permuted row of each slot
    const float* w;             //   [T*k] gate weights
    uint16_t* y;                //   bf16 [T][d], or null (the sum is a separate launch)
    Ctrl* ctrl;
    float* part;                // split gate/up tiles: fp32 partial sums [T*k][I/128][ks][256]
    int ks;                     // K parts per gate/up tile (1: whole tiles)
    int mx8;                    // h rounded to MXFP8 (else bf16) before its pieces are formed
    int nst;                    // stages of the ring (dec_stages)
    // Routing inside the kernel (route != 0; up to kRouteMaxT tokens, E at most the grid): every CTA
    // computes the logits of its expert and a share of the token pieces, and after one grid-wide
    // arrival every CTA takes the top-k and builds the plan itself; CTA 0 writes the routing
    // outputs (ids, w, the permutation and the plan, as the one-launch router does).  Otherwise the
    // plan, offsets, perm_token, inv_pos, w and the token pieces come from the preceding kernels.
    int route;
    const uint16_t* x;          // bf16 [T][d]
    const float* W_r;           // fp32 [E][d]
    const float* bias;          // fp32 [E] or null
    float* logits;              // [T][E] (workspace)
    int32_t* ids_out;           // [T*k]
    float* w_out;               // [T*k]
    int32_t* counts_out;        // [E]
    int32_t* offsets_out;       // [E+1] (= offsets)
    int32_t* perm_out;          // [T*k] (= perm_token)
    int32_t* inv_out;           // [T*k] (= inv_pos)
    float* row_w_out;           // [T*k]
    uint8_t* xa_w;              // the token pieces this launch writes (= xa, xa_s)
    uint8_t* xa_s_w;
};

constexpr int kRouteMaxT = 8;   // tokens the in-kernel routing takes (one warp per token)

// Sum of the accumulator words of one 32-column tensor-memory load over the eight lanes of a lane
// group (lane bits 0-2), in place: afterwards lane l of the group holds, as fp32 bit patterns in v[0..4), the sums of columns 4 (l & 7) .. 4 (l & 7) + 3.
template <int HALF, int MASK>
__device__ __forceinline__ void group8_stage(uint32_t (&v)[32], int lane) {
    const bool upper = (lane & MASK) != 0;
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
        const float send = __uint_as_float(upper ? v[i] : v[i + HALF]);
        const float recv = __shfl_xor_sync(0xffffffffu, send, MASK);
        v[i] = __float_as_uint(__uint_as_float(upper ? v[i + HALF] : v[i]) + recv);
    }
}

__device__ __forceinline__ void group8_reduce32(uint32_t (&v)[32], int lane) {
    group8_stage<16, 4>(v, lane);
    group8_stage<8, 2>(v, lane);
    group8_stage<4, 1>(v, lane);
}

// One epilogue warp's arrival for 256-feature block p after its y_perm rows of a down tile are
// stored; the last of the 8 x n_act arrivals (every epilogue warp of every tile of the block)
// computes y[t][256p .. 256p + 255] = sum_j w[t][j] * y_perm[inv_pos[t k + j]] in fp32 in slot
// order, rounds it to bf16 and resets the ticket.  A slot whose row lies outside [0, T k)
// contributes nothing.
__device__ __forceinline__ void fused_sum(const DecArgs& a, int p, int n_act, int lane, const int32_t* s_inv,
                                          const float* s_w) {
    __threadfence();  // this lane's y_perm stores before the arrival
    __syncwarp();
    unsigned last = 0;
    if (lane == 0) last = atomicAdd(&a.ctrl->dec_ticket[p], 1u) == (unsigned)(8 * n_act - 1);
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    __threadfence();
    const int P = a.T * a.k, d = a.d;
    const int f = 256 * p + 8 * lane;  // this lane's 8 features
    for (int t = 0; t < a.T; ++t) {
        // lane j holds slot j's row and weight (k <= 32), broadcast below: two dependent loads per
        // token instead of two per slot
        const int rj = lane < a.k ? s_inv[t * a.k + lane] : -1;
        const float wl = lane < a.k ? s_w[t * a.k + lane] : 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < a.k; j0 += 8) {
            uint4 u[8];
            float wj[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int r = __shfl_sync(0xffffffffu, rj, (j0 + jj) & 31);
                wj[jj] = __shfl_sync(0xffffffffu, wl, (j0 + jj) & 31);
                const bool ok = j0 + jj < a.k && (unsigned)r < (unsigned)P;
                u[jj] = ok ? __ldcg(reinterpret_cast<const uint4*>(a.y_perm + (size_t)r * d + f)) : make_uint4(0, 0, 0, 0);
                if (!ok) wj[jj] = 0.f;
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {  // slot order
                const uint32_t v[4] = {u[jj].x, u[jj].y, u[jj].z, u[jj].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    acc[2 * m] = fmaf(wj[jj], bf16_bits_to_f32(v[m] & 0xFFFFu), acc[2 * m]);
                    acc[2 * m + 1] = fmaf(wj[jj], bf16_bits_to_f32(v[m] >> 16), acc[2 * m + 1]);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            o[m] = (uint32_t)f32_to_bf16_bits(acc[2 * m]) | ((uint32_t)f32_to_bf16_bits(acc[2 * m + 1]) << 16);
        *reinterpret_cast<uint4*>(a.y + (size_t)t * d + f) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (lane == 0) a.ctrl->dec_ticket[p] = 0u;  // ready for the next call
}

// A tile of the decode layer: gate/up (slot u, block p of 128 intermediate rows, K part ks of
// args.ks; K = d) or down (slot u, block p of 256 output features; K = I).
struct DecTile {
    bool up;
    int u, p, ks, e;
    int KT;    // K steps of this tile
    int KTT;   // K tiles of a whole row of the operands
    int kbase; // first K tile of this tile
    size_t a_rb, rb0, rb1;  // 128-row blocks: A operand, B rows 0..127, B rows 128..255
    const uint8_t *aq, *as, *bq0, *bs0, *bq1, *bs1;
};

__device__ __forceinline__ DecTile dec_tile(int t, const DecArgs& a, const int32_t* s_act, int n_up) {
    DecTile D;
    const int nbu = a.I / 128, nbd = a.d / 256;
    D.up = t < n_up;
    if (D.up) {
        D.u = t / (nbu * a.ks);
        const int rem = t % (nbu * a.ks);
        D.p = rem / a.ks;
        D.ks = rem % a.ks;
        D.KTT = a.d / 256;
        D.KT = D.KTT / a.ks;
        D.kbase = D.ks * D.KT;
    } else {
        const int l = t - n_up;
        D.u = l / nbd;
        D.p = l % nbd;
        D.ks = 0;
        D.KTT = D.KT = a.I / 256;
        D.kbase = 0;
    }
    D.e = s_act[D.u];
    if (D.up) {
        D.a_rb = 0;
        D.rb0 = D.rb1 = (size_t)D.e * nbu + D.p;
        D.aq = a.xa;
        D.as = a.xa_s;
        D.bq0 = a.gq;
        D.bs0 = a.gs;
        D.bq1 = a.uq;
        D.bs1 = a.us;
    } else {
        D.a_rb = D.u;
        D.rb0 = (size_t)D.e * 2 * nbd + 2 * D.p;
        D.rb1 = D.rb0 + 1;
        D.aq = a.ha;
        D.as = a.ha_s;
        D.bq0 = D.bq1 = a.dq;
        D.bs0 = D.bs1 = a.ds;
    }
    return D;
}

// The 8 pieces of four bf16 h values per lane: lanes of one 8-lane group hold one MX block of h
// (features 4 (lane & 7) .. + 3 of the block); written to rows row0 .. row0 + 7, block blk of the
// slot's down-GEMM operand (nothing is written when store is false).
__device__ __forceinline__ void h_pieces(const DecArgs& args, float (&r)[4], int lane, int blk, size_t row0,
                                         bool store) {
    const int pl = lane & 7;
#pragma unroll 1
    for (int pc = 0; pc < kPieces; ++pc) {
        float amax = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
        uint32_t sb;
        const uint32_t codes = piece4(r, amax, sb);
        if (store) {
            const size_t row = row0 + pc;
            *reinterpret_cast<uint16_t*>(args.ha + mma_tile_offset((int64_t)row, blk, args.I) + 2 * pl) =
                (uint16_t)codes;
            if (pl == 0) args.ha_s[mma_scale_offset((int64_t)row, blk, args.I)] = (uint8_t)sb;
        }
    }
}

// h = SiLU(g) * u of four features, rounded to the down GEMM's operand format: bf16, or (mx8) the
// MXFP8 value of its 32-element block, which the 8 lanes of the lane group hold together.
__device__ __forceinline__ void swiglu_round(const DecArgs& args, const float (&g)[4], const float (&u)[4],
                                             float (&r)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = __fdividef(g[i], 1.f + __expf(-g[i])) * u[i];
    if (!args.mx8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) r[i] = bf16_bits_to_f32(f32_to_bf16_bits(r[i]));
        return;
    }
    float amax = fmaxf(fmaxf(fabsf(r[0]), fabsf(r[1])), fmaxf(fabsf(r[2]), fabsf(r[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    float inv;
    const float scale = e8m0_to_f32(mx8_scale_from_amax(amax, inv));
    mx8_round4(r, inv, scale);
}

// Chunk c of a gate/up tile's columns (32 features = one MX block of h): lane pl of the token's
// group gets features 4pl .. 4pl+3.  Whole tiles: form h and write its pieces.  Split tiles:
// store this part's fp32 sums of g and u for the last part to add.
__device__ __forceinline__ void up_chunk(const DecArgs& args, const DecTile& D, uint32_t (&gv)[32], uint32_t (&uv)[32],
                                         int half, int c, int lane, int j, int r0, size_t row0) {
    group8_reduce32(gv, lane);
    group8_reduce32(uv, lane);
    const int f = 64 * half + 32 * c + 4 * (lane & 7);  // feature within the tile's 128
    if (args.ks > 1) {
        if (j >= 0) {
            float* dst = args.part + (((size_t)(r0 + j) * (args.I / 128) + D.p) * args.ks + D.ks) * 256;
            *reinterpret_cast<float4*>(dst + f) = make_float4(__uint_as_float(gv[0]), __uint_as_float(gv[1]),
                                                              __uint_as_float(gv[2]), __uint_as_float(gv[3]));
            *reinterpret_cast<float4*>(dst + 128 + f) = make_float4(__uint_as_float(uv[0]), __uint_as_float(uv[1]),
                                                                    __uint_as_float(uv[2]), __uint_as_float(uv[3]));
        }
        return;
    }
    const float g[4] = {__uint_as_float(gv[0]), __uint_as_float(gv[1]), __uint_as_float(gv[2]), __uint_as_float(gv[3])};
    const float u[4] = {__uint_as_float(uv[0]), __uint_as_float(uv[1]), __uint_as_float(uv[2]), __uint_as_float(uv[3])};
    float r[4];
    swiglu_round(args, g, u, r);
    h_pieces(args, r, lane, 4 * D.p + 2 * half + c, row0, j >= 0);
}

// Split gate/up tiles: the last of the 8 x ks warp arrivals of (slot u, block p) adds the ks partial
// sums of each of the expert's tokens in part order, forms h and writes its pieces; lane group
// lane >> 3 takes MX block (lane >> 3) of the block's 128 features.
__device__ __forceinline__ void up_finish_split(const DecArgs& args, const DecTile& D, int lane, int r0, int cnt) {
    const int nbu = args.I / 128, g8 = lane >> 3, f = 32 * g8 + 4 * (lane & 7);
    for (int j = 0; j < cnt; ++j) {
        const float* src = args.part + ((size_t)(r0 + j) * nbu + D.p) * args.ks * 256;
        float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
        for (int q = 0; q < args.ks; ++q) {
            const float4 gq = __ldcg(reinterpret_cast<const float4*>(src + (size_t)q * 256 + f));
            const float4 uq = __ldcg(reinterpret_cast<const float4*>(src + (size_t)q * 256 + 128 + f));
            g[0] += gq.x; g[1] += gq.y; g[2] += gq.z; g[3] += gq.w;
            u[0] += uq.x; u[1] += uq.y; u[2] += uq.z; u[3] += uq.w;
        }
        float r[4];
        swiglu_round(args, g, u, r);
        h_pieces(args, r, lane, 4 * D.p + g8, (size_t)D.u * 128 + 8 * (size_t)j, true);
    }
}

// Chunk c of a down tile's columns: lane pl of row group grp gets columns 4pl .. 4pl+3, stores them
// as bf16 into that permuted row of y_perm.
__device__ __forceinline__ void down_chunk(const DecArgs& args, const DecTile& D, uint32_t (&v)[32], int half, int c,
                                           int lane, int grp, int r0, int cnt) {
    const int pl = lane & 7;
    group8_reduce32(v, lane);
    if (grp < cnt) {
        const uint32_t o0 = (uint32_t)f32_to_bf16_bits(__uint_as_float(v[0])) |
                            ((uint32_t)f32_to_bf16_bits(__uint_as_float(v[1])) << 16);
        const uint32_t o1 = (uint32_t)f32_to_bf16_bits(__uint_as_float(v[2])) |
                            ((uint32_t)f32_to_bf16_bits(__uint_as_float(v[3])) << 16);
        uint16_t* dst = args.y_perm + (size_t)(r0 + grp) * args.d + (size_t)D.p * 256 + 128 * half + 32 * c + 4 * pl;
        *reinterpret_cast<uint2*>(dst) = make_uint2(o0, o1);
    }
}

// Gate/up tile epilogue of one warp (lane quarter rows, half of the columns): per token of the
// expert, g and u summed over its 8 piece lanes, h = SiLU(g) * u rounded to bf16, and h's pieces
// written as the slot's down-GEMM operand; then the warp's arrival publishes them.
__device__ __forceinline__ void epilogue_up(const DecArgs& args, const DecTile& D, uint32_t acc, int half, int grp,
                                            int lane, int r0, int cnt, const int32_t* s_perm, uint64_t* acc_empty,
                                            Ctrl* ctrl) {
    const bool live = 4 * (grp >> 2) < args.T;  // this warp's token groups include a real token
    if (live) {
        int j = -1;  // the expert's row index of token grp, or -1 when it did not choose it
        if (grp < args.T)
            for (int i = 0; i < cnt; ++i)
                if (s_perm[r0 + i] == grp) j = i;
        const size_t row0 = (size_t)D.u * 128 + 8 * (size_t)(j < 0 ? 0 : j);
        // one chunk (g and u of 32 features) at a time; the accumulator is released after the last load
        uint32_t gv[32], uv[32];
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
            tmem_ld32(acc + 32 * (2 * half + c), gv);
            tmem_ld32(acc + 128 + 32 * (2 * half + c), uv);
            tmem_ld_wait();
            if (c == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            up_chunk(args, D, gv, uv, half, c, lane, j, r0, row0);
        }
    } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
    }
    if (args.ks > 1) {
        // this warp's partial sums are stored; the last of the tile's 8 x ks warp arrivals finishes it
        __threadfence();
        __syncwarp();
        unsigned* counter = &ctrl->dec_split[D.u * (args.I / 128) + D.p];
        unsigned last = 0;
        if (lane == 0) last = atomicAdd(counter, 1u) == (unsigned)(kEpiWarps * args.ks - 1);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) return;
        __threadfence();
        up_finish_split(args, D, lane, r0, cnt);
        if (lane == 0) *counter = 0u;  // ready for the next call
    }
    // publish: h pieces in place (whole tiles: every warp's share; split tiles: the block)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(&ctrl->dec_ready[D.u], 1u);
}

// Down tile epilogue of one warp: per row of the expert, the sum over its 8 piece lanes rounded to
// bf16 and stored as that permuted row of y_perm; then (fused weighted sum) the warp's arrival.
__device__ __forceinline__ void epilogue_down(const DecArgs& args, const DecTile& D, uint32_t acc, int half, int grp,
                                              int lane, int r0, int cnt, int n_act, uint64_t* acc_empty,
                                              const int32_t* s_inv, const float* s_w) {
    const bool live = 4 * (grp >> 2) < cnt;
    if (live) {
        uint32_t v[32];
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            tmem_ld32(acc + 32 * (4 * half + c), v);
            tmem_ld_wait();
            if (c == 3) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            down_chunk(args, D, v, half, c, lane, grp, r0, cnt);
        }
    } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
    }
    if (args.y != nullptr) fused_sum(args, D.p, n_act, lane, s_inv, s_w);
}

constexpr int kTileQ = 8;  // tile-id queue from the claiming producer to the other roles

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// One persistent CTA per SM.  Roles: warp 0 claims tiles (a global counter: every gate/up tile,
// then every down tile) and streams their weight tiles and scales into the ring; warp 10 streams
// the A operand (the token pieces, or the slot's h pieces once all gate/up tiles of that slot have
// published them); warp 1 copies scales to tensor memory and issues the MMAs; warps 2-9 drain the
// accumulator.  The down tiles' weights stream while their h is still being produced.
__global__ void __launch_bounds__(kThreads + 32, 1) umma_decode_layer_kernel(const DecArgs args) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int kStages = args.nst;
    const int kStageBytes = dec_stage_bytes(args.T), kAReg = dec_a_region(args.T);
    uint64_t* full_b = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* full_a = full_b + kMaxStages;
    uint64_t* empty = full_a + kMaxStages;
    uint64_t* tq_full = empty + kMaxStages;
    uint64_t* tq_empty = tq_full + kTileQ;
    uint64_t* acc_full = tq_empty + kTileQ;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* mma_done = acc_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_tq = const_cast<int*>(abort_flag) + 1;                                           // [kTileQ]
    const int P = args.T * args.k;
    int32_t* s_off = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + kBarBytes);  // [E+1]
    int32_t* s_act = s_off + (args.E + 1);                                                  // [E]
    int32_t* s_cnt = s_act + args.E;                                                        // [E]
    int32_t* s_perm = s_cnt + args.E;                                                       // [P]
    int32_t* s_inv = s_perm + P;                                                            // [P]
    float* s_w = reinterpret_cast<float*>(s_inv + P);                                       // [P]
    int32_t* s_ids = reinterpret_cast<int32_t*>(s_w + P);                                   // [P]
    __shared__ int s_nact;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Ctrl* ctrl = args.ctrl;
    int* status = &ctrl->status;

    auto stage_a = [&](int s) { return smem + (size_t)s * kStageBytes; };
    auto stage_b = [&](int s) { return smem + (size_t)s * kStageBytes + kAReg; };
    auto stage_sfa = [&](int s) { return smem + (size_t)s * kStageBytes + kAReg + 2 * kTile; };
    auto stage_sfb = [&](int s) { return smem + (size_t)s * kStageBytes + kAReg + 2 * kTile + 2 * kAtom; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_b[s], 1);
            mbar_init(&full_a[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < kTileQ; ++q) {
            mbar_init(&tq_full[q], 1);
            mbar_init(&tq_empty[q], 2 + kEpiWarps);  // A producer, MMA warp, epilogue warps
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, kEpiWarps);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    if (args.route) {
        // ---- routing inside the kernel; the ring's memory stages the router rows meanwhile
        float* Ws = reinterpret_cast<float*>(smem);                                     // [d]
        uint16_t* xs = reinterpret_cast<uint16_t*>(smem + sizeof(float) * (size_t)args.d);  // [T][d]
        const int E = args.E, d = args.d, T = args.T, k = args.k;
        if ((int)blockIdx.x < E) route_stage_w(args.W_r, blockIdx.x, d, Ws);  // independent of earlier kernels
        for (int i = threadIdx.x; i < E; i += blockDim.x) s_cnt[i] = 0;
        pdl_wait();
        if ((int)blockIdx.x < E) route_stage_x(args.x, T, d, xs);
        // this CTA's share of the token pieces (items spread over the CTAs first, then the threads),
        // while the router rows are in flight
        for (int i = blockIdx.x + gridDim.x * threadIdx.x; i < T * (d / 32); i += gridDim.x * blockDim.x)
            x_pieces_item(args.x, i, d, args.mx8, args.xa_w, args.xa_s_w);
        if ((int)blockIdx.x < E) {  // the logits of expert blockIdx.x (E <= the grid)
            const float2 acc = route_dot_staged(Ws, xs + (size_t)(warp < T ? warp : 0) * d, nullptr, d, warp < T);
            if (warp < T && lane == 0)
                args.logits[(size_t)warp * E + blockIdx.x] = acc.x + (args.bias ? args.bias[blockIdx.x] : 0.f);
        }
        // one arrival per CTA; every CTA waits for all of them (bounded)
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(&ctrl->route_ticket, 1u);
            const long long t0 = clock64();
            while (ld_acquire_u32(&ctrl->route_ticket) < gridDim.x) {
                if (clock64() - t0 > kWaitCycles) {
                    set_status(status, MOE_ERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                __nanosleep(32);
            }
        }
        __syncthreads();
        asm volatile("fence.proxy.async.global;" ::: "memory");  // others' piece stores -> this CTA's bulk copies
        if (!*abort_flag) {
            // all T x E logits into shared memory at once (the staging area is free now), then the
            // top-k and softmax per token (warp t), the picks counted in s_cnt
            float* s_logits = Ws;
            for (int i = threadIdx.x; i < T * E; i += blockDim.x) s_logits[i] = __ldcg(args.logits + i);
            __syncthreads();
            if (warp < T) topk_softmax_warp<true>(s_logits + (size_t)warp * E, E, k, s_ids + warp * k, s_w + warp * k, s_cnt);
            __syncthreads();
            if (warp == 0) {  // offsets and the active list (and, in CTA 0, the workspace plan)
                if (blockIdx.x == 0) build_plan_warp(s_cnt, E, args.counts_out, args.offsets_out, args.plan, s_off);
                const int chunk = (E + 31) / 32, lo = min(E, lane * chunk), hi = min(E, lo + chunk);
                int c_sum = 0, a_sum = 0;
                for (int e = lo; e < hi; ++e) {
                    c_sum += s_cnt[e];
                    a_sum += s_cnt[e] > 0;
                }
                int c_inc = c_sum, a_inc = a_sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int cu = __shfl_up_sync(0xffffffffu, c_inc, o), au = __shfl_up_sync(0xffffffffu, a_inc, o);
                    if (lane >= o) {
                        c_inc += cu;
                        a_inc += au;
                    }
                }
                int c_off = c_inc - c_sum, a_off = a_inc - a_sum;
                for (int e = lo; e < hi; ++e) {
                    s_off[e] = c_off;
                    c_off += s_cnt[e];
                    if (s_cnt[e] > 0) s_act[a_off++] = e;
                }
                if (lane == 31) {
                    s_off[E] = c_inc;
                    s_nact = a_inc;
                }
            }
            __syncthreads();
            for (int p = threadIdx.x; p < P; p += blockDim.x) {  // rows ordered by (expert, token, slot)
                const int t = p / k, ex = s_ids[p];
                int rank = 0;  // tokens before t that chose ex (a token picks an expert at most once)
                for (int t2 = 0; t2 < t; ++t2)
                    for (int j = 0; j < k; ++j) rank += (s_ids[t2 * k + j] == ex);
                const int r = s_off[ex] + rank;
                s_perm[r] = t;
                s_inv[p] = r;
                if (blockIdx.x == 0) {
                    args.ids_out[p] = ex;
                    args.w_out[p] = s_w[p];
                    args.perm_out[r] = t;
                    args.inv_out[p] = r;
                    args.row_w_out[r] = s_w[p];
                }
            }
        } else if (threadIdx.x == 0) {
            s_nact = 0;  // timed out: no tiles, straight to the teardown
        }
    } else {
        pdl_wait();  // the routing plan and the token pieces come from the preceding kernels
        if (threadIdx.x == 0) s_nact = args.plan.scalars[0];
        for (int i = threadIdx.x; i <= args.E; i += blockDim.x) {
            s_off[i] = args.offsets[i];
            if (i < args.E) s_act[i] = args.plan.active[i];
        }
        for (int i = threadIdx.x; i < P; i += blockDim.x) {
            s_perm[i] = args.perm_token[i];
            if (args.y != nullptr) {
                s_inv[i] = args.inv_pos[i];
                s_w[i] = args.w[i];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_act = s_nact;

    const int nbu = args.I / 128;
    const int n_up = n_act * nbu * args.ks, n_tiles = n_up + n_act * (args.d / 256);

    // next tile id from the queue (every role but the claiming producer); -1 ends the loop
    auto next_tile = [&](int q, bool arrive) -> int {
        if (!mbar_wait(&tq_full[q % kTileQ], (uint32_t)(q / kTileQ) & 1u, abort_flag, status)) return -1;
        const int t = s_tq[q % kTileQ];
        if (arrive) mbar_arrive(&tq_empty[q % kTileQ]);
        return t;
    };

    if (warp == 0) {
        // ---------------------------------------------------------- tile claims + weight copies
        if (lane == 0) {
            int kiter = 0;
            const uint64_t l2_stream = l2_policy_evict_first();
            for (int q = 0;; ++q) {
                if (!mbar_wait(&tq_empty[q % kTileQ], ((uint32_t)(q / kTileQ) & 1u) ^ 1u, abort_flag, status)) break;
                // the first tile of every CTA is its own index; later ones are claimed from the
                // counter, which starts past them
                const unsigned c = q == 0 ? blockIdx.x : gridDim.x + atomicAdd(&ctrl->dec_tile, 1u);
                const int t = c < (unsigned)n_tiles ? (int)c : -1;
                s_tq[q % kTileQ] = t;
                mbar_arrive(&tq_full[q % kTileQ]);
                if (t < 0) break;
                const DecTile D = dec_tile(t, args, s_act, n_up);
                const int apr = D.KTT * 2;  // scale atoms per 128-row block
                const int kt0 = t % D.KT;   // concurrent tiles start at different K steps
                bool ok = true;
                for (int kk = 0; kk < D.KT; ++kk, ++kiter) {
                    const int s = kiter % kStages;
                    const int kt = D.kbase + (kk + kt0 < D.KT ? kk + kt0 : kk + kt0 - D.KT);
                    if (!mbar_wait(&empty[s], ((uint32_t)(kiter / kStages) & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_b[s], 2 * kTile + 4 * kAtom);
                    // the weights are read once per call: evict them first from L2
                    bulk_load_hint(stage_b(s), D.bq0 + (D.rb0 * D.KTT + kt) * kTile, kTile, &full_b[s], l2_stream);
                    bulk_load_hint(stage_b(s) + kTile, D.bq1 + (D.rb1 * D.KTT + kt) * kTile, kTile, &full_b[s],
                                   l2_stream);
                    bulk_load_hint(stage_sfb(s), D.bs0 + (D.rb0 * apr + 2 * kt) * kAtom, 2 * kAtom, &full_b[s],
                                   l2_stream);
                    bulk_load_hint(stage_sfb(s) + 2 * kAtom, D.bs1 + (D.rb1 * apr + 2 * kt) * kAtom, 2 * kAtom,
                                   &full_b[s], l2_stream);
                }
                if (!ok) break;
            }
            if (*abort_flag) {  // let the copies already issued land before shared memory is released
                volatile int never = 0;
                for (int i = 0; i < kStages && i < kiter; ++i) {
                    const int it = kiter - 1 - i;
                    mbar_wait(&full_b[it % kStages], (it / kStages) & 1, &never, nullptr, 100000000LL);
                }
            }
        }
    } else if (warp == kThreads / 32) {
        // ---------------------------------------------------------- A operand copies
        if (lane == 0) {
            int kiter = 0;
            for (int q = 0;; ++q) {
                const int t = next_tile(q, true);
                if (t < 0) break;
                const DecTile D = dec_tile(t, args, s_act, n_up);
                const int cnt = s_off[D.e + 1] - s_off[D.e];
                const int rows = 8 * (D.up ? args.T : cnt);
                const uint32_t a_bytes = (uint32_t)(rows < 128 ? rows : 128) * 128;
                const int kt0 = t % D.KT;
                bool ok = true;
                // Down tiles wait for the slot's h pieces, published by every epilogue warp of a whole
                // gate/up tile or once per 128-row block by a split tile's last part.  (Waiting per
                // block, just before the K step that reads it, was measured slower: each acquiring
                // poll costs a round trip under full load.)
                auto wait_ready = [&](const unsigned* ctr, unsigned need) {
                    const long long t0 = clock64();
                    while (ld_acquire_u32(ctr) < need) {
                        if (*abort_flag || clock64() - t0 > kWaitCycles) {
                            set_status(status, MOE_ERR_TIMEOUT);
                            *abort_flag = 1;
                            return false;
                        }
                        __nanosleep(64);
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");  // generic stores -> bulk copies
                    return true;
                };
                const unsigned per_block = (unsigned)(args.ks > 1 ? 1 : kEpiWarps);
                if (!D.up) ok = wait_ready(&ctrl->dec_ready[D.u], per_block * nbu);
                for (int kk = 0; kk < D.KT && ok; ++kk, ++kiter) {
                    const int s = kiter % kStages;
                    const int kt = D.kbase + (kk + kt0 < D.KT ? kk + kt0 : kk + kt0 - D.KT);
                    if (!mbar_wait(&empty[s], ((uint32_t)(kiter / kStages) & 1u) ^ 1u, abort_flag, status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_a[s], a_bytes + 2 * kAtom);
                    bulk_load(stage_a(s), D.aq + (D.a_rb * D.KTT + kt) * kTile, a_bytes, &full_a[s]);
                    bulk_load(stage_sfa(s), D.as + (D.a_rb * D.KTT * 2 + 2 * kt) * kAtom, 2 * kAtom, &full_a[s]);
                }
                if (!ok) break;
            }
            if (*abort_flag) {
                volatile int never = 0;
                for (int i = 0; i < kStages && i < kiter; ++i) {
                    const int it = kiter - 1 - i;
                    mbar_wait(&full_a[it % kStages], (it / kStages) & 1, &never, nullptr, 100000000LL);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer (whole warp)
        int kiter = 0, it = 0;
        const uint32_t idesc = idesc_mxf4(128, 256);
        for (int q = 0;; ++q, ++it) {
            int t = next_tile(q, false);
            if (lane == 0 && t >= 0) mbar_arrive(&tq_empty[q % kTileQ]);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t < 0) break;
            const DecTile D = dec_tile(t, args, s_act, n_up);
            if (!mbar_wait_warp(acc_empty, (it & 1) ^ 1, abort_flag, status)) break;
            tc_fence_after();
            bool ok = true;
            for (int kt = 0; kt < D.KT; ++kt, ++kiter) {
                const int s = kiter % kStages;
                const uint32_t ph = (kiter / kStages) & 1;
                if (!mbar_wait_warp(&full_b[s], ph, abort_flag, status) ||
                    !mbar_wait_warp(&full_a[s], ph, abort_flag, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sf = tmem + kSfBase + s * kSfCols;
                stage_scales_to_tmem(sf, desc_sf(stage_sfa(s)), desc_sf(stage_sfa(s) + kAtom), desc_sf(stage_sfb(s)),
                                     desc_sf(stage_sfb(s) + 2 * kAtom), desc_sf(stage_sfb(s) + kAtom),
                                     desc_sf(stage_sfb(s) + 3 * kAtom));
                stage_mmas_commit(tmem, desc_sw128(stage_a(s)), desc_sw128(stage_b(s)), idesc,
                                  idesc | (2u << 29) | (2u << 4), sf, kt > 0 ? 1u : 0u, &empty[s]);
            }
            if (!ok) break;
            tc_commit(acc_full);
        }
        tc_commit(mma_done);
        volatile int never = 0;
        mbar_wait_warp(mma_done, 0, &never, nullptr, 100000000LL);
    } else {
        // ---------------------------------------------------------- epilogue (warps 2-9)
        const int q4 = warp & 3;          // tensor-memory lane quarter: rows 32q4 .. 32q4 + 31
        const int half = (warp - 2) / 4;  // half of the accumulator columns
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const int grp = 4 * q4 + (lane >> 3);  // 8-row group: token grp (gate/up) or the expert's row grp (down)
        int it = 0;
        for (int q = 0;; ++q, ++it) {
            int t = next_tile(q, false);
            if (lane == 0 && t >= 0) mbar_arrive(&tq_empty[q % kTileQ]);
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t < 0) break;
            const DecTile D = dec_tile(t, args, s_act, n_up);
            const int r0 = s_off[D.e], cnt = s_off[D.e + 1] - r0;
            if (!mbar_wait(acc_full, it & 1, abort_flag, status)) break;
            tc_fence_after();
            if (D.up)
                epilogue_up(args, D, tmem + lane_base, half, grp, lane, r0, cnt, s_perm, acc_empty, ctrl);
            else
                epilogue_down(args, D, tmem + lane_base, half, grp, lane, r0, cnt, n_act, acc_empty, s_inv, s_w);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (threadIdx.x == 0 && !(*abort_flag)) {
        // the last CTA out resets the claim counter and the slots' arrival counts for the next call
        __threadfence();
        if (atomicAdd(&ctrl->dec_done, 1u) == gridDim.x - 1) {
            for (int u = 0; u < n_act; ++u) ctrl->dec_ready[u] = 0u;
            ctrl->dec_tile = 0u;
            if (args.route) ctrl->route_ticket = 0u;
            __threadfence();
            ctrl->dec_done = 0u;
        }
    }
    pdl_launch_dependents();
}

}  // namespace

static_assert(kDecMaxT == kMmaDecodeMaxT, "decode tile geometry");

bool mma_decode_supported(int T, int d, int E, int k, int I, const moe_expert_weights* W) {
    return mma_decode_shape(T, d, I) && (T * k < E ? T * k : E) <= kDecSlots && W->wfmt == MOE_W_MXFP4 &&
           W->gate_q_mma && W->gate_s_mma && W->up_q_mma && W->up_s_mma && W->down_q_mma && W->down_s_mma;
}

bool mma_decode_fused_sum(int T, int d) { return T <= 4 && d / 256 <= kDecTickets; }

bool mma_decode_route_supported(int T, int d, int E, int k) {
    const int nst = dec_stages(T, E, k);
    return T >= 1 && T <= kRouteMaxT && E <= sm_count() &&
           sizeof(float) * (size_t)d + sizeof(uint16_t) * (size_t)T * d <= (size_t)nst * dec_stage_bytes(T);
}

cudaError_t launch_x_pieces(const uint16_t* x, int T, int d, bool mx8, uint8_t* xa, uint8_t* xa_s, cudaStream_t st,
                            bool pdl) {
    const int n = T * (d / 32);
    int m8 = mx8 ? 1 : 0;
    void* args[] = {&x, &T, &d, &m8, &xa, &xa_s};
    return launch_kernel((const void*)x_pieces_kernel, dim3((n + 255) / 256), dim3(256), 0, st, pdl, args);
}

cudaError_t launch_mma_decode(const uint8_t* xa, const uint8_t* xa_s, uint8_t* ha, uint8_t* ha_s, float* part,
                              PlanView plan, const int32_t* offsets, const int32_t* perm_token, int T, int d, int E,
                              int k, int I, const moe_expert_weights* W, bool mx8, uint16_t* y_perm,
                              const int32_t* inv_pos, const float* w, uint16_t* y, Ctrl* ctrl, cudaStream_t st,
                              bool pdl, const DecRoute* route) {
    DecArgs a = {};
    a.mx8 = mx8 ? 1 : 0;
    if (route != nullptr) {
        a.route = 1;
        a.x = route->x;
        a.W_r = route->W_r;
        a.bias = route->b;
        a.logits = route->logits;
        a.ids_out = route->ids;
        a.w_out = route->w;
        a.counts_out = route->counts;
        a.row_w_out = route->row_w;
        a.offsets_out = const_cast<int32_t*>(offsets);
        a.perm_out = const_cast<int32_t*>(perm_token);
        a.inv_out = const_cast<int32_t*>(inv_pos);
        a.xa_w = const_cast<uint8_t*>(xa);
        a.xa_s_w = const_cast<uint8_t*>(xa_s);
    }
    const int slots = T * k < E ? T * k : E;
    a.ks = slots * (I / 128) <= kDecSplitCounters ? mma_decode_ksplit(T, d) : 1;
    a.part = part;
    a.xa = xa;
    a.xa_s = xa_s;
    a.ha = ha;
    a.ha_s = ha_s;
    a.gq = W->gate_q_mma;
    a.gs = W->gate_s_mma;
    a.uq = W->up_q_mma;
    a.us = W->up_s_mma;
    a.dq = W->down_q_mma;
    a.ds = W->down_s_mma;
    a.plan = plan;
    a.offsets = offsets;
    a.perm_token = perm_token;
    a.T = T;
    a.E = E;
    a.k = k;
    a.d = d;
    a.I = I;
    a.y_perm = y_perm;
    a.inv_pos = inv_pos;
    a.w = w;
    a.y = (y != nullptr && mma_decode_fused_sum(T, d)) ? y : nullptr;
    a.ctrl = ctrl;
    a.nst = dec_stages(T, E, k);
    void* kargs[] = {&a};
    return launch_kernel((const void*)umma_decode_layer_kernel, dim3(sm_count()), dim3(kThreads + 32),
                         dec_fixed_smem(E, T * k) + (size_t)a.nst * dec_stage_bytes(T), st, pdl, kargs);
}

}  // namespace moe
