// common.cuh -- shared device helpers and the workspace layout of the MoE layer library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kPadRows = 128;   // expert row groups of the MXFP4 path start at multiples of this
constexpr int kTokTile = 128;   // token tile (MMA N) of the tcgen05 grouped GEMMs

// ------------------------------------------------------------------ workspace layout
// Control block (first 8 KB, zeroed by moe_workspace_init): status word, decode-route ticket, and
// the counters of the tensor-core decode kernel (decode_mma.cu): its tile claims and finished
// CTAs, per active slot the epilogue arrivals that publish the slot's h operand, per 256-feature
// block the arrivals of the down tiles (the last computes the block's weighted sum).  Every counter
// is back at zero when a call completes (after a device-side timeout, initialise the workspace
// again).
constexpr int kDecTickets = 64;
constexpr int kDecSlots = 512;
constexpr int kDecSplitCounters = 1024;  // (slot, block) arrival counters of split gate/up tiles
struct Ctrl {
    int status;
    unsigned route_ticket;
    unsigned dec_tile;
    unsigned dec_done;
    unsigned dec_ticket[kDecTickets];
    unsigned dec_ready[kDecSlots];
    unsigned dec_split[kDecSplitCounters];
    int pad[444];
};
static_assert(sizeof(Ctrl) == 8192, "control block size");

// Per-call plan written by the permutation and read by the expert kernels (int32 words).
struct PlanView {
    int32_t* counts;       // [E]   scratch counts (zeroed by the count pass)
    int32_t* pad_offsets;  // [E+1] padded row start of each expert (multiples of kPadRows)
    int32_t* ttile_prefix; // [E+1] exclusive prefix of ceil(count / kTokTile)
    int32_t* active;       // [E]   experts with count > 0, ascending
    int32_t* scalars;      // [8]   0: n_active, 1: total token tiles, 2: padded rows used
};

struct WsLayout {
    size_t ctrl = 0, logits = 0, plan = 0, ids = 0, w = 0, counts = 0, offsets = 0, perm = 0, inv = 0, row_w = 0,
           xq = 0, xs = 0, xa = 0, xa_s = 0, h = 0, h_s = 0, y_perm = 0, total = 0;
    size_t dxa = 0, dxa_s = 0, dha = 0, dha_s = 0;  // decode on the tensor cores: x and h pieces
    size_t dpart = 0;                                // its split gate/up tiles' fp32 partial sums
    size_t xa_s16 = 0, h_s16 = 0, xrf = 0, hrf = 0;  // NVFP4 weights: operand scales per 16, row factors
    size_t rs_bhi = 0, rs_blo = 0, rs_wn2 = 0, rs_part = 0, rs_xn2 = 0, rs_cnt = 0, rs_list = 0;  // screened router
    size_t rs_stat = 0;
    int64_t pad_rows = 0;
};

// Decode on the tensor cores (decode_mma.cu): at most 16 tokens, whose activation rows are fed to
// the block-scaled FP4 MMAs as 8 MXFP4 pieces each (rows of one 128-row operand tile).
constexpr int kMmaDecodeMaxT = 16;
inline bool mma_decode_shape(int T, int d, int I) { return T >= 1 && T <= kMmaDecodeMaxT && d % 256 == 0 && I % 256 == 0; }
// K splits of a gate/up tile (1 = whole tiles): with one or two tokens there are too few gate/up
// tiles to occupy every SM, so each tile's K range is split into two parts of at least 8 K steps
// whose fp32 partial sums are added by the part that finishes last.  (Measured at one token,
// d = 8192: 54.6 us per step with whole tiles, 51.1 with two parts, 53.8 with four -- more parts
// fill the SMs but lengthen the partial-sum hand-off that the down tiles wait for; half tiles of
// 64 gate + 64 up rows with the full K range, which need no partial sums, took 60.1 us with 16 KB
// weight stages and 54.0 us with two K steps per stage (twice the MMAs and scale copies per weight
// byte); the two parts on the two CTAs of a cluster, partial sums exchanged through distributed
// shared memory, took 56.9 us, also when only the gate/up tiles are claimed in pairs and the down
// tiles alone (57.1 us; the same code with the pairing switched off: 51.8 us).)
inline int mma_decode_ksplit(int T, int d) {
    const int kt = d / 256;
    if (T > 2) return 1;
    return (kt % 2 == 0 && kt / 2 >= 8) ? 2 : 1;
}
// bytes of those partial sums: per token row of the layer, per 128-row block, per part, 128 g + 128 u
inline size_t mma_decode_part_bytes(int T, int d, int k, int I) {
    const int ks = mma_decode_ksplit(T, d);
    return ks > 1 ? (size_t)T * k * (I / 128) * ks * 256 * sizeof(float) : 0;
}

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Router of many tokens (route_screen.cu): tensor-core screen of the logits with a certified bound,
// fixed-order logits for the candidates only.  S = K splits of the screen (0: the dense fixed-order
// kernel routes this shape).
struct RouterScreenSizes {
    int S;
    size_t b_bytes, wn2_bytes, part_bytes, xn2_bytes, cnt_bytes, list_bytes, stat_bytes;
};
struct RouterScreenBufs {
    uint8_t* bhi;   // bf16 high parts of W_r, tensor-core tiles [E_pad/128][d/64]
    uint8_t* blo;   // bf16 low parts
    float* wn2;     // [4][E] shares of ||w_e||^2 (quarters of the row)
    float* part;    // [S][T][E_pad] screened values per K split
    float* xn2;     // [S][T] ||x_t||^2 per K split
    int32_t* cnt;   // [E] candidates per expert
    int32_t* list;  // [E][T] candidate tokens of each expert
    uint32_t* stat; // [4] max ||w_e||^2, max |b_e| (bit patterns), all finite (1 / 0)
};
int router_screen_splits(int T, int d, int E);
RouterScreenSizes router_screen_sizes(int T, int d, int E);

inline int64_t padded_rows(int T, int k, int E) {
    int64_t P = (int64_t)T * k;
    int64_t touched = P < E ? P : E;
    return align_up((size_t)(P + touched * (kPadRows - 1)), kPadRows);
}

inline size_t mma_scale_bytes(int64_t rows, int64_t K) {
    if (rows % 128 != 0 || K % 128 != 0) return 0;
    return (size_t)(rows / 128) * (size_t)(K / 128) * 512;
}

inline WsLayout ws_layout(int T, int d, int E, int k, int I, moe_act_fmt fmt) {
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    int64_t P = (int64_t)T * k;
    L.ctrl = take(sizeof(Ctrl));
    L.logits = take(sizeof(float) * (size_t)T * E);
    L.plan = take(sizeof(int32_t) * (size_t)(4 * E + 2 + 8));
    L.ids = take(sizeof(int32_t) * (size_t)P);
    L.w = take(sizeof(float) * (size_t)P);
    L.counts = take(sizeof(int32_t) * (size_t)E);
    L.offsets = take(sizeof(int32_t) * (size_t)(E + 1));
    L.perm = take(sizeof(int32_t) * (size_t)P);
    L.inv = take(sizeof(int32_t) * (size_t)P);
    L.row_w = take(sizeof(float) * (size_t)P);
    const RouterScreenSizes rs = router_screen_sizes(T, d, E);
    if (rs.S) {
        L.rs_bhi = take(rs.b_bytes);
        L.rs_blo = take(rs.b_bytes);
        L.rs_wn2 = take(rs.wn2_bytes);
        L.rs_part = take(rs.part_bytes);
        L.rs_xn2 = take(rs.xn2_bytes);
        L.rs_cnt = take(rs.cnt_bytes);
        L.rs_list = take(rs.list_bytes);
        L.rs_stat = take(rs.stat_bytes);
    }
    if (fmt == MOE_ACT_MXFP4 || fmt == MOE_ACT_MXFP8) {
        const size_t per_byte = fmt == MOE_ACT_MXFP4 ? 2 : 1;  // values per code byte
        L.pad_rows = padded_rows(T, k, E);
        L.xq = take((size_t)T * d / per_byte);
        L.xs = take((size_t)T * d / 32);
        L.xa = take((size_t)L.pad_rows * d / per_byte);
        L.xa_s = take(mma_scale_bytes(L.pad_rows, d));
        L.h = take((size_t)L.pad_rows * I / per_byte);
        L.h_s = take(mma_scale_bytes(L.pad_rows, I));
        L.y_perm = take(sizeof(uint16_t) * (size_t)P * d);
        if (fmt == MOE_ACT_MXFP4) {  // NVFP4 weights on the tensor cores
            L.xa_s16 = take(mma_scale_bytes(L.pad_rows, 2 * (int64_t)d));
            L.h_s16 = take(mma_scale_bytes(L.pad_rows, 2 * (int64_t)I));
            L.xrf = take(sizeof(float) * (size_t)L.pad_rows);
            L.hrf = take(sizeof(float) * (size_t)L.pad_rows);
        }
    } else {
        L.h = take(sizeof(uint16_t) * (size_t)P * I);
        L.y_perm = take(sizeof(uint16_t) * (size_t)P * d);  // expert outputs (normalised layer, tensor-core decode)
    }
    if (fmt != MOE_ACT_MXFP4 && mma_decode_shape(T, d, I)) {  // decode on the tensor cores (bf16, MXFP8)
        const size_t slots = (size_t)(P < E ? P : E);
        L.dxa = take((size_t)128 * d / 2);
        L.dxa_s = take(mma_scale_bytes(128, d));
        L.dha = take(slots * 128 * I / 2);
        L.dha_s = take(slots * mma_scale_bytes(128, I));
        L.dpart = take(mma_decode_part_bytes(T, d, k, I));
    }
    L.total = off;
    return L;
}

// Workspace of the dense MXFP4 linear map (y = x W^T, x [T][K], W [N][K]), run as the down GEMM
// of one expert holding every row: control block, one-expert plan, offsets, identity permutation
// and, for MOE_ACT_MXFP4 / MXFP8, the quantised rows and the padded operand tiles of width K.
inline WsLayout dense_layout(int T, int K, int N, moe_act_fmt fmt) {
    (void)N;
    WsLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.ctrl = take(sizeof(Ctrl));
    L.plan = take(sizeof(int32_t) * (size_t)(4 * 1 + 2 + 8));
    L.offsets = take(sizeof(int32_t) * 2);
    L.perm = take(sizeof(int32_t) * (size_t)T);
    if (fmt == MOE_ACT_MXFP4 || fmt == MOE_ACT_MXFP8) {
        const size_t per_byte = fmt == MOE_ACT_MXFP4 ? 2 : 1;  // values per code byte
        L.pad_rows = padded_rows(T, 1, 1);
        L.xq = take((size_t)T * K / per_byte);
        L.xs = take((size_t)T * K / 32);
        L.xa = take((size_t)L.pad_rows * K / per_byte);
        L.xa_s = take(mma_scale_bytes(L.pad_rows, K));
    }
    L.total = off;
    return L;
}

inline PlanView plan_view(void* ws, const WsLayout& L, int E) {
    int32_t* p = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + L.plan);
    PlanView v;
    v.counts = p;
    v.pad_offsets = p + E;
    v.ttile_prefix = p + 2 * E + 1;
    v.active = p + 3 * E + 2;
    v.scalars = p + 4 * E + 2;
    return v;
}

// ------------------------------------------------------------------ device helpers
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// E8M0 scale byte -> 2^(s-127) as fp32 (s = 0 is the subnormal 2^-127; 255 is never produced).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

// Record the first device-side error in the workspace status word.
__device__ __forceinline__ void set_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Eight E2M1 codes of one 32-bit word (element 2m in the low nibble of byte m) -> 4 f16x2.
// The hardware conversion puts the low nibble of each byte in the low half.
__device__ __forceinline__ void e2m1x8_to_h2(uint32_t word, uint32_t (&h)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(word));
}

__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
    __half2 v = *reinterpret_cast<__half2*>(&h);
    return __half22float2(v);
}

// MX quantisation of eight elements already divided by the block scale 2^X (an exact power-of-
// two product): each is rounded to nearest on the E2M1 magnitude grid {0, .5, 1, 1.5, 2, 3, 4, 6},
// ties to the even code, saturating at 6 (OCP MX rule).  That is what the hardware conversion to
// E2M1 does (round to nearest even, satfinite); it returns -0 for a negative value that rounds to
// zero, which is cleared to code 0.  Element 0 lands in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8_encode(const float* a) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
    const uint32_t mag = r & 0x77777777u;
    const uint32_t nonzero = (mag + 0x77777777u) & 0x88888888u;  // bit 3 of a nibble: magnitude != 0
    return mag | (r & nonzero);
}

// Two E4M3 bytes (OCP OFP8: bias 7, subnormals, largest finite 448) -> their values as fp32; the
// byte in bits 0..7 becomes .x.  Every E4M3 value is an f16 value, so the hardware conversion to
// f16 pairs is exact.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two) {
    uint32_t h;
    asm("{\n\t.reg .b16 p;\n\t"
        "cvt.u16.u32 p, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, p;\n\t}"
        : "=r"(h)
        : "r"(two));
    return h2_to_f2(h);
}

// fp32 t >= 0 -> the nearest E4M3 byte, ties to even, saturating at 448 (hardware conversion).
__device__ __forceinline__ uint32_t f32_to_e4m3_sat(float t) {
    uint32_t r;
    asm("{\n\t.reg .b16 p;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 p, %1, %1;\n\t"
        "cvt.u32.u16 %0, p;\n\t}"
        : "=r"(r)
        : "f"(t));
    return r & 0xFFu;  // both halves hold the same conversion
}

// Block exponent X = floor(log2(amax)) - 2 clamped to [-127, 127] (amax = 0 gives -127).
// Returns the scale byte X + 127 and writes 2^-X (exact) to inv_scale.
__device__ __forceinline__ uint32_t mx_scale_from_amax(float amax, float& inv_scale) {
    int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // biased exponent; 0 for zero/subnormal
    int X = ef - 127 - 2;
    if (X < -127) X = -127;
    inv_scale = __uint_as_float((uint32_t)(127 - X) << 23);
    return (uint32_t)(X + 127);
}

// ------------------------------------------------------------------ MXFP8 (E4M3 elements)
// Block exponent of the 8-bit MX format: X = floor(log2(amax)) - 8 (8 = the exponent of E4M3's
// largest normal, 448 = 1.75 * 2^8) clamped to [-127, 127]; amax = 0 or below 2^-126 gives -127.
// Returns the scale byte X + 127 and writes 2^-X (exact) to inv_scale.
__device__ __forceinline__ uint32_t mx8_scale_from_amax(float amax, float& inv_scale) {
    int X = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 8;
    if (X < -127) X = -127;
    inv_scale = __uint_as_float((uint32_t)(127 - X) << 23);
    return (uint32_t)(X + 127);
}

// Four values already divided by the block scale -> four E4M3 bytes (element 0 in bits 0..7):
// nearest E4M3 value, ties to even, saturating at 448 (the hardware conversion), with the sign
// of the value unless its magnitude rounds to zero (a zero is stored as +0).
__device__ __forceinline__ uint32_t e4m3x4_encode(float a0, float a1, float a2, float a3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    const uint32_t mag = r & 0x7F7F7F7Fu;
    const uint32_t nonzero = (mag + 0x7F7F7F7Fu) & 0x80808080u;  // bit 7 of a byte: magnitude != 0
    return mag | (r & nonzero);
}

// A whole 32-element block in MXFP8: returns the scale byte and writes the 32 code bytes (element
// i in byte i % 16 of c[i / 16]).
__device__ __forceinline__ uint32_t mx8_block_encode(const float (&v)[32], uint4 (&c)[2]) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float inv;
    const uint32_t sb = mx8_scale_from_amax(amax, inv);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = e4m3x4_encode(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    c[0] = make_uint4(w[0], w[1], w[2], w[3]);
    c[1] = make_uint4(w[4], w[5], w[6], w[7]);
    return sb;
}

// Four values of a block rounded in place to their MXFP8 values (E4M3 value * 2^X, exact in fp32)
// given the block's 2^-X and 2^X.
__device__ __forceinline__ void mx8_round4(float (&v)[4], float inv, float scale) {
    const uint32_t c = e4m3x4_encode(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
    const float2 lo = e4m3x2_to_f2(c & 0xFFFFu), hi = e4m3x2_to_f2(c >> 16);
    v[0] = lo.x * scale;
    v[1] = lo.y * scale;
    v[2] = hi.x * scale;
    v[3] = hi.y * scale;
}

// A whole 32-element block: returns the scale byte and writes the 16 bytes of codes
// (v is overwritten with v / 2^X).
__device__ __forceinline__ uint32_t mx_block_encode(float (&v)[32], uint4& codes) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    float inv;
    const uint32_t sb = mx_scale_from_amax(amax, inv);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= inv;
    codes.x = e2m1x8_encode(v);
    codes.y = e2m1x8_encode(v + 8);
    codes.z = e2m1x8_encode(v + 16);
    codes.w = e2m1x8_encode(v + 24);
    return sb;
}

// Byte offset of (row, scale column) in the tensor-core scale layout of a matrix whose rows
// carry K/32 scale columns.
__host__ __device__ __forceinline__ size_t mma_scale_offset(int64_t row, int64_t col, int64_t K) {
    int64_t atoms_per_row_block = K / 128;
    int64_t atom = (row / 128) * atoms_per_row_block + col / 4;
    return (size_t)atom * 512 + (size_t)((row % 32) * 16 + ((row / 32) % 4) * 4 + (col % 4));
}

// Byte offset of the 16-byte code chunk of (row, 32-element block blk) in the tensor-core code
// tiles of a matrix with K values per row: tiles of 128 rows x 256 values (16384 bytes) at tile
// index (row/128)*(K/256) + blk/8, chunk blk%8 of row r stored at r*128 + ((blk%8) ^ (r%8))*16.
__host__ __device__ __forceinline__ size_t mma_tile_offset(int64_t row, int64_t blk, int64_t K) {
    const int64_t tile = (row / 128) * (K / 256) + blk / 8;
    const int64_t r = row % 128;
    return (size_t)tile * 16384 + (size_t)(r * 128 + (((blk % 8) ^ (r % 8)) * 16));
}

// Byte offset of the 16-byte chunk c (elements 16c .. 16c+15) of a row in the tensor-core tiles of
// an E4M3 matrix with K values (bytes) per row: tiles of 128 rows x 128 values (16384 bytes) at
// tile index (row/128)*(K/128) + c/8, chunk c%8 of row r stored at r*128 + ((c%8) ^ (r%8))*16.
__host__ __device__ __forceinline__ size_t mma8_tile_offset(int64_t row, int64_t c, int64_t K) {
    const int64_t tile = (row / 128) * (K / 128) + c / 8;
    const int64_t r = row % 128;
    return (size_t)tile * 16384 + (size_t)(r * 128 + (((c % 8) ^ (r % 8)) * 16));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------------ mbarriers and bulk copies
constexpr long long kWaitCycles = 4000000000LL;  // bound of a device-side wait: about two seconds at GB300 clocks

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false when the CTA is
// aborting (another role timed out) or this wait ran out (then it records the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (*abort_flag) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) {
            set_status(status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// L2 policy for data read once per call: evicted first, so that a stream larger than L2 does not
// push out what later calls reuse (the code of the kernels, router weights, control counters).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_load with an L2 cache policy (l2_policy_evict_first).
__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's results / let the next
// kernel start its prologue.  No-ops when the launch did not use the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace moe

// ------------------------------------------------------------------ host-side checks (api.cu)
namespace moe {
moe_status check_device();                 // MOE_ERR_DEVICE unless the current device is sm_103
moe_status from_cuda(cudaError_t e);       // MOE_ERR_CUDA (recorded for moe_last_cuda_error) or MOE_OK
// Shape rules of the layer entry points (MOE_ERR_UNSUPPORTED_SHAPE / MOE_ERR_INVALID_ARG).
moe_status check_shape(int T, int d, int E, int k, int I, moe_act_fmt fmt);
}  // namespace moe

// ------------------------------------------------------------------ host-side launch entry points
// (one per kernel family; defined in the .cu files, called by api.cu)
namespace moe {
// Raise a kernel's dynamic shared-memory limit on the current device once; later calls with the
// same or a smaller size do not touch the runtime (so launches inside a stream capture make no
// attribute calls once the first, uncaptured call has run).
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);
// Launch with the programmatic-dependent-launch attribute when pdl is true.
cudaError_t launch_kernel(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool pdl,
                          void** args);
int sm_count();  // SMs of the current device

cudaError_t launch_synth(uint64_t seed, uint32_t tensor_id, uint32_t expert_first, uint32_t n_experts, int64_t rows,
                         int64_t K, float c, float* out, cudaStream_t st);
cudaError_t launch_pack(const float* w, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, cudaStream_t st);
cudaError_t launch_unpack(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K, float* w, cudaStream_t st);
cudaError_t launch_scales_to_mma(const uint8_t* s, int64_t rows, int64_t K, uint8_t* s_mma, cudaStream_t st);
cudaError_t launch_nvfp4_pack(const float* w, int64_t n_mats, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                              float* gs, cudaStream_t st);
cudaError_t launch_nvfp4_unpack(const uint8_t* q, const uint8_t* s, const float* gs, int64_t n_mats, int64_t rows,
                                int64_t K, float* w, cudaStream_t st);
cudaError_t launch_codes_to_mma(const uint8_t* q, int64_t rows, int64_t K, uint8_t* q_mma, cudaStream_t st);

// zero_counts (optional): counts[E] zeroed for the counting top-k that follows.
cudaError_t launch_route_logits(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E,
                                float* logits, cudaStream_t st, bool pdl, int32_t* zero_counts = nullptr);
// counts (optional): the picks also counted per expert into counts[E], which the caller has zeroed.
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t st, bool pdl,
                        int32_t* counts = nullptr);
// The screened router (route_screen.cu): logits (exact fixed-order values for every candidate, -inf
// for the experts the screen ruled out), then launch_topk's ids and w.
// cudaErrorNotSupported when the shape or the operands' alignment does not allow it or the
// tensor-map encoder is missing (route with the dense kernel).
// counts (optional): zeroed by the route's first launch, then the picks counted per expert.
cudaError_t launch_router_screen(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                 const RouterScreenBufs& rb, float* logits, int32_t* ids, float* w, int* status,
                                 cudaStream_t st, bool pdl, int32_t* counts = nullptr);
// Decode route: logits, then the last CTA runs top-k and the whole permutation (small T).
cudaError_t launch_route_decode(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                float* logits, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                int32_t* perm_token, int32_t* inv_pos, float* row_w, PlanView plan, Ctrl* ctrl,
                                cudaStream_t st, bool pdl);
bool route_decode_supported(int T, int d, int E, int k);

// The permutation from counts a counting top-k left in plan.counts (one launch: offsets, plan,
// permuted rows); the other arguments as launch_permute's.
cudaError_t launch_permute_counted(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                                   int32_t* perm_token, int32_t* inv_pos, PlanView plan, cudaStream_t st, bool pdl,
                                   const float* w = nullptr, float* row_w = nullptr);
// row_w (optional, with w): gate weight of each permuted row, row_w[inv_pos[t*k+j]] = w[t][j].
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_pos, PlanView plan, cudaStream_t st, bool pdl,
                           const float* w = nullptr, float* row_w = nullptr);
// The token operand of the prefill GEMMs: each row of x quantised once (xq, xs), then gathered into
// padded expert-grouped tensor-core tiles (xa, xa_s).  fp8: MXFP8 (E4M3 bytes), else MXFP4.
cudaError_t launch_act_quant_gather(const uint16_t* x, int T, int d, int E, int k, const int32_t* offsets,
                                    const int32_t* perm_token, PlanView plan, int64_t pad_rows, uint8_t* xq,
                                    uint8_t* xs, uint8_t* xa, uint8_t* xa_s, bool fp8, cudaStream_t st, bool pdl);
// The two halves of it: each row of x quantised once (reads x only, so it may run before the
// router), then the gather into the padded tiles (after the permutation).  zero_pad = false leaves
// each expert's padding rows unwritten: the expert GEMMs' rows are independent and padding rows'
// results are never stored, so the layer call skips those writes (a fifth of the gather's bytes at
// the prefill workload); the step call moe_permute writes them as zeros.
cudaError_t launch_act_quant(const uint16_t* x, int T, int d, uint8_t* xq, uint8_t* xs, bool fp8, cudaStream_t st,
                             bool pdl);
// Quantise each token row once and write it straight to the padded rows of its k picks (the
// permutation of ids / inv_pos / offsets / plan already built); padding rows are left as they are.
cudaError_t launch_act_quant_scatter(const uint16_t* x, int T, int d, int k, const int32_t* ids,
                                     const int32_t* inv_pos, const int32_t* offsets, PlanView plan, uint8_t* xa,
                                     uint8_t* xa_s, bool fp8, cudaStream_t st, bool pdl);
cudaError_t launch_act_gather(const uint8_t* xq, const uint8_t* xs, int d, int E, const int32_t* offsets,
                              const int32_t* perm_token, PlanView plan, int64_t pad_rows, uint8_t* xa, uint8_t* xa_s,
                              bool fp8, cudaStream_t st, bool pdl, bool zero_pad = true);

cudaError_t launch_gemv_up(const uint16_t* x, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                           int T, int d, int E, int k, int I, const moe_expert_weights* W, uint16_t* h,
                           cudaStream_t st, bool pdl);
// y != nullptr: fused weighted sum into y [T][d] using row_w; otherwise bf16 y_perm [P][d].
// pdl: the kernel for up to four tokens reads the plan (and offsets) before its dependency wait, so with
// pdl = true the plan must come from a kernel that completed before the preceding kernel's own wait.
cudaError_t launch_gemv_down(const uint16_t* h, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                             const float* row_w, int T, int d, int E, int k, int I, const moe_expert_weights* W,
                             uint16_t* y_perm, uint16_t* y, int* status, cudaStream_t st, bool pdl);
bool gemv_supported(int d, int I);
cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                           uint16_t* y, cudaStream_t st, bool pdl);
// The plan of one expert holding rows 0..T-1 in order (a dense product as a grouped one).
cudaError_t launch_dense_plan(int T, PlanView plan, int32_t* offsets, int32_t* perm_token, cudaStream_t st,
                              bool pdl);
// Weighted sum of the expert outputs, each first divided by its RMS over d (sqrt(mean + eps)).
cudaError_t launch_combine_norm(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                                float eps, uint16_t* y, cudaStream_t st, bool pdl);

// Decode on the tensor cores (decode_mma.cu), MXFP4 weights with their tensor-core copies.
bool mma_decode_supported(int T, int d, int E, int k, int I, const moe_expert_weights* W);
// x bf16 [T][d] -> 8 MXFP4 pieces per row: rows 8t + p of a [128][d] operand tile (code tiles xa,
// scale atoms xa_s); mx8: of the row's MXFP8 values.  Reads x before its dependency wait (the
// preceding kernel must have passed its own wait before letting this one start).
cudaError_t launch_x_pieces(const uint16_t* x, int T, int d, bool mx8, uint8_t* xa, uint8_t* xa_s, cudaStream_t st,
                            bool pdl);
// Both expert GEMMs in one persistent launch: gate/up tiles, then down tiles (each waits for its
// slot's h operand), expert outputs to y_perm; with y != nullptr (T <= 4, d <= 64 * 256) the weighted
// sum y[t] = sum_j w[t][j] y_perm[inv_pos[t k + j]] (fp32, slot order, then bf16) is fused too.
// mx8: h is rounded to MXFP8 (else bf16) before its pieces are formed.
// route != nullptr (mma_decode_route_supported): the launch also routes -- it computes the logits,
// the token pieces (into xa / xa_s), the top-k and the plan itself and writes ids, w, counts,
// offsets, perm_token, inv_pos, row_w and the plan like the one-launch router; otherwise all of them
// come from the preceding kernels.
struct DecRoute {
    const uint16_t* x;
    const float* W_r;
    const float* b;
    float* logits;
    int32_t* ids;
    float* w;
    int32_t* counts;
    float* row_w;
};
bool mma_decode_route_supported(int T, int d, int E, int k);
cudaError_t launch_mma_decode(const uint8_t* xa, const uint8_t* xa_s, uint8_t* ha, uint8_t* ha_s, float* part,
                              PlanView plan, const int32_t* offsets, const int32_t* perm_token, int T, int d, int E,
                              int k, int I, const moe_expert_weights* W, bool mx8, uint16_t* y_perm,
                              const int32_t* inv_pos, const float* w, uint16_t* y, Ctrl* ctrl, cudaStream_t st,
                              bool pdl, const DecRoute* route = nullptr);
bool mma_decode_fused_sum(int T, int d);

// Grouped prefill GEMMs (umma.cu).  fp8: MXFP8 token operand and h (kind::mxf8f6f4, the weights
// read from their canonical codes through tensor maps); else MXFP4 (kind::mxf4, tensor-core tiles).
// NVFP4 weights (W->wfmt) with MXFP4 operands: kind::mxf4nvf4; xa_s / h_s are then the operands'
// UE4M3 scales and rf their row factors (launch_nv_operand_scales).
cudaError_t launch_umma_up(const uint8_t* xa, const uint8_t* xa_s, PlanView plan, const int32_t* offsets,
                           int T, int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W,
                           bool fp8, const float* rf, uint8_t* h, uint8_t* h_s, int* status, cudaStream_t st,
                           bool pdl);
cudaError_t launch_umma_down(const uint8_t* h, const uint8_t* h_s, PlanView plan, const int32_t* offsets,
                             int T, int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W,
                             bool fp8, const float* rf, uint16_t* y_perm, int* status, cudaStream_t st, bool pdl);
// Whether the kind::mxf4nvf4 GEMMs fit shared memory for E experts.
bool umma_nv_supported(int E);
// E8M0 scales of an MXFP4 operand (tensor-core layout of width K, rows_used[0] padded rows) as
// UE4M3 scales per 16 values (layout of width 2K) and one power-of-two factor per row (nvfp4.cu).
cudaError_t launch_nv_operand_scales(const uint8_t* s32, const int32_t* rows_used, int64_t pad_rows, int K,
                                     uint8_t* s16, float* rf, cudaStream_t st, bool pdl);
}  // namespace moe

