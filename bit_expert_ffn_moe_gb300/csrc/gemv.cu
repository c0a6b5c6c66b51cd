// gemv.cu -- decode-shape expert kernels (MOE_ACT_BF16): bf16 activations, MXFP4 or NVFP4
// weights (template flag NV: two E4M3 scales per 32-element block and a global scale per matrix,
// applied to each 16-element half-sum and to the finished dot product).
//
// At decode sizes every chosen expert sees one or a few tokens, so the expert matrices are read
// once and used for very little arithmetic: the time is the weight read (Muse Spark Open
// explainer, section 13: at one token per expert about 98% of the time waits on the 4-bit weight
// read; DGX Spark news item, section 1: batch-1 generation is bound by weight reads).  These
// kernels stream each weight row once with coalesced 128-bit loads (16 bytes = one 32-element
// MXFP4 block) and keep the work per weight byte small:
//   - E2M1 codes become exact f16 pairs with the hardware conversion (cvt.rn.f16x2.e2m1x2);
//   - activation rows are staged once per CTA as f16, each row prescaled by a power of two so
//     that its largest magnitude lies in [2^14, 2^15) (a bf16 value then converts exactly unless
//     it is more than 2^28 times smaller than the row maximum);
//   - products w*x are exact and accumulate in fp32 (fma.rn.f32.f16); the block scale and the
//     row's prescale are applied once per 32-element partial.
// One warp owns whole weight rows: lane l takes K-blocks l, l+32, ..., so each row's dot product
// is finished with warp shuffles and no CTA-wide barrier sits in the streaming loop.  Activation
// blocks are read from shared memory in an order where the lanes of a warp touch consecutive
// 16-byte units, and each read serves every weight row of the batch.
#include "common.cuh"

namespace moe {

constexpr int kThr = 256;  // threads per CTA (8 warps)
constexpr int kWarps = kThr / 32;
constexpr int kQ = 4;               // activation rows staged per pass (gate/up)
constexpr int kDownMaxRows = 64;    // staged permuted rows per down CTA
// rows per warp in the down kernel: fewer for long rows so the double-buffered weights fit
__host__ __device__ constexpr int down_rows_per_warp(int bpl) { return bpl <= 2 ? 4 : bpl == 4 ? 2 : 1; }
constexpr int kUpOutsPerWarp = 4;

// ------------------------------------------------------------------ helpers

// acc += w.lo * x.lo + w.hi * x.hi with f16 operands and an fp32 accumulator (exact products).
__device__ __forceinline__ float dot2_f16(uint32_t w2, uint32_t x2, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

// Unscaled dot product of one 32-element MXFP4 block (16 bytes of codes) with 32 f16 activations
// held as 16 f16x2 words (elements 2m, 2m+1 in word m, low half first).
__device__ __forceinline__ float block_dot(const uint4& codes, const uint32_t (&x)[16]) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t h[4];
        e2m1x8_to_h2(words[m], h);  // elements 8m .. 8m+7 as 4 f16x2
        a0 = dot2_f16(h[0], x[4 * m + 0], a0);
        a1 = dot2_f16(h[1], x[4 * m + 1], a1);
        a0 = dot2_f16(h[2], x[4 * m + 2], a0);
        a1 = dot2_f16(h[3], x[4 * m + 3], a1);
    }
    return a0 + a1;
}

// NVFP4: acc + the dot product of one 32-element block with 32 f16 activations, each 16-element
// half scaled by its E4M3 scale (sc: elements 0..15 in bits 0..7, 16..31 in bits 8..15).
__device__ __forceinline__ float block_dot_nv(const uint4& codes, const uint32_t (&x)[16], uint32_t sc, float acc) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
    float a[4] = {0.f, 0.f, 0.f, 0.f};  // a[0], a[1]: elements 0..15; a[2], a[3]: 16..31
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t h[4];
        e2m1x8_to_h2(words[m], h);
        const int p = (m >> 1) * 2;
        a[p] = dot2_f16(h[0], x[4 * m + 0], a[p]);
        a[p + 1] = dot2_f16(h[1], x[4 * m + 1], a[p + 1]);
        a[p] = dot2_f16(h[2], x[4 * m + 2], a[p]);
        a[p + 1] = dot2_f16(h[3], x[4 * m + 3], a[p + 1]);
    }
    const float2 s = e4m3x2_to_f2(sc);
    return fmaf(a[2] + a[3], s.y, fmaf(a[0] + a[1], s.x, acc));
}

// Scale word of one 32-element block (idx = row * K/32 + block): MXFP4 one E8M0 byte, NVFP4 the
// block's two E4M3 bytes.  The NVFP4 pair is read like the weight codes (a streaming load issued
// where it is written, so that a batch's scales stay in flight with its codes).
template <bool NV>
__device__ __forceinline__ uint32_t load_block_scale(const uint8_t* s, size_t idx) {
    if constexpr (NV) {
        uint32_t v;
        asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];"
                     : "=r"(v)
                     : "l"(reinterpret_cast<const unsigned short*>(s) + idx));
        return v;
    } else {
        return __ldg(s + idx);
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ int prescale_exp(uint32_t mx) {
    const int p = (mx == 0) ? 0 : 141 - (int)(mx >> 7);  // row maximum * 2^p in [2^14, 2^15)
    return max(-126, min(126, p));
}

// All threads of the CTA stage nq activation rows (bf16, K elements) as prescaled f16 in
// block-interleaved order: 16-byte unit c (elements 8c..8c+7) of block b of staged row q sits at
// uint4 index (q * 4 + c) * nb + b.  inv[q] = 2^-p undoes the row's prescale.  smax: nq words of
// shared scratch.  Ends with __syncthreads.
__device__ void stage_rows_f16(const uint16_t* __restrict__ src, const int* rows, int nq, int K, uint4* dst,
                               float* inv, unsigned* smax) {
    const int tid = threadIdx.x, nb = K / 32, units = K / 8, total = nq * units;
    if (tid < nq) smax[tid] = 0;
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < total; i += blockDim.x) {
        const int q = i / units, u = i - q * units;
        const uint4 v = reinterpret_cast<const uint4*>(src + (size_t)rows[q] * K)[u];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t mx = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        atomicMax(&smax[q], mx);
    }
    __syncthreads();
#pragma unroll 4
    for (int i = tid; i < total; i += blockDim.x) {
        const int q = i / units, u = i - q * units;
        const uint4 v = reinterpret_cast<const uint4*>(src + (size_t)rows[q] * K)[u];
        const float up = __uint_as_float((uint32_t)(127 + prescale_exp(smax[q])) << 23);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half lo = __float2half_rn(bf16_bits_to_f32(w[j] & 0xFFFFu) * up);
            const __half hi = __float2half_rn(bf16_bits_to_f32(w[j] >> 16) * up);
            o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        dst[((size_t)q * 4 + (u & 3)) * nb + (u >> 2)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid < nq) inv[tid] = __uint_as_float((uint32_t)(127 - prescale_exp(smax[tid])) << 23);
    __syncthreads();
}

__device__ __forceinline__ void load_x_block(const uint4* xs, int q, int nb, int b, uint32_t (&x)[16]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint4 v = xs[((size_t)q * 4 + c) * nb + b];
        x[4 * c + 0] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
    }
}

struct GemvArgs {
    const uint8_t* q0;  // up: gate codes; down: down codes
    const uint8_t* s0;
    const uint8_t* q1;  // up: up codes
    const uint8_t* s1;
    const float* gs0;   // NVFP4: global scale per expert of q0 / q1
    const float* gs1;
    const uint16_t* act;  // up: x [T][d]; down: h [P][I]
    const int32_t* perm_token;
    const int32_t* offsets;
    PlanView plan;
    const float* row_w;  // down, fused: gate weight of each permuted row
    int T, K, M_exp, P, E;
    int tch;       // down: tokens per chunk
    int maxrows;   // down: staged rows per CTA (tch * k)
    int outs;      // up: output features per CTA; down: rows per CTA
    uint16_t* out; // up: h [P][I]; down: y_perm [P][d] or y [T][d]
    int* status;   // device status word (first error wins)
};

// ------------------------------------------------------------------ gate/up + SwiGLU
// Grid (I / outs, slots): slot u is the u-th active expert.  Warp w computes outputs
// i = blockIdx.x * outs + w * kUpOutsPerWarp + o, reading gate row i and up row i (lane l owns
// K-blocks l + 32 j, j < BPL) and the staged activation blocks of up to kQ tokens.
template <int BPL, bool NV>
__global__ void __launch_bounds__(kThr, 2)
gemv_up_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int nb = a.K / 32;
    uint4* xs = reinterpret_cast<uint4*>(smem);                                 // [kQ][K/8]
    float* inv = reinterpret_cast<float*>(smem + (size_t)kQ * a.K * 2);        // [kQ]
    unsigned* smax = reinterpret_cast<unsigned*>(inv + kQ);                    // [kQ]
    int* rows = reinterpret_cast<int*>(smax + kQ);                             // [kQ]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    pdl_wait();
    // the next kernel (the down GEMV) may start now: before its own wait it only reads the routing
    // plan, which the kernel before this one wrote, and the weights
    pdl_launch_dependents();
    const int slot = blockIdx.y;
    if (slot >= a.plan.scalars[0]) return;
    const int e = a.plan.active[slot];
    const size_t row_bytes = (size_t)a.K / 2;
    const int i0 = blockIdx.x * a.outs + warp * kUpOutsPerWarp;
    const float gsg = NV ? __ldg(a.gs0 + e) : 1.f, gsu = NV ? __ldg(a.gs1 + e) : 1.f;  // NVFP4 global scales

    auto load_out = [&](int i, uint4 (&wg)[BPL], uint4 (&wu)[BPL], uint32_t (&sg)[BPL], uint32_t (&su)[BPL]) {
        const size_t grow = (size_t)e * a.M_exp + i;
#pragma unroll
        for (int j = 0; j < BPL; ++j) {
            const int b = lane + 32 * j;
            if (b < nb) {
                wg[j] = ldg_stream(a.q0 + grow * row_bytes + 16 * (size_t)b);
                wu[j] = ldg_stream(a.q1 + grow * row_bytes + 16 * (size_t)b);
                sg[j] = load_block_scale<NV>(a.s0, grow * nb + b);
                su[j] = load_block_scale<NV>(a.s1, grow * nb + b);
            }
        }
    };
    uint4 wg[BPL], wu[BPL];
    uint32_t sg[BPL], su[BPL];
    load_out(i0, wg, wu, sg, su);  // weights depend only on the expert: start streaming now

    const int r0 = a.offsets[e], n = a.offsets[e + 1] - r0;
    for (int tc0 = 0; tc0 < n; tc0 += kQ) {
        const int nq = min(kQ, n - tc0);
        if (tc0 > 0) {
            __syncthreads();
            load_out(i0, wg, wu, sg, su);
        }
        if (tid < nq) rows[tid] = a.perm_token[r0 + tc0 + tid];
        __syncthreads();
        stage_rows_f16(a.act, rows, nq, a.K, xs, inv, smax);
        for (int o = 0; o < kUpOutsPerWarp; ++o) {
            float g[kQ], u[kQ];
#pragma unroll
            for (int q = 0; q < kQ; ++q) g[q] = u[q] = 0.f;
#pragma unroll
            for (int j = 0; j < BPL; ++j) {
                const int b = lane + 32 * j;
                if (b < nb) {
                    const float fg = e8m0_to_f32(sg[j]), fu = e8m0_to_f32(su[j]);
#pragma unroll
                    for (int q = 0; q < kQ; ++q) {
                        if (q < nq) {
                            uint32_t x[16];
                            load_x_block(xs, q, nb, b, x);
                            if constexpr (NV) {
                                g[q] = block_dot_nv(wg[j], x, sg[j], g[q]);
                                u[q] = block_dot_nv(wu[j], x, su[j], u[q]);
                            } else {
                                g[q] = fmaf(block_dot(wg[j], x), fg, g[q]);
                                u[q] = fmaf(block_dot(wu[j], x), fu, u[q]);
                            }
                        }
                    }
                }
            }
            // next output's rows are independent of this one's arithmetic
            if (o + 1 < kUpOutsPerWarp) load_out(i0 + o + 1, wg, wu, sg, su);
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                if (q < nq) {
                    float gs = warp_sum(g[q]) * inv[q], us = warp_sum(u[q]) * inv[q];
                    if constexpr (NV) {
                        gs *= gsg;
                        us *= gsu;
                    }
                    if (lane == q) {
                        const float hv = gs / (1.f + expf(-gs)) * us;  // SiLU(g) * u
                        a.out[(size_t)(r0 + tc0 + q) * a.M_exp + i0 + o] = f32_to_bf16_bits(hv);
                    }
                }
            }
        }
    }
    pdl_launch_dependents();
}


// ------------------------------------------------------------------ gate/up + SwiGLU, T <= 4
// For up to four tokens a CTA-wide split of K is faster than whole rows per warp: the weight
// rows of a batch are prefetched into registers one batch ahead and every thread owns one
// K-block, so the activations need no shared-memory traffic per row.  (The down GEMV takes the
// same split, with its weights fed through a copy-engine ring.)
constexpr int kR = 8;  // weight rows per batch per row group

// Sum V values over the 32 lanes of a warp; afterwards lane l holds the warp sum of value
// l >> (5 - log2 V), for V in {8, 16, 32}.
template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&a)[V], int lane) {
#pragma unroll
    for (int half = V / 2, mask = 16; half >= 1; half /= 2, mask /= 2) {
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? a[i] : a[i + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, mask);
            a[i] = (upper ? a[i + half] : a[i]) + recv;
        }
    }
    float v = a[0];
#pragma unroll
    for (int mask = (32 / V) / 2; mask >= 1; mask /= 2) v += __shfl_xor_sync(0xffffffffu, v, mask);
    return v;
}

// Row-group geometry for a contraction of K elements: nb = K/32 blocks, bpt blocks per thread,
// G threads per group (a power of two >= 32 covering nb / bpt), RG = kThr / G groups per CTA.
struct CtaGeo {
    int nb, bpt, G, RG;
};

__host__ __device__ inline CtaGeo make_cta_geo(int K) {
    CtaGeo g;
    g.nb = K / 32;
    g.bpt = (g.nb + kThr - 1) / kThr;
    const int need = (g.nb + g.bpt - 1) / g.bpt;
    int G = 32;
    while (G < need) G *= 2;
    g.G = G;
    g.RG = kThr / G;
    return g;
}

// Stage activation rows (bf16, K elements each) as prescaled f16 in block-interleaved order:
// 16-byte unit c (elements 8c..8c+7) of block b of staged row q sits at uint4 index
// (q * 4 + c) * nb + b, so threads owning consecutive blocks read consecutive units.
// inv[q] receives 2^-p, the factor that undoes the row's prescale 2^p.  One warp per row.
__device__ void stage_rows_warp(const uint16_t* __restrict__ src, const int* rows, int nq, int K, uint4* dst,
                               float* inv) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int nb = K / 32, units = K / 8;
    for (int q = warp; q < nq; q += nwarps) {
        const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)rows[q] * K);
        uint32_t mx = 0;
        for (int u = lane; u < units; u += 32) {
            const uint4 v = s[u];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = max(mx, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
        }
        mx = __reduce_max_sync(0xffffffffu, mx);
        // biased exponent E of max |x|; p = 141 - E puts the maximum in [2^14, 2^15)
        int p = (mx == 0) ? 0 : 141 - (int)(mx >> 7);
        p = max(-126, min(126, p));
        const float up = __uint_as_float((uint32_t)(127 + p) << 23);
        const float down = __uint_as_float((uint32_t)(127 - p) << 23);
        for (int u = lane; u < units; u += 32) {
            const uint4 v = s[u];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half lo = __float2half_rn(bf16_bits_to_f32(w[i] & 0xFFFFu) * up);
                const __half hi = __float2half_rn(bf16_bits_to_f32(w[i] >> 16) * up);
                o[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
            }
            const int b = u >> 2, c = u & 3;
            dst[((size_t)q * 4 + c) * nb + b] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) inv[q] = down;
    }
}

// Weight rows of one batch into registers (rows[j] = global row index, or -1 to skip).
template <int BPT, bool NV>
__device__ __forceinline__ void load_rows_cta(const uint8_t* const (&q)[kR], const uint8_t* const (&s)[kR],
                                          const size_t (&grow)[kR], int gl, const CtaGeo& geo, size_t row_bytes,
                                          uint4 (&wv)[kR][BPT], uint32_t (&sv)[kR][BPT]) {
#pragma unroll
    for (int j = 0; j < kR; ++j)
#pragma unroll
        for (int c = 0; c < BPT; ++c) {
            const int b = gl + c * geo.G;
            if (b < geo.nb) {
                wv[j][c] = ldg_stream(q[j] + grow[j] * row_bytes + 16 * (size_t)b);
                sv[j][c] = load_block_scale<NV>(s[j], grow[j] * geo.nb + b);
            }
        }
}

// kR x Q partial dot products of the thread's blocks: acc[qq * kR + j] for staged row q0 + qq
// (qq < nq) against weight row j.
template <int BPT, int Q, bool NV>
__device__ __forceinline__ void batch_dots(const uint4* xs, int q0, int nq, int gl, const CtaGeo& geo,
                                           const uint4 (&wv)[kR][BPT], const uint32_t (&sv)[kR][BPT],
                                           float (&acc)[kR * Q]) {
#pragma unroll
    for (int v = 0; v < kR * Q; ++v) acc[v] = 0.f;
#pragma unroll
    for (int qq = 0; qq < Q; ++qq) {
        if (qq < nq) {
#pragma unroll
            for (int c = 0; c < BPT; ++c) {
                const int b = gl + c * geo.G;
                if (b < geo.nb) {
                    uint32_t x[16];
                    load_x_block(xs, q0 + qq, geo.nb, b, x);
#pragma unroll
                    for (int j = 0; j < kR; ++j) {
                        if constexpr (NV)
                            acc[qq * kR + j] = block_dot_nv(wv[j][c], x, sv[j][c], acc[qq * kR + j]);
                        else
                            acc[qq * kR + j] = fmaf(block_dot(wv[j][c], x), e8m0_to_f32(sv[j][c]), acc[qq * kR + j]);
                    }
                }
            }
        }
    }
}

// Grid (M_exp / outs, slots): slot u is the u-th active expert.  A batch gives each row group
// kR/2 output features i (gate row i and up row i), for up to Q of the expert's tokens; an
// expert with more rows takes them Q at a time (its weights are read again per pass).
// One block per thread: bounded to two CTAs per SM (128 registers; the two-row instantiations
// would otherwise take more and fit one CTA per SM).
template <int BPT, int Q, bool NV>
__global__ void __launch_bounds__(kThr, BPT == 1 ? 2 : 0)
gemv_up_cta_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int kOut = kR / 2;
    constexpr int V = kR * Q;
    const CtaGeo geo = make_cta_geo(a.K);
    uint4* xs = reinterpret_cast<uint4*>(smem);                              // [Q][K/8]
    float* inv = reinterpret_cast<float*>(smem + (size_t)Q * a.K * 2);      // [Q]
    float* red = inv + Q;                                                   // [2][8 warps][32]
    int* rows = reinterpret_cast<int*>(red + 2 * 8 * 32);                   // [Q]
    unsigned* smax = reinterpret_cast<unsigned*>(rows + Q);                 // [Q]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid / geo.G, gl = tid % geo.G;
    const int wpg = geo.G / 32;  // warps per group

    pdl_wait();
    // the next kernel (the down GEMV) may start now: before its own wait it only reads the routing
    // plan, which the kernel before this one wrote, and the weights
    pdl_launch_dependents();
    const int slot = blockIdx.y;
    if (slot >= a.plan.scalars[0]) return;
    const int e = a.plan.active[slot];
    const size_t row_bytes = (size_t)a.K / 2;
    const float gsg = NV ? __ldg(a.gs0 + e) : 1.f, gsu = NV ? __ldg(a.gs1 + e) : 1.f;  // NVFP4 global scales
    const int outs_per_group = a.outs / geo.RG;
    const int nbatch = outs_per_group / kOut;
    const int i_base = blockIdx.x * a.outs + grp * outs_per_group;
    const uint8_t* const qsel[kR] = {a.q0, a.q0, a.q0, a.q0, a.q1, a.q1, a.q1, a.q1};
    const uint8_t* const ssel[kR] = {a.s0, a.s0, a.s0, a.s0, a.s1, a.s1, a.s1, a.s1};
    auto grows = [&](int bi, size_t (&g)[kR]) {
#pragma unroll
        for (int j = 0; j < kR; ++j) g[j] = (size_t)e * a.M_exp + i_base + bi * kOut + (j % kOut);
    };

    uint4 wcur[kR][BPT], wnxt[kR][BPT];
    uint32_t scur[kR][BPT], snxt[kR][BPT];
    {
        size_t g[kR];
        grows(0, g);
        load_rows_cta<BPT, NV>(qsel, ssel, g, gl, geo, row_bytes, wcur, scur);  // weights depend only on e
    }
    const int r0 = a.offsets[e], n = a.offsets[e + 1] - r0;

    for (int tc0 = 0; tc0 < n; tc0 += Q) {
        const int nq = min(Q, n - tc0);
        __syncthreads();
        if (tid < nq) rows[tid] = a.perm_token[r0 + tc0 + tid];
        __syncthreads();
        stage_rows_f16(a.act, rows, nq, a.K, xs, inv, smax);  // all warps; ends with a barrier
        for (int bi = 0; bi < nbatch; ++bi) {
            const bool more = bi + 1 < nbatch || tc0 + Q < n;
            if (more) {
                size_t g[kR];
                grows(bi + 1 < nbatch ? bi + 1 : 0, g);
                load_rows_cta<BPT, NV>(qsel, ssel, g, gl, geo, row_bytes, wnxt, snxt);
            }
            float acc[V];
            batch_dots<BPT, Q, NV>(xs, 0, nq, gl, geo, wcur, scur, acc);
            // partial sums go to alternating halves of red, so one barrier per batch suffices: the
            // leader warp finishes batch bi's features while the others compute batch bi + 1
            float* rb = red + (bi & 1) * (8 * 32);
            rb[warp * 32 + lane] = warp_transpose_reduce<V>(acc, lane);
            __syncthreads();
            if (gl < 32) {
                // lane l holds value v = l >> (5 - log2 V); v = qq * kR + j
                const int v = lane >> (5 - (V == 8 ? 3 : V == 16 ? 4 : 5));
                const int qq = v / kR, j = v % kR;
                const bool leader = (lane & ((32 / V) - 1)) == 0;
                if (leader && qq < nq && j < kOut) {
                    float g = 0.f, u = 0.f;
                    for (int w = 0; w < wpg; ++w) {
                        const int wi = (grp * wpg + w) * 32;
                        g += rb[wi + lane];
                        u += rb[wi + lane + kOut * (32 / V)];
                    }
                    g *= inv[qq];
                    u *= inv[qq];
                    if constexpr (NV) {
                        g *= gsg;
                        u *= gsu;
                    }
                    const float hv = g / (1.f + expf(-g)) * u;  // SiLU(g) * u
                    const int i = i_base + bi * kOut + j;
                    a.out[(size_t)(r0 + tc0 + qq) * a.M_exp + i] = f32_to_bf16_bits(hv);
                }
            }
            if (more) {
#pragma unroll
                for (int j = 0; j < kR; ++j)
#pragma unroll
                    for (int c = 0; c < BPT; ++c) {
                        wcur[j][c] = wnxt[j][c];
                        scur[j][c] = snxt[j][c];
                    }
            }
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ down (+ weighted sum), T <= 4
// The same CTA-wide split of K as the gate/up kernel above, with the weights fed through a ring
// of shared-memory stages by the copy engine.  A CTA owns feats = RG * kR output features and
// walks the active experts in ascending order (each token's slot order); batch u is the feats
// rows of expert active[u], whose codes (feats * K/2 bytes) and scales (feats * K/32 bytes) are
// each one contiguous range: two bulk copies fill a stage, and kDownStages batches are in
// flight.  Row group g takes rows kR*g .. kR*g + kR - 1 of the batch; thread gl of the group owns
// K-block gl of each.
// The batch's h rows (bf16, at most Q) are converted once per CTA, a batch ahead, into a double
// buffer of f16 blocks: four threads share a 32-element block (8 elements each), scale it by a
// power of two that puts the block maximum in [2^14, 2^15), and the block's partial sums are
// scaled back by the inverse, an exact rescaling.
// FUSED: ys[t][f] accumulates w * bf16(expert output) batch after batch (the same lane updates a
// given (t, f) in expert order); otherwise the bf16 outputs go to y_perm.
// MXFP4, Q = 1: three stages; otherwise two (for Q = 2, 4 the h rows take the third stage's
// shared memory, and the NVFP4 stages are larger by their second scale byte per block, so that
// two CTAs still fit an SM).  8-element h pieces per thread and batch: 2 for Q <= 2
// (Q K/8 <= 2 kThr), Q for Q = 4.
template <int Q, bool NV> __host__ __device__ constexpr int down_stages() { return Q == 1 && !NV ? 3 : 2; }
template <int Q> __host__ __device__ constexpr int down_hunits() { return Q <= 2 ? 2 : Q; }

// Bytes of one stage: codes, then scales (one byte per 32-element block, two for NVFP4).
__host__ __device__ inline uint32_t down_stage_bytes(int K, bool nv) {
    const CtaGeo g = make_cta_geo(K);
    return (uint32_t)(g.RG * kR) * (uint32_t)(K / 2 + (K / 32) * (nv ? 2 : 1));
}

template <int Q, bool NV>
__host__ __device__ inline size_t down_ring_smem(int K, int P) {
    const CtaGeo g = make_cta_geo(K);
    return (size_t)down_stages<Q, NV>() * down_stage_bytes(K, NV) + (size_t)2 * Q * K * 2 /* h blocks */ +
           sizeof(float) * ((size_t)2 * Q * g.nb /* inverse scales */ + 2 * 8 * 32 + (size_t)Q * g.RG * kR) +
           sizeof(uint64_t) * down_stages<Q, NV>() + sizeof(int) * 3 * (size_t)P;
}

template <int Q, bool FUSED, bool NV>
__global__ void __launch_bounds__(kThr, 2)
gemv_down_ring_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int V = kR * Q;
    constexpr int kDownStages = down_stages<Q, NV>();
    constexpr int kDownHUnits = down_hunits<Q>();
    constexpr uint32_t kScaleBytes = NV ? 2 : 1;  // per 32-element block
    const CtaGeo geo = make_cta_geo(a.K);
    const int feats = geo.RG * kR, nb = geo.nb;
    const uint32_t code_bytes = (uint32_t)feats * (a.K / 2),
                   stage_bytes = code_bytes + (uint32_t)feats * (a.K / 32) * kScaleBytes;
    uint4* hb = reinterpret_cast<uint4*>(smem + (size_t)kDownStages * stage_bytes);  // [2][Q][4][nb] f16 blocks
    float* hinv = reinterpret_cast<float*>(hb + (size_t)2 * Q * 4 * nb);               // [2][Q][nb]
    float* red = hinv + 2 * Q * nb;                                                     // [2][8 warps][32]
    float* ys = red + 2 * 8 * 32;                                                       // [Q][feats]
    uint64_t* full = reinterpret_cast<uint64_t*>(ys + (size_t)Q * feats);              // [kDownStages]
    int* sl_r0 = reinterpret_cast<int*>(full + kDownStages);                           // [P] first row of slot u
    int* sl_cnt = sl_r0 + a.P;                                                          // [P] its rows (<= Q)
    int* sl_e = sl_cnt + a.P;                                                           // [P] its expert
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int grp = tid / geo.G, gl = tid % geo.G;
    const int wpg = geo.G / 32;
    const int f0 = blockIdx.x * feats;
    const int K2 = a.K / 2;
    const int hunits = Q * nb * 4;  // 8-element pieces of the batch's h rows

    if (tid == 0) {
        for (int s = 0; s < kDownStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    for (int i = tid; i < Q * feats; i += blockDim.x) ys[i] = 0.f;
    // The routing plan comes from the kernel two launches back, which completed before the gate/up
    // kernel passed its own wait and let this one start; it is read through L2 before this
    // kernel's wait, and the first weight stages are issued, so only h waits for gate/up.
    const int n_act = __ldcg(a.plan.scalars);
    if (tid < n_act) {
        const int e = __ldcg(a.plan.active + tid);
        const int r0 = __ldcg(a.offsets + e);
        sl_e[tid] = e;
        sl_r0[tid] = r0;
        sl_cnt[tid] = min(Q, __ldcg(a.offsets + e + 1) - r0);
    }
    __syncthreads();

    auto stage = [&](int s) { return smem + (size_t)s * stage_bytes; };
    auto issue = [&](int u) {  // thread 0: batch u into stage u % kDownStages
        const int s = u % kDownStages;
        const size_t R = (size_t)sl_e[u] * a.M_exp + f0;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        bulk_load(stage(s), a.q0 + R * K2, code_bytes, &full[s]);
        bulk_load(stage(s) + code_bytes, a.s0 + R * (a.K / 32) * kScaleBytes, stage_bytes - code_bytes, &full[s]);
    };
    int issued = 0;
    if (tid == 0)
        for (; issued < min(n_act, kDownStages); ++issued) issue(issued);
    pdl_wait();

    // piece i = (qq, b, c): elements 8c .. 8c+7 of block b of h row qq of the batch
    auto load_h = [&](int u, uint4 (&hv)[kDownHUnits]) {
#pragma unroll
        for (int m = 0; m < kDownHUnits; ++m) {
            const int i = tid + m * kThr;
            const int qq = i / (4 * nb), rem = i % (4 * nb);
            hv[m] = (u < n_act && i < hunits && qq < sl_cnt[u])
                        ? __ldcg(reinterpret_cast<const uint4*>(a.act + (size_t)(sl_r0[u] + qq) * a.K) + rem)
                        : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    auto convert_h = [&](int u, const uint4 (&hv)[kDownHUnits], int buf) {
#pragma unroll
        for (int m = 0; m < kDownHUnits; ++m) {
            const int i = tid + m * kThr;  // the four pieces of a block are adjacent lanes
            const int qq = i / (4 * nb), rem = i % (4 * nb), b = rem >> 2, c = rem & 3;
            const bool valid = u < n_act && i < hunits && qq < sl_cnt[u];
            const uint32_t w[4] = {hv[m].x, hv[m].y, hv[m].z, hv[m].w};
            uint32_t mx = 0;
            if (valid)
#pragma unroll
                for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
            if (m * kThr < hunits) {  // warp-uniform: whole warps hold valid pieces or none
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            }
            if (valid) {
                const int p = prescale_exp(mx);
                const float up = __uint_as_float((uint32_t)(127 + p) << 23);
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __half2 h2 = __floats2half2_rn(bf16_bits_to_f32(w[j] & 0xFFFFu) * up,
                                                         bf16_bits_to_f32(w[j] >> 16) * up);
                    o[j] = *reinterpret_cast<const uint32_t*>(&h2);
                }
                hb[(((size_t)buf * Q + qq) * 4 + c) * nb + b] = make_uint4(o[0], o[1], o[2], o[3]);
                if (c == 0) hinv[((size_t)buf * Q + qq) * nb + b] = __uint_as_float((uint32_t)(127 - p) << 23);
            }
        }
    };
    uint4 hv[kDownHUnits];
    load_h(0, hv);
    convert_h(0, hv, 0);
    __syncthreads();

    bool ok = true;
    for (int u = 0; u < n_act; ++u) {
        const int s = u % kDownStages, buf = u & 1;
        const int r0 = sl_r0[u], cnt = sl_cnt[u];
        load_h(u + 1, hv);  // converted after this batch's arithmetic
        const bool arrived = mbar_wait(&full[s], (uint32_t)(u / kDownStages) & 1u, &s_abort, a.status);
        float acc[V];
#pragma unroll
        for (int v = 0; v < V; ++v) acc[v] = 0.f;
        if (gl < nb) {
            const unsigned char* st = stage(s);
#pragma unroll
            for (int qq = 0; qq < Q; ++qq) {
                if (qq < cnt) {
                    uint32_t x[16];
                    load_x_block(hb + (size_t)buf * Q * 4 * nb, qq, nb, gl, x);
                    const float inv = hinv[((size_t)buf * Q + qq) * nb + gl];
#pragma unroll
                    for (int j = 0; j < kR; ++j) {
                        const int row = grp * kR + j;
                        const uint4 w = *reinterpret_cast<const uint4*>(st + (size_t)row * K2 + 16 * gl);
                        if constexpr (NV) {
                            const uint32_t sc = reinterpret_cast<const uint16_t*>(st + code_bytes)[(size_t)row * nb + gl];
                            acc[qq * kR + j] = block_dot_nv(w, x, sc, 0.f) * inv;
                        } else {
                            const uint32_t sc = st[code_bytes + (size_t)row * nb + gl];
                            acc[qq * kR + j] = block_dot(w, x) * e8m0_to_f32(sc) * inv;
                        }
                    }
                }
            }
        }
        convert_h(u + 1, hv, buf ^ 1);
        float* rb = red + (u & 1) * (8 * 32);
        rb[warp * 32 + lane] = warp_transpose_reduce<V>(acc, lane);
        ok = __syncthreads_and(arrived);  // stage s read, next h blocks and rb written; one verdict
        if (!ok) break;
        if (tid == 0 && issued < n_act) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(issued++);
        }
        if (gl < 32) {
            const int v = lane >> (5 - (V == 8 ? 3 : V == 16 ? 4 : 5));
            const int qq = v / kR, j = v % kR;
            const bool leader = (lane & ((32 / V) - 1)) == 0;
            if (leader && qq < cnt) {
                float o = 0.f;
                for (int w = 0; w < wpg; ++w) o += rb[(grp * wpg + w) * 32 + lane];
                if constexpr (NV) o *= __ldg(a.gs0 + sl_e[u]);
                const uint16_t ob = f32_to_bf16_bits(o);
                if (FUSED) {
                    const int t = a.perm_token[r0 + qq];
                    float& yv = ys[t * feats + grp * kR + j];
                    yv = fmaf(a.row_w[r0 + qq], bf16_bits_to_f32(ob), yv);
                } else {
                    a.out[(size_t)(r0 + qq) * a.M_exp + f0 + grp * kR + j] = ob;
                }
            }
        }
    }
    if (!ok) {
        // a copy did not arrive in time: wait (bounded) for the last batch issued to each stage,
        // so that no copy still writes into this CTA's shared memory, then leave
        if (tid == 0) {
            volatile int never = 0;
            for (int u = max(0, issued - kDownStages); u < issued; ++u)
                mbar_wait(&full[u % kDownStages], (uint32_t)(u / kDownStages) & 1u, &never, nullptr, kWaitCycles / 4);
        }
        __syncthreads();
        return;
    }
    if (FUSED) {
        __syncthreads();
        for (int i = tid; i < a.T * feats; i += blockDim.x) {
            const int t = i / feats, f = i % feats;
            a.out[(size_t)t * a.M_exp + f0 + f] = f32_to_bf16_bits(ys[i]);
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ down (+ weighted sum)
// Grid (d / outs, token chunks).  The CTA stages every permuted row whose token lies in its chunk
// (rows are expert-major, so each active expert forms a consecutive segment).  Warp w owns rows
// n = blockIdx.x * outs + w * RPW + rr and walks the segments in ascending expert
// order, prefetching the next segment's weight rows.
// FUSED: y[t] accumulates w * bf16(expert output) in that order, which is the slot order j of the
// token (ids are ascending); otherwise the bf16 expert outputs go to y_perm.
template <int BPL, bool FUSED, bool NV>
__global__ void __launch_bounds__(kThr, 2)
gemv_down_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int RPW = down_rows_per_warp(BPL);
    const int nb = a.K / 32, mr = a.maxrows;
    uint4* hs = reinterpret_cast<uint4*>(smem);                                  // [mr][K/8]
    float* inv = reinterpret_cast<float*>(smem + (size_t)mr * a.K * 2);         // [mr]
    unsigned* smax = reinterpret_cast<unsigned*>(inv + mr);                     // [mr]
    float* ys = reinterpret_cast<float*>(smax + mr);                            // [tch][outs]
    int* s_row = reinterpret_cast<int*>(ys + (size_t)a.tch * a.outs);          // [mr]
    int* s_tok = s_row + mr;
    int* s_exp = s_tok + mr;
    float* s_w = reinterpret_cast<float*>(s_exp + mr);
    int* s_off = reinterpret_cast<int*>(s_w + mr);                              // [E+1]
    __shared__ int wtot[kWarps];
    __shared__ int s_cnt;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.y * a.tch, t1 = min(a.T, t0 + a.tch);
    const size_t row_bytes = (size_t)a.K / 2;
    const int nl0 = warp * RPW;                       // first local row of this warp
    const int n0 = blockIdx.x * a.outs + nl0;         // first global row of this warp

    pdl_wait();
    for (int i = tid; i <= a.E; i += blockDim.x) s_off[i] = a.offsets[i];
    for (int i = tid; i < a.tch * a.outs; i += blockDim.x) ys[i] = 0.f;
    if (tid == 0) s_cnt = 0;
    __syncthreads();
    // rows of the chunk in permuted order (stable compaction over all P rows), with their expert
    for (int base = 0; base < a.P; base += blockDim.x) {
        const int r = base + tid;
        const int t = r < a.P ? a.perm_token[r] : -1;
        const bool in = (t >= t0 && t < t1);
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        if (lane == 0) wtot[warp] = __popc(bal);
        __syncthreads();
        int before = s_cnt;
        for (int w = 0; w < warp; ++w) before += wtot[w];
        if (in) {
            const int pos = before + __popc(bal & ((1u << lane) - 1u));
            int lo = 0, hi = a.E;  // expert of row r: last e with offsets[e] <= r
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= r) lo = mid; else hi = mid;
            }
            s_row[pos] = r;
            s_tok[pos] = t - t0;
            s_exp[pos] = lo;
            s_w[pos] = FUSED ? a.row_w[r] : 0.f;
        }
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < kWarps; ++w) tot += wtot[w];
            s_cnt += tot;
        }
        __syncthreads();
    }
    const int nrows = s_cnt;

    auto load_rows = [&](int e, uint4 (&wv)[RPW][BPL], uint32_t (&sv)[RPW][BPL]) {
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const size_t grow = (size_t)e * a.M_exp + n0 + rr;
#pragma unroll
            for (int j = 0; j < BPL; ++j) {
                const int b = lane + 32 * j;
                if (b < nb) {
                    wv[rr][j] = ldg_stream(a.q0 + grow * row_bytes + 16 * (size_t)b);
                    sv[rr][j] = load_block_scale<NV>(a.s0, grow * nb + b);
                }
            }
        }
    };
    uint4 wcur[RPW][BPL], wnxt[RPW][BPL];
    uint32_t scur[RPW][BPL], snxt[RPW][BPL];
    int qs = 0;
    if (nrows > 0) load_rows(s_exp[0], wcur, scur);  // in flight while h is staged
    stage_rows_f16(a.act, s_row, nrows, a.K, hs, inv, smax);
    while (qs < nrows) {
        const int e = s_exp[qs];
        const float gsd = NV ? __ldg(a.gs0 + e) : 1.f;  // NVFP4: the expert's global scale
        int qe = qs + 1;
        while (qe < nrows && s_exp[qe] == e) ++qe;
        const bool more = qe < nrows;
        if (more) load_rows(s_exp[qe], wnxt, snxt);
        for (int q = qs; q < qe; ++q) {
            float acc[RPW];
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) acc[rr] = 0.f;
#pragma unroll
            for (int j = 0; j < BPL; ++j) {
                const int b = lane + 32 * j;
                if (b < nb) {
                    uint32_t x[16];
                    load_x_block(hs, q, nb, b, x);
#pragma unroll
                    for (int rr = 0; rr < RPW; ++rr) {
                        if constexpr (NV)
                            acc[rr] = block_dot_nv(wcur[rr][j], x, scur[rr][j], acc[rr]);
                        else
                            acc[rr] = fmaf(block_dot(wcur[rr][j], x), e8m0_to_f32(scur[rr][j]), acc[rr]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
                float s = warp_sum(acc[rr]) * inv[q];
                if constexpr (NV) s *= gsd;
                if (lane == rr) {
                    const uint16_t sb = f32_to_bf16_bits(s);
                    if (FUSED) {
                        float& yv = ys[s_tok[q] * a.outs + nl0 + rr];
                        yv = fmaf(s_w[q], bf16_bits_to_f32(sb), yv);
                    } else {
                        a.out[(size_t)s_row[q] * a.M_exp + n0 + rr] = sb;
                    }
                }
            }
        }
        if (more) {
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                for (int j = 0; j < BPL; ++j) {
                    wcur[rr][j] = wnxt[rr][j];
                    scur[rr][j] = snxt[rr][j];
                }
        }
        qs = qe;
    }
    if (FUSED) {
        __syncthreads();
        for (int i = tid; i < a.outs * (t1 - t0); i += blockDim.x) {
            const int tt = i / a.outs, nn = i % a.outs;
            a.out[(size_t)(t0 + tt) * a.M_exp + blockIdx.x * a.outs + nn] = f32_to_bf16_bits(ys[tt * a.outs + nn]);
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ weighted sum (unfused)
// One thread per (token, 8 consecutive features): y = sum_j w[t][j] * y_perm[inv_pos[t*k+j]]; a row
// index outside [0, T k) is not read (that slot contributes nothing).
__global__ void combine_kernel(const uint16_t* __restrict__ y_perm, const int32_t* __restrict__ inv_pos,
                               const float* __restrict__ w, int T, int k, int d, uint16_t* __restrict__ y) {
    pdl_wait();
    const int per_row = d / 8;
    const int64_t total = (int64_t)T * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / per_row), c = (int)(i % per_row);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        // up to 8 slots at a time: their rows' loads are issued before the sums (in slot order)
        for (int j0 = 0; j0 < k; j0 += 8) {
            uint4 u[8];
            float wj[8];
            bool ok[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int j = j0 + q;
                const int r = j < k ? __ldg(inv_pos + (size_t)t * k + j) : -1;
                ok[q] = (unsigned)r < (unsigned)(T * k);  // else not a row of y_perm: contributes nothing
                wj[q] = ok[q] ? __ldg(w + (size_t)t * k + j) : 0.f;
                // each y_perm row is read once: streaming loads, so that they do not displace the rest of L2
                u[q] = ok[q] ? __ldcs(reinterpret_cast<const uint4*>(y_perm + (size_t)r * d + 8 * c)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (!ok[q]) continue;
                const uint32_t v[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    acc[2 * m] = fmaf(wj[q], bf16_bits_to_f32(v[m] & 0xFFFF), acc[2 * m]);
                    acc[2 * m + 1] = fmaf(wj[q], bf16_bits_to_f32(v[m] >> 16), acc[2 * m + 1]);
                }
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            o[m] = (uint32_t)f32_to_bf16_bits(acc[2 * m]) | ((uint32_t)f32_to_bf16_bits(acc[2 * m + 1]) << 16);
        *reinterpret_cast<uint4*>(y + (size_t)t * d + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ weighted sum of normalised expert outputs
// Muse Spark Open explainer, section 9: each chosen expert's output is normalised before the
// router-weighted sum; the normalisation is RMSNorm over the d features (no learned scale).
// One CTA per token.  Pass 1: the sum of squares of each slot row, per thread over its 8-feature
// units in increasing order, then a warp butterfly, then the warps in order; the slot's factor
// is w[t][j] / sqrt(ss / d + eps).  Pass 2: y = sum_j factor_j * y_perm[row_j], fp32 in slot order.
// A row index outside [0, T k) is not read: that slot contributes nothing.
__global__ void __launch_bounds__(1024) combine_norm_kernel(const uint16_t* __restrict__ y_perm,
                                                            const int32_t* __restrict__ inv_pos,
                                                            const float* __restrict__ w, int T, int k, int d,
                                                            float eps, uint16_t* __restrict__ y) {
    __shared__ float red[kMaxK][32];
    __shared__ float factor[kMaxK];
    __shared__ int rows[kMaxK];
    pdl_wait();
    const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int units = d / 8;
    if (tid < k) {
        const int r = inv_pos[(size_t)t * k + tid];
        rows[tid] = ((unsigned)r < (unsigned)(T * k)) ? r : -1;
    }
    __syncthreads();
    for (int j = 0; j < k; ++j) {
        float ss = 0.f;
        if (rows[j] >= 0)
            for (int c = tid; c < units; c += blockDim.x) {
                const uint4 u = *reinterpret_cast<const uint4*>(y_perm + (size_t)rows[j] * d + 8 * c);
                const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float lo = bf16_bits_to_f32(v[m] & 0xFFFF), hi = bf16_bits_to_f32(v[m] >> 16);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
        ss = warp_sum(ss);
        if (lane == 0) red[j][warp] = ss;
    }
    __syncthreads();
    if (tid < k) {
        float ss = 0.f;
        for (int i = 0; i < nwarps; ++i) ss += red[tid][i];
        factor[tid] = rows[tid] >= 0 ? w[(size_t)t * k + tid] / sqrtf(ss / (float)d + eps) : 0.f;
    }
    __syncthreads();
    for (int c = tid; c < units; c += blockDim.x) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            if (rows[j] < 0) continue;
            const float fj = factor[j];
            const uint4 u = *reinterpret_cast<const uint4*>(y_perm + (size_t)rows[j] * d + 8 * c);
            const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acc[2 * m] = fmaf(fj, bf16_bits_to_f32(v[m] & 0xFFFF), acc[2 * m]);
                acc[2 * m + 1] = fmaf(fj, bf16_bits_to_f32(v[m] >> 16), acc[2 * m + 1]);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            o[m] = (uint32_t)f32_to_bf16_bits(acc[2 * m]) | ((uint32_t)f32_to_bf16_bits(acc[2 * m + 1]) << 16);
        *reinterpret_cast<uint4*>(y + (size_t)t * d + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
    pdl_launch_dependents();
}


// ------------------------------------------------------------------ launchers

static int bpl_for(int K) {
    const int nb = K / 32;
    return nb <= 32 ? 1 : nb <= 64 ? 2 : nb <= 128 ? 4 : nb <= 256 ? 8 : 0;
}

bool gemv_supported(int d, int I) { return bpl_for(d) != 0 && bpl_for(I) != 0; }

template <bool NV>
static const void* up_cta_kernel(int bpt, int Q) {
    if (bpt == 1) return Q == 1 ? (const void*)gemv_up_cta_kernel<1, 1, NV> : (const void*)gemv_up_cta_kernel<1, 2, NV>;
    return Q == 1 ? (const void*)gemv_up_cta_kernel<2, 1, NV> : (const void*)gemv_up_cta_kernel<2, 2, NV>;
}

template <bool NV>
static const void* up_warp_kernel(int bpl) {
    return bpl == 1 ? (const void*)gemv_up_kernel<1, NV> : bpl == 2 ? (const void*)gemv_up_kernel<2, NV>
         : bpl == 4 ? (const void*)gemv_up_kernel<4, NV> : (const void*)gemv_up_kernel<8, NV>;
}

template <bool F, bool NV>
static const void* down_kernel(int bpl) {
    return bpl == 1 ? (const void*)gemv_down_kernel<1, F, NV> : bpl == 2 ? (const void*)gemv_down_kernel<2, F, NV>
         : bpl == 4 ? (const void*)gemv_down_kernel<4, F, NV> : (const void*)gemv_down_kernel<8, F, NV>;
}

template <bool NV>
static const void* ring_kernel(int T, bool fused) {
    if (T == 1) return fused ? (const void*)gemv_down_ring_kernel<1, true, NV> : (const void*)gemv_down_ring_kernel<1, false, NV>;
    if (T == 2) return fused ? (const void*)gemv_down_ring_kernel<2, true, NV> : (const void*)gemv_down_ring_kernel<2, false, NV>;
    return fused ? (const void*)gemv_down_ring_kernel<4, true, NV> : (const void*)gemv_down_ring_kernel<4, false, NV>;
}

template <bool NV>
static size_t ring_smem(int T, int K, int P) {
    return T == 1 ? down_ring_smem<1, NV>(K, P) : T == 2 ? down_ring_smem<2, NV>(K, P) : down_ring_smem<4, NV>(K, P);
}

cudaError_t launch_gemv_up(const uint16_t* x, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                           int T, int d, int E, int k, int I, const moe_expert_weights* W, uint16_t* h,
                           cudaStream_t st, bool pdl) {
    const int P = T * k;
    if (P == 0) return cudaSuccess;
    const int bpl = bpl_for(d);
    const bool nv = W->wfmt == MOE_W_NVFP4;
    if (T <= 4 && make_cta_geo(d).bpt <= 2) {
        // up to four tokens: CTA-wide split of K (see gemv_up_cta_kernel), two token rows per pass
        const CtaGeo geo = make_cta_geo(d);
        const int unit = geo.RG * (kR / 2);
        if (I % unit != 0) return cudaErrorInvalidValue;
        int outs = unit;  // outputs per CTA: a multiple of unit dividing I, at most 64
        for (int o = unit; o <= 64 && o <= I; o += unit)
            if (I % o == 0) outs = o;
        GemvArgs a = {};
        a.q0 = W->gate_q;
        a.s0 = W->gate_s;
        a.q1 = W->up_q;
        a.s1 = W->up_s;
        a.gs0 = W->gate_gs;
        a.gs1 = W->up_gs;
        a.act = x;
        a.perm_token = perm_token;
        a.offsets = offsets;
        a.plan = plan;
        a.T = T;
        a.K = d;
        a.M_exp = I;
        a.P = P;
        a.E = E;
        a.outs = outs;
        a.out = h;
        const int Q = T < 2 ? T : 2;
        const size_t smem = (size_t)Q * d * 2 + sizeof(float) * (Q + 2 * 8 * 32) + sizeof(int) * Q + sizeof(unsigned) * Q;
        void* args[] = {&a};
        const dim3 grid(I / outs, P < E ? P : E);
        const void* f = nv ? up_cta_kernel<true>(geo.bpt, Q) : up_cta_kernel<false>(geo.bpt, Q);
        return launch_kernel(f, grid, dim3(kThr), smem, st, pdl, args);
    }
    const int outs = kWarps * kUpOutsPerWarp;
    if (bpl == 0 || I % outs != 0) return cudaErrorInvalidValue;
    GemvArgs a = {};
    a.q0 = W->gate_q;
    a.s0 = W->gate_s;
    a.q1 = W->up_q;
    a.s1 = W->up_s;
    a.gs0 = W->gate_gs;
    a.gs1 = W->up_gs;
    a.act = x;
    a.perm_token = perm_token;
    a.offsets = offsets;
    a.plan = plan;
    a.T = T;
    a.K = d;
    a.M_exp = I;
    a.P = P;
    a.E = E;
    a.outs = outs;
    a.out = h;
    const size_t smem = (size_t)kQ * d * 2 + sizeof(float) * kQ + sizeof(unsigned) * kQ + sizeof(int) * kQ;
    void* args[] = {&a};
    const dim3 grid(I / outs, P < E ? P : E);
    const void* f = nv ? up_warp_kernel<true>(bpl) : up_warp_kernel<false>(bpl);
    return launch_kernel(f, grid, dim3(kThr), smem, st, pdl, args);
}

cudaError_t launch_gemv_down(const uint16_t* h, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                             const float* row_w, int T, int d, int E, int k, int I, const moe_expert_weights* W,
                             uint16_t* y_perm, uint16_t* y, int* status, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    const CtaGeo dgeo = make_cta_geo(I);
    const int P = T * k, feats = dgeo.RG * kR;
    const bool nv = W->wfmt == MOE_W_NVFP4;
    const size_t ring_bytes = nv ? ring_smem<true>(T, I, P) : ring_smem<false>(T, I, P);
    const bool aligned16 = ((uintptr_t)W->down_q % 16 == 0) && ((uintptr_t)W->down_s % 16 == 0);
    // two CTAs per SM: 2 x (ring_smem + 1 KB reserved) within the SM's 228 KB
    const int hunits = T <= 2 ? down_hunits<2>() : down_hunits<4>();
    if (T <= 4 && dgeo.bpt == 1 && d % feats == 0 && aligned16 && T * dgeo.nb * 4 <= hunits * kThr &&
        ring_bytes <= 113 * 1024) {
        // up to four tokens: CTA-split of K, weights through the copy-engine ring
        GemvArgs a = {};
        a.q0 = W->down_q;
        a.s0 = W->down_s;
        a.gs0 = W->down_gs;
        a.act = h;
        a.perm_token = perm_token;
        a.offsets = offsets;
        a.plan = plan;
        a.row_w = row_w;
        a.T = T;
        a.K = I;
        a.M_exp = d;
        a.P = P;
        a.E = E;
        a.out = y ? y : y_perm;
        a.status = status;
        void* args[] = {&a};
        const dim3 grid(d / feats);
        const void* f = nv ? ring_kernel<true>(T, y != nullptr) : ring_kernel<false>(T, y != nullptr);
        return launch_kernel(f, grid, dim3(kThr), ring_bytes, st, pdl, args);
    }
    const int bpl = bpl_for(I);
    const int outs = kWarps * down_rows_per_warp(bpl);
    if (bpl == 0 || d % outs != 0) return cudaErrorInvalidValue;
    // tokens per chunk: at most 8, at most kDownMaxRows staged rows, staged h <= 100 KB
    int tch = 8;
    while (tch > 1 && ((size_t)tch * k > kDownMaxRows || (size_t)tch * k * I * 2 > 100 * 1024)) tch /= 2;
    if (tch > T) tch = T;
    if ((size_t)tch * k > kDownMaxRows || (size_t)tch * k * I * 2 > 200 * 1024) return cudaErrorInvalidValue;
    GemvArgs a = {};
    a.q0 = W->down_q;
    a.s0 = W->down_s;
    a.gs0 = W->down_gs;
    a.act = h;
    a.perm_token = perm_token;
    a.offsets = offsets;
    a.plan = plan;
    a.row_w = row_w;
    a.T = T;
    a.K = I;
    a.M_exp = d;
    a.P = T * k;
    a.E = E;
    a.tch = tch;
    a.maxrows = tch * k;
    a.outs = outs;
    a.out = y ? y : y_perm;
    const size_t mr = (size_t)tch * k;
    const size_t smem = mr * I * 2 + sizeof(float) * mr + sizeof(unsigned) * mr + sizeof(float) * tch * outs +
                        sizeof(int) * 3 * mr + sizeof(float) * mr + sizeof(int) * (E + 1);
    void* args[] = {&a};
    const dim3 grid(d / outs, (T + tch - 1) / tch);
    const void* f = nv ? (y ? down_kernel<true, true>(bpl) : down_kernel<false, true>(bpl))
                       : (y ? down_kernel<true, false>(bpl) : down_kernel<false, false>(bpl));
    return launch_kernel(f, grid, dim3(kThr), smem, st, pdl, args);
}

cudaError_t launch_combine_norm(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                                float eps, uint16_t* y, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    // few tokens (decode): wide CTAs, so that one token's rows stream with many loads in flight
    const int threads = T < 2 * sm_count() ? 1024 : 256;
    void* args[] = {&y_perm, &inv_pos, &w, &T, &k, &d, &eps, &y};
    return launch_kernel((const void*)combine_norm_kernel, dim3((unsigned)T), dim3(threads), 0, st, pdl, args);
}

cudaError_t launch_combine(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                           uint16_t* y, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    int64_t total = (int64_t)T * (d / 8);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    void* args[] = {&y_perm, &inv_pos, &w, &T, &k, &d, &y};
    return launch_kernel((const void*)combine_kernel, dim3((unsigned)blocks), dim3(256), 0, st, pdl, args);
}

}  // namespace moe
