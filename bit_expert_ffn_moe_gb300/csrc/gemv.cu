// gemv.cu -- decode-shape expert kernels (MOE_ACT_BF16): bf16 activations, MXFP4 weights.
//
// At decode sizes every chosen expert sees one or a few tokens, so the expert matrices are read
// once and used for very little arithmetic: the time is the weight read (Muse Spark Open
// explainer, section 13: about 98% of the time waiting on the 4-bit weight read at one token per
// expert; DGX Spark news item, section 1: batch-1 generation is bound by weight reads).  These
// kernels therefore stream each weight row once with coalesced 128-bit loads (one 16-byte load
// = one 32-element MXFP4 block), decode E2M1 with the hardware conversion, and accumulate in
// fp32 with packed fp32x2 FMAs; the block scale is applied once per 32-element partial.
//
// Activations are held in shared memory as fp32 in a "block-interleaved" order: float4 number q
// (elements 4q..4q+3) of block b sits at float4 index q*NB + b, so the 32 lanes of a warp,
// which work on 32 consecutive blocks, read 32 consecutive float4s (no bank conflicts).
#include "common.cuh"

namespace moe {

constexpr int kGemvThreads = 256;  // 8 warps
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = 8 * kRowsPerWarp;

// Stage one bf16 row of n elements (n % 32 == 0) into shared memory in block-interleaved fp32.
__device__ __forceinline__ void stage_row_bf16(const uint16_t* __restrict__ src, int n, float4* dst) {
    const int nb = n / 32;
    for (int i = threadIdx.x; i < n / 8; i += blockDim.x) {  // 8 bf16 = 16 bytes per step
        uint4 u = *reinterpret_cast<const uint4*>(src + 8 * i);
        const int b = i / 4, q = (i % 4) * 2;  // elements 8i..8i+7 = float4s q, q+1 of block b
        dst[q * nb + b] = make_float4(bf16_bits_to_f32(u.x & 0xFFFF), bf16_bits_to_f32(u.x >> 16),
                                      bf16_bits_to_f32(u.y & 0xFFFF), bf16_bits_to_f32(u.y >> 16));
        dst[(q + 1) * nb + b] = make_float4(bf16_bits_to_f32(u.z & 0xFFFF), bf16_bits_to_f32(u.z >> 16),
                                            bf16_bits_to_f32(u.w & 0xFFFF), bf16_bits_to_f32(u.w >> 16));
    }
}

// Partial dot product of one 32-element MXFP4 block (16 bytes of codes) with a block of
// activations in block-interleaved shared memory; returns the unscaled fp32 sum.
__device__ __forceinline__ float block_dot(const uint4& codes, const float4* __restrict__ act, int nb, int b) {
    float2 acc = make_float2(0.f, 0.f);
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t h[4];
        e2m1x8_to_h2(words[m], h);
        const float4 xa = act[(2 * m) * nb + b];
        const float4 xb = act[(2 * m + 1) * nb + b];
        acc = __ffma2_rn(h2_to_f2(h[0]), make_float2(xa.x, xa.y), acc);
        acc = __ffma2_rn(h2_to_f2(h[1]), make_float2(xa.z, xa.w), acc);
        acc = __ffma2_rn(h2_to_f2(h[2]), make_float2(xb.x, xb.y), acc);
        acc = __ffma2_rn(h2_to_f2(h[3]), make_float2(xb.z, xb.w), acc);
    }
    return acc.x + acc.y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// ------------------------------------------------------------------ gate/up + SwiGLU
// Grid: (I / kRowsPerCta, slots).  Slot u handles the u-th active expert; each warp computes
// kRowsPerWarp rows i of W_g and W_u for the expert's tokens, TC tokens at a time.
// CPL = 16-byte chunks per lane per pass over a row.
template <int TC, int CPL>
__global__ void __launch_bounds__(kGemvThreads)
gemv_up_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm_token,
               const int32_t* __restrict__ offsets, PlanView plan, int d, int I, const uint8_t* __restrict__ gq,
               const uint8_t* __restrict__ gs, const uint8_t* __restrict__ uq, const uint8_t* __restrict__ us,
               uint16_t* __restrict__ h) {
    extern __shared__ float4 xs4[];  // [TC][d/4] block-interleaved
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    pdl_wait();
    const int slot = blockIdx.y;
    if (slot >= plan.scalars[0]) return;
    const int e = plan.active[slot];
    const int r0 = offsets[e], n = offsets[e + 1] - r0;
    const int nb = d / 32;
    const size_t row_bytes = (size_t)d / 2;

    for (int tc0 = 0; tc0 < n; tc0 += TC) {
        const int nt = min(TC, n - tc0);
        __syncthreads();
        for (int t = 0; t < nt; ++t)
            stage_row_bf16(x + (size_t)perm_token[r0 + tc0 + t] * d, d, xs4 + (size_t)t * (d / 4));
        __syncthreads();
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int i = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp + rr;
            const size_t grow = (size_t)e * I + i;
            const uint8_t* gq_row = gq + grow * row_bytes;
            const uint8_t* uq_row = uq + grow * row_bytes;
            const uint8_t* gs_row = gs + grow * nb;
            const uint8_t* us_row = us + grow * nb;
            float ag[TC], au[TC];
#pragma unroll
            for (int t = 0; t < TC; ++t) ag[t] = au[t] = 0.f;
            for (int cb = 0; cb < nb; cb += 32 * CPL) {
                uint4 wg[CPL], wu[CPL];
                uint32_t sg[CPL], su[CPL];
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int b = cb + lane + 32 * c;
                    if (b < nb) {
                        wg[c] = ldg_stream(gq_row + 16 * (size_t)b);
                        wu[c] = ldg_stream(uq_row + 16 * (size_t)b);
                        sg[c] = __ldg(gs_row + b);
                        su[c] = __ldg(us_row + b);
                    }
                }
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    const int b = cb + lane + 32 * c;
                    if (b < nb) {
                        const float fg = e8m0_to_f32(sg[c]), fu = e8m0_to_f32(su[c]);
#pragma unroll
                        for (int t = 0; t < TC; ++t) {
                            if (t < nt) {
                                const float4* act = xs4 + (size_t)t * (d / 4);
                                ag[t] = fmaf(block_dot(wg[c], act, nb, b), fg, ag[t]);
                                au[t] = fmaf(block_dot(wu[c], act, nb, b), fu, au[t]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < TC; ++t) {
                if (t < nt) {
                    const float g = warp_sum(ag[t]), u = warp_sum(au[t]);
                    if (lane == t) {
                        const float hv = g / (1.f + expf(-g)) * u;  // SiLU(g) * u
                        h[(size_t)(r0 + tc0 + t) * I + i] = f32_to_bf16_bits(hv);
                    }
                }
            }
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ down (+ weighted sum)
// Grid: (d / kRowsPerCta, token chunks of TCH <= 8 tokens).  The CTA stages, for every permuted
// row whose token lies in its chunk, the bf16 h row (as fp32) and the pair's gate weight.  Rows
// are in expert-major order, so the active experts form consecutive segments of at most TCH
// pairs.  Each warp computes kRowsPerWarp output features for every segment, prefetching the
// next segment's weight rows while it computes the current one.
// FUSED: y[t] accumulates w * bf16(expert output) in ascending expert order, which is the slot
// order j of the token (ids are ascending); otherwise the bf16 expert outputs go to y_perm.
constexpr int kDownMaxPairs = 64;
constexpr int kDownMaxTok = 8;

template <int CPL>
__device__ __forceinline__ void load_down_rows(const uint8_t* __restrict__ dq, const uint8_t* __restrict__ ds, int e,
                                               int d, int nb, int n0, int cb, int lane,
                                               uint4 (&wv)[kRowsPerWarp][CPL], uint32_t (&sv)[kRowsPerWarp][CPL]) {
    const size_t row_bytes = (size_t)nb * 16;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const size_t grow = (size_t)e * d + n0 + rr;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int b = cb + lane + 32 * c;
            if (b < nb) {
                wv[rr][c] = ldg_stream(dq + grow * row_bytes + 16 * (size_t)b);
                sv[rr][c] = __ldg(ds + grow * nb + b);
            }
        }
    }
}

template <int CPL, bool FUSED>
__global__ void __launch_bounds__(kGemvThreads)
gemv_down_kernel(const uint16_t* __restrict__ h, const int32_t* __restrict__ perm_token,
                 const int32_t* __restrict__ offsets, PlanView plan, const int32_t* __restrict__ ids,
                 const float* __restrict__ wts, int T, int TCH, int d, int k, int I, const uint8_t* __restrict__ dq,
                 const uint8_t* __restrict__ ds, uint16_t* __restrict__ y_perm, uint16_t* __restrict__ y) {
    extern __shared__ float4 hs4[];  // [pairs][I/4] block-interleaved
    __shared__ int s_row[kDownMaxPairs], s_tok[kDownMaxPairs], s_exp[kDownMaxPairs];
    __shared__ float s_w[kDownMaxPairs];
    __shared__ int s_np;
    __shared__ float ys[kRowsPerCta][kDownMaxTok];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.y * TCH, t1 = min(T, t0 + TCH);
    const int nb = I / 32;
    pdl_wait();

    if (threadIdx.x == 0) {
        int np = 0;
        const int n_act = plan.scalars[0];
        for (int u = 0; u < n_act; ++u) {
            const int e = plan.active[u];
            for (int r = offsets[e]; r < offsets[e + 1]; ++r) {
                const int t = perm_token[r];
                if (t < t0 || t >= t1) continue;
                float wv = 0.f;
                if (FUSED) {
                    int j = 0;
                    while (j < k - 1 && ids[(size_t)t * k + j] != e) ++j;
                    wv = wts[(size_t)t * k + j];
                }
                s_row[np] = r;
                s_tok[np] = t - t0;
                s_exp[np] = e;
                s_w[np] = wv;
                ++np;
            }
        }
        s_np = np;
    }
    for (int i = threadIdx.x; i < kRowsPerCta * kDownMaxTok; i += blockDim.x) (&ys[0][0])[i] = 0.f;
    __syncthreads();
    const int np = s_np;
    for (int q = 0; q < np; ++q) stage_row_bf16(h + (size_t)s_row[q] * I, I, hs4 + (size_t)q * (I / 4));
    __syncthreads();

    const int n0 = blockIdx.x * kRowsPerCta + warp * kRowsPerWarp;
    const bool single = nb <= 32 * CPL;
    uint4 wcur[kRowsPerWarp][CPL], wnxt[kRowsPerWarp][CPL];
    uint32_t scur[kRowsPerWarp][CPL], snxt[kRowsPerWarp][CPL];
    if (np > 0 && single) load_down_rows<CPL>(dq, ds, s_exp[0], d, nb, n0, 0, lane, wcur, scur);
    int q0 = 0;
    while (q0 < np) {
        const int e = s_exp[q0];
        int q1 = q0 + 1;
        while (q1 < np && s_exp[q1] == e) ++q1;
        float acc[kRowsPerWarp][kDownMaxTok];
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
            for (int qi = 0; qi < kDownMaxTok; ++qi) acc[rr][qi] = 0.f;
        for (int cb = 0; cb < nb; cb += 32 * CPL) {
            if (single) {
                if (q1 < np) load_down_rows<CPL>(dq, ds, s_exp[q1], d, nb, n0, 0, lane, wnxt, snxt);
            } else {
                load_down_rows<CPL>(dq, ds, e, d, nb, n0, cb, lane, wcur, scur);
            }
#pragma unroll
            for (int qi = 0; qi < kDownMaxTok; ++qi) {
                if (q0 + qi < q1) {
                    const float4* act = hs4 + (size_t)(q0 + qi) * (I / 4);
#pragma unroll
                    for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
                        for (int c = 0; c < CPL; ++c) {
                            const int b = cb + lane + 32 * c;
                            if (b < nb)
                                acc[rr][qi] = fmaf(block_dot(wcur[rr][c], act, nb, b), e8m0_to_f32(scur[rr][c]),
                                                   acc[rr][qi]);
                        }
                }
            }
        }
#pragma unroll
        for (int qi = 0; qi < kDownMaxTok; ++qi) {
            if (q0 + qi < q1) {
#pragma unroll
                for (int rr = 0; rr < kRowsPerWarp; ++rr) {
                    const float s = warp_sum(acc[rr][qi]);
                    if (lane == 0) {
                        const uint16_t sb = f32_to_bf16_bits(s);
                        if (FUSED) {
                            float& a = ys[warp * kRowsPerWarp + rr][s_tok[q0 + qi]];
                            a = fmaf(s_w[q0 + qi], bf16_bits_to_f32(sb), a);
                        } else {
                            y_perm[(size_t)s_row[q0 + qi] * d + n0 + rr] = sb;
                        }
                    }
                }
            }
        }
        if (single && q1 < np) {
#pragma unroll
            for (int rr = 0; rr < kRowsPerWarp; ++rr)
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    wcur[rr][c] = wnxt[rr][c];
                    scur[rr][c] = snxt[rr][c];
                }
        }
        q0 = q1;
    }
    if (FUSED) {
        __syncthreads();
        for (int i = threadIdx.x; i < kRowsPerCta * (t1 - t0); i += blockDim.x) {
            const int tt = i / kRowsPerCta, rr = i % kRowsPerCta;
            y[(size_t)(t0 + tt) * d + blockIdx.x * kRowsPerCta + rr] = f32_to_bf16_bits(ys[rr][tt]);
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ weighted sum (unfused)
// One thread per (token, 8 consecutive features): y = sum_j w[t][j] * y_perm[inv_pos[t*k+j]].
__global__ void combine_kernel(const uint16_t* __restrict__ y_perm, const int32_t* __restrict__ inv_pos,
                               const float* __restrict__ w, int T, int k, int d, uint16_t* __restrict__ y) {
    pdl_wait();
    const int per_row = d / 8;
    const int64_t total = (int64_t)T * per_row;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / per_row), c = (int)(i % per_row);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const float wj = w[(size_t)t * k + j];
            const uint4 u = *reinterpret_cast<const uint4*>(y_perm + (size_t)inv_pos[(size_t)t * k + j] * d + 8 * c);
            const uint32_t v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                acc[2 * m] = fmaf(wj, bf16_bits_to_f32(v[m] & 0xFFFF), acc[2 * m]);
                acc[2 * m + 1] = fmaf(wj, bf16_bits_to_f32(v[m] >> 16), acc[2 * m + 1]);
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


template <int TC, int CPL>
static cudaError_t up_variant(dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args) {
    const void* f = (const void*)gemv_up_kernel<TC, CPL>;
    return launch_kernel(f, grid, dim3(kGemvThreads), smem, st, pdl, args);
}

template <int TC>
static cudaError_t up_cpl(int nb, dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args) {
    if (nb <= 32) return up_variant<TC, 1>(grid, smem, st, pdl, args);
    if (nb <= 64) return up_variant<TC, 2>(grid, smem, st, pdl, args);
    if (nb <= 128) return up_variant<TC, 4>(grid, smem, st, pdl, args);
    return up_variant<TC, 8>(grid, smem, st, pdl, args);
}

cudaError_t launch_gemv_up(const uint16_t* x, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                           int T, int d, int E, int k, int I, const moe_expert_weights* W, uint16_t* h,
                           cudaStream_t st, bool pdl) {
    const int P = T * k;
    if (P == 0) return cudaSuccess;
    const int slots = P < E ? P : E;
    // token chunk: all of a decode step's tokens when they fit in <= 128 KB of fp32 staging
    int TC = 1;
    while (TC < T && TC < 4 && (size_t)(2 * TC) * d * 4 <= 128 * 1024) TC *= 2;
    const size_t smem = (size_t)TC * d * 4;
    dim3 grid(I / kRowsPerCta, slots);
    const int nb = d / 32;
    const uint8_t *gq = W->gate_q, *gs = W->gate_s, *uq = W->up_q, *us = W->up_s;
    void* args[] = {&x, &perm_token, &offsets, &plan, &d, &I, &gq, &gs, &uq, &us, &h};
    switch (TC) {
        case 1: return up_cpl<1>(nb, grid, smem, st, pdl, args);
        case 2: return up_cpl<2>(nb, grid, smem, st, pdl, args);
        default: return up_cpl<4>(nb, grid, smem, st, pdl, args);
    }
}

template <int CPL, bool FUSED>
static cudaError_t down_variant(dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args) {
    const void* f = (const void*)gemv_down_kernel<CPL, FUSED>;
    return launch_kernel(f, grid, dim3(kGemvThreads), smem, st, pdl, args);
}

template <bool FUSED>
static cudaError_t down_cpl(int nb, dim3 grid, size_t smem, cudaStream_t st, bool pdl, void** args) {
    if (nb <= 32) return down_variant<1, FUSED>(grid, smem, st, pdl, args);
    if (nb <= 64) return down_variant<2, FUSED>(grid, smem, st, pdl, args);
    return down_variant<4, FUSED>(grid, smem, st, pdl, args);
}

cudaError_t launch_gemv_down(const uint16_t* h, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                             const int32_t* ids, const float* w, int T, int d, int E, int k, int I,
                             const moe_expert_weights* W, uint16_t* y_perm, uint16_t* y, cudaStream_t st, bool pdl) {
    (void)E;
    if (T == 0) return cudaSuccess;
    // token chunk: at most kDownMaxTok tokens and kDownMaxPairs pairs, staged h <= 160 KB
    int TCH = T < kDownMaxTok ? T : kDownMaxTok;
    while (TCH > 1 && ((size_t)TCH * k > kDownMaxPairs || (size_t)TCH * k * I * 4 > 160 * 1024)) TCH /= 2;
    if ((size_t)TCH * k > kDownMaxPairs || (size_t)TCH * k * I * 4 > 200 * 1024) return cudaErrorInvalidValue;
    const size_t smem = (size_t)TCH * k * I * 4;
    dim3 grid(d / kRowsPerCta, (T + TCH - 1) / TCH);
    const int nb = I / 32;
    const uint8_t *dq = W->down_q, *ds = W->down_s;
    void* args[] = {&h, &perm_token, &offsets, &plan, &ids, &w, &T, &TCH, &d, &k, &I, &dq, &ds, &y_perm, &y};
    if (y != nullptr) return down_cpl<true>(nb, grid, smem, st, pdl, args);
    return down_cpl<false>(nb, grid, smem, st, pdl, args);
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
