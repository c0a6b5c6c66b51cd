// route_screen.cu -- router logits of many tokens: a tensor-core screen with a certified error bound,
// then the fixed-order fp32 logits only for the experts the screen cannot rule out.
//
// The router is one fp32 matrix product followed by a top-k (Muse Spark Open explainer, section 8);
// the choice is a set.  The logits are defined by a fixed fp32 reduction order (route_common.cuh)
// so that the chosen ids are reproducible bit for bit, and at prefill sizes those T d E sequential
// fmas are most of the routing time.  But the top-k only needs the logits of the experts that can
// still be among a token's k largest, and the weights only the logits of the chosen ones:
//
//   1. router_split_kernel   W_r = hi + lo + r with hi = bf16(w), lo = bf16(w - hi), so |r| <= 2^-16 |w|;
//                            hi and lo stored as tensor-core operand tiles; ||w_e||^2 per expert;
//   2. router_screen_kernel  a = x hi^T + x lo^T on the tensor cores (tcgen05 kind::f16: bf16 operands,
//                            fp32 accumulators; x is bf16 already, so every product is exact; the hi
//                            and lo rows of 128 experts are one N = 256 operand), with ||x_t||^2 summed
//                            from the staged token tiles;
//   3. router_cand_kernel    per token a bound eps_t >= |a_e - l_e| for every expert e (l = the
//                            fixed-order logit), the k-th largest screened value v, and the
//                            candidates a_e >= v - 2 eps_t; every other expert gets the logit -inf;
//   4. router_exact_kernel   the fixed-order logits of the candidates, grouped by expert;
//   5. topk_kernel           the usual top-k + softmax over the logits (route.cu).
//
// Why the candidates hold the exact top-k: the k experts with the largest a all have
// l >= a - eps >= v - eps, so the k-th largest l is at least v - eps; an expert of the exact top-k has
// l at least that, so a >= l - eps >= v - 2 eps.  An expert outside has l < v - eps, strictly below the
// k-th largest l, so no tie with it is decided differently either.
//
// The bound (all sums over the d elements of one logit; S = sum_i |x_i w_i| <= ||x|| ||w|| by
// Cauchy-Schwarz):
//   - the split: sum |x_i r_i| <= 2^-16 S;
//   - the tensor-core accumulation: each accumulation step (one MMA: 16 exact products added to the
//     fp32 accumulator) is taken to err by at most 2^-17 (|acc| + sum of its |products|), eight times
//     the error of an fp32 sum that truncates each of its 17 aligned terms; over n steps into one
//     accumulator that is at most n 2^-17 (1 + n 2^-17) S.  The PTX ISA does not specify the
//     accumulation's internal rounding, so this is an assumption about the hardware, stated here and
//     kept loose; the GPU tests compare the chosen ids with the oracle's on every workload;
//   - the fp32 sums of the accumulators (hi and lo parts of R of them), of the K-split partial sums
//     and the bias: (2 R S_k + 2) 2^-24 S plus 2^-23 max|b|;
//   - the fixed-order logit itself: d/32 sequential fmas per partial sum and a 5-level butterfly, at
//     most (d/32 + 6) 2^-24 S from the exact value;
//   - flushed subnormals: at most 2^-124 sqrt(d) (||x|| + ||w||).
// The norms are summed in fp32 and inflated by their own worst-case relative error, the final
// products and sums are rounded upward and the threshold downward.  A token whose screened values,
// norms or bound are not finite takes every expert as a candidate (then nothing is screened out).
#include <cmath>

#include "route_common.cuh"
#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kScrTile = 128 * 128;          // operand tile: 128 rows x 64 bf16 values (128 bytes)
constexpr int kScrStages = 4;
constexpr int kScrStageBytes = 3 * kScrTile;  // token tile, hi tile, lo tile
constexpr int kScrAcc = 2;                    // accumulators (256 columns: hi, lo), taken in turn by the stages
constexpr int kScrEpiWarps = 4;
constexpr int kScrThreads = 64 + 32 * kScrEpiWarps;  // producer, MMA issuer, 4 epilogue warps
constexpr int kScrBarBytes = 128;
constexpr size_t kScrSmem = (size_t)kScrStages * kScrStageBytes + 1024 + kScrBarBytes;
constexpr int kScrMinT = 256;         // fewer tokens: the dense fixed-order kernel
constexpr int kScrTargetCtas = 148;   // K splits fill about this many CTAs (one per SM)
constexpr int kSplitParts = 4;        // CTAs per router row in the split kernel
constexpr int kScrMaxD = 32768;       // the exact kernel holds one fp32 router row in shared memory
constexpr int kXTile = 32;            // candidate tokens per work item of the exact kernel (4 per warp)
constexpr int kXThreads = 256;
constexpr int kXBatch = 8;            // x loads in flight per lane and token

// ------------------------------------------------------------------ 1. split of W_r
// CTA (e, part) writes a quarter of row e of the hi and lo operand matrices ([E_pad][d] bf16, in
// 128 x 64 tiles with the 128-byte swizzle: 16-byte chunk j of row r at chunk position j ^ (r % 8));
// rows past E are zero.  Also that quarter's share of ||w_e||^2 (wn2 [kSplitParts][E]) and the
// reset of the expert's candidate count (and of its pick count, when the top-k counts picks).
__global__ void __launch_bounds__(256) router_split_kernel(const float* __restrict__ W_r, int E, int d,
                                                           uint8_t* __restrict__ bhi, uint8_t* __restrict__ blo,
                                                           float* __restrict__ wn2, int32_t* __restrict__ cnt,
                                                           int32_t* __restrict__ counts) {
    __shared__ float red[8];
    pdl_wait();
    const int e = blockIdx.x, KB = d / 64, rb = e / 128, r = e % 128;
    const int c_per = d / 8 / kSplitParts;  // 16-byte output chunks of this CTA (d % 128 == 0)
    float s2 = 0.f;
    for (int c = blockIdx.y * c_per + threadIdx.x; c < (blockIdx.y + 1) * c_per; c += blockDim.x) {
        float v[8];
        if (e < E) {
            const float4 p0 = __ldg(reinterpret_cast<const float4*>(W_r + (size_t)e * d) + 2 * c);
            const float4 p1 = __ldg(reinterpret_cast<const float4*>(W_r + (size_t)e * d) + 2 * c + 1);
            v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
            v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        uint32_t hw[4], lw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * i]), h1 = __float2bfloat16_rn(v[2 * i + 1]);
            // w - hi is exact in fp32 (hi is w rounded to fewer bits)
            const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * i] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * i + 1] - __bfloat162float(h1));
            hw[i] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
            lw[i] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            s2 = fmaf(v[2 * i], v[2 * i], s2);
            s2 = fmaf(v[2 * i + 1], v[2 * i + 1], s2);
        }
        const int kb = c / 8, j = c % 8;
        const size_t off = ((size_t)rb * KB + kb) * kScrTile + (size_t)r * 128 + (size_t)((j ^ (r & 7)) * 16);
        *reinterpret_cast<uint4*>(bhi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4*>(blo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s2;
    __syncthreads();
    if (threadIdx.x == 0 && e < E) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        wn2[(size_t)blockIdx.y * E + e] = t;
        if (blockIdx.y == 0) {
            cnt[e] = 0;
            if (counts) counts[e] = 0;  // the per-expert pick counts the top-k adds to
        }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ 2. tensor-core screen
struct ScreenArgs {
    CUtensorMap tmap_x;  // x bf16 [T][d]: boxes of 64 values x 128 rows, 128-byte swizzle, zeros past T
    const uint8_t* bhi;  // [E_pad / 128][d / 64] tiles of 16 KB
    const uint8_t* blo;
    float* part;  // [S][T][E_pad] screened partial values of each K split
    float* xn2;   // [S][T] partial ||x_t||^2 of each K split
    const float* wn2;  // [4][E] shares of ||w_e||^2, and the bias: CTA (0, 0, 0) writes their maxima to stat
    const float* b;
    uint32_t* stat;    // max ||w_e||^2, max |b_e| (bit patterns), 1 when all are finite
    int T, E, E_pad, KB, kb_per;  // KB = d / 64 stages in all, kb_per of them per K split
    int* status;
};

// CTA (token tile, 128-expert tile, K split).  Warp 0: copies (the token box through the tensor map,
// the hi and lo tiles as 1-D bulk copies, which land as one 256-row operand); warp 1: tensor memory
// and the MMAs (M = 128 tokens, N = 256: hi rows in accumulator columns 0..127, lo rows in
// 128..255), stage s into accumulator s % 2; warps 2-5: while the stages stream, each thread sums
// the squares of its token row's values in the staged token tile (the stage is freed by the MMAs'
// commit and these four warps); at the end it adds the hi and lo parts of its row's accumulators in
// fixed order and stores them.
__global__ void __launch_bounds__(kScrThreads, 1) router_screen_kernel(const __grid_constant__ ScreenArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kScrStages * kScrStageBytes);
    uint64_t* empty = full + kScrStages;
    uint64_t* acc_full = empty + kScrStages;
    uint64_t* mma_done = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * 128, nb = blockIdx.y, split = blockIdx.z;
    const int kb0 = split * a.kb_per, nk = a.kb_per;
    auto stage = [&](int s) { return smem + (size_t)s * kScrStageBytes; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kScrStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + kScrEpiWarps);
        }
        mbar_init(acc_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();  // the operand tiles come from the split kernel

    if (warp == 0) {
        if (lane == 0) {
            int i = 0;
            for (; i < nk; ++i) {
                const int s = i % kScrStages;
                if (!mbar_wait(&empty[s], ((i / kScrStages) & 1) ^ 1, abort_flag, a.status)) break;
                const int kb = kb0 + i;
                const size_t tile = ((size_t)nb * a.KB + kb) * kScrTile;
                mbar_arrive_expect_tx(&full[s], kScrStageBytes);
                tma_load_2d(stage(s), &a.tmap_x, kb * 64, m0, &full[s]);
                bulk_load(stage(s) + kScrTile, a.bhi + tile, kScrTile, &full[s]);
                bulk_load(stage(s) + 2 * kScrTile, a.blo + tile, kScrTile, &full[s]);
            }
            if (*abort_flag) {  // let the issued copies land before shared memory is released
                volatile int never = 0;
                for (int q = 0; q < kScrStages && q < i; ++q) {
                    const int it = i - 1 - q;
                    mbar_wait(&full[it % kScrStages], (it / kScrStages) & 1, &never, nullptr, 100000000LL);
                }
            }
        }
    } else if (warp == 1) {
        const uint32_t idesc = idesc_f16_bf16(128, 256);
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
            const int s = i % kScrStages;
            if (!mbar_wait_warp(&full[s], (i / kScrStages) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            stage_mmas_bf16_commit(tmem + (uint32_t)((i % kScrAcc) * 256), desc_sw128(stage(s)),
                                   desc_sw128(stage(s) + kScrTile), idesc, i >= kScrAcc ? 1u : 0u, &empty[s]);
        }
        if (ok) tc_commit(acc_full);
        tc_commit(mma_done);
        volatile int never = 0;  // every MMA has completed before tensor memory is freed
        mbar_wait_warp(mma_done, 0, &never, nullptr, 100000000LL);
    } else {
        const int q = warp & 3;  // tensor-memory lane quarter
        const int m = 32 * q + lane;
        if (warp == 2 && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
            // the maxima the candidate bounds use, the same for every token
            uint32_t wm = 0, bm = 0;  // bit patterns of non-negative floats order like the values
            bool fin = true;
            for (int e = lane; e < a.E; e += 32) {
                float w2 = 0.f;
                for (int p4 = 0; p4 < kSplitParts; ++p4) w2 += __ldcg(a.wn2 + (size_t)p4 * a.E + e);
                const float be = a.b ? __ldg(a.b + e) : 0.f;
                fin = fin && isfinite(w2) && isfinite(be);
                wm = max(wm, __float_as_uint(w2));
                bm = max(bm, __float_as_uint(fabsf(be)));
            }
            wm = __reduce_max_sync(0xffffffffu, wm);
            bm = __reduce_max_sync(0xffffffffu, bm);
            fin = __all_sync(0xffffffffu, fin);
            if (lane == 0) {
                a.stat[0] = wm;
                a.stat[1] = bm;
                a.stat[2] = fin ? 1u : 0u;
            }
        }
        float s2 = 0.f;
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
            const int s = i % kScrStages;
            if (!mbar_wait_warp(&full[s], (i / kScrStages) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            // the row's 16-byte chunks in their swizzled order (the sum is bounded, not pinned): lanes
            // m .. m + 7 then read eight different bank groups
            const uint4* row = reinterpret_cast<const uint4*>(stage(s) + (size_t)m * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 u = row[j ^ (m & 7)];
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float x0 = __uint_as_float(w4[h] << 16), x1 = __uint_as_float(w4[h] & 0xFFFF0000u);
                    s2 = fmaf(x0, x0, s2);
                    s2 = fmaf(x1, x1, s2);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (ok && mbar_wait_warp(acc_full, 0, abort_flag, a.status)) {
            tc_fence_after();
            const int t = m0 + m;
            const uint32_t lane_base = (uint32_t)(32 * q) << 16;
            const int n_used = nk < kScrAcc ? nk : kScrAcc;
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                float sum[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(32 * c), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) sum[i] = __uint_as_float(v[i]);
                for (int r = 0; r < n_used; ++r) {  // hi of accumulator 0 taken; then lo 0, hi 1, lo 1
                    if (r > 0) {
                        tmem_ld32(tmem + lane_base + (uint32_t)(256 * r + 32 * c), v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(v[i]);
                    }
                    tmem_ld32(tmem + lane_base + (uint32_t)(256 * r + 128 + 32 * c), v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) sum[i] += __uint_as_float(v[i]);
                }
                if (t < a.T) {
                    float4* dst = reinterpret_cast<float4*>(a.part + ((size_t)split * a.T + t) * a.E_pad +
                                                            (size_t)nb * 128 + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(sum[4 * i], sum[4 * i + 1], sum[4 * i + 2], sum[4 * i + 3]);
                }
            }
            if (nb == 0 && t < a.T) a.xn2[(size_t)split * a.T + t] = s2;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ 3. candidates
// 32 tokens per CTA, one warp per token at a time (lane l holds experts l + 32 i).  The candidates
// are counted per expert in shared memory first, so that each CTA adds to an expert's global count
// once (the load is skewed: a popular expert is a candidate of most tokens), then written to the
// experts' lists.  C: the relative bound factor (host side), tiny: sqrt(d) 2^-124.
// tokens per CTA of the candidate kernel (16 warps): one per warp up to 128 experts, two beyond
// (fewer CTAs, half the global count atomics; measured 8.9 / 11.9 us at 128 experts with one / two,
// 23.4 / 19.9 us at 256)
template <int NV>
__host__ __device__ constexpr int cand_tokens() { return NV <= 4 ? 16 : 32; }
template <int NV>
__global__ void __launch_bounds__(512, 2) router_cand_kernel(const float* __restrict__ part, const float* __restrict__ xn2,
                                                          int S, int T, int d, int E, int E_pad, int k,
                                                          const float* __restrict__ b,
                                                          const uint32_t* __restrict__ stat, float C, float tiny,
                                                          float* __restrict__ logits, int32_t* __restrict__ cnt,
                                                          int32_t* __restrict__ list) {
    __shared__ int lcnt[kMaxE];
    constexpr int kCandTok = cand_tokens<NV>();
    __shared__ uint32_t mask[kCandTok][NV];  // candidate bits of each token: bit l of word i = expert l + 32 i
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __shared__ uint32_t s_wm, s_bm;  // bit patterns of non-negative floats order like the values
    __shared__ int s_fin;
    pdl_wait();
    if (threadIdx.x == 0) {  // max ||w_e||^2 and max |b_e| over the experts (the screen kernel's)
        s_wm = __ldcg(stat);
        s_bm = __ldcg(stat + 1);
        s_fin = (int)__ldcg(stat + 2);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x) lcnt[e] = 0;
    __syncthreads();
    for (int u = 0; u < kCandTok / 16; ++u) {
        const int tl = warp + 16 * u, t = blockIdx.x * kCandTok + tl;
        if (t >= T) {
            if (lane < NV) mask[tl][lane] = 0u;
            continue;
        }
        // the loads of up to four K splits are issued before the sums that wait for them (in split order)
        float av[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            av[i] = e < E ? __ldcg(part + (size_t)t * E_pad + e) : 0.f;
        }
        float nx2 = __ldcg(xn2 + t);
        constexpr int kB = NV <= 4 ? 4 : NV <= 8 ? 2 : 1;
        for (int sp0 = 1; sp0 < S; sp0 += kB) {
            float pv[kB][NV], xv[kB];
#pragma unroll
            for (int q = 0; q < kB; ++q) {
                const int sp = sp0 + q;
                xv[q] = 0.f;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int e = lane + 32 * i;
                    pv[q][i] = sp < S && e < E ? __ldcg(part + ((size_t)sp * T + t) * E_pad + e) : 0.f;
                }
                if (sp < S) xv[q] = __ldcg(xn2 + (size_t)sp * T + t);
            }
#pragma unroll
            for (int q = 0; q < kB; ++q)
                if (sp0 + q < S) {
#pragma unroll
                    for (int i = 0; i < NV; ++i) av[i] += pv[q][i];
                    nx2 += xv[q];
                }
        }
        bool fin = s_fin != 0;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (e < E) {
                av[i] = av[i] + (b ? __ldg(b + e) : 0.f);
                fin = fin && isfinite(av[i]);
            }
        }
        fin = __all_sync(0xffffffffu, fin);
        const float wmax2 = __uint_as_float(s_wm), bmax = __uint_as_float(s_bm);
        // the fp32 sums of squares carry a relative error below (terms) 2^-24
        const float infl = 1.f + (float)(d + S + 8) * 0x1p-23f;
        const float nx = __fsqrt_ru(__fmul_ru(nx2, infl));
        const float wx = __fsqrt_ru(__fmul_ru(wmax2, infl));
        float eps = __fmul_ru(__fmul_ru(C, nx), wx);
        eps = __fadd_ru(eps, __fmul_ru(0x1p-22f, bmax));
        eps = __fadd_ru(eps, __fmul_ru(tiny, __fadd_ru(nx, wx)));
        const bool all = !fin || !(eps <= 1.0e37f);
        float thr = -INFINITY;
        if (!all) {
            // the k-th largest screened value: k rounds of the warp maximum over the keys not yet taken
            uint32_t key[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i) key[i] = lane + 32 * i < E ? logit_key(av[i]) : 0u;
            uint32_t taken = 0, wb = 0;
            for (int r = 0; r < k; ++r) {
                uint32_t lb = 0;
                int li = 0;
#pragma unroll
                for (int i = 0; i < NV; ++i)
                    if (!((taken >> i) & 1u) && key[i] > lb) {
                        lb = key[i];
                        li = i;
                    }
                wb = __reduce_max_sync(0xffffffffu, lb);
                const int id = __reduce_min_sync(0xffffffffu, (lb == wb) ? lane + 32 * li : 0x7fffffff);
                if ((id & 31) == lane) taken |= 1u << (id >> 5);
            }
            thr = __fsub_rd(key_logit(wb), __fmul_ru(2.f, eps));
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            const bool c = e < E && (all || av[i] >= thr);
            const uint32_t bits = __ballot_sync(0xffffffffu, c);
            if (lane == 0) mask[tl][i] = bits;
            if (c) atomicAdd(lcnt + e, 1);
            else if (e < E) logits[(size_t)t * E + e] = -INFINITY;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {  // this CTA's slice of each expert's list
        const int n = lcnt[e];
        lcnt[e] = n ? atomicAdd(cnt + e, n) : 0;
    }
    __syncthreads();
    for (int u = 0; u < kCandTok / 16; ++u) {
        const int tl = warp + 16 * u, t = blockIdx.x * kCandTok + tl;
        if (t >= T) continue;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if ((mask[tl][i] >> lane) & 1u) {
                const int e = lane + 32 * i;
                list[(size_t)e * T + atomicAdd(lcnt + e, 1)] = t;
            }
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ 4. exact logits of the candidates
// Work items: (expert e, 32 of its candidate tokens), numbered expert by expert; each CTA takes a
// contiguous range of items, so it reloads the expert's router row (fp32, shared memory) only when
// the expert changes.  Warp w computes tokens 4w .. 4w + 3 of an item in the fixed order: lane c
// accumulates the elements i with (i/4) % 32 == c in increasing i (two tokens per packed fma), then
// the butterfly and the bias.
__global__ void __launch_bounds__(kXThreads, 2) router_exact_kernel(const uint16_t* __restrict__ x,
                                                                 const float* __restrict__ W_r,
                                                                 const float* __restrict__ b, int T, int d, int E,
                                                                 const int32_t* __restrict__ cnt,
                                                                 const int32_t* __restrict__ list,
                                                                 float* __restrict__ logits) {
    extern __shared__ __align__(16) unsigned char xsm[];
    float* wsm = reinterpret_cast<float*>(xsm);                  // [d]
    int32_t* pre = reinterpret_cast<int32_t*>(xsm + (size_t)d * 4);  // [E + 1]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    if (warp == 0) {  // exclusive prefix of the items per expert
        int run = 0;
        for (int e0 = 0; e0 < E; e0 += 32) {
            const int e = e0 + lane;
            const int n = e < E ? (__ldcg(cnt + e) + kXTile - 1) / kXTile : 0;
            int incl = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (e < E) pre[e] = run + incl - n;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) pre[E] = run;
    }
    __syncthreads();
    const int total = pre[E];
    const int it0 = (int)((long long)total * blockIdx.x / gridDim.x);
    const int it1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
    int cur = -1;
    for (int it = it0; it < it1; ++it) {
        int lo = 0, hi = E - 1;  // the last expert whose items start at or before `it`
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= it) lo = mid;
            else hi = mid - 1;
        }
        const int e = lo;
        if (e != cur) {
            __syncthreads();
            for (int i = 4 * tid; i < d; i += 4 * kXThreads)
                *reinterpret_cast<float4*>(wsm + i) = __ldg(reinterpret_cast<const float4*>(W_r + (size_t)e * d + i));
            __syncthreads();
            cur = e;
        }
        const int j = it - pre[e];
        const int n = min(kXTile, __ldcg(cnt + e) - j * kXTile);
        const int32_t* lst = list + (size_t)e * T + (size_t)j * kXTile;
        int tk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) tk[u] = 4 * warp + u < n ? __ldcg(lst + 4 * warp + u) : -1;
        if (tk[0] < 0) continue;
        const uint2* xr[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) xr[u] = reinterpret_cast<const uint2*>(x + (size_t)(tk[u] >= 0 ? tk[u] : tk[0]) * d);
        float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
        // lane c takes groups g = c + 32 j (elements 4g .. 4g + 3) for j = 0 .. d/128 - 1 in order; the
        // x loads of eight consecutive j are issued before their fmas
        const int nj = d / 128;
        for (int j0 = 0; j0 < nj; j0 += kXBatch) {
            uint2 xv[kXBatch][4];
#pragma unroll
            for (int u = 0; u < kXBatch; ++u)
                if (j0 + u < nj) {
                    const int g = lane + 32 * (j0 + u);
#pragma unroll
                    for (int q = 0; q < 4; ++q) xv[u][q] = __ldg(xr[q] + g);
                }
#pragma unroll
            for (int u = 0; u < kXBatch; ++u)
                if (j0 + u < nj) {
                    const float4 wv = *reinterpret_cast<const float4*>(wsm + 4 * (lane + 32 * (j0 + u)));
                    const float w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) {
                        const int h = qd >> 1;
                        const bool up = qd & 1;
                        const uint32_t p0 = h ? xv[u][0].y : xv[u][0].x, p1 = h ? xv[u][1].y : xv[u][1].x;
                        const uint32_t p2 = h ? xv[u][2].y : xv[u][2].x, p3 = h ? xv[u][3].y : xv[u][3].x;
                        const float x0 = __uint_as_float(up ? (p0 & 0xFFFF0000u) : (p0 << 16));
                        const float x1 = __uint_as_float(up ? (p1 & 0xFFFF0000u) : (p1 << 16));
                        const float x2 = __uint_as_float(up ? (p2 & 0xFFFF0000u) : (p2 << 16));
                        const float x3 = __uint_as_float(up ? (p3 & 0xFFFF0000u) : (p3 << 16));
                        const float2 wq = make_float2(w4[qd], w4[qd]);
                        acc01 = fma2(make_float2(x0, x1), wq, acc01);
                        acc23 = fma2(make_float2(x2, x3), wq, acc23);
                    }
                }
        }
        const float s0 = warp_butterfly_sum(acc01.x), s1 = warp_butterfly_sum(acc01.y);
        const float s2 = warp_butterfly_sum(acc23.x), s3 = warp_butterfly_sum(acc23.y);
        if (lane == 0) {
            const float be = b ? __ldg(b + e) : 0.f;
            const float s[4] = {s0, s1, s2, s3};
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (tk[u] >= 0) logits[(size_t)tk[u] * E + e] = s[u] + be;
        }
    }
    pdl_launch_dependents();
}

// Tensor map of x bf16 [T][d] in boxes of 64 values x 128 rows with the 128-byte swizzle (zeros past T).
cudaError_t x_tensor_map(CUtensorMap* m, const uint16_t* x, int T, int d) {
    encode_tiled_fn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)T};
    const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int router_screen_splits(int T, int d, int E) {
    // the candidate lists and the screened values take 4 T E bytes each (and the values once per K
    // split): beyond 2^25 token-expert pairs the dense kernel routes, with no such buffers
    if (T < kScrMinT || d % 128 != 0 || d > kScrMaxD || E > kMaxE || (int64_t)T * E > ((int64_t)1 << 25)) return 0;
    const int KB = d / 64;
    const int tiles = ((T + 127) / 128) * ((E + 127) / 128);
    int S = 1;
    while (tiles * S * 2 <= kScrTargetCtas && KB % (2 * S) == 0 && KB / (2 * S) >= 2) S *= 2;
    return S;
}

RouterScreenSizes router_screen_sizes(int T, int d, int E) {
    RouterScreenSizes z{};
    z.S = router_screen_splits(T, d, E);
    if (!z.S) return z;
    const size_t E_pad = (size_t)(E + 127) / 128 * 128;
    z.b_bytes = E_pad * d * 2;
    z.wn2_bytes = sizeof(float) * kSplitParts * E;
    z.part_bytes = sizeof(float) * z.S * (size_t)T * E_pad;
    z.xn2_bytes = sizeof(float) * z.S * (size_t)T;
    z.cnt_bytes = sizeof(int32_t) * E;
    z.list_bytes = sizeof(int32_t) * (size_t)E * T;
    z.stat_bytes = 16;
    return z;
}

cudaError_t launch_router_screen(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                 const RouterScreenBufs& rb, float* logits, int32_t* ids, float* w, int* status,
                                 cudaStream_t st, bool pdl, int32_t* counts) {
    const int S = router_screen_splits(T, d, E);
    if (!S || ((uintptr_t)x & 15) || ((uintptr_t)W_r & 15)) return cudaErrorNotSupported;
    const int E_pad = (E + 127) / 128 * 128, KB = d / 64;
    ScreenArgs a;
    cudaError_t err = x_tensor_map(&a.tmap_x, x, T, d);
    if (err != cudaSuccess) return err;
    // 1. split
    {
        void* args[] = {&W_r, &E, &d, (void*)&rb.bhi, (void*)&rb.blo, (void*)&rb.wn2, (void*)&rb.cnt, &counts};
        err = launch_kernel((const void*)router_split_kernel, dim3(E_pad, kSplitParts), dim3(256), 0, st, pdl, args);
        if (err != cudaSuccess) return err;
    }
    // 2. screen
    a.bhi = rb.bhi;
    a.blo = rb.blo;
    a.part = rb.part;
    a.xn2 = rb.xn2;
    a.wn2 = rb.wn2;
    a.b = b;
    a.stat = rb.stat;
    a.E = E;
    a.T = T;
    a.E_pad = E_pad;
    a.KB = KB;
    a.kb_per = KB / S;
    a.status = status;
    {
        void* args[] = {&a};
        err = launch_kernel((const void*)router_screen_kernel, dim3((T + 127) / 128, E_pad / 128, S),
                            dim3(kScrThreads), kScrSmem, st, true, args);
        if (err != cudaSuccess) return err;
    }
    // 3. candidates: the relative bound factor of the bound described at the top of this file
    {
        const double steps = 4.0 * ((a.kb_per + kScrAcc - 1) / kScrAcc);  // MMAs into one accumulator
        const double tc = steps * 0x1p-17 * (1.0 + steps * 0x1p-17);
        const double sums = (double)(2 * kScrAcc * S + 2) * 0x1p-24;
        const double exact = (double)(d / 32 + 6) * 0x1p-24;
        // (1 + 2^-8)^2 covers |hi| + |lo| against |w|; 1.05 covers the products of small terms dropped
        float C = (float)(1.05 * ((tc + sums) * (1.0 + 0x1p-7) + 0x1p-16 + exact));
        float tiny = (float)(std::sqrt((double)d) * 0x1p-124);
        const void* f = E_pad <= 128   ? (const void*)router_cand_kernel<4>
                        : E_pad <= 256 ? (const void*)router_cand_kernel<8>
                        : E_pad <= 512 ? (const void*)router_cand_kernel<16>
                                       : (const void*)router_cand_kernel<32>;
        const int per_cta = E_pad <= 128 ? cand_tokens<4>() : cand_tokens<8>();
        void* args[] = {(void*)&rb.part, (void*)&rb.xn2, (void*)&S, &T, &d, &E, (void*)&E_pad, &k, &b,
                        (void*)&rb.stat, &C, &tiny, &logits, (void*)&rb.cnt, (void*)&rb.list};
        err = launch_kernel(f, dim3((T + per_cta - 1) / per_cta), dim3(512), 0, st, true, args);
        if (err != cudaSuccess) return err;
    }
    // 4. exact logits of the candidates
    {
        const size_t smem = (size_t)d * 4 + (size_t)(E + 1) * 4;
        void* args[] = {&x, &W_r, &b, &T, &d, &E, (void*)&rb.cnt, (void*)&rb.list, &logits};
        err = launch_kernel((const void*)router_exact_kernel, dim3(2 * sm_count()), dim3(kXThreads), smem, st, true,
                            args);
        if (err != cudaSuccess) return err;
    }
    // 5. top-k + softmax
    return launch_topk(logits, T, E, k, ids, w, st, true, counts);
}

}  // namespace moe
