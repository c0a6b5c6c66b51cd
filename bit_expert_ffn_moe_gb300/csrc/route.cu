// route.cu -- router logits, top-k + softmax, and the permutation by expert.
//
// Router: Muse Spark Open explainer, section 8 -- one FP32 matrix product scores every expert,
// the best k are kept as a set, no shared expert.  Weights: section 9 -- the chosen experts'
// outputs are weighted by renormalised router scores (the printed example sums to 1).
// Permutation: section 12 -- pairs are gathered per expert so each expert runs one batch.
//
// Fixed fp32 reduction order of a logit (so that routing is reproducible bit for bit): 32
// partial sums; partial c accumulates with fma, from +0, the elements i with (i/4) % 32 == c in
// increasing i; then an xor butterfly p_c += p_{c^m} for m = 16, 8, 4, 2, 1; then + b[e].
// Lane c of a warp owns partial c.
#include <float.h>

#include "route_common.cuh"

namespace moe {

// ------------------------------------------------------------------ decode route (small T)
// Grid: one CTA per expert.  W_r[e] and x (T <= 8 rows) are staged in shared memory with
// cp.async in kRouteChunks commit groups, so the dot products of chunk c overlap the copies of
// the later chunks; warps compute the T logits of expert e.  The last CTA to finish (atomic
// ticket) runs top-k for every token and the whole permutation, so a decode step needs one launch.
constexpr int kRouteDecodeThreads = 128;
constexpr int kRouteDecodeMaxT = 8;
__global__ void __launch_bounds__(kRouteDecodeThreads)
route_decode_kernel(const uint16_t* __restrict__ x, const float* __restrict__ W_r, const float* __restrict__ b,
                    int T, int d, int E, int k, float* logits, int32_t* ids, float* w, int32_t* counts,
                    int32_t* offsets, int32_t* perm_token, int32_t* inv_pos, float* row_w, PlanView plan,
                    Ctrl* ctrl) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* Ws = reinterpret_cast<float*>(smem);                      // [d]
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + sizeof(float) * d);  // [T][d]
    __shared__ int s_last;
    __shared__ int s_cnt[kMaxE];
    __shared__ int s_off[kMaxE + 1];
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // the router weights do not depend on the preceding kernel: their copies start before its wait,
    // the token rows after it
    route_stage_w(W_r, e, d, Ws);
    pdl_wait();
    // the next kernel may start now: what it reads before its own dependency wait (x) is ready
    pdl_launch_dependents();
    route_stage_x(x, T, d, xs);
    for (int i = tid; i < E; i += blockDim.x) s_cnt[i] = 0;

    const float bias = b ? b[e] : 0.f;
    // warp w: tokens w and w + 4 (T <= 8)
    const float2 acc = route_dot_staged(Ws, xs + (size_t)(warp < T ? warp : 0) * d,
                                        warp + 4 < T ? xs + (size_t)(warp + 4) * d : nullptr, d, warp < T);
    if (warp < T && lane == 0) logits[(size_t)warp * E + e] = acc.x + bias;
    if (warp + 4 < T && lane == 0) logits[(size_t)(warp + 4) * E + e] = acc.y + bias;

    // ---- last CTA: top-k + permutation
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        unsigned ticket = atomicAdd(&ctrl->route_ticket, 1u);
        s_last = (ticket == (unsigned)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid == 0) ctrl->route_ticket = 0;  // ready for the next call on this workspace

    __shared__ int32_t s_ids[kRouteDecodeMaxT * kMaxK];
    __shared__ float s_w[kRouteDecodeMaxT * kMaxK];
    for (int t = warp; t < T; t += blockDim.x / 32)  // other CTAs' logits, read from L2
        topk_softmax_warp(logits + (size_t)t * E, E, k, s_ids + t * k, s_w + t * k, s_cnt);
    __syncthreads();
    const int P = T * k;
    for (int p = tid; p < P; p += blockDim.x) {
        ids[p] = s_ids[p];
        w[p] = s_w[p];
    }
    if (warp == 0) build_plan_warp(s_cnt, E, counts, offsets, plan, s_off);
    __syncthreads();
    for (int p = tid; p < P; p += blockDim.x) {
        const int t = p / k, ex = s_ids[p];
        int rank = 0;  // tokens before t that chose ex (each token picks an expert at most once)
        for (int t2 = 0; t2 < t; ++t2)
            for (int j = 0; j < k; ++j) rank += (s_ids[t2 * k + j] == ex);
        const int r = s_off[ex] + rank;
        perm_token[r] = t;
        inv_pos[p] = r;
        row_w[r] = s_w[p];
    }
    pdl_launch_dependents();
}

static size_t route_decode_smem(int T, int d) {
    return sizeof(float) * (size_t)d + sizeof(uint16_t) * (size_t)T * d;  // W_r[e] and x staging
}

bool route_decode_supported(int T, int d, int E, int k) {
    return T >= 1 && T <= kRouteDecodeMaxT && E <= kMaxE && k <= kMaxK && route_decode_smem(T, d) <= 200 * 1024;
}

cudaError_t launch_route_decode(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                float* logits, int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                                int32_t* perm_token, int32_t* inv_pos, float* row_w, PlanView plan, Ctrl* ctrl,
                                cudaStream_t st, bool pdl) {
    const size_t smem = route_decode_smem(T, d);
    void* args[] = {&x, &W_r, &b, &T, &d, &E, &k, &logits, &ids, &w, &counts, &offsets, &perm_token, &inv_pos,
                    &row_w, &plan, &ctrl};
    return launch_kernel((const void*)route_decode_kernel, dim3(E), dim3(kRouteDecodeThreads), smem, st, pdl, args);
}

// ------------------------------------------------------------------ tiled logits (any T)
// Pure fp32 FMA work in the fixed order (lanes are the 32 partial sums).  CTA tile: 32 tokens x
// 16 experts, 8 warps as 4 (tokens) x 2 (experts), warp tile 8 x 8 (64 accumulators per lane).
// K is streamed through a 3-stage cp.async ring of 256-element chunks (64 groups of 4; lane c
// takes groups c and c + 32 of a chunk, i.e. its elements in increasing order).  1024 CTAs of 256
// threads for 4096 tokens x 128 experts: two resident per SM, about 7 per SM in all, so the last
// wave is nearly full.
constexpr int kLT = 32, kLE = 16, kLKC = 256, kLStages = 3, kLThreads = 256;
constexpr int kLStageBytes = kLT * kLKC * 2 + kLE * kLKC * 4;  // bf16 x chunk + fp32 W_r chunk

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(valid ? 16 : 0) : "memory");
}

__global__ void __launch_bounds__(kLThreads, 2)
route_logits_tiled_kernel(const uint16_t* __restrict__ x, const float* __restrict__ W_r, const float* __restrict__ b,
                          int T, int d, int E, float* __restrict__ logits, int32_t* __restrict__ zero_counts) {
    extern __shared__ __align__(16) unsigned char lsm[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * kLT, e0 = blockIdx.y * kLE;
    const int wt = (warp >> 1) * 8, we = (warp & 1) * 8;
    auto xs = [&](int st) { return reinterpret_cast<uint16_t*>(lsm + (size_t)st * kLStageBytes); };
    auto ws = [&](int st) { return reinterpret_cast<float*>(lsm + (size_t)st * kLStageBytes + kLT * kLKC * 2); };
    const int nchunks = (d + kLKC - 1) / kLKC;
    // stage chunk kc (16-byte pieces: x 32 rows x 32, W_r 16 rows x 64; zero-filled past T, E, d)
    auto load_chunk = [&](int kc) {
        const int st = kc % kLStages, k0 = kc * kLKC;
        uint16_t* xd = xs(st);
        float* wd = ws(st);
        for (int i = tid; i < kLT * (kLKC / 8); i += kLThreads) {
            const int r = i / (kLKC / 8), c = i % (kLKC / 8);
            const bool ok = t0 + r < T && k0 + 8 * c < d;
            cp_async16(xd + r * kLKC + 8 * c, ok ? x + (size_t)(t0 + r) * d + k0 + 8 * c : x, ok);
        }
        for (int i = tid; i < kLE * (kLKC / 4); i += kLThreads) {
            const int r = i / (kLKC / 4), c = i % (kLKC / 4);
            const bool ok = e0 + r < E && k0 + 4 * c < d;
            cp_async16(wd + r * kLKC + 4 * c, ok ? W_r + (size_t)(e0 + r) * d + k0 + 4 * c : W_r, ok);
        }
    };
    // acc[p][c] = partial sums of tokens wt + 2p (x) and wt + 2p + 1 (y) against expert we + c;
    // each is the same sequential fma chain as a scalar accumulator, two per instruction.
    float2 acc[4][8];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[p][c] = make_float2(0.f, 0.f);

    pdl_wait();
    if (zero_counts && blockIdx.x == 0 && blockIdx.y == 0)  // the pick counts the top-k adds to next
        for (int e = tid; e < E; e += kLThreads) zero_counts[e] = 0;
#pragma unroll
    for (int kc = 0; kc < kLStages - 1; ++kc) {
        if (kc < nchunks) load_chunk(kc);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int kc = 0; kc < nchunks; ++kc) {
        asm volatile("cp.async.wait_group %0;" ::"n"(kLStages - 2) : "memory");
        __syncthreads();  // chunk kc is in; every warp is done with the stage refilled below
        if (kc + kLStages - 1 < nchunks) load_chunk(kc + kLStages - 1);
        asm volatile("cp.async.commit_group;" ::: "memory");
        const uint16_t* xc = xs(kc % kLStages);
        const float* wc = ws(kc % kLStages);
        const int k0 = kc * kLKC;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi) {
            if (k0 + 128 * gi >= d) break;  // d % 128 == 0: a group of 32 lanes is all in or all out
            const int g = lane + 32 * gi;
            float2 xv[4][4];  // [token pair][element of the group]
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const uint2 u0 = *reinterpret_cast<const uint2*>(xc + (wt + 2 * p) * kLKC + 4 * g);
                const uint2 u1 = *reinterpret_cast<const uint2*>(xc + (wt + 2 * p + 1) * kLKC + 4 * g);
                xv[p][0] = make_float2(bf16_bits_to_f32(u0.x & 0xFFFF), bf16_bits_to_f32(u1.x & 0xFFFF));
                xv[p][1] = make_float2(bf16_bits_to_f32(u0.x >> 16), bf16_bits_to_f32(u1.x >> 16));
                xv[p][2] = make_float2(bf16_bits_to_f32(u0.y & 0xFFFF), bf16_bits_to_f32(u1.y & 0xFFFF));
                xv[p][3] = make_float2(bf16_bits_to_f32(u0.y >> 16), bf16_bits_to_f32(u1.y >> 16));
            }
            float wv[8][4];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const float4 f = *reinterpret_cast<const float4*>(wc + (we + c) * kLKC + 4 * g);
                wv[c][0] = f.x;
                wv[c][1] = f.y;
                wv[c][2] = f.z;
                wv[c][3] = f.w;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float2 wq = make_float2(wv[c][q], wv[c][q]);
#pragma unroll
                    for (int p = 0; p < 4; ++p) acc[p][c] = fma2(xv[p][q], wq, acc[p][c]);
                }
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            float s = warp_butterfly_sum((a & 1) ? acc[a >> 1][c].y : acc[a >> 1][c].x);
            int t = t0 + wt + a, e = e0 + we + c;
            if (lane == ((a * 8 + c) & 31) && t < T && e < E) logits[(size_t)t * E + e] = s + (b ? b[e] : 0.f);
        }
    pdl_launch_dependents();
}

// One warp per token; NV = keys per lane (E <= 32 NV), one instantiation per width so that each
// holds only the registers its own width needs.  counts != nullptr: the picks are also counted per
// expert (a shared-memory histogram per CTA, then one global add per expert and CTA); the caller
// has zeroed counts.
template <int NV>
__global__ void topk_kernel(const float* __restrict__ logits, int T, int E, int k, int32_t* ids, float* w,
                            int32_t* counts) {
    __shared__ int hist[kMaxE];
    pdl_wait();
    if (counts) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
        __syncthreads();
    }
    const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (t < T)
        topk_softmax_regs<NV, false>(logits + (size_t)t * E, E, k, ids + (size_t)t * k, w + (size_t)t * k,
                                     counts ? hist : nullptr);
    if (counts) {
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            if (hist[e] != 0) atomicAdd(counts + e, hist[e]);
    }
    pdl_launch_dependents();
}

cudaError_t launch_route_logits(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E,
                                float* logits, cudaStream_t st, bool pdl, int32_t* zero_counts) {
    if (T == 0) return cudaSuccess;
    void* args[] = {&x, &W_r, &b, &T, &d, &E, &logits, &zero_counts};
    dim3 grid((T + kLT - 1) / kLT, (E + kLE - 1) / kLE);
    return launch_kernel((const void*)route_logits_tiled_kernel, grid, dim3(kLThreads),
                         (size_t)kLStages * kLStageBytes, st, pdl, args);
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* w, cudaStream_t st, bool pdl,
                        int32_t* counts) {
    if (T == 0) return cudaSuccess;
    void* args[] = {&logits, &T, &E, &k, &ids, &w, &counts};
    const int nv = (E + 31) / 32;
    const void* f = nv <= 1   ? (const void*)topk_kernel<1>
                    : nv <= 2 ? (const void*)topk_kernel<2>
                    : nv <= 4 ? (const void*)topk_kernel<4>
                    : nv <= 8 ? (const void*)topk_kernel<8>
                    : nv <= 16 ? (const void*)topk_kernel<16>
                               : (const void*)topk_kernel<32>;
    return launch_kernel(f, dim3((T + 7) / 8), dim3(256), 0, st, pdl, args);
}

// ------------------------------------------------------------------ permutation (any T)

// Histogram of the chosen experts: each CTA counts its share of the pairs in shared memory, then
// adds its nonzero counts to the global ones (few global atomics even when the load is skewed).
__global__ void count_kernel(const int32_t* __restrict__ ids, int P, int E, int32_t* counts) {
    __shared__ int hist[kMaxE];
    pdl_wait();
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < P; p += gridDim.x * blockDim.x) {
        const int e = ids[p];
        if ((unsigned)e < (unsigned)E) atomicAdd(&hist[e], 1);  // an id outside [0, E) is not counted
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (hist[e] != 0) atomicAdd(&counts[e], hist[e]);
}

__global__ void plan_kernel(int E, int32_t* counts_out, int32_t* offsets, PlanView plan) {
    pdl_wait();
    if (threadIdx.x < 32) build_plan_warp(plan.counts, E, counts_out, offsets, plan);
}

// One expert (0) holding rows 0..T-1 in order: the plan a dense product runs with.
__global__ void dense_plan_kernel(int T, PlanView plan, int32_t* offsets, int32_t* perm_token) {
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int tiles = (T + kTokTile - 1) / kTokTile;
        const int used = (T + kPadRows - 1) / kPadRows * kPadRows;  // the expert's padded rows
        plan.counts[0] = T;
        plan.pad_offsets[0] = 0;
        plan.pad_offsets[1] = used;
        plan.ttile_prefix[0] = 0;
        plan.ttile_prefix[1] = tiles;
        plan.active[0] = 0;
        plan.scalars[0] = T > 0 ? 1 : 0;
        plan.scalars[1] = tiles;
        plan.scalars[2] = used;
        offsets[0] = 0;
        offsets[1] = T;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T; i += gridDim.x * blockDim.x) perm_token[i] = i;
    pdl_launch_dependents();
}

// One CTA per expert: a stable block-wide compaction over the tokens that chose it, 2048 tokens
// per pass (each thread's ids of two tokens loaded at once, as 16-byte vectors when k % 4 == 0),
// compacted in token order: the first 1024 tokens of the pass, then the next 1024.  Per 1024
// tokens: the warps' counts (ballots) to shared memory, one barrier, warp 0 scans the 32 counts, a
// second barrier.  (The warp_tot writes for the next 1024 tokens come after every thread passed the
// second barrier, by which point warp 0 has read the counts; warp 0's next warp_pre writes come
// after the next first barrier, by which point every thread has read the previous warp_pre.)
__device__ __forceinline__ void warp_exclusive_scan(const int* warp_tot, int* warp_pre) {
    const int lane = threadIdx.x & 31;
    const int v = warp_tot[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    warp_pre[lane] = incl - v;
    if (lane == 31) warp_pre[32] = incl;
}

__device__ __forceinline__ int find_slot(const int32_t* __restrict__ ids, int t, int T, int k, int e) {
    int j_found = -1;
    if (t < T) {
        if ((k & 3) == 0) {
            const int4* p = reinterpret_cast<const int4*>(ids + (size_t)t * k);
            for (int q = 0; q < k / 4; ++q) {
                const int4 v = __ldg(p + q);
                if (v.x == e) j_found = 4 * q;
                if (v.y == e) j_found = 4 * q + 1;
                if (v.z == e) j_found = 4 * q + 2;
                if (v.w == e) j_found = 4 * q + 3;
            }
        } else {
            for (int j = 0; j < k; ++j)
                if (__ldg(ids + (size_t)t * k + j) == e) j_found = j;
        }
    }
    return j_found;
}

__global__ void __launch_bounds__(1024)
scatter_kernel(const int32_t* __restrict__ ids, int T, int k, const int32_t* __restrict__ offsets, PlanView plan,
               int32_t* perm_token, int32_t* inv_pos, const float* __restrict__ w, float* row_w) {
    __shared__ int warp_tot[32], warp_pre[33];
    pdl_wait();
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (plan.counts[e] == 0) return;
    int running = offsets[e];
    for (int t0 = 0; t0 < T; t0 += 2048) {
        const int ta = t0 + tid, tb = t0 + 1024 + tid;
        const int ja = find_slot(ids, ta, T, k, e), jb = find_slot(ids, tb, T, k, e);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = h ? tb : ta, j_found = h ? jb : ja;
            const unsigned bal = __ballot_sync(0xffffffffu, j_found >= 0);
            const int before = __popc(bal & ((1u << lane) - 1u));
            if (lane == 0) warp_tot[warp] = __popc(bal);
            __syncthreads();
            if (warp == 0) warp_exclusive_scan(warp_tot, warp_pre);
            __syncthreads();
            if (j_found >= 0) {
                const int r = running + warp_pre[warp] + before;
                perm_token[r] = t;
                inv_pos[(size_t)t * k + j_found] = r;
                if (row_w) row_w[r] = w[(size_t)t * k + j_found];
            }
            running += warp_pre[32];
        }
    }
}

// The permutation when the top-k has already counted the picks into plan.counts: CTA e takes its
// expert's offset from the counts of the experts before it, CTA 0 also writes the whole plan
// (counts, offsets, padded offsets, tile prefix, active list), and every CTA scatters as above.
__global__ void __launch_bounds__(1024)
scatter_plan_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int32_t* counts_out, int32_t* offsets,
                    PlanView plan, int32_t* perm_token, int32_t* inv_pos, const float* __restrict__ w,
                    float* row_w) {
    __shared__ int warp_tot[32], warp_pre[33];
    __shared__ int s_base;
    pdl_wait();
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (e == 0 && warp == 0) build_plan_warp(plan.counts, E, counts_out, offsets, plan);
    int v = tid < e ? __ldcg(plan.counts + tid) : 0;  // E <= 1024 = blockDim.x
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) warp_tot[warp] = v;
    __syncthreads();
    if (tid == 0) {
        int b = 0;
        for (int q = 0; q < 32; ++q) b += warp_tot[q];
        s_base = b;
    }
    __syncthreads();
    if (__ldcg(plan.counts + e) == 0) return;  // block-uniform
    int running = s_base;
    for (int t0 = 0; t0 < T; t0 += 2048) {
        const int ta = t0 + tid, tb = t0 + 1024 + tid;
        const int ja = find_slot(ids, ta, T, k, e), jb = find_slot(ids, tb, T, k, e);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = h ? tb : ta, j_found = h ? jb : ja;
            const unsigned bal = __ballot_sync(0xffffffffu, j_found >= 0);
            const int before = __popc(bal & ((1u << lane) - 1u));
            if (lane == 0) warp_tot[warp] = __popc(bal);
            __syncthreads();
            if (warp == 0) warp_exclusive_scan(warp_tot, warp_pre);
            __syncthreads();
            if (j_found >= 0) {
                const int r = running + warp_pre[warp] + before;
                perm_token[r] = t;
                inv_pos[(size_t)t * k + j_found] = r;
                if (row_w) row_w[r] = w[(size_t)t * k + j_found];
            }
            running += warp_pre[32];
        }
    }
}

cudaError_t launch_permute_counted(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                                   int32_t* perm_token, int32_t* inv_pos, PlanView plan, cudaStream_t st, bool pdl,
                                   const float* w, float* row_w) {
    if (w == nullptr) row_w = nullptr;
    void* args[] = {&ids, &T, &k, &E, &counts, &offsets, &plan, &perm_token, &inv_pos, &w, &row_w};
    return launch_kernel((const void*)scatter_plan_kernel, dim3(E), dim3(1024), 0, st, pdl, args);
}

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_pos, PlanView plan, cudaStream_t st, bool pdl,
                           const float* w, float* row_w) {
    cudaError_t err = cudaMemsetAsync(plan.counts, 0, sizeof(int32_t) * (size_t)E, st);
    if (err != cudaSuccess) return err;
    int P = T * k;
    if (P > 0) {
        int blocks = (P + 1023) / 1024;  // about 1024 pairs per CTA
        if (blocks > 256) blocks = 256;
        void* a1[] = {&ids, &P, &E, &plan.counts};
        err = launch_kernel((const void*)count_kernel, dim3(blocks), dim3(256), 0, st, false, a1);
        if (err != cudaSuccess) return err;
    }
    void* a2[] = {&E, &counts, &offsets, &plan};
    err = launch_kernel((const void*)plan_kernel, dim3(1), dim3(32), 0, st, pdl, a2);
    if (err != cudaSuccess) return err;
    if (P == 0) return cudaSuccess;
    if (w == nullptr) row_w = nullptr;
    void* a3[] = {&ids, &T, &k, &offsets, &plan, &perm_token, &inv_pos, &w, &row_w};
    return launch_kernel((const void*)scatter_kernel, dim3(E), dim3(1024), 0, st, pdl, a3);
}

cudaError_t launch_dense_plan(int T, PlanView plan, int32_t* offsets, int32_t* perm_token, cudaStream_t st,
                              bool pdl) {
    int blocks = (T + 255) / 256;
    if (blocks < 1) blocks = 1;
    if (blocks > 152) blocks = 152;
    void* args[] = {&T, &plan, &offsets, &perm_token};
    return launch_kernel((const void*)dense_plan_kernel, dim3(blocks), dim3(256), 0, st, pdl, args);
}

// ------------------------------------------------------------------ MX activation operand
// Quantise each token row once (one thread per 32-element block), then gather the rows into
// padded expert-grouped order with the scales in the tensor-core layout.  FP8: MXFP8 (32 E4M3
// bytes per block, tiles of 128 values per 128-byte line), else MXFP4 (16 bytes of E2M1 codes per
// block, 256 values per line).

template <bool FP8>
__global__ void act_quant_kernel(const uint16_t* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ xq,
                                 uint8_t* __restrict__ xs) {
    pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblocks; blk += stride) {
        const uint4* src = reinterpret_cast<const uint4*>(x + blk * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 u = src[i];
            uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                v[8 * i + 2 * m] = bf16_bits_to_f32(ww[m] & 0xFFFF);
                v[8 * i + 2 * m + 1] = bf16_bits_to_f32(ww[m] >> 16);
            }
        }
        if (FP8) {
            uint4 c[2];
            const uint32_t sb = mx8_block_encode(v, c);
            reinterpret_cast<uint4*>(xq)[2 * blk] = c[0];
            reinterpret_cast<uint4*>(xq)[2 * blk + 1] = c[1];
            xs[blk] = (uint8_t)sb;
        } else {
            uint4 codes;
            const uint32_t sb = mx_block_encode(v, codes);
            reinterpret_cast<uint4*>(xq)[blk] = codes;
            xs[blk] = (uint8_t)sb;
        }
    }
}

// One warp per padded row: the row's expert comes from a binary search over the padded offsets
// cached in shared memory; lanes copy consecutive 16-byte chunks of the token's quantised row
// into the tensor-core code tiles (8 lanes fill one 128-byte line), then its scale bytes four
// at a time.
template <bool FP8>
__global__ void __launch_bounds__(256)
act_gather_kernel(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xs, int d, int E, int64_t pad_rows,
                  const int32_t* __restrict__ offsets, const int32_t* __restrict__ perm_token, PlanView plan,
                  uint8_t* __restrict__ xa, uint8_t* __restrict__ xa_s, int zero_pad) {
    extern __shared__ int32_t s_pad[];  // [E+1]
    pdl_wait();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) s_pad[i] = plan.pad_offsets[i];
    __syncthreads();
    const int nb = d / 32, lane = threadIdx.x & 31;
    const int nc = FP8 ? d / 16 : d / 32;  // 16-byte chunks of a quantised row
    const int64_t used = plan.scalars[2];
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < used; r += nwarps) {
        int lo = 0, hi = E;  // expert of padded row r: last e with s_pad[e] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_pad[mid] <= r) lo = mid; else hi = mid;
        }
        const int64_t local = r - s_pad[lo];
        const bool real = local < plan.counts[lo];
        if (!real && !zero_pad) continue;  // the caller leaves padding rows as they are
        const int t = real ? perm_token[offsets[lo] + local] : 0;
        const uint4* src = reinterpret_cast<const uint4*>(xq + (size_t)t * (size_t)nc * 16);
        constexpr int kGB = 8;  // a lane's loads of up to 8 chunks are issued before its stores
        for (int c0 = lane; c0 < nc; c0 += 32 * kGB) {
            uint4 v[kGB];
#pragma unroll
            for (int u = 0; u < kGB; ++u) {
                const int c = c0 + 32 * u;
                v[u] = real && c < nc ? src[c] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kGB; ++u) {
                const int c = c0 + 32 * u;
                if (c < nc)
                    *reinterpret_cast<uint4*>(xa + (FP8 ? mma8_tile_offset(r, c, d) : mma_tile_offset(r, c, d))) = v[u];
            }
        }
        // scales: blocks 4q .. 4q+3 of a row are 4 consecutive bytes of one scale atom (and of xs)
        const uint32_t* srcs = reinterpret_cast<const uint32_t*>(xs + (size_t)t * nb);
        for (int q = lane; q < nb / 4; q += 32)
            *reinterpret_cast<uint32_t*>(xa_s + mma_scale_offset(r, 4 * q, d)) = real ? srcs[q] : 0u;
    }
    (void)pad_rows;
}

// The layer call's operand in one pass, once the permutation is known.  Work item = (token t, a
// segment of 64 of its 32-element blocks); lane j < k first finds the padded row of pick j (its
// expert's padded start + its row within the expert), then lane l loads the blocks
// seg + l and seg + 32 + l of the token row (both before any store), encodes them (as
// act_quant_kernel) and writes each block's codes to all k rows; the scale bytes of four
// consecutive blocks (four neighbouring lanes) go out as one 4-byte store per row.  Padding rows
// are left as they are.  ids == nullptr: the identity of a dense map (k = 1, token t to row t).
template <bool FP8>
__global__ void __launch_bounds__(256)
act_quant_scatter_kernel(const uint16_t* __restrict__ x, int T, int d, int k, const int32_t* __restrict__ ids,
                         const int32_t* __restrict__ inv_pos, const int32_t* __restrict__ offsets, PlanView plan,
                         uint8_t* __restrict__ xa, uint8_t* __restrict__ xa_s) {
    pdl_wait();
    const int lane = threadIdx.x & 31, nb = d / 32, nseg = (nb + 63) / 64;
    const int64_t items = (int64_t)T * nseg;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t it = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); it < items; it += nwarps) {
        const int64_t t = it / nseg;
        const int b0 = (int)(it % nseg) * 64;
        int my_row = 0;
        if (lane < k) {
            if (ids) {
                const int e = __ldg(ids + t * k + lane);
                my_row = __ldg(plan.pad_offsets + e) + (__ldg(inv_pos + t * k + lane) - __ldg(offsets + e));
            } else {
                my_row = (int)t;
            }
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + t * d);  // 4 chunks of 16 bytes per block
        uint4 u[2][4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int blk = b0 + 32 * h + lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) u[h][i] = blk < nb ? __ldg(src + (size_t)blk * 4 + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // warp-uniform: the shuffles below need every lane
            const int blk = b0 + 32 * h + lane;
            float v[32];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t ww[4] = {u[h][i].x, u[h][i].y, u[h][i].z, u[h][i].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    v[8 * i + 2 * m] = bf16_bits_to_f32(ww[m] & 0xFFFF);
                    v[8 * i + 2 * m + 1] = bf16_bits_to_f32(ww[m] >> 16);
                }
            }
            uint4 c[2];
            const uint32_t sb = FP8 ? mx8_block_encode(v, c) : mx_block_encode(v, c[0]);
            const int q0 = lane & ~3;
            const uint32_t s4 = (__shfl_sync(0xffffffffu, sb, q0) & 0xFF) |
                                ((__shfl_sync(0xffffffffu, sb, q0 + 1) & 0xFF) << 8) |
                                ((__shfl_sync(0xffffffffu, sb, q0 + 2) & 0xFF) << 16) |
                                ((__shfl_sync(0xffffffffu, sb, q0 + 3) & 0xFF) << 24);
            for (int j = 0; j < k; ++j) {
                const int64_t r = __shfl_sync(0xffffffffu, my_row, j);
                if (blk < nb) {
                    if (FP8) {
                        *reinterpret_cast<uint4*>(xa + mma8_tile_offset(r, 2 * blk, d)) = c[0];
                        *reinterpret_cast<uint4*>(xa + mma8_tile_offset(r, 2 * blk + 1, d)) = c[1];
                    } else {
                        *reinterpret_cast<uint4*>(xa + mma_tile_offset(r, blk, d)) = c[0];
                    }
                    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(xa_s + mma_scale_offset(r, blk, d)) = s4;
                }
            }
        }
    }
}

cudaError_t launch_act_quant_scatter(const uint16_t* x, int T, int d, int k, const int32_t* ids,
                                     const int32_t* inv_pos, const int32_t* offsets, PlanView plan, uint8_t* xa,
                                     uint8_t* xa_s, bool fp8, cudaStream_t st, bool pdl) {
    if (T == 0) return cudaSuccess;
    const int64_t items = (int64_t)T * ((d / 32 + 63) / 64);
    int64_t blocks = (items + 7) / 8;  // 8 warps (work items) per CTA
    if (blocks > 152 * 8) blocks = 152 * 8;
    void* args[] = {&x, &T, &d, &k, &ids, &inv_pos, &offsets, &plan, &xa, &xa_s};
    const void* f = fp8 ? (const void*)act_quant_scatter_kernel<true> : (const void*)act_quant_scatter_kernel<false>;
    return launch_kernel(f, dim3((unsigned)blocks), dim3(256), 0, st, pdl, args);
}

cudaError_t launch_act_quant(const uint16_t* x, int T, int d, uint8_t* xq, uint8_t* xs, bool fp8, cudaStream_t st,
                             bool pdl) {
    int64_t nb = (int64_t)T * (d / 32);
    if (nb <= 0) return cudaSuccess;
    int64_t blocks = (nb + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    void* a1[] = {&x, &nb, &xq, &xs};
    const void* f = fp8 ? (const void*)act_quant_kernel<true> : (const void*)act_quant_kernel<false>;
    return launch_kernel(f, dim3((unsigned)blocks), dim3(256), 0, st, pdl, a1);
}

cudaError_t launch_act_gather(const uint8_t* xq, const uint8_t* xs, int d, int E, const int32_t* offsets,
                              const int32_t* perm_token, PlanView plan, int64_t pad_rows, uint8_t* xa, uint8_t* xa_s,
                              bool fp8, cudaStream_t st, bool pdl, bool zero_pad) {
    if (pad_rows == 0) return cudaSuccess;
    int64_t blocks = (pad_rows + 7) / 8;  // 8 warps (rows) per CTA
    if (blocks > 152 * 8) blocks = 152 * 8;
    int zp = zero_pad ? 1 : 0;
    void* a2[] = {&xq, &xs, &d, &E, &pad_rows, &offsets, &perm_token, &plan, &xa, &xa_s, &zp};
    const void* g = fp8 ? (const void*)act_gather_kernel<true> : (const void*)act_gather_kernel<false>;
    return launch_kernel(g, dim3((unsigned)blocks), dim3(256), sizeof(int32_t) * (size_t)(E + 1), st, pdl, a2);
}

cudaError_t launch_act_quant_gather(const uint16_t* x, int T, int d, int E, int k, const int32_t* offsets,
                                    const int32_t* perm_token, PlanView plan, int64_t pad_rows, uint8_t* xq,
                                    uint8_t* xs, uint8_t* xa, uint8_t* xa_s, bool fp8, cudaStream_t st, bool pdl) {
    (void)k;
    cudaError_t err = launch_act_quant(x, T, d, xq, xs, fp8, st, pdl);
    if (err != cudaSuccess) return err;
    return launch_act_gather(xq, xs, d, E, offsets, perm_token, plan, pad_rows, xa, xa_s, fp8, st, pdl);
}

}  // namespace moe
