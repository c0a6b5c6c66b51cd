// route_common.cuh -- device helpers of the router shared by the router kernels (route.cu) and the
// decode kernel that routes its own tokens (decode_mma.cu): the fixed-order fp32 dot products of
// the logits, and the warp top-k + softmax.
//
// Fixed fp32 reduction order of a logit (so that routing is reproducible bit for bit): 32
// partial sums; partial c accumulates with fma, from +0, the elements i with (i/4) % 32 == c in
// increasing i; then an xor butterfly p_c += p_{c^m} for m = 16, 8, 4, 2, 1; then + b[e].
// Lane c of a warp owns partial c.
#pragma once

#include "common.cuh"

namespace moe {

// Two independent fp32 fmas (round to nearest each) on packed pairs: (a.x*b.x + c.x, a.y*b.y + c.y).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float warp_butterfly_sum(float p) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) p = p + __shfl_xor_sync(0xffffffffu, p, m);
    return p;
}

// Order-preserving key of a logit: a larger float gives a larger unsigned key, +0 and -0 give the
// same key, and no finite value or infinity maps to 0, which marks "no candidate".
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp selects the top-k of logits[0..E) (largest first; ties -> lower id), sorts the set by
// ascending id and writes ids[0..k) and the softmax weights w[0..k); when cnt is given it also
// counts each pick there (shared-memory histogram).  Lane l holds the keys of ids l + 32 i in
// registers; a round takes the lane maxima (strict > over increasing i keeps the lower id), the
// warp maximum of the keys and then the least id among the lanes holding it.
template <int NV, bool SHARED>
__device__ __forceinline__ void topk_softmax_regs(const float* logits, int E, int k, int32_t* ids, float* w, int* cnt) {
    const int lane = threadIdx.x & 31;
    uint32_t key[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        // global logits come from other CTAs: read through L2
        const float v = lane + 32 * i < E ? (SHARED ? logits[lane + 32 * i] : __ldcg(logits + lane + 32 * i)) : 0.f;
        key[i] = lane + 32 * i < E ? logit_key(v) : 0u;
    }
    int my_id = 0x7fffffff;
    uint32_t my_key = 0, taken = 0;  // bit i: id lane + 32 i already chosen
    for (int r = 0; r < k; ++r) {
        uint32_t lb = 0;
        int li = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (!((taken >> i) & 1u) && key[i] > lb) {
                lb = key[i];
                li = i;
            }
        const uint32_t wb = __reduce_max_sync(0xffffffffu, lb);
        const int id = __reduce_min_sync(0xffffffffu, (lb == wb) ? lane + 32 * li : 0x7fffffff);
        if ((id & 31) == lane) taken |= 1u << (id >> 5);
        if (lane == r) {
            my_id = id;
            my_key = wb;
        }
    }
    // ascending-id order of the chosen set
    int rank = 0;
    for (int s = 0; s < k; ++s) {
        int o = __shfl_sync(0xffffffffu, my_id, s);
        if (lane < k && o < my_id) ++rank;
    }
    const float my_logit = key_logit(my_key);
    const float m = __shfl_sync(0xffffffffu, my_logit, 0);  // the first pick is the largest logit
    float ex = lane < k ? expf(my_logit - m) : 0.f;
    float sum = warp_butterfly_sum(ex);
    if (lane < k) {
        ids[rank] = my_id;
        w[rank] = ex / sum;
        if (cnt) atomicAdd(cnt + my_id, 1);
    }
}

// logits in global memory (SHARED = false) or in this block's shared memory (SHARED = true)
template <bool SHARED = false>
__device__ __forceinline__ void topk_softmax_warp(const float* logits, int E, int k, int32_t* ids, float* w, int* cnt = nullptr) {
    const int nv = (E + 31) / 32;
    if (nv <= 1) topk_softmax_regs<1, SHARED>(logits, E, k, ids, w, cnt);
    else if (nv <= 2) topk_softmax_regs<2, SHARED>(logits, E, k, ids, w, cnt);
    else if (nv <= 4) topk_softmax_regs<4, SHARED>(logits, E, k, ids, w, cnt);
    else if (nv <= 8) topk_softmax_regs<8, SHARED>(logits, E, k, ids, w, cnt);
    else if (nv <= 16) topk_softmax_regs<16, SHARED>(logits, E, k, ids, w, cnt);
    else topk_softmax_regs<32, SHARED>(logits, E, k, ids, w, cnt);
}

// Warp 0 of a block: counts[E] -> offsets, padded offsets, token-tile prefix, active list
// (offsets also to shared memory when offsets_smem is given).
__device__ __forceinline__ void build_plan_warp(const int32_t* counts_in, int E, int32_t* counts_out, int32_t* offsets, PlanView plan,
                                int32_t* offsets_smem = nullptr) {
    const int lane = threadIdx.x & 31;
    const int chunk = (E + 31) / 32;
    const int lo = min(E, lane * chunk), hi = min(E, lo + chunk);
    int s_cnt = 0, s_pad = 0, s_tile = 0, s_act = 0;
    for (int e = lo; e < hi; ++e) {
        int c = counts_in[e];
        s_cnt += c;
        s_pad += (c + kPadRows - 1) / kPadRows * kPadRows;
        s_tile += (c + kTokTile - 1) / kTokTile;
        s_act += c > 0;
    }
    int x_cnt = s_cnt, x_pad = s_pad, x_tile = s_tile, x_act = s_act;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int a = __shfl_up_sync(0xffffffffu, x_cnt, o), b = __shfl_up_sync(0xffffffffu, x_pad, o);
        int c = __shfl_up_sync(0xffffffffu, x_tile, o), d = __shfl_up_sync(0xffffffffu, x_act, o);
        if (lane >= o) {
            x_cnt += a;
            x_pad += b;
            x_tile += c;
            x_act += d;
        }
    }
    int c_off = x_cnt - s_cnt, p_off = x_pad - s_pad, t_off = x_tile - s_tile, a_off = x_act - s_act;
    for (int e = lo; e < hi; ++e) {
        int c = counts_in[e];
        if (counts_out) counts_out[e] = c;
        plan.counts[e] = c;
        offsets[e] = c_off;
        if (offsets_smem) offsets_smem[e] = c_off;
        plan.pad_offsets[e] = p_off;
        plan.ttile_prefix[e] = t_off;
        if (c > 0) plan.active[a_off++] = e;
        c_off += c;
        p_off += (c + kPadRows - 1) / kPadRows * kPadRows;
        t_off += (c + kTokTile - 1) / kTokTile;
    }
    if (lane == 31) {
        offsets[E] = x_cnt;
        if (offsets_smem) offsets_smem[E] = x_cnt;
        plan.pad_offsets[E] = x_pad;
        plan.ttile_prefix[E] = x_tile;
        plan.scalars[0] = x_act;
        plan.scalars[1] = x_tile;
        plan.scalars[2] = x_pad;
    }
}

// Chunked staging of one expert's router row and the T token rows for the fixed-order dot
// products: kRouteChunks cp.async commit groups of W_r[e] (issued first: they do not depend on a
// preceding kernel), then kRouteChunks groups of x; chunk c holds the 4-element groups
// [c*Gc, (c+1)*Gc) of a row (clamped to d/4), Gc a multiple of 32 so that group g stays with lane
// g % 32.
constexpr int kRouteChunks = 4;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ int route_chunk_groups(int d) {
    const int ng = d / 4;
    return ((ng + kRouteChunks - 1) / kRouteChunks + 31) / 32 * 32;
}

// Issue the kRouteChunks commit groups of W_r[e] into Ws[d] (all threads of the block).
__device__ __forceinline__ void route_stage_w(const float* W_r, int e, int d, float* Ws) {
    const int ng = d / 4, Gc = route_chunk_groups(d);
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c) {
        const int lo = min(c * Gc, ng), hi = min(lo + Gc, ng);
        for (int g = lo + (int)threadIdx.x; g < hi; g += blockDim.x) cp_async16(Ws + 4 * g, W_r + (size_t)e * d + 4 * g);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
}

// Issue the kRouteChunks commit groups of the T token rows into xs[T][d] (all threads).
__device__ __forceinline__ void route_stage_x(const uint16_t* x, int T, int d, uint16_t* xs) {
    const int ng = d / 4, Gc = route_chunk_groups(d);
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c) {
        const int lo = min(c * Gc, ng), hi = min(lo + Gc, ng);
        const int n8 = (hi - lo) / 2;  // 8-element pieces of a token row in this chunk
        for (int i = (int)threadIdx.x; i < T * n8; i += blockDim.x) {
            const int t = i / n8, p8 = lo / 2 + i % n8;
            cp_async16(xs + (size_t)t * d + 8 * p8, x + (size_t)t * d + 8 * p8);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
}

// Wait for the staged chunks (W_r groups, then x groups, as issued above) one at a time and
// accumulate the fixed-order partial sums of the token rows xr0 (and xr1 when not null) against
// Ws.  Every thread of the block calls it (it holds the block barriers); `active` warps
// accumulate.  Returns the butterfly-combined sums (before the bias) in every lane.
__device__ __forceinline__ float2 route_dot_staged(const float* Ws, const uint16_t* xr0, const uint16_t* xr1, int d,
                                                   bool active) {
    const int ng = d / 4, Gc = route_chunk_groups(d), lane = threadIdx.x & 31;
    float acc = 0.f, acc2 = 0.f;
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c) {
        if (c == 0) cp_async_wait_group<kRouteChunks - 1>();
        else if (c == 1) cp_async_wait_group<kRouteChunks - 2>();
        else if (c == 2) cp_async_wait_group<kRouteChunks - 3>();
        else cp_async_wait_group<0>();
        __syncthreads();
        const int lo = min(c * Gc, ng), hi = min(lo + Gc, ng);
        if (active) {
            const int n = (hi - lo) / 32;  // groups of this lane in the chunk (hi - lo is a multiple of 32)
#pragma unroll 4
            for (int m = 0; m < n; ++m) {
                const int g = lo + lane + 32 * m;
                const float4 wv = *reinterpret_cast<const float4*>(Ws + 4 * g);
                const uint2 xv = *reinterpret_cast<const uint2*>(xr0 + 4 * g);
                acc = fmaf(bf16_bits_to_f32(xv.x & 0xFFFF), wv.x, acc);
                acc = fmaf(bf16_bits_to_f32(xv.x >> 16), wv.y, acc);
                acc = fmaf(bf16_bits_to_f32(xv.y & 0xFFFF), wv.z, acc);
                acc = fmaf(bf16_bits_to_f32(xv.y >> 16), wv.w, acc);
            }
            if (xr1 != nullptr) {
#pragma unroll 4
                for (int m = 0; m < n; ++m) {
                    const int g = lo + lane + 32 * m;
                    const float4 wv = *reinterpret_cast<const float4*>(Ws + 4 * g);
                    const uint2 xv = *reinterpret_cast<const uint2*>(xr1 + 4 * g);
                    acc2 = fmaf(bf16_bits_to_f32(xv.x & 0xFFFF), wv.x, acc2);
                    acc2 = fmaf(bf16_bits_to_f32(xv.x >> 16), wv.y, acc2);
                    acc2 = fmaf(bf16_bits_to_f32(xv.y & 0xFFFF), wv.z, acc2);
                    acc2 = fmaf(bf16_bits_to_f32(xv.y >> 16), wv.w, acc2);
                }
            }
        }
    }
    return make_float2(warp_butterfly_sum(acc), warp_butterfly_sum(acc2));
}

}  // namespace moe
