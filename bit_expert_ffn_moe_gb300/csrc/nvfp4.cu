// nvfp4.cu -- NVFP4 weight helpers: pack (fp32 -> E2M1 codes, one E4M3 scale per 16 elements,
// one fp32 global scale per matrix) and unpack.
// Format: Muse Spark Open explainer, section 11 (the expert weights are 4-bit values of which 16
// share a small scale, about 4.5 bits per value); the scale is an E4M3 number (OCP OFP8) and the
// global scale puts the largest block scale of a matrix at the top of the E4M3 range.
// Every step of the rule runs in fp32 with round-to-nearest-even: the divisions and products are
// written with the _rn intrinsics so that no contraction or approximation can change a code.
#include "common.cuh"

namespace moe {

// Largest |w| of each matrix as fp32 bits in amax_bits[m] (non-negative fp32 values order like
// their bit patterns, so an integer atomicMax finds the maximum).  Grid (chunks, n_mats).
__global__ void nv_amax_kernel(const float* __restrict__ w, int64_t per_mat, unsigned* __restrict__ amax_bits) {
    const int m = blockIdx.y;
    const float4* src = reinterpret_cast<const float4*>(w + (int64_t)m * per_mat);
    const int64_t n4 = per_mat / 4;
    float mx = 0.f;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
        const float4 v = src[i];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    __shared__ float red[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    if (warp == 0) {
        mx = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.f;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) atomicMax(amax_bits + m, __float_as_uint(mx));
    }
}

// In place: the maximum's bits -> the global scale max / (6 * 448), or 1 when that is 0.
__global__ void nv_global_kernel(float* gs, int64_t n_mats) {
    for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < n_mats; m += (int64_t)gridDim.x * blockDim.x) {
        const float g = __fdiv_rn(gs[m], 2688.f);
        gs[m] = g == 0.f ? 1.f : g;
    }
}

// One thread per 32 elements of a row (two 16-element blocks): 16 bytes of codes, 2 scale bytes.
__global__ void nv_pack_kernel(const float* __restrict__ w, int64_t units_per_mat, int64_t n_units,
                               const float* __restrict__ gs, uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += stride) {
        const float g = gs[u / units_per_mat];
        const float4* src = reinterpret_cast<const float4*>(w + u * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 f = src[i];
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
        uint32_t cw[4];
        uint32_t sb2 = 0;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float* vh = v + 16 * half;
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(vh[i]));
            const uint32_t sb = f32_to_e4m3_sat(__fdiv_rn(__fdiv_rn(amax, g), 6.f));
            const float D = __fmul_rn(e4m3x2_to_f2(sb).x, g);
            if (D == 0.f) {
                cw[2 * half] = cw[2 * half + 1] = 0u;
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) vh[i] = __fdiv_rn(vh[i], D);
                cw[2 * half] = e2m1x8_encode(vh);
                cw[2 * half + 1] = e2m1x8_encode(vh + 8);
            }
            sb2 |= sb << (8 * half);
        }
        reinterpret_cast<uint4*>(q)[u] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        reinterpret_cast<uint16_t*>(s)[u] = (uint16_t)sb2;
    }
}

// One thread per 32 elements: value = (E2M1 * E4M3) * global, the exact product rounded once.
__global__ void nv_unpack_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                 const float* __restrict__ gs, int64_t units_per_mat, int64_t n_units,
                                 float* __restrict__ w) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; u < n_units; u += stride) {
        const float g = gs[u / units_per_mat];
        const uint4 c = reinterpret_cast<const uint4*>(q)[u];
        const float2 sc = e4m3x2_to_f2(reinterpret_cast<const uint16_t*>(s)[u]);
        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
        float4* dst = reinterpret_cast<float4*>(w + u * 32);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float sv = m < 2 ? sc.x : sc.y;  // words 0, 1: elements 0..15; words 2, 3: 16..31
            uint32_t h[4];
            e2m1x8_to_h2(words[m], h);
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 p = h2_to_f2(h[j]);
                f[2 * j] = __fmul_rn(__fmul_rn(p.x, sv), g);
                f[2 * j + 1] = __fmul_rn(__fmul_rn(p.y, sv), g);
            }
            dst[2 * m] = make_float4(f[0], f[1], f[2], f[3]);
            dst[2 * m + 1] = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
}

// ------------------------------------------------------------------ MXFP4 rows against NVFP4 weights
// The tensor cores take NVFP4 weights (kind::mxf4nvf4) only with both operands' scales in UE4M3, one
// per 16 values.  An MXFP4 operand row keeps its codes; each 32-element block's scale 2^X_b becomes
// the UE4M3 power of two 2^(X_b - F) on both of its 16-element halves, with one factor 2^F per row,
// F = max_b X_b - 8, that the GEMM epilogue multiplies back in.  UE4M3 holds the powers of two
// 2^-9 .. 2^8, so this is exact for every block within 17 binades of the row's largest; a block
// further below (whose values are below 2^-15 of the row's largest block scale) gets scale 0.
// One warp per padded row; s32 and s16 in the tensor-core scale layout of width K and 2K.
__global__ void __launch_bounds__(256) nv_operand_scales_kernel(const uint8_t* __restrict__ s32,
                                                                const int32_t* __restrict__ rows_used, int K,
                                                                uint8_t* __restrict__ s16, float* __restrict__ rf) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t used = *rows_used;
    const int nb = K / 32, lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < used; r += nwarps) {
        int smax = 0;  // largest scale byte (X + 127) of the row
        for (int b = lane; b < nb; b += 32) smax = max(smax, (int)s32[mma_scale_offset(r, b, K)]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) smax = max(smax, __shfl_xor_sync(0xffffffffu, smax, o));
        const int F = smax - 127 - 8;
        for (int b = lane; b < nb; b += 32) {
            const int e = (int)s32[mma_scale_offset(r, b, K)] - 127 - F;  // <= 8
            // UE4M3 of 2^e: normal for e >= -6 (exponent field e + 7), subnormal 2^-7 .. 2^-9
            const uint32_t u = e >= -6 ? (uint32_t)(e + 7) << 3 : e >= -9 ? 1u << (e + 9) : 0u;
            *reinterpret_cast<uint16_t*>(s16 + mma_scale_offset(r, 2 * b, 2 * K)) = (uint16_t)(u | (u << 8));
        }
        if (lane == 0)  // 2^F, F in [-135, 119]: subnormal below 2^-126
            rf[r] = F >= -126 ? __uint_as_float((uint32_t)(F + 127) << 23) : __uint_as_float(1u << (F + 149));
    }
}

cudaError_t launch_nv_operand_scales(const uint8_t* s32, const int32_t* rows_used, int64_t pad_rows, int K,
                                     uint8_t* s16, float* rf, cudaStream_t st, bool pdl) {
    if (pad_rows == 0) return cudaSuccess;
    int64_t blocks = (pad_rows + 7) / 8;  // 8 warps (rows) per CTA
    if (blocks > 152 * 8) blocks = 152 * 8;
    void* args[] = {&s32, &rows_used, &K, &s16, &rf};
    return launch_kernel((const void*)nv_operand_scales_kernel, dim3((unsigned)blocks), dim3(256), 0, st, pdl, args);
}

static unsigned nv_grid(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    if (b > 152 * 64) b = 152 * 64;
    return (unsigned)(b < 1 ? 1 : b);
}

cudaError_t launch_nvfp4_pack(const float* w, int64_t n_mats, int64_t rows, int64_t K, uint8_t* q, uint8_t* s,
                              float* gs, cudaStream_t st) {
    const int64_t per_mat = rows * K;
    if (n_mats == 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(gs, 0, sizeof(float) * (size_t)n_mats, st);
    if (e != cudaSuccess) return e;
    if (per_mat > 0) {
        int64_t chunks = (per_mat / 4 + 255) / 256;
        if (chunks > 1024) chunks = 1024;
        nv_amax_kernel<<<dim3((unsigned)chunks, (unsigned)n_mats), 256, 0, st>>>(w, per_mat,
                                                                              reinterpret_cast<unsigned*>(gs));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    nv_global_kernel<<<nv_grid(n_mats, 256), 256, 0, st>>>(gs, n_mats);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t units = n_mats * rows * (K / 32);
    if (units == 0) return cudaSuccess;
    nv_pack_kernel<<<nv_grid(units, 256), 256, 0, st>>>(w, rows * (K / 32), units, gs, q, s);
    return cudaGetLastError();
}

cudaError_t launch_nvfp4_unpack(const uint8_t* q, const uint8_t* s, const float* gs, int64_t n_mats, int64_t rows,
                                int64_t K, float* w, cudaStream_t st) {
    const int64_t units = n_mats * rows * (K / 32);
    if (units == 0) return cudaSuccess;
    nv_unpack_kernel<<<nv_grid(units, 256), 256, 0, st>>>(q, s, gs, rows * (K / 32), units, w);
    return cudaGetLastError();
}

}  // namespace moe
