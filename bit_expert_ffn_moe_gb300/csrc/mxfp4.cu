// mxfp4.cu -- MXFP4 helpers: pack (fp32 -> E2M1 codes + E8M0 block scales), unpack, and the
// re-layout of block scales into the tensor-core scale layout.
// Format: DGX Spark MoE inference optimizations (section 2, block-scaled 4-bit MXFP4 expert
// path); Muse Spark Open explainer (section 11, 4-bit values sharing a small scale).  Rounding
// rule of OCP MX v1.0 (shared exponent floor(log2 amax) - 2, RNE onto the E2M1 grid, saturate).
#include "common.cuh"

namespace moe {

// One thread per 32-element block.
__global__ void pack_kernel(const float* __restrict__ w, int64_t nblocks, uint8_t* __restrict__ q,
                            uint8_t* __restrict__ s) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblocks; blk += stride) {
        const float4* src = reinterpret_cast<const float4*>(w + blk * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 f = src[i];
            v[4 * i] = f.x;
            v[4 * i + 1] = f.y;
            v[4 * i + 2] = f.z;
            v[4 * i + 3] = f.w;
        }
        uint4 codes;
        const uint32_t sb = mx_block_encode(v, codes);
        reinterpret_cast<uint4*>(q)[blk] = codes;
        s[blk] = (uint8_t)sb;
    }
}

// One thread per 32-element block; uses the hardware E2M1 -> f16 conversion.
__global__ void unpack_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t nblocks,
                              float* __restrict__ w) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; blk < nblocks; blk += stride) {
        uint4 c = reinterpret_cast<const uint4*>(q)[blk];
        float sc = e8m0_to_f32(s[blk]);
        uint32_t words[4] = {c.x, c.y, c.z, c.w};
        float4* dst = reinterpret_cast<float4*>(w + blk * 32);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t h[4];
            e2m1x8_to_h2(words[m], h);
            float2 a = h2_to_f2(h[0]), b = h2_to_f2(h[1]), cc = h2_to_f2(h[2]), dd = h2_to_f2(h[3]);
            dst[2 * m] = make_float4(a.x * sc, a.y * sc, b.x * sc, b.y * sc);
            dst[2 * m + 1] = make_float4(cc.x * sc, cc.y * sc, dd.x * sc, dd.y * sc);
        }
    }
}

// One thread per scale byte.
__global__ void scales_to_mma_kernel(const uint8_t* __restrict__ s, int64_t rows, int64_t K, uint8_t* __restrict__ out) {
    const int64_t cols = K / 32, total = rows * cols;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        int64_t r = i / cols, c = i % cols;
        out[mma_scale_offset(r, c, K)] = s[i];
    }
}

// Code tiles: one thread per 16-byte chunk (one 32-element block) of the output.
__global__ void codes_to_mma_kernel(const uint8_t* __restrict__ q, int64_t rows, int64_t K, uint8_t* __restrict__ out) {
    const int64_t nb = K / 32;  // 16-byte chunks per row
    const int64_t total = rows * nb;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t r = i / nb, blk = i % nb;
        *reinterpret_cast<uint4*>(out + mma_tile_offset(r, blk, K)) = reinterpret_cast<const uint4*>(q)[i];
    }
}

static unsigned grid_for(int64_t n, int threads) {
    int64_t b = (n + threads - 1) / threads;
    if (b > 152 * 64) b = 152 * 64;
    return (unsigned)(b < 1 ? 1 : b);
}

cudaError_t launch_pack(const float* w, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, cudaStream_t st) {
    int64_t nb = rows * (K / 32);
    if (nb == 0) return cudaSuccess;
    pack_kernel<<<grid_for(nb, 256), 256, 0, st>>>(w, nb, q, s);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K, float* w, cudaStream_t st) {
    int64_t nb = rows * (K / 32);
    if (nb == 0) return cudaSuccess;
    unpack_kernel<<<grid_for(nb, 256), 256, 0, st>>>(q, s, nb, w);
    return cudaGetLastError();
}

cudaError_t launch_scales_to_mma(const uint8_t* s, int64_t rows, int64_t K, uint8_t* s_mma, cudaStream_t st) {
    int64_t n = rows * (K / 32);
    if (n == 0) return cudaSuccess;
    scales_to_mma_kernel<<<grid_for(n, 256), 256, 0, st>>>(s, rows, K, s_mma);
    return cudaGetLastError();
}

cudaError_t launch_codes_to_mma(const uint8_t* q, int64_t rows, int64_t K, uint8_t* q_mma, cudaStream_t st) {
    int64_t n = rows * (K / 32);
    if (n == 0) return cudaSuccess;
    codes_to_mma_kernel<<<grid_for(n, 256), 256, 0, st>>>(q, rows, K, q_mma);
    return cudaGetLastError();
}

}  // namespace moe
