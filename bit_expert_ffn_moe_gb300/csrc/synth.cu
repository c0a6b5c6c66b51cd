// synth.cu -- device-side synthetic weight generator (input generation only; holds none of the
// layer's arithmetic).  Counter-based SplitMix64 (Steele, Lea & Flood, OOPSLA 2014): element n of
// expert e's matrix is float32(2*(u0+u1+u2+u3) - 262140) * c with u0..u3 the 16-bit fields of
// mix(key + (n+1) * golden), key = mix((seed << 32) | (tensor_id << 24) | e).
#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

__global__ void synth_weights_kernel(uint64_t seed, uint32_t tensor_id, uint32_t expert_first, int64_t per_expert,
                                     int64_t total, float c, float* __restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
        uint64_t e = expert_first + (uint64_t)(idx / per_expert);
        uint64_t n = (uint64_t)(idx % per_expert);
        uint64_t key = splitmix64_mix((seed << 32) | ((uint64_t)tensor_id << 24) | e);
        uint64_t z = splitmix64_mix(key + (n + 1) * 0x9E3779B97F4A7C15ull);
        int s = (int)(z & 0xFFFF) + (int)((z >> 16) & 0xFFFF) + (int)((z >> 32) & 0xFFFF) + (int)((z >> 48) & 0xFFFF);
        out[idx] = __fmul_rn((float)(2 * s - 262140), c);
    }
}

cudaError_t launch_synth(uint64_t seed, uint32_t tensor_id, uint32_t expert_first, uint32_t n_experts, int64_t rows,
                         int64_t K, float c, float* out, cudaStream_t st) {
    int64_t per = rows * K, total = per * (int64_t)n_experts;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    synth_weights_kernel<<<(unsigned)blocks, 256, 0, st>>>(seed, tensor_id, expert_first, per, total, c, out);
    return cudaGetLastError();
}

}  // namespace moe
