// noalloc.cu -- a router entry point that allocates nothing and takes no workspace.
//
// Some callers cannot allocate device memory, or own a scratch buffer, at the point where they
// route tokens: code that runs while a stream is being captured into a CUDA graph in the global
// capture mode (allocation calls are not permitted there), hosts that hand the whole device to a
// fixed memory pool and refuse further allocations, and thin foreign-function callers that have
// no means to size and keep a workspace alive.  moe_route_noalloc serves them: the router's only
// scratch, the T x E fp32 logits, lives in a fixed array in this library's own device memory.
//
// The array is a file-scope static __device__ object, so host code cannot use its name as a
// device address; its address is looked up once per device with cudaGetSymbolAddress (on the
// first call made with that device current) and passed to the existing router kernels.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kNoallocMaxLogits = 512 * 1024;  // T * E <= 524288 (2 MiB of fp32)
static __device__ __align__(256) float g_noalloc_logits[kNoallocMaxLogits];

// Device address of g_noalloc_logits on the current device (looked up once per device).
cudaError_t noalloc_scratch(float** out) {
    static std::mutex mu;
    static float* ptrs[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (ptrs[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_logits);
        if (err != cudaSuccess) return err;
        ptrs[dev] = static_cast<float*>(p);
    }
    *out = ptrs[dev];
    return cudaSuccess;
}

bool is_sm103() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    return major == 10 && minor == 3;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E,
                                        int k, int32_t* ids, float* w, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || d <= 0 || d % 128 != 0 || E <= 0 || E > kMaxE || k <= 0 || k > kMaxK || k > E)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((size_t)T * (size_t)E > kNoallocMaxLogits) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!x || !W_r || !ids || !w || (reinterpret_cast<uintptr_t>(x) % 16) || (reinterpret_cast<uintptr_t>(W_r) % 16))
        return MOE_ERR_INVALID_ARG;
    if (!is_sm103()) return MOE_ERR_DEVICE;
    float* logits = nullptr;
    if (noalloc_scratch(&logits) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    if (launch_route_logits(x, W_r, b, T, d, E, logits, st, false) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_topk(logits, T, E, k, ids, w, st, false) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}
