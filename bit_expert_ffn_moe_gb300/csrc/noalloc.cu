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
// device address.  Its address is looked up with cudaGetSymbolAddress, with the device current,
// once per CUDA context: the cache is keyed on the device and on the id of the context current
// when the call is made, so a new context (after cudaDeviceReset, or a caller that binds its own
// driver context) gets a fresh lookup instead of a stale address.
#include <mutex>

#include "common.cuh"

namespace moe {
namespace {

constexpr size_t kNoallocMaxLogits = 512 * 1024;  // T * E <= 524288 (2 MiB of fp32)
static __device__ __align__(256) float g_noalloc_logits[kNoallocMaxLogits];

// Driver calls that identify the current context, taken through the runtime's entry-point query
// (no link-time dependency on the driver library).  Null when the driver does not provide them.
typedef int (*ctx_get_current_fn)(void** ctx);
typedef int (*ctx_get_id_fn)(void* ctx, unsigned long long* id);

struct CtxQuery {
    ctx_get_current_fn get_current = nullptr;
    ctx_get_id_fn get_id = nullptr;
};

const CtxQuery& ctx_query() {
    static CtxQuery q;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            q.get_current = reinterpret_cast<ctx_get_current_fn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            q.get_id = reinterpret_cast<ctx_get_id_fn>(f);
    });
    return q;
}

// Id of the context current on this thread; false when it cannot be determined.
bool current_ctx_id(unsigned long long* id) {
    const CtxQuery& q = ctx_query();
    if (!q.get_current || !q.get_id) return false;
    void* ctx = nullptr;
    if (q.get_current(&ctx) != 0 || ctx == nullptr) return false;
    return q.get_id(ctx, id) == 0;
}

// Device address of g_noalloc_logits in the current context (looked up once per context; on
// every call when the context cannot be identified).
cudaError_t noalloc_scratch(float** out) {
    static std::mutex mu;
    struct Entry {
        bool valid;
        unsigned long long ctx;
        float* ptr;
    };
    static Entry cache[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    unsigned long long ctx = 0;
    const bool known = current_ctx_id(&ctx);
    std::lock_guard<std::mutex> lock(mu);
    if (known && cache[dev].valid && cache[dev].ctx == ctx) {
        *out = cache[dev].ptr;
        return cudaSuccess;
    }
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_logits);
    if (err != cudaSuccess) return err;
    // the lookup makes the device's primary context current if none was: identify it now
    if (!known && current_ctx_id(&ctx)) cache[dev] = {true, ctx, static_cast<float*>(p)};
    else if (known) cache[dev] = {true, ctx, static_cast<float*>(p)};
    *out = static_cast<float*>(p);
    return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E,
                                        int k, int32_t* ids, float* w, moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_shape(T, d, E, k, 32, MOE_ACT_BF16);  // the same rules as moe_route
    if (st != MOE_OK) return st;
    if ((size_t)T * (size_t)E > kNoallocMaxLogits) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!x || !W_r || !ids || !w || (reinterpret_cast<uintptr_t>(x) % 16) || (reinterpret_cast<uintptr_t>(W_r) % 16))
        return MOE_ERR_INVALID_ARG;
    st = check_device();
    if (st != MOE_OK) return st;
    float* logits = nullptr;
    st = from_cuda(noalloc_scratch(&logits));
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    st = from_cuda(launch_route_logits(x, W_r, b, T, d, E, logits, s, false));
    if (st != MOE_OK) return st;
    return from_cuda(launch_topk(logits, T, E, k, ids, w, s, false));
}
