// selftest.cu -- failure-detection self-test of the bounded device waits.
//
// Every barrier wait in this library's kernels gives up after a bounded time, records
// MOE_ERR_TIMEOUT in the workspace status word and lets its kernel finish, so a copy or a signal
// that never arrives surfaces as an error status that the host reads, not as a hung GPU.
// moe_selftest_wait_timeout exercises exactly that path without faulting anything: one thread
// waits on an mbarrier phase that no thread ever completes, with a short time limit; the wait
// runs out, the status is recorded and the kernel returns normally, leaving the context usable.
#include "common.cuh"

namespace moe {
namespace {

__global__ void wait_timeout_kernel(int* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(&bar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    bool done = false;
    while (true) {
        uint32_t ok;
        // phase 0 of a barrier expecting one arrival that never comes
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(a)
            : "memory");
        if (ok) {
            done = true;
            break;
        }
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > limit_ns) break;
    }
    if (!done) set_status(status, MOE_ERR_TIMEOUT);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(a) : "memory");
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int limit_us, moe_stream_t stream) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % 256) != 0 || ws_bytes < sizeof(Ctrl))
        return MOE_ERR_WORKSPACE;
    if (limit_us < 1 || limit_us > 1000000) return MOE_ERR_INVALID_ARG;
    Ctrl* ctrl = static_cast<Ctrl*>(ws);
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(&ctrl->status, 1000ull * (unsigned long long)limit_us);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
