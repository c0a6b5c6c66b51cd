// api.cu -- the extern "C" entry points declared in include/moe.h: argument checks, workspace
// carving and the launch sequence of each layer step.  No entry point allocates device memory.
#include <stdio.h>

#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

using namespace moe;

namespace moe {

// The kernels are compiled for sm_103a only; refuse other devices before launching.
moe_status check_device() {
    static int verdict[64] = {0};  // 0 unknown, 1 ok, 2 bad
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev >= 0 && dev < 64 && verdict[dev] == 1) return MOE_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const bool ok = (major == 10 && minor == 3);
    if (dev >= 0 && dev < 64) verdict[dev] = ok ? 1 : 2;
    return ok ? MOE_OK : MOE_ERR_DEVICE;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

moe_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    g_last_cuda_error = e;
    return MOE_ERR_CUDA;
}

moe_status check_shape(int T, int d, int E, int k, int I, moe_act_fmt fmt) {
    if (T < 0 || d <= 0 || E <= 0 || k <= 0 || I <= 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (fmt != MOE_ACT_BF16 && fmt != MOE_ACT_MXFP4 && fmt != MOE_ACT_MXFP8) return MOE_ERR_INVALID_ARG;
    if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (d % (fmt == MOE_ACT_BF16 ? 128 : 256) != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (I % (fmt == MOE_ACT_BF16 ? 32 : 256) != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((int64_t)T * k > (int64_t)1 << 30 || (int64_t)T * d > ((int64_t)1 << 40)) return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

}  // namespace moe

namespace {

constexpr int kAbiVersion = 13;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define MOE_TRY(expr)                               \
    do {                                            \
        moe_status _s = (expr);                     \
        if (_s != MOE_OK) return _s;                \
    } while (0)
#define MOE_CUDA(expr) MOE_TRY(from_cuda(expr))

moe_status check_ws(void* ws, size_t ws_bytes, const WsLayout& L) {
    if (ws == nullptr || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status check_weights(const moe_expert_weights* W, moe_act_fmt fmt, bool need_up, bool need_down) {
    if (W == nullptr) return MOE_ERR_INVALID_ARG;
    if (W->wfmt != MOE_W_MXFP4 && W->wfmt != MOE_W_NVFP4) return MOE_ERR_INVALID_ARG;
    if (W->wfmt == MOE_W_NVFP4) {  // the GEMVs (E4M3 scale pairs read as 16-bit words) or kind::mxf4nvf4
        if (fmt == MOE_ACT_MXFP8) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (need_up && (!W->gate_gs || !W->up_gs || !aligned(W->gate_s, 2) || !aligned(W->up_s, 2)))
            return MOE_ERR_INVALID_ARG;
        if (need_down && (!W->down_gs || !aligned(W->down_s, 2))) return MOE_ERR_INVALID_ARG;
    }
    // MOE_ACT_MXFP8 reads the canonical codes through tensor maps (32-byte aligned) as well as the
    // tensor-core copies
    const size_t q_align = fmt == MOE_ACT_MXFP8 ? 32 : 16;
    const bool mma = fmt != MOE_ACT_BF16;
    if (need_up) {
        if (!W->gate_q || !W->gate_s || !W->up_q || !W->up_s) return MOE_ERR_INVALID_ARG;
        if (!aligned(W->gate_q, q_align) || !aligned(W->up_q, q_align)) return MOE_ERR_INVALID_ARG;
        if (mma && (!W->gate_q_mma || !W->gate_s_mma || !W->up_q_mma || !W->up_s_mma || !aligned(W->gate_q_mma, 16) ||
                    !aligned(W->gate_s_mma, 16) || !aligned(W->up_q_mma, 16) || !aligned(W->up_s_mma, 16)))
            return MOE_ERR_INVALID_ARG;
    }
    if (need_down) {
        if (!W->down_q || !W->down_s || !aligned(W->down_q, q_align)) return MOE_ERR_INVALID_ARG;
        if (mma && (!W->down_q_mma || !W->down_s_mma || !aligned(W->down_q_mma, 16) || !aligned(W->down_s_mma, 16)))
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

char* at(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

// route (+ permutation when fused) into the given buffers
moe_status run_route(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                     int32_t* ids, float* w, void* ws, const WsLayout& L, cudaStream_t st, bool pdl,
                     int32_t* counts = nullptr) {
    float* logits = reinterpret_cast<float*>(at(ws, L.logits));
    cudaError_t e = cudaErrorNotSupported;
    if (L.rs_list) {  // many tokens: tensor-core screen, fixed-order logits of the candidates only
        const RouterScreenBufs rb = {reinterpret_cast<uint8_t*>(at(ws, L.rs_bhi)),
                                     reinterpret_cast<uint8_t*>(at(ws, L.rs_blo)),
                                     reinterpret_cast<float*>(at(ws, L.rs_wn2)),
                                     reinterpret_cast<float*>(at(ws, L.rs_part)),
                                     reinterpret_cast<float*>(at(ws, L.rs_xn2)),
                                     reinterpret_cast<int32_t*>(at(ws, L.rs_cnt)),
                                     reinterpret_cast<int32_t*>(at(ws, L.rs_list)),
                                     reinterpret_cast<uint32_t*>(at(ws, L.rs_stat))};
        e = launch_router_screen(x, W_r, b, T, d, E, k, rb, logits, ids, w,
                                 &reinterpret_cast<Ctrl*>(at(ws, L.ctrl))->status, st, pdl, counts);
        if (e != cudaErrorNotSupported) {
            MOE_CUDA(e);
            return MOE_OK;
        }
    }
    MOE_CUDA(launch_route_logits(x, W_r, b, T, d, E, logits, st, pdl, counts));
    MOE_CUDA(launch_topk(logits, T, E, k, ids, w, st, true, counts));
    return MOE_OK;
}

// route + permutation of the layer call: the top-k counts the picks per expert into plan.counts
// (zeroed by the route's first launch), then one launch builds offsets, plan and the permuted rows
// (with row weights)
moe_status route_counted(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                         int32_t* ids, float* w, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                         float* row_w, const PlanView& plan, void* ws, const WsLayout& L, cudaStream_t st) {
    MOE_TRY(run_route(x, W_r, b, T, d, E, k, ids, w, ws, L, st, true, plan.counts));
    MOE_CUDA(launch_permute_counted(ids, T, E, k, counts, offsets, perm, inv, plan, st, true, w, row_w));
    return MOE_OK;
}

// Events of a host-buffer call's staging buffer (moe_layer_forward_host with copy streams): "ready"
// (its input copy landed, or the layer wrote it), "consumed" (the last layer that read it is done),
// "drained" (the last copy out of it is done).  Created on first use of a buffer address, kept for
// the process in a small table: beyond 64 buffers the least recently used entry is released,
// after the host has waited for its events -- a buffer met again later then has no pending work
// that its fresh events would fail to order.
struct StagingEvents {
    cudaEvent_t ready = nullptr, consumed = nullptr, drained = nullptr;
    bool consumed_recorded = false, drained_recorded = false;
};

StagingEvents* staging_events(const void* buf) {
    static std::mutex mu;
    static std::vector<std::pair<const void*, StagingEvents*>> table;
    std::lock_guard<std::mutex> lock(mu);
    for (size_t i = 0; i < table.size(); ++i)
        if (table[i].first == buf) {  // most recently used at the back, so that the entries of one
            auto hit = table[i];      // call (x and y) are never the one evicted for the other
            table.erase(table.begin() + (ptrdiff_t)i);
            table.push_back(hit);
            return hit.second;
        }
    if (table.size() >= 64) {
        StagingEvents* old = table.front().second;
        if (cudaEventSynchronize(old->ready) != cudaSuccess || cudaEventSynchronize(old->consumed) != cudaSuccess ||
            cudaEventSynchronize(old->drained) != cudaSuccess)
            return nullptr;
        cudaEventDestroy(old->ready);
        cudaEventDestroy(old->consumed);
        cudaEventDestroy(old->drained);
        delete old;
        table.erase(table.begin());
    }
    StagingEvents* ev = new StagingEvents();
    if (cudaEventCreateWithFlags(&ev->ready, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev->consumed, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev->drained, cudaEventDisableTiming) != cudaSuccess) {
        delete ev;
        return nullptr;
    }
    table.emplace_back(buf, ev);
    return ev;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    }
    return "MOE_ERR_UNKNOWN";
}

int moe_abi_version(void) { return kAbiVersion; }

const char* moe_last_cuda_error(void) {
    return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

// ---------------------------------------------------------------- MXFP4 helpers

moe_status moe_mxfp4_pack(const float* w, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, moe_stream_t stream) {
    if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !s || !aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_pack(w, rows, K, q, s, (cudaStream_t)stream));
}

moe_status moe_mxfp4_unpack(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K, float* w,
                            moe_stream_t stream) {
    if (rows < 0 || K <= 0 || K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MOE_OK;
    if (!w || !q || !s || !aligned(w, 16) || !aligned(q, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_unpack(q, s, rows, K, w, (cudaStream_t)stream));
}

// ---------------------------------------------------------------- NVFP4 helpers

static moe_status check_nvfp4(const void* w, int64_t n_mats, int64_t rows, int64_t K, const void* q, const void* s,
                              const void* gs) {
    if (n_mats < 0 || n_mats > 65535 || rows < 0 || K <= 0 || K % 32 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (n_mats == 0) return MOE_OK;
    if (!gs || !aligned(gs, 4)) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!w || !q || !s || !aligned(w, 16) || !aligned(q, 16) || !aligned(s, 2))) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status moe_nvfp4_pack(const float* w, int64_t n_mats, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, float* gs,
                          moe_stream_t stream) {
    MOE_TRY(check_nvfp4(w, n_mats, rows, K, q, s, gs));
    if (n_mats == 0) return MOE_OK;
    MOE_TRY(check_device());
    return from_cuda(launch_nvfp4_pack(w, n_mats, rows, K, q, s, gs, (cudaStream_t)stream));
}

moe_status moe_nvfp4_unpack(const uint8_t* q, const uint8_t* s, const float* gs, int64_t n_mats, int64_t rows,
                            int64_t K, float* w, moe_stream_t stream) {
    MOE_TRY(check_nvfp4(w, n_mats, rows, K, q, s, gs));
    if (n_mats == 0 || rows == 0) return MOE_OK;
    MOE_TRY(check_device());
    return from_cuda(launch_nvfp4_unpack(q, s, gs, n_mats, rows, K, w, (cudaStream_t)stream));
}

size_t moe_mxfp4_mma_scale_bytes(int64_t rows, int64_t K) {
    if (rows <= 0 || K <= 0) return 0;
    return mma_scale_bytes(rows, K);
}

moe_status moe_mxfp4_scales_to_mma(const uint8_t* s, int64_t rows, int64_t K, uint8_t* s_mma, moe_stream_t stream) {
    if (rows <= 0 || K <= 0 || rows % 128 != 0 || K % 128 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!s || !s_mma) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_scales_to_mma(s, rows, K, s_mma, (cudaStream_t)stream));
}

moe_status moe_mxfp4_codes_to_mma(const uint8_t* q, int64_t rows, int64_t K, uint8_t* q_mma, moe_stream_t stream) {
    if (rows <= 0 || K <= 0 || rows % 128 != 0 || K % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!q || !q_mma || !aligned(q, 16) || !aligned(q_mma, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_codes_to_mma(q, rows, K, q_mma, (cudaStream_t)stream));
}

// ---------------------------------------------------------------- workspace

size_t moe_workspace_size(int T, int d, int E, int k, int I, moe_act_fmt fmt) {
    if (check_shape(T, d, E, k, I, fmt) != MOE_OK) return 0;
    return ws_layout(T, d, E, k, I, fmt).total;
}

int64_t moe_padded_rows(int T, int k, int E) {
    if (T < 0 || k <= 0 || E <= 0) return 0;
    return padded_rows(T, k, E);
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (ws == nullptr || !aligned(ws, 256) || ws_bytes < sizeof(Ctrl)) return MOE_ERR_WORKSPACE;
    MOE_TRY(check_device());
    return from_cuda(cudaMemsetAsync(ws, 0, sizeof(Ctrl), (cudaStream_t)stream));
}

moe_status moe_get_device_status(void* ws, moe_stream_t stream, moe_status* out) {
    if (ws == nullptr || out == nullptr || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int host = 0;
    MOE_CUDA(cudaMemcpyAsync(&host, ws, sizeof(int), cudaMemcpyDeviceToHost, st));
    MOE_CUDA(cudaMemsetAsync(ws, 0, sizeof(int), st));
    MOE_CUDA(cudaStreamSynchronize(st));
    *out = (moe_status)host;
    return MOE_OK;
}

// ---------------------------------------------------------------- layer steps

moe_status moe_workspace_routing(void* ws, size_t ws_bytes, int T, int d, int E, int k, int I, moe_act_fmt fmt,
                                 int32_t** counts, int32_t** offsets, int32_t** perm_token, int32_t** inv_pos) {
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (!counts || !offsets || !perm_token || !inv_pos) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    *counts = reinterpret_cast<int32_t*>(at(ws, L.counts));
    *offsets = reinterpret_cast<int32_t*>(at(ws, L.offsets));
    *perm_token = reinterpret_cast<int32_t*>(at(ws, L.perm));
    *inv_pos = reinterpret_cast<int32_t*>(at(ws, L.inv));
    return MOE_OK;
}


moe_status moe_route(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k, int32_t* ids,
                     float* w, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_shape(T, d, E, k, 32, MOE_ACT_BF16));
    if (T == 0) return MOE_OK;
    if (!x || !W_r || !ids || !w || !aligned(x, 16) || !aligned(W_r, 16)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, 32, MOE_ACT_BF16);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    if (route_decode_supported(T, d, E, k)) {  // few tokens: the one-launch router (its plan goes to ws)
        return from_cuda(launch_route_decode(
            x, W_r, b, T, d, E, k, reinterpret_cast<float*>(at(ws, L.logits)), ids, w,
            reinterpret_cast<int32_t*>(at(ws, L.counts)), reinterpret_cast<int32_t*>(at(ws, L.offsets)),
            reinterpret_cast<int32_t*>(at(ws, L.perm)), reinterpret_cast<int32_t*>(at(ws, L.inv)),
            reinterpret_cast<float*>(at(ws, L.row_w)), plan_view(ws, L, E), reinterpret_cast<Ctrl*>(at(ws, L.ctrl)),
            (cudaStream_t)stream, false));
    }
    return run_route(x, W_r, b, T, d, E, k, ids, w, ws, L, (cudaStream_t)stream, false);
}

moe_status moe_permute(const uint16_t* x, const int32_t* ids, int T, int d, int E, int k, moe_act_fmt fmt,
                       int32_t* counts, int32_t* offsets, int32_t* perm_token, int32_t* inv_pos, uint8_t* xa,
                       uint8_t* xa_s, void* ws, size_t ws_bytes, moe_stream_t stream) {
    // the buffers this call uses do not depend on I: check against the smallest valid I
    const int I_min = fmt == MOE_ACT_BF16 ? 32 : 256;
    MOE_TRY(check_shape(T, d, E, k, I_min, fmt));
    if (!ids || !counts || !offsets || !perm_token || !inv_pos) return MOE_ERR_INVALID_ARG;
    // the token operand of the prefill GEMMs (MXFP4 / MXFP8), unless both buffers are NULL
    const bool operand = fmt != MOE_ACT_BF16 && (xa != nullptr || xa_s != nullptr);
    if (operand && (!x || !xa || !xa_s || !aligned(x, 16) || !aligned(xa, 16))) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I_min, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    cudaStream_t st = (cudaStream_t)stream;
    PlanView plan = plan_view(ws, L, E);
    MOE_CUDA(launch_permute(ids, T, E, k, counts, offsets, perm_token, inv_pos, plan, st, false));
    if (operand)
        MOE_CUDA(launch_act_quant_gather(x, T, d, E, k, offsets, perm_token, plan, L.pad_rows,
                                         reinterpret_cast<uint8_t*>(at(ws, L.xq)),
                                         reinterpret_cast<uint8_t*>(at(ws, L.xs)), xa, xa_s, fmt == MOE_ACT_MXFP8, st,
                                         true));
    return MOE_OK;
}

size_t moe_decode_pieces_bytes(int T, int d, int scales) {
    if (!mma_decode_shape(T, d, 256)) return 0;
    return scales ? mma_scale_bytes(128, d) : (size_t)128 * d / 2;
}

moe_status moe_decode_pieces(const uint16_t* x, int T, int d, moe_act_fmt fmt, uint8_t* xa, uint8_t* xa_s,
                             moe_stream_t stream) {
    if (fmt != MOE_ACT_BF16 && fmt != MOE_ACT_MXFP8) return MOE_ERR_INVALID_ARG;
    if (T == 0) return d > 0 && d % 256 == 0 ? MOE_OK : MOE_ERR_UNSUPPORTED_SHAPE;
    if (!mma_decode_shape(T, d, 256)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!x || !xa || !xa_s || !aligned(x, 16) || !aligned(xa, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_x_pieces(x, T, d, fmt == MOE_ACT_MXFP8, xa, xa_s, (cudaStream_t)stream, false));
}

moe_status moe_expert_ffn_decode(const uint8_t* xa, const uint8_t* xa_s, moe_act_fmt fmt, const int32_t* perm_token,
                                 const int32_t* offsets, const int32_t* inv_pos, const float* w, int T, int d, int E,
                                 int k, int I, const moe_expert_weights* W, uint16_t* y_perm, uint16_t* y, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
    if (fmt != MOE_ACT_BF16 && fmt != MOE_ACT_MXFP8) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(W, fmt, true, true));
    if (!mma_decode_supported(T, d, E, k, I, W)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (y != nullptr && !mma_decode_fused_sum(T, d)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!xa || !xa_s || !perm_token || !offsets || !y_perm || !aligned(xa, 16) || !aligned(y_perm, 16))
        return MOE_ERR_INVALID_ARG;
    if (y != nullptr && (!inv_pos || !w || !aligned(y, 16))) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(ws, L.ctrl));
    return from_cuda(launch_mma_decode(xa, xa_s, reinterpret_cast<uint8_t*>(at(ws, L.dha)),
                                       reinterpret_cast<uint8_t*>(at(ws, L.dha_s)),
                                       reinterpret_cast<float*>(at(ws, L.dpart)), plan_view(ws, L, E), offsets,
                                       perm_token, T, d, E, k, I, W, fmt == MOE_ACT_MXFP8, y_perm, inv_pos, w, y, ctrl,
                                       (cudaStream_t)stream, false));
}

moe_status moe_expert_up_swiglu(const uint16_t* x, const uint8_t* xa, const uint8_t* xa_s, moe_act_fmt fmt,
                                const int32_t* perm_token, const int32_t* offsets, int T, int d, int E, int k, int I,
                                const moe_expert_weights* W, void* h, uint8_t* h_s, void* ws, size_t ws_bytes,
                                moe_stream_t stream) {
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(W, fmt, true, false));
    if (!offsets || !h) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    cudaStream_t st = (cudaStream_t)stream;
    PlanView plan = plan_view(ws, L, E);
    if (fmt == MOE_ACT_BF16) {
        if (!x || !perm_token || !aligned(x, 16)) return MOE_ERR_INVALID_ARG;
        if (!gemv_supported(d, I)) return MOE_ERR_UNSUPPORTED_SHAPE;
        return from_cuda(launch_gemv_up(x, perm_token, offsets, plan, T, d, E, k, I, W,
                                        static_cast<uint16_t*>(h), st, false));
    }
    if (!xa || !xa_s || !h_s || !aligned(xa, 16) || !aligned(h, 16)) return MOE_ERR_INVALID_ARG;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(ws, L.ctrl));
    if (W->wfmt == MOE_W_NVFP4) {  // the token operand's scales as UE4M3 per 16 (workspace)
        if (!umma_nv_supported(E)) return MOE_ERR_UNSUPPORTED_SHAPE;
        uint8_t* s16 = reinterpret_cast<uint8_t*>(at(ws, L.xa_s16));
        float* rf = reinterpret_cast<float*>(at(ws, L.xrf));
        MOE_CUDA(launch_nv_operand_scales(xa_s, plan.scalars + 2, L.pad_rows, d, s16, rf, st, false));
        return from_cuda(launch_umma_up(xa, s16, plan, offsets, T, d, E, k, I, L.pad_rows, W, false, rf,
                                        static_cast<uint8_t*>(h), h_s, &ctrl->status, st, true));
    }
    return from_cuda(launch_umma_up(xa, xa_s, plan, offsets, T, d, E, k, I, L.pad_rows, W, fmt == MOE_ACT_MXFP8,
                                    nullptr, static_cast<uint8_t*>(h), h_s, &ctrl->status, st, false));
}

moe_status moe_expert_down(const void* h, const uint8_t* h_s, moe_act_fmt fmt, const int32_t* perm_token,
                           const int32_t* offsets, int T, int d, int E, int k, int I, const moe_expert_weights* W,
                           uint16_t* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(W, fmt, false, true));
    if (!h || !offsets || !y_perm || !aligned(h, 16)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    cudaStream_t st = (cudaStream_t)stream;
    PlanView plan = plan_view(ws, L, E);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(ws, L.ctrl));
    if (fmt == MOE_ACT_BF16) {
        if (!perm_token) return MOE_ERR_INVALID_ARG;
        if (!gemv_supported(d, I)) return MOE_ERR_UNSUPPORTED_SHAPE;
        return from_cuda(launch_gemv_down(static_cast<const uint16_t*>(h), perm_token, offsets, plan, nullptr, T, d, E,
                                          k, I, W, y_perm, nullptr, &ctrl->status, st, false));
    }
    if (!h_s) return MOE_ERR_INVALID_ARG;
    if (W->wfmt == MOE_W_NVFP4) {  // h's scales as UE4M3 per 16 (workspace)
        if (!umma_nv_supported(E)) return MOE_ERR_UNSUPPORTED_SHAPE;
        uint8_t* s16 = reinterpret_cast<uint8_t*>(at(ws, L.h_s16));
        float* rf = reinterpret_cast<float*>(at(ws, L.hrf));
        MOE_CUDA(launch_nv_operand_scales(h_s, plan.scalars + 2, L.pad_rows, I, s16, rf, st, false));
        return from_cuda(launch_umma_down(static_cast<const uint8_t*>(h), s16, plan, offsets, T, d, E, k, I,
                                          L.pad_rows, W, false, rf, y_perm, &ctrl->status, st, true));
    }
    return from_cuda(launch_umma_down(static_cast<const uint8_t*>(h), h_s, plan, offsets, T, d, E, k, I, L.pad_rows, W,
                                      fmt == MOE_ACT_MXFP8, nullptr, y_perm, &ctrl->status, st, false));
}

moe_status moe_combine(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d, uint16_t* y,
                       moe_stream_t stream) {
    if (T < 0 || k <= 0 || k > kMaxK || d <= 0 || d % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MOE_OK;
    if (!y_perm || !inv_pos || !w || !y || !aligned(y_perm, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_combine(y_perm, inv_pos, w, T, k, d, y, (cudaStream_t)stream, false));
}

moe_status moe_combine_norm(const uint16_t* y_perm, const int32_t* inv_pos, const float* w, int T, int k, int d,
                            float eps, uint16_t* y, moe_stream_t stream) {
    if (T < 0 || k <= 0 || k > kMaxK || d <= 0 || d % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!(eps > 0.f && eps <= 1.f)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y_perm || !inv_pos || !w || !y || !aligned(y_perm, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_combine_norm(y_perm, inv_pos, w, T, k, d, eps, y, (cudaStream_t)stream, false));
}

// The layer; norm: each expert output row is divided by its RMS over d before the weighted sum.
static moe_status layer_forward(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k, int I,
                                const moe_expert_weights* W, moe_act_fmt fmt, bool norm, float eps, uint16_t* y,
                                int32_t* ids, float* w, void* ws, size_t ws_bytes, cudaStream_t st) {
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (norm && !(eps > 0.f && eps <= 1.f)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    MOE_TRY(check_weights(W, fmt, true, true));
    if (!x || !W_r || !y || !aligned(x, 16) || !aligned(W_r, 16) || !aligned(y, 16)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, I, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    PlanView plan = plan_view(ws, L, E);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(ws, L.ctrl));
    int32_t* ids_b = ids ? ids : reinterpret_cast<int32_t*>(at(ws, L.ids));
    float* w_b = w ? w : reinterpret_cast<float*>(at(ws, L.w));
    int32_t* counts = reinterpret_cast<int32_t*>(at(ws, L.counts));
    int32_t* offsets = reinterpret_cast<int32_t*>(at(ws, L.offsets));
    int32_t* perm = reinterpret_cast<int32_t*>(at(ws, L.perm));
    int32_t* inv = reinterpret_cast<int32_t*>(at(ws, L.inv));
    float* row_w = reinterpret_cast<float*>(at(ws, L.row_w));

    if (fmt != MOE_ACT_MXFP4 && mma_decode_supported(T, d, E, k, I, W)) {
        // few tokens, MXFP4 weights with their tensor-core copies: the expert GEMMs on the tensor
        // cores, each activation row (bf16, or its MXFP8 values) fed as 8 MXFP4 pieces (decode_mma.cu)
        const bool mx8 = fmt == MOE_ACT_MXFP8;
        uint8_t* dxa = reinterpret_cast<uint8_t*>(at(ws, L.dxa));
        uint8_t* dxa_s = reinterpret_cast<uint8_t*>(at(ws, L.dxa_s));
        uint8_t* dha = reinterpret_cast<uint8_t*>(at(ws, L.dha));
        uint8_t* dha_s = reinterpret_cast<uint8_t*>(at(ws, L.dha_s));
        uint16_t* y_perm = reinterpret_cast<uint16_t*>(at(ws, L.y_perm));
        const bool fused = !norm && mma_decode_fused_sum(T, d);
        if (mma_decode_route_supported(T, d, E, k)) {
            // one launch: the kernel routes its tokens and builds their pieces itself
            const DecRoute r = {x, W_r, b, reinterpret_cast<float*>(at(ws, L.logits)), ids_b, w_b, counts, row_w};
            MOE_CUDA(launch_mma_decode(dxa, dxa_s, dha, dha_s, reinterpret_cast<float*>(at(ws, L.dpart)), plan,
                                       offsets, perm, T, d, E, k, I, W, mx8, y_perm, inv, w_b, fused ? y : nullptr,
                                       ctrl, st, true, &r));
            if (norm) MOE_CUDA(launch_combine_norm(y_perm, inv, w_b, T, k, d, eps, y, st, true));
            else if (!fused) MOE_CUDA(launch_combine(y_perm, inv, w_b, T, k, d, y, st, true));
            return MOE_OK;
        }
        if (route_decode_supported(T, d, E, k)) {
            MOE_CUDA(launch_route_decode(x, W_r, b, T, d, E, k, reinterpret_cast<float*>(at(ws, L.logits)), ids_b, w_b,
                                         counts, offsets, perm, inv, row_w, plan, ctrl, st, true));
        } else {
            MOE_TRY(route_counted(x, W_r, b, T, d, E, k, ids_b, w_b, counts, offsets, perm, inv, row_w, plan, ws, L,
                                  st));
        }
        MOE_CUDA(launch_x_pieces(x, T, d, mx8, dxa, dxa_s, st, true));
        MOE_CUDA(launch_mma_decode(dxa, dxa_s, dha, dha_s, reinterpret_cast<float*>(at(ws, L.dpart)), plan, offsets,
                                   perm, T, d, E, k, I, W, mx8, y_perm, inv, w_b, fused ? y : nullptr, ctrl, st,
                                   true));
        if (norm) MOE_CUDA(launch_combine_norm(y_perm, inv, w_b, T, k, d, eps, y, st, true));
        else if (!fused) MOE_CUDA(launch_combine(y_perm, inv, w_b, T, k, d, y, st, true));
        return MOE_OK;
    }
    if (fmt == MOE_ACT_BF16) {
        if (!gemv_supported(d, I)) return MOE_ERR_UNSUPPORTED_SHAPE;
        if (route_decode_supported(T, d, E, k)) {
            MOE_CUDA(launch_route_decode(x, W_r, b, T, d, E, k, reinterpret_cast<float*>(at(ws, L.logits)), ids_b, w_b,
                                         counts, offsets, perm, inv, row_w, plan, ctrl, st, true));
        } else {
            MOE_TRY(route_counted(x, W_r, b, T, d, E, k, ids_b, w_b, counts, offsets, perm, inv, row_w, plan, ws, L,
                                  st));
        }
        uint16_t* h = reinterpret_cast<uint16_t*>(at(ws, L.h));
        MOE_CUDA(launch_gemv_up(x, perm, offsets, plan, T, d, E, k, I, W, h, st, true));
        if (!norm) {
            MOE_CUDA(launch_gemv_down(h, perm, offsets, plan, row_w, T, d, E, k, I, W, nullptr, y, &ctrl->status, st,
                                      true));
            return MOE_OK;
        }
        uint16_t* y_perm = reinterpret_cast<uint16_t*>(at(ws, L.y_perm));
        MOE_CUDA(launch_gemv_down(h, perm, offsets, plan, nullptr, T, d, E, k, I, W, y_perm, nullptr, &ctrl->status,
                                  st, true));
        MOE_CUDA(launch_combine_norm(y_perm, inv, w_b, T, k, d, eps, y, st, true));
        return MOE_OK;
    }
    uint8_t* xa = reinterpret_cast<uint8_t*>(at(ws, L.xa));
    uint8_t* xa_s = reinterpret_cast<uint8_t*>(at(ws, L.xa_s));
    const bool fp8 = fmt == MOE_ACT_MXFP8;
    const bool nv = W->wfmt == MOE_W_NVFP4;  // kind::mxf4nvf4: operand scales as UE4M3 per 16
    if (nv && !umma_nv_supported(E)) return MOE_ERR_UNSUPPORTED_SHAPE;
    // route (its first launch zeroes the pick counts, its top-k fills them), the permutation in one
    // launch, then each token row quantised once and written to its k padded operand rows
    MOE_TRY(run_route(x, W_r, b, T, d, E, k, ids_b, w_b, ws, L, st, true, plan.counts));
    MOE_CUDA(launch_permute_counted(ids_b, T, E, k, counts, offsets, perm, inv, plan, st, true));
    MOE_CUDA(launch_act_quant_scatter(x, T, d, k, ids_b, inv, offsets, plan, xa, xa_s, fp8, st, true));
    uint8_t* h = reinterpret_cast<uint8_t*>(at(ws, L.h));
    uint8_t* h_s = reinterpret_cast<uint8_t*>(at(ws, L.h_s));
    uint16_t* y_perm = reinterpret_cast<uint16_t*>(at(ws, L.y_perm));
    const uint8_t* up_s = xa_s;
    const uint8_t* down_s = h_s;
    float* xrf = nullptr;
    float* hrf = nullptr;
    if (nv) {
        uint8_t* xa_s16 = reinterpret_cast<uint8_t*>(at(ws, L.xa_s16));
        xrf = reinterpret_cast<float*>(at(ws, L.xrf));
        MOE_CUDA(launch_nv_operand_scales(xa_s, plan.scalars + 2, L.pad_rows, d, xa_s16, xrf, st, true));
        up_s = xa_s16;
    }
    MOE_CUDA(launch_umma_up(xa, up_s, plan, offsets, T, d, E, k, I, L.pad_rows, W, fp8, xrf, h, h_s, &ctrl->status,
                            st, true));
    if (nv) {
        uint8_t* h_s16 = reinterpret_cast<uint8_t*>(at(ws, L.h_s16));
        hrf = reinterpret_cast<float*>(at(ws, L.hrf));
        MOE_CUDA(launch_nv_operand_scales(h_s, plan.scalars + 2, L.pad_rows, I, h_s16, hrf, st, true));
        down_s = h_s16;
    }
    MOE_CUDA(launch_umma_down(h, down_s, plan, offsets, T, d, E, k, I, L.pad_rows, W, fp8, hrf, y_perm,
                              &ctrl->status, st, true));
    if (norm) MOE_CUDA(launch_combine_norm(y_perm, inv, w_b, T, k, d, eps, y, st, true));
    else MOE_CUDA(launch_combine(y_perm, inv, w_b, T, k, d, y, st, true));
    return MOE_OK;
}

moe_status moe_layer_forward(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k, int I,
                             const moe_expert_weights* W, moe_act_fmt fmt, uint16_t* y, int32_t* ids, float* w,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
    return layer_forward(x, W_r, b, T, d, E, k, I, W, fmt, false, 0.f, y, ids, w, ws, ws_bytes, (cudaStream_t)stream);
}

moe_status moe_layer_forward_host(const uint16_t* x_host, const float* W_r, const float* b, int T, int d, int E,
                                  int k, int I, const moe_expert_weights* W, moe_act_fmt fmt, uint16_t* y_host,
                                  int32_t* ids, float* w, uint16_t* x_dev, uint16_t* y_dev, void* ws,
                                  size_t ws_bytes, moe_stream_t stream, moe_stream_t in_stream,
                                  moe_stream_t out_stream) {
    MOE_TRY(check_shape(T, d, E, k, I, fmt));
    if (T == 0) return MOE_OK;
    if (!x_host || !y_host || !x_dev || !y_dev || !aligned(x_dev, 16) || !aligned(y_dev, 16) || x_dev == y_dev)
        return MOE_ERR_INVALID_ARG;
    const cudaStream_t st = (cudaStream_t)stream;
    const size_t bytes = sizeof(uint16_t) * (size_t)T * (size_t)d;
    if (!in_stream || !out_stream) {
        MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st));
        MOE_TRY(layer_forward(x_dev, W_r, b, T, d, E, k, I, W, fmt, false, 0.f, y_dev, ids, w, ws, ws_bytes, st));
        MOE_CUDA(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st));
        return MOE_OK;
    }
    const cudaStream_t is = (cudaStream_t)in_stream, os = (cudaStream_t)out_stream;
    StagingEvents* ex = staging_events(x_dev);
    StagingEvents* ey = staging_events(y_dev);
    if (!ex || !ey) return MOE_ERR_CUDA;
    // a buffer may serve as x_dev in one call and as y_dev in another: each write into it waits for
    // every earlier reader of it (layers reading it as x, copies out of it as y)
    if (ex->consumed_recorded) MOE_CUDA(cudaStreamWaitEvent(is, ex->consumed, 0));  // the last layer read x_dev
    if (ex->drained_recorded) MOE_CUDA(cudaStreamWaitEvent(is, ex->drained, 0));    // the last copy out of it
    MOE_CUDA(cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, is));
    MOE_CUDA(cudaEventRecord(ex->ready, is));
    MOE_CUDA(cudaStreamWaitEvent(st, ex->ready, 0));
    if (ey->drained_recorded) MOE_CUDA(cudaStreamWaitEvent(st, ey->drained, 0));  // the last copy out of y_dev
    if (ey->consumed_recorded) MOE_CUDA(cudaStreamWaitEvent(st, ey->consumed, 0));  // the last layer read of it
    MOE_TRY(layer_forward(x_dev, W_r, b, T, d, E, k, I, W, fmt, false, 0.f, y_dev, ids, w, ws, ws_bytes, st));
    MOE_CUDA(cudaEventRecord(ex->consumed, st));
    ex->consumed_recorded = true;
    MOE_CUDA(cudaEventRecord(ey->ready, st));  // y_dev written
    MOE_CUDA(cudaStreamWaitEvent(os, ey->ready, 0));
    MOE_CUDA(cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, os));
    MOE_CUDA(cudaEventRecord(ey->drained, os));
    ey->drained_recorded = true;
    return MOE_OK;
}

moe_status moe_layer_forward_norm(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E, int k,
                                  int I, const moe_expert_weights* W, moe_act_fmt fmt, float eps, uint16_t* y,
                                  int32_t* ids, float* w, void* ws, size_t ws_bytes, moe_stream_t stream) {
    return layer_forward(x, W_r, b, T, d, E, k, I, W, fmt, true, eps, y, ids, w, ws, ws_bytes, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- dense MXFP4 linear map

static moe_status check_dense_shape(int T, int K, int N, moe_act_fmt fmt) {
    if (T < 0 || K <= 0 || N <= 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (fmt == MOE_ACT_MXFP4 || fmt == MOE_ACT_MXFP8) {
        if (K % 256 != 0 || N % 256 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    } else if (fmt == MOE_ACT_BF16) {
        if (K % 128 != 0 || N % 128 != 0 || !gemv_supported(N, K)) return MOE_ERR_UNSUPPORTED_SHAPE;
    } else {
        return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

size_t moe_dense_workspace_size(int T, int K, int N, moe_act_fmt fmt) {
    if (check_dense_shape(T, K, N, fmt) != MOE_OK) return 0;
    return dense_layout(T, K, N, fmt).total;
}

moe_status moe_dense_linear(const uint16_t* x, int T, int K, int N, const moe_mxfp4_matrix* W, moe_act_fmt fmt,
                            uint16_t* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_dense_shape(T, K, N, fmt));
    if (T == 0) return MOE_OK;
    if (!x || !y || !W || !W->q || !W->s || !aligned(x, 16) || !aligned(y, 16) || !aligned(W->q, 16))
        return MOE_ERR_INVALID_ARG;
    if (fmt == MOE_ACT_MXFP4 && (!W->q_mma || !W->s_mma || !aligned(W->q_mma, 16) || !aligned(W->s_mma, 16)))
        return MOE_ERR_INVALID_ARG;
    if (fmt == MOE_ACT_MXFP8 && (!W->s_mma || !aligned(W->q, 32) || !aligned(W->s_mma, 16))) return MOE_ERR_INVALID_ARG;
    const WsLayout L = dense_layout(T, K, N, fmt);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    MOE_TRY(check_device());
    cudaStream_t st = (cudaStream_t)stream;
    PlanView plan = plan_view(ws, L, 1);
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(at(ws, L.ctrl));
    int32_t* offsets = reinterpret_cast<int32_t*>(at(ws, L.offsets));
    int32_t* perm = reinterpret_cast<int32_t*>(at(ws, L.perm));
    // the matrix as the down weights of one expert that holds every row
    moe_expert_weights Wd = {};
    Wd.down_q = W->q;
    Wd.down_s = W->s;
    Wd.down_q_mma = W->q_mma;
    Wd.down_s_mma = W->s_mma;
    MOE_CUDA(launch_dense_plan(T, plan, offsets, perm, st, false));
    if (fmt == MOE_ACT_BF16) {
        // launched after the plan kernel has completed: the down GEMV reads the plan before its
        // own dependency wait, which needs the plan's writer two launches back
        MOE_CUDA(launch_gemv_down(x, perm, offsets, plan, nullptr, T, N, 1, 1, K, &Wd, y, nullptr, &ctrl->status, st,
                                  false));
        return MOE_OK;
    }
    uint8_t* xa = reinterpret_cast<uint8_t*>(at(ws, L.xa));
    uint8_t* xa_s = reinterpret_cast<uint8_t*>(at(ws, L.xa_s));
    const bool fp8 = fmt == MOE_ACT_MXFP8;
    // each row quantised straight into its operand row (the identity permutation: row t = token t)
    MOE_CUDA(launch_act_quant_scatter(x, T, K, 1, nullptr, nullptr, nullptr, plan, xa, xa_s, fp8, st, true));
    MOE_CUDA(launch_umma_down(xa, xa_s, plan, offsets, T, N, 1, 1, K, L.pad_rows, &Wd, fp8, nullptr, y,
                              &ctrl->status, st, true));
    return MOE_OK;
}

// ---------------------------------------------------------------- synthetic inputs

moe_status moe_synth_weights(uint64_t seed, uint32_t tensor_id, uint32_t expert_first, uint32_t n_experts,
                             int64_t rows, int64_t K, float c, float* out, moe_stream_t stream) {
    if (seed >= (1ull << 32) || tensor_id >= 256 || rows < 0 || K < 0) return MOE_ERR_INVALID_ARG;
    if ((uint64_t)expert_first + n_experts > (1ull << 24)) return MOE_ERR_INVALID_ARG;
    if (rows * K * (int64_t)n_experts == 0) return MOE_OK;
    if (!out) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_device());
    return from_cuda(launch_synth(seed, tensor_id, expert_first, n_experts, rows, K, c, out, (cudaStream_t)stream));
}

}  // extern "C"
