// umma.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a) with
// block-scaled FP4 operands (kind::mxf4: E2M1 values, one E8M0 scale per 32 elements along K).
//
// The expert FFN is a dense contraction per expert (Muse Spark Open explainer, section 9: gate,
// up and down matrices; section 12: each expert computes the tokens gathered for it as one
// batch).  Expert weights and activations are both MXFP4 (DGX Spark news item, section 2: the
// block-scaled 4-bit MXFP4 expert path), so the MMA consumes them without any dequantisation.
//
// Roles: the weights are the MMA "A" operand (M = 128 weight rows per tile) and the tokens of
// one expert are "B" (N = 32..128 tokens), so an expert with few tokens costs a narrow MMA rather
// than a padded 128-token tile.  D[m][n] = sum_k A[m][k] * B[n][k] lives in tensor memory.
//
// One persistent CTA per SM walks the tile list (expert, 128-row weight block, token tile):
//   warp 0    TMA producer: weight and activation tiles (128-byte swizzle) + their block
//             scales (1-D bulk copies of the pre-arranged scale atoms) into a ring of stages;
//   warp 1    allocates tensor memory, copies each stage's scales into it (tcgen05.cp) and
//             issues the MMAs from one thread; tcgen05.commit releases stages / publishes tiles;
//   warps 2-5 epilogue: tcgen05.ld of the accumulators;
//             up:   h = SiLU(g) * u, quantised to MXFP4 along I (one warp = one 32-block),
//                   written as the down GEMM's padded activation operand;
//             down: bf16 expert outputs y_perm in compact permuted row order.
// Every barrier wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, stops issuing work,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include <cuda.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer warp, MMA warp, 4 epilogue warps
constexpr int kTileA = 128 * 128;               // 128 rows x 128 bytes (256 FP4 values) per stage
constexpr int kTileB = 128 * 128;
constexpr int kSfBytes = 1024;                  // two 512-byte scale atoms = 128 rows x 8 scales
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitCycles = 4000000000LL;  // about two seconds at GB300 clocks

template <bool IS_UP>
struct Shape {
    static constexpr int kNumA = IS_UP ? 2 : 1;
    static constexpr int kStages = IS_UP ? 4 : 6;
    static constexpr int kStageBytes = kNumA * kTileA + kTileB + (kNumA + 1) * kSfBytes;
    static constexpr int kSfCols = (kNumA + 1) * 8;  // tensor-memory columns of one stage's scales
    static constexpr int kSfBase = 256;              // accumulators use columns [0, 256)
    static constexpr int kAccBufs = IS_UP ? 1 : 2;
    static constexpr int kSmem = kStages * kStageBytes + 1024 /* alignment */ + 512 /* barriers */;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false when the CTA is
// aborting (another role timed out) or this wait ran out (then it records the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                          long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (*abort_flag) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) {
            set_status(status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand tile with 128-byte swizzle; 8-row groups of
// 8 x 128 bytes lie 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(const void* p) {
    const uint64_t a = smem_u32(p);
    return ((a >> 4) & 0x3FFFull) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Descriptor of one 512-byte scale atom: 32 rows x 16 bytes, no swizzle (8-row core matrices
// of 128 contiguous bytes).
__device__ __forceinline__ uint64_t desc_sf(const void* p) {
    const uint64_t a = smem_u32(p);
    return ((a >> 4) & 0x3FFFull) | (1ull << 16) | ((uint64_t)(128 >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::mxf4 with block scaling: A and B E2M1 (format code 1), K-major,
// UE8M0 scales, D fp32, shape M x N; the scale-factor byte selectors are added per MMA.
__device__ __forceinline__ uint32_t idesc_mxf4(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ kernel arguments / tiles
struct UmmaArgs {
    const uint8_t* sfa0;   // weight scales (tensor-core layout): gate (up) or down
    const uint8_t* sfa1;   // up-matrix scales (up only)
    const uint8_t* sfb;    // activation scales (tensor-core layout, padded rows)
    PlanView plan;
    const int32_t* offsets;
    int E;
    int K;        // contraction length: d (up) or I (down)
    int M_exp;    // weight rows per expert: I (up) or d (down)
    uint8_t* h;   // up: MXFP4 codes [pad_rows][I/2]
    uint8_t* h_s; // up: scales, tensor-core layout
    uint16_t* y_perm;  // down: bf16 [P][d]
    int* status;
};

struct Tile {
    int e, mb, j, n_valid, N, a_row, b_row;
};

__device__ __forceinline__ Tile decode_tile(int t, const UmmaArgs& a) {
    const int MB = a.M_exp / 128;
    int lo = 0, hi = a.E;  // last expert e with ttile_prefix[e] * MB <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.plan.ttile_prefix[mid] * MB <= t) lo = mid; else hi = mid;
    }
    Tile T;
    T.e = lo;
    const int ntt = a.plan.ttile_prefix[lo + 1] - a.plan.ttile_prefix[lo];
    const int local = t - a.plan.ttile_prefix[lo] * MB;
    T.mb = local / ntt;
    T.j = local % ntt;
    T.n_valid = min(kTokTile, a.plan.counts[lo] - T.j * kTokTile);
    T.N = (T.n_valid + 31) / 32 * 32;
    T.a_row = lo * a.M_exp + T.mb * 128;
    T.b_row = a.plan.pad_offsets[lo] + T.j * kTokTile;
    return T;
}

// ------------------------------------------------------------------ the kernel
template <bool IS_UP>
__global__ void __launch_bounds__(kThreads, 1)
umma_grouped_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB, const UmmaArgs args) {
    using S = Shape<IS_UP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kStages * S::kStageBytes);
    uint64_t* empty = full + S::kStages;
    uint64_t* acc_full = empty + S::kStages;     // [kAccBufs]
    uint64_t* acc_empty = acc_full + 2;          // [kAccBufs]
    uint64_t* mma_done = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto stage_a = [&](int s, int i) { return smem + (size_t)s * S::kStageBytes + (size_t)i * kTileA; };
    auto stage_b = [&](int s) { return smem + (size_t)s * S::kStageBytes + S::kNumA * kTileA; };
    auto stage_sf = [&](int s, int i) {  // i < kNumA: weight scales; i == kNumA: activation scales
        return smem + (size_t)s * S::kStageBytes + S::kNumA * kTileA + kTileB + (size_t)i * kSfBytes;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kEpiWarps);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    pdl_wait();  // the plan, offsets and activation operand come from the preceding kernels
    const int MB = args.M_exp / 128;
    const int n_tiles = args.plan.scalars[1] * MB;
    const int KT = args.K / 256;  // K tiles of 256 FP4 values (128 bytes per row)

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            int kiter = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile T = decode_tile(t, args);
                const uint32_t bytes = S::kNumA * kTileA + T.N * 128 + (S::kNumA + 1) * kSfBytes;
                const size_t sfa_base = ((size_t)(T.a_row / 128) * (args.K / 128)) * 512;
                const size_t sfb_base = ((size_t)(T.b_row / 128) * (args.K / 128)) * 512;
                for (int kt = 0; kt < KT; ++kt, ++kiter) {
                    const int s = kiter % S::kStages;
                    const uint32_t ph = (kiter / S::kStages) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[s], bytes);
                    tma_load_2d(stage_a(s, 0), &tmA0, &full[s], kt * 128, T.a_row);
                    if (IS_UP) tma_load_2d(stage_a(s, 1), &tmA1, &full[s], kt * 128, T.a_row);
                    for (int c = 0; c < T.N / 32; ++c)
                        tma_load_2d(stage_b(s) + c * 32 * 128, &tmB, &full[s], kt * 128, T.b_row + 32 * c);
                    bulk_load(stage_sf(s, 0), args.sfa0 + sfa_base + (size_t)kt * 1024, kSfBytes, &full[s]);
                    if (IS_UP) bulk_load(stage_sf(s, 1), args.sfa1 + sfa_base + (size_t)kt * 1024, kSfBytes, &full[s]);
                    bulk_load(stage_sf(s, S::kNumA), args.sfb + sfb_base + (size_t)kt * 1024, kSfBytes, &full[s]);
                }
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA's shared memory is released
                for (int q = 0; q < S::kStages && q < kiter; ++q) {
                    const int it = kiter - 1 - q;
                    mbar_wait(&full[it % S::kStages], (it / S::kStages) & 1, abort_flag, nullptr, 100000000LL);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int kiter = 0, it = 0;
            bool ok = true;
            const uint32_t idesc0 = 0;
            (void)idesc0;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++it) {
                const Tile T = decode_tile(t, args);
                const int buf = it % S::kAccBufs;
                const uint32_t use = it / S::kAccBufs;
                if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, abort_flag, args.status)) break;
                tc_fence_after();
                const uint32_t d0 = tmem + (IS_UP ? 0u : (uint32_t)(buf * 128));
                const uint32_t idesc = idesc_mxf4(128, T.N);
                for (int kt = 0; kt < KT; ++kt, ++kiter) {
                    const int s = kiter % S::kStages;
                    const uint32_t ph = (kiter / S::kStages) & 1;
                    if (!mbar_wait(&full[s], ph, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf_col = tmem + S::kSfBase + s * S::kSfCols;
                    for (int i = 0; i <= S::kNumA; ++i)
                        for (int hh = 0; hh < 2; ++hh)
                            tc_cp_sf(sf_col + i * 8 + hh * 4, desc_sf(stage_sf(s, i) + hh * 512));
                    const uint64_t adesc0 = desc_sw128(stage_a(s, 0));
                    const uint64_t adesc1 = IS_UP ? desc_sw128(stage_a(s, 1)) : 0;
                    const uint64_t bdesc = desc_sw128(stage_b(s));
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        const uint32_t sfid = (uint32_t)(sub & 1) * 2;
                        const uint32_t id = idesc | (sfid << 29) | (sfid << 4);
                        const uint32_t col = (uint32_t)(sub >> 1) * 4;
                        const uint32_t acc = (kt > 0 || sub > 0) ? 1u : 0u;
                        mma_mxf4(d0, adesc0 + 2 * sub, bdesc + 2 * sub, id, sf_col + col, sf_col + S::kNumA * 8 + col,
                                 acc);
                        if (IS_UP)
                            mma_mxf4(tmem + 128, adesc1 + 2 * sub, bdesc + 2 * sub, id, sf_col + 8 + col,
                                     sf_col + S::kNumA * 8 + col, acc);
                    }
                    tc_commit(&empty[s]);  // the stage is free once these MMAs have read it
                }
                if (!ok) break;
                tc_commit(&acc_full[buf]);
            }
            // all MMAs and scale copies issued by this thread have completed once this fires
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, abort_flag, nullptr, 100000000LL);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may access
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        int it = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const Tile T = decode_tile(t, args);
            const int buf = it % S::kAccBufs;
            const uint32_t use = it / S::kAccBufs;
            if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, args.status)) break;
            tc_fence_after();
            const uint32_t acc0 = tmem + lane_base + (IS_UP ? 0u : (uint32_t)(buf * 128));
            const int m = 32 * q + lane;  // weight row within the tile
            for (int c0 = 0; c0 < T.n_valid; c0 += 32) {
                uint32_t g[32];
                tmem_ld32(acc0 + c0, g);
                if (IS_UP) {
                    uint32_t u[32];
                    tmem_ld32(tmem + lane_base + 128 + c0, u);
                    tmem_ld_wait();
                    const int I = args.M_exp;
                    const int blk = (T.mb * 128 + 32 * q) / 32;  // 32-block of h along I
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const int n = c0 + cc;
                        if (n >= T.n_valid) continue;  // uniform across the warp
                        const float gv = __uint_as_float(g[cc]), uv = __uint_as_float(u[cc]);
                        const float hv = gv / (1.f + expf(-gv)) * uv;  // SiLU(g) * u
                        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
                        float inv;
                        const uint32_t sb = mx_scale_from_amax(__uint_as_float(amax_bits), inv);
                        const uint32_t code = e2m1_encode(hv, inv);
                        // gather the 32 nibbles of the warp (lane l = element l of the block)
                        uint32_t v = code | (__shfl_down_sync(0xffffffffu, code, 1) << 4);  // even lanes: a byte
                        v = v | (__shfl_down_sync(0xffffffffu, v, 2) << 8);                 // lanes % 4 == 0
                        v = v | (__shfl_down_sync(0xffffffffu, v, 4) << 16);                // lanes % 8 == 0
                        const uint32_t w1 = __shfl_sync(0xffffffffu, v, 8);
                        const uint32_t w2 = __shfl_sync(0xffffffffu, v, 16);
                        const uint32_t w3 = __shfl_sync(0xffffffffu, v, 24);
                        if (lane == 0) {
                            const size_t row = (size_t)(T.b_row + n);
                            *reinterpret_cast<uint4*>(args.h + row * (I / 2) + (size_t)blk * 16) = make_uint4(v, w1, w2, w3);
                            args.h_s[mma_scale_offset((int64_t)row, blk, I)] = (uint8_t)sb;
                        }
                    }
                } else {
                    tmem_ld_wait();
                    const int d = args.M_exp;
                    const size_t row0 = (size_t)args.offsets[T.e] + (size_t)T.j * kTokTile;
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const int n = c0 + cc;
                        if (n >= T.n_valid) continue;
                        args.y_perm[(row0 + n) * d + T.mb * 128 + m] = f32_to_bf16_bits(__uint_as_float(g[cc]));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    pdl_launch_dependents();
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// 2-D byte tensor [rows][row_bytes], box 128 bytes x box_rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rows == 0) return false;
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

template <bool IS_UP>
cudaError_t launch_grouped(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, const UmmaArgs& args,
                           cudaStream_t st, bool pdl) {
    const void* f = (const void*)umma_grouped_kernel<IS_UP>;
    void* kargs[] = {const_cast<CUtensorMap*>(&a0), const_cast<CUtensorMap*>(&a1), const_cast<CUtensorMap*>(&b),
                     const_cast<UmmaArgs*>(&args)};
    return launch_kernel(f, dim3(sm_count()), dim3(kThreads), Shape<IS_UP>::kSmem, st, pdl, kargs);
}

}  // namespace

cudaError_t launch_umma_up(const uint8_t* xa, const uint8_t* xa_s, PlanView plan, const int32_t* offsets, int T,
                           int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W, uint8_t* h,
                           uint8_t* h_s, int* status, cudaStream_t st, bool pdl) {
    (void)T;
    (void)k;
    if (pad_rows == 0) return cudaSuccess;
    alignas(64) CUtensorMap ma0, ma1, mb;
    if (!make_map(&ma0, W->gate_q, (uint64_t)E * I, d / 2, 128) || !make_map(&ma1, W->up_q, (uint64_t)E * I, d / 2, 128) ||
        !make_map(&mb, xa, (uint64_t)pad_rows, d / 2, 32))
        return cudaErrorInvalidValue;
    UmmaArgs a = {};
    a.sfa0 = W->gate_s_mma;
    a.sfa1 = W->up_s_mma;
    a.sfb = xa_s;
    a.plan = plan;
    a.offsets = offsets;
    a.E = E;
    a.K = d;
    a.M_exp = I;
    a.h = h;
    a.h_s = h_s;
    a.status = status;
    return launch_grouped<true>(ma0, ma1, mb, a, st, pdl);
}

cudaError_t launch_umma_down(const uint8_t* h, const uint8_t* h_s, PlanView plan, const int32_t* offsets, int T,
                             int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W,
                             uint16_t* y_perm, int* status, cudaStream_t st, bool pdl) {
    (void)T;
    (void)k;
    if (pad_rows == 0) return cudaSuccess;
    alignas(64) CUtensorMap ma0, mb;
    if (!make_map(&ma0, W->down_q, (uint64_t)E * d, I / 2, 128) || !make_map(&mb, h, (uint64_t)pad_rows, I / 2, 32))
        return cudaErrorInvalidValue;
    UmmaArgs a = {};
    a.sfa0 = W->down_s_mma;
    a.sfa1 = nullptr;
    a.sfb = h_s;
    a.plan = plan;
    a.offsets = offsets;
    a.E = E;
    a.K = I;
    a.M_exp = d;
    a.y_perm = y_perm;
    a.status = status;
    return launch_grouped<false>(ma0, ma0, mb, a, st, pdl);
}

}  // namespace moe
