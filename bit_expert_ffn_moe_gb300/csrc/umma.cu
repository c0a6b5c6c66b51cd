// umma.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a) with
// block-scaled FP4 operands (kind::mxf4: E2M1 values, one E8M0 scale per 32 elements along K).
//
// The expert FFN is a dense contraction per expert (Muse Spark Open explainer, section 9: gate,
// up and down matrices; section 12: each expert computes the tokens gathered for it as one
// batch).  Expert weights and activations are both MXFP4 (DGX Spark news item, section 2: the
// block-scaled 4-bit MXFP4 expert path), so the MMA consumes them without any dequantisation.
//
// Roles: the tokens of one expert are the MMA "A" operand (M = 128 padded token rows) and 256
// weight rows are "B" (N = 256).  D[m][n] = sum_k A[m][k] * B[n][k] lives in tensor memory with
// lane m = token and column n = weight row, so an epilogue thread owns one token row and one
// tcgen05.ld of 32 columns hands it a whole 32-element block of the output: the SwiGLU result is
// requantised to MXFP4 with no cross-lane traffic, and y rows are written as contiguous 64-byte
// pieces.
//   up:   B = 128 gate rows followed by the same 128 up rows, so D holds g in columns 0..127 and
//         u in columns 128..255 of 128 consecutive intermediate rows.
//   down: B = 256 rows of W_down (256 output features).
// Why N = 256: an MMA reads its operands from shared memory, which the copy engine also has to
// fill, and at M = N = 128 that traffic (not the tensor math) bounds the K loop on GB300; N = 256
// moves 25% fewer shared-memory bytes per flop and hides the scale copies behind the MMAs.  Its
// 256 accumulator columns leave room for one accumulator buffer only (tensor memory holds 512
// columns and the scale slots need the rest), so the MMAs wait while the epilogue drains it.
// Tiles are (expert e, token tile j, weight block p) with p fastest: CTAs that run at the same
// time share a token tile through L2 and walk the expert's weight blocks, each of which stays in
// L2 while the expert's other token tiles use it.
//
// One persistent CTA per SM walks the tile list:
//   warp 0    producer: per K step, six bulk copies (the copy engine) into a ring of stages --
//             the 16 KB token tile, two 16 KB weight tiles and their 1 KB scale pieces.  All
//             operands are stored pre-arranged in the tensor-core layouts (code tiles already
//             in the 128-byte swizzle, scale atoms), so every piece is one contiguous copy; on
//             GB300 these run markedly faster than 2-D tensor boxes of 128-byte rows, from L2 as
//             well as from HBM;
//   warp 1    allocates tensor memory; with all 32 lanes, copies each stage's scales into it
//             (tcgen05.cp) and issues the MMAs (one elected lane); tcgen05.commit frees stages
//             and publishes the accumulator;
//   warps 2-9 epilogue: two warps per tensor-memory lane quarter (32 token rows), each taking
//             half of the accumulator columns into registers and freeing tensor memory at once,
//             then converting and storing them while the next tile's MMAs run.
// Every barrier wait is bounded: on expiry the CTA records MOE_ERR_TIMEOUT, stops issuing work,
// waits (bounded) for its own copies and MMAs, frees tensor memory and exits.
#include <cuda.h>

#include <mutex>

#include "tcgen05.cuh"

namespace moe {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer warp, MMA warp, 8 epilogue warps
constexpr int kTile = 128 * 128;                // 128 rows x 128 bytes (256 FP4 values)
constexpr int kAtom = 512;                      // scale atom: 128 rows x 4 scales
constexpr int kStages = 4;
// MMA kinds of the grouped GEMMs: MXFP4 tokens x MXFP4 weights (kind::mxf4), MXFP8 tokens x MXFP4
// weights (kind::mxf8f6f4), MXFP4 tokens x NVFP4 weights (kind::mxf4nvf4, 16-element UE4M3 scales)
constexpr int kMxf4 = 0, kMxf8 = 1, kNvf4 = 2;
// Bytes of a stage: the A tile, two B tiles (256 weight rows) and the scale atoms -- kind::mxf4:
// 256 values of K, 2 atoms of A scales and 2 + 2 of B scales; kind::mxf8f6f4: 128 values of K (E4M3
// tokens, the FP4 weights widened to one byte per value), one atom each (A's in a 2-atom slot, so
// that every stage starts on the 1024-byte boundary the 128-byte swizzle needs); kind::mxf4nvf4:
// 256 values of K with 16-element scales, 4 atoms of A scales and 4 + 4 of B scales.
template <int KIND>
__host__ __device__ constexpr int stage_bytes() { return 3 * kTile + (KIND == kMxf8 ? 4 : KIND == kNvf4 ? 12 : 6) * kAtom; }
static_assert(stage_bytes<kMxf4>() % 1024 == 0 && stage_bytes<kMxf8>() % 1024 == 0 &&
                  stage_bytes<kNvf4>() % 1024 == 0,
              "stages start on 1024-byte boundaries");
// bytes an MXFP8 stage's copies signal: a widened weight box counts its packed global bytes (8 KB)
constexpr int kStageTx8 = kTile + 2 * (kTile / 2) + 3 * kAtom;
constexpr int kAccBufs = 1;
constexpr int kAccCols = 256;
constexpr int kSfBase = kAccBufs * kAccCols;  // scale slots after the accumulator
// tensor-memory scale columns per stage: A 8 + B 16 (A 16 + B 32 for 16-element scales)
template <int KIND>
__host__ __device__ constexpr int sf_cols() { return KIND == kNvf4 ? 48 : 24; }
constexpr uint32_t kTmemCols = 512;
constexpr int kBarBytes = 256;
static_assert(kSfBase + kStages * sf_cols<kNvf4>() <= (int)kTmemCols, "tensor memory budget");

template <int KIND>
constexpr size_t smem_bytes(int E) {
    return (size_t)kStages * stage_bytes<KIND>() + 1024 /* alignment */ + kBarBytes +
           (size_t)4 * (E + 1) * sizeof(int32_t);
}
constexpr size_t kMaxSmem = 232448;  // 227 KB per CTA

// ------------------------------------------------------------------ kernel arguments / tiles
struct UmmaArgs {
    CUtensorMap tmap_b0;  // MXFP8: B rows 0..127 / 128..255 read from the canonical weight codes
    CUtensorMap tmap_b1;
    const uint8_t* qa;   // token-operand code tiles (padded rows)
    const uint8_t* sfa;  // token-operand scales (tensor-core layout over padded rows)
    const uint8_t* qb0;  // B rows 0..127: gate (up) or down code tiles
    const uint8_t* sfb0;
    const uint8_t* qb1;  // B rows 128..255: up (up) or down code tiles
    const uint8_t* sfb1;
    int b1_step;         // 128-row block of B rows 128..255 relative to rows 0..127: 0 (up), 1 (down)
    PlanView plan;
    const int32_t* offsets;
    int E;
    int K;       // contraction length: d (up) or I (down)
    int NB;      // weight blocks per expert: I/128 (up) or d/256 (down)
    int n_out;   // output row length: I (h, up) or d (y_perm, down)
    uint8_t* h;    // up: MXFP4 (MXFP8) code tiles of [pad_rows][I]
    uint8_t* h_s;  // up: scales, tensor-core layout
    uint16_t* y_perm;  // down: bf16 [P][d]
    int* status;
    // NVFP4 weights: per padded A row the power-of-two factor its UE4M3 scales leave out, and the
    // weight matrices' global scales per expert (B rows 0..127 / 128..255)
    const float* rf;
    const float* gs0;
    const float* gs1;
};

// Plan copied to shared memory once per CTA.
struct SmemPlan {
    int32_t* ttile_prefix;  // [E+1]
    int32_t* counts;        // [E]
    int32_t* pad_offsets;   // [E+1]
    int32_t* offsets;       // [E+1]
};

struct Tile {
    int e, j, p, n_valid, a_row, y_row, b_rb;
};

// Advance `e` (monotone over a CTA's tiles) to the expert owning tile t and fill in the tile.
template <bool IS_UP>
__device__ __forceinline__ Tile decode_tile(int t, int& e, const SmemPlan& sp, const UmmaArgs& a) {
    while (sp.ttile_prefix[e + 1] * a.NB <= t) ++e;
    Tile T;
    T.e = e;
    const int local = t - sp.ttile_prefix[e] * a.NB;
    T.j = local / a.NB;
    T.p = local % a.NB;
    T.n_valid = min(kTokTile, sp.counts[e] - T.j * kTokTile);
    T.a_row = sp.pad_offsets[e] + T.j * kTokTile;
    T.y_row = sp.offsets[e] + T.j * kTokTile;
    // 128-row block of B rows 0..127 in the weight matrix ([E*I] rows up, [E*d] rows down)
    T.b_rb = IS_UP ? e * a.NB + T.p : e * 2 * a.NB + 2 * T.p;
    return T;
}

// ------------------------------------------------------------------ the kernel
template <bool IS_UP, int KIND>
__global__ void __launch_bounds__(kThreads, 1) umma_grouped_kernel(const __grid_constant__ UmmaArgs args) {
    constexpr bool FP8 = KIND == kMxf8, NV = KIND == kNvf4;
    constexpr int kStageBytes = stage_bytes<KIND>();
    constexpr int kSfCols = sf_cols<KIND>();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;       // [kAccBufs]
    uint64_t* acc_empty = acc_full + kAccBufs;  // [kAccBufs]
    uint64_t* mma_done = acc_empty + kAccBufs;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int32_t* plan_smem = reinterpret_cast<int32_t*>(smem + kStages * kStageBytes + kBarBytes);
    const int E = args.E;
    SmemPlan sp;
    sp.ttile_prefix = plan_smem;
    sp.counts = plan_smem + (E + 1);
    sp.pad_offsets = plan_smem + 2 * (E + 1);
    sp.offsets = plan_smem + 3 * (E + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    auto stage_a = [&](int s) { return smem + (size_t)s * kStageBytes; };
    auto stage_b = [&](int s) { return smem + (size_t)s * kStageBytes + kTile; };  // 256 rows
    auto stage_sfa = [&](int s) { return smem + (size_t)s * kStageBytes + 3 * kTile; };
    // B scales: rows 0..127, then rows 128..255 (each 2 atoms; 1 for 8-bit tokens, after A's 2-atom
    // slot; 4 with 16-element scales)
    auto stage_sfb = [&](int s) { return smem + (size_t)s * kStageBytes + 3 * kTile + (NV ? 4 : 2) * kAtom; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
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

    pdl_wait();  // the plan, offsets and token operand come from the preceding kernels
    for (int i = threadIdx.x; i <= E; i += kThreads) {
        sp.ttile_prefix[i] = args.plan.ttile_prefix[i];
        sp.pad_offsets[i] = args.plan.pad_offsets[i];
        sp.offsets[i] = args.offsets[i];
        if (i < E) sp.counts[i] = args.plan.counts[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_tiles = args.plan.scalars[1] * args.NB;
    const int KT = args.K / (FP8 ? 128 : 256);  // K steps: 128 bytes of every operand row
    const int atoms_per_rowblk = args.K / (NV ? 64 : 128);

    if (warp == 0) {
        // ---------------------------------------------------------- copy producer
        if (lane == 0) {
            int kiter = 0, e = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                const Tile T = decode_tile<IS_UP>(t, e, sp, args);
                const size_t rb1 = (size_t)T.b_rb + args.b1_step;
                const uint8_t* qa = args.qa + (size_t)(T.a_row / 128) * KT * kTile;
                const uint8_t* qb0 = args.qb0 + (size_t)T.b_rb * KT * kTile;
                const uint8_t* qb1 = args.qb1 + rb1 * KT * kTile;
                const uint8_t* sfa = args.sfa + ((size_t)(T.a_row / 128) * atoms_per_rowblk) * kAtom;
                const uint8_t* sfb0 = args.sfb0 + ((size_t)T.b_rb * atoms_per_rowblk) * kAtom;
                const uint8_t* sfb1 = args.sfb1 + (rb1 * atoms_per_rowblk) * kAtom;
                for (int kt = 0; kt < KT; ++kt, ++kiter) {
                    const int s = kiter % kStages;
                    const uint32_t ph = (kiter / kStages) & 1;
                    if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    if (FP8) {
                        // the weight boxes come widened from the canonical codes through the tensor
                        // maps (128 values x 128 rows, 16 KB each in shared memory)
                        mbar_arrive_expect_tx(&full[s], kStageTx8);
                        bulk_load(stage_a(s), qa + (size_t)kt * kTile, kTile, &full[s]);
                        tma_load_2d(stage_b(s), &args.tmap_b0, 128 * kt, 128 * T.b_rb, &full[s]);
                        tma_load_2d(stage_b(s) + kTile, &args.tmap_b1, 128 * kt, 128 * (int)rb1, &full[s]);
                        bulk_load(stage_sfa(s), sfa + (size_t)kt * kAtom, kAtom, &full[s]);
                        bulk_load(stage_sfb(s), sfb0 + (size_t)kt * kAtom, kAtom, &full[s]);
                        bulk_load(stage_sfb(s) + kAtom, sfb1 + (size_t)kt * kAtom, kAtom, &full[s]);
                        continue;
                    }
                    constexpr int kStageAtoms = NV ? 4 : 2;  // scale atoms per operand block per K step
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    bulk_load(stage_a(s), qa + (size_t)kt * kTile, kTile, &full[s]);
                    bulk_load(stage_b(s), qb0 + (size_t)kt * kTile, kTile, &full[s]);
                    bulk_load(stage_b(s) + kTile, qb1 + (size_t)kt * kTile, kTile, &full[s]);
                    bulk_load(stage_sfa(s), sfa + (size_t)kt * kStageAtoms * kAtom, kStageAtoms * kAtom, &full[s]);
                    bulk_load(stage_sfb(s), sfb0 + (size_t)kt * kStageAtoms * kAtom, kStageAtoms * kAtom, &full[s]);
                    bulk_load(stage_sfb(s) + kStageAtoms * kAtom, sfb1 + (size_t)kt * kStageAtoms * kAtom,
                              kStageAtoms * kAtom, &full[s]);
                }
            }
            if (*abort_flag) {
                // let the copies already issued land before the CTA's shared memory is released
                // (bounded waits that the abort flag does not cut short)
                volatile int never = 0;
                for (int q = 0; q < kStages && q < kiter; ++q) {
                    const int it = kiter - 1 - q;
                    mbar_wait(&full[it % kStages], (it / kStages) & 1, &never, nullptr, 100000000LL);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer (whole warp)
        int kiter = 0, it = 0;
        bool ok = true;
        const uint32_t idesc = FP8 ? idesc_mxf8_e4m3_e2m1(128, 256)
                                   : NV ? idesc_mxf4nvf4_ue4m3(128, 256) : idesc_mxf4(128, 256);
        for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++it) {
            const int buf = it % kAccBufs;
            const uint32_t use = it / kAccBufs;
            if (!mbar_wait_warp(&acc_empty[buf], (use & 1) ^ 1, abort_flag, args.status)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(buf * kAccCols);
            for (int kt = 0; kt < KT; ++kt, ++kiter) {
                const int s = kiter % kStages;
                const uint32_t ph = (kiter / kStages) & 1;
                if (!mbar_wait_warp(&full[s], ph, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sf = tmem + kSfBase + s * kSfCols;
                // the stage is free once these MMAs have read it
                if (NV) {
                    stage_scales_nv_to_tmem(sf, desc_sf(stage_sfa(s)), desc_sf(stage_sfb(s)),
                                            desc_sf(stage_sfb(s) + 4 * kAtom));
                    stage_mmas_nv_commit(d_tmem, desc_sw128(stage_a(s)), desc_sw128(stage_b(s)), idesc, sf,
                                         kt > 0 ? 1u : 0u, &empty[s]);
                    continue;
                }
                if (FP8) {
                    stage_scales8_to_tmem(sf, desc_sf(stage_sfa(s)), desc_sf(stage_sfb(s)), desc_sf(stage_sfb(s) + kAtom));
                    stage_mmas8_commit(d_tmem, desc_sw128(stage_a(s)), desc_sw128(stage_b(s)), idesc, sf,
                                       kt > 0 ? 1u : 0u, &empty[s]);
                    continue;
                }
                stage_scales_to_tmem(sf, desc_sf(stage_sfa(s)), desc_sf(stage_sfa(s) + kAtom), desc_sf(stage_sfb(s)),
                                     desc_sf(stage_sfb(s) + 2 * kAtom), desc_sf(stage_sfb(s) + kAtom),
                                     desc_sf(stage_sfb(s) + 3 * kAtom));
                stage_mmas_commit(d_tmem, desc_sw128(stage_a(s)), desc_sw128(stage_b(s)), idesc,
                                  idesc | (2u << 29) | (2u << 4), sf, kt > 0 ? 1u : 0u, &empty[s]);
            }
            if (!ok) break;
            tc_commit(&acc_full[buf]);
        }
        // all MMAs and scale copies issued by this warp have completed once this fires
        tc_commit(mma_done);
        volatile int never = 0;  // wait even when aborting: tensor memory is freed next
        mbar_wait_warp(mma_done, 0, &never, nullptr, 100000000LL);
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                // tensor-memory lane quarter this warp may access
        const int half = (warp - 2) / 4;       // half of the accumulator columns it drains
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const int m = 32 * q + lane;  // token row within the tile
        int it = 0, e = 0;
        for (int t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const Tile T = decode_tile<IS_UP>(t, e, sp, args);
            const int buf = it % kAccBufs;
            const uint32_t use = it / kAccBufs;
            if (!mbar_wait(&acc_full[buf], use & 1, abort_flag, args.status)) break;
            tc_fence_after();
            const uint32_t acc = tmem + lane_base + (uint32_t)(buf * kAccCols);
            // Copy this warp's 128 accumulator columns to registers and free tensor memory at once,
            // so that the next tile's MMAs run while these values are converted and stored.
            uint32_t v[4][32];
            if (IS_UP) {  // g and u of chunks 2*half, 2*half + 1
                tmem_ld32(acc + 32 * (2 * half), v[0]);
                tmem_ld32(acc + 32 * (2 * half + 1), v[1]);
                tmem_ld32(acc + 128 + 32 * (2 * half), v[2]);
                tmem_ld32(acc + 128 + 32 * (2 * half + 1), v[3]);
            } else {  // chunks 4*half .. 4*half + 3
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(acc + 32 * (4 * half + c), v[c]);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            // NVFP4 weights: the accumulators miss the A row's power-of-two factor and the weight
            // matrices' global scales
            float f0 = 1.f, f1 = 1.f;
            if (NV) {
                const float r = __ldg(args.rf + T.a_row + m);
                f0 = r * __ldg(args.gs0 + T.e);
                f1 = r * __ldg(args.gs1 + T.e);
            }
            if (IS_UP) {
                const int I = args.n_out;
                const size_t row = (size_t)T.a_row + m;  // every padded row is written (zeros there)
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float gv = __uint_as_float(v[cc][i]), uv = __uint_as_float(v[2 + cc][i]);
                        if (NV) {
                            gv *= f0;
                            uv *= f1;
                        }
                        hv[i] = __fdividef(gv, 1.f + __expf(-gv)) * uv;  // SiLU(g) * u
                    }
                    const int blk = 4 * T.p + 2 * half + cc;  // 32-block of h along I
                    uint32_t sb;
                    if (FP8) {
                        uint4 c8[2];
                        sb = mx8_block_encode(hv, c8);
                        *reinterpret_cast<uint4*>(args.h + mma8_tile_offset((int64_t)row, 2 * blk, I)) = c8[0];
                        *reinterpret_cast<uint4*>(args.h + mma8_tile_offset((int64_t)row, 2 * blk + 1, I)) = c8[1];
                    } else {
                        uint4 codes;
                        sb = mx_block_encode(hv, codes);
                        *reinterpret_cast<uint4*>(args.h + mma_tile_offset((int64_t)row, blk, I)) = codes;
                    }
                    args.h_s[mma_scale_offset((int64_t)row, blk, I)] = (uint8_t)sb;
                }
            } else {
                // Each thread holds 32 columns (64 bytes) of its own token row per chunk; after a
                // 4 x 4 transpose of 16-byte pieces inside groups of four lanes, store j writes 64
                // contiguous bytes of 8 rows (row 4g + j of each group) instead of 16 bytes of 32.
                const int d = args.n_out;
                const int rbase = 32 * q + 4 * (lane >> 2), piece = lane & 3;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 pc[4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        uint32_t w4[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[c][8 * a + 2 * i]) * f0,
                                                                      __uint_as_float(v[c][8 * a + 2 * i + 1]) * f0);
                            w4[i] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                        pc[a] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                    transpose4_pieces(pc, lane);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = rbase + j;  // token row within the tile
                        if (r < T.n_valid)
                            *reinterpret_cast<uint4*>(args.y_perm + ((size_t)T.y_row + r) * d + (size_t)T.p * 256 +
                                                      32 * (4 * half + c) + 8 * piece) = pc[j];
                    }
                }
            }
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
template <bool IS_UP, int KIND>
cudaError_t launch_grouped(const UmmaArgs& args, cudaStream_t st, bool pdl) {
    const void* f = (const void*)umma_grouped_kernel<IS_UP, KIND>;
    void* kargs[] = {const_cast<UmmaArgs*>(&args)};
    return launch_kernel(f, dim3(sm_count()), dim3(kThreads), smem_bytes<KIND>(args.E), st, pdl, kargs);
}

// Tensor map of a canonical MXFP4 code matrix q[rows][K/2] read in boxes of 128 values x 128 rows,
// each 4-bit value given a byte's place in shared memory (16 values in 8 bytes, then 8 empty
// bytes: the FP4 operand layout of kind::mxf8f6f4) with the 128-byte swizzle.  q must be 32-byte
// aligned and K a multiple of 128.
cudaError_t fp4_widening_map(CUtensorMap* m, const uint8_t* q, int64_t rows, int64_t K) {
    encode_tiled_fn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    const cuuint32_t box[2] = {128, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(q), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

// The driver's tensor-map encoder, taken through the runtime's entry-point query.
encode_tiled_fn tensor_map_encoder() {
    static encode_tiled_fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &r) ==
                cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<encode_tiled_fn>(f);
    });
    return fn;
}

bool umma_nv_supported(int E) { return smem_bytes<kNvf4>(E) <= kMaxSmem; }

cudaError_t launch_umma_up(const uint8_t* xa, const uint8_t* xa_s, PlanView plan, const int32_t* offsets, int T,
                           int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W, bool fp8,
                           const float* rf, uint8_t* h, uint8_t* h_s, int* status, cudaStream_t st, bool pdl) {
    (void)T;
    (void)k;
    if (pad_rows == 0) return cudaSuccess;
    UmmaArgs a = {};
    a.qa = xa;
    a.sfa = xa_s;
    a.qb0 = W->gate_q_mma;
    a.sfb0 = W->gate_s_mma;
    a.qb1 = W->up_q_mma;
    a.sfb1 = W->up_s_mma;
    a.b1_step = 0;
    a.plan = plan;
    a.offsets = offsets;
    a.E = E;
    a.K = d;
    a.NB = I / 128;
    a.n_out = I;
    a.h = h;
    a.h_s = h_s;
    a.status = status;
    if (W->wfmt == MOE_W_NVFP4) {
        a.rf = rf;
        a.gs0 = W->gate_gs;
        a.gs1 = W->up_gs;
        return launch_grouped<true, kNvf4>(a, st, pdl);
    }
    if (!fp8) return launch_grouped<true, kMxf4>(a, st, pdl);
    cudaError_t err = fp4_widening_map(&a.tmap_b0, W->gate_q, (int64_t)E * I, d);
    if (err == cudaSuccess) err = fp4_widening_map(&a.tmap_b1, W->up_q, (int64_t)E * I, d);
    return err == cudaSuccess ? launch_grouped<true, kMxf8>(a, st, pdl) : err;
}

cudaError_t launch_umma_down(const uint8_t* h, const uint8_t* h_s, PlanView plan, const int32_t* offsets, int T,
                             int d, int E, int k, int I, int64_t pad_rows, const moe_expert_weights* W, bool fp8,
                             const float* rf, uint16_t* y_perm, int* status, cudaStream_t st, bool pdl) {
    (void)T;
    (void)k;
    if (pad_rows == 0) return cudaSuccess;
    UmmaArgs a = {};
    a.qa = h;
    a.sfa = h_s;
    a.qb0 = W->down_q_mma;
    a.sfb0 = W->down_s_mma;
    a.qb1 = W->down_q_mma;
    a.sfb1 = W->down_s_mma;
    a.b1_step = 1;
    a.plan = plan;
    a.offsets = offsets;
    a.E = E;
    a.K = I;
    a.NB = d / 256;
    a.n_out = d;
    a.y_perm = y_perm;
    a.status = status;
    if (W->wfmt == MOE_W_NVFP4) {
        a.rf = rf;
        a.gs0 = a.gs1 = W->down_gs;
        return launch_grouped<false, kNvf4>(a, st, pdl);
    }
    if (!fp8) return launch_grouped<false, kMxf4>(a, st, pdl);
    cudaError_t err = fp4_widening_map(&a.tmap_b0, W->down_q, (int64_t)E * d, I);
    if (err == cudaSuccess) a.tmap_b1 = a.tmap_b0;
    return err == cudaSuccess ? launch_grouped<false, kMxf8>(a, st, pdl) : err;
}

}  // namespace moe
