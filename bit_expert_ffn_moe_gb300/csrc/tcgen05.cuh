// tcgen05.cuh -- PTX wrappers of the 5th-generation tensor cores (sm_103a) shared by the grouped
// expert GEMMs: tensor-memory scale copies, block-scaled MMAs (kind::mxf4: E2M1 operands;
// kind::mxf8f6f4: E4M3 tokens x E2M1 weights; one E8M0 scale per 32 elements in both;
// kind::mxf4nvf4: E2M1 operands with one UE4M3 scale per 16 elements),
// shared-memory and instruction descriptors, tensor-map copies, tensor-memory loads and the
// commit / fence instructions.  The bit fields are the ones the PTX ISA defines.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

constexpr int kStageTileBytes = 128 * 128;  // operand tile: 128 rows x 128 bytes (256 FP4 values)
constexpr int kScaleAtomBytes = 512;        // scale atom: 128 rows x 4 scales

// One K step of 256 values: the six scale-atom copies of the stage into tensor memory, then the
// four K = 64 MMAs and the commit that frees the stage, each group issued by one elected lane.
// Scale slot of a stage (24 columns from sf): A scales of K values 0..127 at sf, 128..255 at
// sf + 4; B scales of K values 0..127 at sf + 8 (rows 0..127) and sf + 12 (rows 128..255), of
// K values 128..255 at sf + 16 and sf + 20.
__device__ __forceinline__ void stage_scales_to_tmem(uint32_t sf, uint64_t a0, uint64_t a1, uint64_t b00,
                                                     uint64_t b10, uint64_t b01, uint64_t b11) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%2], %3;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%6], %7;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%8], %9;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%10], %11;\n\t}" ::"r"(sf),
        "l"(a0), "r"(sf + 4), "l"(a1), "r"(sf + 8), "l"(b00), "r"(sf + 12), "l"(b10), "r"(sf + 16), "l"(b01),
        "r"(sf + 20), "l"(b11)
        : "memory");
}

// MMAs of one stage: sub-steps 0..3 use A/B descriptors advanced by 32 bytes each and scale bytes
// (sub & 1) * 2 of the A/B scale columns of K values 0..127 (subs 0, 1) or 128..255 (subs 2, 3).
__device__ __forceinline__ void stage_mmas_commit(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id0, uint32_t id2,
                                                  uint32_t sf, uint32_t accumulate, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, q;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "setp.eq.b32 q, %5, %5;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%6], [%7], p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %8, %9, %4, [%6], [%7], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %10, %11, %3, [%12], [%13], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %14, %15, %4, [%12], [%13], q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%16];\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(id0), "r"(id2), "r"(accumulate), "r"(sf), "r"(sf + 8), "l"(ad + 2), "l"(bd + 2),
        "l"(ad + 4), "l"(bd + 4), "r"(sf + 4), "r"(sf + 16), "l"(ad + 6), "l"(bd + 6), "r"(smem_u32(bar))
        : "memory");
}

// 8-bit operands (kind::mxf8f6f4, one E8M0 scale per 32 values, K = 32 per MMA): one K step of 128
// values.  Scale slot: A scales at sf (4 columns), B scales of rows 0..127 at sf + 4 and of rows
// 128..255 at sf + 8.
__device__ __forceinline__ void stage_scales8_to_tmem(uint32_t sf, uint64_t a, uint64_t b0, uint64_t b1) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%2], %3;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t}" ::"r"(sf),
        "l"(a), "r"(sf + 4), "l"(b0), "r"(sf + 8), "l"(b1)
        : "memory");
}

// The four K = 32 MMAs of an 8-bit stage: sub-step i reads the operands 32 bytes further along
// each row and scale byte i of the A and B scale columns (selectors in instruction-descriptor
// bits 29-30 and 4-5), then the commit that frees the stage.
__device__ __forceinline__ void stage_mmas8_commit(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sf,
                                                   uint32_t accumulate, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, q;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %7, %8, %9, [%5], [%6], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %10, %11, %12, [%5], [%6], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %13, %14, %15, [%5], [%6], q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%16];\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(sf), "r"(sf + 4), "l"(ad + 2), "l"(bd + 2),
        "r"(idesc | (1u << 29) | (1u << 4)), "l"(ad + 4), "l"(bd + 4), "r"(idesc | (2u << 29) | (2u << 4)),
        "l"(ad + 6), "l"(bd + 6), "r"(idesc | (3u << 29) | (3u << 4)), "r"(smem_u32(bar))
        : "memory");
}

// 4-bit operands with 16-element UE4M3 scales (kind::mxf4nvf4, scale_vec::4X, K = 64 per MMA): one
// K step of 256 values takes four scale atoms per 128 rows (each atom: 4 scales of every row, one
// MMA's K range).  Scale slot (48 columns from sf): A atom i at sf + 4i, B atoms of K range i at
// sf + 16 + 8i (rows 0..127) and sf + 20 + 8i (rows 128..255).  a, b0, b1: the stage's first
// atoms (A, B rows 0..127, B rows 128..255), each followed by its next three.
__device__ __forceinline__ void stage_scales_nv_to_tmem(uint32_t sf, uint64_t a, uint64_t b0, uint64_t b1) {
    // a descriptor's start address field counts 16-byte units: one 512-byte atom is 32
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%2], %3;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%4], %5;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%6], %7;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%8], %9;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%10], %11;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%12], %13;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%14], %15;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%16], %17;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%18], %19;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%20], %21;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%22], %23;\n\t}" ::"r"(sf),
        "l"(a), "r"(sf + 4), "l"(a + 32), "r"(sf + 8), "l"(a + 64), "r"(sf + 12), "l"(a + 96), "r"(sf + 16),
        "l"(b0), "r"(sf + 20), "l"(b1), "r"(sf + 24), "l"(b0 + 32), "r"(sf + 28), "l"(b1 + 32), "r"(sf + 32),
        "l"(b0 + 64), "r"(sf + 36), "l"(b1 + 64), "r"(sf + 40), "l"(b0 + 96), "r"(sf + 44), "l"(b1 + 96)
        : "memory");
}

// The four K = 64 MMAs of a stage with 16-element UE4M3 scales (scale byte selectors 0: an MMA
// reads all four bytes of its scale columns), then the commit that frees the stage.
__device__ __forceinline__ void stage_mmas_nv_commit(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t sf,
                                                     uint32_t accumulate, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, q;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %7, %8, %3, [%9], [%10], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %11, %12, %3, [%13], [%14], q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %15, %16, %3, [%17], [%18], q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%19];\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate), "r"(sf), "r"(sf + 16), "l"(ad + 2), "l"(bd + 2), "r"(sf + 4),
        "r"(sf + 24), "l"(ad + 4), "l"(bd + 4), "r"(sf + 8), "r"(sf + 32), "l"(ad + 6), "l"(bd + 6), "r"(sf + 12),
        "r"(sf + 40), "r"(smem_u32(bar))
        : "memory");
}

// mbar_wait by every lane of a warp with a warp-uniform verdict.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status,
                                               long long limit = kWaitCycles) {
    const bool ok = mbar_wait(bar, parity, abort_flag, status, limit);
    return __all_sync(0xffffffffu, ok);
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

// Instruction descriptor of kind::mxf4nvf4 with 16-element block scaling: A and B E2M1 (format
// code 1), K-major, UE4M3 scales (bit 23 clear), D fp32, shape M x N.
__device__ __forceinline__ uint32_t idesc_mxf4nvf4_ue4m3(int M, int N) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E4M3 (format code 0), B E2M1
// (format code 5, read from the widened shared-memory layout: 16 values in 8 bytes, then 8 empty
// bytes), K-major, UE8M0 scales, D fp32, shape M x N; scale byte selectors added per MMA.
__device__ __forceinline__ uint32_t idesc_mxf8_e4m3_e2m1(int M, int N) {
    return (0u << 7) | (5u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::f16 with bf16 A and B (format code 1), K-major, D fp32 (format
// code 1), shape M x N, no sparsity, negation or saturation.
__device__ __forceinline__ uint32_t idesc_f16_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// One stage of 64 bf16 values of K: the four K = 16 MMAs (descriptors advanced by 32 bytes each);
// `accumulate` = 0 makes the first one overwrite the accumulator.  Then the commit that frees the
// stage.
__device__ __forceinline__ void stage_mmas_bf16_commit(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc,
                                                       uint32_t accumulate, uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, q;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %3, 0;\n\t"
        "setp.eq.b32 q, %3, %3;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %4, p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %6, %4, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %8, %4, q;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %9, %10, %4, q;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%11];\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(accumulate), "r"(idesc), "l"(ad + 2), "l"(bd + 2), "l"(ad + 4), "l"(bd + 4), "l"(ad + 6),
        "l"(bd + 6), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tensor-map copy of one box into shared memory, completing on an mbarrier (x: innermost
// coordinate in elements, y: row).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The MMA warp runs its loop with all 32 lanes (warp-uniform control flow, so every operand is
// warp-uniform) and each tcgen05 instruction is issued by one lane chosen by elect.sync inside
// the instruction's own asm block.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
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

// 4 x 4 transpose of 16-byte pieces among the lanes of each aligned group of four: on entry lane
// 4g + i holds pieces p[0..3] of row i of the group, on return p[j] = piece i of row j.  Two xor
// stages (swap the off-diagonal 2 x 2 blocks, then the off-diagonal pieces inside each block).
__device__ __forceinline__ void transpose4_pieces(uint4 (&p)[4], int lane) {
    const bool i1 = (lane >> 1) & 1, i0 = lane & 1;
#pragma unroll
    for (int j0 = 0; j0 < 2; ++j0) {  // stage A: exchange pieces whose bit 1 differs from the lane's
        uint4& lo = p[j0];
        uint4& hi = p[2 | j0];
        uint4 snd = i1 ? lo : hi;
        uint4 rcv;
        rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, 2);
        rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, 2);
        rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, 2);
        rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, 2);
        if (i1) lo = rcv; else hi = rcv;
    }
#pragma unroll
    for (int j1 = 0; j1 < 2; ++j1) {  // stage B: exchange pieces whose bit 0 differs from the lane's
        uint4& lo = p[2 * j1];
        uint4& hi = p[2 * j1 + 1];
        uint4 snd = i0 ? lo : hi;
        uint4 rcv;
        rcv.x = __shfl_xor_sync(0xffffffffu, snd.x, 1);
        rcv.y = __shfl_xor_sync(0xffffffffu, snd.y, 1);
        rcv.z = __shfl_xor_sync(0xffffffffu, snd.z, 1);
        rcv.w = __shfl_xor_sync(0xffffffffu, snd.w, 1);
        if (i0) lo = rcv; else hi = rcv;
    }
}

// The driver's tensor-map encoder (cuTensorMapEncodeTiled), taken through the runtime's entry-point
// query so that the library needs no link-time dependency on the driver library; null when
// unavailable.
typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
encode_tiled_fn tensor_map_encoder();

}  // namespace moe
