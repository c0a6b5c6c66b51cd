// gemv_pipe.cu -- decode-shape expert kernels (MOE_ACT_BF16, T <= 4) with a bulk-copy weight
// pipeline.
//
// Decode is bound by reading the chosen experts' weights once (Muse Spark Open explainer,
// section 13; DGX Spark news item, section 1), so the design goal is to keep enough bytes in
// flight per SM to run HBM at full rate while the arithmetic per byte stays small:
//   - one producer thread streams contiguous weight-row ranges (codes and E8M0 scales) into a ring
//     of shared-memory stages with 1-D bulk copies (TMA engine) completing on mbarriers, so the
//     bytes in flight per SM are the ring size, not a register budget;
//   - 256 consumer threads (8 warps) own fixed 32-element K blocks: thread j of a row group reads
//     16 bytes of codes per row from the stage, keeps the activations of its block in registers
//     (f16, prescaled per row by a power of two, exact for bf16 inputs), forms exact products with
//     fp32 accumulation, and applies the block scale once per partial;
//   - partial dot products are summed per row group by a warp transpose-reduction and one
//     cross-warp exchange through shared memory per stage.
// Work split: the persistent grid (one CTA per SM) gives each CTA an equal contiguous range of
// output features (gate/up: over the flattened (active expert, i) space; down: a range of d rows
// that the CTA computes for every active expert in ascending order, fusing the weighted sum in the
// slot order of each token).
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCons = 256;                // consumer threads
constexpr int kPipeThreads = kCons + 32;  // + producer warp
constexpr int kRowsPerGroup = 8;          // weight rows per row group per stage
constexpr int kRedId = 1;                 // named barrier of the consumer warps

struct Geo {
    int nb, bpt, G, RG;
};

__host__ __device__ inline Geo make_geo(int K) {
    Geo g;
    g.nb = K / 32;
    g.bpt = (g.nb + kCons - 1) / kCons;
    const int need = (g.nb + g.bpt - 1) / g.bpt;
    int G = 32;
    while (G < need) G *= 2;
    g.G = G;
    g.RG = kCons / G;
    return g;
}

struct PipeArgs {
    const uint8_t* q0;  // up: gate codes / down: down codes
    const uint8_t* s0;
    const uint8_t* q1;  // up: up codes
    const uint8_t* s1;
    const uint16_t* act;  // up: x [T][d]; down: h [P][I]
    const int32_t* perm_token;
    const int32_t* offsets;
    PlanView plan;
    const float* row_w;  // down: gate weight of each permuted row
    int T, K, M_exp, E, stages;
    int xs_rows;    // staged activation rows: Q, or all P permuted rows when stage_all
    int stage_all;  // down: stage every h row once at the start
    size_t stage_bytes, codes_bytes, scale_bytes;  // per stage: codes region (per matrix), scales region
    uint16_t* out;  // up: h [P][I]; down: y [T][d]
    int* status;
};

// acc += w.lo * x.lo + w.hi * x.hi (f16 operands, exact products, fp32 accumulator).
__device__ __forceinline__ float dot2_f16(uint32_t w2, uint32_t x2, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\t"
        "mov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc)
        : "r"(w2), "r"(x2));
    return acc;
}

__device__ __forceinline__ float block_dot(const uint4& codes, const uint32_t* x) {
    const uint32_t words[4] = {codes.x, codes.y, codes.z, codes.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        uint32_t h[4];
        e2m1x8_to_h2(words[m], h);
        a0 = dot2_f16(h[0], x[4 * m + 0], a0);
        a1 = dot2_f16(h[1], x[4 * m + 1], a1);
        a0 = dot2_f16(h[2], x[4 * m + 2], a0);
        a1 = dot2_f16(h[3], x[4 * m + 3], a1);
    }
    return a0 + a1;
}

template <int V>
__device__ __forceinline__ float warp_transpose_reduce(float (&a)[V], int lane) {
#pragma unroll
    for (int half = V / 2, mask = 16; half >= 1; half /= 2, mask /= 2) {
        const bool upper = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? a[i] : a[i + half];
            const float recv = __shfl_xor_sync(0xffffffffu, send, mask);
            a[i] = (upper ? a[i + half] : a[i]) + recv;
        }
    }
    float v = a[0];
#pragma unroll
    for (int mask = (32 / V) / 2; mask >= 1; mask /= 2) v += __shfl_xor_sync(0xffffffffu, v, mask);
    return v;
}

// Prescale exponent p of a row whose largest |bf16| has bit pattern mx (sign cleared): the row
// maximum times 2^p lies in [2^14, 2^15).
__device__ __forceinline__ int prescale_exp(uint32_t mx) {
    const int p = (mx == 0) ? 0 : 141 - (int)(mx >> 7);
    return max(-126, min(126, p));
}

// All consumer threads stage nq activation rows as prescaled f16, block-interleaved: 16-byte
// unit c of block b of staged row q at uint4 index (q * 4 + c) * nb + b.  inv[q] = 2^-p.
// smax: nq ints of shared scratch.  Ends with the consumer barrier.
__device__ void stage_rows(const uint16_t* __restrict__ src, const int* rows, int nq, int K, uint4* dst, float* inv,
                           unsigned* smax, int tid) {
    const int nb = K / 32, units = K / 8, total = nq * units;
    if (tid < nq) smax[tid] = 0;
    ptx::named_sync(kRedId, kCons);
#pragma unroll 4
    for (int i = tid; i < total; i += kCons) {
        const int q = i / units, u = i - q * units;
        const uint4 v = reinterpret_cast<const uint4*>(src + (size_t)rows[q] * K)[u];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t mx = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) mx = max(mx, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        atomicMax(&smax[q], mx);
    }
    ptx::named_sync(kRedId, kCons);
#pragma unroll 4
    for (int i = tid; i < total; i += kCons) {
        const int q = i / units, u = i - q * units;
        const uint4 v = reinterpret_cast<const uint4*>(src + (size_t)rows[q] * K)[u];
        const float up = __uint_as_float((uint32_t)(127 + prescale_exp(smax[q])) << 23);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half lo = __float2half_rn(bf16_bits_to_f32(w[j] & 0xFFFFu) * up);
            const __half hi = __float2half_rn(bf16_bits_to_f32(w[j] >> 16) * up);
            o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
        }
        dst[((size_t)q * 4 + (u & 3)) * nb + (u >> 2)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (tid < nq) inv[tid] = __uint_as_float((uint32_t)(127 - prescale_exp(smax[tid])) << 23);
    ptx::named_sync(kRedId, kCons);
}

// Item of the producer / consumer sequence: matrix rows [row, row + m) of expert e.
struct Item {
    int e, row, m, slot;
};

// Gate/up sequence of CTA c: outputs [f0, f1) of the flattened (active slot, i) space, cut into
// items of at most mmax outputs that do not cross experts.
struct UpSeq {
    long long f, f1;
    int I, mmax;
    const int32_t* active;
    __device__ bool next(Item& it) {
        if (f >= f1) return false;
        const int slot = (int)(f / I), i = (int)(f % I);
        int m = min(mmax, I - i);
        if ((long long)m > f1 - f) m = (int)(f1 - f);
        it.slot = slot;
        it.e = active[slot];
        it.row = i;
        it.m = m;
        f += m;
        return true;
    }
};

// Down sequence of CTA c: its rows [n0, n1) for every active expert (ascending), cut into items
// of at most mmax rows.
struct DownSeq {
    int u, n_act, n0, n1, r, mmax;
    const int32_t* active;
    __device__ bool next(Item& it) {
        if (n1 <= n0) return false;
        if (r >= n1) {
            ++u;
            r = n0;
        }
        if (u >= n_act) return false;
        it.slot = u;
        it.e = active[u];
        it.row = r;
        it.m = min(mmax, n1 - r);
        r += it.m;
        return true;
    }
};

// Producer: copy the codes and scales of one item into stage s.
__device__ __forceinline__ void issue_item(const PipeArgs& a, bool up, const Item& it, unsigned char* st, uint64_t* bar) {
    const size_t row_bytes = (size_t)a.K / 2, srow = (size_t)a.K / 32;
    const size_t g0 = (size_t)it.e * a.M_exp + it.row;
    const uint32_t cbytes = (uint32_t)(it.m * row_bytes);
    const size_t s_lo = g0 * srow, s_hi = (g0 + it.m) * srow;
    const size_t s_lo16 = s_lo & ~size_t(15), s_hi16 = (s_hi + 15) & ~size_t(15);
    const uint32_t sbytes = (uint32_t)(s_hi16 - s_lo16);
    const int nmat = up ? 2 : 1;
    ptx::mbar_arrive_expect_tx(bar, nmat * (cbytes + sbytes));
    ptx::bulk_load(st, a.q0 + g0 * row_bytes, cbytes, bar);
    ptx::bulk_load(st + nmat * a.codes_bytes, a.s0 + s_lo16, sbytes, bar);
    if (up) {
        ptx::bulk_load(st + a.codes_bytes, a.q1 + g0 * row_bytes, cbytes, bar);
        ptx::bulk_load(st + nmat * a.codes_bytes + a.scale_bytes, a.s1 + s_lo16, sbytes, bar);
    }
}

// ------------------------------------------------------------------ the kernel
// UP: h[r0 + qq][i] = SiLU(g) * u for the expert's tokens; DOWN: y[t] += w * bf16(W_d h).
template <bool UP, int Q, int BPT>
__global__ void __launch_bounds__(kPipeThreads, 1)
gemv_pipe_kernel(const PipeArgs a) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    constexpr int V = kRowsPerGroup * Q;
    const Geo geo = make_geo(a.K);
    unsigned char* stages = smem;
    const int XR = a.xs_rows;                                                           // Q, or P when staged once
    uint4* xs = reinterpret_cast<uint4*>(smem + (size_t)a.stages * a.stage_bytes);     // [XR][K/8]
    float* inv = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(xs) + (size_t)XR * a.K * 2);  // [XR]
    unsigned* smax = reinterpret_cast<unsigned*>(inv + XR);                             // [XR]
    float* red = reinterpret_cast<float*>(smax + XR);                                   // [2][8][32]
    int* rows = reinterpret_cast<int*>(red + 2 * 8 * 32);                               // [XR]
    int* toks = rows + XR;                                                              // [Q]
    float* pw = reinterpret_cast<float*>(toks + Q);                                     // [Q]
    float* ys = pw + Q;                                                                 // [T][rows per CTA]
    const int ys_rows = UP ? 0 : (a.M_exp + gridDim.x - 1) / gridDim.x;
    uint64_t* full = reinterpret_cast<uint64_t*>(
        (reinterpret_cast<uintptr_t>(ys + (UP ? 0 : a.T * ys_rows)) + 7) & ~uintptr_t(7));
    uint64_t* empty = full + a.stages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + a.stages);
    volatile int* s_ok = abort_flag + 1;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < a.stages; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], kCons / 32);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    pdl_wait();  // routing and the activation rows come from the preceding kernels

    const int n_act = a.plan.scalars[0];
    UpSeq useq;
    DownSeq dseq;
    const int mmax = UP ? 4 * geo.RG : kRowsPerGroup * geo.RG;
    int n0 = 0, n1 = 0;
    if (UP) {
        const long long N = (long long)n_act * a.M_exp;
        useq = UpSeq{N * blockIdx.x / gridDim.x, N * (blockIdx.x + 1) / gridDim.x, a.M_exp, mmax, a.plan.active};
    } else {
        n0 = (int)((long long)a.M_exp * blockIdx.x / gridDim.x);
        n1 = (int)((long long)a.M_exp * (blockIdx.x + 1) / gridDim.x);
        dseq = DownSeq{0, n_act, n0, n1, n0, mmax, a.plan.active};
    }
    auto next_item = [&](Item& it) { return UP ? useq.next(it) : dseq.next(it); };

    if (warp == kCons / 32) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            Item it;
            int n = 0;
            while (next_item(it)) {
                const int s = n % a.stages;
                const uint32_t ph = (n / a.stages) & 1;
                if (!ptx::mbar_wait(&empty[s], ph ^ 1, abort_flag, a.status)) break;
                issue_item(a, UP, it, stages + (size_t)s * a.stage_bytes, &full[s]);
                ++n;
            }
            if (*abort_flag)  // let issued copies land before the CTA's shared memory is released
                for (int q = 0; q < a.stages && q < n; ++q) {
                    const int k = n - 1 - q;
                    ptx::mbar_wait(&full[k % a.stages], (k / a.stages) & 1, abort_flag, nullptr, 100000000LL);
                }
        }
    } else {
        // ------------------------------------------------------------ consumers
        const int grp = tid / geo.G, gl = tid % geo.G, wpg = geo.G / 32;
        const int cwarp = warp;
        (void)cwarp;
        uint32_t xr[Q][BPT][16];
        int cur_slot = -1, nq = 0, r0 = 0, xbase = 0;
        Item it;
        int n = 0;
        if (!UP)
            for (int i = tid; i < a.T * ys_rows; i += kCons) ys[i] = 0.f;
        if (a.stage_all) {
            // down, small P: stage every permuted h row once (rows are compact permuted rows)
            for (int i = tid; i < XR; i += kCons) rows[i] = i;
            ptx::named_sync(kRedId, kCons);
            stage_rows(a.act, rows, XR, a.K, xs, inv, smax, tid);
        }
        while (next_item(it)) {
            if (it.slot != cur_slot) {
                // new expert: its tokens' activation rows (or its pairs' h rows) into registers
                cur_slot = it.slot;
                r0 = a.offsets[it.e];
                nq = a.offsets[it.e + 1] - r0;
                if (nq > Q) nq = Q;  // callers guarantee at most Q rows per expert (T <= Q)
                ptx::named_sync(kRedId, kCons);  // the previous item's output phase is done
                if (tid < nq) {
                    if (!a.stage_all) rows[tid] = UP ? a.perm_token[r0 + tid] : r0 + tid;
                    toks[tid] = a.perm_token[r0 + tid];
                    pw[tid] = UP ? 0.f : a.row_w[r0 + tid];
                }
                ptx::named_sync(kRedId, kCons);
                if (!a.stage_all) stage_rows(a.act, rows, nq, a.K, xs, inv, smax, tid);
                xbase = a.stage_all ? r0 : 0;
#pragma unroll
                for (int qq = 0; qq < Q; ++qq)
#pragma unroll
                    for (int c = 0; c < BPT; ++c) {
                        const int b = gl + c * geo.G;
#pragma unroll
                        for (int cu = 0; cu < 4; ++cu) {
                            uint4 v = make_uint4(0, 0, 0, 0);
                            if (qq < nq && b < geo.nb) v = xs[((size_t)(xbase + qq) * 4 + cu) * geo.nb + b];
                            xr[qq][c][4 * cu + 0] = v.x;
                            xr[qq][c][4 * cu + 1] = v.y;
                            xr[qq][c][4 * cu + 2] = v.z;
                            xr[qq][c][4 * cu + 3] = v.w;
                        }
                    }
            }
            const int s = n % a.stages;
            const uint32_t ph = (n / a.stages) & 1;
            ++n;
            // one consumer thread waits (bounded) for the stage and shares the verdict, so every
            // consumer warp leaves the loop at the same item if the wait gives up
            if (tid == 0) *s_ok = ptx::mbar_wait(&full[s], ph, abort_flag, a.status) ? 1 : 0;
            ptx::named_sync(kRedId, kCons);
            if (*s_ok == 0) break;
            const unsigned char* st = stages + (size_t)s * a.stage_bytes;
            const size_t row_bytes = (size_t)a.K / 2, srow = (size_t)a.K / 32;
            const size_t g0 = (size_t)it.e * a.M_exp + it.row;
            const int sadj = (int)((g0 * srow) & 15);
            // rows of this group in the stage: up: outputs 4*grp .. 4*grp+3 (gate j, up j);
            // down: rows 8*grp .. 8*grp+7
            float acc[V];
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = 0.f;
#pragma unroll
            for (int j = 0; j < kRowsPerGroup; ++j) {
                const int mat = UP ? (j / 4) : 0;
                const int lr = UP ? (4 * grp + (j % 4)) : (kRowsPerGroup * grp + j);
                if (lr < it.m) {
                    const unsigned char* codes = st + (size_t)mat * a.codes_bytes + (size_t)lr * row_bytes;
                    const unsigned char* scl =
                        st + (UP ? 2 : 1) * a.codes_bytes + (size_t)mat * a.scale_bytes + sadj + (size_t)lr * srow;
#pragma unroll
                    for (int c = 0; c < BPT; ++c) {
                        const int b = gl + c * geo.G;
                        if (b < geo.nb) {
                            const uint4 w = *reinterpret_cast<const uint4*>(codes + 16 * (size_t)b);
                            const float sc = e8m0_to_f32(scl[b]);
#pragma unroll
                            for (int qq = 0; qq < Q; ++qq)
                                if (qq < nq) acc[qq * kRowsPerGroup + j] = fmaf(block_dot(w, xr[qq][c]), sc,
                                                                                acc[qq * kRowsPerGroup + j]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&empty[s]);  // this warp is done with the stage
            float* rb = red + (n & 1) * 8 * 32;
            rb[cwarp * 32 + lane] = warp_transpose_reduce<V>(acc, lane);
            ptx::named_sync(kRedId, kCons);
            if (gl < 32) {
                constexpr int sh = (V == 8 ? 2 : V == 16 ? 1 : 0);  // lane l holds value l >> sh
                const int v = lane >> sh, qq = v / kRowsPerGroup, j = v % kRowsPerGroup;
                const bool leader = (lane & ((1 << sh) - 1)) == 0;
                if (leader && qq < nq) {
                    if (UP) {
                        const int lr = 4 * grp + j;
                        if (j < 4 && lr < it.m) {
                            float g = 0.f, u = 0.f;
                            for (int w = 0; w < wpg; ++w) {
                                g += rb[(grp * wpg + w) * 32 + lane];
                                u += rb[(grp * wpg + w) * 32 + lane + (4 << sh)];
                            }
                            g *= inv[xbase + qq];
                            u *= inv[xbase + qq];
                            const float hv = g / (1.f + expf(-g)) * u;  // SiLU(g) * u
                            a.out[(size_t)(r0 + qq) * a.M_exp + it.row + lr] = f32_to_bf16_bits(hv);
                        }
                    } else {
                        const int lr = kRowsPerGroup * grp + j;
                        if (lr < it.m) {
                            float sum = 0.f;
                            for (int w = 0; w < wpg; ++w) sum += rb[(grp * wpg + w) * 32 + lane];
                            const float yv = bf16_bits_to_f32(f32_to_bf16_bits(sum * inv[xbase + qq]));
                            float& acc_y = ys[toks[qq] * ys_rows + (it.row + lr - n0)];
                            acc_y = fmaf(pw[qq], yv, acc_y);
                        }
                    }
                }
            }
        }
        if (!UP) {
            ptx::named_sync(kRedId, kCons);
            for (int i = tid; i < a.T * (n1 - n0); i += kCons) {
                const int t = i / (n1 - n0), rr = i % (n1 - n0);
                a.out[(size_t)t * a.M_exp + n0 + rr] = f32_to_bf16_bits(ys[t * ys_rows + rr]);
            }
        }
    }
    __syncthreads();
    pdl_launch_dependents();
}

int sm_count_cached() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

template <bool UP, int Q>
const void* pick_kernel(int bpt) {
    return bpt == 1 ? (const void*)gemv_pipe_kernel<UP, Q, 1> : (const void*)gemv_pipe_kernel<UP, Q, 2>;
}

template <bool UP>
const void* pick_q(int q, int bpt) {
    if (q == 1) return pick_kernel<UP, 1>(bpt);
    if (q == 2) return pick_kernel<UP, 2>(bpt);
    return pick_kernel<UP, 4>(bpt);
}

int q_for(int T) { return T <= 1 ? 1 : T <= 2 ? 2 : 4; }

// Shared memory of a configuration, or 0 when it does not fit.
size_t pipe_smem(bool up, int T, int K, int M_exp, int E, int stages, size_t* stage_bytes, size_t* codes_bytes,
                 size_t* scale_bytes, int ctas, int xs_rows) {
    const Geo geo = make_geo(K);
    const int mmax = up ? 4 * geo.RG : kRowsPerGroup * geo.RG;
    const int Q = q_for(T);
    *codes_bytes = (size_t)mmax * K / 2;
    *scale_bytes = ((size_t)mmax * K / 32 + 32 + 15) & ~size_t(15);
    const size_t nmat = up ? 2 : 1;  // gate and up matrices, or the down matrix
    *stage_bytes = ((nmat * *codes_bytes + nmat * *scale_bytes) + 127) & ~size_t(127);
    const int ys_rows = up ? 0 : (M_exp + ctas - 1) / ctas;
    const int XR = xs_rows;
    size_t bytes = (size_t)stages * *stage_bytes + (size_t)XR * K * 2 + sizeof(float) * XR + sizeof(unsigned) * XR +
                   sizeof(float) * 2 * 8 * 32 + sizeof(int) * (XR + Q) + sizeof(float) * Q +
                   sizeof(float) * (size_t)T * ys_rows + 16 + sizeof(uint64_t) * 2 * stages + 32 + 128;
    (void)E;
    return bytes;
}

}  // namespace

bool gemv_pipe_supported(int T, int d, int I) {
    const Geo gu = make_geo(d), gd = make_geo(I);
    const int Q = q_for(T);
    return T >= 1 && T <= 4 && gu.bpt <= 2 && gd.bpt <= 2 && Q * gu.bpt <= 4 && Q * gd.bpt <= 4 &&
           (I % (4 * gu.RG)) == 0;
}

static cudaError_t launch_pipe(bool up, PipeArgs& a, int T, int P, cudaStream_t st, bool pdl) {
    const int ctas = sm_count_cached();
    const Geo geo = make_geo(a.K);
    const int Q = q_for(T);
    // down: stage all P = T*k permuted h rows once when they take at most 48 KB
    a.stage_all = (!up && (size_t)P * a.K * 2 <= 48 * 1024) ? 1 : 0;
    a.xs_rows = a.stage_all ? P : Q;
    int stages = 8;
    size_t smem = 0;
    for (; stages >= 3; --stages) {
        smem = pipe_smem(up, T, a.K, a.M_exp, a.E, stages, &a.stage_bytes, &a.codes_bytes, &a.scale_bytes, ctas,
                         a.xs_rows);
        if (smem <= 220 * 1024) break;
    }
    if (stages < 3) return cudaErrorInvalidValue;
    a.stages = stages;
    void* args[] = {&a};
    const void* f = up ? pick_q<true>(q_for(T), geo.bpt) : pick_q<false>(q_for(T), geo.bpt);
    return launch_kernel(f, dim3(ctas), dim3(kPipeThreads), smem, st, pdl, args);
}

cudaError_t launch_gemv_up_pipe(const uint16_t* x, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                                int T, int d, int E, int k, int I, const moe_expert_weights* W, uint16_t* h, int* status,
                                cudaStream_t st, bool pdl) {
    PipeArgs a = {};
    a.q0 = W->gate_q;
    a.s0 = W->gate_s;
    a.q1 = W->up_q;
    a.s1 = W->up_s;
    a.act = x;
    a.perm_token = perm_token;
    a.offsets = offsets;
    a.plan = plan;
    a.T = T;
    a.K = d;
    a.M_exp = I;
    a.E = E;
    a.out = h;
    a.status = status;
    return launch_pipe(true, a, T, T * k, st, pdl);
}

cudaError_t launch_gemv_down_pipe(const uint16_t* h, const int32_t* perm_token, const int32_t* offsets, PlanView plan,
                                  const float* row_w, int T, int d, int E, int k, int I, const moe_expert_weights* W,
                                  uint16_t* y, int* status, cudaStream_t st, bool pdl) {
    PipeArgs a = {};
    a.q0 = W->down_q;
    a.s0 = W->down_s;
    a.act = h;
    a.perm_token = perm_token;
    a.offsets = offsets;
    a.plan = plan;
    a.row_w = row_w;
    a.T = T;
    a.K = I;
    a.M_exp = d;
    a.E = E;
    a.out = y;
    a.status = status;
    return launch_pipe(false, a, T, T * k, st, pdl);
}

}  // namespace moe
