/*
 * moe_oracle.c -- plain, slow CPU oracle for the MoE expert-FFN layer
 * (router top-k -> permute by expert -> gate/up + SwiGLU -> down -> weighted sum).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call
 * this file: only the tests, the package's smoke check and the CPU-baseline leg of
 * the benchmark use it.  It shares no code, header, table or helper with the CUDA
 * library; both sides are written independently from the same sources:
 *
 *   [MUSE]  "Muse Spark Open を段階的に分解する" (illustrated explainer of Muse Spark Open)
 *             section 8  -- router: one FP32 matrix product scores every expert, the best 8 of
 *                            256 are kept, no shared expert, the choice is a set.
 *             section 9  -- each chosen expert is gate/up/down; outputs are weighted by the router
 *                            scores and summed; the printed weights 0.21 ... 0.06 sum to 1.
 *             section 11 -- expert weights are kept as 4-bit values sharing a small block scale.
 *             section 12 -- tokens are gathered per expert and computed as one batch.
 *   [SPARK] "DGX Spark MoE inference optimizations" (devotd news), section 2 -- the expert
 *             compute path is the block-scaled 4-bit MXFP4 format.
 *   [OCP-MX] OCP Microscaling Formats (MX) v1.0 -- E2M1 element grid, E8M0 scale,
 *             shared exponent = floor(log2(amax)) - emax_elem (emax_elem = 2 for E2M1).
 *   [OFP8]  OCP 8-bit Floating Point Specification (OFP8) v1.0 -- the E4M3 encoding (bias 7,
 *             subnormals, S.1111.111 NaN, no infinity, largest finite 448).
 *
 * Readings taken where the sources are silent (each also listed in the design notes):
 *   R1  router reduction order: the sources only say "FP32".  Logits are formed from 32
 *       partial sums; partial c accumulates, with fmaf and starting from +0, the elements i
 *       whose 4-element group index (i/4) is congruent to c mod 32, in increasing i; the 32
 *       partials are combined by an xor butterfly (m = 16, 8, 4, 2, 1: p_c <- p_c + p_{c^m});
 *       the logit is p_0 + b_e (b_e = +0 when there is no bias).
 *   R2  top-k ties go to the lower expert id; ids are stored in ascending order (a set).
 *   R3  the gate weights are a softmax over the k selected logits (bias included), computed
 *       in fp64 and rounded once to fp32.
 *   R4  permuted rows are ordered by (expert, token, slot).
 *   R5  SwiGLU: h = SiLU(g) * u = g / (1 + exp(-g)) * u.
 *   R6  an all-zero block gets scale byte 0 and zero codes; -0 is encoded as +0; values are
 *       rounded to nearest on the E2M1 grid with ties to the even code, saturating at 6.
 *   R7  activation formats mirror the path under test:
 *         ACT_BF16  -- x used as its bf16 values; h rounded to fp32 then to bf16 (RNE);
 *         ACT_MXFP4 -- x quantised per token row with the R6 rule; h rounded to fp32 then
 *                      quantised with the R6 rule;
 *         ACT_EXACT -- x as bf16 values, h kept in fp64 (informational only).
 *       Expert outputs (y_perm) are rounded to fp32 then bf16, as the GPU stores them; the
 *       weighted sum is formed in fp64 over the k slots in slot order, rounded to fp32, then
 *       to bf16.
 *   R9  shared latent projections (optional; [MUSE] s.9: one matrix shared by the 8 experts
 *       narrows the token from 8192 to 4096 before them and one widens the weighted sum back
 *       to 8192): plain MXFP4 matrix products, out[n] = sum_c a[c] W[n][c], with the input row
 *       in the activation format of R7 (bf16 values, or MXFP4-quantised), fp64 accumulation,
 *       the output rounded to fp32 then bf16 like an expert output.
 *   R8  expert output normalisation (optional; [MUSE] s.9 says each chosen expert's output is
 *       normalised before the weighted sum, without naming the normalisation): RMSNorm over
 *       the d output features of the expert's (bf16) output row, v / sqrt(mean(v^2) + eps),
 *       eps = 1e-6 unless given, no learned scale; computed in fp64 and rounded to fp32, then
 *       summed as in R7.
 *   R10 NVFP4 expert weights (optional; [MUSE] s.11 describes the weights as 4-bit values of
 *       which 16 share a small scale, about 4.5 bits each, without giving the scale's format):
 *       E2M1 codes as in MXFP4, one E4M3 scale [OFP8] per 16 consecutive elements of a row and
 *       one fp32 global scale per matrix; value = E2M1 * E4M3 * global.  Quantiser, in fp32:
 *       global = amax(matrix) / (6 * 448) (1 if that is 0); per block t = (amax(block) / global)
 *       / 6, scale = nearest E4M3 to t (ties even, saturating at 448); D = scale * global;
 *       each code = nearest E2M1 to |v| / D (ties even, saturating at 6), signed unless 0;
 *       D = 0 gives zero codes.
 *   R11 MXFP8 activations (optional, ACT_MXFP8; [SPARK] s.2 names the baseline configuration
 *       "4-bit weights, 8-bit activations" without the 8-bit format): the MX format of the same
 *       family as the MXFP4 path [OCP-MX], E4M3 elements [OFP8] with one E8M0 scale per 32:
 *       X = floor(log2(amax)) - 8 (8 = exponent of E4M3's largest normal, 448 = 1.75 * 2^8),
 *       clamped to [-127, 127]; each element is |v| / 2^X rounded to the nearest E4M3 value
 *       (ties even, saturating at 448), signed unless its magnitude code is 0; an all-zero block
 *       gets scale byte 0.  x rows and the fp32 h rows are quantised this way (as R7 does with
 *       MXFP4); the weights stay MXFP4 (or NVFP4).
 * Accumulations inside the expert matrices are fp64 (closer to exact than the kernels).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ACT_BF16 0
#define ACT_MXFP4 1
#define ACT_EXACT 2
#define ACT_MXFP8 3

/* Threads of the OpenMP loops for later calls (the environment is read only once). */
void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ scalar formats */

/* bf16 bits -> fp32: the bf16 value is the top half of an fp32 word. */
static float bf16_bits_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16 bits, round to nearest, ties to even (finite inputs). */
static uint16_t float_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

static float round_to_bf16(float f) { return bf16_bits_to_float(float_to_bf16_bits(f)); }

/* E2M1 magnitudes for codes 0..7 [OCP-MX]; bit 3 of a code is the sign. */
static const double kE2M1Magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(int code) {
    double m = kE2M1Magnitude[code & 7];
    return (code & 8) ? -m : m;
}

/* E8M0 scale byte -> 2^(s-127); 0xFF is NaN [OCP-MX]. */
double oracle_e8m0_value(int s) {
    if (s == 255) return NAN;
    return ldexp(1.0, s - 127);
}

/* Nearest E2M1 magnitude code for a >= 0 (already divided by the block scale).
 * Ties go to the even code; values beyond the largest magnitude saturate (R6). */
int oracle_e2m1_encode_magnitude(double a) {
    int best = 0;
    double best_dist = fabs(a - kE2M1Magnitude[0]);
    for (int c = 1; c < 8; ++c) {
        double dist = fabs(a - kE2M1Magnitude[c]);
        if (dist < best_dist || (dist == best_dist && (c % 2) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return best;
}

/* Quantise one block of n values to E2M1 codes with one shared E8M0 scale [OCP-MX], (R6).
 * Shared exponent X = floor(log2(amax)) - 2, clamped to the E8M0 range. */
void oracle_mx_block_quantize(const double* v, int n, uint8_t* codes, uint8_t* scale_byte) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) {
        *scale_byte = 0;
        for (int i = 0; i < n; ++i) codes[i] = 0;
        return;
    }
    int ex;
    (void)frexp(amax, &ex); /* amax = f * 2^ex, f in [0.5, 1)  =>  floor(log2(amax)) = ex - 1 */
    int X = (ex - 1) - 2;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    *scale_byte = (uint8_t)(X + 127);
    for (int i = 0; i < n; ++i) {
        double a = ldexp(fabs(v[i]), -X);
        int c = oracle_e2m1_encode_magnitude(a);
        if (c != 0 && v[i] < 0.0) c |= 8;
        codes[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------ MXFP4 tensors */

/* Pack fp32 rows [rows][K] into MXFP4: q[rows][K/2] (element 2i in the low nibble, 2i+1 in
 * the high nibble) and s[rows][K/32] (one E8M0 byte per 32 consecutive elements of a row).
 * Returns 0, or -1 when K is not a multiple of 32. */
int oracle_mxfp4_pack(const float* w, int64_t rows, int64_t K, uint8_t* q, uint8_t* s) {
    if (K % 32 != 0) return -1;
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double v[32];
        uint8_t codes[32];
        for (int64_t b = 0; b < nb; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = (double)w[r * K + b * 32 + i];
            oracle_mx_block_quantize(v, 32, codes, &s[r * nb + b]);
            for (int i = 0; i < 16; ++i)
                q[r * (K / 2) + b * 16 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        }
    }
    return 0;
}

/* Dequantise MXFP4 rows back to fp32 (exact: every E2M1 value times 2^(s-127) is an fp32
 * number for s in 0..254).  Returns 0, or -1 if a scale byte is 0xFF (NaN). */
int oracle_mxfp4_unpack(const uint8_t* q, const uint8_t* s, int64_t rows, int64_t K, float* w) {
    if (K % 32 != 0) return -1;
    int64_t nb = K / 32;
    int bad = 0;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < K; ++i) {
            uint8_t sb = s[r * nb + i / 32];
            if (sb == 255) bad = 1;
            uint8_t byte = q[r * (K / 2) + i / 2];
            int code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            w[r * K + i] = (float)(oracle_e2m1_value(code) * oracle_e8m0_value(sb));
        }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ NVFP4 tensors  (R10) */

/* E4M3 byte -> value [OFP8]: sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0;
 * exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
double oracle_e4m3_value(int code) {
    int e = (code >> 3) & 0xF, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return (code & 0x80) ? -v : v;
}

/* Nearest non-negative finite E4M3 code to a >= 0: a search over the 127 codes 0x00..0x7E,
 * ties to the even code, values beyond 448 saturating to 448 (R10). */
int oracle_e4m3_encode_nonneg(double a) {
    int best = 0;
    double best_dist = fabs(a);
    for (int c = 1; c <= 0x7E; ++c) {
        double dist = fabs(a - oracle_e4m3_value(c));
        if (dist < best_dist || (dist == best_dist && (c % 2) == 0)) {
            best = c;
            best_dist = dist;
        }
    }
    return best;
}

/* Global scale of one NVFP4 matrix from its largest magnitude (R10): amax / (6 * 448) in fp32,
 * so that the largest block scale lands at the top of the E4M3 range; 1 when that is 0. */
float oracle_nvfp4_global_scale(float amax) {
    float gs = amax / 2688.0f;
    return gs == 0.0f ? 1.0f : gs;
}

/* Quantise one block of n values (16 in NVFP4) with the matrix's global scale gs (R10), every
 * step in fp32 in this order: t = (amax / gs) / 6; scale byte = nearest E4M3 to t (ties even,
 * saturating); D = value(scale byte) * gs; code of v = nearest E2M1 to |v| / D (ties even,
 * saturating at 6), with the sign of v unless the magnitude code is 0; D = 0 gives zero codes. */
void oracle_nv_block_quantize(const float* v, int n, float gs, uint8_t* codes, uint8_t* scale_byte) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    float t = (amax / gs) / 6.0f;
    int sb = oracle_e4m3_encode_nonneg((double)t);
    *scale_byte = (uint8_t)sb;
    float D = (float)oracle_e4m3_value(sb) * gs;
    for (int i = 0; i < n; ++i) {
        if (D == 0.0f) {
            codes[i] = 0;
            continue;
        }
        float a = fabsf(v[i]) / D;
        int c = oracle_e2m1_encode_magnitude((double)a);
        if (c != 0 && v[i] < 0.0f) c |= 8;
        codes[i] = (uint8_t)c;
    }
}

/* Pack n_mats fp32 matrices [n_mats][rows][K] into NVFP4 (R10): codes q[n_mats*rows][K/2]
 * (same nibble order as MXFP4), scales s[n_mats*rows][K/16] (one E4M3 byte per 16 consecutive
 * elements of a row) and one fp32 global scale gs[m] per matrix.  Returns 0, or -1 when K is
 * not a multiple of 16. */
int oracle_nvfp4_pack(const float* w, int64_t n_mats, int64_t rows, int64_t K, uint8_t* q, uint8_t* s, float* gs) {
    if (K % 16 != 0) return -1;
    int64_t nb = K / 16;
    for (int64_t m = 0; m < n_mats; ++m) {
        const float* wm = w + m * rows * K;
        float amax = 0.0f;
        for (int64_t i = 0; i < rows * K; ++i) {
            float a = fabsf(wm[i]);
            if (a > amax) amax = a;
        }
        float g = oracle_nvfp4_global_scale(amax);
        gs[m] = g;
#pragma omp parallel for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            uint8_t codes[16];
            int64_t row = m * rows + r;
            for (int64_t b = 0; b < nb; ++b) {
                oracle_nv_block_quantize(wm + r * K + b * 16, 16, g, codes, &s[row * nb + b]);
                for (int i = 0; i < 8; ++i)
                    q[row * (K / 2) + b * 8 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
            }
        }
    }
    return 0;
}

/* Dequantise NVFP4 matrices to fp64 (exact: code value * scale value has at most 6 significant
 * bits, times the fp32 global scale at most 30).  Returns 0, or -1 if a scale byte is NaN. */
int oracle_nvfp4_unpack(const uint8_t* q, const uint8_t* s, const float* gs, int64_t n_mats, int64_t rows, int64_t K,
                        double* w) {
    if (K % 16 != 0) return -1;
    int64_t nb = K / 16;
    int bad = 0;
    for (int64_t m = 0; m < n_mats; ++m)
        for (int64_t r = 0; r < rows; ++r) {
            int64_t row = m * rows + r;
            for (int64_t i = 0; i < K; ++i) {
                uint8_t sb = s[row * nb + i / 16];
                if ((sb & 0x7F) == 0x7F) bad = 1;
                uint8_t byte = q[row * (K / 2) + i / 2];
                int code = (i % 2 == 0) ? (byte & 0xF) : (byte >> 4);
                w[row * K + i] = oracle_e2m1_value(code) * oracle_e4m3_value(sb) * (double)gs[m];
            }
        }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ MXFP8 blocks  (R11) */

/* Quantise one block of n values to E4M3 codes (sign in bit 7) with one shared E8M0 scale. */
void oracle_mx8_block_quantize(const double* v, int n, uint8_t* codes, uint8_t* scale_byte) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) {
        double a = fabs(v[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0) {
        *scale_byte = 0;
        for (int i = 0; i < n; ++i) codes[i] = 0;
        return;
    }
    int ex;
    (void)frexp(amax, &ex); /* floor(log2(amax)) = ex - 1 */
    int X = (ex - 1) - 8;
    if (X < -127) X = -127;
    if (X > 127) X = 127;
    *scale_byte = (uint8_t)(X + 127);
    for (int i = 0; i < n; ++i) {
        int c = oracle_e4m3_encode_nonneg(ldexp(fabs(v[i]), -X));
        if (c != 0 && v[i] < 0.0) c |= 0x80;
        codes[i] = (uint8_t)c;
    }
}

/* ------------------------------------------------------------------ router  [MUSE] s.8 */

/* logits[t][e] = b[e] + sum_i x[t][i] * W_r[e][i] with the R1 reduction order.
 * x is bf16 bits [T][d], W_r fp32 [E][d], b fp32 [E] or NULL.  Requires d % 4 == 0. */
void oracle_router_logits(const uint16_t* x, const float* W_r, const float* b, int T, int d, int E,
                          float* logits) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float p[32];
            for (int c = 0; c < 32; ++c) {
                float acc = 0.0f;
                for (int g = c; g < d / 4; g += 32)
                    for (int q4 = 0; q4 < 4; ++q4) {
                        int i = 4 * g + q4;
                        acc = fmaf(bf16_bits_to_float(x[(int64_t)t * d + i]), W_r[(int64_t)e * d + i], acc);
                    }
                p[c] = acc;
            }
            for (int m = 16; m >= 1; m >>= 1) {
                float nxt[32];
                for (int c = 0; c < 32; ++c) nxt[c] = p[c] + p[c ^ m];
                memcpy(p, nxt, sizeof p);
            }
            logits[(int64_t)t * E + e] = p[0] + (b ? b[e] : 0.0f);
        }
    }
}

/* Top-k selection (R2) and softmax over the selected logits (R3).
 * ids[t][j] ascending expert ids, w[t][j] the matching gate weights. */
void oracle_topk_softmax(const float* logits, int T, int E, int k, int32_t* ids, float* w) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        unsigned char* taken = (unsigned char*)calloc((size_t)E, 1);
        int32_t chosen[1024];
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e; /* strict: equal values keep the lower id */
            }
            taken[best] = 1;
            chosen[j] = best;
        }
        free(taken);
        /* ascending order of the chosen set (insertion sort, k <= 32) */
        for (int a = 1; a < k; ++a) {
            int32_t v = chosen[a];
            int z = a - 1;
            while (z >= 0 && chosen[z] > v) {
                chosen[z + 1] = chosen[z];
                --z;
            }
            chosen[z + 1] = v;
        }
        double m = -INFINITY;
        for (int j = 0; j < k; ++j) m = fmax(m, (double)l[chosen[j]]);
        double sum = 0.0;
        double ex[1024];
        for (int j = 0; j < k; ++j) {
            ex[j] = exp((double)l[chosen[j]] - m);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j) {
            ids[(int64_t)t * k + j] = chosen[j];
            w[(int64_t)t * k + j] = (float)(ex[j] / sum);
        }
    }
}

/* ------------------------------------------------------------------ permute  [MUSE] s.12 */

/* Group the T*k (token, slot) pairs by expert (R4).
 * counts[e]; offsets[e] exclusive scan (E+1 entries); perm_token[r] = token of row r;
 * inv_pos[t*k + j] = row of pair (t, j).  Returns 0, or -1 on an id outside [0, E). */
int oracle_permute(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets,
                   int32_t* perm_token, int32_t* inv_pos) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t p = 0; p < (int64_t)T * k; ++p) {
        if (ids[p] < 0 || ids[p] >= E) return -1;
        counts[ids[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = ids[(int64_t)t * k + j];
            int r = fill[e]++;
            perm_token[r] = t;
            inv_pos[(int64_t)t * k + j] = r;
        }
    free(fill);
    return 0;
}

/* ------------------------------------------------------------------ activations (R7) */

/* The activation operand of one token row as the GEMMs see it (fp32 values).
 * ACT_MXFP4: quantise each 32-block (R6) and return the dequantised values, plus the codes
 * and scales if q / s are non-NULL (q: [d/2] packed like weights, s: [d/32]).
 * ACT_MXFP8: the same with the R11 rule (q: [d] E4M3 code bytes, s: [d/32]). */
void oracle_activation_row(const uint16_t* x_row, int d, int act_fmt, float* out, uint8_t* q, uint8_t* s) {
    double v[32];
    uint8_t codes[32], sb;
    if (act_fmt == ACT_MXFP8) { /* R11: one E4M3 code byte per element */
        for (int b = 0; b < d / 32; ++b) {
            for (int i = 0; i < 32; ++i) v[i] = (double)bf16_bits_to_float(x_row[b * 32 + i]);
            oracle_mx8_block_quantize(v, 32, codes, &sb);
            for (int i = 0; i < 32; ++i) out[b * 32 + i] = (float)(oracle_e4m3_value(codes[i]) * oracle_e8m0_value(sb));
            if (q)
                for (int i = 0; i < 32; ++i) q[b * 32 + i] = codes[i];
            if (s) s[b] = sb;
        }
        return;
    }
    if (act_fmt != ACT_MXFP4) {
        for (int i = 0; i < d; ++i) out[i] = bf16_bits_to_float(x_row[i]);
        return;
    }
    for (int b = 0; b < d / 32; ++b) {
        for (int i = 0; i < 32; ++i) v[i] = (double)bf16_bits_to_float(x_row[b * 32 + i]);
        oracle_mx_block_quantize(v, 32, codes, &sb);
        for (int i = 0; i < 32; ++i) out[b * 32 + i] = (float)(oracle_e2m1_value(codes[i]) * oracle_e8m0_value(sb));
        if (q)
            for (int i = 0; i < 16; ++i) q[b * 16 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
        if (s) s[b] = sb;
    }
}

/* ------------------------------------------------------------------ one expert  [MUSE] s.9 */

/* Decode one MXFP4 weight row (K elements) into fp64. */
static void weight_row(const uint8_t* q, const uint8_t* s, int64_t row, int K, double* out) {
    const uint8_t* qr = q + row * (K / 2);
    const uint8_t* sr = s + row * (K / 32);
    for (int i = 0; i < K; ++i) {
        int code = (i % 2 == 0) ? (qr[i / 2] & 0xF) : (qr[i / 2] >> 4);
        out[i] = oracle_e2m1_value(code) * oracle_e8m0_value(sr[i / 32]);
    }
}

/* One weight matrix of an expert: MXFP4 (q, s), or NVFP4 (q, s, gs) (R10). */
#define W_MXFP4 0
#define W_NVFP4 1
typedef struct {
    const uint8_t* q;
    const uint8_t* s;
    int fmt;
    double gs;
} wmat;

/* Decode one weight row of either format into fp64 (exact in both). */
static void wmat_row(const wmat* W, int64_t row, int K, double* out) {
    if (W->fmt == W_MXFP4) {
        weight_row(W->q, W->s, row, K, out);
        return;
    }
    const uint8_t* qr = W->q + row * (K / 2);
    const uint8_t* sr = W->s + row * (K / 16);
    for (int i = 0; i < K; ++i) {
        int code = (i % 2 == 0) ? (qr[i / 2] & 0xF) : (qr[i / 2] >> 4);
        out[i] = oracle_e2m1_value(code) * oracle_e4m3_value(sr[i / 16]) * W->gs;
    }
}

/* Expert FFN for n activation rows of one expert.
 *   a      [n][d]  activation operand values (from oracle_activation_row)
 *   W_g, W_u [I][d];  W_d [d][I]  (MXFP4 (q, s), or NVFP4 (q, s, global scale), R10)
 *   h_out  [n][I]  the down-GEMM operand after the R7 rounding (may be NULL)
 *   hq/hs  [n][I/2], [n][I/32]  MXFP4 codes/scales of h when act_fmt == ACT_MXFP4; [n][I] E4M3
 *          codes and [n][I/32] scales when act_fmt == ACT_MXFP8 (may be NULL)
 *   y_out  [n][d]  expert output rounded to fp32 then bf16 (R7)
 * g and u accumulate in fp64 and are rounded to fp32, as the kernels hold them in fp32. */
static void expert_ffn(const float* a, int n, int d, int I, const wmat* Wg, const wmat* Wu, const wmat* Wd,
                       int act_fmt, float* h_out, uint8_t* hq, uint8_t* hs, float* y_out) {
    double* h = (double*)malloc(sizeof(double) * (size_t)n * I);
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (size_t)(d > I ? d : I));
        double* urow = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 16)
        for (int i = 0; i < I; ++i) {
            wmat_row(Wg, i, d, wrow);
            wmat_row(Wu, i, d, urow);
            for (int r = 0; r < n; ++r) {
                const float* ar = a + (int64_t)r * d;
                double g = 0.0, u = 0.0;
                for (int c = 0; c < d; ++c) g += (double)ar[c] * wrow[c];
                for (int c = 0; c < d; ++c) u += (double)ar[c] * urow[c];
                double gf = (double)(float)g, uf = (double)(float)u;
                h[(int64_t)r * I + i] = gf / (1.0 + exp(-gf)) * uf; /* R5 */
            }
        }
        free(wrow);
        free(urow);
    }
    /* R7: round h to the operand format of the down GEMM */
    for (int r = 0; r < n; ++r) {
        double* hr = h + (int64_t)r * I;
        if (act_fmt == ACT_BF16) {
            for (int i = 0; i < I; ++i) hr[i] = (double)round_to_bf16((float)hr[i]);
        } else if (act_fmt == ACT_MXFP4) {
            double v[32];
            uint8_t codes[32], sb;
            for (int b = 0; b < I / 32; ++b) {
                for (int i = 0; i < 32; ++i) v[i] = (double)(float)hr[b * 32 + i];
                oracle_mx_block_quantize(v, 32, codes, &sb);
                for (int i = 0; i < 32; ++i) hr[b * 32 + i] = oracle_e2m1_value(codes[i]) * oracle_e8m0_value(sb);
                if (hq)
                    for (int i = 0; i < 16; ++i)
                        hq[(int64_t)r * (I / 2) + b * 16 + i] = (uint8_t)(codes[2 * i] | (codes[2 * i + 1] << 4));
                if (hs) hs[(int64_t)r * (I / 32) + b] = sb;
            }
        } else if (act_fmt == ACT_MXFP8) { /* R11 */
            double v[32];
            uint8_t codes[32], sb;
            for (int b = 0; b < I / 32; ++b) {
                for (int i = 0; i < 32; ++i) v[i] = (double)(float)hr[b * 32 + i];
                oracle_mx8_block_quantize(v, 32, codes, &sb);
                for (int i = 0; i < 32; ++i) hr[b * 32 + i] = oracle_e4m3_value(codes[i]) * oracle_e8m0_value(sb);
                if (hq)
                    for (int i = 0; i < 32; ++i) hq[(int64_t)r * I + b * 32 + i] = codes[i];
                if (hs) hs[(int64_t)r * (I / 32) + b] = sb;
            }
        }
        if (h_out)
            for (int i = 0; i < I; ++i) h_out[(int64_t)r * I + i] = (float)hr[i];
    }
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 16)
        for (int c = 0; c < d; ++c) {
            wmat_row(Wd, c, I, wrow);
            for (int r = 0; r < n; ++r) {
                const double* hr = h + (int64_t)r * I;
                double y = 0.0;
                for (int i = 0; i < I; ++i) y += hr[i] * wrow[i];
                y_out[(int64_t)r * d + c] = round_to_bf16((float)y);
            }
        }
        free(wrow);
    }
    free(h);
}

void oracle_expert_ffn(const float* a, int n, int d, int I, const uint8_t* Wg_q, const uint8_t* Wg_s,
                       const uint8_t* Wu_q, const uint8_t* Wu_s, const uint8_t* Wd_q, const uint8_t* Wd_s,
                       int act_fmt, float* h_out, uint8_t* hq, uint8_t* hs, float* y_out) {
    wmat g = {Wg_q, Wg_s, W_MXFP4, 1.0}, u = {Wu_q, Wu_s, W_MXFP4, 1.0}, dn = {Wd_q, Wd_s, W_MXFP4, 1.0};
    expert_ffn(a, n, d, I, &g, &u, &dn, act_fmt, h_out, hq, hs, y_out);
}

/* The same expert with NVFP4 weights (R10): scales [rows][K/16] E4M3 and one global scale per
 * matrix (gs_g, gs_u, gs_d). */
void oracle_expert_ffn_nvfp4(const float* a, int n, int d, int I, const uint8_t* Wg_q, const uint8_t* Wg_s,
                             const uint8_t* Wu_q, const uint8_t* Wu_s, const uint8_t* Wd_q, const uint8_t* Wd_s,
                             float gs_g, float gs_u, float gs_d, int act_fmt, float* h_out, uint8_t* hq,
                             uint8_t* hs, float* y_out) {
    wmat g = {Wg_q, Wg_s, W_NVFP4, gs_g}, u = {Wu_q, Wu_s, W_NVFP4, gs_u}, dn = {Wd_q, Wd_s, W_NVFP4, gs_d};
    expert_ffn(a, n, d, I, &g, &u, &dn, act_fmt, h_out, hq, hs, y_out);
}

/* ------------------------------------------------------------------ weighted sum  [MUSE] s.9 */

/* y[t][c] = sum_j w[t][j] * y_perm[row(t, j)][c], formed in fp64 in slot order, rounded to
 * fp32 then bf16 (R7).  rows[t*k + j] gives the y_perm row of pair (t, j); only the n_tok
 * tokens listed in tokens[] are produced (y has n_tok rows). */
void oracle_combine(const float* y_perm, const int32_t* rows, const float* w, int n_tok, const int32_t* tokens,
                    int k, int d, float* y) {
    for (int s = 0; s < n_tok; ++s) {
        int t = tokens[s];
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < k; ++j)
                acc += (double)w[(int64_t)t * k + j] * (double)y_perm[(int64_t)rows[(int64_t)t * k + j] * d + c];
            y[(int64_t)s * d + c] = round_to_bf16((float)acc);
        }
    }
}

/* Dense MXFP4 linear map (R9): out[r][n] = sum_c a[r][c] * W[n][c] for n_rows rows of the
 * activation operand a [n_rows][K] (from oracle_activation_row), W MXFP4 [N][K]; fp64
 * accumulation, rounded to fp32 then bf16. */
void oracle_dense_linear(const float* a, int n_rows, int K, int N, const uint8_t* Wq, const uint8_t* Ws, float* out) {
#pragma omp parallel
    {
        double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 16)
        for (int n = 0; n < N; ++n) {
            weight_row(Wq, Ws, n, K, wrow);
            for (int r = 0; r < n_rows; ++r) {
                double acc = 0.0;
                for (int c = 0; c < K; ++c) acc += (double)a[(int64_t)r * K + c] * wrow[c];
                out[(int64_t)r * N + n] = round_to_bf16((float)acc);
            }
        }
        free(wrow);
    }
}

/* Expert output normalisation (R8): out[r] = y[r] / sqrt(mean_c y[r][c]^2 + eps), fp64, rounded
 * to fp32.  An all-zero row stays zero. */
void oracle_expert_norm(const float* y, int64_t rows, int d, double eps, float* out) {
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) ss += (double)y[r * d + c] * (double)y[r * d + c];
        double inv = 1.0 / sqrt(ss / d + eps);
        for (int c = 0; c < d; ++c) out[r * d + c] = (float)((double)y[r * d + c] * inv);
    }
}

/* bf16 helpers exported for the tests (pinned against torch's own conversion). */
uint16_t oracle_float_to_bf16_bits(float f) { return float_to_bf16_bits(f); }
float oracle_bf16_bits_to_float(uint16_t h) { return bf16_bits_to_float(h); }
