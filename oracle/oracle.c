/*
 * Oracle for the fused MoE expert forward: a plain, slow CPU restatement in
 * fp64.  TEST INFRASTRUCTURE ONLY: it is built and called by tests/, by the
 * smoke check and by the benchmark's CPU-baseline leg, never by the product
 * path.  It shares no code with the CUDA kernels.
 *
 * Sources it follows (titles and section names in English translation; the
 * printed titles follow in brackets):
 *  - "MegaMoE: fusing the MoE forward into one comm/compute kernel"
 *    [MegaMoE：把 MoE 前向路径压进一个通信计算融合核] (code-reading notes),
 *    section "Stage 3: FP8 x FP4 two-layer GEMM"
 *    (layer equations Z_e = X_e W1_e^T, Y_e = H_e W2_e^T), "Stage 4: SwiGLU
 *    and requantisation in the L1 epilogue" (gate/up cast to BF16 first,
 *    silu(a) = a / (1 + exp(-a)), times the top-k weight, per-32-channel
 *    amax -> power-of-two UE8M0 scale -> E4M3), "Stage 5/6" (L2 output cast
 *    to BF16, FP32 sum of the BF16 top-k slots, cast to BF16), and the MoE
 *    equation y_t = sum_j g_tj W2 SwiGLU(W1 x_t) of "Problem background".
 *  - "MegaMoE" blog, section 7.3 "L1 weight interleave" (gate/up rows
 *    interleaved with granularity 8) and 7.1 "precision configuration".
 *  - "Fused comm/compute operators (5): practice" [通算融合算子（五）：实战——
 *    两个 kernel 写完一个 TP MoE 融合层], section 2 "schedule tables"
 *    (expert-sorted pool, each expert padded to 128 rows, one slot table
 *    [token][k], slack per 128-row block).
 *
 * Readings taken where the pages are silent or garbled (all listed in the
 * design notes): OCP MX element formats (E4M3 bias 7 max 448 no Inf;
 * E2M1 {0,.5,1,1.5,2,3,4,6}; UE8M0 = 2^(e-127), 0xFF NaN); weight scales
 * are 1x32 along K; the requantisation exponent is the smallest e with
 * amax <= 448 * 2^e (amax = 0 -> e = 0); FP8 rounding is RNE with
 * saturation; slot order inside an expert is stable in t*k+j; top-k ties
 * go to the lower expert index; the top-k weight is applied in the L1
 * epilogue, the combine is an unweighted sum.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* element formats                                                          */
/* ------------------------------------------------------------------------ */

/* E4M3 (OCP "fn" variant): s.eeee.mmm, bias 7, subnormals m*2^-9,
 * s.1111.111 = NaN, no infinities. */
double oracle_e4m3_decode(uint8_t code) {
    int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* E2M1: s.ee.m, bias 1, e = 0 subnormal (m * 0.5); no NaN/Inf. */
double oracle_e2m1_decode(uint8_t code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* UE8M0: 2^(code - 127), 0xFF = NaN. */
double oracle_ue8m0_decode(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* Round a real value to the nearest E4M3 code, ties to even mantissa,
 * saturating to +-448 (never reached for requantised values, see below). */
uint8_t oracle_e4m3_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 = 2^-6 is code 0x08 */
        double m = nearbyint(ldexp(a, 9)); /* default rounding mode: half-even */
        return sign | (uint8_t)m;
    }
    int q;
    double f = frexp(a, &q);          /* a = f * 2^q, f in [0.5, 1) */
    int ex = q - 1;                   /* a = (2f) * 2^ex, 2f in [1, 2) */
    double mm = nearbyint((2.0 * f - 1.0) * 8.0);
    if (mm >= 8.0) { mm = 0.0; ex += 1; }
    int code = ((ex + 7) << 3) | (int)mm;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* Round to the nearest bfloat16 value (8 significant bits), ties to even.
 * bfloat16 shares fp32's exponent range: subnormal spacing 2^-133. */
double oracle_bf16_round(double v) {
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    double a = fabs(v);
    double r;
    if (a < ldexp(1.0, -126)) {
        r = ldexp(nearbyint(ldexp(a, 133)), -133);
    } else {
        int q;
        double f = frexp(a, &q);               /* f in [0.5,1) */
        r = ldexp(nearbyint(ldexp(f, 8)), q - 8);
        if (r > 3.3895313892515355e38) r = INFINITY; /* beyond bf16 max */
    }
    return v < 0 ? -r : r;
}

/* bfloat16 bit pattern of a value that is already a bfloat16 value. */
uint16_t oracle_bf16_bits(double v) {
    float f = (float)oracle_bf16_round(v);  /* exact: bf16 values are floats */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

double oracle_silu(double a) { return a / (1.0 + exp(-a)); }

/* Requantisation exponent for a 32-value group: the smallest integer e in
 * [-127, 127] with amax <= 448 * 2^e; amax = 0 gives e = 0. */
int oracle_requant_exponent(double amax) {
    if (!(amax > 0.0)) return 0;
    int e = -127;
    while (e < 127 && amax > ldexp(448.0, e)) ++e;
    return e;
}

/* ------------------------------------------------------------------------ */
/* routing: softmax over router logits, top-k, renormalise                  */
/* ------------------------------------------------------------------------ */

/* The pages do not say what a NaN router logit means; it is read here as
 * -inf: it ranks below every number and has softmax weight 0. */
void oracle_route(const float* logits, int T, int E, int k, int64_t* idx, float* w) {
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    double* l = (double*)malloc(sizeof(double) * (size_t)E);
    char* taken = (char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* lt = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) l[e] = isnan(lt[e]) ? -INFINITY : (double)lt[e];
        double lmax = -INFINITY;
        for (int e = 0; e < E; ++e) if (l[e] > lmax) lmax = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) { p[e] = exp(l[e] - lmax); z += p[e]; }
        for (int e = 0; e < E; ++e) p[e] /= z;             /* softmax */
        memset(taken, 0, (size_t)E);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {                       /* top-k by logit */
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;  /* ties: lower index */
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
            sel += p[best];
        }
        for (int j = 0; j < k; ++j)                         /* renormalise */
            w[(size_t)t * k + j] = (float)(p[idx[(size_t)t * k + j]] / sel);
    }
    free(p);
    free(l);
    free(taken);
}

/* ------------------------------------------------------------------------ */
/* schedule tables (naive host loop)                                        */
/* ------------------------------------------------------------------------ */

/* counts[E], offsets[E+1] (each expert padded to `block` rows), slots[T*k]
 * (-1 for an empty entry), row2tk[P] (-1 for padding rows), slack[P/block].
 * row2tk/slack may be NULL (sizes unknown before the call); returns P. */
int oracle_layout(const int64_t* idx, int T, int k, int E, int block,
                  int32_t* counts, int32_t* offsets, int32_t* slots,
                  int32_t* row2tk, int32_t* slack) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int i = 0; i < T * k; ++i) if (idx[i] >= 0) counts[idx[i]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + (counts[e] + block - 1) / block * block;
    int P = offsets[E];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (row2tk) for (int r = 0; r < P; ++r) row2tk[r] = -1;
    for (int i = 0; i < T * k; ++i) {          /* scan in t*k+j order */
        int64_t e = idx[i];
        if (e < 0) { slots[i] = -1; continue; }
        int s = offsets[e] + fill[e]++;
        slots[i] = s;
        if (row2tk) row2tk[s] = i;
    }
    if (slack) {
        for (int b = 0; b < P / block; ++b) {
            int real = 0;
            for (int r = b * block; r < (b + 1) * block; ++r) real += (row2tk && row2tk[r] >= 0);
            slack[b] = block - real;
        }
    }
    free(fill);
    return P;
}

/* Pool capacity of the MegaMoE layout ("pool capacity" formula):
 * align(R*T*min(k,E_loc) + E_loc*(B_M-1), align_to). */
int64_t oracle_pool_capacity(int64_t R, int64_t T, int64_t k, int64_t E_loc,
                             int64_t block_m, int64_t align_to) {
    int64_t m = k < E_loc ? k : E_loc;
    int64_t n = R * T * m + E_loc * (block_m - 1);
    return (n + align_to - 1) / align_to * align_to;
}

/* SF pool rows: (pool / B_M) * align(B_M, 128). */
int64_t oracle_sf_pool_rows(int64_t pool, int64_t block_m) {
    return (pool / block_m) * ((block_m + 127) / 128 * 128);
}

/* ------------------------------------------------------------------------ */
/* forward: direct per-(token, k) loop                                      */
/* ------------------------------------------------------------------------ */

static inline uint8_t scale_byte(const uint32_t* sf_row, int kblk32) {
    return (uint8_t)(sf_row[kblk32 >> 2] >> (8 * (kblk32 & 3)));
}

/* Decoded values of every code, filled from the decoders above (a lookup
 * gives the same double as the call; it only saves the call per element). */
static double g_e2m1[16], g_e4m3[256];
static void fill_tables(void) {
    for (int c = 0; c < 16; ++c) g_e2m1[c] = oracle_e2m1_decode((uint8_t)c);
    for (int c = 0; c < 256; ++c) g_e4m3[c] = oracle_e4m3_decode((uint8_t)c);
}

/* dot product of a packed E2M1 weight row (with per-32 UE8M0 scales) and
 * a decoded activation vector of length K */
static double dot_w_row(const uint8_t* wrow, const uint32_t* sfrow,
                        const double* a, int K) {
    double acc = 0.0;
    for (int b = 0; b < K / 32; ++b) {
        double s = oracle_ue8m0_decode(scale_byte(sfrow, b));
        double part = 0.0;
        for (int i = b * 32; i < b * 32 + 32; ++i) {
            uint8_t byte = wrow[i >> 1];
            uint8_t code = (i & 1) ? (byte >> 4) : (byte & 0xF);
            part += g_e2m1[code] * a[i];
        }
        acc += s * part;
    }
    return acc;
}

/*
 * For each listed token t (token_list[0..n_list), or all T tokens if
 * token_list is NULL):
 *   y[i][:]   bf16 bits of y_t                      (i = position in list)
 *   q[i][j][:] E4M3 codes of the requantised L1 output h for slot j (opt.)
 *   qe[i][j][:] requant exponents e* per 32-channel group (opt.)
 * Empty slots (idx < 0) produce q = 0, qe = 0 and add nothing to y.
 * clamp > 0 enables the optional activation clamp (gate <= clamp,
 * -clamp <= up <= clamp) applied to the BF16 gate/up values.
 */
void oracle_forward(int T, int H, int I, int E, int k,
                    const uint8_t* x, const uint32_t* x_sf,
                    const int64_t* idx, const float* topk_w,
                    const uint8_t* w1, const uint32_t* w1_sf,
                    const uint8_t* w2, const uint32_t* w2_sf,
                    const int32_t* token_list, int n_list,
                    uint16_t* y, uint8_t* q, int8_t* qe,
                    double clamp, int nthreads) {
    (void)E;
    const size_t w1_row = (size_t)H / 2, w1_sfrow = (size_t)H / 128;
    const size_t w2_row = (size_t)I / 2, w2_sfrow = (size_t)I / 128;
    int n = token_list ? n_list : T;
    fill_tables();
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
    {
        double* xh = (double*)malloc(sizeof(double) * (size_t)H);
        double* h = (double*)malloc(sizeof(double) * (size_t)I);
        double* ysum = (double*)malloc(sizeof(double) * (size_t)H);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int li = 0; li < n; ++li) {
            int t = token_list ? token_list[li] : li;
            /* decode x_t */
            for (int c = 0; c < H; ++c) {
                double s = oracle_ue8m0_decode(scale_byte(x_sf + (size_t)t * (H / 128), c / 32));
                xh[c] = g_e4m3[x[(size_t)t * H + c]] * s;
            }
            for (int d = 0; d < H; ++d) ysum[d] = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t e = idx[(size_t)t * k + j];
                uint8_t* qo = q ? q + ((size_t)li * k + j) * I : NULL;
                int8_t* qeo = qe ? qe + ((size_t)li * k + j) * (I / 32) : NULL;
                if (e < 0) {
                    if (qo) memset(qo, 0, (size_t)I);
                    if (qeo) memset(qeo, 0, (size_t)I / 32);
                    continue;
                }
                double wt = (double)topk_w[(size_t)t * k + j];
                const uint8_t* W1 = w1 + (size_t)e * 2 * I * w1_row;
                const uint32_t* S1 = w1_sf + (size_t)e * 2 * I * w1_sfrow;
                /* L1 + SwiGLU x top-k weight */
                for (int c = 0; c < I; ++c) {
                    int rg = 16 * (c / 8) + c % 8;       /* gate row under the interleave */
                    int ru = rg + 8;                     /* matching up row */
                    double zg = dot_w_row(W1 + rg * w1_row, S1 + rg * w1_sfrow, xh, H);
                    double zu = dot_w_row(W1 + ru * w1_row, S1 + ru * w1_sfrow, xh, H);
                    double g = oracle_bf16_round(zg);
                    double u = oracle_bf16_round(zu);
                    if (clamp > 0.0) {
                        if (g > clamp) g = clamp;
                        if (u > clamp) u = clamp;
                        if (u < -clamp) u = -clamp;
                    }
                    h[c] = oracle_silu(g) * u * wt;
                }
                /* amax -> UE8M0 -> E4M3 per 32 channels; dequantised in place */
                for (int G = 0; G < I / 32; ++G) {
                    double amax = 0.0;
                    for (int c = G * 32; c < G * 32 + 32; ++c) if (fabs(h[c]) > amax) amax = fabs(h[c]);
                    int es = oracle_requant_exponent(amax);
                    if (qeo) qeo[G] = (int8_t)es;
                    for (int c = G * 32; c < G * 32 + 32; ++c) {
                        uint8_t code = oracle_e4m3_encode(ldexp(h[c], -es));
                        if (qo) qo[c] = code;
                        h[c] = oracle_e4m3_decode(code) * ldexp(1.0, es);
                    }
                }
                /* L2, BF16 per slot, accumulate */
                const uint8_t* W2 = w2 + (size_t)e * H * w2_row;
                const uint32_t* S2 = w2_sf + (size_t)e * H * w2_sfrow;
                for (int d = 0; d < H; ++d) {
                    double yd = dot_w_row(W2 + d * w2_row, S2 + d * w2_sfrow, h, I);
                    ysum[d] += oracle_bf16_round(yd);
                }
            }
            for (int d = 0; d < H; ++d) y[(size_t)li * H + d] = oracle_bf16_bits(ysum[d]);
        }
        free(xh);
        free(h);
        free(ysum);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
