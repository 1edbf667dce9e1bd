/*
 * CPU oracle for the NVFP4 (nvfp4/g16) weight-only GEMV.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library. The CUDA library never links, includes
 * or calls it, and this file includes no header of the CUDA library.
 *
 * What it computes (plain definition, fp64, no blocking or reordering):
 *
 *     y[m, n] = g * sum_k E2M1(q[n, k]) * E4M3(s[n, k / 16]) * bf16(x[m, k])
 *
 * Sources on the pages:
 *   - "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[4], [6], [8],
 *     [9] and [33], field `note`: the W4A16 weight is NVFP4, i.e. E2M1 values
 *     with an unsigned E4M3 scale for every 16 weights; the activation is BF16.
 *   - "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json", node l0.kda.q, field
 *     `steps`: activation read as bf16, the nvfp4/g16 weight widened to bf16,
 *     bf16 x bf16 products accumulated in f32, then an f32 scale.
 *   - "GLM-5.3-Flash-NVFP4" blueprint page, section Precision, table of weight
 *     and activation formats: nvfp4/g16 weight with bf16 activation.
 * Readings where the pages are silent (each listed in the design notes):
 *   - element 2j of a row is the LOW nibble of byte j, element 2j+1 the high one;
 *   - packed codes are [N, K/2] bytes and scales [N, K/16] bytes, row-major;
 *   - g is one FP32 scale per weight tensor, applied after the sum;
 *   - the E4M3 sign bit is decoded as in standard E4M3 (the pages say the
 *     scale is unsigned, so valid data never sets it); 0x7F/0xFF are NaN;
 *   - MoE: slot s = t * top_k + j uses expert ids[s] and its own g; x row t
 *     (shared per token) or row s (one row per slot).
 *
 * The FFN block (nvfp4_oracle_ffn_swiglu) composes these: gate/up GEMVs, the clamped SiLU
 * product in fp64, bf16 rounding of that product (nearest, ties to even), then the down GEMV
 * on the rounded values.
 *
 * Decoders follow the bit definitions of the two minifloat formats (OCP
 * Microscaling Formats v1.0): E2M1 has 1 sign, 2 exponent (bias 1) and
 * 1 mantissa bit; E4M3 has 1 sign, 4 exponent (bias 7) and 3 mantissa bits,
 * no infinities, and NaN where all exponent and mantissa bits are set.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. */
double nvfp4_oracle_e2m1(int code) {
    int sign = (code >> 3) & 1;
    int exp_field = (code >> 1) & 3;
    int mant = code & 1;
    double mag;
    if (exp_field == 0) {
        /* subnormal: (mant / 2) * 2^(1 - bias) with bias 1 */
        mag = 0.5 * (double)mant;
    } else {
        mag = ldexp(1.0 + 0.5 * (double)mant, exp_field - 1);
    }
    return sign ? -mag : mag;
}

/* E4M3 (FN variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa. */
double nvfp4_oracle_e4m3(int code) {
    int sign = (code >> 7) & 1;
    int exp_field = (code >> 3) & 15;
    int mant = code & 7;
    double mag;
    if (exp_field == 15 && mant == 7) return NAN;
    if (exp_field == 0) {
        /* subnormal: (mant / 8) * 2^(1 - bias) */
        mag = ldexp((double)mant / 8.0, -6);
    } else {
        mag = ldexp(1.0 + (double)mant / 8.0, exp_field - 7);
    }
    return sign ? -mag : mag;
}

/* bf16 is the top half of an IEEE binary32. */
double nvfp4_oracle_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int nvfp4_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void nvfp4_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Code n of the packed row: the low nibble of byte j is element 2j. */
static int nibble_at(const uint8_t *wrow, int64_t k) {
    return (wrow[k / 2] >> (4 * (k & 1))) & 0xF;
}

/* One output element: returns sum_k E2M1 * E4M3 * x and sum_k |E2M1 * E4M3 * x|. */
static void dot_row(const uint8_t *wrow, const uint8_t *srow, const uint16_t *xrow,
                    int64_t K, double *sum_out, double *abs_out) {
    double sum = 0.0, abs_sum = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double q = nvfp4_oracle_e2m1(nibble_at(wrow, k));
        double s = nvfp4_oracle_e4m3(srow[k / 16]);
        double xv = nvfp4_oracle_bf16(xrow[k]);
        double term = q * s * xv;
        sum += term;
        abs_sum += fabs(term);
    }
    *sum_out = sum;
    *abs_out = abs_sum;
}

/*
 * Dense GEMV.  w: [N, K/2] bytes, s: [N, K/16] bytes, x: [M, K] bf16 bits.
 * rows: the output columns n to compute (NULL = all N, in order); nrows their count.
 * y, yabs: [M, nrows] row-major; yabs[m, i] = |g| * sum_k |term|.
 * Returns 0, or -1 on a bad argument.
 */
int nvfp4_oracle_gemv(const uint8_t *w, const uint8_t *s, double g, const uint16_t *x,
                      int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                      double *y, double *yabs) {
    if (K % 16 != 0 || M < 0 || N < 0 || K < 0) return -1;
    if (rows == NULL) nrows = N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (n < 0 || n >= N) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        const uint8_t *wrow = w + n * (K / 2);
        const uint8_t *srow = s + n * (K / 16);
        for (int64_t m = 0; m < M; ++m) {
            double sum, abs_sum;
            dot_row(wrow, srow, x + m * K, K, &sum, &abs_sum);
            y[m * nrows + i] = g * sum;
            yabs[m * nrows + i] = fabs(g) * abs_sum;
        }
    }
    return 0;
}

/*
 * Gate and up projections of one input, written side by side:
 * y[m, 0:N] = gate GEMV, y[m, N:2N] = up GEMV (the fused "gate|up" projection
 * of "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[9] shape).
 * rows index the 2N concatenated outputs (NULL = all).
 */
int nvfp4_oracle_gemv_gate_up(const uint8_t *wg, const uint8_t *sg, double gg,
                              const uint8_t *wu, const uint8_t *su, double gu,
                              const uint16_t *x, int64_t M, int64_t N, int64_t K,
                              const int64_t *rows, int64_t nrows, double *y, double *yabs) {
    if (K % 16 != 0 || M < 0 || N < 0 || K < 0) return -1;
    if (rows == NULL) nrows = 2 * N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        if (r < 0 || r >= 2 * N) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t r = rows ? rows[i] : i;
        int up = r >= N;
        int64_t n = up ? r - N : r;
        const uint8_t *wrow = (up ? wu : wg) + n * (K / 2);
        const uint8_t *srow = (up ? su : sg) + n * (K / 16);
        double g = up ? gu : gg;
        for (int64_t m = 0; m < M; ++m) {
            double sum, abs_sum;
            dot_row(wrow, srow, x + m * K, K, &sum, &abs_sum);
            y[m * nrows + i] = g * sum;
            yabs[m * nrows + i] = fabs(g) * abs_sum;
        }
    }
    return 0;
}

/*
 * The fused gate/up activation (the swiglu_clamp and silu_mul nodes that follow the gate/up
 * projection in "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json", block l0.mlp; the pages name
 * a clamp but give no limit, so the limit is an argument, +inf for none):
 *     c(v) = v > lim ? lim : (v < -lim ? -lim : v)      (NaN stays NaN)
 *     silu(v) = v / (1 + exp(-v))
 *     swiglu(gate, up) = silu(c(gate)) * c(up).
 */
double nvfp4_oracle_swiglu(double gate, double up, double lim) {
    double gc = gate > lim ? lim : (gate < -lim ? -lim : gate);
    double uc = up > lim ? lim : (up < -lim ? -lim : up);
    return gc / (1.0 + exp(-gc)) * uc;
}

/*
 * Gate/up GEMVs followed by the fused activation: y[m, i] = swiglu(gate[m, n], up[m, n]) for
 * the output columns n = rows[i] (NULL = all N), in fp64. The gate and up values and their
 * |g| * sum |term| scales are returned too ([M, nrows] each; NULL pointers skip them), so a
 * caller can bound how errors in gate and up carry through the activation.
 */
int nvfp4_oracle_gate_up_swiglu(const uint8_t *wg, const uint8_t *sg, double gg,
                                const uint8_t *wu, const uint8_t *su, double gu,
                                const uint16_t *x, double lim, int64_t M, int64_t N, int64_t K,
                                const int64_t *rows, int64_t nrows, double *y,
                                double *gate, double *gate_abs, double *up, double *up_abs) {
    if (K % 16 != 0 || M < 0 || N < 0 || K < 0 || !(lim > 0.0)) return -1;
    if (rows == NULL) nrows = N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (n < 0 || n >= N) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        for (int64_t m = 0; m < M; ++m) {
            double sg_sum, sg_abs, su_sum, su_abs;
            dot_row(wg + n * (K / 2), sg + n * (K / 16), x + m * K, K, &sg_sum, &sg_abs);
            dot_row(wu + n * (K / 2), su + n * (K / 16), x + m * K, K, &su_sum, &su_abs);
            double gv = gg * sg_sum, uv = gu * su_sum;
            y[m * nrows + i] = nvfp4_oracle_swiglu(gv, uv, lim);
            if (gate) gate[m * nrows + i] = gv;
            if (gate_abs) gate_abs[m * nrows + i] = fabs(gg) * sg_abs;
            if (up) up[m * nrows + i] = uv;
            if (up_abs) up_abs[m * nrows + i] = fabs(gu) * su_abs;
        }
    }
    return 0;
}

/*
 * Routed-expert GEMV over slots (the routed gate/up slot GEMV of
 * "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[33]).
 * w: [E, N, K/2], s: [E, N, K/16], gs: [E] per-expert global scales (float).
 * ids: [T * top_k], slot s = t * top_k + j, token-major.
 * x: [T, K] when x_per_slot == 0 (row t), [T * top_k, K] when 1 (row s).
 * rows: output columns to compute (NULL = all N).  y, yabs: [T * top_k, nrows].
 * A slot whose id is outside [0, E) gets zeros and is counted in *bad_ids.
 */
int nvfp4_oracle_moe_gemv(const uint8_t *w, const uint8_t *s, const float *gs, int64_t E,
                          const int32_t *ids, int64_t T, int64_t top_k,
                          const uint16_t *x, int x_per_slot, int64_t N, int64_t K,
                          const int64_t *rows, int64_t nrows, double *y, double *yabs,
                          int64_t *bad_ids) {
    if (K % 16 != 0 || E < 0 || T < 0 || top_k < 0 || N < 0 || K < 0) return -1;
    if (rows == NULL) nrows = N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (n < 0 || n >= N) return -1;
    }
    int64_t slots = T * top_k;
    int64_t bad = 0;
    for (int64_t sl = 0; sl < slots; ++sl)
        if (ids[sl] < 0 || ids[sl] >= E) ++bad;
    if (bad_ids) *bad_ids = bad;
    int64_t sl;
#pragma omp parallel for schedule(static)
    for (sl = 0; sl < slots; ++sl) {
        int64_t e = ids[sl];
        int64_t xrow = x_per_slot ? sl : sl / top_k;
        for (int64_t i = 0; i < nrows; ++i) {
            if (e < 0 || e >= E) {
                y[sl * nrows + i] = 0.0;
                yabs[sl * nrows + i] = 0.0;
                continue;
            }
            int64_t n = rows ? rows[i] : i;
            const uint8_t *wrow = w + (e * N + n) * (K / 2);
            const uint8_t *srow = s + (e * N + n) * (K / 16);
            double g = (double)gs[e];
            double sum, abs_sum;
            dot_row(wrow, srow, x + xrow * K, K, &sum, &abs_sum);
            y[sl * nrows + i] = g * sum;
            yabs[sl * nrows + i] = fabs(g) * abs_sum;
        }
    }
    return 0;
}

/*
 * Scale-dictionary NVFP4 ("glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[64],
 * field `note`: routed gate+up weights at 4.3125 bit/weight with a scale dictionary, while a
 * tensor kept plain reads 4.5). Reading (the pages give only the bit budget):
 *   - the E2M1 codes stay [N, K/2] bytes (4 bits per weight);
 *   - the [N, K/16] E4M3 block scales are replaced by one 5-bit index per 16-element block
 *     into a table `dict` of 32 E4M3 codes for the whole tensor: 4 + 5/16 = 4.3125 bits per
 *     weight. A tensor whose scales need more than 32 codes stays plain (4 + 8/16 = 4.5), so
 *     the coding is exact: block b of row n has the scale E4M3(dict[index(n, b)]);
 *   - index layout: K % 256 == 0; for each 16-row tile r (rows 16r .. 16r + 15; N rounded up
 *     to a multiple of 16) and 256-column segment c (blocks 16c .. 16c + 15) a 160-byte record
 *     at byte (r * (K / 256) + c) * 160 holds the 256 indices of (row 16r + i, block 16c + j)
 *     at position q = 16 i + j, as bits 5q .. 5q + 4 (least significant first) of the record
 *     read as a bit stream in which bit p is bit p % 8 of byte p / 8.
 */
int nvfp4_oracle_sdict_index(const uint8_t *idx, int64_t K, int64_t n, int64_t b) {
    const uint8_t *rec = idx + ((n / 16) * (K / 256) + b / 16) * 160;
    int64_t q = (n % 16) * 16 + (b % 16);
    int v = 0;
    for (int i = 0; i < 5; ++i) {
        int64_t bit = 5 * q + i;
        v |= ((rec[bit / 8] >> (bit % 8)) & 1) << i;
    }
    return v;
}

/* Bytes of the index plane of one [N, K] tensor. */
int64_t nvfp4_oracle_sdict_idx_bytes(int64_t N, int64_t K) {
    return ((N + 15) / 16) * (K / 256) * 160;
}

/* Row n's block scales as plain E4M3 codes: srow[b] = dict[index(n, b)]. */
static void sdict_scale_row(const uint8_t *idx, const uint8_t *dict, int64_t K, int64_t n, uint8_t *srow) {
    for (int64_t b = 0; b < K / 16; ++b) srow[b] = dict[nvfp4_oracle_sdict_index(idx, K, n, b)];
}

/*
 * Dense GEMV with dictionary scales: w [N, K/2], idx (layout above), dict [32] E4M3 codes.
 * Otherwise as nvfp4_oracle_gemv. Returns 0, or -1 on a bad argument (K % 256 != 0 included).
 */
int nvfp4_oracle_gemv_sdict(const uint8_t *w, const uint8_t *idx, const uint8_t *dict, double g,
                            const uint16_t *x, int64_t M, int64_t N, int64_t K, const int64_t *rows,
                            int64_t nrows, double *y, double *yabs) {
    if (K % 256 != 0 || M < 0 || N < 0 || K < 0) return -1;
    if (rows == NULL) nrows = N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (n < 0 || n >= N) return -1;
    }
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        uint8_t srow[4096];
        uint8_t *sr = K / 16 <= 4096 ? srow : (uint8_t *)malloc((size_t)(K / 16));
        sdict_scale_row(idx, dict, K, n, sr);
        for (int64_t m = 0; m < M; ++m) {
            double sum, abs_sum;
            dot_row(w + n * (K / 2), sr, x + m * K, K, &sum, &abs_sum);
            y[m * nrows + i] = g * sum;
            yabs[m * nrows + i] = fabs(g) * abs_sum;
        }
        if (sr != srow) free(sr);
    }
    return 0;
}

/*
 * Routed-expert GEMV with dictionary scales: expert e's index plane starts at
 * idx + e * nvfp4_oracle_sdict_idx_bytes(N, K) and its table at dict + 32 e. Otherwise as
 * nvfp4_oracle_moe_gemv.
 */
int nvfp4_oracle_moe_gemv_sdict(const uint8_t *w, const uint8_t *idx, const uint8_t *dict, const float *gs,
                                int64_t E, const int32_t *ids, int64_t T, int64_t top_k,
                                const uint16_t *x, int x_per_slot, int64_t N, int64_t K,
                                const int64_t *rows, int64_t nrows, double *y, double *yabs,
                                int64_t *bad_ids) {
    if (K % 256 != 0 || E < 0 || T < 0 || top_k < 0 || N < 0 || K < 0) return -1;
    if (rows == NULL) nrows = N;
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t n = rows ? rows[i] : i;
        if (n < 0 || n >= N) return -1;
    }
    int64_t slots = T * top_k;
    int64_t bad = 0;
    for (int64_t sl = 0; sl < slots; ++sl)
        if (ids[sl] < 0 || ids[sl] >= E) ++bad;
    if (bad_ids) *bad_ids = bad;
    int64_t plane = nvfp4_oracle_sdict_idx_bytes(N, K);
    int64_t sl;
#pragma omp parallel for schedule(static)
    for (sl = 0; sl < slots; ++sl) {
        int64_t e = ids[sl];
        int64_t xrow = x_per_slot ? sl : sl / top_k;
        uint8_t srow[4096];
        uint8_t *sr = K / 16 <= 4096 ? srow : (uint8_t *)malloc((size_t)(K / 16));
        for (int64_t i = 0; i < nrows; ++i) {
            if (e < 0 || e >= E) {
                y[sl * nrows + i] = 0.0;
                yabs[sl * nrows + i] = 0.0;
                continue;
            }
            int64_t n = rows ? rows[i] : i;
            sdict_scale_row(idx + e * plane, dict + 32 * e, K, n, sr);
            double g = (double)gs[e];
            double sum, abs_sum;
            dot_row(w + (e * N + n) * (K / 2), sr, x + xrow * K, K, &sum, &abs_sum);
            y[sl * nrows + i] = g * sum;
            yabs[sl * nrows + i] = fabs(g) * abs_sum;
        }
        if (sr != srow) free(sr);
    }
    return 0;
}

/*
 * bf16 nearest-even rounding of an fp64 value, returned as the bf16 bit pattern. bf16 has 8
 * significant bits and binary32's exponent range: the quantum is 2^(e - 7) for
 * 2^e <= |v| < 2^(e + 1), e >= -126, and 2^-133 below 2^-126. A value that rounds to 2^128 or
 * more is infinite; NaN maps to the quiet NaN 0x7FC0. This is the rounding of the silu_mul
 * node's bf16 output in "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json" (l3.moe.shared_act).
 */
uint16_t nvfp4_oracle_bf16_rne(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);  /* a = f * 2^e with 0.5 <= f < 1, so 2^(e - 1) <= a < 2^e */
    int ex = e - 1;
    double q = ex >= -126 ? ldexp(1.0, ex - 7) : ldexp(1.0, -133);
    double m = rint(a / q);  /* nearest, ties to even (the default rounding mode) */
    double r = m * q;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r;      /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/*
 * The shared-expert FFN of "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json" (block l3.moe,
 * nodes shared_gate_up, shared_clamp, shared_act and shared_down, which the plan runs as one
 * group), in the nodes' order:
 *   1. gate and up GEMVs over x [M, H] (weights [I, H/2], scales [I, H/16]);
 *   2. h = silu(clamp(gate)) * clamp(up) (nvfp4_oracle_swiglu), in fp64;
 *   3. h rounded to bf16 (the silu_mul node's output precision);
 *   4. the down GEMV y = gd * W_down . h (weights [H, I/2], scales [H, I/16]).
 * rows: output columns of y to compute (NULL = all H). h_out (fp64, before rounding) and
 * hbits_out (the bf16 h of step 3) are [M, I] and may be NULL; gate, up and their
 * |g| * sum |term| scales go to aux [4][M, I] when aux is not NULL (order: gate, gate_abs,
 * up, up_abs). y and yabs are [M, nrows]; yabs is the down GEMV's |gd| * sum |term| on h.
 */
int nvfp4_oracle_ffn_swiglu(const uint8_t *wg, const uint8_t *sg, double gg,
                            const uint8_t *wu, const uint8_t *su, double gu,
                            const uint8_t *wd, const uint8_t *sd, double gd,
                            const uint16_t *x, double lim, int64_t M, int64_t H, int64_t I,
                            const int64_t *rows, int64_t nrows, double *y, double *yabs,
                            double *h_out, uint16_t *hbits_out, double *aux) {
    if (H % 16 != 0 || I % 16 != 0 || M < 0 || H < 0 || I < 0 || !(lim > 0.0)) return -1;
    double *h = (double *)malloc(sizeof(double) * (size_t)(M * I > 0 ? M * I : 1));
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(M * I > 0 ? M * I : 1));
    if (!h || !hb) {
        free(h);
        free(hb);
        return -2;
    }
    int rc = nvfp4_oracle_gate_up_swiglu(wg, sg, gg, wu, su, gu, x, lim, M, I, H, NULL, I, h,
                                         aux ? aux : NULL, aux ? aux + M * I : NULL,
                                         aux ? aux + 2 * M * I : NULL, aux ? aux + 3 * M * I : NULL);
    if (rc == 0) {
        for (int64_t j = 0; j < M * I; ++j) hb[j] = nvfp4_oracle_bf16_rne(h[j]);
        rc = nvfp4_oracle_gemv(wd, sd, gd, hb, M, H, I, rows, nrows, y, yabs);
        if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)(M * I));
        if (hbits_out) memcpy(hbits_out, hb, sizeof(uint16_t) * (size_t)(M * I));
    }
    free(h);
    free(hb);
    return rc;
}
