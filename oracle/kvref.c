/*
 * kvref.c -- float64 CPU oracle for KVarN-style KV-cache block quantization
 * and for the decode attention that reads the quantized cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline leg do.  It shares no code, header, table or constant with the
 * CUDA path: every layout constant below is restated here on purpose.
 *
 * Method source: "KVarN: Huawei'den KV-Cache Kuantizasyonu icin Yerel vLLM
 * Backend'i" (blog.edumints.com), section "KVarN Nasil Calisir?" (How KVarN
 * works).  That section quantizes the KV cache in fixed-size token blocks and
 * passes every block through four stages:
 *   1. the raw FP16 block ("Onbellek"),
 *   2. an orthonormal Hadamard rotation along the channel dimension
 *      ("Dondurulmus Onbellek"), which spreads outliers and keeps attention
 *      scores unchanged,
 *   3. a Sinkhorn-like row and column variance normalization in the log
 *      domain ("Normalize Edilmis Onbellek"),
 *   4. low-bit asymmetric round-to-nearest, 4-bit keys and 2-bit values
 *      ("Kuantize Edilmis Onbellek").
 * The same page names the format kvarn_k4v2_g128 (section "Yazilim
 * Gelistirme ve Ogrenme Acisindan Pratik Cikarimlar"): group size 128.
 * Decode attention and paging follow "KV Cache (Anahtar-Deger Onbellegi)"
 * (yapayzekasozluk.tr), sections "KV Cache Nasil Calisir?" and "Paged
 * Attention (vLLM)".
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   - block = 128 tokens x 128 channels of one KV head; K and V are separate
 *     tiles and both pass through all four stages;
 *   - Hadamard = Sylvester construction in natural order, scaled by
 *     1/sqrt(128); row y_t = H x_t;
 *   - Sinkhorn: rows = tokens, columns = channels, log scales a_t, b_d start
 *     at 0; one iteration = row step then column step; each step adds
 *     log(sigma) where sigma is the centred population standard deviation
 *     (divide by n) of Z = Y * exp(-a_t - b_d); a step is skipped for a row or
 *     column whose variance is <= 1e-10 * mean(Z^2) of that row or column;
 *     format variant "_rms": sigma is the uncentred root mean square instead
 *     (Sinkhorn-Knopp on the squares), a step skipped only for a zero row or
 *     column;
 *   - group = the 128 channels of one token (per-token groups);
 *   - RTN: z = min, s = (max - min)/(2^b - 1), q = clamp(rint(u)) with
 *     u = (x - z)/s, ties to even; a constant group gives s = 0, q = 0;
 *   - stored metadata is fp32: s' = fp32(r_t s), z' = fp32(r_t z), column
 *     scale c_d = fp32(exp(b_d)); dequantized rotated value
 *     yhat_td = c_d (s'_t q_td + z'_t);
 *   - attention: softmax(q . k * scale) v over every cached token (the
 *     quantized pages, then the newest len mod 128 tokens kept as fp16).
 *
 * Page record (one per page and KV head, 15360 bytes): the K part, then the
 * V part, each holding codes, per-token metadata and per-channel scales:
 *   [0,     8192)  K codes, token-major: row t at 64 t; byte j holds channel
 *                  2j in bits 0-3 and channel 2j+1 in bits 4-7
 *   [8192,  9216)  K per-token {s', z'} fp32 pairs, token t at 8192 + 8 t
 *   [9216,  9728)  K per-channel c_d fp32
 *   [9728, 13824)  V codes, 2 bits each, as 1024 little-endian 32-bit words
 *                  in 16-channel groups: write channel c = 16m + 8e + r
 *                  (m < 8, e < 2, r < 8) and token t = 16k + 8f + 2j + s
 *                  (k < 8, f < 2, j < 4, s < 2); the code of (c, t) is crumb
 *                  i = 2(k mod 4) + f + 8s (bits 2i, 2i+1) of word
 *                  128m + 16r + 4j + 2e + floor(k/4).  This is a fixed
 *                  permutation of the 4096 code bytes (see kvref_v_code_pos)
 *   [13824,14848)  V per-token {s', z'} fp32 pairs
 *   [14848,15360)  V per-channel c_d fp32
 * Pool = [num_pages][num_kv_heads][15360 bytes].
 *
 * Format variant "_m16" (fp16 metadata, 108 B per token-head): the
 * same codes, the same fp32 arithmetic, and every stored s', z', c_d rounded
 * once more to fp16 (IEEE binary16, round to nearest even, overflow to
 * infinity).  Record of 13824 bytes:
 *   [0,     8192)  K codes (as above)
 *   [8192,  8704)  K per-token {s', z'} fp16 pairs, token t at 8192 + 4 t
 *   [8704,  8960)  K per-channel c_d fp16
 *   [8960, 13056)  V codes (the same permutation)
 *   [13056,13568)  V per-token {s', z'} fp16 pairs
 *   [13568,13824)  V per-channel c_d fp16
 *
 * Format variant "_pc" (per-channel grouping): after the same rotation and normalization, one RTN group is
 * one channel's 128 tokens of the tile, so s_d, z_d are per channel and the
 * row scale r_t cannot be folded into them; it is stored per token.  With
 * x_td = Y_td / (r_t c_d): z_d = min_t x_td, s_d = (max_t - min_t) / (2^b - 1),
 * q = rint((x - z_d) / s_d), and yhat_td = r_t (cs_d q_td + cz_d) with
 * cs_d = fp32(c_d s_d), cz_d = fp32(c_d z_d).  Record of 15360 bytes:
 *   [0,     8192)  K codes (as above)
 *   [8192,  8704)  K per-token r_t fp32
 *   [8704,  9728)  K per-channel {cs_d, cz_d} fp32 pairs
 *   [9728, 13824)  V codes (the same permutation)
 *   [13824,14336)  V per-token r_t fp32
 *   [14336,15360)  V per-channel {cs_d, cz_d} fp32 pairs
 *
 * Format variant "k4v2_g64" (group size 64, the "g" of the KVarN page's format
 * name kvarn_k4v2_g128): the same
 * stages with two RTN groups per token, channels 0-63 and 64-127, each with
 * its own {s', z'} (the row scale folded in as in the default).  Record of
 * 17408 bytes (136 B per token-head):
 *   [0,     8192)  K codes (as above)
 *   [8192, 10240)  K {s'_0, z'_0, s'_1, z'_1} fp32 per token (token t at 8192 + 16 t)
 *   [10240,10752)  K per-channel c_d fp32
 *   [10752,14848)  V codes (the same permutation)
 *   [14848,16896)  V {s'_0, z'_0, s'_1, z'_1} fp32 per token
 *   [16896,17408)  V per-channel c_d fp32
 *
 * Format variant "k4v4_g128" (4-bit values, the "v" of the format name): the
 * same stages
 * with 4-bit RTN on V as on K.  The V codes are a fixed permutation of
 * channel-major order chosen like the 2-bit one (see kvref_v4_code_pos):
 * with channel c = 16m + 8e + r and token t = 16k + 8f + 2j + s, the code of
 * (c, t) is nibble n = 4s + 2(k mod 2) + f of 32-bit word
 * 256m + 32r + 8j + 4e + floor(k/2).  Record of 19456 bytes (152 B per
 * token-head):
 *   [0,     9728)  the K part (as in the default)
 *   [9728, 17920)  V codes, 4 bits each, 2048 little-endian 32-bit words
 *   [17920,18944)  V {s', z'} fp32 per token
 *   [18944,19456)  V per-channel c_d fp32
 *
 * Format variant "k8v4_g128" (8-bit keys, 4-bit values): the same stages
 * with 8-bit RTN on K and 4-bit RTN on V.  K codes are token-major, one byte
 * per channel, the 16-byte chunks of odd tokens swapped pairwise: the code of
 * (channel d, token t) is byte 128 t + (d XOR 16 (t mod 2)) (see
 * kvref_k8_code_pos).  V codes as in "k4v4_g128".  Record of 27648 bytes (216 B per token-head):
 *   [0,    16384)  K codes
 *   [16384,17408)  K {s', z'} fp32 per token
 *   [17408,17920)  K per-channel c_d fp32
 *   [17920,26112)  V codes (the 4-bit permutation)
 *   [26112,27136)  V {s', z'} fp32 per token
 *   [27136,27648)  V per-channel c_d fp32
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define NCH 128            /* head_dim = group size */
#define NTOK 128           /* tokens per block / page */
#define REC_BYTES 15360
#define OFF_KCODES 0
#define OFF_KSZ 8192
#define OFF_KC 9216
#define OFF_VCODES 9728
#define OFF_VSZ 13824
#define OFF_VC 14848
#define REC_BYTES_M16 13824
#define REC_BYTES_G64 17408
#define REC_BYTES_V4 19456
#define REC_BYTES_K8 27648
#define G64 64

/* Offsets of the record parts for the two metadata widths. */
typedef struct {
    long rec, kcodes, ksz, kc, vcodes, vsz, vc;
    int msz;   /* bytes of one stored metadata value: 4 (fp32) or 2 (fp16) */
} rec_layout;

/* fmt: 0 = fp32 metadata, 1 = "_m16" (fp16 metadata), 2 = "_pc" (per-channel
 * groups; ksz / vsz hold r_t, kc / vc the {cs, cz} pairs), 3 = "g64" (two
 * groups per token; ksz / vsz hold two {s', z'} pairs per token) */
static rec_layout layout_of(int fmt)
{
    rec_layout L;
    if (fmt == 1) {
        L.rec = REC_BYTES_M16; L.kcodes = 0; L.ksz = 8192; L.kc = 8704;
        L.vcodes = 8960; L.vsz = 13056; L.vc = 13568; L.msz = 2;
    } else if (fmt == 2) {
        L.rec = REC_BYTES; L.kcodes = 0; L.ksz = 8192; L.kc = 8704;
        L.vcodes = 9728; L.vsz = 13824; L.vc = 14336; L.msz = 4;
    } else if (fmt == 3) {
        L.rec = REC_BYTES_G64; L.kcodes = 0; L.ksz = 8192; L.kc = 10240;
        L.vcodes = 10752; L.vsz = 14848; L.vc = 16896; L.msz = 4;
    } else if (fmt == 4) {
        L.rec = REC_BYTES_V4; L.kcodes = 0; L.ksz = 8192; L.kc = 9216;
        L.vcodes = 9728; L.vsz = 17920; L.vc = 18944; L.msz = 4;
    } else if (fmt == 5) {
        L.rec = REC_BYTES_K8; L.kcodes = 0; L.ksz = 16384; L.kc = 17408;
        L.vcodes = 17920; L.vsz = 26112; L.vc = 27136; L.msz = 4;
    } else {
        L.rec = REC_BYTES; L.kcodes = OFF_KCODES; L.ksz = OFF_KSZ; L.kc = OFF_KC;
        L.vcodes = OFF_VCODES; L.vsz = OFF_VSZ; L.vc = OFF_VC; L.msz = 4;
    }
    return L;
}

long kvref_record_bytes(int fmt) { return layout_of(fmt).rec; }

/* ------------------------------------------------------------------ */
/* fp16 <-> double, written out from the IEEE-754 binary16 definition */
/* ------------------------------------------------------------------ */

double kvref_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)mant, -24);              /* subnormal or zero */
    } else if (expo == 31) {
        v = mant ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + mant), expo - 25);
    }
    return sign ? -v : v;
}

/* float -> binary16, round to nearest even, from the definition: the value
 * is an integer multiple of the fp16 spacing 2^(e - 10) of its binade (2^-24
 * for the subnormals); the exact quotient is rounded to the nearest integer,
 * ties to the even one, and a result of 2^11 spacings carries into the next
 * binade.  Beyond the largest finite value (65504, or from 65520 on after
 * rounding) the result is infinity; NaN stays NaN. */
uint16_t kvref_f32_to_f16(float f)
{
    double x = (double)f, a = fabs(x), m, fl;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    int e;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    if (a == 0.0) return sign;
    e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a) e -= 1;          /* guard the log2 rounding */
    if (ldexp(1.0, e + 1) <= a) e += 1;
    if (e < -14) e = -14;                    /* subnormal spacing 2^-24 */
    m = ldexp(a, 10 - e);                    /* spacings of 2^(e - 10), exact */
    fl = floor(m);
    if (m - fl > 0.5 || (m - fl == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    if (fl >= 2048.0) {                      /* carried into the next binade */
        fl /= 2.0;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7c00);
    if (fl < 1024.0) return (uint16_t)(sign | (uint16_t)fl);          /* subnormal */
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(fl - 1024.0));
}

/* ------------------------------------------------------------------ */
/* Stage 2: orthonormal Hadamard rotation along channels               */
/* KVarN page, "KVarN Nasil Calisir?", stage "Dondurulmus Onbellek".    */
/* ------------------------------------------------------------------ */

/* Sylvester recursion H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]], then the
 * whole matrix is scaled by 1/sqrt(n) so that H H^T = I.  n: power of two. */
void kvref_hadamard(int n, double *H)
{
    int m, i, j;
    for (i = 0; i < n * n; ++i) H[i] = 0.0;
    H[0] = 1.0;
    for (m = 1; m < n; m *= 2) {
        for (i = 0; i < m; ++i) {
            for (j = 0; j < m; ++j) {
                double h = H[i * n + j];
                H[i * n + (j + m)] = h;
                H[(i + m) * n + j] = h;
                H[(i + m) * n + (j + m)] = -h;
            }
        }
    }
    for (i = 0; i < n * n; ++i) H[i] /= sqrt((double)n);
}

/* Y = X H^T, y_t = H x_t for every token row, as an explicit matrix product
 * taken in two exact-then-rounded steps: each row of H is (+-1) / sqrt(n), so
 * y_td = (sum_j sign(H_dj) x_tj) / sqrt(n).  The signed sum of fp16 inputs is
 * exact in float64 (every fp16 value is a multiple of 2^-24 below 2^16, so
 * any sum of 128 of them fits in 53 bits); the division rounds once.  A
 * rotated value that is zero in exact arithmetic is therefore exactly zero
 * here, which the skip rules of the normalization rely on.
 * x: NTOK x NCH fp16 bit patterns, token t at x + t * ld_tok.  Y: NTOK x NCH. */
void kvref_rotate_tile(const uint16_t *x, long ld_tok, const double *H, double *Y)
{
    int t, d, j;
    double xt[NCH];
    const double root = sqrt((double)NCH);
    for (t = 0; t < NTOK; ++t) {
        for (j = 0; j < NCH; ++j) xt[j] = kvref_half_to_double(x[t * ld_tok + j]);
        for (d = 0; d < NCH; ++d) {
            double acc = 0.0;
            for (j = 0; j < NCH; ++j) acc += H[d * NCH + j] > 0.0 ? xt[j] : -xt[j];
            Y[t * NCH + d] = acc / root;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Stage 3: Sinkhorn-like row/column variance normalization, log domain */
/* KVarN page, "KVarN Nasil Calisir?", stage "Normalize Edilmis Onbellek" */
/* ------------------------------------------------------------------ */

/* Whether a row or column step updates its scale.  Centred statistic (the
 * reading of the KVarN page's "variance"): the step is skipped when the
 * variance is at most 1e-10 of the mean square (constant or zero rows).
 * Uncentred statistic (format variant "_rms": the literal Sinkhorn-Knopp
 * scaling of the squares, sigma = root mean square): skipped only for an
 * all-zero row or column. */
static int step_applies(int stat, double var, double msq)
{
    return stat ? msq > 0.0 : var > 1e-10 * msq;
}

/* Centred population statistics of v[0..n-1], two passes. */
static void centred_stats(const double *v, int n, double *var, double *mean_sq)
{
    int i;
    double mean = 0.0, acc = 0.0, sq = 0.0;
    for (i = 0; i < n; ++i) mean += v[i];
    mean /= n;
    for (i = 0; i < n; ++i) {
        double e = v[i] - mean;
        acc += e * e;
        sq += v[i] * v[i];
    }
    *var = acc / n;
    *mean_sq = sq / n;
}

/* Runs `iters` iterations (row step, then column step) on the rotated tile Y
 * (NTOK x NCH) with the centred statistic (stat = 0) or the uncentred one
 * (stat = 1, below).  Output: log row scales a[NTOK] and log column scales
 * b[NCH].
 * trace (nullable, 4*iters entries): for iteration k, trace[4k] is the largest
 * |log sigma| over the rows that the row step updated and trace[4k+1] the
 * spread (largest minus smallest log sigma) over those rows; trace[4k+2] and
 * trace[4k+3] are the same two figures for the column step.  The centred
 * statistics admit no exact joint fixed point in general (row and column means
 * differ), so log sigma settles to a common per-step offset while the spread
 * goes to zero: the spread is the convergence measure. */
void kvref_sinkhorn_stat(const double *Y, int iters, int stat, double *a, double *b,
                         double *trace)
{
    int k, t, d;
    double z[NTOK > NCH ? NTOK : NCH];
    double ea[NTOK], eb[NCH];
    for (t = 0; t < NTOK; ++t) a[t] = 0.0;
    for (d = 0; d < NCH; ++d) b[d] = 0.0;
    for (k = 0; k < iters; ++k) {
        double worst = 0.0, lo = INFINITY, hi = -INFINITY;
        /* row step: normalise each token row by its current std */
        for (d = 0; d < NCH; ++d) eb[d] = exp(-b[d]);
        for (t = 0; t < NTOK; ++t) {
            double var, msq;
            double e = exp(-a[t]);
            for (d = 0; d < NCH; ++d) z[d] = Y[t * NCH + d] * e * eb[d];
            centred_stats(z, NCH, &var, &msq);
            if (step_applies(stat, var, msq)) {
                double ls = log(sqrt(stat ? msq : var));
                a[t] += ls;
                if (fabs(ls) > worst) worst = fabs(ls);
                if (ls < lo) lo = ls;
                if (ls > hi) hi = ls;
            }
        }
        if (trace) {
            trace[4 * k] = worst;
            trace[4 * k + 1] = hi >= lo ? hi - lo : 0.0;
        }
        worst = 0.0;
        lo = INFINITY;
        hi = -INFINITY;
        /* column step: normalise each channel column by its current std */
        for (t = 0; t < NTOK; ++t) ea[t] = exp(-a[t]);
        for (d = 0; d < NCH; ++d) {
            double var, msq;
            double e = exp(-b[d]);
            for (t = 0; t < NTOK; ++t) z[t] = Y[t * NCH + d] * ea[t] * e;
            centred_stats(z, NTOK, &var, &msq);
            if (step_applies(stat, var, msq)) {
                double ls = log(sqrt(stat ? msq : var));
                b[d] += ls;
                if (fabs(ls) > worst) worst = fabs(ls);
                if (ls < lo) lo = ls;
                if (ls > hi) hi = ls;
            }
        }
        if (trace) {
            trace[4 * k + 2] = worst;
            trace[4 * k + 3] = hi >= lo ? hi - lo : 0.0;
        }
    }
}

/* The default (centred) statistic. */
void kvref_sinkhorn(const double *Y, int iters, double *a, double *b, double *trace)
{
    kvref_sinkhorn_stat(Y, iters, 0, a, b, trace);
}

/* ------------------------------------------------------------------ */
/* Stage 4: asymmetric round-to-nearest, per-token groups of 128        */
/* KVarN page, "KVarN Nasil Calisir?", stage "Kuantize Edilmis Onbellek"; */
/* format name kvarn_k4v2_g128 (4-bit K, 2-bit V, group 128).           */
/* ------------------------------------------------------------------ */

/* Normalised tile Xn_td = Y_td / (r_t c32_d), then per row t:
 * z = min_d Xn, s = (max - min)/(2^bits - 1), u = (Xn - z)/s,
 * q = clamp(rint(u), 0, 2^bits - 1); metadata s' = fp32(r s), z' = fp32(r z).
 * u (nullable) receives the pre-rounding value for the boundary rule. */
void kvref_rtn(const double *Y, const double *r, const float *c32, int bits,
               uint8_t *q, float *s32, float *z32, double *u)
{
    int t, d;
    int qmax = (1 << bits) - 1;
    for (t = 0; t < NTOK; ++t) {
        double xn[NCH];
        double mn = INFINITY, mx = -INFINITY, s, z;
        for (d = 0; d < NCH; ++d) {
            xn[d] = Y[t * NCH + d] / (r[t] * (double)c32[d]);
            if (xn[d] < mn) mn = xn[d];
            if (xn[d] > mx) mx = xn[d];
        }
        z = mn;
        s = (mx - mn) / qmax;
        s32[t] = (float)(r[t] * s);
        z32[t] = (float)(r[t] * z);
        for (d = 0; d < NCH; ++d) {
            double ud = 0.0;
            long qi = 0;
            if (s > 0.0) {
                ud = (xn[d] - z) / s;
                qi = (long)nearbyint(ud);          /* ties to even */
                if (qi < 0) qi = 0;
                if (qi > qmax) qi = qmax;
            }
            q[t * NCH + d] = (uint8_t)qi;
            if (u) u[t * NCH + d] = ud;
        }
    }
}

/* Format "_pc": RTN with one group per channel (over the 128 tokens of the
 * tile).  Outputs the codes, r32_t = fp32(r_t), and per channel
 * cs32_d = fp32(c_d s_d), cz32_d = fp32(c_d z_d); u as in kvref_rtn. */
void kvref_rtn_pc(const double *Y, const double *r, const float *c32, int bits, uint8_t *q,
                  float *r32, float *cs32, float *cz32, double *u)
{
    int t, d;
    int qmax = (1 << bits) - 1;
    for (t = 0; t < NTOK; ++t) r32[t] = (float)r[t];
    for (d = 0; d < NCH; ++d) {
        double mn = INFINITY, mx = -INFINITY, s, z;
        for (t = 0; t < NTOK; ++t) {
            double x = Y[t * NCH + d] / (r[t] * (double)c32[d]);
            if (x < mn) mn = x;
            if (x > mx) mx = x;
        }
        z = mn;
        s = (mx - mn) / qmax;
        cs32[d] = (float)((double)c32[d] * s);
        cz32[d] = (float)((double)c32[d] * z);
        for (t = 0; t < NTOK; ++t) {
            double x = Y[t * NCH + d] / (r[t] * (double)c32[d]);
            double ud = 0.0;
            long qi = 0;
            if (s > 0.0) {
                ud = (x - z) / s;
                qi = (long)nearbyint(ud);          /* ties to even */
                if (qi < 0) qi = 0;
                if (qi > qmax) qi = qmax;
            }
            q[t * NCH + d] = (uint8_t)qi;
            if (u) u[t * NCH + d] = ud;
        }
    }
}

/* Format "g64": RTN with two groups of 64 channels per token.  s32, z32:
 * [NTOK][2] (group g of token t at 2 t + g); u as in kvref_rtn. */
void kvref_rtn_g64(const double *Y, const double *r, const float *c32, int bits, uint8_t *q,
                   float *s32, float *z32, double *u)
{
    int t, d, g;
    int qmax = (1 << bits) - 1;
    for (t = 0; t < NTOK; ++t) {
        for (g = 0; g < NCH / G64; ++g) {
            double xn[G64];
            double mn = INFINITY, mx = -INFINITY, s, z;
            for (d = 0; d < G64; ++d) {
                int c = g * G64 + d;
                xn[d] = Y[t * NCH + c] / (r[t] * (double)c32[c]);
                if (xn[d] < mn) mn = xn[d];
                if (xn[d] > mx) mx = xn[d];
            }
            z = mn;
            s = (mx - mn) / qmax;
            s32[2 * t + g] = (float)(r[t] * s);
            z32[2 * t + g] = (float)(r[t] * z);
            for (d = 0; d < G64; ++d) {
                int c = g * G64 + d;
                double ud = 0.0;
                long qi = 0;
                if (s > 0.0) {
                    ud = (xn[d] - z) / s;
                    qi = (long)nearbyint(ud);      /* ties to even */
                    if (qi < 0) qi = 0;
                    if (qi > qmax) qi = qmax;
                }
                q[t * NCH + c] = (uint8_t)qi;
                if (u) u[t * NCH + c] = ud;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Packing into a page record                                          */
/* ------------------------------------------------------------------ */

static void put_f32(uint8_t *p, float v) { memcpy(p, &v, 4); }
static float get_f32(const uint8_t *p) { float v; memcpy(&v, p, 4); return v; }

/* Where the 2-bit V code of channel c, token t lives inside the V code region:
 * byte offset and bit shift.  The split of c and t into digits and the word /
 * crumb formulas are the layout stated in the header comment of this file:
 * c = 16m + 8e + r, t = 16k + 8f + 2j + s, word 128m + 16r + 4j + 2e + k/4,
 * crumb 2(k%4) + f + 8s, little-endian words. */
void kvref_v_code_pos(int c, int t, int *byte, int *shift)
{
    int m = c / 16, e = (c / 8) % 2, r = c % 8;
    int k = t / 16, f = (t / 8) % 2, j = (t / 2) % 4, s = t % 2;
    int word = 128 * m + 16 * r + 4 * j + 2 * e + k / 4;
    int crumb = 2 * (k % 4) + f + 8 * s;
    *byte = 4 * word + crumb / 4;
    *shift = 2 * (crumb % 4);
}

static void put_meta(uint8_t *p, float v, int meta16)
{
    if (meta16) {
        uint16_t h = kvref_f32_to_f16(v);
        memcpy(p, &h, 2);
    } else {
        put_f32(p, v);
    }
}

static float get_meta(const uint8_t *p, int meta16)
{
    if (meta16) {
        uint16_t h;
        memcpy(&h, p, 2);
        return (float)kvref_half_to_double(h);   /* exact */
    }
    return get_f32(p);
}

/* Where the 4-bit V code of channel c, token t lives inside the V code
 * region of the "k4v4_g128" record: byte offset and bit shift.  Digits as in
 * kvref_v_code_pos; word 256m + 32r + 8j + 4e + floor(k/2), nibble
 * 4s + 2(k mod 2) + f (nibble n at bits 4n of the little-endian word). */
/* Byte of the 8-bit K code of channel d, token t (format "k8v4_g128"). */
int kvref_k8_code_pos(int d, int t)
{
    return NCH * t + (d ^ (16 * (t & 1)));
}

void kvref_v4_code_pos(int c, int t, int *byte, int *shift)
{
    int m = c / 16, e = (c / 8) % 2, r = c % 8;
    int k = t / 16, f = (t / 8) % 2, j = (t / 2) % 4, s = t % 2;
    int word = 256 * m + 32 * r + 8 * j + 4 * e + k / 2;
    int nib = 4 * s + 2 * (k % 2) + f;
    *byte = 4 * word + nib / 2;
    *shift = 4 * (nib % 2);
}

/* is_v = 0: K part (4-bit, token-major); is_v = 1: V part (2-bit, permuted;
 * 4-bit for fmt 4).  fmt: the record format (layout_of); fmt 1 stores the
 * metadata as fp16. */
void kvref_pack_part_fmt(uint8_t *rec, int is_v, const uint8_t *q, const float *s32,
                         const float *z32, const float *c32, int fmt)
{
    rec_layout L = layout_of(fmt);
    long sz = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    const int meta16 = fmt == 1;
    int t, d, j;
    if (!is_v && fmt == 5) {
        for (t = 0; t < NTOK; ++t)
            for (d = 0; d < NCH; ++d) rec[L.kcodes + kvref_k8_code_pos(d, t)] = q[t * NCH + d];
    } else if (is_v && (fmt == 4 || fmt == 5)) {
        memset(rec + L.vcodes, 0, NTOK * NCH / 2);
        for (t = 0; t < NTOK; ++t)
            for (d = 0; d < NCH; ++d) {
                int byte, shift;
                kvref_v4_code_pos(d, t, &byte, &shift);
                rec[L.vcodes + byte] |= (uint8_t)((q[t * NCH + d] & 15) << shift);
            }
    } else if (!is_v) {
        for (t = 0; t < NTOK; ++t)
            for (j = 0; j < NCH / 2; ++j)
                rec[L.kcodes + t * 64 + j] =
                    (uint8_t)((q[t * NCH + 2 * j] & 15) | ((q[t * NCH + 2 * j + 1] & 15) << 4));
    } else {
        memset(rec + L.vcodes, 0, NTOK * NCH / 4);
        for (t = 0; t < NTOK; ++t)
            for (d = 0; d < NCH; ++d) {
                int byte, shift;
                kvref_v_code_pos(d, t, &byte, &shift);
                rec[L.vcodes + byte] |= (uint8_t)((q[t * NCH + d] & 3) << shift);
            }
    }
    for (t = 0; t < NTOK; ++t) {
        put_meta(rec + sz + 2 * L.msz * t, s32[t], meta16);
        put_meta(rec + sz + 2 * L.msz * t + L.msz, z32[t], meta16);
    }
    for (d = 0; d < NCH; ++d) put_meta(rec + cc + L.msz * d, c32[d], meta16);
}

void kvref_pack_part(uint8_t *rec, int is_v, const uint8_t *q, const float *s32,
                     const float *z32, const float *c32)
{
    kvref_pack_part_fmt(rec, is_v, q, s32, z32, c32, 0);
}

/* Inverse of kvref_pack_part_fmt for the codes and metadata (fp16 metadata
 * returned as the floats it represents). */
void kvref_unpack_part_fmt(const uint8_t *rec, int is_v, uint8_t *q, float *s32, float *z32,
                           float *c32, int fmt)
{
    rec_layout L = layout_of(fmt);
    long sz = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    const int meta16 = fmt == 1;
    int t, d;
    for (t = 0; t < NTOK; ++t) {
        for (d = 0; d < NCH; ++d) {
            if (!is_v && fmt == 5) {
                q[t * NCH + d] = rec[L.kcodes + kvref_k8_code_pos(d, t)];
            } else if (is_v && (fmt == 4 || fmt == 5)) {
                int byte, shift;
                kvref_v4_code_pos(d, t, &byte, &shift);
                q[t * NCH + d] = (uint8_t)((rec[L.vcodes + byte] >> shift) & 15);
            } else if (!is_v) {
                uint8_t byte = rec[L.kcodes + t * 64 + d / 2];
                q[t * NCH + d] = (uint8_t)((byte >> (4 * (d % 2))) & 15);
            } else {
                int byte, shift;
                kvref_v_code_pos(d, t, &byte, &shift);
                q[t * NCH + d] = (uint8_t)((rec[L.vcodes + byte] >> shift) & 3);
            }
        }
        s32[t] = get_meta(rec + sz + 2 * L.msz * t, meta16);
        z32[t] = get_meta(rec + sz + 2 * L.msz * t + L.msz, meta16);
    }
    for (d = 0; d < NCH; ++d) c32[d] = get_meta(rec + cc + L.msz * d, meta16);
}

void kvref_unpack_part(const uint8_t *rec, int is_v, uint8_t *q, float *s32, float *z32,
                       float *c32)
{
    kvref_unpack_part_fmt(rec, is_v, q, s32, z32, c32, 0);
}

/* Format "_pc": codes as in the other formats, r_t per token, {cs_d, cz_d}
 * per channel. */
void kvref_pack_part_pc(uint8_t *rec, int is_v, const uint8_t *q, const float *r32,
                        const float *cs32, const float *cz32)
{
    rec_layout L = layout_of(2);
    long rr = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    float zero[NTOK];
    int t, d;
    memset(zero, 0, sizeof(zero));
    /* the codes: the shared packer, metadata overwritten below */
    kvref_pack_part_fmt(rec, is_v, q, zero, zero, zero, 0);
    for (t = 0; t < NTOK; ++t) put_f32(rec + rr + 4 * t, r32[t]);
    for (d = 0; d < NCH; ++d) {
        put_f32(rec + cc + 8 * d, cs32[d]);
        put_f32(rec + cc + 8 * d + 4, cz32[d]);
    }
}

void kvref_unpack_part_pc(const uint8_t *rec, int is_v, uint8_t *q, float *r32, float *cs32,
                          float *cz32)
{
    rec_layout L = layout_of(2);
    long rr = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    float s32[NTOK], z32[NTOK], c32[NCH];
    int t, d;
    kvref_unpack_part_fmt(rec, is_v, q, s32, z32, c32, 0);   /* the codes */
    for (t = 0; t < NTOK; ++t) r32[t] = get_f32(rec + rr + 4 * t);
    for (d = 0; d < NCH; ++d) {
        cs32[d] = get_f32(rec + cc + 8 * d);
        cz32[d] = get_f32(rec + cc + 8 * d + 4);
    }
}

/* Format "g64": codes as in the other formats (at this format's offsets), two
 * {s', z'} pairs per token, c_d per channel.  s32, z32: [NTOK][2]. */
void kvref_pack_part_g64(uint8_t *rec, int is_v, const uint8_t *q, const float *s32,
                         const float *z32, const float *c32)
{
    rec_layout L = layout_of(3), L0 = layout_of(0);
    long sz = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    uint8_t tmp[REC_BYTES];
    float zero[NTOK];
    int t, d, g;
    memset(zero, 0, sizeof(zero));
    /* the codes: the shared packer into a scratch record, copied across */
    kvref_pack_part_fmt(tmp, is_v, q, zero, zero, zero, 0);
    if (is_v)
        memcpy(rec + L.vcodes, tmp + L0.vcodes, NTOK * NCH / 4);
    else
        memcpy(rec + L.kcodes, tmp + L0.kcodes, NTOK * NCH / 2);
    for (t = 0; t < NTOK; ++t)
        for (g = 0; g < 2; ++g) {
            put_f32(rec + sz + 16 * t + 8 * g, s32[2 * t + g]);
            put_f32(rec + sz + 16 * t + 8 * g + 4, z32[2 * t + g]);
        }
    for (d = 0; d < NCH; ++d) put_f32(rec + cc + 4 * d, c32[d]);
}

void kvref_unpack_part_g64(const uint8_t *rec, int is_v, uint8_t *q, float *s32, float *z32,
                           float *c32)
{
    rec_layout L = layout_of(3), L0 = layout_of(0);
    long sz = is_v ? L.vsz : L.ksz, cc = is_v ? L.vc : L.kc;
    uint8_t tmp[REC_BYTES];
    float a[NTOK], b[NTOK], c[NCH];
    int t, d, g;
    memset(tmp, 0, sizeof(tmp));
    if (is_v)
        memcpy(tmp + L0.vcodes, rec + L.vcodes, NTOK * NCH / 4);
    else
        memcpy(tmp + L0.kcodes, rec + L.kcodes, NTOK * NCH / 2);
    kvref_unpack_part_fmt(tmp, is_v, q, a, b, c, 0);   /* the codes */
    for (t = 0; t < NTOK; ++t)
        for (g = 0; g < 2; ++g) {
            s32[2 * t + g] = get_f32(rec + sz + 16 * t + 8 * g);
            z32[2 * t + g] = get_f32(rec + sz + 16 * t + 8 * g + 4);
        }
    for (d = 0; d < NCH; ++d) c32[d] = get_f32(rec + cc + 4 * d);
}

/* Dequantized rotated tile from a record: yhat_td = c_d (s'_t q_td + z'_t), or
 * for "_pc" yhat_td = r_t (cs_d q_td + cz_d), or for "g64"
 * yhat_td = c_d (s'_{t,g} q_td + z'_{t,g}) with g = d / 64. */
void kvref_dequant_part_fmt(const uint8_t *rec, int is_v, int fmt, double *yhat)
{
    uint8_t q[NTOK * NCH];
    float a32[NTOK], b32[NTOK > NCH ? NTOK : NCH], c32[NCH];
    int t, d;
    if (fmt == 3) {
        float s2[2 * NTOK], z2[2 * NTOK];
        kvref_unpack_part_g64(rec, is_v, q, s2, z2, c32);
        for (t = 0; t < NTOK; ++t)
            for (d = 0; d < NCH; ++d) {
                int g = d / G64;
                yhat[t * NCH + d] = (double)c32[d] * ((double)s2[2 * t + g] * q[t * NCH + d] +
                                                      (double)z2[2 * t + g]);
            }
        return;
    }
    if (fmt == 2) {
        kvref_unpack_part_pc(rec, is_v, q, a32, b32, c32);
        for (t = 0; t < NTOK; ++t)
            for (d = 0; d < NCH; ++d)
                yhat[t * NCH + d] =
                    (double)a32[t] * ((double)b32[d] * q[t * NCH + d] + (double)c32[d]);
        return;
    }
    kvref_unpack_part_fmt(rec, is_v, q, a32, b32, c32, fmt);
    for (t = 0; t < NTOK; ++t)
        for (d = 0; d < NCH; ++d)
            yhat[t * NCH + d] = (double)c32[d] * ((double)a32[t] * q[t * NCH + d] + (double)b32[t]);
}

void kvref_dequant_part(const uint8_t *rec, int is_v, double *yhat)
{
    kvref_dequant_part_fmt(rec, is_v, 0, yhat);
}

/* ------------------------------------------------------------------ */
/* One tile through all four stages                                    */
/* ------------------------------------------------------------------ */

/* Quantizes one 128x128 fp16 tile (token t at x + t*ld_tok) and packs it into
 * the K (is_v = 0, 4 bits) or V (is_v = 1, 2 bits) part of `rec`.  The
 * optional outputs expose every intermediate for the tests:
 * Y (rotated), a, b (log scales), q (codes), u (pre-rounding values). */
void kvref_quantize_tile_fmt(const uint16_t *x, long ld_tok, int is_v, int iters, int stat,
                             int fmt, uint8_t *rec, double *Y_out, double *a_out,
                             double *b_out, uint8_t *q_out, double *u_out)
{
    static double H[NCH * NCH];
    static int have_h = 0;
    double *Y = (double *)malloc(sizeof(double) * NTOK * NCH);
    double a[NTOK], b[NCH], r[NTOK];
    float c32[NCH], s32[NTOK], z32[NTOK];
    uint8_t q[NTOK * NCH];
    int t, d, bits = is_v ? (fmt == 4 || fmt == 5 ? 4 : 2) : (fmt == 5 ? 8 : 4);
#pragma omp critical(kvref_h)
    {
        if (!have_h) {
            kvref_hadamard(NCH, H);
            have_h = 1;
        }
    }
    kvref_rotate_tile(x, ld_tok, H, Y);
    kvref_sinkhorn_stat(Y, iters, stat, a, b, NULL);
    for (t = 0; t < NTOK; ++t) r[t] = exp(a[t]);
    for (d = 0; d < NCH; ++d) c32[d] = (float)exp(b[d]);
    if (fmt == 2) {
        float r32[NTOK], cs32[NCH], cz32[NCH];
        kvref_rtn_pc(Y, r, c32, bits, q, r32, cs32, cz32, u_out);
        if (rec) kvref_pack_part_pc(rec, is_v, q, r32, cs32, cz32);
    } else if (fmt == 3) {
        float s2[2 * NTOK], z2[2 * NTOK];
        kvref_rtn_g64(Y, r, c32, bits, q, s2, z2, u_out);
        if (rec) kvref_pack_part_g64(rec, is_v, q, s2, z2, c32);
    } else {
        kvref_rtn(Y, r, c32, bits, q, s32, z32, u_out);
        if (rec) kvref_pack_part_fmt(rec, is_v, q, s32, z32, c32, fmt);
    }
    if (Y_out) memcpy(Y_out, Y, sizeof(double) * NTOK * NCH);
    if (a_out) memcpy(a_out, a, sizeof(a));
    if (b_out) memcpy(b_out, b, sizeof(b));
    if (q_out) memcpy(q_out, q, sizeof(q));
    free(Y);
}

void kvref_quantize_tile_stat(const uint16_t *x, long ld_tok, int is_v, int iters, int stat,
                              uint8_t *rec, double *Y_out, double *a_out, double *b_out,
                              uint8_t *q_out, double *u_out)
{
    kvref_quantize_tile_fmt(x, ld_tok, is_v, iters, stat, 0, rec, Y_out, a_out, b_out, q_out,
                            u_out);
}

void kvref_quantize_tile(const uint16_t *x, long ld_tok, int is_v, int iters, uint8_t *rec,
                         double *Y_out, double *a_out, double *b_out, uint8_t *q_out,
                         double *u_out)
{
    kvref_quantize_tile_stat(x, ld_tok, is_v, iters, 0, rec, Y_out, a_out, b_out, q_out, u_out);
}

/* ------------------------------------------------------------------ */
/* Prefill: every full 128-token block into its page, the rest to the tail */
/* Paging: "KV Cache (Anahtar-Deger Onbellegi)", "Paged Attention (vLLM)". */
/* ------------------------------------------------------------------ */

/* k, v: fp16 [B][S][Hkv][128] addressed with element strides sb, st, sh.
 * block_table: [B][max_blocks] page ids.  pool: [num_pages][Hkv][15360].
 * tail_k, tail_v: fp16 [B][Hkv][128 slots][128].  u_k, u_v (nullable):
 * pre-rounding values, [B][max_blocks][Hkv][128][128] doubles, for the
 * boundary rule.  Returns 0, or -1 on a page id outside [0, num_pages). */
int kvref_quantize_blocks_fmt(const uint16_t *k, const uint16_t *v, long sb, long st, long sh,
                              int B, const int32_t *seq_lens, const int32_t *block_table,
                              int max_blocks, int hkv, int iters, int stat, int fmt,
                              uint8_t *pool, long num_pages, uint16_t *tail_k, uint16_t *tail_v,
                              double *u_k, double *u_v)
{
    int bad = 0;
    const long rec_bytes = layout_of(fmt).rec;
    long item, n_items = (long)B * max_blocks * hkv;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
    for (item = 0; item < n_items; ++item) {
        int b = (int)(item / ((long)max_blocks * hkv));
        int j = (int)((item / hkv) % max_blocks);
        int h = (int)(item % hkv);
        int nfull = seq_lens[b] / NTOK;
        long page;
        uint8_t *rec;
        long uoff = (((long)b * max_blocks + j) * hkv + h) * NTOK * NCH;
        if (j >= nfull) continue;
        page = block_table[(long)b * max_blocks + j];
        if (page < 0 || page >= num_pages) { bad = 1; continue; }
        rec = pool + (page * hkv + h) * rec_bytes;
        kvref_quantize_tile_fmt(k + b * sb + (long)j * NTOK * st + h * sh, st, 0, iters, stat,
                                fmt, rec, NULL, NULL, NULL, NULL, u_k ? u_k + uoff : NULL);
        kvref_quantize_tile_fmt(v + b * sb + (long)j * NTOK * st + h * sh, st, 1, iters, stat,
                                fmt, rec, NULL, NULL, NULL, NULL, u_v ? u_v + uoff : NULL);
    }
    {
        int b, h, s, d;
        for (b = 0; b < B; ++b) {
            int nfull = seq_lens[b] / NTOK, rem = seq_lens[b] % NTOK;
            for (h = 0; h < hkv; ++h)
                for (s = 0; s < rem; ++s) {
                    long src = b * sb + ((long)nfull * NTOK + s) * st + h * sh;
                    long dst = (((long)b * hkv + h) * NTOK + s) * NCH;
                    for (d = 0; d < NCH; ++d) {
                        tail_k[dst + d] = k[src + d];
                        tail_v[dst + d] = v[src + d];
                    }
                }
        }
    }
    return bad ? -1 : 0;
}

int kvref_quantize_blocks_stat(const uint16_t *k, const uint16_t *v, long sb, long st, long sh,
                               int B, const int32_t *seq_lens, const int32_t *block_table,
                               int max_blocks, int hkv, int iters, int stat, uint8_t *pool,
                               long num_pages, uint16_t *tail_k, uint16_t *tail_v, double *u_k,
                               double *u_v)
{
    return kvref_quantize_blocks_fmt(k, v, sb, st, sh, B, seq_lens, block_table, max_blocks,
                                     hkv, iters, stat, 0, pool, num_pages, tail_k, tail_v, u_k,
                                     u_v);
}

int kvref_quantize_blocks(const uint16_t *k, const uint16_t *v, long sb, long st, long sh,
                          int B, const int32_t *seq_lens, const int32_t *block_table,
                          int max_blocks, int hkv, int iters, uint8_t *pool, long num_pages,
                          uint16_t *tail_k, uint16_t *tail_v, double *u_k, double *u_v)
{
    return kvref_quantize_blocks_stat(k, v, sb, st, sh, B, seq_lens, block_table, max_blocks,
                                      hkv, iters, 0, pool, num_pages, tail_k, tail_v, u_k, u_v);
}

/* Decode-time append: token `pos[b]` (the length before the append) goes to
 * tail slot pos mod 128; when that slot is 127 the now-full tail is quantized
 * into page block_table[b][pos / 128].  pos < 0 marks an idle slot. */
int kvref_append_token_fmt(const uint16_t *k_new, const uint16_t *v_new, const int32_t *pos,
                           int B, const int32_t *block_table, int max_blocks, int hkv,
                           int iters, int stat, int fmt, uint8_t *pool, long num_pages,
                           uint16_t *tail_k, uint16_t *tail_v)
{
    int b, bad = 0;
    const long rec_bytes = layout_of(fmt).rec;
    for (b = 0; b < B; ++b) {
        int p = pos[b], h, d, slot;
        if (p < 0) continue;
        slot = p % NTOK;
        for (h = 0; h < hkv; ++h) {
            long dst = (((long)b * hkv + h) * NTOK + slot) * NCH;
            long src = ((long)b * hkv + h) * NCH;
            for (d = 0; d < NCH; ++d) {
                tail_k[dst + d] = k_new[src + d];
                tail_v[dst + d] = v_new[src + d];
            }
        }
        if (slot == NTOK - 1) {
            long page;
            if (p / NTOK >= max_blocks) { bad = 1; continue; }
            page = block_table[(long)b * max_blocks + p / NTOK];
            if (page < 0 || page >= num_pages) { bad = 1; continue; }
            for (h = 0; h < hkv; ++h) {
                uint8_t *rec = pool + (page * hkv + h) * rec_bytes;
                const uint16_t *tk = tail_k + ((long)b * hkv + h) * NTOK * NCH;
                const uint16_t *tv = tail_v + ((long)b * hkv + h) * NTOK * NCH;
                kvref_quantize_tile_fmt(tk, NCH, 0, iters, stat, fmt, rec, NULL, NULL, NULL,
                                        NULL, NULL);
                kvref_quantize_tile_fmt(tv, NCH, 1, iters, stat, fmt, rec, NULL, NULL, NULL,
                                        NULL, NULL);
            }
        }
    }
    return bad ? -1 : 0;
}

int kvref_append_token_stat(const uint16_t *k_new, const uint16_t *v_new, const int32_t *pos,
                            int B, const int32_t *block_table, int max_blocks, int hkv,
                            int iters, int stat, uint8_t *pool, long num_pages,
                            uint16_t *tail_k, uint16_t *tail_v)
{
    return kvref_append_token_fmt(k_new, v_new, pos, B, block_table, max_blocks, hkv, iters,
                                  stat, 0, pool, num_pages, tail_k, tail_v);
}

int kvref_append_token(const uint16_t *k_new, const uint16_t *v_new, const int32_t *pos, int B,
                       const int32_t *block_table, int max_blocks, int hkv, int iters,
                       uint8_t *pool, long num_pages, uint16_t *tail_k, uint16_t *tail_v)
{
    return kvref_append_token_stat(k_new, v_new, pos, B, block_table, max_blocks, hkv, iters, 0,
                                   pool, num_pages, tail_k, tail_v);
}

/* ------------------------------------------------------------------ */
/* Decode attention over quantized pages plus the fp16 tail            */
/* "KV Cache (Anahtar-Deger Onbellegi)", "KV Cache Nasil Calisir?": one new */
/* token attends to every cached K,V; grouped heads per the GQA answer in */
/* "Sik Sorulan Sorular".  Rotation invariance: KVarN page, stage 2.      */
/* ------------------------------------------------------------------ */

/* route 0 (textbook): x_hat = H yhat for every cached token, then
 *   o = softmax(scale * q . x_hat) V_hat with the fp16 tail appended.
 * route 1 (rotated): q_rot = H q, scores from yhat directly, the value sum
 *   accumulated in rotated space and rotated back once: o = H o_rot + o_tail.
 * q: fp16 [B][Hq][128].  out: double [B][Hq][128].  A sequence of length 0
 * yields a zero output.  Returns -1 on a page id outside [0, num_pages). */
int kvref_decode_attention_fmt(const uint16_t *q, const uint8_t *pool, long num_pages,
                               const int32_t *block_table, int max_blocks,
                               const int32_t *seq_lens, int B, int hq, int hkv,
                               const uint16_t *tail_k, const uint16_t *tail_v, double scale,
                               int route, int fmt, double *out)
{
    const long rec_bytes = layout_of(fmt).rec;
    static double H[NCH * NCH];
    static int have_h = 0;
    int bad = 0;
    long item, n_items = (long)B * hq;
    int g = hq / hkv;
#pragma omp critical(kvref_h)
    {
        if (!have_h) {
            kvref_hadamard(NCH, H);
            have_h = 1;
        }
    }
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (item = 0; item < n_items; ++item) {
        int b = (int)(item / hq), h = (int)(item % hq), kvh = h / g;
        int len = seq_lens[b], nfull = len / NTOK, rem = len % NTOK;
        double qv[NCH], qr[NCH], acc[NCH], acc_tail[NCH];
        double *scores = (double *)malloc(sizeof(double) * (len > 0 ? len : 1));
        double *yk = (double *)malloc(sizeof(double) * NTOK * NCH);
        double *yv = (double *)malloc(sizeof(double) * NTOK * NCH);
        double mx = -INFINITY, l = 0.0, xk[NCH];
        int j, t, d, e, pagebad = 0;
        for (d = 0; d < NCH; ++d) qv[d] = kvref_half_to_double(q[item * NCH + d]);
        for (d = 0; d < NCH; ++d) {
            double s = 0.0;
            for (e = 0; e < NCH; ++e) s += H[d * NCH + e] * qv[e];
            qr[d] = s;
        }
        /* pass 1: scores */
        for (j = 0; j < nfull; ++j) {
            long page = block_table[(long)b * max_blocks + j];
            if (page < 0 || page >= num_pages) { pagebad = 1; break; }
            kvref_dequant_part_fmt(pool + (page * hkv + kvh) * rec_bytes, 0, fmt, yk);
            for (t = 0; t < NTOK; ++t) {
                double s = 0.0;
                if (route == 0) {
                    for (d = 0; d < NCH; ++d) {
                        double x = 0.0;
                        for (e = 0; e < NCH; ++e) x += H[d * NCH + e] * yk[t * NCH + e];
                        xk[d] = x;
                    }
                    for (d = 0; d < NCH; ++d) s += qv[d] * xk[d];
                } else {
                    for (d = 0; d < NCH; ++d) s += qr[d] * yk[t * NCH + d];
                }
                scores[j * NTOK + t] = s * scale;
            }
        }
        if (pagebad) {
            bad = 1;
            for (d = 0; d < NCH; ++d) out[item * NCH + d] = NAN;
            free(scores); free(yk); free(yv);
            continue;
        }
        for (t = 0; t < rem; ++t) {
            const uint16_t *kt = tail_k + (((long)b * hkv + kvh) * NTOK + t) * NCH;
            double s = 0.0;
            for (d = 0; d < NCH; ++d) s += qv[d] * kvref_half_to_double(kt[d]);
            scores[nfull * NTOK + t] = s * scale;
        }
        for (t = 0; t < len; ++t) if (scores[t] > mx) mx = scores[t];
        for (t = 0; t < len; ++t) { scores[t] = exp(scores[t] - mx); l += scores[t]; }
        /* pass 2: weighted value sum */
        for (d = 0; d < NCH; ++d) { acc[d] = 0.0; acc_tail[d] = 0.0; }
        for (j = 0; j < nfull; ++j) {
            long page = block_table[(long)b * max_blocks + j];
            kvref_dequant_part_fmt(pool + (page * hkv + kvh) * rec_bytes, 1, fmt, yv);
            for (t = 0; t < NTOK; ++t) {
                double p = scores[j * NTOK + t];
                if (route == 0) {
                    for (d = 0; d < NCH; ++d) {
                        double x = 0.0;
                        for (e = 0; e < NCH; ++e) x += H[d * NCH + e] * yv[t * NCH + e];
                        acc[d] += p * x;
                    }
                } else {
                    for (d = 0; d < NCH; ++d) acc[d] += p * yv[t * NCH + d];
                }
            }
        }
        for (t = 0; t < rem; ++t) {
            const uint16_t *vt = tail_v + (((long)b * hkv + kvh) * NTOK + t) * NCH;
            double p = scores[nfull * NTOK + t];
            for (d = 0; d < NCH; ++d) acc_tail[d] += p * kvref_half_to_double(vt[d]);
        }
        for (d = 0; d < NCH; ++d) {
            double o;
            if (len == 0) { out[item * NCH + d] = 0.0; continue; }
            if (route == 0) {
                o = acc[d] + acc_tail[d];
            } else {
                double x = 0.0;
                for (e = 0; e < NCH; ++e) x += H[d * NCH + e] * acc[e];
                o = x + acc_tail[d];
            }
            out[item * NCH + d] = o / l;
        }
        free(scores); free(yk); free(yv);
    }
    return bad ? -1 : 0;
}

int kvref_decode_attention(const uint16_t *q, const uint8_t *pool, long num_pages,
                           const int32_t *block_table, int max_blocks, const int32_t *seq_lens,
                           int B, int hq, int hkv, const uint16_t *tail_k, const uint16_t *tail_v,
                           double scale, int route, double *out)
{
    return kvref_decode_attention_fmt(q, pool, num_pages, block_table, max_blocks, seq_lens, B,
                                      hq, hkv, tail_k, tail_v, scale, route, 0, out);
}

/* ------------------------------------------------------------------ */
/* The FP8 paged cache: the common halving of the KV cache by 8-bit    */
/* floats ("KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr,   */
/* "Sik Sorulan Sorular": INT8/FP8 KV quantization), the second baseline */
/* the quantized cache is compared with.                                 */
/* Readings: e4m3 ("fn": bias 7, 3 mantissa bits, largest finite 448,    */
/* no infinities), one fp32 scale per token and KV head, s = max|x| / 448 */
/* and codes e4m3(x / s) rounded to nearest even and saturated to +-448;  */
/* both divisions are single-precision, as the codes are a decision taken */
/* in fp32 on both sides.  Page (per page and KV head, 33792 bytes):      */
/*   [0, 16384) K codes [128 tokens][128 channels]                        */
/*   [16384, 32768) V codes, same                                         */
/*   [32768, 33280) K scales fp32 [128 tokens], [33280, 33792) V scales.  */
/* ------------------------------------------------------------------ */

#define FP8_PAGE_BYTES 33792

/* value of an e4m3 code (NaN for the two NaN codes) */
double kvref_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    v = e == 0 ? ldexp((double)m, -9) : ldexp(8.0 + m, e - 10);
    return sign ? -v : v;
}

/* nearest e4m3 code to u, ties to even, magnitudes above 448 saturated */
uint8_t kvref_e4m3_encode(float u)
{
    double a = fabs((double)u), t;
    int sign = u < 0 || (u == 0 && signbit(u)), e, m;
    if (u != u) return 0x7F;
    if (a >= 448.0) return (uint8_t)((sign << 7) | 0x7E);
    if (a < ldexp(1.0, -6)) {                 /* subnormal: multiples of 2^-9 */
        m = (int)nearbyint(ldexp(a, 9));      /* 0..8; 8 is the smallest normal */
        return (uint8_t)((sign << 7) | m);
    }
    e = (int)floor(log2(a));
    if (ldexp(1.0, e) > a) --e;               /* guard log2 rounding */
    if (ldexp(1.0, e + 1) <= a) ++e;
    t = ldexp(a, 3 - e);                      /* 8 (1 + f), in [8, 16) */
    m = (int)nearbyint(t) - 8;
    if (m == 8) { m = 0; ++e; }
    if (e > 8 || (e == 8 && m == 7)) return (uint8_t)((sign << 7) | 0x7E);
    return (uint8_t)((sign << 7) | ((e + 7) << 3) | m);
}

/* one token of one head: scale and codes */
void kvref_fp8_quantize_token(const uint16_t *x, uint8_t *codes, float *scale)
{
    float amax = 0.0f, s;
    int d;
    for (d = 0; d < NCH; ++d) {
        float a = (float)fabs(kvref_half_to_double(x[d]));
        if (a > amax) amax = a;
    }
    s = amax / 448.0f;
    *scale = s;
    for (d = 0; d < NCH; ++d)
        codes[d] = s > 0.0f ? kvref_e4m3_encode((float)kvref_half_to_double(x[d]) / s) : 0;
}

/* tokens [0, seq_lens[b]) of k, v fp16 [B][S][Hkv][128] (element strides
 * sb, st, sh) into the pages block_table[b][t / 128]; returns -1 on a page id
 * outside [0, num_pages) */
int kvref_fp8_write_blocks(const uint16_t *k, const uint16_t *v, long sb, long st, long sh,
                           int B, int hkv, const int32_t *seq_lens, const int32_t *block_table,
                           int max_blocks, uint8_t *pool, long num_pages)
{
    int b, h, t, bad = 0;
    for (b = 0; b < B; ++b)
        for (t = 0; t < seq_lens[b]; ++t) {
            long page = block_table[(long)b * max_blocks + t / NTOK];
            int tt = t % NTOK;
            if (page < 0 || page >= num_pages) { bad = 1; continue; }
            for (h = 0; h < hkv; ++h) {
                uint8_t *pg = pool + (page * hkv + h) * (long)FP8_PAGE_BYTES;
                float s;
                long src = b * sb + (long)t * st + h * sh;
                kvref_fp8_quantize_token(k + src, pg + tt * NCH, &s);
                memcpy(pg + 32768 + 4 * tt, &s, 4);
                kvref_fp8_quantize_token(v + src, pg + 16384 + tt * NCH, &s);
                memcpy(pg + 33280 + 4 * tt, &s, 4);
            }
        }
    return bad ? -1 : 0;
}

/* decode attention over the fp8 pages: out[b][h] = sum_t softmax_t(scale
 * q . k_t) v_t with k_t = s^K_t e4m3(codes), the textbook definition in
 * float64; returns -1 on a page id outside the pool */
int kvref_fp8_decode_attention(const uint16_t *q, const uint8_t *pool, long num_pages,
                               const int32_t *block_table, int max_blocks,
                               const int32_t *seq_lens, int B, int hq, int hkv, double scale,
                               double *out)
{
    int bad = 0;
    long item, n_items = (long)B * hq;
    int g = hq / hkv;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (item = 0; item < n_items; ++item) {
        int b = (int)(item / hq), h = (int)(item % hq), kvh = h / g;
        int len = seq_lens[b], t, d;
        double qv[NCH], acc[NCH], mx = -INFINITY, l = 0.0;
        double *sc = (double *)malloc(sizeof(double) * (len > 0 ? len : 1));
        for (d = 0; d < NCH; ++d) { qv[d] = kvref_half_to_double(q[item * NCH + d]); acc[d] = 0.0; }
        for (t = 0; t < len && !bad; ++t) {
            long page = block_table[(long)b * max_blocks + t / NTOK];
            const uint8_t *pg;
            float s;
            double x = 0.0;
            if (page < 0 || page >= num_pages) { bad = 1; break; }
            pg = pool + (page * hkv + kvh) * (long)FP8_PAGE_BYTES;
            memcpy(&s, pg + 32768 + 4 * (t % NTOK), 4);
            for (d = 0; d < NCH; ++d) x += qv[d] * (double)s * kvref_e4m3_decode(pg[(t % NTOK) * NCH + d]);
            sc[t] = x * scale;
            if (sc[t] > mx) mx = sc[t];
        }
        if (!bad) {
            for (t = 0; t < len; ++t) {
                long page = block_table[(long)b * max_blocks + t / NTOK];
                const uint8_t *pg = pool + (page * hkv + kvh) * (long)FP8_PAGE_BYTES;
                float s;
                double p = exp(sc[t] - mx);
                memcpy(&s, pg + 33280 + 4 * (t % NTOK), 4);
                l += p;
                for (d = 0; d < NCH; ++d)
                    acc[d] += p * (double)s * kvref_e4m3_decode(pg[16384 + (t % NTOK) * NCH + d]);
            }
        }
        for (d = 0; d < NCH; ++d) out[item * NCH + d] = len > 0 && !bad ? acc[d] / l : 0.0;
        free(sc);
    }
    return bad ? -1 : 0;
}
