/*
 * CPU oracle for the CSA2 global-attention decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark may load this library.  It shares no code with the
 * GPU library: it is a plain, slow restatement of what the pages define, in
 * fp64, written so that each step can be checked against the pages by eye.
 *
 * Sources (all "DeepSeek-V4.1-Flash" pages):
 *   [study]  "An infra-oriented diagram of the DeepSeek-V4.1-Flash architecture",
 *            reading notes (k=v 512-wide latent, 64 heads, RoPE on 64 dims
 *            un-rotated on the output; m=2 gated pooling; FP4 E2M1 main cache
 *            with one E4M3 scale per 16 channels; lightning indexer with 32 FP4
 *            heads x 128, ReLU, per-head weights, top-512; Reindex layers score
 *            a 16,384-entry pool chosen by blocks of 8) and section "The KV
 *            cache" (288 B entry, 68 B indexer key with E8M0 per 32, 528 B FP8
 *            SWA entry, 2.5 entries per token, 890 B per token).
 *   [perchy] "perchy.ai/models/deepseek", card "Full. Reindex. Reuse."
 *            (512 selected entries alongside SWA; 16,384 candidate cap).
 *   [helix]  "DeepSeek V4.1 Flash: Why Its Encoder, Engram and KV Cache Matter",
 *            section "CSA2 makes long context cheaper to retain" (128-token SWA,
 *            FP4 with one scale per 16 channels, 0.87 GiB at 1,048,576 tokens).
 *
 * Where the pages leave a step open, the reading taken is stated at the step.
 * Parity status: every function here is pinned by the CPU tests in tests/
 * against closed forms, library format definitions, brute force or textbook
 * special cases; the absolute numerics of DeepSeek's own kernels (score scale,
 * E8M0 rounding rule, SWA byte split, block aggregator, RoPE pairing) cannot be
 * pinned from the pages, so only the readings below are.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DIM 512        /* latent width, k = v                     [study] */
#define ORC_HEADS 64       /* attention query heads                   [study] */
#define ORC_IDIM 128       /* indexer key / query head width          [study] */
#define ORC_IHEADS 32      /* indexer query heads                     [study] */
#define ORC_KV_BYTES 288   /* 512 FP4 + 32 E4M3 scales                [study, "The KV cache"] */
#define ORC_IDX_BYTES 68   /* 128 FP4 + 4 E8M0 scales                 [study, "The KV cache"] */
#define ORC_SWA_BYTES 528  /* 512 E4M3 + 16 E8M0 (reading of "528 FP8 bytes") */

int orc_kv_bytes(void) { return ORC_KV_BYTES; }
int orc_idx_bytes(void) { return ORC_IDX_BYTES; }
int orc_swa_bytes(void) { return ORC_SWA_BYTES; }

/* ------------------------------------------------------------------ formats */
/* FP4 E2M1: sign bit 3, magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} (OCP MX formats). */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(int code) {
    double v = E2M1_MAG[code & 7];
    return (code & 8) ? -v : v;
}

/* FP8 E4M3 ("FN" variant): bias 7, no infinities, 0x7F/0xFF are NaN,
 * subnormals m * 2^-9, max finite 448. */
double orc_e4m3_value(int byte) {
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* E8M0: 2^(b - 127); 0xFF is NaN. */
double orc_e8m0_value(int byte) {
    if ((byte & 255) == 255) return NAN;
    return ldexp(1.0, (byte & 255) - 127);
}

/* Round |a| to the nearest of `n` ascending magnitudes, ties to the even code,
 * saturating at the largest (round-to-nearest-even with satfinite). */
static int rne_pick(double a, const double *mag, int n) {
    if (a >= mag[n - 1]) return n - 1;
    int best = 0;
    double bd = fabs(a - mag[0]);
    for (int c = 1; c < n; c++) {
        double d = fabs(a - mag[c]);
        if (d < bd || (d == bd && (c & 1) == 0)) { best = c; bd = d; }
    }
    return best;
}

static double E4M3_MAG[127];
static int e4m3_ready = 0;
static void e4m3_init(void) {
    if (e4m3_ready) return;
    for (int c = 0; c < 127; c++) E4M3_MAG[c] = orc_e4m3_value(c);
    e4m3_ready = 1;
}

/* Encoders keep the sign of x (IEEE style: a negative value that rounds to a
 * zero magnitude gives the negative-zero code). */
int orc_e2m1_encode(double x) {
    int c = rne_pick(fabs(x), E2M1_MAG, 8);
    return signbit(x) ? (c | 8) : c;
}

int orc_e4m3_encode(double x) {
    e4m3_init();
    int c = rne_pick(fabs(x), E4M3_MAG, 127);
    return signbit(x) ? (c | 0x80) : c;
}

/* bf16 <-> double */
double orc_bf16_value(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Round a double to bfloat16, nearest-even (one rounding, straight from fp64). */
uint16_t orc_bf16_from_double(double v) {
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    int ex;
    frexp(a, &ex);                 /* a = f * 2^ex, f in [0.5, 1) */
    int q = ex - 8;                /* 8 significant bits -> ulp 2^(ex-8) */
    if (q < -133) q = -133;        /* bf16 subnormal spacing */
    double r = nearbyint(ldexp(a, -q));   /* default rounding mode: ties to even */
    float f = (float)ldexp(r, q);  /* exact: r*2^q has <= 9 bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t b = (uint16_t)(u >> 16);
    return signbit(v) ? (uint16_t)(b | 0x8000) : b;
}

/* Smallest e with lim * 2^e >= amax, clamped to the E8M0 range [-127, 127]:
 * the power-of-two scale is the smallest one that needs no saturation. */
static int pow2_scale_exp(double amax, double lim) {
    int e = (int)ceil(log2(amax / lim));
    while (ldexp(lim, e) < amax) e++;
    while (ldexp(lim, e - 1) >= amax) e--;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

/* ------------------------------------------------------------ cache packing */
/* S1: main KV entry.  Per 16 channels: scale = E4M3_RNE(amax / 6); each
 * element = E2M1_RNE(x / scale).  Bytes 0..255 hold the 512 nibbles (low
 * nibble = even channel), bytes 256..287 the 32 scales.  A group whose scale
 * rounds to zero (amax = 0, or underflow) stores all-zero codes.  [study] */
void orc_pack_kv_row(const uint16_t *x, uint8_t *out) {
    memset(out, 0, ORC_KV_BYTES);
    for (int g = 0; g < 32; g++) {
        double amax = 0.0;
        for (int i = 0; i < 16; i++) {
            double a = fabs(orc_bf16_value(x[16 * g + i]));
            if (a > amax) amax = a;
        }
        int sc = orc_e4m3_encode(amax / 6.0);
        double s = orc_e4m3_value(sc);
        out[256 + g] = (uint8_t)sc;
        for (int i = 0; i < 16; i++) {
            int c = 16 * g + i;
            int code = (s == 0.0) ? 0 : orc_e2m1_encode(orc_bf16_value(x[c]) / s);
            out[c >> 1] |= (uint8_t)(code << (4 * (c & 1)));
        }
    }
}

/* S2 (indexer key) and S4 (indexer query head): 128 FP4 + 4 E8M0 scales, one
 * per 32 channels (reading: the smallest power of two >= amax / 6).  Logical
 * 68-byte record: 64 nibble bytes then 4 scale bytes.  [study] */
void orc_pack_idx_row(const uint16_t *x, uint8_t *out) {
    memset(out, 0, ORC_IDX_BYTES);
    for (int g = 0; g < 4; g++) {
        double amax = 0.0;
        for (int i = 0; i < 32; i++) {
            double a = fabs(orc_bf16_value(x[32 * g + i]));
            if (a > amax) amax = a;
        }
        if (amax == 0.0) { out[64 + g] = 0; continue; }
        int e = pow2_scale_exp(amax, 6.0);
        out[64 + g] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; i++) {
            int c = 32 * g + i;
            int code = orc_e2m1_encode(ldexp(orc_bf16_value(x[c]), -e));
            out[c >> 1] |= (uint8_t)(code << (4 * (c & 1)));
        }
    }
}

/* S3: SWA entry, 528 FP8 bytes read as 512 E4M3 values + 16 E8M0 scales (one
 * per 32 channels, smallest power of two >= amax / 448).  [study] */
void orc_pack_swa_row(const uint16_t *x, uint8_t *out) {
    memset(out, 0, ORC_SWA_BYTES);
    for (int g = 0; g < 16; g++) {
        double amax = 0.0;
        for (int i = 0; i < 32; i++) {
            double a = fabs(orc_bf16_value(x[32 * g + i]));
            if (a > amax) amax = a;
        }
        if (amax == 0.0) { out[512 + g] = 0; continue; }
        int e = pow2_scale_exp(amax, 448.0);
        out[512 + g] = (uint8_t)(e + 127);
        for (int i = 0; i < 32; i++) {
            int c = 32 * g + i;
            out[c] = (uint8_t)orc_e4m3_encode(ldexp(orc_bf16_value(x[c]), -e));
        }
    }
}

/* m=2 gated pooling: two consecutive tokens become one entry; per channel
 * e = sum_t softmax_t(z_t) x_t over the pair, computed in fp64 and rounded to
 * bf16 before packing.  [study, Full-layer global KV note] */
void orc_pool_m2_row(const uint16_t *x0, const uint16_t *x1, const float *z0, const float *z1,
                     uint16_t *out) {
    for (int c = 0; c < ORC_DIM; c++) {
        double a = (double)z0[c], b = (double)z1[c];
        double m = a > b ? a : b;
        double ea = exp(a - m), eb = exp(b - m);
        double v = (ea * orc_bf16_value(x0[c]) + eb * orc_bf16_value(x1[c])) / (ea + eb);
        out[c] = orc_bf16_from_double(v);
    }
}

void orc_pack_kv(const uint16_t *x, int64_t rows, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) orc_pack_kv_row(x + r * ORC_DIM, out + r * ORC_KV_BYTES);
}

void orc_pack_idx(const uint16_t *x, int64_t rows, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) orc_pack_idx_row(x + r * ORC_IDIM, out + r * ORC_IDX_BYTES);
}

void orc_pack_swa(const uint16_t *x, int64_t rows, uint8_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) orc_pack_swa_row(x + r * ORC_DIM, out + r * ORC_SWA_BYTES);
}

/* rows_out entries from 2*rows_out tokens (x, z are [2*rows_out][512]). */
void orc_pool_m2(const uint16_t *x, const float *z, int64_t rows_out, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows_out; r++)
        orc_pool_m2_row(x + (2 * r) * ORC_DIM, x + (2 * r + 1) * ORC_DIM, z + (2 * r) * ORC_DIM,
                        z + (2 * r + 1) * ORC_DIM, out + r * ORC_DIM);
}

/* Indexer-key projection: the indexer's 128-wide key is a 512 -> 128
 * projection of the same latent the main cache stores [study, reading notes on
 * the Full layer's global KV].  The weights are not on the pages (synthetic
 * here).  Reading: out[r][n] = sum_c x[r][c] * w[n][c] over the bf16 latent
 * (the m=2 pooled one for encoder entries) and bf16 weights, exact in fp64 and
 * rounded once to bf16, the input of the key's FP4 packing.
 * x: [rows][512], w: [128][512], out: [rows][128], all bf16 bits. */
void orc_project_keys(const uint16_t *x, int64_t rows, const uint16_t *w, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int n = 0; n < ORC_IDIM; n++) {
            double acc = 0.0;
            for (int c = 0; c < ORC_DIM; c++)
                acc += orc_bf16_value(x[r * ORC_DIM + c]) * orc_bf16_value(w[(int64_t)n * ORC_DIM + c]);
            out[r * ORC_IDIM + n] = orc_bf16_from_double(acc);
        }
    }
}

/* ---------------------------------------------------------------- dequant */
void orc_dequant_kv(const uint8_t *rec, double *out) {
    for (int c = 0; c < ORC_DIM; c++) {
        int code = (rec[c >> 1] >> (4 * (c & 1))) & 15;
        out[c] = orc_e2m1_value(code) * orc_e4m3_value(rec[256 + c / 16]);
    }
}

void orc_dequant_idx(const uint8_t *rec, double *out) {
    for (int c = 0; c < ORC_IDIM; c++) {
        int code = (rec[c >> 1] >> (4 * (c & 1))) & 15;
        out[c] = orc_e2m1_value(code) * orc_e8m0_value(rec[64 + c / 32]);
    }
}

void orc_dequant_swa(const uint8_t *rec, double *out) {
    for (int c = 0; c < ORC_DIM; c++)
        out[c] = orc_e4m3_value(rec[c]) * orc_e8m0_value(rec[512 + c / 32]);
}

/* ----------------------------------------------------------- indexer score */
/* Lightning indexer [study]: s_j = sum_h w_h * ReLU(qhat_h . khat_j), with
 * 32 FP4 query heads of 128 dims and one shared key per entry.  No extra
 * global scale (reading: a positive factor does not change the order).
 * keys: [n][68] logical records; qidx: [32][68]; w: [32]. */
void orc_index_score(const uint8_t *keys, int64_t n, const uint8_t *qidx, const float *w,
                     double *out) {
    double q[ORC_IHEADS][ORC_IDIM];
    for (int h = 0; h < ORC_IHEADS; h++) orc_dequant_idx(qidx + h * ORC_IDX_BYTES, q[h]);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; j++) {
        double k[ORC_IDIM];
        orc_dequant_idx(keys + j * ORC_IDX_BYTES, k);
        double s = 0.0;
        for (int h = 0; h < ORC_IHEADS; h++) {
            double d = 0.0;
            for (int c = 0; c < ORC_IDIM; c++) d += q[h][c] * k[c];
            s += (double)w[h] * (d > 0.0 ? d : 0.0);
        }
        out[j] = s;
    }
}

/* ---------------------------------------------------------------- top-k */
/* Top-k by (score descending, index ascending): lower index wins ties.  The
 * selected indices are returned in ascending order and padded with -1.
 * [perchy: the main selection keeps 512 entries; study, lightning indexer] */
static const double *g_sort_keys;
static int cmp_desc_then_idx(const void *a, const void *b) {
    int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
    double si = g_sort_keys[i], sj = g_sort_keys[j];
    if (si > sj) return -1;
    if (si < sj) return 1;
    return (i < j) ? -1 : (i > j);
}
static int cmp_i64(const void *a, const void *b) {
    int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
    return (i < j) ? -1 : (i > j);
}

/* returns the number selected, min(k, n) */
int orc_topk(const double *s, int64_t n, int k, int32_t *out) {
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (n > 0 ? n : 1));
    for (int64_t i = 0; i < n; i++) idx[i] = i;
    g_sort_keys = s;
    qsort(idx, (size_t)n, sizeof(int64_t), cmp_desc_then_idx);
    int m = (int)(n < k ? n : k);
    qsort(idx, (size_t)m, sizeof(int64_t), cmp_i64);
    for (int i = 0; i < k; i++) out[i] = i < m ? (int32_t)idx[i] : -1;
    free(idx);
    return m;
}

/* Candidate pool [study, lightning-indexer note: 16,384 positions chosen as
 * 2,048 blocks of 8 by an earlier layer]: block score = max of the Full-layer scores of the block's
 * entries j < n (reading: max), top `nb` blocks by (block score desc, block id
 * asc), returned ascending and padded with -1.  Returns the number selected. */
int orc_pool_blocks(const double *s, int64_t n, int block, int nb, int32_t *out) {
    int64_t nblk = (n + block - 1) / block;
    double *bs = (double *)malloc(sizeof(double) * (nblk > 0 ? nblk : 1));
    for (int64_t b = 0; b < nblk; b++) {
        double m = -INFINITY;
        for (int64_t j = b * block; j < (b + 1) * block && j < n; j++)
            if (s[j] > m) m = s[j];
        bs[b] = m;
    }
    int r = orc_topk(bs, nblk, nb, out);
    free(bs);
    return r;
}

/* ------------------------------------------------------- sparse attention */
/* One query, all 64 heads [study: k = v, one 512-wide latent shared by all
 * heads; attention covers the SWA window and the 512 selected entries; RoPE
 * on 64 of 512 dims, un-rotated on the output]:
 *   l_i  = sm_scale * q_h . k_i        over the n entries given (the selected
 *                                      entries and the SWA window; no dedup,
 *                                      no sink)
 *   p    = softmax(l)                  (fp64)
 *   o_h  = sum_i p_i k_i               (values are the keys)
 *   then dims (rope_off + 2i, rope_off + 2i + 1), i < rope_dim/2, are rotated
 *   by -pos with theta_i = pos * rope_base^(-2i / rope_dim).
 * q: [64][512], k: [n][512], both already in fp64 (dequantised).  out:
 * [64][512]; lse (optional): [64], log sum_i exp(l_i), -inf when n == 0. */
void orc_attn_f64(const double *q, const double *k, int n, int64_t pos, double sm_scale, double rope_base,
                  int rope_off, int rope_dim, double *out, double *lse) {
#pragma omp parallel for schedule(static)
    for (int h = 0; h < ORC_HEADS; h++) {
        double *o = out + (size_t)h * ORC_DIM;
        const double *qh = q + (size_t)h * ORC_DIM;
        for (int c = 0; c < ORC_DIM; c++) o[c] = 0.0;
        if (lse) lse[h] = -INFINITY;
        if (n == 0) continue;
        double *l = (double *)malloc(sizeof(double) * (size_t)n);
        double mx = -INFINITY;
        for (int i = 0; i < n; i++) {
            double d = 0.0;
            for (int c = 0; c < ORC_DIM; c++) d += qh[c] * k[(size_t)i * ORC_DIM + c];
            l[i] = sm_scale * d;
            if (l[i] > mx) mx = l[i];
        }
        double den = 0.0;
        for (int i = 0; i < n; i++) { l[i] = exp(l[i] - mx); den += l[i]; }
        if (lse) lse[h] = mx + log(den);   /* log sum_i exp(l_i) */
        for (int i = 0; i < n; i++) {
            double p = l[i] / den;
            for (int c = 0; c < ORC_DIM; c++) o[c] += p * k[(size_t)i * ORC_DIM + c];
        }
        free(l);
        for (int i = 0; i < rope_dim / 2; i++) {
            double th = (double)pos * pow(rope_base, -2.0 * i / (double)rope_dim);
            double cs = cos(th), sn = sin(th);
            double a = o[rope_off + 2 * i], b = o[rope_off + 2 * i + 1];
            o[rope_off + 2 * i] = a * cs + b * sn;
            o[rope_off + 2 * i + 1] = -a * sn + b * cs;
        }
    }
}

/* The cache-record form: q [64][512] bf16, kv_rows [n_sel][288] records of the
 * selected entries, swa_rows [n_swa][528]; dequantised (exactly, in fp64) and
 * passed to orc_attn_f64 in that order. */
static void orc_sparse_attn_impl(const uint16_t *q, const uint8_t *kv_rows, int n_sel, const uint8_t *swa_rows,
                                 int n_swa, int64_t pos, double sm_scale, double rope_base, int rope_off,
                                 int rope_dim, double *out, double *lse) {
    int n = n_sel + n_swa;
    double *k = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORC_DIM);
    double *qd = (double *)malloc(sizeof(double) * ORC_HEADS * ORC_DIM);
    for (int i = 0; i < n_sel; i++) orc_dequant_kv(kv_rows + (size_t)i * ORC_KV_BYTES, k + (size_t)i * ORC_DIM);
    for (int i = 0; i < n_swa; i++)
        orc_dequant_swa(swa_rows + (size_t)i * ORC_SWA_BYTES, k + (size_t)(n_sel + i) * ORC_DIM);
    for (int i = 0; i < ORC_HEADS * ORC_DIM; i++) qd[i] = orc_bf16_value(q[i]);
    orc_attn_f64(qd, k, n, pos, sm_scale, rope_base, rope_off, rope_dim, out, lse);
    free(qd);
    free(k);
}

void orc_sparse_attn(const uint16_t *q, const uint8_t *kv_rows, int n_sel, const uint8_t *swa_rows,
                     int n_swa, int64_t pos, double sm_scale, double rope_base, int rope_off,
                     int rope_dim, double *out) {
    orc_sparse_attn_impl(q, kv_rows, n_sel, swa_rows, n_swa, pos, sm_scale, rope_base, rope_off, rope_dim, out,
                         NULL);
}

/* The same, also writing lse[h] = log sum_i exp(l_i) over the entries given
 * (-inf when there are none): the weight with which this output enters a
 * softmax over a larger set of entries (log-sum-exp merge of partial sets). */
void orc_sparse_attn_lse(const uint16_t *q, const uint8_t *kv_rows, int n_sel, const uint8_t *swa_rows,
                         int n_swa, int64_t pos, double sm_scale, double rope_base, int rope_off,
                         int rope_dim, double *out, double *lse) {
    orc_sparse_attn_impl(q, kv_rows, n_sel, swa_rows, n_swa, pos, sm_scale, rope_base, rope_off, rope_dim, out,
                         lse);
}
