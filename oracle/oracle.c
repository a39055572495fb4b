/*
 * oracle.c -- plain float64 CPU reference of the paged q_len=1 decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this file.  It shares no code,
 * header, table or helper with the CUDA library and includes none of it.
 *
 * What it computes (each function below cites the passage it follows):
 *   oracle_rope_kv_append  -- optional per-head RMSNorm, then RoPE on the new
 *                             q and k of every active row at
 *                             position seq_len-1, then the append of the
 *                             rotated k (rounded to the element type, bf16
 *                             or fp16) and of v into the row's current page;
 *   oracle_decode_attn     -- single-token GQA attention over the page table,
 *                             written as the plain softmax definition;
 *   oracle_decode_attn_split + oracle_lse_combine
 *                          -- the same attention computed as per-segment
 *                             partial softmax results merged by their
 *                             log-sum-exp (the long-sequence path), used only
 *                             to check the combine algebra.
 *
 * Numbers: bf16 / fp16 inputs are read as exact doubles; all arithmetic is
 * float64; the only rounding to a narrow type is the round-to-nearest-even of
 * the rotated key to the element type before it is stored in the cache.
 *
 * Readings of the pages that this file encodes (where they are silent):
 *   - RoPE pairs element i with element i + D/2 ("rotate half"), or 2i with
 *     2i + 1 when asked ("interleaved"), and uses angle pos * theta^(-2i/D),
 *     i = 0 .. D/2-1;
 *   - the cached keys are stored already rotated; only the new key is rotated;
 *   - seq_len counts the new token, which lands in logical slot seq_len-1;
 *   - the softmax scale is 1/sqrt(D) unless the caller passes another;
 *   - q head g reads kv head g / (Hq/Hkv);
 *   - rows with active == 0 produce an all-zero output and write nothing.
 *
 * bf16 / fp16 arrays are passed as uint16_t bit patterns.  Strides are in elements.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> double ------------------------------------------------- */

static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), in one rounding step.
 * bf16 keeps 8 significant bits and the float32 exponent range, so the
 * quantum of a normal value in [2^(e-1), 2^e) is 2^(e-8), and the quantum of
 * a subnormal value is 2^-133. */
uint16_t oracle_bf16_from_double(double x) {
    if (isnan(x)) return 0x7FC0;
    if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    int e;
    frexp(x, &e);
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    double r = nearbyint(ldexp(x, -qexp)); /* default rounding: nearest, ties to even */
    double y = ldexp(r, qexp);
    const double max_bf16 = 3.3895313892515355e38; /* (2 - 2^-7) * 2^127 */
    if (y > max_bf16) return 0x7F80;
    if (y < -max_bf16) return 0xFF80;
    float f = (float)y; /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }

/* ---- fp16 (IEEE binary16) <-> double ---------------------------------- */

static double f16_to_double(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0x1F) v = m ? NAN : INFINITY;
    else if (e == 0) v = ldexp((double)m, -24);            /* subnormal: m * 2^-24 */
    else v = ldexp((double)(m | 0x400), e - 25);            /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

/* Nearest binary16 to a double (ties to even), one rounding step: 11
 * significant bits, exponent range [-14, 15], subnormal quantum 2^-24. */
uint16_t oracle_f16_from_double(double x) {
    if (isnan(x)) return 0x7E00;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                     /* a in [2^(e-1), 2^e) */
    int qexp = e - 11;
    if (qexp < -24) qexp = -24;
    double r = nearbyint(ldexp(a, -qexp));
    double y = ldexp(r, qexp);
    if (y >= 65520.0) return sign | 0x7C00;  /* beyond max (65504) + half ulp: inf */
    /* encode y exactly */
    if (y < ldexp(1.0, -14)) return sign | (uint16_t)nearbyint(ldexp(y, 24));
    int ey;
    double fy = frexp(y, &ey);        /* y = fy * 2^ey, fy in [0.5, 1) */
    int E = ey - 1 + 15;
    int M = (int)nearbyint(ldexp(fy, 11)) - 1024;
    return sign | (uint16_t)(E << 10) | (uint16_t)M;
}

double oracle_f16_to_double(uint16_t h) { return f16_to_double(h); }

/* element type of q / k / v / cache / out: 0 = bf16, 1 = fp16 */
static double elem_to_double(uint16_t h, int dtype) { return dtype ? f16_to_double(h) : bf16_to_double(h); }
static uint16_t elem_from_double(double x, int dtype) { return dtype ? oracle_f16_from_double(x) : oracle_bf16_from_double(x); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- RMSNorm ----------------------------------------------------------- */

/* Per-head RMSNorm with float64 variance (the pages keep "RMSNorm variance" in
 * fp32 or better for alignment, "Engineering TTS inference in vLLM-Omni",
 * Qwen3-TTS section 4):  x_d <- w_d * x_d / sqrt(mean_e(x_e^2) + eps).
 * w == NULL: no normalisation. */
static void rms_norm(double* x, int D, const double* w, double eps) {
    if (!w) return;
    double ss = 0.0;
    for (int d = 0; d < D; ++d) ss += x[d] * x[d];
    double r = 1.0 / sqrt(ss / (double)D + eps);
    for (int d = 0; d < D; ++d) x[d] = w[d] * (x[d] * r);
}

/* ---- RoPE + append ---------------------------------------------------- */

/* Rotate one head vector x[0..D) in place by position pos.  Pair i of
 * frequency a_i = pos * theta^(-2i/D) is (i, i + D/2) ("rotate half") or, with
 * interleaved, (2i, 2i + 1):
 *   x'_first  = x_first cos a_i - x_second sin a_i
 *   x'_second = x_second cos a_i + x_first sin a_i
 * The pages ask for RoPE cos/sin in fp32 or better for alignment with the
 * reference model ("Engineering TTS inference in vLLM-Omni", Qwen3-TTS,
 * section 4 "numerical precision: fp32 alignment"); here they are float64. */
static void rope_rotate(double* x, int D, double pos, double theta, int interleaved) {
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double a = pos * pow(theta, -2.0 * (double)i / (double)D);
        double c = cos(a), s = sin(a);
        int i0 = interleaved ? 2 * i : i, i1 = interleaved ? 2 * i + 1 : i + half;
        double lo = x[i0], hi = x[i1];
        x[i0] = lo * c - hi * s;
        x[i1] = hi * c + lo * s;
    }
}

/* RoPE on the new q/k of every active row, then append of k (rotated, bf16)
 * and v into slot seq_len-1 of the row's logical sequence, reached through
 * the page table: page = page_table[b][slot / P], offset = slot % P.
 * The step follows the append-then-attend interface of the vox-serve
 * "Adding a Model" page (section "1. The model code": keys and values are
 * written into the paged cache, then attention runs over it), and its rule
 * that padding entries write nothing (section "How a program runs").
 *
 * q, k_new, v_new: [B][Hq][D], [B][Hkv][D], [B][Hkv][D] of the element type
 *   dtype (0 = bf16, 1 = fp16; the Fish kernel takes fp16 or bf16); the
 *   rotated key is rounded to that type.  interleaved selects the RoPE pairing.
 * positions: NULL means seq_len - 1.
 * q_norm_w, k_norm_w: per-dim RMSNorm weights [D] applied to every q / new-k
 *   head before RoPE, or NULL for none; norm_eps is the epsilon.
 * q_rot: float64 [B][Hq][D] out; rows with active == 0 are left untouched.
 * k_rot: float64 [B][Hkv][D] out or NULL: the rotated key before its
 *        rounding (rows that are skipped are left untouched).
 * k_pre: float64 [B][Hkv][D] out or NULL: the key fed to RoPE (after the
 *        RMSNorm when there is one).
 * Returns the number of active rows whose slot could not be placed
 * (seq_len outside [1, MPS*P] or a page id outside [0, num_pages)); those
 * rows write nothing.
 */
int oracle_rope_kv_append(const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                          const int32_t* positions,
                          const double* q_norm_w, const double* k_norm_w, double norm_eps,
                          uint16_t* k_cache, uint16_t* v_cache,
                          int64_t page_stride, int64_t token_stride,
                          const int32_t* page_table, int max_pages_per_seq, int num_pages,
                          const int32_t* seq_lens, const int32_t* active,
                          double* q_rot, double* k_rot, double* k_pre,
                          int B, int Hq, int Hkv, int D, int P, double theta, int dtype, int interleaved) {
    int bad = 0;
    double* tmp = (double*)malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b) {
        if (!active[b]) continue;
        int L = seq_lens[b];
        if (L < 1 || (int64_t)L > (int64_t)max_pages_per_seq * P) { ++bad; continue; }
        double pos = positions ? (double)positions[b] : (double)(L - 1);
        for (int g = 0; g < Hq; ++g) {
            const uint16_t* src = q + ((size_t)b * Hq + g) * D;
            for (int d = 0; d < D; ++d) tmp[d] = elem_to_double(src[d], dtype);
            rms_norm(tmp, D, q_norm_w, norm_eps);
            rope_rotate(tmp, D, pos, theta, interleaved);
            memcpy(q_rot + ((size_t)b * Hq + g) * D, tmp, sizeof(double) * (size_t)D);
        }
        int slot = L - 1;
        int page = page_table[(size_t)b * max_pages_per_seq + slot / P];
        if (page < 0 || (num_pages > 0 && page >= num_pages)) { ++bad; continue; }
        int off = slot % P;
        for (int h = 0; h < Hkv; ++h) {
            const uint16_t* ks = k_new + ((size_t)b * Hkv + h) * D;
            const uint16_t* vs = v_new + ((size_t)b * Hkv + h) * D;
            for (int d = 0; d < D; ++d) tmp[d] = elem_to_double(ks[d], dtype);
            rms_norm(tmp, D, k_norm_w, norm_eps);
            if (k_pre) memcpy(k_pre + ((size_t)b * Hkv + h) * D, tmp, sizeof(double) * (size_t)D);
            rope_rotate(tmp, D, pos, theta, interleaved);
            if (k_rot) memcpy(k_rot + ((size_t)b * Hkv + h) * D, tmp, sizeof(double) * (size_t)D);
            uint16_t* kd = k_cache + (int64_t)page * page_stride + (int64_t)off * token_stride + (int64_t)h * D;
            uint16_t* vd = v_cache + (int64_t)page * page_stride + (int64_t)off * token_stride + (int64_t)h * D;
            for (int d = 0; d < D; ++d) {
                kd[d] = elem_from_double(tmp[d], dtype);
                vd[d] = vs[d];
            }
        }
    }
    free(tmp);
    return bad;
}

/* ---- attention -------------------------------------------------------- */

static const uint16_t* key_row(const uint16_t* cache, int64_t page_stride, int64_t token_stride,
                               const int32_t* pt_row, int P, int j, int h, int D) {
    int page = pt_row[j / P];
    return cache + (int64_t)page * page_stride + (int64_t)(j % P) * token_stride + (int64_t)h * D;
}

/* Softmax attention of one q head over keys [j0, j1) of row b.  Writes the
 * normalised output o[0..D) and returns lse = m + ln(sum exp(s - m)) (natural
 * log).  Plain definition: s_j = sm_scale * <q, K_j>, p = exp(s - max s),
 * o = sum p_j V_j / sum p_j. */
static double attend_range(const double* qv, const uint16_t* k_cache, const uint16_t* v_cache,
                           int64_t page_stride, int64_t token_stride, const int32_t* pt_row,
                           int P, int h, int D, int j0, int j1, double sm_scale,
                           double* s, double* o, int dtype) {
    double m = -INFINITY;
    for (int j = j0; j < j1; ++j) {
        const uint16_t* kr = key_row(k_cache, page_stride, token_stride, pt_row, P, j, h, D);
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qv[d] * elem_to_double(kr[d], dtype);
        s[j - j0] = acc * sm_scale;
        if (s[j - j0] > m) m = s[j - j0];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = j0; j < j1; ++j) {
        double p = exp(s[j - j0] - m);
        l += p;
        const uint16_t* vr = key_row(v_cache, page_stride, token_stride, pt_row, P, j, h, D);
        for (int d = 0; d < D; ++d) o[d] += p * elem_to_double(vr[d], dtype);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    return m + log(l);
}

/* Single-token GQA decode attention over the paged cache ("Engineering TTS
 * inference in vLLM-Omni", Fish Speech S2 Pro, "model-specific attention
 * kernel": q_len = 1, one kv head serves its group of q heads, keys reached
 * through the block table).
 *
 * q_rot: float64 [B][Hq][D]; out: float64 [B][Hq][D].
 * rows / n_rows: the rows to compute (NULL: all B rows).  Rows not listed are
 * left untouched.  Inactive rows get zeros (padding entries "compute garbage
 * that is ignored", vox-serve "Adding a Model", "How a program runs"; zero is
 * the defined value here).
 * sm_scale <= 0 means 1/sqrt(D).
 * lse_out (may be NULL): float64 [B][Hq], natural-log log-sum-exp per head.
 */
void oracle_decode_attn(const double* q_rot, const uint16_t* k_cache, const uint16_t* v_cache,
                        int64_t page_stride, int64_t token_stride,
                        const int32_t* page_table, int max_pages_per_seq,
                        const int32_t* seq_lens, const int32_t* active,
                        double* out, double* lse_out, double sm_scale,
                        const int32_t* rows, int n_rows,
                        int B, int Hq, int Hkv, int D, int P, int dtype) {
    if (sm_scale <= 0.0) sm_scale = 1.0 / sqrt((double)D);
    int G = Hq / Hkv;
    int nr = rows ? n_rows : B;
    int64_t total = (int64_t)nr * Hq;
#pragma omp parallel
    {
        double* s = NULL;
        int cap = 0;
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < total; ++t) {
            int r = (int)(t / Hq), g = (int)(t % Hq);
            int b = rows ? rows[r] : r;
            double* o = out + ((size_t)b * Hq + g) * D;
            if (!active[b]) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (lse_out) lse_out[(size_t)b * Hq + g] = -INFINITY;
                continue;
            }
            int L = seq_lens[b];
            if (L > cap) { free(s); cap = L; s = (double*)malloc(sizeof(double) * (size_t)cap); }
            const int32_t* pt_row = page_table + (size_t)b * max_pages_per_seq;
            double lse = attend_range(q_rot + ((size_t)b * Hq + g) * D, k_cache, v_cache,
                                      page_stride, token_stride, pt_row, P, g / G, D, 0, L,
                                      sm_scale, s, o, dtype);
            if (lse_out) lse_out[(size_t)b * Hq + g] = lse;
        }
        free(s);
    }
}

/* Merge S partial results of one head: o_s (normalised) and lse_s.  Splits
 * with lse = -inf (no keys) get weight 0.  M = max lse_s over non-empty
 * splits; w_s = exp(lse_s - M); o = sum w_s o_s / sum w_s.  This is the
 * online-softmax recurrence applied to whole segments ("Engineering TTS
 * inference in vLLM-Omni", Fish Speech S2 Pro: the long path splits the
 * sequence, computes partial m/l/acc per segment and merges them).
 * Returns the merged lse, or -inf if every split is empty (o is then zero). */
double oracle_lse_combine(const double* o_parts, const double* lse_parts, int S, int D, double* o) {
    double M = -INFINITY;
    for (int k = 0; k < S; ++k)
        if (lse_parts[k] > M) M = lse_parts[k];
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) return -INFINITY;
    double wsum = 0.0;
    for (int k = 0; k < S; ++k) {
        if (lse_parts[k] == -INFINITY) continue;
        double w = exp(lse_parts[k] - M);
        wsum += w;
        for (int d = 0; d < D; ++d) o[d] += w * o_parts[(size_t)k * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= wsum;
    return M + log(wsum);
}

/* The attention of oracle_decode_attn, computed as n_splits contiguous
 * segments of every row's keys, segment k = [floor(k L / S), floor((k+1) L / S)),
 * each reduced to (o_k, lse_k) and then merged by oracle_lse_combine.  Exists
 * only to pin the combine algebra against the unsplit definition. */
void oracle_decode_attn_split(const double* q_rot, const uint16_t* k_cache, const uint16_t* v_cache,
                              int64_t page_stride, int64_t token_stride,
                              const int32_t* page_table, int max_pages_per_seq,
                              const int32_t* seq_lens, const int32_t* active,
                              double* out, double sm_scale, int n_splits,
                              int B, int Hq, int Hkv, int D, int P, int dtype) {
    if (sm_scale <= 0.0) sm_scale = 1.0 / sqrt((double)D);
    int G = Hq / Hkv;
    for (int b = 0; b < B; ++b) {
        for (int g = 0; g < Hq; ++g) {
            double* o = out + ((size_t)b * Hq + g) * D;
            if (!active[b]) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                continue;
            }
            int L = seq_lens[b];
            int S = n_splits;
            double* op = (double*)malloc(sizeof(double) * (size_t)S * D);
            double* lp = (double*)malloc(sizeof(double) * (size_t)S);
            double* s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            const int32_t* pt_row = page_table + (size_t)b * max_pages_per_seq;
            for (int k = 0; k < S; ++k) {
                int j0 = (int)(((int64_t)k * L) / S), j1 = (int)(((int64_t)(k + 1) * L) / S);
                if (j1 <= j0) {
                    lp[k] = -INFINITY;
                    for (int d = 0; d < D; ++d) op[(size_t)k * D + d] = 0.0;
                    continue;
                }
                lp[k] = attend_range(q_rot + ((size_t)b * Hq + g) * D, k_cache, v_cache, page_stride,
                                     token_stride, pt_row, P, g / G, D, j0, j1, sm_scale, s,
                                     op + (size_t)k * D, dtype);
            }
            oracle_lse_combine(op, lp, S, D, o);
            free(op);
            free(lp);
            free(s);
        }
    }
}
