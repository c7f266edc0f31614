/*
 * qsa_oracle.c -- plain, slow CPU oracle for QSA block-sparse GQA decode and
 * speculative verify over an NVFP4 paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file.  It shares no code, header,
 * table or constant with the CUDA library, and the library never calls it.
 *
 * Arithmetic: fp64 for floating point, int64 for the index dot products.  No
 * blocking, no online softmax, no splits: each function is the definition
 * written out, with explicit sorts where the definition ranks.  OpenMP only
 * distributes independent query rows over cores.
 *
 * Sources (TensorRT-LLM pull-request pages):
 *   - PR #20276 "Qwen3.8-Flash-Next NVFP4 target", Features table: NVFP4 KV
 *     cache = uint8 e2m1 pages + e4m3 block scales; canonical QSA selection =
 *     a pure function of the scores, the window and k: every block strictly
 *     above the k-th score, ties to the highest index.
 *   - PR #20276, Decisions: canonical rows are identical launch to launch.
 *   - PR #20937 "GB300 perf work on qwen3_8_flash_next_nvfp4__sm_103__tp1",
 *     What changes / Verify: request-tiled index scores; split-K sparse GQA
 *     with a per-row merge.
 *   - e2m1 / e4m3 bit fields: OCP Microscaling Formats v1.0 (element formats).
 *
 * Readings where the pages are silent:
 *   R1 block score = max over the block's visible tokens of the token score;
 *   R2 token score = sum over all query heads of the int8 dot product;
 *   R3 one selection per query row, shared by every head;
 *   R4 the window counts toward k and trails the row's last visible token;
 *   R5 an invalid block inside the window is dropped and its slot refilled;
 *   R7 row j of R rows of a request sees L - R + 1 + j tokens (clamped to
 *      [0, MB*P]);
 *   R9 low nibble = even element; tensor scale is a dequant multiplier.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_SENTINEL INT32_MIN

/* ---- element decoders (OCP MX v1.0 bit fields) ------------------------- */

/* e2m1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0. */
double qsa_oracle_e2m1(int code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;                                  /* subnormal */
    else
        v = ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* e4m3 (fn variant): sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0;
 * exponent 15 with mantissa 7 is NaN; there is no infinity. */
double qsa_oracle_e4m3(int byte)
{
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp(m / 8.0, -6);                       /* subnormal */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int qsa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads the following calls use (n >= 1); for single-thread timings. */
void qsa_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Tokens visible to row j of a request with L cached tokens (R7). */
static int64_t visible_tokens(int64_t L, int R, int j, int64_t cap)
{
    int64_t n = L - R + 1 + j;
    if (n < 0)
        n = 0;
    if (n > cap)
        n = cap;
    return n;
}

/* ---- A1: index scores --------------------------------------------------- */
/*
 * scores[r, beta] = max over tokens t of block beta with t < n_r of
 *                   sum_h sum_d iq[r, h, d] * ik[page, t - beta*P, d]      (R1, R2)
 * or INT32_MIN when the page entry is invalid (< 0 or >= NP) or no token of the
 * block is visible.  Rows [row_begin, row_end) are written; others untouched.
 */
int qsa_oracle_index_scores(int B, int R, int Hq, int Di, int P, int MB, int NP,
                            const int8_t *iq, const int8_t *ik_pool,
                            const int32_t *page_table, const int32_t *seqlens,
                            int row_begin, int row_end, int32_t *scores)
{
    int T = B * R;
    if (row_begin < 0) row_begin = 0;
    if (row_end > T) row_end = T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
    for (int r = row_begin; r < row_end; r++) {
        int b = r / R, j = r % R;
        int64_t n = visible_tokens(seqlens[b], R, j, (int64_t)MB * P);
        for (int beta = 0; beta < MB; beta++) {
            int32_t page = page_table[(int64_t)b * MB + beta];
            int32_t *dst = &scores[(int64_t)r * MB + beta];
            if (page < 0 || page >= NP || (int64_t)beta * P >= n) {
                *dst = ORACLE_SENTINEL;
                continue;
            }
            int64_t best = INT64_MIN;
            for (int tau = 0; tau < P; tau++) {
                if ((int64_t)beta * P + tau >= n)
                    break;
                const int8_t *key = ik_pool + ((int64_t)page * P + tau) * Di;
                int64_t s = 0;
                for (int h = 0; h < Hq; h++) {
                    const int8_t *qv = iq + ((int64_t)r * Hq + h) * Di;
                    for (int d = 0; d < Di; d++)
                        s += (int64_t)qv[d] * (int64_t)key[d];
                }
                if (s > best)
                    best = s;
            }
            if (best <= (int64_t)INT32_MIN || best > (int64_t)INT32_MAX)
                bad = 1;
            *dst = (int32_t)best;
        }
    }
    return bad ? -1 : 0;
}

/* ---- A2: canonical selection ------------------------------------------- */

typedef struct {
    int32_t score;
    int32_t beta;
} cand_t;

/* Rank order: higher score first; on equal scores the higher block index. */
static int cmp_rank(const void *a, const void *b)
{
    const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
    if (x->score != y->score)
        return x->score > y->score ? -1 : 1;
    if (x->beta != y->beta)
        return x->beta > y->beta ? -1 : 1;
    return 0;
}

static int cmp_int_asc(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * Per row: valid blocks are the visible blocks (beta < ceil(n_r / P)) whose
 * score is not the invalid sentinel.  The window is the valid blocks among the
 * last W visible ones (R4, R5).  The other valid blocks are ranked by (score
 * desc, beta desc) with a full sort and the first k - |window| are taken.  The
 * output lists window and taken blocks in ascending order, padded with -1;
 * nsel is their count.
 */
int qsa_oracle_select(int B, int R, int P, int MB, const int32_t *scores,
                      const int32_t *seqlens, int k, int W, int row_begin,
                      int row_end, int32_t *sel, int32_t *nsel)
{
    int T = B * R;
    if (k < 1 || W < 0 || W > k)
        return -1;
    if (row_begin < 0) row_begin = 0;
    if (row_end > T) row_end = T;
    int oom = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : oom)
    for (int r = row_begin; r < row_end; r++) {
        int b = r / R, j = r % R;
        int64_t n = visible_tokens(seqlens[b], R, j, (int64_t)MB * P);
        int nb = (int)((n + P - 1) / P);
        int wlo = nb - W > 0 ? nb - W : 0;
        const int32_t *row = scores + (int64_t)r * MB;
        int32_t *chosen = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
        cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)(nb > 0 ? nb : 1));
        if (!chosen || !cand) {
            free(chosen);
            free(cand);
            oom = 1;
            continue;
        }
        int nc = 0;
        for (int beta = wlo; beta < nb; beta++)
            if (row[beta] != ORACLE_SENTINEL)
                chosen[nc++] = beta;
        int ncand = 0;
        for (int beta = 0; beta < wlo; beta++)
            if (row[beta] != ORACLE_SENTINEL) {
                cand[ncand].score = row[beta];
                cand[ncand].beta = beta;
                ncand++;
            }
        qsort(cand, (size_t)ncand, sizeof(cand_t), cmp_rank);
        int take = k - nc;
        if (take > ncand)
            take = ncand;
        for (int i = 0; i < take; i++)
            chosen[nc++] = cand[i].beta;
        qsort(chosen, (size_t)nc, sizeof(int32_t), cmp_int_asc);
        for (int i = 0; i < k; i++)
            sel[(int64_t)r * k + i] = i < nc ? chosen[i] : -1;
        nsel[r] = nc;
        free(chosen);
        free(cand);
    }
    return oom ? -2 : 0;
}

/* ---- A3: sparse GQA attention over the selected NVFP4 pages ------------- */

/* Dequantised element (page p, KV head g, token tau, dim d) (R9). */
static double nvfp4_elem(const uint8_t *pool, const uint8_t *sf, double tscale,
                         int Hkv, int P, int D, int64_t p, int g, int tau, int d)
{
    int64_t row = ((p * Hkv + g) * P + tau);
    uint8_t byte = pool[row * (D / 2) + d / 2];
    int code = (d & 1) ? (byte >> 4) : (byte & 15);
    uint8_t s = sf[row * (D / 16) + d / 16];
    return qsa_oracle_e2m1(code) * qsa_oracle_e4m3(s) * tscale;
}

/*
 * For row r (request b = r / R) and query head h (KV head g = h / (Hq/Hkv)):
 * the tokens are those of the distinct blocks listed in sel[r, :] (entries in
 * [0, MB)) whose page entry is valid, restricted to t < n_r.  z_t = sm_scale * q . K_t,
 * lse = ln sum_t exp(z_t), out = sum_t exp(z_t - lse) V_t, computed two-pass
 * (max, then sum) in double.  No tokens: out = 0, lse = -inf.
 * out is [T, Hq, D] double, lse is [T, Hq] double.
 */
int qsa_oracle_attention(int B, int R, int Hq, int Hkv, int D, int P, int MB,
                         int NP, const uint16_t *q_bf16, const uint8_t *k_pool,
                         const uint8_t *k_sf, const uint8_t *v_pool,
                         const uint8_t *v_sf, double k_scale, double v_scale,
                         double sm_scale, const int32_t *page_table,
                         const int32_t *seqlens, const int32_t *sel, int k,
                         int row_begin, int row_end, double *out, double *lse)
{
    int T = B * R;
    if (Hkv <= 0 || Hq % Hkv != 0 || D % 16 != 0)
        return -1;
    int G = Hq / Hkv;
    if (row_begin < 0) row_begin = 0;
    if (row_end > T) row_end = T;
    int64_t cap_tokens = (int64_t)k * P;
    int oom = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : oom)
    for (int r = row_begin; r < row_end; r++) {
        for (int h = 0; h < Hq; h++) {
            int b = r / R, j = r % R, g = h / G;
            int64_t n = visible_tokens(seqlens[b], R, j, (int64_t)MB * P);
            double *z = (double *)malloc(sizeof(double) * (size_t)(cap_tokens > 0 ? cap_tokens : 1));
            int64_t *tp = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cap_tokens > 0 ? cap_tokens : 1));
            int *tt = (int *)malloc(sizeof(int) * (size_t)(cap_tokens > 0 ? cap_tokens : 1));
            if (!z || !tp || !tt) {
                free(z); free(tp); free(tt);
                oom = 1;
                continue;
            }
            const uint16_t *qv = q_bf16 + ((int64_t)r * Hq + h) * D;
            int64_t nt = 0;
            for (int i = 0; i < k; i++) {
                int32_t beta = sel[(int64_t)r * k + i];
                if (beta < 0 || beta >= MB)
                    continue;
                int dup = 0;                  /* a block counts once */
                for (int i2 = 0; i2 < i; i2++)
                    if (sel[(int64_t)r * k + i2] == beta)
                        dup = 1;
                if (dup)
                    continue;
                int32_t page = page_table[(int64_t)b * MB + beta];
                if (page < 0 || page >= NP)
                    continue;
                for (int tau = 0; tau < P; tau++) {
                    if ((int64_t)beta * P + tau >= n)
                        break;
                    double dot = 0.0;
                    for (int d = 0; d < D; d++)
                        dot += bf16_to_double(qv[d]) *
                               nvfp4_elem(k_pool, k_sf, k_scale, Hkv, P, D, page, g, tau, d);
                    z[nt] = sm_scale * dot;
                    tp[nt] = page;
                    tt[nt] = tau;
                    nt++;
                }
            }
            double *o = out + ((int64_t)r * Hq + h) * D;
            if (nt == 0) {
                for (int d = 0; d < D; d++)
                    o[d] = 0.0;
                lse[(int64_t)r * Hq + h] = -INFINITY;
            } else {
                double m = z[0];
                for (int64_t t = 1; t < nt; t++)
                    if (z[t] > m)
                        m = z[t];
                double l = 0.0;
                for (int64_t t = 0; t < nt; t++)
                    l += exp(z[t] - m);
                double L = m + log(l);
                for (int d = 0; d < D; d++) {
                    double acc = 0.0;
                    for (int64_t t = 0; t < nt; t++)
                        acc += exp(z[t] - L) *
                               nvfp4_elem(v_pool, v_sf, v_scale, Hkv, P, D, tp[t], g, tt[t], d);
                    o[d] = acc;
                }
                lse[(int64_t)r * Hq + h] = L;
            }
            free(z); free(tp); free(tt);
        }
    }
    return oom ? -2 : 0;
}

/* ---- decode prologue: NVFP4 quantiser and token store ------------------
 *
 * TensorRT-LLM PR #20937 "GB300 perf work on
 * qwen3_8_flash_next_nvfp4__sm_103__tp1", What changes: a decode prologue over
 * the NVFP4 KV cache that also serves verify steps; Walkthrough, changes
 * table: NVFP4 storage in the decode prologue.  The pages print no quantiser;
 * the recipe below is the plain per-16-element NVFP4 reading:
 *   sf     = e4m3_rne_satfinite((max|x| / 6) / scale)
 *   code_i = e2m1_rne_satfinite(x_i / (e4m3(sf) * scale))
 * Where floating point decides a code, the decision is taken in IEEE fp32
 * (the pages fix no precision; fp32 is what the library computes in), with
 * the divisions and the product in that order.  The encoders are written from
 * the element definitions: the nearest representable magnitude, a tie going
 * to the code whose lowest bit is 0 (the even mantissa), saturating at the
 * largest finite value.  A code whose magnitude is zero is stored as +0.
 */

/* e4m3 byte (sign 0) nearest to q >= 0. */
int qsa_oracle_e4m3_encode(float q)
{
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; c++) {                 /* 0x7F is NaN */
        double d = fabs((double)q - qsa_oracle_e4m3(c));
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    return best;
}

/* e2m1 code nearest to y (sign bit 3; magnitude zero stored as +0). */
int qsa_oracle_e2m1_encode(float y)
{
    double a = fabs((double)y);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 7; c++) {
        double d = fabs(a - qsa_oracle_e2m1(c));
        if (d < bd || (d == bd && (c & 1) == 0)) {
            best = c;
            bd = d;
        }
    }
    if (best != 0 && y < 0.0f)
        best |= 8;
    return best;
}

/* One 16-element block: 16 codes and the scale byte. */
void qsa_oracle_quantize_block(const float *x, float scale, uint8_t *codes, uint8_t *sf_out)
{
    float a = 0.0f;
    for (int i = 0; i < 16; i++) {
        float v = fabsf(x[i]);
        if (v > a)
            a = v;
    }
    float q = (a / 6.0f) / scale;     /* ISO C, no contraction: each op rounds */
    int sf = qsa_oracle_e4m3_encode(q);
    float den = (float)qsa_oracle_e4m3(sf) * scale;
    for (int i = 0; i < 16; i++) {
        if (den == 0.0f) {
            codes[i] = 0;
        } else {
            codes[i] = (uint8_t)qsa_oracle_e2m1_encode(x[i] / den);
        }
    }
    *sf_out = (uint8_t)sf;
}

static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Row r = b*R + j is the token at position L_b - R + j of request b: block
 * pos / P, slot pos % P of page page_table[b, pos / P]; skipped when
 * pos < 0, pos >= MB*P or the page is invalid.  k_new / v_new: bf16
 * [T, Hkv, D]; ik_new: int8 [T, Di].  The pools are updated in place.
 */
int qsa_oracle_store_kv(int B, int R, int Hkv, int D, int Di, int P, int MB, int NP,
                        const uint16_t *k_new, const uint16_t *v_new, const int8_t *ik_new,
                        float k_scale, float v_scale, const int32_t *page_table,
                        const int32_t *seqlens, uint8_t *k_pool, uint8_t *k_sf,
                        uint8_t *v_pool, uint8_t *v_sf, int8_t *ik_pool)
{
    if (D % 16 != 0)
        return -1;
    for (int b = 0; b < B; b++) {
        for (int j = 0; j < R; j++) {
            int64_t pos = (int64_t)seqlens[b] - R + j;
            if (pos < 0 || pos >= (int64_t)MB * P)
                continue;
            int beta = (int)(pos / P), slot = (int)(pos % P);
            int32_t page = page_table[(int64_t)b * MB + beta];
            if (page < 0 || page >= NP)
                continue;
            int64_t r = (int64_t)b * R + j;
            for (int g = 0; g < Hkv; g++) {
                int64_t row = ((int64_t)page * Hkv + g) * P + slot;
                for (int kv = 0; kv < 2; kv++) {
                    const uint16_t *src = (kv ? v_new : k_new) + (r * Hkv + g) * D;
                    uint8_t *pool = kv ? v_pool : k_pool;
                    uint8_t *sfp = kv ? v_sf : k_sf;
                    float scale = kv ? v_scale : k_scale;
                    for (int blk = 0; blk < D / 16; blk++) {
                        float x[16];
                        uint8_t codes[16], sf;
                        for (int i = 0; i < 16; i++)
                            x[i] = bf16_to_float(src[blk * 16 + i]);
                        qsa_oracle_quantize_block(x, scale, codes, &sf);
                        for (int i = 0; i < 16; i += 2)
                            pool[row * (D / 2) + blk * 8 + i / 2] =
                                (uint8_t)(codes[i] | (codes[i + 1] << 4));
                        sfp[row * (D / 16) + blk] = sf;
                    }
                }
            }
            memcpy(ik_pool + ((int64_t)page * P + slot) * Di, ik_new + r * Di, (size_t)Di);
        }
    }
    return 0;
}

/* ---- speculative rollback of the cache planes ---------------------------
 *
 * TensorRT-LLM PR #20937 "GB300 perf work on
 * qwen3_8_flash_next_nvfp4__sm_103__tp1", What changes (Rollback and PLE):
 * batched rollback of the QSA index planes; rollback gather / restore of the
 * planes, whose test restores the rejected rows' old values and leaves kept
 * rows untouched.  Row r = b*R + j owns the slot at position L_b - R + j
 * (skipped when negative, at or past MB*P, or on an invalid page).  Saved
 * state of row r, at r * (144*Hkv + 64): per KV head K codes (D/2), K scales
 * (D/16), V codes (D/2), V scales (D/16); then the index key (Di).
 */
static int row_slot(int b, int R, int j, int P, int MB, int NP, const int32_t *page_table,
                    const int32_t *seqlens, int32_t *page, int *slot)
{
    int64_t pos = (int64_t)seqlens[b] - R + j;
    if (pos < 0 || pos >= (int64_t)MB * P)
        return 0;
    *page = page_table[(int64_t)b * MB + pos / P];
    if (*page < 0 || *page >= NP)
        return 0;
    *slot = (int)(pos % P);
    return 1;
}

/* restore == 0: pools -> saved (every row with a slot);
 * restore != 0: saved -> pools (rows with a slot and rejected[r] != 0). */
int qsa_oracle_rollback(int restore, int B, int R, int Hkv, int D, int Di, int P, int MB, int NP,
                        const int32_t *page_table, const int32_t *seqlens,
                        const int32_t *rejected, uint8_t *k_pool, uint8_t *k_sf,
                        uint8_t *v_pool, uint8_t *v_sf, int8_t *ik_pool, uint8_t *saved)
{
    int64_t row_bytes = (int64_t)Hkv * (2 * (D / 2 + D / 16)) + Di;
    for (int b = 0; b < B; b++) {
        for (int j = 0; j < R; j++) {
            int64_t r = (int64_t)b * R + j;
            int32_t page;
            int slot;
            if (!row_slot(b, R, j, P, MB, NP, page_table, seqlens, &page, &slot))
                continue;
            if (restore && rejected[r] == 0)
                continue;
            uint8_t *s = saved + r * row_bytes;
            for (int g = 0; g < Hkv; g++) {
                int64_t row = ((int64_t)page * Hkv + g) * P + slot;
                uint8_t *parts[4] = {k_pool + row * (D / 2), k_sf + row * (D / 16),
                                     v_pool + row * (D / 2), v_sf + row * (D / 16)};
                int sizes[4] = {D / 2, D / 16, D / 2, D / 16};
                for (int q = 0; q < 4; q++) {
                    if (restore)
                        memcpy(parts[q], s, (size_t)sizes[q]);
                    else
                        memcpy(s, parts[q], (size_t)sizes[q]);
                    s += sizes[q];
                }
            }
            int8_t *key = ik_pool + ((int64_t)page * P + slot) * Di;
            if (restore)
                memcpy(key, s, (size_t)Di);
            else
                memcpy(s, key, (size_t)Di);
        }
    }
    return 0;
}
