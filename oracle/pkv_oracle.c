/*
 * pkv_oracle.c -- plain fp64 CPU oracle for one paged grouped-query decode-attention step.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference arm may
 * load this library. The product path (serving_paged_gqa_gb300) never links, imports or calls it, and this file
 * shares no code, header, table or constant with the CUDA path.
 *
 * What it computes follows "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity
 * GPUs" (arXiv 2606.26666):
 *   - problem statement (gist.science technical summary, "Methodologie" 1): grouped-query attention where
 *     G = Hq/Hkv query heads share one KV head, executed directly over the native block-table page layout;
 *   - sequence splitting into S disjoint ranges, each a partial online-softmax state, combined exactly by a merge
 *     (same section, "Sequentie Splitting");
 *   - row-local bounds: split ranges come from each row's real length; empty splits hold a neutral state
 *     (same section, "Row-Local Bounds");
 *   - the compact workqueue of non-empty (row, KV head, split) tasks (same section, "Compact Workqueue"; abstract).
 * The attention itself is the textbook definition written out: for query head hq of row b, with hkv = hq / G,
 *   s_j = scale * <q[b,hq,:], k_j>,  w_j = exp(s_j - max s) / sum exp(s - max s),  out = sum_j w_j v_j,
 * over the row's tokens j = 0..L_b-1, token j living in slot j % ps of physical page block_table[b][j / ps].
 * Everything is fp64; fp16 inputs are widened exactly.
 *
 * Parity pins (tests/test_oracle_pins.py): fp16 widening checked on all 65536 bit patterns against numpy; dense
 * numpy attention on the gathered contiguous KV; a pure-Python brute force on tiny inputs; closed forms (L=1,
 * q=0, equal keys, one dominant key, all-ones values); physical-page permutation invariance; split/merge
 * invariance; hand-derived worklists and the closed-form task count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_EPAGE (-2)
#define OR_ENOMEM (-3)

/* IEEE 754 binary16 -> double: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. Exact. */
double pkv_oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

int pkv_oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Shapes shared by the calls below. q is [B][Hq][d], pools are [num_pages][ps][Hkv][d], block_table is
 * [B][max_pages], seq_lens is [B]; all row-major and contiguous, fp16 stored as raw uint16 bits. */
typedef struct {
    int B, Hq, Hkv, d, ps, num_pages, max_pages;
} or_shape;

static int shape_ok(const or_shape* s) {
    return s->B >= 0 && s->Hq > 0 && s->Hkv > 0 && s->Hq % s->Hkv == 0 && s->d > 0 && s->ps > 0 &&
           s->num_pages >= 0 && s->max_pages >= 0;
}

/* Physical address of token j's row for KV head hkv of row b, or NULL if the block table points outside the pool. */
static const uint16_t* token_row(const or_shape* s, const uint16_t* pool, const int32_t* block_table, int b,
                                 int64_t j, int hkv) {
    int64_t p = j / s->ps, slot = j % s->ps;
    int32_t phys = block_table[(int64_t)b * s->max_pages + p];
    if (phys < 0 || phys >= s->num_pages) return NULL;
    return pool + (((int64_t)phys * s->ps + slot) * s->Hkv + hkv) * s->d;
}

/* Partial online-softmax state of query head hq of row b over tokens [t0, t1):
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  acc = sum_j exp(s_j - m) v_j.
 * An empty range gives the neutral state m = -inf, l = 0, acc = 0. With t0 = 0 and t1 = L_b, acc / l is the
 * attention output. scores must hold t1 - t0 doubles. */
static int state_range(const or_shape* s, const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                       const int32_t* block_table, double scale, int b, int hq, int64_t t0, int64_t t1,
                       double* scores, double* m_out, double* l_out, double* acc) {
    int G = s->Hq / s->Hkv;
    int hkv = hq / G;
    const uint16_t* qr = q + ((int64_t)b * s->Hq + hq) * s->d;
    for (int i = 0; i < s->d; ++i) acc[i] = 0.0;
    if (t1 <= t0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return OR_OK;
    }
    double m = -INFINITY;
    for (int64_t j = t0; j < t1; ++j) {
        const uint16_t* kr = token_row(s, k_pool, block_table, b, j, hkv);
        if (!kr) return OR_EPAGE;
        double dot = 0.0;
        for (int i = 0; i < s->d; ++i) dot += pkv_oracle_half_to_double(qr[i]) * pkv_oracle_half_to_double(kr[i]);
        scores[j - t0] = dot * scale;
        if (scores[j - t0] > m) m = scores[j - t0];
    }
    double l = 0.0;
    for (int64_t j = t0; j < t1; ++j) {
        const uint16_t* vr = token_row(s, v_pool, block_table, b, j, hkv);
        if (!vr) return OR_EPAGE;
        double w = exp(scores[j - t0] - m);
        l += w;
        for (int i = 0; i < s->d; ++i) acc[i] += w * pkv_oracle_half_to_double(vr[i]);
    }
    *m_out = m;
    *l_out = l;
    return OR_OK;
}

/* Attention output for n_pairs (b, hq) pairs given as pairs[2*i], pairs[2*i+1]; out is [n_pairs][d].
 * pairs == NULL means all B*Hq pairs in (b, hq) order. A row with L_b = 0 has output 0. */
int pkv_oracle_attention(int B, int Hq, int Hkv, int d, int ps, int num_pages, int max_pages, const uint16_t* q,
                         const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* block_table,
                         const int32_t* seq_lens, double scale, const int32_t* pairs, int64_t n_pairs,
                         double* out) {
    or_shape s = {B, Hq, Hkv, d, ps, num_pages, max_pages};
    if (!shape_ok(&s)) return OR_EINVAL;
    if (!pairs) n_pairs = (int64_t)B * Hq;
    int64_t maxlen = 0;
    for (int b = 0; b < B; ++b) {
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_pages * ps) return OR_EINVAL;
        if (seq_lens[b] > maxlen) maxlen = seq_lens[b];
    }
    int err = OR_OK;
#pragma omp parallel
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
        if (!scores) {
#pragma omp atomic write
            err = OR_ENOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_pairs; ++i) {
            if (!scores) continue;
            int b = pairs ? pairs[2 * i] : (int)(i / Hq);
            int hq = pairs ? pairs[2 * i + 1] : (int)(i % Hq);
            double* o = out + i * d;
            if (b < 0 || b >= B || hq < 0 || hq >= Hq) {
#pragma omp atomic write
                err = OR_EINVAL;
                continue;
            }
            double m, l;
            int rc = state_range(&s, q, k_pool, v_pool, block_table, scale, b, hq, 0, seq_lens[b], scores, &m, &l, o);
            if (rc != OR_OK) {
#pragma omp atomic write
                err = rc;
                continue;
            }
            if (l > 0.0)
                for (int k = 0; k < d; ++k) o[k] /= l;
        }
        free(scores);
    }
    return err;
}

/* Partial state (m, l, acc[d]) of pair (b, hq) over tokens [t0, t1), clipped to [0, L_b). */
int pkv_oracle_split_state(int B, int Hq, int Hkv, int d, int ps, int num_pages, int max_pages, const uint16_t* q,
                           const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* block_table,
                           const int32_t* seq_lens, double scale, int b, int hq, int64_t t0, int64_t t1, double* m,
                           double* l, double* acc) {
    or_shape s = {B, Hq, Hkv, d, ps, num_pages, max_pages};
    if (!shape_ok(&s) || b < 0 || b >= B || hq < 0 || hq >= Hq) return OR_EINVAL;
    int64_t L = seq_lens[b];
    if (t0 < 0) t0 = 0;
    if (t1 > L) t1 = L;
    double* scores = (double*)malloc(sizeof(double) * (size_t)(t1 > t0 ? t1 - t0 : 1));
    if (!scores) return OR_ENOMEM;
    int rc = state_range(&s, q, k_pool, v_pool, block_table, scale, b, hq, t0, t1, scores, m, l, acc);
    free(scores);
    return rc;
}

/* Exact combination of S partial states over disjoint ranges of one (b, hq):
 *   M = max_s m_s over non-neutral states,  w_s = exp(m_s - M),  out = sum_s w_s acc_s / sum_s w_s l_s.
 * Neutral states (l_s = 0) contribute nothing; if every state is neutral the output is 0. */
void pkv_oracle_merge(int64_t S, int d, const double* m, const double* l, const double* acc, double* out) {
    double M = -INFINITY;
    for (int64_t s = 0; s < S; ++s)
        if (l[s] > 0.0 && m[s] > M) M = m[s];
    for (int i = 0; i < d; ++i) out[i] = 0.0;
    if (M == -INFINITY) return;
    double den = 0.0;
    for (int64_t s = 0; s < S; ++s) {
        if (!(l[s] > 0.0)) continue;
        double w = exp(m[s] - M);
        den += w * l[s];
        for (int i = 0; i < d; ++i) out[i] += w * acc[s * d + i];
    }
    for (int i = 0; i < d; ++i) out[i] /= den;
}

/* Reference compact worklist: the non-empty (row, KV head, split) tasks in lexicographic (b, h, s) order.
 * Row b has P_b = ceil(L_b / ps) pages and S_b = ceil(P_b / c) splits of c pages (0 if L_b = 0); split s covers
 * logical pages [s*c, min((s+1)*c, P_b)). Each task is 5 int32: b, h, s, page_begin, page_end. Returns the task
 * count (sum_b Hkv * S_b); writes at most cap tasks; negative on bad arguments. */
int64_t pkv_oracle_worklist(int B, const int32_t* seq_lens, int ps, int Hkv, int c, int32_t* tasks, int64_t cap) {
    if (B < 0 || ps <= 0 || Hkv <= 0 || c <= 0) return OR_EINVAL;
    int64_t n = 0;
    for (int b = 0; b < B; ++b) {
        int64_t L = seq_lens[b];
        if (L < 0) return OR_EINVAL;
        int64_t P = (L + ps - 1) / ps;
        int64_t S = (P + c - 1) / c;
        for (int h = 0; h < Hkv; ++h) {
            for (int64_t sp = 0; sp < S; ++sp) {
                if (n < cap && tasks) {
                    int64_t pb = sp * c, pe = (sp + 1) * c < P ? (sp + 1) * c : P;
                    int32_t* t = tasks + 5 * n;
                    t[0] = b;
                    t[1] = h;
                    t[2] = (int32_t)sp;
                    t[3] = (int32_t)pb;
                    t[4] = (int32_t)pe;
                }
                ++n;
            }
        }
    }
    return n;
}
