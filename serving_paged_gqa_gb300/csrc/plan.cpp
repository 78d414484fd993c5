// Host planner: workspace layout and the roofline-style cost-model policy.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs": the v2 abstract
// names a calibrated roofline-style policy whose cost-model constants are fixed on calibration traces and which
// routes each step to one execution path; the gist.science technical summary, "Calibrated Adaptive Policy", keys
// that choice on batch size B and the longest context N_max. Here the candidates are this library's own
// single-pass kernel, the rectangular split grid and the compact workqueue, each over a set of split sizes c
// (pages per split) and with the separate or the fused merge; the model (include/pkv.h, pkv_policy) predicts each
// candidate's step time and the cheapest is kept. Its constants come from policy_constants.h, which the
// calibration tool writes.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "pkv_internal.h"
#include "policy_constants.h"

namespace {

using namespace pkv;

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8 || g == 16; }

}  // namespace

extern "C" int pkv_check_problem(const pkv_problem* pr) {
    if (!pr) return PKV_E_NULLPTR;
    if (pr->batch < 0 || pr->num_q_heads <= 0 || pr->num_kv_heads <= 0 || pr->head_dim <= 0 ||
        pr->page_size <= 0 || pr->num_pages < 0 || pr->max_pages_per_seq < 0)
        return PKV_E_INVAL;
    if (pr->num_q_heads % pr->num_kv_heads != 0) return PKV_E_UNSUPPORTED;
    if (pr->head_dim != kHeadDim || pr->page_size != kPageSize) return PKV_E_UNSUPPORTED;
    if (!supported_group(pr->num_q_heads / pr->num_kv_heads)) return PKV_E_UNSUPPORTED;
    if (pr->batch > PKV_MAX_BATCH) return PKV_E_UNSUPPORTED;
    if (pr->num_kv_heads > 0x7fff) return PKV_E_UNSUPPORTED;
    if ((int64_t)pr->max_pages_per_seq * kPageSize > 0x7fffffffLL) return PKV_E_UNSUPPORTED;
    return PKV_OK;
}

extern "C" void pkv_policy_default(pkv_policy* pol) {
    if (!pol) return;
    std::memset(pol, 0, sizeof(*pol));
    pol->launch_us = PKV_FIT_LAUNCH_US;
    pol->hbm_gbs = PKV_FIT_HBM_GBS;
    pol->cta_gbs = PKV_FIT_CTA_GBS;
    pol->wq_cta_gbs = PKV_FIT_WQ_CTA_GBS;
    pol->task_us = PKV_FIT_TASK_US;
    pol->tail = PKV_FIT_TAIL;
    pol->merge_us = PKV_FIT_MERGE_US;
    pol->merge_state_us = PKV_FIT_MERGE_STATE_US;
    pol->fused_us = PKV_FIT_FUSED_US;
    pol->fused_state_us = PKV_FIT_FUSED_STATE_US;
    pol->build_us = PKV_FIT_BUILD_US;
    pol->ctas_per_sm = kDecodeCtasPerSm;
    pol->max_splits = 1024;
    pol->allow_variants = (1 << PKV_VARIANT_SINGLE) | (1 << PKV_VARIANT_SPLIT) | (1 << PKV_VARIANT_WORKQUEUE);
    pol->allow_fused = 1;
    pol->split_max_batch = 2;
}

namespace {

int fill_plan(const pkv_problem* pr, const int32_t* lens, int32_t num_sms, int32_t variant, int32_t chunk,
              int32_t ctas_per_sm, pkv_plan_t* plan) {
    int rc = pkv_check_problem(pr);
    if (rc != PKV_OK) return rc;
    if (!plan || (pr->batch > 0 && !lens)) return PKV_E_NULLPTR;
    if (num_sms <= 0) return PKV_E_INVAL;
    if (variant < PKV_VARIANT_SINGLE || variant > PKV_VARIANT_WORKQUEUE) return PKV_E_INVAL;
    if (ctas_per_sm <= 0) ctas_per_sm = 2;
    const int B = pr->batch, Hkv = pr->num_kv_heads, G = pr->num_q_heads / pr->num_kv_heads;
    // never more CTAs per SM than fit in its registers and shared memory: the persistent grid is one wave
    ctas_per_sm = std::min(ctas_per_sm, kDecodeCtasPerSm);
    const int smem = decode_smem_bytes(G);
    if (smem > 0) ctas_per_sm = std::max(1, std::min(ctas_per_sm, kSmemPerSm / (smem + kSmemReservedPerCta)));
    int64_t max_pages = 0, sum_len = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 0 || (int64_t)lens[b] > (int64_t)pr->max_pages_per_seq * kPageSize) return PKV_E_INVAL;
        max_pages = std::max<int64_t>(max_pages, (lens[b] + kPageSize - 1) / kPageSize);
        sum_len += lens[b];
    }
    if (variant == PKV_VARIANT_SINGLE) {
        chunk = std::max<int32_t>(1, pr->max_pages_per_seq);
    } else if (chunk < 1) {
        return PKV_E_INVAL;
    }
    int64_t splits = 0, wq_tasks = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t P = (lens[b] + kPageSize - 1) / kPageSize;
        const int64_t S = (P + chunk - 1) / chunk;
        splits = std::max(splits, S);
        wq_tasks += (int64_t)Hkv * S;
    }
    if (variant == PKV_VARIANT_SINGLE) splits = 1;
    if (splits > 0xffff) return PKV_E_UNSUPPORTED;
    splits = std::max<int64_t>(splits, 1);
    int64_t tasks;
    if (variant == PKV_VARIANT_WORKQUEUE)
        tasks = wq_tasks;
    else
        tasks = (int64_t)B * Hkv * splits;
    if (tasks > 0x7fffffffLL / G) return PKV_E_UNSUPPORTED;

    std::memset(plan, 0, sizeof(*plan));
    plan->variant = variant;
    plan->chunk_pages = chunk;
    plan->num_splits = (int32_t)splits;
    plan->num_tasks = (int32_t)tasks;
    plan->fuse_merge = variant == PKV_VARIANT_SINGLE ? 0 : 1;
    plan->list_in_decode = variant == PKV_VARIANT_WORKQUEUE && B <= PKV_MAX_ROWS_IN_DECODE ? 1 : 0;
    plan->group = G;
    plan->num_sms = num_sms;
    plan->problem = *pr;
    const int64_t grid_cap = (int64_t)ctas_per_sm * num_sms;
    plan->grid_ctas = (int32_t)std::max<int64_t>(1, std::min<int64_t>(tasks, grid_cap));
    plan->task_capacity = variant == PKV_VARIANT_WORKQUEUE ? tasks : 0;
    plan->state_capacity = variant == PKV_VARIANT_SINGLE ? 0 : tasks * G;

    int64_t off = kWsAlign;  // header
    plan->off_counters = off;
    off = align_up(off + 4 * (int64_t)B * Hkv, kWsAlign);
    plan->off_row_off = off;
    off = align_up(off + 4 * (int64_t)B, kWsAlign);
    plan->off_row_splits = off;
    off = align_up(off + 4 * (int64_t)B, kWsAlign);
    plan->off_tasks = off;
    off = align_up(off + (int64_t)sizeof(pkv_task) * plan->task_capacity, kWsAlign);
    plan->off_ml = off;
    off = align_up(off + 8 * plan->state_capacity, kWsAlign);
    plan->off_acc = off;
    off = align_up(off + 4 * (int64_t)kHeadDim * plan->state_capacity, kWsAlign);
    plan->ws_bytes = off;
    plan->kv_bytes = (double)kTokenHeadBytes * Hkv * (double)sum_len +
                     2.0 * 2.0 * (double)B * pr->num_q_heads * kHeadDim;
    (void)max_pages;
    return PKV_OK;
}

// What the model needs of a candidate plan (the rest of pkv_plan_t is workspace layout).
struct Cand {
    int32_t variant, chunk, group, list_in_decode, fuse;
    int64_t splits, tasks, grid, p_max;
    double kv_bytes;
};

int64_t max_row_pages(const int32_t* lens, int B) {
    int64_t p_max = 0;
    for (int b = 0; b < B; ++b) p_max = std::max<int64_t>(p_max, ((int64_t)lens[b] + kPageSize - 1) / kPageSize);
    return p_max;
}

Cand cand_of(const pkv_plan_t* plan, const int32_t* lens) {
    Cand c;
    c.variant = plan->variant;
    c.chunk = plan->chunk_pages;
    c.group = plan->group;
    c.list_in_decode = plan->list_in_decode;
    c.fuse = plan->fuse_merge;
    c.splits = plan->num_splits;
    c.tasks = plan->num_tasks;
    c.grid = plan->grid_ctas;
    c.p_max = max_row_pages(lens, plan->problem.batch);
    c.kv_bytes = plan->kv_bytes;
    return c;
}

// Step time of a candidate under the model documented with pkv_policy (include/pkv.h).
double predict(const pkv_policy* pol, const Cand& c) {
    const double T = (double)c.tasks;
    if (T <= 0) return pol->launch_us;
    const double W = (double)std::max<int64_t>(1, c.grid);
    const double A = std::min(T, W);
    const double pages_per_task = c.variant == PKV_VARIANT_SINGLE ? (double)c.p_max
                                                                   : (double)std::min<int64_t>(c.chunk, c.p_max);
    const double task_bytes = pages_per_task * kPageSize * kTokenHeadBytes;
    const double gb = 1e3;  // bytes / (GB/s * 1e3) = microseconds
    double t;
    if (c.variant == PKV_VARIANT_WORKQUEUE) {
        const double stream = c.kv_bytes / (std::min(pol->hbm_gbs, A * pol->wq_cta_gbs) * gb);
        const double makespan = std::ceil(T / W) * task_bytes / (pol->wq_cta_gbs * gb);
        t = pol->launch_us + stream + (T / W) * pol->task_us + pol->tail * std::max(0.0, makespan - stream);
    } else {
        const double share = std::min(pol->cta_gbs, pol->hbm_gbs / A) * gb;
        t = pol->launch_us + std::ceil(T / W) * (pol->task_us + (c.kv_bytes / T) / share);
    }
    if (c.variant != PKV_VARIANT_SINGLE) {
        const double s_max = c.variant == PKV_VARIANT_SPLIT ? (double)c.splits
                                                            : std::ceil((double)c.p_max / std::max(1, c.chunk));
        if (c.fuse)
            t += pol->fused_us + pol->fused_state_us * s_max * c.group;
        else
            t += pol->merge_us + pol->merge_state_us * s_max;
    }
    if (c.variant == PKV_VARIANT_WORKQUEUE && !c.list_in_decode) t += pol->build_us;
    return t;
}

// The cheaper merge mode for a candidate (the fused one only if allowed and not single pass); returns its time.
double choose_merge(const pkv_policy* pol, Cand& c) {
    c.fuse = 0;
    const double sep = predict(pol, c);
    if (c.variant == PKV_VARIANT_SINGLE || !pol->allow_fused) return sep;
    c.fuse = 1;
    const double fused = predict(pol, c);
    if (fused < sep) return fused;
    c.fuse = 0;
    return sep;
}

}  // namespace

extern "C" int pkv_plan_fixed(const pkv_problem* pr, const int32_t* lens, int32_t num_sms, int32_t variant,
                              int32_t chunk_pages, int32_t ctas_per_sm, pkv_plan_t* plan) {
    int rc = fill_plan(pr, lens, num_sms, variant, chunk_pages, ctas_per_sm, plan);
    if (rc != PKV_OK) return rc;
    pkv_policy pol;
    pkv_policy_default(&pol);
    Cand c = cand_of(plan, lens);
    plan->predicted_us = choose_merge(&pol, c);
    plan->fuse_merge = c.fuse;
    return PKV_OK;
}

extern "C" int pkv_plan(const pkv_problem* pr, const int32_t* lens, int32_t num_sms, const pkv_policy* policy,
                        pkv_plan_t* plan) {
    int rc = pkv_check_problem(pr);
    if (rc != PKV_OK) return rc;
    if (!plan || (pr->batch > 0 && !lens)) return PKV_E_NULLPTR;
    pkv_policy pol;
    if (policy)
        pol = *policy;
    else
        pkv_policy_default(&pol);
    if (pol.ctas_per_sm <= 0 || pol.max_splits <= 0 || !(pol.hbm_gbs > 0) || !(pol.cta_gbs > 0) ||
        !(pol.wq_cta_gbs > 0))
        return PKV_E_INVAL;
    if (num_sms <= 0) return PKV_E_INVAL;
    const int B = pr->batch, Hkv = pr->num_kv_heads, G = pr->num_q_heads / pr->num_kv_heads;
    int64_t max_pages = 0, sum_len = 0;
    for (int b = 0; b < B; ++b) {
        if (lens[b] < 0 || (int64_t)lens[b] > (int64_t)pr->max_pages_per_seq * kPageSize) return PKV_E_INVAL;
        max_pages = std::max<int64_t>(max_pages, (lens[b] + kPageSize - 1) / kPageSize);
        sum_len += lens[b];
    }
    // the grid limit fill_plan applies: CTAs per SM within registers and shared memory
    int ctas_per_sm = std::min<int>(pol.ctas_per_sm, kDecodeCtasPerSm);
    const int smem = decode_smem_bytes(G);
    if (smem > 0) ctas_per_sm = std::max(1, std::min(ctas_per_sm, kSmemPerSm / (smem + kSmemReservedPerCta)));
    const int64_t grid_cap = (int64_t)ctas_per_sm * num_sms;
    // candidate split sizes: powers of two and 1.5x powers of two, bounded so that S <= max_splits
    int32_t chunks[128];
    int nchunks = 0;
    const int64_t cmin = std::max<int64_t>(1, (max_pages + pol.max_splits - 1) / pol.max_splits);
    for (int64_t c = 1; c <= std::max<int64_t>(1, max_pages) && nchunks < 126; c *= 2) {
        if (c >= cmin) chunks[nchunks++] = (int32_t)c;
        const int64_t c3 = c + c / 2;
        if (c3 > c && c3 >= cmin && c3 <= max_pages) chunks[nchunks++] = (int32_t)c3;
    }
    if (nchunks == 0) chunks[nchunks++] = (int32_t)std::max<int64_t>(1, cmin);
    // per-row page counts once, then per candidate split size c: max_b S_b and sum_b S_b, S_b = ceil(P_b / c) (a
    // reciprocal multiply with an exact one-step correction per row instead of an integer division: at B = 4096 the
    // divisions were most of the planner's time)
    static_assert(PKV_MAX_BATCH <= 4096, "page-count scratch on the stack");
    int32_t pages[PKV_MAX_BATCH];
    for (int b = 0; b < B; ++b) pages[b] = (int32_t)(((int64_t)lens[b] + kPageSize - 1) / kPageSize);
    int64_t smax[128], ssum[128];
    for (int i = 0; i < nchunks; ++i) {
        const int64_t c = chunks[i];
        const double inv = 1.0 / (double)c;
        int64_t mx = 0, sum = 0;
        for (int b = 0; b < B; ++b) {
            const int64_t m = (int64_t)pages[b] + c - 1;
            int64_t q = (int64_t)((double)m * inv);
            if (q * c > m)
                --q;
            else if ((q + 1) * c <= m)
                ++q;
            mx = std::max(mx, q);
            sum += q;
        }
        smax[i] = mx;
        ssum[i] = sum;
    }
    // every candidate is scored on the few numbers the model reads; only the winner's workspace layout is filled
    const double kv_bytes = (double)kTokenHeadBytes * Hkv * (double)sum_len + 2.0 * 2.0 * (double)B * pr->num_q_heads * kHeadDim;
    bool have = false;
    Cand best{};
    double best_us = 0.0;
    for (int v = PKV_VARIANT_SINGLE; v <= PKV_VARIANT_WORKQUEUE; ++v) {
        if (!(pol.allow_variants & (1 << v))) continue;
        if (v == PKV_VARIANT_SPLIT && B > pol.split_max_batch) continue;
        const int n = v == PKV_VARIANT_SINGLE ? 1 : nchunks;
        for (int i = 0; i < n; ++i) {
            const int32_t chunk = v == PKV_VARIANT_SINGLE ? std::max<int32_t>(1, pr->max_pages_per_seq) : chunks[i];
            int64_t splits = 1, wq_tasks = 0;
            if (v != PKV_VARIANT_SINGLE) {
                splits = smax[i];
                wq_tasks = (int64_t)Hkv * ssum[i];
            }
            if (splits > 0xffff) continue;
            splits = std::max<int64_t>(splits, 1);
            const int64_t tasks = v == PKV_VARIANT_WORKQUEUE ? wq_tasks : (int64_t)B * Hkv * splits;
            if (tasks > 0x7fffffffLL / G) continue;
            Cand c;
            c.variant = v;
            c.chunk = chunk;
            c.group = G;
            c.list_in_decode = v == PKV_VARIANT_WORKQUEUE && B <= PKV_MAX_ROWS_IN_DECODE ? 1 : 0;
            c.splits = splits;
            c.tasks = tasks;
            c.grid = std::max<int64_t>(1, std::min<int64_t>(tasks, grid_cap));
            c.p_max = max_pages;
            c.kv_bytes = kv_bytes;
            const double us = choose_merge(&pol, c);
            if (!have || us < best_us) {
                best = c;
                best_us = us;
                have = true;
            }
        }
    }
    if (!have) return PKV_E_INVAL;
    rc = fill_plan(pr, lens, num_sms, best.variant, best.chunk, pol.ctas_per_sm, plan);
    if (rc != PKV_OK) return rc;
    plan->fuse_merge = best.fuse;
    plan->predicted_us = best_us;
    return PKV_OK;
}

extern "C" int pkv_plan_launches(const pkv_plan_t* plan) {
    if (!plan) return 0;
    const int merge = plan->fuse_merge ? 0 : 1;
    switch (plan->variant) {
        case PKV_VARIANT_SINGLE: return 1;
        case PKV_VARIANT_SPLIT: return 1 + merge;
        case PKV_VARIANT_WORKQUEUE: return (plan->list_in_decode ? 1 : 2) + merge;
        default: return 0;
    }
}
