// Host planner: workspace layout and the roofline-style cost-model policy.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs": the v2 abstract
// names a calibrated roofline-style policy whose cost-model constants are fixed on calibration traces and which
// routes each step to one execution path; the gist.science technical summary, "Calibrated Adaptive Policy", keys
// that choice on batch size B and the longest context N_max. Here the candidates are this library's own
// single-pass kernel, the rectangular split grid and the compact workqueue, each over a set of split sizes c
// (pages per split), and the model predicts a step's time as
//   launches * launch_us
//   + max(KV bytes / hbm_gbs, sum_i cost_i / W, max_i cost_i)        (decode; W = resident CTAs, cost_i =
//                                                                      task_us + bytes_i / cta_gbs per task)
//   + merge_us + 2 * state bytes / state_gbs                          (split and workqueue)
//   + build_us                                                         (workqueue)
// and keeps the cheapest candidate.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "pkv_internal.h"

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
    pol->launch_us = 2.5;
    pol->hbm_gbs = 5500.0;
    pol->cta_gbs = 40.0;
    pol->task_us = 1.5;
    pol->merge_us = 1.0;
    pol->build_us = 1.0;
    pol->state_gbs = 3000.0;
    pol->ctas_per_sm = 2;
    pol->max_splits = 256;
    pol->allow_variants = (1 << PKV_VARIANT_SINGLE) | (1 << PKV_VARIANT_SPLIT) | (1 << PKV_VARIANT_WORKQUEUE);
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

double predict_us(const pkv_policy* pol, const pkv_plan_t* plan, const int32_t* lens) {
    const pkv_problem& pr = plan->problem;
    const int B = pr.batch, Hkv = pr.num_kv_heads, G = plan->group;
    const int c = plan->chunk_pages;
    const double W = (double)std::max(1, plan->grid_ctas);
    const double per_tok = (double)kTokenHeadBytes;  // K + V bytes of one token for one KV head
    double sum_cost = 0.0, max_cost = 0.0;
    for (int b = 0; b < B; ++b) {
        const int64_t L = lens[b];
        const int64_t P = (L + kPageSize - 1) / kPageSize;
        const int64_t S = plan->variant == PKV_VARIANT_SINGLE ? 1 : (P + c - 1) / c;
        int64_t S_grid = S;
        if (plan->variant == PKV_VARIANT_SPLIT) S_grid = plan->num_splits;
        for (int64_t s = 0; s < S_grid; ++s) {
            int64_t t0 = s * c * kPageSize, t1 = std::min<int64_t>((s + 1) * (int64_t)c * kPageSize, L);
            if (plan->variant == PKV_VARIANT_SINGLE) t0 = 0, t1 = L;
            const double tok = t1 > t0 ? (double)(t1 - t0) : 0.0;
            const double cost = pol->task_us + tok * per_tok / (pol->cta_gbs * 1e3);
            sum_cost += cost * Hkv;
            max_cost = std::max(max_cost, cost);
        }
    }
    const double stream_us = plan->kv_bytes / (pol->hbm_gbs * 1e3);
    double t = pol->launch_us + std::max(stream_us, std::max(sum_cost / W, max_cost));
    if (plan->variant != PKV_VARIANT_SINGLE) {
        const double states = (double)plan->num_tasks * G;
        t += pol->launch_us + pol->merge_us + 2.0 * states * kStateBytes / (pol->state_gbs * 1e3);
    }
    if (plan->variant == PKV_VARIANT_WORKQUEUE) t += pol->launch_us + pol->build_us;
    return t;
}

}  // namespace

extern "C" int pkv_plan_fixed(const pkv_problem* pr, const int32_t* lens, int32_t num_sms, int32_t variant,
                              int32_t chunk_pages, int32_t ctas_per_sm, pkv_plan_t* plan) {
    int rc = fill_plan(pr, lens, num_sms, variant, chunk_pages, ctas_per_sm, plan);
    if (rc != PKV_OK) return rc;
    pkv_policy pol;
    pkv_policy_default(&pol);
    pol.ctas_per_sm = ctas_per_sm > 0 ? ctas_per_sm : pol.ctas_per_sm;
    plan->predicted_us = predict_us(&pol, plan, lens);
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
    if (pol.ctas_per_sm <= 0 || pol.max_splits <= 0 || pol.hbm_gbs <= 0 || pol.cta_gbs <= 0 ||
        pol.state_gbs <= 0)
        return PKV_E_INVAL;
    int64_t max_pages = 0;
    for (int b = 0; b < pr->batch; ++b) {
        if (lens[b] < 0) return PKV_E_INVAL;
        max_pages = std::max<int64_t>(max_pages, (lens[b] + kPageSize - 1) / kPageSize);
    }
    // candidate split sizes: powers of two and 1.5x powers of two, bounded so that S <= max_splits
    std::vector<int32_t> chunks;
    const int64_t cmin = std::max<int64_t>(1, (max_pages + pol.max_splits - 1) / pol.max_splits);
    for (int64_t c = 1; c <= std::max<int64_t>(1, max_pages); c *= 2) {
        if (c >= cmin) chunks.push_back((int32_t)c);
        const int64_t c3 = c + c / 2;
        if (c3 > c && c3 >= cmin && c3 <= max_pages) chunks.push_back((int32_t)c3);
    }
    if (chunks.empty()) chunks.push_back((int32_t)std::max<int64_t>(1, cmin));
    bool have = false;
    pkv_plan_t best{}, cand{};
    for (int v = PKV_VARIANT_SINGLE; v <= PKV_VARIANT_WORKQUEUE; ++v) {
        if (!(pol.allow_variants & (1 << v))) continue;
        const size_t n = v == PKV_VARIANT_SINGLE ? 1 : chunks.size();
        for (size_t i = 0; i < n; ++i) {
            if (fill_plan(pr, lens, num_sms, v, chunks[i], pol.ctas_per_sm, &cand) != PKV_OK) continue;
            cand.predicted_us = predict_us(&pol, &cand, lens);
            if (!have || cand.predicted_us < best.predicted_us) {
                best = cand;
                have = true;
            }
        }
    }
    if (!have) return PKV_E_INVAL;
    *plan = best;
    return PKV_OK;
}

extern "C" int pkv_plan_launches(const pkv_plan_t* plan) {
    if (!plan) return 0;
    const int merge = plan->fuse_merge ? 0 : 1;
    switch (plan->variant) {
        case PKV_VARIANT_SINGLE: return 1;
        case PKV_VARIANT_SPLIT: return 1 + merge;
        case PKV_VARIANT_WORKQUEUE: return 2 + merge;
        default: return 0;
    }
}
