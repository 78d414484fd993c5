// Persistent split-KV paged GQA decode kernel for sm_103a; optionally with the log-sum-exp merge of the split states
// fused in (run by the CTA whose task of a (row, KV head) finishes last).
//
// Computes, for every task (row b, KV head h, logical pages [page_begin, page_end)), the online-softmax state of
// the G = Hq/Hkv query heads that share KV head h ("PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs", v1/v2 abstracts: work mapped by KV-head group so the grouped query heads reuse each
// K/V tile; gist.science technical summary, "Methodologie" 1: native block-table execution ("Layout"), sequence
// splitting into partial online-softmax states combined exactly ("Sequentie Splitting"), row-local bounds with
// neutral states for empty splits ("Row-Local Bounds"), compact workqueue ("Compact Workqueue")).
//
// CTA layout (persistent over tasks; grid = one wave of resident CTAs):
//   warp NCW+2  scheduler: takes tasks (split / single: a static stride over the (b, h, s) task space; workqueue:
//               task blockIdx.x first, then an atomic queue head; a list the decode derives itself from seq_lens is
//               claimed split by split within a row (the KV heads of one split, which read the same pages, one after
//               the other), a list written by the worklist builder in its order, after waiting for the builder
//               grid), bulk-copies the G query rows of the task into a shared-memory
//               task slot (completion on their own barrier), fetches the row length and the task's first 32
//               block-table entries together and publishes them in the slot. With the merge fused it also publishes
//               merge tasks that the epilogue warp requests, and ends only after the epilogue has seen every task;
//   warp NCW+1  loader: per page, one elected lane issues four 3-D TMA tensor copies (K and V of KV head h, each as
//               two 64-column boxes of the page's 16 token rows, 128-byte swizzled) into a ring stage, counted in
//               bytes on the stage's mbarrier; block-table entries past the slot's 32 are read one chunk ahead. When
//               the CTA's first task is known before the CTA barrier (static plans, and a workqueue derived in the
//               decode) it reads that task's entries itself and issues its first page copies at once. A merge
//               task's partial states go through the same ring, 16 states (8 KB of acc) per stage, by bulk copies;
//   warps 0..NCW-1 consumers: page j of the CTA's page sequence (counted across tasks) lives in stage j % NS and
//               goes to warp j % NCW (NS % NCW == 0, so a stage always has the same consumer). The products are
//               taken transposed, so the 16 tokens (scores) and the head dimension (output) fill the 16-row side of
//               mma.sync m16n8k16 and the G query heads the 8-column side: S^T = K Q^T (8 MMAs per page for G <= 8),
//               masking of slots past the row length, online softmax in base 2 per head column, P^T rebuilt in the
//               B-operand layout with four shuffles, O^T += V^T P^T (8 MMAs). At the end of a task each warp hands
//               its (m, l, O) to the epilogue warp through a double-buffered shared-memory slot and moves on. In a
//               merge task a warp folds the states of its stages into a running (M, D, A) per query head instead.
//   warp NCW    epilogue: combines the NCW warps' partials of a task and writes the normalised output (single pass,
//               merge task) or the partial state (m, l, acc) of each query head. With the merge fused it then counts
//               the task in the (b, h) arrival counter; the last of the S_b tasks of (b, h) to arrive re-arms the
//               counter and asks the scheduler (a shared-memory mailbox) for a merge task of (b, h), which the
//               loader, the consumers and this warp then run like any task: all of the pair's states are in flight
//               at once through the ring. Nobody waits for another CTA.
// Every wait is bounded (global timer); on timeout the kernel sets PKV_STATUS_TIMEOUT in the workspace, the other
// warps see an abort flag, every warp that issued bulk copies waits (bounded) for them, and the CTA returns.
#include <cuda_fp16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kBoxBytes = kPageSize * 128;   // one TMA box: 16 token rows x 64 fp16 columns (128 B, swizzled)
constexpr int kStageBytes = 4 * kBoxBytes;   // K columns 0-63, K 64-127, V 0-63, V 64-127
constexpr int kCombRow = kHeadDim + 4;       // floats per partial output row (132: rows land 4 banks apart)
constexpr int kSlotEntries = 32;             // block-table entries the scheduler prefetches per task
constexpr int kMergeStates = kStageBytes / (kHeadDim * 4);  // partial states per ring stage in a merge task (16)
constexpr int kMailbox = 32;                 // merge requests the epilogue may post ahead of the scheduler
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Task kinds: the pages of a task, or the merge of the split states of one (row, KV head) pair.
constexpr int kKindPages = 0;
constexpr int kKindMerge = 1;

struct TaskSlot {
    int32_t b, h, s, task;                  // task: canonical index; the task's states are task * G + g
    int32_t page_begin, npages, seq_len, nsplit;  // nsplit: tasks of (b, h) (arrivals of the fused merge; 0 = none)
    int32_t kind, pad0, pad1, pad2;         // merge: task = the pair's first task, npages = state chunks
    int32_t ent[kSlotEntries];              // physical page of logical page page_begin + i (i < min(npages, 32))
};

// What the epilogue warp needs to know about a task (written by consumer warp 0; npages < 0 ends the CTA).
struct EpiHeader {
    int32_t b, h, s, task, nsplit, npages, kind, pad;
};

// A merge the epilogue warp asks the scheduler for: the pair (b, h) whose nsplit tasks from `first` on have all
// written their states.
struct MergeReq {
    int32_t b, h, first, nsplit;
};

template <int G, int NCW, int NS, int NTS>
struct Layout {
    static constexpr int kNT = (G + 7) / 8;  // 8-head column tiles of the MMAs
    static constexpr int kQRowsBytes = ((G * kRowBytes + 127) / 128) * 128;
    static constexpr int kCombFloats = NCW * G * kCombRow;  // one slot: every consumer warp's O rows
    static constexpr int off_stage = 0;  // 1024-byte aligned (128-byte swizzle atom)
    static constexpr int off_q = off_stage + NS * kStageBytes;
    static constexpr int off_comb = off_q + NTS * kQRowsBytes;
    static constexpr int off_comb_ml = off_comb + 2 * kCombFloats * 4;    // float2 (m, l) per slot/warp/head
    static constexpr int off_ehdr = off_comb_ml + 2 * NCW * G * 8;
    static constexpr int off_rows = off_ehdr + 2 * (int)sizeof(EpiHeader);  // in-decode list: off, S_b, L_b per row
    static constexpr int off_mreq = off_rows + 3 * PKV_MAX_ROWS_IN_DECODE * 4;  // merge-request mailbox
    static constexpr int off_slots = off_mreq + kMailbox * (int)sizeof(MergeReq);
    static constexpr int off_bars = ((off_slots + NTS * (int)sizeof(TaskSlot) + 15) / 16) * 16;
    static constexpr int nbars = 2 * NS + 3 * NTS + 4;
    static constexpr int off_flag = off_bars + nbars * 8;  // abort flag, requests posted, requests taken, verdicts
    static constexpr int used = off_flag + 16;
    static constexpr int total = used + 1024;  // slack to align the base to 1024 bytes
};

struct WaitCtx {
    volatile int* abort_flag;
    uint32_t* status;
};

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

// Warp-collective bounded wait on an mbarrier phase. Returns false if the wait gave up (abort or timeout).
// try_wait suspends the thread until the phase completes or a short hardware time slice ends; the abort flag and
// the global timer are consulted only every kPollEvery slices.
constexpr uint32_t kPollEvery = 256;

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtx& ctx) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (it % kPollEvery == 0) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            const bool stop = (*ctx.abort_flag != 0) || (now - t0 > kWaitLimitNs);
            if (__any_sync(0xffffffffu, stop)) {
                if ((threadIdx.x & 31) == 0 && *ctx.abort_flag == 0) {
                    *ctx.abort_flag = 1;
                    raise_status(ctx.status, PKV_STATUS_TIMEOUT);
                }
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain a warp's own copies before it returns).
__device__ __forceinline__ void warp_drain(uint64_t* bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t it = 1; !__all_sync(0xffffffffu, mbar_try_wait(bar, parity)); ++it) {
        if (it % kPollEvery == 0) {
            const uint64_t now = global_timer_ns();
            if (t0 == 0) t0 = now;
            if (__any_sync(0xffffffffu, now - t0 > kWaitLimitNs)) return;
        }
    }
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of token row `row` inside a 128-byte-swizzled box: the TMA
// stores chunk c of row r at position c ^ (r % 8) of the row's 128-byte line.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Physical page of logical page `lp` of row b (the appended token's page; read once per (row, KV head)).
__device__ __forceinline__ int32_t logical_page_phys(const DecodeParams& p, int b, int lp) {
    return __ldg(p.block_table + (size_t)b * p.max_pages + lp);
}

__device__ __forceinline__ void store_half4(__half* dst, float4 v, float scale) {
    uint2 pk;
    pk.x = pack_half2(v.x * scale, v.y * scale);
    pk.y = pack_half2(v.z * scale, v.w * scale);
    *reinterpret_cast<uint2*>(dst) = pk;
}

// Task t of a static plan (split grid or single pass): its row, KV head, split and logical page range. Split tasks
// are in (b, h, s) order, splits fastest: the CTAs that run at the same time read different page ranges of one head
// (measured faster on GB300 than eight CTAs reading the eight heads of the same pages).
struct StaticTask {
    int b, h, s, pb, pe;
};

__device__ __forceinline__ StaticTask static_task(const DecodeParams& p, int t) {
    StaticTask k;
    if (p.variant == PKV_VARIANT_SPLIT) {
        const int S = p.num_splits;
        const int per_row = p.Hkv * S;
        k.b = t / per_row;
        const int r = t - k.b * per_row;
        k.h = r / S;
        k.s = r - k.h * S;
        k.pb = k.s * p.chunk_pages;
        k.pe = k.pb + p.chunk_pages;
    } else {
        k.b = t / p.Hkv;
        k.h = t - k.b * p.Hkv;
        k.s = 0;
        k.pb = 0;
        k.pe = p.max_pages;
    }
    return k;
}

// The CTA's first task (claim blockIdx.x) when it can be known before the CTA barrier: for a static plan from the
// task index, for a workqueue whose compact list the decode derives itself from seq_lens (a warp-collective scan
// of Hkv * S_b over the rows, the arithmetic of the list derivation below). Plans that run a list written by the
// worklist builder are launched after it and read nothing before griddepcontrol.wait: no first task here. Returns
// false when there is no such task.
__device__ __forceinline__ bool first_task(const DecodeParams& p, int lane, StaticTask& k, int& len) {
    const int t = blockIdx.x;
    if (p.variant != PKV_VARIANT_WORKQUEUE) {
        if (t >= p.num_tasks) return false;
        k = static_task(p, t);
        if (!(k.b >= 0 && k.b < p.B && k.h >= 0 && k.h < p.Hkv && k.pb >= 0 && k.pe >= k.pb)) return false;
        len = p.seq_lens[k.b];
        return true;
    }
    if (!p.list_in_decode || p.B > PKV_MAX_ROWS_IN_DECODE) return false;
    int run = 0, found = -1, fl = 0, foff = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int l = b < p.B ? p.seq_lens[b] : 0;
        if (l < 0 || l > p.max_pages * kPageSize) l = 0;
        const int S = ((l + kPageSize - 1) / kPageSize + p.chunk_pages - 1) / p.chunk_pages;
        const int x = b < p.B ? p.Hkv * S : 0;
        int incl = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int off = run + incl - x;
        const unsigned hit = __ballot_sync(0xffffffffu, x > 0 && off <= t && t < off + x);
        if (found < 0 && hit) {
            const int src = __ffs(hit) - 1;
            found = b0 + src;
            fl = __shfl_sync(0xffffffffu, l, src);
            foff = __shfl_sync(0xffffffffu, off, src);
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found < 0 || t >= min(run, p.task_capacity)) return false;
    const int r = t - foff;  // claim order within the row: split by split, the KV heads of a split together
    k.b = found;
    k.s = r / p.Hkv;
    k.h = r - k.s * p.Hkv;
    k.pb = k.s * p.chunk_pages;
    k.pe = min(k.pb + p.chunk_pages, (fl + kPageSize - 1) / kPageSize);
    len = fl;
    return true;
}

// Pages of a task that lie within its row: the row length is validated (an out-of-range length counts as 0).
__device__ __forceinline__ int task_pages(const DecodeParams& p, int len, int pb, int pe) {
    if (len < 0 || len > p.max_pages * kPageSize) len = 0;
    return max(0, min(pe, (len + kPageSize - 1) / kPageSize) - pb);
}

// Loader side of a merge task: the pair's S_b * G states (written by other CTAs before their arrivals, which the
// epilogue warp's counter acquired) go through the ring by bulk copies, kMergeStates states (8 KB of acc) per stage,
// read through the async proxy. Returns the new ring position, or -1 if a wait gave up.
template <int G, int NS>
__device__ __noinline__ int load_merge_chunks(const DecodeParams& p, uint8_t* stages, uint64_t* full, uint64_t* empty,
                                              int seq, int first, int nsplit, int nchunks, WaitCtx ctx, int lane) {
    fence_proxy_async_global();
    const int nstates = nsplit * G;
    const float* src = p.acc + (size_t)first * G * kHeadDim;
    for (int c = 0; c < nchunks; ++c) {
        const int st = seq % NS;
        if (!warp_wait(&empty[st], ((seq / NS) & 1) ^ 1, ctx)) return -1;
        if (lane == 0) {
            const uint32_t bytes = min(kMergeStates, nstates - c * kMergeStates) * kHeadDim * 4;
            mbar_arrive_expect_tx(&full[st], bytes);
            bulk_g2s(stages + st * kStageBytes, src + (size_t)c * kMergeStates * kHeadDim, bytes, &full[st]);
        }
        __syncwarp();
        ++seq;
    }
    return seq;
}

// Consumer side of a merge task: warp w folds the states of its stages (chunk i of the task is in stage (seq + i) %
// NS and belongs to warp (seq + i) % NCW) into a running (M, D, A) per query head (M in base 2; lane k owns dims
// 4k..4k+3), then hands (M, D) and A to the epilogue warp through the partial-output slot `co` / `cml` once `eempty`
// allows. The (m, l) pairs come from L2 (those of the warp's first kMlAhead chunks requested at once). Returns
// false if a wait gave up.
template <int G, int NS, int NCW>
__device__ __noinline__ bool fold_merge_chunks(const DecodeParams& p, const uint8_t* stages, uint64_t* full,
                                               uint64_t* empty, uint64_t* eempty_e, uint32_t eparity, int seq, int w,
                                               int nchunks, int first, int nsplit, float* co, float2* cml, WaitCtx ctx,
                                               int lane) {
    const int nstates = nsplit * G;
    const float2* mlp = reinterpret_cast<const float2*>(p.ml) + (size_t)first * G;
    const int i0 = (w - seq % NCW + NCW) % NCW;
    constexpr int kMlAhead = 8;
    float2 mlv[kMlAhead];
#pragma unroll
    for (int u = 0; u < kMlAhead; ++u) {
        const int c0 = (i0 + u * NCW) * kMergeStates;
        mlv[u] = c0 + lane < nstates && lane < kMergeStates ? __ldcg(mlp + c0 + lane) : make_float2(-INFINITY, 0.f);
    }
    float Mg[G], Dg[G];
    float4 Ag[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        Mg[g] = -INFINITY;
        Dg[g] = 0.f;
        Ag[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = i0, u = 0; i < nchunks; i += NCW, ++u) {
        const int j = seq + i;
        const int st = j % NS;
        const int c0 = i * kMergeStates;
        const int cnt = min(kMergeStates, nstates - c0);
        float2 ml = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int v = 0; v < kMlAhead; ++v)
            if (v == u) ml = mlv[v];
        if (u >= kMlAhead && lane < cnt) ml = __ldcg(mlp + c0 + lane);
        if (!warp_wait(&full[st], (j / NS) & 1, ctx)) return false;
        const float* chunk = reinterpret_cast<const float*>(stages + st * kStageBytes);
#pragma unroll
        for (int jj = 0; jj < kMergeStates / G; ++jj) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int li = jj * G + g;
                const float m2 = __shfl_sync(0xffffffffu, ml.x, li) * kLog2e;
                const float l = __shfl_sync(0xffffffffu, ml.y, li);
                if (li < cnt && l > 0.f) {
                    const float4 v = *reinterpret_cast<const float4*>(chunk + li * kHeadDim + lane * 4);
                    const float mn = fmaxf(Mg[g], m2);
                    const float fo = fast_exp2(Mg[g] - mn), fn = fast_exp2(m2 - mn);
                    Dg[g] = Dg[g] * fo + fn * l;
                    Ag[g].x = Ag[g].x * fo + fn * v.x;
                    Ag[g].y = Ag[g].y * fo + fn * v.y;
                    Ag[g].z = Ag[g].z * fo + fn * v.z;
                    Ag[g].w = Ag[g].w * fo + fn * v.w;
                    Mg[g] = mn;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (!warp_wait(eempty_e, eparity, ctx)) return false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        *reinterpret_cast<float4*>(co + g * kCombRow + lane * 4) = Ag[g];
        if (lane == 0) cml[g] = make_float2(Mg[g], Dg[g]);
    }
    return true;
}

// Resident CTAs per SM the kernel is compiled for: two up to G = 8; one for G = 16, whose query rows and
// partial-output slots do not leave room for a second CTA's shared memory.
constexpr int ctas_per_sm(int group) { return group >= 16 ? 1 : kDecodeCtasPerSm; }

template <int G, int NCW, int NS, int NTS>
__global__ void __launch_bounds__((NCW + 3) * 32, ctas_per_sm(G)) decode_kernel(const __grid_constant__ DecodeParams p) {
    static_assert(NS % NCW == 0, "each ring stage must map to one consumer warp");
    using L = Layout<G, NCW, NS, NTS>;
    constexpr int kNT = L::kNT;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::off_bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + NS;
    uint64_t* tmeta = bars + 2 * NS;  // task slot published (row, pages, block-table entries)
    uint64_t* tq = tmeta + NTS;       // the slot's query rows have landed
    uint64_t* tempty = tq + NTS;      // the slot has been read by the loader and every consumer
    uint64_t* efull = tempty + NTS;   // [2] every consumer warp has written its partial of the task into the slot
    uint64_t* eempty = efull + 2;     // [2] the epilogue warp has read the slot
    TaskSlot* slots = reinterpret_cast<TaskSlot*>(smem + L::off_slots);
    EpiHeader* ehdr = reinterpret_cast<EpiHeader*>(smem + L::off_ehdr);
    float* comb_o = reinterpret_cast<float*>(smem + L::off_comb);
    float2* comb_ml = reinterpret_cast<float2*>(smem + L::off_comb_ml);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_flag);
    volatile int* posted = abort_flag + 1;    // merge requests the epilogue has posted
    volatile int* taken = abort_flag + 2;     // merge requests the scheduler has published as tasks
    volatile int* verdicts = abort_flag + 3;  // page tasks the epilogue has finished
    MergeReq* mreq = reinterpret_cast<MergeReq*>(smem + L::off_mreq);
    const WaitCtx ctx{abort_flag, &p.hdr->status};
    // the merge of a pair runs as a task of the CTA whose task of the pair arrived last
    const bool fused = p.fuse_merge != 0 && p.variant != PKV_VARIANT_SINGLE;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NTS; ++i) {
            mbar_init(&tmeta[i], 1);
            mbar_init(&tempty[i], NCW + 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&efull[i], NCW);
            mbar_init(&eempty[i], 1);
        }
        *abort_flag = 0;
        *posted = 0;
        *taken = 0;
        *verdicts = 0;
        mbar_fence_init();
    }
    // The loader and the scheduler both work out the CTA's first task before the CTA barrier (first_task): the
    // scheduler's lane 0, which owns the query barriers, copies its query rows into slot 0 at once, and both read
    // its row length and block-table entries, so the loader's first page copies wait neither for the barrier set-up
    // nor for the task slot.
    int pre_np = 0, pre_h = 0, pre_ent = -1, pre_len = 0;
    bool pre_ok = false;
    if (warp == NCW + 1 || warp == NCW + 2) {
        StaticTask k;
        int len = 0;
        if (p.inputs_after_wait) grid_dependency_wait();  // the kernel before may still be writing the inputs
        pre_ok = first_task(p, lane, k, len);
        if (warp == NCW + 2 && lane == 0) {
            for (int i = 0; i < NTS; ++i) mbar_init(&tq[i], 1);
            mbar_fence_init();
            if (pre_ok && !p.overlap_prev) {  // overlapping the kernel before: q may still be in the making
                mbar_arrive_expect_tx(&tq[0], G * kRowBytes);
                bulk_g2s(smem + L::off_q,
                         static_cast<const __half*>(p.q) + ((size_t)k.b * p.Hq + (size_t)k.h * G) * kHeadDim,
                         G * kRowBytes, &tq[0]);
            }
        }
        if (pre_ok) {
            const int nent = max(0, min(min(k.pe, p.max_pages) - k.pb, kSlotEntries));
            pre_ent = lane < nent ? p.block_table[(size_t)k.b * p.max_pages + k.pb + lane] : -1;
            pre_len = len;
            pre_np = min(task_pages(p, pre_len, k.pb, k.pe), nent);
            pre_h = k.h;
        }
    }
    __syncthreads();
    // A separate merge grid launched after this one waits for its completion before reading anything; it may be
    // scheduled now and sit resident beside this grid.
    grid_launch_dependents();

    const int Hq = p.Hq, Hkv = p.Hkv;

    if (warp == NCW + 2) {
        // ------------------------------------------------------------------ scheduler
        // Everything this grid reads from global memory is read after this point (the other warps only follow the
        // slots published below), so the grid may start while the worklist builder is still running.
        grid_dependency_wait();
        const int variant = p.variant;
        const bool wq = variant == PKV_VARIANT_WORKQUEUE;
        const bool in_decode = wq && p.list_in_decode;
        int* row_off_s = reinterpret_cast<int*>(smem + L::off_rows);
        int* row_S_s = row_off_s + PKV_MAX_ROWS_IN_DECODE;
        int* row_L_s = row_S_s + PKV_MAX_ROWS_IN_DECODE;
        int count = p.num_tasks;
        if (in_decode) {
            // The compact list of the step, derived here: S_b = ceil(ceil(L_b / page_size) / c) and the exclusive
            // scan of Hkv * S_b over the rows (the builder's arithmetic, "Compact Workqueue"). Task t of the list
            // belongs to the last row b with off_b <= t.
            int run = 0;
            for (int b0 = 0; b0 < p.B; b0 += 32) {
                const int b = b0 + lane;
                int len = b < p.B ? p.seq_lens[b] : 0;
                if (len < 0 || len > p.max_pages * kPageSize) {
                    if (blockIdx.x == 0) raise_status(ctx.status, PKV_STATUS_BAD_LEN);
                    len = 0;
                }
                const int S = ((len + kPageSize - 1) / kPageSize + p.chunk_pages - 1) / p.chunk_pages;
                const int x = b < p.B ? Hkv * S : 0;
                int incl = x;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (b < p.B) {
                    row_off_s[b] = run + incl - x;
                    row_S_s[b] = S;
                    row_L_s[b] = len;
                    if (blockIdx.x == 0) {  // published for the separate merge kernel (and for inspection)
                        p.row_off[b] = run + incl - x;
                        p.row_splits[b] = S;
                    }
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            __syncwarp();
            count = min(run, p.task_capacity);
            if (blockIdx.x == 0 && lane == 0) {
                p.hdr->task_count = count;
                if (run > p.task_capacity) raise_status(ctx.status, PKV_STATUS_TASKS);
            }
        } else if (wq) {
            count = min(*reinterpret_cast<volatile int32_t*>(&p.hdr->task_count), p.task_capacity);
        }
        const __half* q = static_cast<const __half*>(p.q);
        int tseq = 0;      // slots published
        int k = 0;         // page tasks claimed
        int regular = 0;   // page tasks published
        bool more = true;  // page tasks may remain
        uint64_t idle_t0 = 0;
        uint32_t idle_it = 0;
        for (;;) {
            // Next slot: a merge the epilogue asked for, else the CTA's next page task; with the merge fused the
            // end comes only after the epilogue has finished every page task (any of them may still ask for a
            // merge). The posted count is read after the verdicts, so a request posted before the last verdict
            // is always seen.
            int kind, t = 0;
            bool first = false;  // the CTA's first task (task blockIdx.x), worked out before the CTA barrier
            // lane 0 reads the mailbox counters (they change under the warp) and the warp follows its decision
            int pend = 0, idle = 0;  // a request is pending; (fused, no page task left) the epilogue is still busy
            if (lane == 0 && fused) {
                if (*posted > *taken) {
                    pend = 1;
                } else if (!more) {
                    const int v = *verdicts;
                    __threadfence_block();
                    pend = *posted > *taken;
                    idle = !pend && v < regular;
                }
            }
            pend = __shfl_sync(0xffffffffu, pend, 0);
            idle = __shfl_sync(0xffffffffu, idle, 0);
            if (pend) {
                kind = kKindMerge;
            } else if (more) {
                if (wq && k > 0) {  // the first wave is static: CTA i starts with task i, no atomic on its critical
                    int c = 0;      // path
                    if (lane == 0) c = static_cast<int>(gridDim.x + atomicAdd(&p.hdr->queue_head, 1u));
                    t = __shfl_sync(0xffffffffu, c, 0);
                } else {
                    t = blockIdx.x + k * gridDim.x;
                }
                first = k == 0;
                ++k;
                if (t >= count) {
                    more = false;
                    continue;
                }
                kind = kKindPages;
            } else if (idle) {  // bounded wait for the epilogue
                if (++idle_it % kPollEvery == 0) {
                    const uint64_t now = global_timer_ns();
                    if (idle_t0 == 0) idle_t0 = now;
                    const bool stop = (*abort_flag != 0) || (now - idle_t0 > kWaitLimitNs);
                    if (__any_sync(0xffffffffu, stop)) {
                        if (lane == 0 && *abort_flag == 0) {
                            *abort_flag = 1;
                            raise_status(ctx.status, PKV_STATUS_TIMEOUT);
                        }
                        break;
                    }
                }
                __nanosleep(64);
                continue;
            } else {
                kind = -1;
            }
            const int ts = tseq % NTS;
            if (!warp_wait(&tempty[ts], ((tseq / NTS) & 1) ^ 1, ctx)) break;
            TaskSlot* sl = &slots[ts];
            if (kind < 0) {
                if (lane == 0) {
                    sl->npages = -1;
                    mbar_arrive(&tmeta[ts]);
                }
                break;
            }
            if (kind == kKindMerge) {
                if (lane == 0) {
                    __threadfence_block();  // the entry was written before the posted count
                    const MergeReq r = mreq[*taken % kMailbox];
                    *taken = *taken + 1;
                    sl->b = r.b;
                    sl->h = r.h;
                    sl->s = 0;
                    sl->task = r.first;
                    sl->page_begin = 0;
                    sl->npages = (r.nsplit * G + kMergeStates - 1) / kMergeStates;
                    sl->seq_len = 0;
                    sl->nsplit = r.nsplit;
                    sl->kind = kKindMerge;
                    mbar_arrive(&tq[ts]);  // no query rows
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmeta[ts]);
                __syncwarp();
                ++tseq;
                continue;
            }
            int b, h, s, pb, pe, task, nsplit = 1;
            if (in_decode) {
                int lo = 0, hi = p.B - 1;  // rows without tasks share their successor's offset and are skipped
                while (lo < hi) {
                    const int mid = (lo + hi + 1) >> 1;
                    if (row_off_s[mid] <= t)
                        lo = mid;
                    else
                        hi = mid - 1;
                }
                b = lo;
                const int Sb = max(row_S_s[b], 1);
                // Claimed split by split (the Hkv tasks of one split read the same pages at about the same time,
                // measured faster on GB300 than claiming a head's splits in turn); the list and its states stay in
                // (b, h, s) order.
                const int r = t - row_off_s[b];
                s = r / Hkv;
                h = r - s * Hkv;
                pb = s * p.chunk_pages;
                pe = min(pb + p.chunk_pages, (row_L_s[b] + kPageSize - 1) / kPageSize);
                task = row_off_s[b] + h * Sb + s;
            } else if (wq) {
                const pkv_task tk = p.tasks[t];
                b = tk.row;
                h = tk.head_split >> 16;
                s = tk.head_split & 0xffff;
                pb = tk.page_begin;
                pe = tk.page_end;
                task = t;
            } else {
                const StaticTask st = static_task(p, t);
                b = st.b;
                h = st.h;
                s = st.s;
                pb = st.pb;
                pe = st.pe;
                task = t;
                if (variant == PKV_VARIANT_SPLIT) nsplit = p.num_splits;
            }
            const bool bad = b < 0 || b >= p.B || h < 0 || h >= Hkv || s < 0 || pb < 0 || pe < pb;
            if (bad) {  // a task that is not from this plan: it writes a neutral state and takes no part in a merge
                b = 0;
                h = 0;
                pb = pe = 0;
            }
            // the row length and the task's first block-table entries, fetched together (for the CTA's first static
            // task they were read before the CTA barrier)
            const bool prefetched = first && pre_ok && !bad;
            const bool q_copied = prefetched && !p.overlap_prev;  // the first task's query rows are in slot 0
            const int nent = max(0, min(min(pe, p.max_pages) - pb, kSlotEntries));
            const int ent = prefetched ? pre_ent : (lane < nent ? p.block_table[(size_t)b * p.max_pages + pb + lane] : -1);
            int len = prefetched ? pre_len : p.seq_lens[b];
            const int row_splits = in_decode ? row_S_s[b] : (wq ? p.row_splits[b] : 0);
            if (len < 0 || len > p.max_pages * kPageSize) {
                if (lane == 0) raise_status(ctx.status, PKV_STATUS_BAD_LEN);
                len = 0;
            }
            const int np_row = (len + kPageSize - 1) / kPageSize;
            const int np = task_pages(p, len, pb, pe);
            // A row with pages past its last task (its length grew after the plan was made) is flagged; its tasks
            // still take part in the merge, so the arrival counters stay consistent.
            bool grown, foreign = bad;
            if (wq) {  // the builder's split count of the row: the number of tasks of (b, h) in the list
                nsplit = row_splits;
                // the states of (b, h) are tasks [t - s, t - s + S_b) of the list
                foreign = foreign || s >= row_splits || task - s < 0 || task - s + row_splits > count;
                grown = s == row_splits - 1 && np_row > pe;
            } else {
                grown = np_row > pe && (variant == PKV_VARIANT_SINGLE || s == p.num_splits - 1);
            }
            if ((grown || foreign) && lane == 0) raise_status(ctx.status, PKV_STATUS_TASKS);
            if (foreign) nsplit = 0;
            sl->ent[lane] = ent;
            if (lane == 0) {
                sl->b = b;
                sl->h = h;
                sl->s = s;
                sl->task = task;
                sl->page_begin = pb;
                sl->npages = np;
                sl->seq_len = len;
                sl->nsplit = nsplit;
                sl->kind = kKindPages;
            }
            __syncwarp();
            // Published before the query copy is issued (that copy may queue behind the loader's page copies). The
            // G query rows of this KV head are contiguous in q; the consumers wait for them on their own barrier.
            // The CTA's first static task had its rows copied before the CTA barrier.
            if (lane == 0) {
                mbar_arrive(&tmeta[ts]);
                if (!q_copied) {
                    if (!bad) {
                        mbar_arrive_expect_tx(&tq[ts], G * kRowBytes);
                        bulk_g2s(smem + L::off_q + ts * L::kQRowsBytes,
                                 q + ((size_t)b * Hq + (size_t)h * G) * kHeadDim, G * kRowBytes, &tq[ts]);
                    } else {
                        mbar_arrive(&tq[ts]);
                    }
                }
            }
            __syncwarp();
            ++tseq;
            ++regular;
        }
        // Before the warp leaves, every query copy it issued has landed (only after an abort can one be pending),
        // including the first task's copy when the warp stopped before publishing its slot.
        if (tseq == 0 && pre_ok && !p.overlap_prev) warp_drain(&tq[0], 0);
        for (int j = max(0, tseq - NTS); j < tseq; ++j) warp_drain(&tq[j % NTS], (j / NTS) & 1);
        // Workqueue with the merge fused: rows without tokens have no task, so their (zero) output is written here.
        if (wq && p.fuse_merge) {
            for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
                if (p.seq_lens[b] == 0) {
                    uint4* o = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + (size_t)b * Hq * kHeadDim);
                    for (int i = lane; i < Hq * kHeadDim / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        // Workqueue: the last CTA to finish claiming re-arms the queue head, so the same list can be run again.
        if (wq && lane == 0) {
            __threadfence();
            if (atomicAdd(&p.hdr->ctas_done, 1u) == gridDim.x - 1) {
                atomicExch(&p.hdr->queue_head, 0u);
                atomicExch(&p.hdr->ctas_done, 0u);
            }
        }
    } else if (warp == NCW + 1) {
        // ------------------------------------------------------------------ loader
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_k);
            prefetch_tensormap(&p.tmap_v);
        }
        const uint64_t pol = policy_evict_first();
        int seq = 0;
        bool stop = false;
        // the first pages of the CTA's first task, from the entries read before the CTA barrier (its ring stages are
        // fresh, so nothing is waited for)
        const int pre = min(pre_np, NS);
        for (int i = 0; i < pre; ++i) {
            const int phys = __shfl_sync(0xffffffffu, pre_ent, i);
            const bool ok = phys >= 0 && phys < p.num_pages;
            if (lane == 0) {
                if (ok) {
                    uint8_t* dst = smem + L::off_stage + i * kStageBytes;
                    const int z = phys * kPageSize;
                    mbar_arrive_expect_tx(&full[i], kStageBytes);
                    tma_load_3d(dst, &p.tmap_k, 0, pre_h, z, &full[i], pol);
                    tma_load_3d(dst + kBoxBytes, &p.tmap_k, 64, pre_h, z, &full[i], pol);
                    tma_load_3d(dst + 2 * kBoxBytes, &p.tmap_v, 0, pre_h, z, &full[i], pol);
                    tma_load_3d(dst + 3 * kBoxBytes, &p.tmap_v, 64, pre_h, z, &full[i], pol);
                } else {
                    raise_status(ctx.status, PKV_STATUS_BAD_PAGE);
                    mbar_arrive(&full[i]);
                }
            }
        }
        seq = pre;
        for (int tseq = 0; !stop; ++tseq) {
            const int ts = tseq % NTS;
            if (!warp_wait(&tmeta[ts], (tseq / NTS) & 1, ctx)) break;
            const int np = slots[ts].npages;
            const int b = slots[ts].b, h = slots[ts].h, pb = slots[ts].page_begin;
            const int kind = slots[ts].kind, mfirst = slots[ts].task, mnsplit = slots[ts].nsplit;
            int ent = slots[ts].ent[lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ts]);
            if (np < 0) break;
            if (kind == kKindMerge) {
                seq = load_merge_chunks<G, NS>(p, smem + L::off_stage, full, empty, seq, mfirst, mnsplit, np, ctx,
                                               lane);
                if (seq < 0) break;
                continue;
            }
            const int skip = tseq == 0 ? pre : 0;  // pages issued before the slot was read
            if (np < skip || (skip > 0 && h != pre_h)) {  // the slot disagrees with the prefetch: never expected
                if (lane == 0) {
                    raise_status(ctx.status, PKV_STATUS_TASKS);
                    *abort_flag = 1;
                }
                break;
            }
            const int32_t* bt = p.block_table + (size_t)b * p.max_pages + pb;
            int ent_next = kSlotEntries + lane < np ? bt[kSlotEntries + lane] : 0;
            for (int c0 = 0; c0 < np; c0 += 32) {
                if (c0 > 0) {
                    ent = ent_next;
                    if (c0 + 32 + lane < np) ent_next = bt[c0 + 32 + lane];
                }
                const int n = min(32, np - c0);
                for (int i = c0 == 0 ? skip : 0; i < n; ++i) {
                    const int phys = __shfl_sync(0xffffffffu, ent, i);
                    const bool ok = phys >= 0 && phys < p.num_pages;
                    if (!ok && lane == 0) raise_status(ctx.status, PKV_STATUS_BAD_PAGE);
                    const int st = seq % NS;
                    if (!warp_wait(&empty[st], ((seq / NS) & 1) ^ 1, ctx)) {
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        if (ok) {
                            uint8_t* dst = smem + L::off_stage + st * kStageBytes;
                            const int z = phys * kPageSize;
                            mbar_arrive_expect_tx(&full[st], kStageBytes);
                            tma_load_3d(dst, &p.tmap_k, 0, h, z, &full[st], pol);
                            tma_load_3d(dst + kBoxBytes, &p.tmap_k, 64, h, z, &full[st], pol);
                            tma_load_3d(dst + 2 * kBoxBytes, &p.tmap_v, 0, h, z, &full[st], pol);
                            tma_load_3d(dst + 3 * kBoxBytes, &p.tmap_v, 64, h, z, &full[st], pol);
                        } else {
                            mbar_arrive(&full[st]);
                        }
                    }
                    __syncwarp();
                    ++seq;
                }
                if (stop) break;
            }
        }
        // Wait for every copy this warp issued before the CTA may exit.
        for (int j = max(0, seq - NS); j < seq; ++j) warp_drain(&full[j % NS], (j / NS) & 1);
    } else if (warp == NCW) {
        // ------------------------------------------------------------------ epilogue
        for (int tseq = 0;; ++tseq) {
            const int e = tseq & 1;
            if (!warp_wait(&efull[e], (tseq >> 1) & 1, ctx)) break;
            const EpiHeader hd = ehdr[e];
            if (hd.npages < 0) break;
            const bool merge = hd.kind == kKindMerge;
            const float* co = comb_o + e * L::kCombFloats;
            const float2* cml = comb_ml + e * NCW * G;
            for (int g = 0; g < G; ++g) {
                float M = -INFINITY;
#pragma unroll
                for (int wi = 0; wi < NCW; ++wi) M = fmaxf(M, cml[wi * G + g].x);
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                float lsum = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int wi = 0; wi < NCW; ++wi) {
                        const float2 ml = cml[wi * G + g];
                        const float f = fast_exp2(ml.x - M);
                        lsum += f * ml.y;
                        const float4 v = *reinterpret_cast<const float4*>(co + (wi * G + g) * kCombRow + lane * 4);
                        a.x += f * v.x;
                        a.y += f * v.y;
                        a.z += f * v.z;
                        a.w += f * v.w;
                    }
                }
                if (p.variant == PKV_VARIANT_SINGLE || merge) {  // out = acc / l of the whole row
                    store_half4(static_cast<__half*>(p.out) + ((size_t)hd.b * Hq + hd.h * G + g) * kHeadDim + lane * 4,
                                a, lsum > 0.f ? 1.f / lsum : 0.f);
                } else {
                    const size_t state = (size_t)hd.task * G + g;
                    if (lane == 0)
                        reinterpret_cast<float2*>(p.ml)[state] =
                            make_float2(M == -INFINITY ? -INFINITY : M * kLn2, lsum);
                    reinterpret_cast<float4*>(p.acc + state * kHeadDim)[lane] = a;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&eempty[e]);  // the consumers may refill the slot
            if (fused && !merge) {
                // count the task in (b, h); the last arriver asks for the merge of the pair's S_b states
                fence_acq_rel_gpu();  // this lane's state stores are performed before the arrival
                __syncwarp();
                if (lane == 0) {
                    uint32_t* cnt = p.counters + (size_t)hd.b * Hkv + hd.h;
                    bool last = false;
                    if (hd.nsplit > 0) {
                        const uint32_t old = atomicAdd(cnt, 1u);
                        last = old + 1u == (uint32_t)hd.nsplit;
                        if (last) {
                            fence_acq_rel_gpu();  // the other tasks' states, published before their arrivals
                            const int n = *posted;
                            if (n - *taken >= kMailbox) {  // never expected: requests are taken one per slot
                                raise_status(ctx.status, PKV_STATUS_TASKS);
                                *abort_flag = 1;
                            } else {
                                MergeReq r;
                                r.b = hd.b;
                                r.h = hd.h;
                                r.first = hd.task - hd.s;
                                r.nsplit = hd.nsplit;
                                mreq[n % kMailbox] = r;
                                __threadfence_block();
                                *posted = n + 1;
                            }
                        }
                    }
                    __threadfence_block();  // a request is posted before the verdict that lets the scheduler end
                    *verdicts = *verdicts + 1;
                    if (last) atomicExch(cnt, 0u);  // re-armed for the next step (off the merge's critical path)
                }
                __syncwarp();
            }
        }
    } else {
        // ------------------------------------------------------------------ consumers
        const int w = warp;
        const int g8 = lane >> 2;  // groupID: token row of S^T / dim row of O^T; head column of the B operand
        const int t4 = lane & 3;   // thread in group: head columns 2*t4, 2*t4 + 1 of S^T and O^T
        const int mi = lane >> 3, mr = lane & 7;
        // ldmatrix row addresses. K as the A operand (rows = tokens): matrix mi holds tokens (mi & 1) * 8 + mr at
        // 16-byte chunk parity mi >> 1. V^T as the A operand via .trans (rows = dims): matrix mi holds tokens
        // (mi >> 1) * 8 + mr at chunk parity mi & 1.
        const int k_row = ((mi & 1) << 3) + mr, k_par = mi >> 1;
        const int v_row = ((mi >> 1) << 3) + mr, v_par = mi & 1;
        // P^T in the B-operand layout: lane (g, t) needs P[token 2t (+1, +8, +9)][head g], which lanes
        // (2t) * 4 + g / 2 and (2t + 1) * 4 + g / 2 hold in the half g % 2 of their packed pairs.
        const int src_a = (2 * t4) * 4 + (g8 >> 1), src_b = (2 * t4 + 1) * 4 + (g8 >> 1);
        const uint32_t sel = (g8 & 1) ? 0x7632u : 0x5410u;
        const uint32_t stage0 = smem_addr(smem + L::off_stage);
        const float sl2 = p.scale_log2;
        int seq = 0;
        for (int tseq = 0;; ++tseq) {
            const int ts = tseq % NTS;
            const int e = tseq & 1;
            if (!warp_wait(&tmeta[ts], (tseq / NTS) & 1, ctx)) break;
            const int npages = slots[ts].npages;
            if (npages < 0) {  // no more tasks: tell the epilogue warp
                if (!warp_wait(&eempty[e], ((tseq >> 1) & 1) ^ 1, ctx)) break;
                if (w == 0 && lane == 0) ehdr[e].npages = -1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&efull[e]);
                break;
            }
            const int sb = slots[ts].b, sh = slots[ts].h, ss = slots[ts].s, stask = slots[ts].task;
            const int spb = slots[ts].page_begin, slen = slots[ts].seq_len, snsplit = slots[ts].nsplit;
            if (!warp_wait(&tq[ts], (tseq / NTS) & 1, ctx)) break;
            if (slots[ts].kind == kKindMerge) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[ts]);
                // Merge task: the fold of this warp's stages and its hand-off to the epilogue warp.
                if (!fold_merge_chunks<G, NS, NCW>(p, smem + L::off_stage, full, empty, &eempty[e],
                                                   ((tseq >> 1) & 1) ^ 1, seq, w, npages, stask, snsplit,
                                                   comb_o + e * L::kCombFloats + w * G * kCombRow,
                                                   comb_ml + e * NCW * G + w * G, ctx, lane))
                    break;
                seq += npages;
                if (w == 0 && lane == 0) {
                    EpiHeader hd;
                    hd.b = sb;
                    hd.h = sh;
                    hd.s = 0;
                    hd.task = stask;
                    hd.nsplit = snsplit;
                    hd.npages = npages;
                    hd.kind = kKindMerge;
                    hd.pad = 0;
                    ehdr[e] = hd;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&efull[e]);
                continue;
            }
            // Q^T as the B operand: b0 = Q[head][16ks + 2t, +1], b1 = Q[head][16ks + 2t + 8, +9], head = 8nt + g
            uint32_t qb[8][kNT][2];
            {
                const uint8_t* qs = smem + L::off_q + ts * L::kQRowsBytes;
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    const int head = nt * 8 + g8;
                    const bool on = head < G && npages > 0;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int col = (ks * 16 + 2 * t4) * 2;
                        qb[ks][nt][0] = on ? *reinterpret_cast<const uint32_t*>(qs + head * kRowBytes + col) : 0u;
                        qb[ks][nt][1] = on ? *reinterpret_cast<const uint32_t*>(qs + head * kRowBytes + col + 16) : 0u;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ts]);

            // O^T accumulators: tile d of 16 dims; c0/c1 = dims 16d + g, heads 2t/2t+1; c2/c3 = dims 16d + g + 8
            float o[kNT][8][4];
            float m_a[kNT], m_b[kNT], l_a[kNT], l_b[kNT];  // running max / partial sum of head columns 2t, 2t+1
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                m_a[nt] = m_b[nt] = -INFINITY;
                l_a[nt] = l_b[nt] = 0.f;
#pragma unroll
                for (int d = 0; d < 8; ++d) o[nt][d][0] = o[nt][d][1] = o[nt][d][2] = o[nt][d][3] = 0.f;
            }
            bool aborted = false;

            // Page j of the CTA's page sequence lives in stage j % NS and is consumed by warp j % NCW. With
            // NS % NCW == 0 a stage is always consumed by the same warp, which has therefore finished the stage's
            // previous page before it waits on the stage again: the parity wait can never match a phase two back.
            for (int i = (w - seq % NCW + NCW) % NCW; i < npages; i += NCW) {
                const int j = seq + i;
                const int st = j % NS;
                if (!warp_wait(&full[st], (j / NS) & 1, ctx)) {
                    aborted = true;
                    break;
                }
                const int nvalid = min(kPageSize, slen - (spb + i) * kPageSize);
                const uint32_t sbase = stage0 + st * kStageBytes;
                if (nvalid < kPageSize) {
                    // The boxes always carry 16 token rows; rows past the row's length hold whatever the pool has
                    // there. Their scores are masked below; their V rows are zeroed so 0 * (non-finite) cannot
                    // reach the accumulator.
                    uint8_t* vbase = smem + L::off_stage + st * kStageBytes + 2 * kBoxBytes;
                    for (int e2 = lane; e2 < 2 * kPageSize * 8; e2 += 32) {
                        const int box = e2 >> 7, r = (e2 >> 3) & 15, c = e2 & 7;
                        if (r >= nvalid)
                            *reinterpret_cast<int4*>(vbase + box * kBoxBytes + r * 128 + c * 16) = make_int4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                const bool append = p.k_new != nullptr && (spb + i) * kPageSize + nvalid == slen;
                if (append) {
                    // The page holds the row's newest token (slot nvalid - 1), appended in this step: its K and V
                    // rows of KV head sh come from k_new / v_new. Lane l moves 16 bytes: pool l / 16 (K, V), box
                    // (l / 8) % 2 (columns 0-63, 64-127), chunk l % 8. Into the staged page (swizzled) for this
                    // step's scores, and into the pool slot for later steps; no other task reads these bytes.
                    const int r = nvalid - 1, pool = lane >> 4, half = (lane >> 3) & 1, chunk = lane & 7;
                    const size_t src = ((size_t)sb * Hkv + sh) * kHeadDim + half * 64 + chunk * 8;
                    const int4 val = *reinterpret_cast<const int4*>(
                        static_cast<const __half*>(pool ? p.v_new : p.k_new) + src);
                    uint8_t* stage = smem + L::off_stage + st * kStageBytes + (2 * pool + half) * kBoxBytes;
                    *reinterpret_cast<int4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4)) = val;
                    const int32_t phys = logical_page_phys(p, sb, spb + i);
                    if (phys >= 0 && phys < p.num_pages) {
                        __half* dst = const_cast<__half*>(static_cast<const __half*>(pool ? p.v_pool : p.k_pool)) +
                                      (((size_t)phys * kPageSize + r) * Hkv + sh) * kHeadDim + half * 64 + chunk * 8;
                        *reinterpret_cast<int4*>(dst) = val;
                    }
                    __syncwarp();
                }
                // S^T = K Q^T: rows = the 16 tokens, columns = 8 heads per tile, k = head_dim in 8 steps of 16
                float sc[kNT][4];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    const uint32_t box = sbase + (ks >> 2) * kBoxBytes;
                    ldsm_x4(box + swz(k_row, ((ks & 3) << 1) | k_par), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) mma_16816(sc[nt], a0, a1, a2, a3, qb[ks][nt][0], qb[ks][nt][1]);
                }
                uint32_t pb0[kNT], pb1[kNT];
#pragma unroll
                for (int nt = 0; nt < kNT; ++nt) {
                    // online softmax (base 2) per head column: this lane holds tokens g and g + 8 of heads 2t, 2t+1
                    float x0 = sc[nt][0] * sl2, x1 = sc[nt][1] * sl2, x2 = sc[nt][2] * sl2, x3 = sc[nt][3] * sl2;
                    if (g8 >= nvalid) x0 = x1 = -INFINITY;
                    if (g8 + 8 >= nvalid) x2 = x3 = -INFINITY;
                    float ma = fmaxf(x0, x2), mb = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, off));
                        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
                    }
                    const float na = fmaxf(m_a[nt], ma), nb = fmaxf(m_b[nt], mb);
                    const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
                    const float alpha_a = fast_exp2(m_a[nt] - ua), alpha_b = fast_exp2(m_b[nt] - ub);
                    const float p0 = fast_exp2(x0 - ua), p2 = fast_exp2(x2 - ua);
                    const float p1 = fast_exp2(x1 - ub), p3 = fast_exp2(x3 - ub);
                    l_a[nt] = l_a[nt] * alpha_a + (p0 + p2);
                    l_b[nt] = l_b[nt] * alpha_b + (p1 + p3);
                    m_a[nt] = na;
                    m_b[nt] = nb;
#pragma unroll
                    for (int d = 0; d < 8; ++d) {
                        o[nt][d][0] *= alpha_a;
                        o[nt][d][1] *= alpha_b;
                        o[nt][d][2] *= alpha_a;
                        o[nt][d][3] *= alpha_b;
                    }
                    // P^T in the B-operand layout (tokens 2t, 2t+1 | 2t+8, 2t+9 of head g)
                    const uint32_t h01 = pack_half2(p0, p1), h23 = pack_half2(p2, p3);
                    const uint32_t va = __shfl_sync(0xffffffffu, h01, src_a);
                    const uint32_t vb = __shfl_sync(0xffffffffu, h01, src_b);
                    const uint32_t vc = __shfl_sync(0xffffffffu, h23, src_a);
                    const uint32_t vd = __shfl_sync(0xffffffffu, h23, src_b);
                    pb0[nt] = __byte_perm(va, vb, sel);
                    pb1[nt] = __byte_perm(vc, vd, sel);
                }
                // O^T += V^T P^T: rows = 16 dims per tile (8 tiles), columns = heads, k = the 16 tokens
#pragma unroll
                for (int d = 0; d < 8; ++d) {
                    uint32_t a0, a1, a2, a3;
                    const uint32_t box = sbase + (2 + (d >> 2)) * kBoxBytes;
                    ldsm_x4_trans(box + swz(v_row, ((d & 3) << 1) | v_par), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < kNT; ++nt) mma_16816(o[nt][d], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                }
                if (nvalid < kPageSize || append) fence_proxy_async_smem();  // our stores before the next TMA write
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (aborted) break;
            seq += npages;

            // ---- hand this warp's partial (m, l, O) of the task to the epilogue warp
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    l_a[nt] += __shfl_xor_sync(0xffffffffu, l_a[nt], off);
                    l_b[nt] += __shfl_xor_sync(0xffffffffu, l_b[nt], off);
                }
            }
            if (!warp_wait(&eempty[e], ((tseq >> 1) & 1) ^ 1, ctx)) break;
            float* co = comb_o + e * L::kCombFloats + w * G * kCombRow;
            float2* cml = comb_ml + e * NCW * G + w * G;
#pragma unroll
            for (int nt = 0; nt < kNT; ++nt) {
                const int ha = nt * 8 + 2 * t4, hb = ha + 1;
                if (ha < G) {
#pragma unroll
                    for (int d = 0; d < 8; ++d) {
                        co[ha * kCombRow + d * 16 + g8] = o[nt][d][0];
                        co[ha * kCombRow + d * 16 + g8 + 8] = o[nt][d][2];
                    }
                    if (g8 == 0) cml[ha] = make_float2(m_a[nt], l_a[nt]);
                }
                if (hb < G) {
#pragma unroll
                    for (int d = 0; d < 8; ++d) {
                        co[hb * kCombRow + d * 16 + g8] = o[nt][d][1];
                        co[hb * kCombRow + d * 16 + g8 + 8] = o[nt][d][3];
                    }
                    if (g8 == 0) cml[hb] = make_float2(m_b[nt], l_b[nt]);
                }
            }
            if (w == 0 && lane == 0) {
                EpiHeader hd;
                hd.b = sb;
                hd.h = sh;
                hd.s = ss;
                hd.task = stask;
                hd.nsplit = snsplit;
                hd.npages = npages;
                hd.kind = kKindPages;
                hd.pad = 0;
                ehdr[e] = hd;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&efull[e]);
        }
    }
}

#ifndef PKV_DECODE_CONSUMERS
#define PKV_DECODE_CONSUMERS 4
#endif
#ifndef PKV_DECODE_STAGES
#define PKV_DECODE_STAGES 8
#endif
constexpr int kNCW = PKV_DECODE_CONSUMERS;  // consumer warps per CTA
constexpr int kNS = PKV_DECODE_STAGES;      // pages in flight per CTA
constexpr int kNTS = 4;                     // task slots (scheduler look-ahead)

template <int G>
int launch_g(const DecodeParams& p, int grid, bool pdl, cudaStream_t stream) {
    using L = Layout<G, kNCW, kNS, kNTS>;
    static int configured_mask = 0;  // one bit per device ordinal (< 32)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 32 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<G, kNCW, kNS, kNTS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::total);
        if (e != cudaSuccess) return e;
        __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_ACQ_REL);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3((kNCW + 3) * 32);
    cfg.dynamicSmemBytes = L::total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_kernel<G, kNCW, kNS, kNTS>, p);
}

}  // namespace

int decode_smem_bytes(int group) {
    switch (group) {
        case 1: return Layout<1, kNCW, kNS, kNTS>::total;
        case 2: return Layout<2, kNCW, kNS, kNTS>::total;
        case 4: return Layout<4, kNCW, kNS, kNTS>::total;
        case 8: return Layout<8, kNCW, kNS, kNTS>::total;
        case 16: return Layout<16, kNCW, kNS, kNTS>::total;
        default: return 0;
    }
}

int launch_decode(const DecodeParams& p, int group, int grid, bool pdl, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (group) {
        case 1: return launch_g<1>(p, grid, pdl, s);
        case 2: return launch_g<2>(p, grid, pdl, s);
        case 4: return launch_g<4>(p, grid, pdl, s);
        case 8: return launch_g<8>(p, grid, pdl, s);
        case 16: return launch_g<16>(p, grid, pdl, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
