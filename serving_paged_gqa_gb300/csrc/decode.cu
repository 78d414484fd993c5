// Persistent split-KV paged GQA decode kernel for sm_103a, with the log-sum-exp merge fused into the last task of
// every (row, KV head).
//
// Computes, for every task (row b, KV head h, logical pages [page_begin, page_end)), the online-softmax state of
// the G = Hq/Hkv query heads that share KV head h ("PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs", v1/v2 abstracts: work mapped by KV-head group so the grouped query heads reuse each
// K/V tile; gist.science technical summary, "Methodologie" 1: native block-table execution ("Layout"), sequence
// splitting into partial online-softmax states combined exactly ("Sequentie Splitting"), row-local bounds with
// neutral states for empty splits ("Row-Local Bounds"), compact workqueue ("Compact Workqueue")).
//
// CTA layout (persistent over tasks; grid = resident CTAs):
//   warp NCW+1  scheduler: takes tasks (split / single: a static stride over the task space, KV heads fastest, so the
//               CTAs that start together read the same pages; workqueue: an atomic queue head over the built list,
//               after waiting for the builder grid), fetches the row length and the task's first 32 block-table
//               entries together, publishes both in a shared-memory task slot, then bulk-copies the G query rows of
//               the task into the slot (completion on a separate barrier, so the loader never waits for q);
//   warp NCW    loader: per page, one elected lane issues four 3-D TMA tensor copies (K and V of KV head h, each as
//               two 64-column boxes of the page's 16 token rows, 128-byte swizzled) into a ring stage, counted in
//               bytes on the stage's mbarrier; block-table entries past the slot's 32 are read one chunk ahead;
//   warps 0..NCW-1 consumers: page j of the CTA's page sequence (counted across tasks) lives in stage j % NS and
//               goes to warp j % NCW (NS % NCW == 0, so a stage always has the same consumer). Per page: S = Q K^T on
//               mma.sync m16n8k16 (rows = the G query heads, columns = the 16 tokens), masking of slots past the row
//               length, online softmax in base 2 in registers with quad shuffles, O += P V on mma.sync. At the end
//               of a task the NCW warps combine their states through shared memory and write the normalised fp16
//               output (single pass) or the partial state (m, l, acc) of each query head. With the merge fused, the
//               task then counts itself in the (b, h) arrival counter; the last of the S_b tasks of (b, h) to arrive
//               reads all S_b states from L2 and writes the merged output, then re-arms the counter. Nobody waits.
// Every wait is bounded (global timer); on timeout the kernel sets PKV_STATUS_TIMEOUT in the workspace, the other
// warps see an abort flag, the loader and the scheduler wait (bounded) for their own copies in flight, and the CTA
// returns.
#include <cuda_fp16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kBoxBytes = kPageSize * 128;   // one TMA box: 16 token rows x 64 fp16 columns (128 B, swizzled)
constexpr int kStageBytes = 4 * kBoxBytes;   // K columns 0-63, K 64-127, V 0-63, V 64-127
constexpr int kCombRow = kHeadDim + 8;       // floats per combined row (padding against bank conflicts)
constexpr int kSlotEntries = 32;             // block-table entries the scheduler prefetches per task
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct TaskSlot {
    int32_t b, h, s, task;                  // task: canonical index; the task's states are task * G + g
    int32_t page_begin, npages, seq_len, nsplit;  // nsplit: tasks of (b, h) (arrivals of the fused merge; 0 = none)
    int32_t ent[kSlotEntries];              // physical page of logical page page_begin + i (i < min(npages, 32))
};

template <int G, int NCW, int NS, int NTS>
struct Layout {
    static constexpr int kQRowsBytes = ((G * kRowBytes + 127) / 128) * 128;
    static constexpr int off_stage = 0;  // 1024-byte aligned (128-byte swizzle atom)
    static constexpr int off_q = off_stage + NS * kStageBytes;
    static constexpr int off_comb = off_q + NTS * kQRowsBytes;
    static constexpr int comb_o_floats = NCW * G * kCombRow;
    static constexpr int off_comb_ml = off_comb + comb_o_floats * 4;
    static constexpr int off_slots = off_comb_ml + NCW * G * 8;
    static constexpr int off_bars = ((off_slots + NTS * (int)sizeof(TaskSlot) + 15) / 16) * 16;
    static constexpr int nbars = 2 * NS + 3 * NTS + 4;
    static constexpr int off_flag = off_bars + nbars * 8;
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

// Exact log-sum-exp merge of the nsplit partial states of query head g of the task group starting at task `first`:
// out = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s over states with l_s > 0 (running maximum, so the states
// are read once). Lane k owns dimensions 4k..4k+3. States were written by other CTAs: read them from L2.
template <int G>
__device__ __forceinline__ void merge_group(const DecodeParams& p, int first, int nsplit, int g, int lane,
                                            __half* out_row) {
    const float2* mlp = reinterpret_cast<const float2*>(p.ml);
    const float4* accp = reinterpret_cast<const float4*>(p.acc);
    float M = -INFINITY, D = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
        float2 ml[8];
        float4 av[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j < nsplit) {
                const size_t st = (size_t)(first + s0 + j) * G + g;
                ml[j] = __ldcg(mlp + st);
                av[j] = __ldcg(accp + st * (kHeadDim / 4) + lane);
            } else {
                ml[j] = make_float2(-INFINITY, 0.f);
                av[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (ml[j].y > 0.f) {
                const float m2 = ml[j].x * kLog2e;
                const float mn = fmaxf(M, m2);
                const float fo = fast_exp2(M - mn), fn = fast_exp2(m2 - mn);
                D = D * fo + fn * ml[j].y;
                A.x = A.x * fo + fn * av[j].x;
                A.y = A.y * fo + fn * av[j].y;
                A.z = A.z * fo + fn * av[j].z;
                A.w = A.w * fo + fn * av[j].w;
                M = mn;
            }
        }
    }
    const float inv = D > 0.f ? 1.f / D : 0.f;
    uint2 pk;
    pk.x = pack_half2(A.x * inv, A.y * inv);
    pk.y = pack_half2(A.z * inv, A.w * inv);
    *reinterpret_cast<uint2*>(out_row + lane * 4) = pk;
}

template <int G, int NCW, int NS, int NTS>
__global__ void __launch_bounds__((NCW + 2) * 32, kDecodeCtasPerSm) decode_kernel(const __grid_constant__ DecodeParams p) {
    static_assert(NS % NCW == 0, "each ring stage must map to one consumer warp");
    using L = Layout<G, NCW, NS, NTS>;
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
    uint64_t* cfull = tempty + NTS;
    uint64_t* cempty = cfull + 1;
    uint64_t* mstate = cempty + 1;    // fused merge: every consumer warp has stored its part of the task's states
    uint64_t* mlast = mstate + 1;     // fused merge: warp 0 has counted the task and published whether it was last
    TaskSlot* slots = reinterpret_cast<TaskSlot*>(smem + L::off_slots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::off_flag);
    volatile int* last_flag = abort_flag + 1;
    const WaitCtx ctx{abort_flag, &p.hdr->status};

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < NTS; ++i) {
            mbar_init(&tmeta[i], 1);
            mbar_init(&tq[i], 1);
            mbar_init(&tempty[i], NCW + 1);
        }
        mbar_init(cfull, NCW);
        mbar_init(cempty, NCW);
        mbar_init(mstate, NCW);
        mbar_init(mlast, 1);
        *abort_flag = 0;
        *last_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();

    const int Hq = p.Hq, Hkv = p.Hkv;

    if (warp == NCW + 1) {
        // ------------------------------------------------------------------ scheduler
        // Everything this grid reads from global memory is read after this point (the other warps only follow the
        // slots published below), so the grid may start while the worklist builder is still running.
        grid_dependency_wait();
        const int variant = p.variant;
        const bool wq = variant == PKV_VARIANT_WORKQUEUE;
        int count = p.num_tasks;
        if (wq) count = min(*reinterpret_cast<volatile int32_t*>(&p.hdr->task_count), p.task_capacity);
        const __half* q = static_cast<const __half*>(p.q);
        int tseq = 0;
        for (int k = 0;; ++k) {
            int t;
            if (wq) {
                int c = 0;
                if (lane == 0) c = static_cast<int>(atomicAdd(&p.hdr->queue_head, 1u));
                t = __shfl_sync(0xffffffffu, c, 0);
            } else {
                t = blockIdx.x + k * gridDim.x;
            }
            const int ts = tseq % NTS;
            if (!warp_wait(&tempty[ts], ((tseq / NTS) & 1) ^ 1, ctx)) break;
            TaskSlot* sl = &slots[ts];
            if (t >= count) {
                if (lane == 0) {
                    sl->npages = -1;
                    mbar_arrive(&tmeta[ts]);
                }
                break;
            }
            int b, h, s, pb, pe, task, nsplit = 1;
            if (wq) {
                const pkv_task tk = p.tasks[t];
                b = tk.row;
                h = tk.head_split >> 16;
                s = tk.head_split & 0xffff;
                pb = tk.page_begin;
                pe = tk.page_end;
                task = t;
            } else if (variant == PKV_VARIANT_SPLIT) {
                const int S = p.num_splits;
                const int per_row = Hkv * S;
                b = t / per_row;
                const int r = t - b * per_row;
                s = r / Hkv;
                h = r - s * Hkv;
                pb = s * p.chunk_pages;
                pe = pb + p.chunk_pages;
                task = (b * Hkv + h) * S + s;
                nsplit = S;
            } else {
                b = t / Hkv;
                h = t - b * Hkv;
                s = 0;
                pb = 0;
                pe = p.max_pages;
                task = t;
            }
            const bool bad = b < 0 || b >= p.B || h < 0 || h >= Hkv || s < 0 || pb < 0 || pe < pb;
            if (bad) {  // a task that is not from this plan: it writes a neutral state and takes no part in a merge
                if (lane == 0) raise_status(ctx.status, PKV_STATUS_TASKS);
                b = 0;
                h = 0;
                pb = pe = 0;
            }
            // the row length and the task's first block-table entries, fetched together
            const int nent = max(0, min(min(pe, p.max_pages) - pb, kSlotEntries));
            const int ent = lane < nent ? p.block_table[(size_t)b * p.max_pages + pb + lane] : -1;
            int len = p.seq_lens[b];
            const int row_splits = wq ? p.row_splits[b] : 0;
            if (len < 0 || len > p.max_pages * kPageSize) {
                if (lane == 0) raise_status(ctx.status, PKV_STATUS_BAD_LEN);
                len = 0;
            }
            const int np_row = (len + kPageSize - 1) / kPageSize;
            const int np = max(0, min(pe, np_row) - pb);
            // A row with pages past its last task (its length grew after the plan was made) is flagged; its tasks
            // still take part in the merge, so the arrival counters stay consistent.
            bool grown, foreign = bad;
            if (wq) {  // the builder's split count of the row: the number of tasks of (b, h) in the list
                nsplit = row_splits;
                // the states of (b, h) are tasks [t - s, t - s + S_b) of the list
                foreign = foreign || s >= row_splits || t - s < 0 || t - s + row_splits > count;
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
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tmeta[ts]);
                if (np > 0) {  // the G query rows of this KV head are contiguous in q
                    mbar_arrive_expect_tx(&tq[ts], G * kRowBytes);
                    bulk_g2s(smem + L::off_q + ts * L::kQRowsBytes, q + ((size_t)b * Hq + (size_t)h * G) * kHeadDim,
                             G * kRowBytes, &tq[ts]);
                } else {
                    mbar_arrive(&tq[ts]);
                }
            }
            __syncwarp();
            ++tseq;
        }
        // Before the warp leaves, every query copy it issued has landed (only after an abort can one be pending).
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
    } else if (warp == NCW) {
        // ------------------------------------------------------------------ loader
        if (lane == 0) {
            prefetch_tensormap(&p.tmap_k);
            prefetch_tensormap(&p.tmap_v);
        }
        const uint64_t pol = policy_evict_first();
        int seq = 0;
        bool stop = false;
        for (int tseq = 0; !stop; ++tseq) {
            const int ts = tseq % NTS;
            if (!warp_wait(&tmeta[ts], (tseq / NTS) & 1, ctx)) break;
            const int np = slots[ts].npages;
            const int b = slots[ts].b, h = slots[ts].h, pb = slots[ts].page_begin;
            int ent = slots[ts].ent[lane];
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ts]);
            if (np < 0) break;
            const int32_t* bt = p.block_table + (size_t)b * p.max_pages + pb;
            int ent_next = kSlotEntries + lane < np ? bt[kSlotEntries + lane] : 0;
            for (int c0 = 0; c0 < np; c0 += 32) {
                if (c0 > 0) {
                    ent = ent_next;
                    if (c0 + 32 + lane < np) ent_next = bt[c0 + 32 + lane];
                }
                const int n = min(32, np - c0);
                for (int i = 0; i < n; ++i) {
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
    } else {
        // ------------------------------------------------------------------ consumers
        const int w = warp;
        const int g0 = lane >> 2;        // query head (row of the mma tile) this lane holds
        const int tq4 = 2 * (lane & 3);  // first token column this lane holds in each 8-token half
        const int mi = lane >> 3, mr = lane & 7;
        // ldmatrix row addresses: K (non-transposed) rows = tokens (mi >> 1) * 8 + mr, chunk parity mi & 1;
        // V (transposed) rows = tokens (mi & 1) * 8 + mr, chunk parity mi >> 1.
        const int k_row = ((mi >> 1) << 3) + mr, k_par = mi & 1;
        const int v_row = ((mi & 1) << 3) + mr, v_par = mi >> 1;
        const uint32_t stage0 = smem_addr(smem + L::off_stage);
        float* comb_o = reinterpret_cast<float*>(smem + L::off_comb);
        float2* comb_ml = reinterpret_cast<float2*>(smem + L::off_comb_ml);
        const float sl2 = p.scale_log2;
        const bool fused = p.fuse_merge != 0 && p.variant != PKV_VARIANT_SINGLE;
        int seq = 0;
        for (int tseq = 0;; ++tseq) {
            const int ts = tseq % NTS;
            if (!warp_wait(&tmeta[ts], (tseq / NTS) & 1, ctx)) break;
            const int npages = slots[ts].npages;
            if (npages < 0) break;
            const int sb = slots[ts].b, sh = slots[ts].h, ss = slots[ts].s, stask = slots[ts].task;
            const int spb = slots[ts].page_begin, slen = slots[ts].seq_len, snsplit = slots[ts].nsplit;
            if (!warp_wait(&tq[ts], (tseq / NTS) & 1, ctx)) break;
            // Query fragments (A operand rows = query heads of the group; rows >= G are zero).
            uint32_t qa[8][4];
            {
                const uint8_t* qs = smem + L::off_q + ts * L::kQRowsBytes;
                const bool lo = g0 < G && npages > 0;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int col = (ks * 16 + tq4) * 2;
                    qa[ks][0] = lo ? *reinterpret_cast<const uint32_t*>(qs + g0 * kRowBytes + col) : 0u;
                    qa[ks][2] = lo ? *reinterpret_cast<const uint32_t*>(qs + g0 * kRowBytes + col + 16) : 0u;
                    if constexpr (G > 8) {
                        const bool hi = g0 + 8 < G && npages > 0;
                        qa[ks][1] = hi ? *reinterpret_cast<const uint32_t*>(qs + (g0 + 8) * kRowBytes + col) : 0u;
                        qa[ks][3] = hi ? *reinterpret_cast<const uint32_t*>(qs + (g0 + 8) * kRowBytes + col + 16) : 0u;
                    } else {
                        qa[ks][1] = 0u;
                        qa[ks][3] = 0u;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ts]);

            float o[16][4];
#pragma unroll
            for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            float m_lo = -INFINITY, l_lo = 0.f, m_hi = -INFINITY, l_hi = 0.f;
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
                    for (int e = lane; e < 2 * kPageSize * 8; e += 32) {
                        const int box = e >> 7, r = (e >> 3) & 15, c = e & 7;
                        if (r >= nvalid)
                            *reinterpret_cast<int4*>(vbase + box * kBoxBytes + r * 128 + c * 16) = make_int4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
                // S = Q K^T: two n8 tiles (tokens 0-7 and 8-15), k = head_dim in 8 steps of 16 columns
                float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    const uint32_t box = sbase + (ks >> 2) * kBoxBytes;
                    ldsm_x4(box + swz(k_row, ((ks & 3) << 1) | k_par), b0, b1, b2, b3);
                    mma_16816(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                    mma_16816(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
                }
                // online softmax (base 2), row g0 and (G > 8) row g0 + 8
                float x[4] = {s0[0] * sl2, s0[1] * sl2, s1[0] * sl2, s1[1] * sl2};
                if (tq4 >= nvalid) x[0] = -INFINITY;
                if (tq4 + 1 >= nvalid) x[1] = -INFINITY;
                if (tq4 + 8 >= nvalid) x[2] = -INFINITY;
                if (tq4 + 9 >= nvalid) x[3] = -INFINITY;
                float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float mn = fmaxf(m_lo, mx);
                const float mu = mn == -INFINITY ? 0.f : mn;
                const float alpha = fast_exp2(m_lo - mu);
                float pr[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) pr[e] = fast_exp2(x[e] - mu);
                l_lo = l_lo * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
                m_lo = mn;
                const uint32_t pa0 = pack_half2(pr[0], pr[1]);
                const uint32_t pa2 = pack_half2(pr[2], pr[3]);
                uint32_t pa1 = 0u, pa3 = 0u;
                float alpha_hi = 1.f;
                if constexpr (G > 8) {
                    float y[4] = {s0[2] * sl2, s0[3] * sl2, s1[2] * sl2, s1[3] * sl2};
                    if (tq4 >= nvalid) y[0] = -INFINITY;
                    if (tq4 + 1 >= nvalid) y[1] = -INFINITY;
                    if (tq4 + 8 >= nvalid) y[2] = -INFINITY;
                    if (tq4 + 9 >= nvalid) y[3] = -INFINITY;
                    float my = fmaxf(fmaxf(y[0], y[1]), fmaxf(y[2], y[3]));
                    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 1));
                    my = fmaxf(my, __shfl_xor_sync(0xffffffffu, my, 2));
                    const float mnh = fmaxf(m_hi, my);
                    const float muh = mnh == -INFINITY ? 0.f : mnh;
                    alpha_hi = fast_exp2(m_hi - muh);
                    float ph[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) ph[e] = fast_exp2(y[e] - muh);
                    l_hi = l_hi * alpha_hi + ((ph[0] + ph[1]) + (ph[2] + ph[3]));
                    m_hi = mnh;
                    pa1 = pack_half2(ph[0], ph[1]);
                    pa3 = pack_half2(ph[2], ph[3]);
                }
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o[n][0] *= alpha;
                    o[n][1] *= alpha;
                    if constexpr (G > 8) {
                        o[n][2] *= alpha_hi;
                        o[n][3] *= alpha_hi;
                    }
                }
                // O += P V: 16 n8 tiles over head_dim, k = the 16 tokens
#pragma unroll
                for (int n2 = 0; n2 < 8; ++n2) {
                    uint32_t b0, b1, b2, b3;
                    const uint32_t box = sbase + (2 + (n2 >> 2)) * kBoxBytes;
                    ldsm_x4_trans(box + swz(v_row, ((n2 & 3) << 1) | v_par), b0, b1, b2, b3);
                    mma_16816(o[2 * n2], pa0, pa1, pa2, pa3, b0, b1);
                    mma_16816(o[2 * n2 + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
                if (nvalid < kPageSize) fence_proxy_async_smem();  // zero stores before the next TMA write
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (aborted) break;
            seq += npages;

            // ---- combine the NCW warps' states of this task
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
            if constexpr (G > 8) {
                l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
                l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
            }
            if (!warp_wait(cempty, (tseq & 1) ^ 1, ctx)) break;
            float* my_o = comb_o + w * G * kCombRow;
            if (g0 < G) {
#pragma unroll
                for (int n = 0; n < 16; ++n)
                    *reinterpret_cast<float2*>(my_o + g0 * kCombRow + n * 8 + tq4) = make_float2(o[n][0], o[n][1]);
                if ((lane & 3) == 0) comb_ml[w * G + g0] = make_float2(m_lo, l_lo);
            }
            if constexpr (G > 8) {
                if (g0 + 8 < G) {
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        *reinterpret_cast<float2*>(my_o + (g0 + 8) * kCombRow + n * 8 + tq4) =
                            make_float2(o[n][2], o[n][3]);
                    if ((lane & 3) == 0) comb_ml[w * G + g0 + 8] = make_float2(m_hi, l_hi);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(cfull);
            if (!warp_wait(cfull, tseq & 1, ctx)) break;
            for (int g = w; g < G; g += NCW) {
                float M = -INFINITY;
#pragma unroll
                for (int wi = 0; wi < NCW; ++wi) M = fmaxf(M, comb_ml[wi * G + g].x);
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                float lsum = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int wi = 0; wi < NCW; ++wi) {
                        const float2 ml = comb_ml[wi * G + g];
                        const float f = fast_exp2(ml.x - M);
                        lsum += f * ml.y;
                        const float4 v = *reinterpret_cast<const float4*>(comb_o + (wi * G + g) * kCombRow + lane * 4);
                        a.x += f * v.x;
                        a.y += f * v.y;
                        a.z += f * v.z;
                        a.w += f * v.w;
                    }
                }
                const int hq = sh * G + g;
                if (p.variant == PKV_VARIANT_SINGLE) {
                    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
                    uint2 pk;
                    pk.x = pack_half2(a.x * inv, a.y * inv);
                    pk.y = pack_half2(a.z * inv, a.w * inv);
                    __half* out = static_cast<__half*>(p.out) + ((size_t)sb * Hq + hq) * kHeadDim;
                    *reinterpret_cast<uint2*>(out + lane * 4) = pk;
                } else {
                    const size_t state = (size_t)stask * G + g;
                    if (lane == 0)
                        reinterpret_cast<float2*>(p.ml)[state] =
                            make_float2(M == -INFINITY ? -INFINITY : M * kLn2, lsum);
                    reinterpret_cast<float4*>(p.acc + state * kHeadDim)[lane] = a;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(cempty);

            if (fused) {
                // ---- fused merge: count this task in (b, h); the last arriver merges all S_b states. Two bounded
                // barrier rounds: every warp's states are stored (and fenced) before warp 0 counts the task; the
                // count's outcome is then broadcast. Phase k of either barrier completes before any warp can arrive
                // for task k + 1, so the parities never alias.
                __threadfence();  // this thread's state stores are visible device-wide before the arrival
                __syncwarp();
                if (lane == 0) mbar_arrive(mstate);
                if (w == 0) {
                    if (!warp_wait(mstate, tseq & 1, ctx)) break;
                    if (lane == 0) {
                        int last = 0;
                        if (snsplit > 0) {
                            uint32_t* cnt = p.counters + (size_t)sb * Hkv + sh;
                            __threadfence();
                            const uint32_t old = atomicAdd(cnt, 1u);
                            last = old + 1u == (uint32_t)snsplit;
                            if (last) atomicExch(cnt, 0u);  // re-armed for the next step
                        }
                        *last_flag = last;
                        mbar_arrive(mlast);
                    }
                    __syncwarp();
                }
                if (!warp_wait(mlast, tseq & 1, ctx)) break;
                if (*last_flag) {
                    __threadfence();  // the other tasks' states, published before their arrivals, are read after
                    for (int g = w; g < G; g += NCW)
                        merge_group<G>(p, stask - ss, snsplit, g, lane,
                                       static_cast<__half*>(p.out) + ((size_t)sb * Hq + (size_t)sh * G + g) * kHeadDim);
                }
            }
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
    cfg.blockDim = dim3((kNCW + 2) * 32);
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
