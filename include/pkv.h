/*
 * pkv.h -- C ABI of the paged grouped-query decode-attention library (libpkv.so, CUDA, sm_103a).
 *
 * One decode step of attention over a block-table (paged) FP16 KV cache, as described in "PersistentKV:
 * Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs" (arXiv 2606.26666):
 *   - each query head hq of row b attends to its row's tokens through the row's block table; G = Hq / Hkv query
 *     heads share KV head hkv = hq / G, and work is mapped by KV-head group so those G heads reuse every K/V tile
 *     (abstract; gist.science technical summary, "Methodologie" 1, "Layout");
 *   - sequence splitting: a row's pages are cut into disjoint ranges, each producing a partial online-softmax
 *     state that a separate merge combines exactly ("Sequentie Splitting");
 *   - row-local bounds: split ranges come from each row's true length; empty splits write a neutral state
 *     ("Row-Local Bounds");
 *   - the compact workqueue: a 1-D list of only the non-empty (row, KV head, split) tasks ("Compact Workqueue");
 *   - a roofline-style host policy choosing the schedule and split size per step (abstract; "Calibrated
 *     Adaptive Policy").
 *
 * Tensor layouts (all row-major, contiguous; fp16 = IEEE binary16):
 *   q            [B][Hq][d]                           fp16, 16-byte aligned
 *   k_pool       [num_pages][page_size][Hkv][d]       fp16, 16-byte aligned
 *   v_pool       [num_pages][page_size][Hkv][d]       fp16, 16-byte aligned
 *   block_table  [B][max_pages_per_seq]               int32; entry p of row b is the physical page of logical
 *                                                     page p; entries past the row's last page are never read
 *   seq_lens     [B]                                  int32, tokens per row this step (0 allowed)
 *   out          [B][Hq][d]                           fp16, 16-byte aligned
 * Token j of row b lives in slot j % page_size of page block_table[b][j / page_size].
 * Supported: head_dim = 128, page_size = 16, G = Hq / Hkv in {1, 2, 4, 8, 16}, B <= PKV_MAX_BATCH.
 *
 * Ownership: the caller owns every buffer, including the workspace (sized by pkv_plan_t.ws_bytes, 256-byte
 * aligned, zeroed once with pkv_workspace_init). The library allocates no memory and keeps no per-call state;
 * the only process-wide state is a once-per-device kernel attribute set-up and a cache of TMA descriptors keyed by
 * pool address. Between steps the workspace's counters are back at zero; after a step that raised
 * PKV_STATUS_TIMEOUT or PKV_STATUS_TASKS, call pkv_workspace_init again before the next step.
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Every device call only
 * enqueues work and returns; pkv_plan is host-only and synchronous.
 * Errors: every call returns PKV_OK (0) or a negative PKV_E_* code and enqueues nothing on error. Errors the
 * kernels detect (a block-table entry outside the pool, a length beyond the table, a wait that timed out) are
 * OR-ed into a status word in the workspace; read it with pkv_read_status. No call traps or aborts.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 3: serving session (pkv_session_*) and PKV_PLAN_INPUTS_AFTER_PREV; the structs are unchanged from 2. */
#define PKV_VERSION 3

#define PKV_OK 0
#define PKV_E_INVAL (-1)        /* bad shape, negative size, inconsistent plan/problem */
#define PKV_E_UNSUPPORTED (-2)  /* head_dim, page_size, group size or batch outside the supported set */
#define PKV_E_NULLPTR (-3)      /* a required pointer is NULL */
#define PKV_E_WS_TOO_SMALL (-4) /* workspace smaller than plan->ws_bytes */
#define PKV_E_ALIGN (-5)        /* a pointer misses its required alignment */
#define PKV_E_CUDA (-6)         /* a CUDA runtime call or kernel launch failed */

/* bits of the device status word (pkv_read_status) */
#define PKV_STATUS_BAD_PAGE 0x1u  /* a block-table entry read by the kernel is outside [0, num_pages) */
#define PKV_STATUS_BAD_LEN 0x2u   /* a seq_len is negative or exceeds max_pages_per_seq * page_size */
#define PKV_STATUS_TIMEOUT 0x4u   /* an internal pipeline wait exceeded its time limit; the kernel returned */
#define PKV_STATUS_TASKS 0x8u     /* the device worklist outgrew the plan's task capacity (seq_lens changed
                                     between pkv_plan and the launch; extra tasks were dropped), or a task or
                                     row range in the workspace did not belong to the plan (it was skipped) */

#define PKV_MAX_BATCH 4096
#define PKV_MAX_ROWS_IN_DECODE 256 /* largest B for which the decode kernel can derive the workqueue itself */

/* schedules */
#define PKV_VARIANT_SINGLE 0    /* one task per (row, KV head), output normalised in the decode kernel */
#define PKV_VARIANT_SPLIT 1     /* rectangular grid over (row, KV head, split); empty splits write neutral states */
#define PKV_VARIANT_WORKQUEUE 2 /* device-built compact list of non-empty tasks, pulled from an atomic queue */

typedef struct pkv_problem {
    int32_t batch;             /* B */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 */
    int32_t head_dim;          /* d (128) */
    int32_t page_size;         /* tokens per page (16) */
    int32_t num_pages;         /* physical pages in each of k_pool / v_pool */
    int32_t max_pages_per_seq; /* columns of block_table */
} pkv_problem;

/*
 * Constants of the roofline cost model pkv_plan minimises (microseconds and GB/s; the v2 abstract's "calibrated
 * roofline-style policy", the gist.science technical summary's "Calibrated Adaptive Policy"). For a candidate plan
 * with T tasks on W resident CTAs, A = min(T, W) of them busy, kv = the step's K/V bytes and task bytes = c pages of
 * one KV head's K and V:
 *   workqueue (dynamic):   stream = kv / min(hbm_gbs, A * wq_cta_gbs)
 *                          decode = launch_us + stream + (T / W) * task_us
 *                                   + tail * max(0, ceil(T / W) * task_bytes / wq_cta_gbs - stream)
 *                          (the last term: the CTAs that run ceil(T / W) tasks at their own rate outlast the stream)
 *   split, single (static): decode = launch_us + ceil(T / W) * (task_us + (kv / T) / min(cta_gbs, hbm_gbs / A))
 *   merge  = merge_us + merge_state_us * S_max              separate merge kernel (launched with PDL)
 *          | fused_us + fused_state_us * S_max * G          merge fused into the last task of each (row, KV head)
 *   build  = build_us                                       workqueue with a builder launch
 *   step   = decode + merge + build
 * The rectangular split grid is a candidate only for B <= split_max_batch. pkv_policy_default returns the constants
 * fitted by serving_paged_gqa_gb300/calibrate.py on the calibration traces (seeds 0-4); its held-out evaluation
 * (seeds 5-9) is committed beside it.
 */
typedef struct pkv_policy {
    double launch_us;       /* decode launch, first bytes and teardown */
    double hbm_gbs;         /* KV streaming bandwidth of the whole GPU */
    double cta_gbs;         /* KV streaming bandwidth of one CTA of the static grid (split, single) */
    double wq_cta_gbs;      /* KV streaming bandwidth of one CTA pulling from the workqueue */
    double task_us;         /* per-task cost on one CTA (scheduling, q, epilogue) */
    double tail;            /* workqueue: weight of the per-CTA makespan beyond the bandwidth-bound stream */
    double merge_us;        /* separate merge: cost it adds to the step */
    double merge_state_us;  /* separate merge: per split of the longest (row, KV head) */
    double fused_us;        /* fused merge: cost of the last arrival and its merge */
    double fused_state_us;  /* fused merge: per partial state one last arriver merges */
    double build_us;        /* worklist builder launch (workqueue without the in-decode list) */
    int32_t ctas_per_sm;    /* resident decode CTAs per SM (clamped to what fits) */
    int32_t max_splits;     /* largest split count per row the policy may choose */
    int32_t allow_variants; /* bit mask of PKV_VARIANT_* (1 << v) the policy may choose */
    int32_t allow_fused;    /* 1: the policy may choose the fused merge */
    int32_t split_max_batch;/* largest B for which the split grid is a candidate */
    int32_t reserved;
} pkv_policy;

typedef struct pkv_plan_t {
    int32_t variant;     /* PKV_VARIANT_* */
    int32_t chunk_pages; /* c: pages per split; row b has S_b = ceil(ceil(L_b / page_size) / c) splits */
    int32_t num_splits;  /* S = max_b S_b (extent of the rectangular grid) */
    int32_t num_tasks;   /* tasks the decode kernel runs (single: B*Hkv; split: B*Hkv*S; wq: sum_b Hkv*S_b) */
    int32_t grid_ctas;   /* persistent decode grid size (resident CTAs, at most one wave) */
    int32_t group;       /* G = Hq / Hkv */
    int32_t num_sms;     /* SM count the plan was made for */
    int32_t fuse_merge;  /* split / workqueue: 1 = pkv_decode merges the split states itself (the CTA whose task of
                            a (row, KV head) finishes last runs the pair's merge as one more task: its states go
                            through that CTA's page ring, and it writes out; pkv_merge is then a no-op);
                            0 = pkv_decode writes partial states only and pkv_merge combines them. The planners pick
                            the mode their cost model predicts faster; a caller may change it (the workspace layout
                            does not depend on it). */
    int32_t list_in_decode; /* workqueue: 1 = the decode kernel derives the compact list itself from seq_lens (every
                               CTA scans the per-row split counts into shared memory; CTA 0 publishes row_off /
                               row_splits / task_count), so no pkv_build_worklist launch is needed; 0 = the decode
                               runs the list pkv_build_worklist wrote. The planners set 1 when B <= PKV_MAX_ROWS_IN_DECODE.
                               Both give the same list and state layout, in (b, h_kv, s) order. The builder's list
                               is claimed in that order; a list derived in the decode is claimed split by split
                               within a row (the Hkv tasks of one split, which read the same pages, together). */
    int32_t flags;          /* PKV_PLAN_* bits, 0 from the planners */
    pkv_problem problem; /* copy of the problem the plan was made for; later calls must pass an equal one */
    int64_t task_capacity;  /* task slots reserved in the workspace */
    int64_t state_capacity; /* partial-state slots reserved in the workspace */
    int64_t ws_bytes;       /* workspace bytes this plan needs */
    int64_t off_counters;   /* byte offsets inside the workspace: uint32 arrivals[B][Hkv] (fused merge) */
    int64_t off_row_off;    /*   int32 row_off[B] */
    int64_t off_row_splits; /*   int32 row_splits[B] */
    int64_t off_tasks;      /*   int4 tasks[task_capacity] */
    int64_t off_ml;         /*   float2 (m, l) per state */
    int64_t off_acc;        /*   float acc[state_capacity][d] */
    double predicted_us;    /* cost-model estimate for the step */
    double kv_bytes;        /* algorithmic bytes of the step: K and V of every token + q + out */
} pkv_plan_t;

/* Packed task as the worklist builder stores it (16 bytes): x = row b, y = (h_kv << 16) | split s,
 * z = first logical page, w = one past the last logical page. */
typedef struct pkv_task {
    int32_t row;
    int32_t head_split;
    int32_t page_begin;
    int32_t page_end;
} pkv_task;

/* Workspace header at offset 0 (256 bytes). */
typedef struct pkv_ws_header {
    uint32_t queue_head;  /* next task to claim (workqueue); re-armed to 0 by the builder and after every decode */
    int32_t task_count;   /* tasks written by the last pkv_build_worklist */
    uint32_t status;      /* PKV_STATUS_* bits, sticky until pkv_read_status clears them */
    uint32_t ctas_done;   /* decode CTAs that finished claiming (workqueue); back to 0 after every decode */
    uint32_t reserved[60];
} pkv_ws_header;

/*
 * Plan flag: the step may start while the kernel enqueued just before it on the same stream is still running
 * (programmatic dependent launch), so its CTAs start, read their block-table entries and lengths and begin copying
 * K/V pages while that kernel finishes; q, k_new and v_new are read, and out and the workspace written, only after
 * that kernel has completed (griddepcontrol.wait). Set it only if that kernel writes none of block_table, seq_lens,
 * k_pool and v_pool (typical of a layer loop: the previous layer produced q, the block table and lengths were
 * written before the first layer). Ignored by plans that run the worklist builder (workqueue with list_in_decode
 * = 0). The separate merge kernel lets the next launch start early as well.
 */
#define PKV_PLAN_OVERLAP_PREV 0x1u

/*
 * Plan flag: the step may start while the kernel enqueued just before it on the same stream is still running, and
 * that kernel may write every input (q, k_new, v_new, block_table, seq_lens; e.g. the copy of the step's packed
 * input into device memory): the CTAs only set up their shared memory and barriers before griddepcontrol.wait and
 * read nothing until that kernel has completed. Takes precedence over PKV_PLAN_OVERLAP_PREV. Ignored by plans that
 * run the worklist builder. pkv_serve_step and the serving session set it on the decode that follows their input
 * copy kernel.
 */
#define PKV_PLAN_INPUTS_AFTER_PREV 0x2u

/* Library version (PKV_VERSION). */
int pkv_version(void);

/* Text for a PKV_E_* code. */
const char* pkv_strerror(int code);

/* Validates a problem against the supported set. Host only. */
int pkv_check_problem(const pkv_problem* problem);

/* Fills *policy with the built-in cost-model constants (fitted on the calibration traces, seeds 0-4). */
void pkv_policy_default(pkv_policy* policy);

/*
 * Plans one decode step (the "calibrated roofline-style policy" of the v2 abstract and of the gist.science
 * summary, "Calibrated Adaptive Policy"): evaluates the cost model for the single-pass, split and workqueue
 * schedules over a set of split sizes and keeps the cheapest. seq_lens_host [B] must equal the seq_lens the
 * device calls will read. policy NULL = pkv_policy_default. num_sms = SMs of the target GPU. Host only.
 */
int pkv_plan(const pkv_problem* problem, const int32_t* seq_lens_host, int32_t num_sms, const pkv_policy* policy,
             pkv_plan_t* plan);

/* Same as pkv_plan with the schedule and split size fixed by the caller (chunk_pages >= 1; ignored for
 * PKV_VARIANT_SINGLE). ctas_per_sm <= 0 means the default. The merge mode (fuse_merge) is the one the default
 * policy predicts faster; the caller may change it. Used by tests and calibration sweeps. */
int pkv_plan_fixed(const pkv_problem* problem, const int32_t* seq_lens_host, int32_t num_sms, int32_t variant,
                   int32_t chunk_pages, int32_t ctas_per_sm, pkv_plan_t* plan);

/* Zeroes the whole workspace (header, arrival counters) on `stream`. Call once after allocating, and again after
 * a step that raised PKV_STATUS_TIMEOUT or PKV_STATUS_TASKS. */
int pkv_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Worklist builder (gist.science technical summary, "Methodologie" 1, "Compact Workqueue": a 1-D grid of tasks for
 * the non-empty row / KV-head / split intervals only). From device seq_lens computes S_b, an exclusive prefix sum of
 * Hkv*S_b, and writes the non-empty tasks in (b, h_kv, s) order, row_off/row_splits, the task count and resets the
 * queue head. Only for plans with variant PKV_VARIANT_WORKQUEUE (returns PKV_E_INVAL otherwise). The decode that
 * follows it on the same stream may start its prologue while the builder runs (programmatic dependent launch); it
 * reads nothing the builder writes before the builder has finished.
 */
int pkv_build_worklist(const pkv_plan_t* plan, const pkv_problem* problem, const int32_t* seq_lens_dev, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * Decode kernel: grouped-query attention of every row over its pages, read in place through block_table (gist.science
 * technical summary, "Methodologie" 1: "Layout" -- no repacking into contiguous tensors; "Sequentie Splitting" --
 * each split computes a partial online-softmax state; "Row-Local Bounds" -- split ranges from each row's true length,
 * empty splits write a neutral state; v1/v2 abstracts: work mapped by KV-head group). For query head hq of row b
 * (KV head hkv = hq / G) it computes softmax(scale * q.K^T) V over the row's seq_lens[b] tokens.
 *   single: one task per (row, KV head); writes the normalised output to out.
 *   split / workqueue: one task per (row, KV head, split) writes the partial (m, l, acc) state of its G query heads
 *     into the workspace (empty rectangular splits write m = -inf, l = 0, acc = 0). With plan->fuse_merge = 1 the
 *     CTA that finishes the last task of each (row, KV head) also merges that pair's states and writes out; with 0,
 *     follow with pkv_merge.
 *   workqueue: with plan->list_in_decode = 0 runs the list the last pkv_build_worklist wrote into ws (call it first,
 *     on the same stream); with 1 derives the same list from seq_lens_dev itself.
 * scale multiplies q.k (use 1/sqrt(head_dim)). out may be NULL only for split / workqueue plans with fuse_merge 0.
 * Rows longer than the plan's lengths (seq_lens grew after pkv_plan) raise PKV_STATUS_TASKS; their extra pages are
 * not read.
 */
int pkv_decode(const pkv_plan_t* plan, const pkv_problem* problem, const void* q, const void* k_pool,
               const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale, void* ws,
               size_t ws_bytes, void* out, void* stream);

/*
 * Log-sum-exp merge ("Sequentie Splitting": a separate merge combines the split states exactly):
 * out[b,hq] = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s with M = max_s m_s over non-neutral states; a row
 * with no non-empty state gets 0. For split and workqueue plans with fuse_merge = 0; for single plans and fused
 * plans it returns PKV_OK without work.
 */
int pkv_merge(const pkv_plan_t* plan, const pkv_problem* problem, void* ws, size_t ws_bytes, void* out,
              void* stream);

/* Convenience: build (workqueue with list_in_decode = 0) + decode + merge (fuse_merge = 0) for one step on one
 * stream. */
int pkv_decode_step(const pkv_plan_t* plan, const pkv_problem* problem, const void* q, const void* k_pool,
                    const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale,
                    void* ws, size_t ws_bytes, void* out, void* stream);

/*
 * One decode step of a model layer with the new token's K/V append fused into it (the step before attention in a
 * decode loop; multi-layer decode calls it once per layer with that layer's pools). seq_lens_dev already counts the
 * new token: row b's token L_b - 1 lives in slot (L_b - 1) % page_size of page block_table[b][(L_b - 1) / page_size],
 * which the caller has allocated. k_new, v_new: [B][Hkv][d] fp16, 16-byte aligned, the token's K and V. The kernel
 * that reads that page writes k_new / v_new into the pools' slot and uses them for this step's scores; rows with
 * L_b = 0 append nothing. Otherwise as pkv_decode_step (plan, workspace, merge, errors). k_pool and v_pool are
 * written (one 256-byte row per (row, KV head)).
 */
int pkv_decode_step_append(const pkv_plan_t* plan, const pkv_problem* problem, const void* q, const void* k_new,
                           const void* v_new, void* k_pool, void* v_pool, const int32_t* block_table,
                           const int32_t* seq_lens_dev, float scale, void* ws, size_t ws_bytes, void* out,
                           void* stream);

/*
 * Byte offsets of the five parts of a packed step input (pkv_serve_step): offsets[0] q [B][Hq][d] fp16, [1] k_new
 * [B][Hkv][d] fp16, [2] v_new [B][Hkv][d] fp16, [3] block_table [B][max_pages_per_seq] int32, [4] seq_lens [B]
 * int32 (counting the new token), each part starting on a 256-byte boundary; *total = the buffer's size in bytes.
 * Host only. Returns PKV_OK, PKV_E_NULLPTR or a pkv_check_problem error.
 */
int pkv_step_input_layout(const pkv_problem* problem, size_t offsets[5], size_t* total);

/*
 * One serving step of a layer from host memory in a single call: plans the step (pkv_plan with `policy`, NULL = the
 * built-in constants, on the seq_lens of host_in, which the CPU reads during the call), then enqueues on `stream` the
 * transfer of the packed input host_in (layout of pkv_step_input_layout) into dev_in, the step with the new token's
 * K/V appended (pkv_decode_step_append on the parts of dev_in), and the transfer of out ([B][Hq][d] fp16) into
 * host_out. Page-locked host buffers mapped into the device's address space (cudaHostAlloc, torch's pin_memory) are
 * moved by the GPU itself: a copy kernel reads host_in through its device address, and the step stores out straight
 * into host_out (dev_out is then not written); other host buffers go through cudaMemcpyAsync (dev_out receives out
 * first). The caller owns every buffer: host_in and host_out (16-byte aligned), dev_in (device, at least the
 * layout's total, 256-byte aligned), the pools, ws (at least the plan's ws_bytes: PKV_E_WS_TOO_SMALL otherwise, with
 * nothing enqueued) and dev_out; nothing is allocated. Synchronise the stream before reading host_out or refilling
 * host_in. If plan_out is not NULL it receives the plan. Errors as pkv_plan and pkv_decode_step_append; on error
 * nothing is enqueued. The pages describe no such call: it is how a server feeds the decode step from the host.
 */
int pkv_serve_step(const pkv_problem* problem, const pkv_policy* policy, int32_t num_sms, const void* host_in,
                   void* dev_in, void* k_pool, void* v_pool, float scale, void* ws, size_t ws_bytes, void* dev_out,
                   void* host_out, void* stream, pkv_plan_t* plan_out);

/* Distinct plans whose captured launches a serving session keeps (least recently used first out). */
#define PKV_SESSION_GRAPHS 16

/*
 * Serving session: the buffers of pkv_serve_step bound once (a server's per-layer buffers do not change between
 * steps), and the step's launches replayed from CUDA graphs. The pages describe no such object; it is how this
 * library takes the host-side launch cost off a decode loop, where the plan repeats for many steps (a row's split
 * count changes once every chunk_pages * page_size tokens).
 *
 * pkv_session_create validates and binds problem, policy (copied; NULL = the built-in constants), num_sms (> 0) and
 * the buffers exactly as pkv_serve_step takes them (same layout, alignment and ownership rules; the caller keeps
 * every buffer alive until pkv_session_destroy); it resolves whether host_in and host_out are mapped page-locked
 * memory and, if both are, creates one private non-blocking stream for capturing. *session receives the handle
 * (NULL on error). Errors: PKV_E_NULLPTR, PKV_E_INVAL (num_sms <= 0), PKV_E_ALIGN, pkv_check_problem errors,
 * PKV_E_CUDA (stream creation).
 *
 * pkv_session_step runs one step with the current contents of host_in: pkv_plan on its seq_lens, then, with both
 * host buffers mapped, the step's launches (input copy kernel, decode with the append, merge) are looked up by the
 * plan's launch fields (every field of pkv_plan_t but predicted_us and kv_bytes); a plan seen before replays its
 * graph with one cudaGraphLaunch on `stream`, a new one is captured on the private stream, instantiated, kept (at
 * most PKV_SESSION_GRAPHS, the least recently used is destroyed) and launched. Otherwise (a pageable host buffer, or
 * `stream` being captured by the caller) the launches are enqueued on `stream` as pkv_serve_step does. Results,
 * asynchrony and errors as pkv_serve_step (synchronise `stream` before reading host_out or refilling host_in);
 * plan_out (optional) receives the plan. One host thread at a time per session.
 *
 * pkv_session_stats: graphs captured and graph launches so far. pkv_session_destroy destroys the graphs and the
 * private stream and frees the handle (NULL is a no-op); no work of the session may be pending on the GPU.
 */
typedef struct pkv_session pkv_session;

int pkv_session_create(const pkv_problem* problem, const pkv_policy* policy, int32_t num_sms, const void* host_in,
                       void* dev_in, void* k_pool, void* v_pool, float scale, void* ws, size_t ws_bytes,
                       void* dev_out, void* host_out, pkv_session** session);
int pkv_session_step(pkv_session* session, void* stream, pkv_plan_t* plan_out);
int pkv_session_stats(const pkv_session* session, int64_t* graphs_captured, int64_t* graph_launches);
int pkv_session_destroy(pkv_session* session);

/* Synchronises `stream`, copies the workspace status word to *status and clears it on the device. */
int pkv_read_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status);

/* Number of kernel launches pkv_decode_step enqueues for this plan. */
int pkv_plan_launches(const pkv_plan_t* plan);

/* Size of the library-owned workspace behind pkv_decode_step_static (16 MiB per GPU). */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * pkv_decode_step for callers that cannot allocate device memory. The paper has no counterpart: it is a
 * convenience of this library. Some callers cannot call cudaMalloc where they run a decode step (a plug-in whose
 * host application owns every allocation, code running inside another framework's memory pool, a serving loop
 * that must not allocate after start-up), so this call takes the same inputs and output as pkv_decode_step but
 * keeps the workspace in a fixed array of PKV_STATIC_SCRATCH_BYTES in the library's own device memory. Every GPU
 * that loads libpkv.so holds that array until the process exits. The call itself allocates nothing.
 *   plan, problem, q, k_pool, v_pool, block_table, seq_lens_dev, scale, out, stream: as for pkv_decode_step
 *     (out is always required).
 *   status_dev: NULL, or a 4-byte aligned device uint32_t that receives this step's PKV_STATUS_* bits (stream
 *     ordered, after the step).
 * Errors: PKV_E_WS_TOO_SMALL if plan->ws_bytes exceeds PKV_STATIC_SCRATCH_BYTES (choose a plan with fewer tasks,
 * e.g. a larger chunk_pages); otherwise the errors of pkv_decode_step. Nothing is enqueued on error.
 * The first call on a device looks up the array's device address (once per device, with that device current);
 * make that first call before any stream capture. All calls share the one array and it keeps the last call's
 * contents; the call clears the status word after each step. Calls whose work overlaps on the GPU (other streams,
 * or other host threads on the same device) race on the array: order them on one stream.
 */
int pkv_decode_step_static(const pkv_plan_t* plan, const pkv_problem* problem, const void* q, const void* k_pool,
                           const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale,
                           void* out, uint32_t* status_dev, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
