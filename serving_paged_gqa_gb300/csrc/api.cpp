// C-ABI entry points of libpkv.so: argument validation and kernel launches (see include/pkv.h).
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>

#include "pkv_internal.h"

namespace {

using namespace pkv;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool same_problem(const pkv_problem& a, const pkv_problem& b) { return std::memcmp(&a, &b, sizeof(a)) == 0; }

int check_plan(const pkv_plan_t* plan, const pkv_problem* pr, const void* ws, size_t ws_bytes) {
    if (!plan || !pr || !ws) return PKV_E_NULLPTR;
    int rc = pkv_check_problem(pr);
    if (rc != PKV_OK) return rc;
    if (!same_problem(plan->problem, *pr)) return PKV_E_INVAL;
    if (plan->variant < PKV_VARIANT_SINGLE || plan->variant > PKV_VARIANT_WORKQUEUE) return PKV_E_INVAL;
    if (plan->group != pr->num_q_heads / pr->num_kv_heads || plan->grid_ctas <= 0 || plan->chunk_pages <= 0 ||
        plan->num_splits <= 0 || plan->num_tasks < 0 || (plan->fuse_merge != 0 && plan->fuse_merge != 1) ||
        (plan->list_in_decode != 0 && plan->list_in_decode != 1))
        return PKV_E_INVAL;
    if (plan->list_in_decode && pr->batch > PKV_MAX_ROWS_IN_DECODE) return PKV_E_UNSUPPORTED;
    if ((uint32_t)plan->flags & ~(PKV_PLAN_OVERLAP_PREV | PKV_PLAN_INPUTS_AFTER_PREV)) return PKV_E_INVAL;
    if (plan->off_counters < (int64_t)sizeof(pkv_ws_header) ||
        plan->off_counters + 4 * (int64_t)pr->batch * pr->num_kv_heads > plan->ws_bytes)
        return PKV_E_INVAL;
    if (!aligned(ws, kWsAlign)) return PKV_E_ALIGN;
    if ((int64_t)ws_bytes < plan->ws_bytes) return PKV_E_WS_TOO_SMALL;
    return PKV_OK;
}

template <typename T>
T* at(void* ws, int64_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int cuda_rc(int e) { return e == cudaSuccess ? PKV_OK : PKV_E_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// TMA descriptor of a K or V pool [num_pages][page_size][Hkv][d] seen as the 3-D tensor (d, Hkv, num_pages *
// page_size) with box (64, 1, page_size) and 128-byte swizzle. Descriptors are cached by (device, pointer, shape).
int pool_tensor_map(const void* pool, int num_pages, int hkv, CUtensorMap* out) {
    struct Entry {
        const void* ptr;
        int num_pages, hkv, dev;
        CUtensorMap map;
    };
    static std::mutex mu;
    static Entry cache[32];
    static int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_E_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < used; ++i) {
            const Entry& e = cache[i];
            if (e.ptr == pool && e.num_pages == num_pages && e.hkv == hkv && e.dev == dev) {
                *out = e.map;
                return PKV_OK;
            }
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return PKV_E_CUDA;
    const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)num_pages * kPageSize};
    const cuuint64_t strides[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)hkv * kRowBytes};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)kPageSize};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap m;
    if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_E_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    Entry& e = cache[next];
    e = Entry{pool, num_pages, hkv, dev, m};
    next = (next + 1) % 32;
    used = std::max(used, next == 0 ? 32 : next);
    *out = m;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_version(void) { return PKV_VERSION; }

extern "C" const char* pkv_strerror(int code) {
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_E_INVAL: return "invalid argument";
        case PKV_E_UNSUPPORTED: return "unsupported problem (head_dim 128, page_size 16, G in {1,2,4,8,16})";
        case PKV_E_NULLPTR: return "null pointer";
        case PKV_E_WS_TOO_SMALL: return "workspace smaller than plan->ws_bytes";
        case PKV_E_ALIGN: return "misaligned pointer";
        case PKV_E_CUDA: return "CUDA error";
        default: return "unknown error";
    }
}

extern "C" int pkv_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws) return PKV_E_NULLPTR;
    if (ws_bytes < sizeof(pkv_ws_header)) return PKV_E_WS_TOO_SMALL;
    if (!aligned(ws, kWsAlign)) return PKV_E_ALIGN;
    return cuda_rc(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

extern "C" int pkv_build_worklist(const pkv_plan_t* plan, const pkv_problem* pr, const int32_t* seq_lens_dev,
                                  void* ws, size_t ws_bytes, void* stream) {
    int rc = check_plan(plan, pr, ws, ws_bytes);
    if (rc != PKV_OK) return rc;
    if (plan->variant != PKV_VARIANT_WORKQUEUE) return PKV_E_INVAL;
    if (pr->batch > 0 && !seq_lens_dev) return PKV_E_NULLPTR;
    if (!aligned(seq_lens_dev, 4)) return PKV_E_ALIGN;
    BuildParams p{};
    p.seq_lens = seq_lens_dev;
    p.row_off = at<int32_t>(ws, plan->off_row_off);
    p.row_splits = at<int32_t>(ws, plan->off_row_splits);
    p.tasks = at<pkv_task>(ws, plan->off_tasks);
    p.hdr = static_cast<pkv_ws_header*>(ws);
    p.B = pr->batch;
    p.Hkv = pr->num_kv_heads;
    p.max_pages = pr->max_pages_per_seq;
    p.chunk_pages = plan->chunk_pages;
    p.task_capacity = (int32_t)plan->task_capacity;
    const int64_t blocks = (plan->task_capacity + 1023) / 1024;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(blocks, 2 * (int64_t)plan->num_sms));
    return cuda_rc(launch_build(p, grid, stream));
}

namespace pkv {

int check_decode_args(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_pool,
                      const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale,
                      void* ws, size_t ws_bytes, void* out) {
    int rc = check_plan(plan, pr, ws, ws_bytes);
    if (rc != PKV_OK) return rc;
    if (pr->batch > 0 && (!q || !k_pool || !v_pool || !block_table || !seq_lens_dev)) return PKV_E_NULLPTR;
    const bool writes_out = plan->variant == PKV_VARIANT_SINGLE || plan->fuse_merge;
    if (writes_out && pr->batch > 0 && !out) return PKV_E_NULLPTR;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens_dev, 4))
        return PKV_E_ALIGN;
    if (!(scale == scale)) return PKV_E_INVAL;
    return PKV_OK;
}

int decode_step(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_new, const void* v_new,
                const void* k_pool, const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev,
                float scale, void* ws, size_t ws_bytes, void* out, void* stream, bool clear_counters) {
    int rc = check_decode_args(plan, pr, q, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes, out);
    if (rc != PKV_OK) return rc;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_E_NULLPTR;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_E_ALIGN;
    if (clear_counters) {
        const size_t n = 4 * (size_t)pr->batch * pr->num_kv_heads;
        if (n > 0 && cudaMemsetAsync(at<char>(ws, plan->off_counters), 0, n, static_cast<cudaStream_t>(stream)) !=
                         cudaSuccess)
            return PKV_E_CUDA;
    }
    if (plan->variant == PKV_VARIANT_WORKQUEUE && !plan->list_in_decode) {
        rc = pkv_build_worklist(plan, pr, seq_lens_dev, ws, ws_bytes, stream);
        if (rc != PKV_OK) return rc;
    }
    rc = decode_launch(plan, pr, q, k_new, v_new, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes, out,
                       stream);
    if (rc != PKV_OK) return rc;
    return pkv_merge(plan, pr, ws, ws_bytes, out, stream);
}

}  // namespace pkv

extern "C" int pkv_decode(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_pool,
                          const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale,
                          void* ws, size_t ws_bytes, void* out, void* stream) {
    return decode_launch(plan, pr, q, nullptr, nullptr, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes,
                         out, stream);
}

int pkv::decode_launch(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_new,
                       const void* v_new, const void* k_pool, const void* v_pool, const int32_t* block_table,
                       const int32_t* seq_lens_dev, float scale, void* ws, size_t ws_bytes, void* out, void* stream) {
    int rc = check_decode_args(plan, pr, q, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes, out);
    if (rc != PKV_OK) return rc;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_E_NULLPTR;
    if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_E_ALIGN;
    // A workqueue plan may hold no task while its rows still need an output (every row empty); other plans have
    // tasks whenever B > 0.
    if (pr->batch == 0) return PKV_OK;
    DecodeParams p{};
    if (pr->num_pages > 0) {
        rc = pool_tensor_map(k_pool, pr->num_pages, pr->num_kv_heads, &p.tmap_k);
        if (rc == PKV_OK) rc = pool_tensor_map(v_pool, pr->num_pages, pr->num_kv_heads, &p.tmap_v);
        if (rc != PKV_OK) return rc;
    }
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.k_new = k_new;
    p.v_new = v_new;
    p.block_table = block_table;
    p.seq_lens = seq_lens_dev;
    p.out = out;
    p.ml = at<float>(ws, plan->off_ml);
    p.acc = at<float>(ws, plan->off_acc);
    p.tasks = at<const pkv_task>(ws, plan->off_tasks);
    p.row_off = at<int32_t>(ws, plan->off_row_off);
    p.row_splits = at<int32_t>(ws, plan->off_row_splits);
    p.counters = at<uint32_t>(ws, plan->off_counters);
    p.hdr = static_cast<pkv_ws_header*>(ws);
    p.B = pr->batch;
    p.Hq = pr->num_q_heads;
    p.Hkv = pr->num_kv_heads;
    p.num_pages = pr->num_pages;
    p.max_pages = pr->max_pages_per_seq;
    p.chunk_pages = plan->chunk_pages;
    p.num_splits = plan->num_splits;
    p.variant = plan->variant;
    p.num_tasks = plan->num_tasks;
    p.task_capacity = (int32_t)plan->task_capacity;
    p.fuse_merge = plan->variant != PKV_VARIANT_SINGLE && plan->fuse_merge;
    p.list_in_decode = plan->variant == PKV_VARIANT_WORKQUEUE && plan->list_in_decode;
    p.scale_log2 = scale * 1.4426950408889634f;
    // The workqueue decode follows its builder: let it start while the builder runs (it reads the builder's output
    // only after griddepcontrol.wait). Otherwise it may start early only if the plan says the kernel before it writes
    // none of what the decode reads before that wait.
    const bool builder = plan->variant == PKV_VARIANT_WORKQUEUE && !plan->list_in_decode;
    const uint32_t flags = (uint32_t)plan->flags;
    const bool pdl = builder || (flags & (PKV_PLAN_OVERLAP_PREV | PKV_PLAN_INPUTS_AFTER_PREV));
    p.inputs_after_wait = !builder && (flags & PKV_PLAN_INPUTS_AFTER_PREV) ? 1 : 0;
    p.overlap_prev = !builder && !p.inputs_after_wait && (flags & PKV_PLAN_OVERLAP_PREV) ? 1 : 0;
    return cuda_rc(launch_decode(p, plan->group, plan->grid_ctas, pdl, stream));
}

extern "C" int pkv_merge(const pkv_plan_t* plan, const pkv_problem* pr, void* ws, size_t ws_bytes, void* out,
                         void* stream) {
    int rc = check_plan(plan, pr, ws, ws_bytes);
    if (rc != PKV_OK) return rc;
    if (plan->variant == PKV_VARIANT_SINGLE || plan->fuse_merge) return PKV_OK;
    if (pr->batch > 0 && !out) return PKV_E_NULLPTR;
    if (!aligned(out, 16)) return PKV_E_ALIGN;
    MergeParams p{};
    p.ml = at<float>(ws, plan->off_ml);
    p.acc = at<float>(ws, plan->off_acc);
    p.row_off = at<int32_t>(ws, plan->off_row_off);
    p.row_splits = at<int32_t>(ws, plan->off_row_splits);
    p.out = out;
    p.B = pr->batch;
    p.Hq = pr->num_q_heads;
    p.Hkv = pr->num_kv_heads;
    p.num_splits = plan->num_splits;
    p.variant = plan->variant;
    p.status = &static_cast<pkv_ws_header*>(ws)->status;
    p.task_capacity = plan->num_tasks;
    return cuda_rc(launch_merge(p, stream));
}

extern "C" int pkv_decode_step(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_pool,
                               const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev,
                               float scale, void* ws, size_t ws_bytes, void* out, void* stream) {
    return decode_step(plan, pr, q, nullptr, nullptr, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes,
                       out, stream, false);
}

extern "C" int pkv_decode_step_append(const pkv_plan_t* plan, const pkv_problem* pr, const void* q,
                                      const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                                      const int32_t* block_table, const int32_t* seq_lens_dev, float scale, void* ws,
                                      size_t ws_bytes, void* out, void* stream) {
    if (pr && pr->batch > 0 && (!k_new || !v_new)) return PKV_E_NULLPTR;
    return decode_step(plan, pr, q, k_new, v_new, k_pool, v_pool, block_table, seq_lens_dev, scale, ws, ws_bytes, out,
                       stream, false);
}

extern "C" int pkv_step_input_layout(const pkv_problem* pr, size_t offsets[5], size_t* total) {
    if (!pr || !offsets || !total) return PKV_E_NULLPTR;
    int rc = pkv_check_problem(pr);
    if (rc != PKV_OK) return rc;
    const size_t B = (size_t)pr->batch;
    const size_t sizes[5] = {B * pr->num_q_heads * pr->head_dim * 2, B * pr->num_kv_heads * pr->head_dim * 2,
                             B * pr->num_kv_heads * pr->head_dim * 2, B * (size_t)pr->max_pages_per_seq * 4, B * 4};
    size_t off = 0;
    for (int i = 0; i < 5; ++i) {
        offsets[i] = off;
        off += (sizes[i] + kWsAlign - 1) / kWsAlign * kWsAlign;
    }
    *total = off;
    return PKV_OK;
}

namespace {

// The device-visible address of page-locked host memory (mapped into the device's address space), or nullptr for
// any other pointer (pageable host memory, device memory, unknown): such buffers are moved with cudaMemcpyAsync.
const void* mapped_host_address(const void* p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // an unregistered pointer is not an error of this call
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// The buffers of a serving step (everything but the step's contents), validated once.
struct ServeBind {
    pkv_problem pr;
    size_t off[5];
    size_t total;
    const void* host_in;
    void* dev_in;
    void* k_pool;
    void* v_pool;
    float scale;
    void* ws;
    size_t ws_bytes;
    void* dev_out;
    void* host_out;
    const void* in_mapped;  // device-visible addresses of the host buffers, or nullptr (copied by cudaMemcpyAsync)
    void* out_mapped;
};

int bind_serve(const pkv_problem* pr, const void* host_in, void* dev_in, void* k_pool, void* v_pool, float scale,
               void* ws, size_t ws_bytes, void* dev_out, void* host_out, ServeBind* sb) {
    if (!pr || !host_in || !dev_in || !ws || !dev_out || !host_out) return PKV_E_NULLPTR;
    int rc = pkv_step_input_layout(pr, sb->off, &sb->total);
    if (rc != PKV_OK) return rc;
    if (!aligned(dev_in, kWsAlign) || !aligned(dev_out, 16)) return PKV_E_ALIGN;
    if (!aligned(host_in, 16) || !aligned(host_out, 16)) return PKV_E_ALIGN;
    sb->pr = *pr;
    sb->host_in = host_in;
    sb->dev_in = dev_in;
    sb->k_pool = k_pool;
    sb->v_pool = v_pool;
    sb->scale = scale;
    sb->ws = ws;
    sb->ws_bytes = ws_bytes;
    sb->dev_out = dev_out;
    sb->host_out = host_out;
    // Page-locked host buffers mapped into the device's address space are read and written by kernels directly
    // (the input by a copy kernel, out by the step's own output stores); others go through cudaMemcpyAsync.
    sb->in_mapped = mapped_host_address(host_in);
    sb->out_mapped = const_cast<void*>(mapped_host_address(host_out));
    return PKV_OK;
}

const int32_t* host_lens(const ServeBind& sb) {
    return reinterpret_cast<const int32_t*>(static_cast<const char*>(sb.host_in) + sb.off[4]);
}

int check_serve(const ServeBind& sb, const pkv_plan_t* plan) {
    if ((int64_t)sb.ws_bytes < plan->ws_bytes) return PKV_E_WS_TOO_SMALL;
    const char* d = static_cast<const char*>(sb.dev_in);
    return check_decode_args(plan, &sb.pr, d + sb.off[0], sb.k_pool, sb.v_pool,
                             reinterpret_cast<const int32_t*>(d + sb.off[3]),
                             reinterpret_cast<const int32_t*>(d + sb.off[4]), sb.scale, sb.ws, sb.ws_bytes,
                             sb.out_mapped ? sb.out_mapped : sb.dev_out);
}

// Enqueues one serving step of `plan` on `s`: the input copy, the decode with the new token appended, the merge and
// the output copy (arguments checked by check_serve).
int serve_enqueue(const ServeBind& sb, const pkv_plan_t* plan, cudaStream_t s) {
    if (sb.pr.batch == 0) return PKV_OK;
    char* d = static_cast<char*>(sb.dev_in);
    void* out = sb.out_mapped ? sb.out_mapped : sb.dev_out;
    pkv_plan_t run = *plan;
    if (sb.in_mapped) {
        if (launch_stage_copy(sb.in_mapped, sb.dev_in, sb.total, s) != cudaSuccess) return PKV_E_CUDA;
        run.flags |= PKV_PLAN_INPUTS_AFTER_PREV;  // the decode's set-up overlaps the copy kernel
    } else if (cudaMemcpyAsync(sb.dev_in, sb.host_in, sb.total, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        return PKV_E_CUDA;
    }
    int rc = decode_step(&run, &sb.pr, d + sb.off[0], d + sb.off[1], d + sb.off[2], sb.k_pool, sb.v_pool,
                         reinterpret_cast<const int32_t*>(d + sb.off[3]),
                         reinterpret_cast<const int32_t*>(d + sb.off[4]), sb.scale, sb.ws, sb.ws_bytes, out, s, false);
    if (rc != PKV_OK) return rc;
    const size_t out_bytes = (size_t)sb.pr.batch * sb.pr.num_q_heads * sb.pr.head_dim * 2;
    if (!sb.out_mapped && cudaMemcpyAsync(sb.host_out, sb.dev_out, out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PKV_E_CUDA;
    return PKV_OK;
}

}  // namespace

extern "C" int pkv_serve_step(const pkv_problem* pr, const pkv_policy* policy, int32_t num_sms, const void* host_in,
                              void* dev_in, void* k_pool, void* v_pool, float scale, void* ws, size_t ws_bytes,
                              void* dev_out, void* host_out, void* stream, pkv_plan_t* plan_out) {
    ServeBind sb;
    int rc = bind_serve(pr, host_in, dev_in, k_pool, v_pool, scale, ws, ws_bytes, dev_out, host_out, &sb);
    if (rc != PKV_OK) return rc;
    pkv_plan_t plan;  // from the lengths in the host copy of the input
    rc = pkv_plan(pr, host_lens(sb), num_sms, policy, &plan);
    if (rc != PKV_OK) return rc;
    if ((int64_t)ws_bytes < plan.ws_bytes) return PKV_E_WS_TOO_SMALL;
    if (plan_out) *plan_out = plan;
    rc = check_serve(sb, &plan);
    if (rc != PKV_OK) return rc;
    return serve_enqueue(sb, &plan, static_cast<cudaStream_t>(stream));
}

// A serving session: the buffers bound once, and every distinct plan's launches captured once into a CUDA graph
// (on a private stream) that later steps with the same plan replay with one cudaGraphLaunch.
struct pkv_session {
    ServeBind sb;
    pkv_policy pol;
    bool have_pol;
    int32_t num_sms;
    bool graphs;             // both host buffers are mapped: the step is kernels only and can be captured
    cudaStream_t capture;    // private stream the graphs are captured on
    struct Entry {
        pkv_plan_t key;      // the plan without its lens-dependent estimates (predicted_us, kv_bytes)
        cudaGraphExec_t exec;
        uint64_t used;
    };
    Entry cache[PKV_SESSION_GRAPHS];
    int n;
    uint64_t clock;
    int64_t captured, replayed;
};

extern "C" int pkv_session_create(const pkv_problem* pr, const pkv_policy* policy, int32_t num_sms,
                                  const void* host_in, void* dev_in, void* k_pool, void* v_pool, float scale, void* ws,
                                  size_t ws_bytes, void* dev_out, void* host_out, pkv_session** session) {
    if (!session) return PKV_E_NULLPTR;
    *session = nullptr;
    if (num_sms <= 0) return PKV_E_INVAL;
    ServeBind sb;
    int rc = bind_serve(pr, host_in, dev_in, k_pool, v_pool, scale, ws, ws_bytes, dev_out, host_out, &sb);
    if (rc != PKV_OK) return rc;
    pkv_session* s = new (std::nothrow) pkv_session();
    if (!s) return PKV_E_CUDA;
    s->sb = sb;
    s->have_pol = policy != nullptr;
    if (policy) s->pol = *policy;
    s->num_sms = num_sms;
    s->graphs = sb.pr.batch > 0 && sb.in_mapped != nullptr && sb.out_mapped != nullptr;
    s->capture = nullptr;
    if (s->graphs && cudaStreamCreateWithFlags(&s->capture, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        delete s;
        return PKV_E_CUDA;
    }
    *session = s;
    return PKV_OK;
}

extern "C" int pkv_session_step(pkv_session* s, void* stream, pkv_plan_t* plan_out) {
    if (!s) return PKV_E_NULLPTR;
    const ServeBind& sb = s->sb;
    pkv_plan_t plan;
    int rc = pkv_plan(&sb.pr, host_lens(sb), s->num_sms, s->have_pol ? &s->pol : nullptr, &plan);
    if (rc != PKV_OK) return rc;
    if (plan_out) *plan_out = plan;
    rc = check_serve(sb, &plan);
    if (rc != PKV_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    bool graph = s->graphs;
    if (graph) {  // a stream the caller is capturing gets the launches themselves
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
            cudaGetLastError();
            graph = false;
        } else if (cs != cudaStreamCaptureStatusNone) {
            graph = false;
        }
    }
    if (!graph) return serve_enqueue(sb, &plan, st);
    pkv_plan_t key = plan;
    key.predicted_us = 0.0;
    key.kv_bytes = 0.0;
    for (int i = 0; i < s->n; ++i) {
        if (std::memcmp(&s->cache[i].key, &key, sizeof(key)) == 0) {
            s->cache[i].used = ++s->clock;
            if (cudaGraphLaunch(s->cache[i].exec, st) != cudaSuccess) return PKV_E_CUDA;
            ++s->replayed;
            return PKV_OK;
        }
    }
    if (cudaStreamBeginCapture(s->capture, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        cudaGetLastError();
        return PKV_E_CUDA;
    }
    rc = serve_enqueue(sb, &plan, s->capture);
    cudaGraph_t g = nullptr;
    const cudaError_t end = cudaStreamEndCapture(s->capture, &g);
    cudaGraphExec_t exec = nullptr;
    if (rc == PKV_OK && (end != cudaSuccess || !g || cudaGraphInstantiate(&exec, g, 0) != cudaSuccess)) rc = PKV_E_CUDA;
    if (g) cudaGraphDestroy(g);
    if (rc != PKV_OK) {
        cudaGetLastError();
        return rc;
    }
    int slot = s->n;
    if (s->n == PKV_SESSION_GRAPHS) {  // the least recently used graph makes room
        slot = 0;
        for (int i = 1; i < s->n; ++i)
            if (s->cache[i].used < s->cache[slot].used) slot = i;
        cudaGraphExecDestroy(s->cache[slot].exec);
    } else {
        ++s->n;
    }
    s->cache[slot].key = key;
    s->cache[slot].exec = exec;
    s->cache[slot].used = ++s->clock;
    ++s->captured;
    if (cudaGraphLaunch(exec, st) != cudaSuccess) return PKV_E_CUDA;
    ++s->replayed;
    return PKV_OK;
}

extern "C" int pkv_session_stats(const pkv_session* s, int64_t* graphs_captured, int64_t* graph_launches) {
    if (!s || !graphs_captured || !graph_launches) return PKV_E_NULLPTR;
    *graphs_captured = s->captured;
    *graph_launches = s->replayed;
    return PKV_OK;
}

extern "C" int pkv_session_destroy(pkv_session* s) {
    if (!s) return PKV_OK;
    int rc = PKV_OK;
    for (int i = 0; i < s->n; ++i)
        if (cudaGraphExecDestroy(s->cache[i].exec) != cudaSuccess) rc = PKV_E_CUDA;
    if (s->capture && cudaStreamDestroy(s->capture) != cudaSuccess) rc = PKV_E_CUDA;
    if (rc != PKV_OK) cudaGetLastError();
    delete s;
    return rc;
}

extern "C" int pkv_read_status(void* ws, size_t ws_bytes, void* stream, uint32_t* status) {
    if (!ws || !status) return PKV_E_NULLPTR;
    if (ws_bytes < sizeof(pkv_ws_header)) return PKV_E_WS_TOO_SMALL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    pkv_ws_header* hdr = static_cast<pkv_ws_header*>(ws);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, &hdr->status, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PKV_E_CUDA;
    if (cudaMemsetAsync(&hdr->status, 0, sizeof(uint32_t), s) != cudaSuccess) return PKV_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_E_CUDA;
    *status = v;
    return PKV_OK;
}
