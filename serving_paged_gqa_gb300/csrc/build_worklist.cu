// Device worklist builder for the compact workqueue schedule.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs", gist.science
// technical summary, "Methodologie" 1, "Compact Workqueue": the scheduler emits a 1-D grid of tasks only for the
// non-empty row / KV-head / split intervals. Row b has P_b = ceil(L_b / page_size) pages and
// S_b = ceil(P_b / c) splits of c pages ("Row-Local Bounds": counts come from each row's true length); its tasks
// start at off_b = sum_{b' < b} Hkv * S_b' and are ordered (h_kv, s). Every CTA recomputes the block-wide
// exclusive scan of Hkv * S_b in shared memory (B <= PKV_MAX_BATCH) and then writes a grid-strided share of the
// tasks, locating each task's row by binary search over the offsets. CTA 0 also publishes row_off, row_splits,
// the task count and resets the queue head the decode kernel claims tasks from.
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 1024;
constexpr int kPerThread = PKV_MAX_BATCH / kThreads;

__global__ void __launch_bounds__(kThreads) build_kernel(const BuildParams p) {
    // The decode launched after this grid waits for its completion before it reads anything written here, so it
    // may be scheduled at once.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int32_t s_off[PKV_MAX_BATCH + 1];
    __shared__ int32_t s_pages[PKV_MAX_BATCH];
    __shared__ int32_t s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.B, c = p.chunk_pages;

    int items[kPerThread];
    int tsum = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int b = tid * kPerThread + k;
        int n = 0;
        if (b < B) {
            int len = p.seq_lens[b];
            if (len < 0 || len > p.max_pages * kPageSize) {
                if (blockIdx.x == 0) atomicOr(&p.hdr->status, PKV_STATUS_BAD_LEN);
                len = 0;
            }
            const int pages = (len + kPageSize - 1) / kPageSize;
            s_pages[b] = pages;
            n = p.Hkv * ((pages + c - 1) / c);
        }
        items[k] = n;
        tsum += n;
    }
    // block-wide exclusive scan of the per-thread sums
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int x = s_warp[lane];
        int xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, xi, o);
            if (lane >= o) xi += y;
        }
        s_warp[lane] = xi - x;
    }
    __syncthreads();
    int run = s_warp[warp] + incl - tsum;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) {
        const int b = tid * kPerThread + k;
        if (b < B) s_off[b] = run;
        run += items[k];
    }
    if (tid == kThreads - 1) s_off[B] = run;  // the last thread's running sum is the grand total
    __syncthreads();

    const int total = s_off[B];
    const int count = min(total, p.task_capacity);
    if (blockIdx.x == 0) {
        for (int b = tid; b < B; b += kThreads) {
            p.row_off[b] = s_off[b];
            p.row_splits[b] = (s_pages[b] + c - 1) / c;
        }
        if (tid == 0) {
            p.hdr->task_count = count;
            p.hdr->queue_head = 0u;
            p.hdr->ctas_done = 0u;
            if (total > p.task_capacity) atomicOr(&p.hdr->status, PKV_STATUS_TASKS);
        }
    }
    for (int t = blockIdx.x * kThreads + tid; t < count; t += gridDim.x * kThreads) {
        // last row b with s_off[b] <= t; rows with no tasks share their successor's offset and are skipped
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= t)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int b = lo;
        const int pages = s_pages[b];
        const int splits = (pages + c - 1) / c;
        const int r = t - s_off[b];
        const int h = r / splits;
        const int s = r - h * splits;
        const int pb = s * c;
        pkv_task tk;
        tk.row = b;
        tk.head_split = (h << 16) | s;
        tk.page_begin = pb;
        tk.page_end = min(pb + c, pages);
        p.tasks[t] = tk;
    }
}

}  // namespace

int launch_build(const BuildParams& p, int grid, void* stream) {
    build_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
