// Internal declarations shared by the host API and the kernel translation units of libpkv.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>

#include "pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;
constexpr int kPageSize = 16;
constexpr int kRowBytes = kHeadDim * 2;               // one token of one KV head, fp16
constexpr int kTokenHeadBytes = 2 * kRowBytes;        // K + V of one token for one KV head
constexpr int kStateBytes = (kHeadDim + 2) * 4;       // (m, l, acc[d]) in fp32
constexpr int kWsAlign = 256;

// Arguments of the decode kernel (passed by value as a __grid_constant__ kernel parameter).
struct DecodeParams {
    // TMA descriptors of the K and V pools viewed as 3-D tensors (d, Hkv, num_pages * page_size), box
    // (64, 1, page_size), 128-byte swizzle: one box is half of one KV head's rows of one page.
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    const void* q;
    const void* k_pool;
    const void* v_pool;
    const void* k_new;     // [B][Hkv][d] fp16: the token appended this step (NULL: nothing to append)
    const void* v_new;
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;             // fp16 [B][Hq][d] (single-pass only)
    float* ml;             // float2 (m, l) per state
    float* acc;            // float [state][d]
    const pkv_task* tasks;      // workqueue only
    int32_t* row_off;           // workqueue only: the list's first task of each row (written here if list_in_decode)
    int32_t* row_splits;        // workqueue only: S_b per row (the builder's, or written here if list_in_decode)
    uint32_t* counters;         // fused merge: arrivals per (row, KV head), zero between steps
    pkv_ws_header* hdr;
    int32_t B, Hq, Hkv, num_pages, max_pages;
    int32_t chunk_pages, num_splits, variant, num_tasks, task_capacity;
    int32_t fuse_merge;         // 1: the last task of each (row, KV head) merges its states and writes out
    int32_t list_in_decode;     // workqueue: derive the compact list from seq_lens in every CTA
    int32_t overlap_prev;       // launched to overlap the kernel before it: q is read only after griddepcontrol.wait
    int32_t inputs_after_wait;  // launched to overlap the kernel before it: nothing is read before griddepcontrol.wait
    float scale_log2;           // scale * log2(e): scores are kept in base-2 units inside the kernel
};

struct BuildParams {
    const int32_t* seq_lens;
    int32_t* row_off;
    int32_t* row_splits;
    pkv_task* tasks;
    pkv_ws_header* hdr;
    int32_t B, Hkv, max_pages, chunk_pages, task_capacity;
};

struct MergeParams {
    const float* ml;
    const float* acc;
    const int32_t* row_off;
    const int32_t* row_splits;
    void* out;
    uint32_t* status;
    int32_t B, Hq, Hkv, num_splits, variant;
    int32_t task_capacity;  // tasks whose states the workspace holds
};

// Kernel launchers (defined in the .cu files). They return the CUDA error of the launch.
int launch_decode(const DecodeParams& p, int group, int grid, bool pdl, void* stream);
int launch_build(const BuildParams& p, int grid, void* stream);
int launch_merge(const MergeParams& p, void* stream);
// Copies `bytes` (a multiple of 16, both addresses 16-byte aligned) from src to dst on the device; src may be pinned
// host memory through its device-visible address.
int launch_stage_copy(const void* src, void* dst, size_t bytes, void* stream);

// Validation shared by pkv_decode and the step entry points (PKV_OK or a PKV_E_* code; enqueues nothing).
int check_decode_args(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_pool,
                      const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev, float scale,
                      void* ws, size_t ws_bytes, void* out);

// build (workqueue) + decode + merge on one stream after validating every argument up front; with clear_counters
// the workspace's arrival counters are zeroed first; k_new / v_new (both or neither) are appended inside the decode.
int decode_step(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_new, const void* v_new,
                const void* k_pool, const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev,
                float scale, void* ws, size_t ws_bytes, void* out, void* stream, bool clear_counters);

// pkv_decode with the appended token (k_new / v_new may be NULL).
int decode_launch(const pkv_plan_t* plan, const pkv_problem* pr, const void* q, const void* k_new, const void* v_new,
                  const void* k_pool, const void* v_pool, const int32_t* block_table, const int32_t* seq_lens_dev,
                  float scale, void* ws, size_t ws_bytes, void* out, void* stream);

// Dynamic shared memory of the decode kernel for a group size (0 if unsupported).
int decode_smem_bytes(int group);

// Resident decode CTAs per SM the kernel is compiled for (its __launch_bounds__ minimum; the register budget of a
// third CTA does not exist).
constexpr int kDecodeCtasPerSm = 2;

// Shared memory of one SM usable by resident CTAs (sm_103: 228 KB) and the per-CTA reservation.
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemReservedPerCta = 1024;

}  // namespace pkv
