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
    const int32_t* block_table;
    const int32_t* seq_lens;
    void* out;             // fp16 [B][Hq][d] (single-pass only)
    float* ml;             // float2 (m, l) per state
    float* acc;            // float [state][d]
    const pkv_task* tasks; // workqueue only
    pkv_ws_header* hdr;
    int32_t B, Hq, Hkv, num_pages, max_pages;
    int32_t chunk_pages, num_splits, variant, num_tasks, task_capacity;
    float scale_log2;      // scale * log2(e): scores are kept in base-2 units inside the kernel
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
int launch_decode(const DecodeParams& p, int group, int grid, void* stream);
int launch_build(const BuildParams& p, int grid, void* stream);
int launch_merge(const MergeParams& p, void* stream);

// Dynamic shared memory of the decode kernel for a group size (0 if unsupported).
int decode_smem_bytes(int group);

}  // namespace pkv
