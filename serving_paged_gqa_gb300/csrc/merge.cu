// Log-sum-exp merge of split states (the separate-kernel schedule).
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs", gist.science
// technical summary, "Methodologie" 1, "Sequentie Splitting": each split produces a partial online-softmax state
// and a separate merge kernel combines them exactly. For query head hq of row b with states (m_s, l_s, acc_s):
//   M = max_s m_s over states with l_s > 0,  out = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s.
// Neutral states (empty splits: m = -inf, l = 0) contribute nothing; a row with none gets 0.
//
// One CTA of 16 warps per (b, hq). The states are split across the warps (warp w takes s = w, w + 16, ...); lane k
// owns dimensions 4k..4k+3, so one state is one coalesced 512-byte load per warp. The (m, l) pairs give M in one
// block-wide pass, while the first round of acc loads is already in flight; then each warp accumulates its states
// 8 at a time (all 8 loads issued before use), and the 16 partial sums meet in shared memory. With 128 states in
// flight per CTA a merge of S states costs about 1 + S/128 memory round trips (the merge is latency-bound: its
// states are a few MB). The grid is launched with programmatic stream serialization after the decode and reads the
// states only after griddepcontrol.wait.
#include <cuda_fp16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 16;
constexpr int kRound = 8;  // states per warp whose loads are in flight together
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const MergeParams p) {
    __shared__ float s_max[kWarps];
    __shared__ float4 s_acc[kWarps][32];
    __shared__ float s_den[kWarps];
    // a grid launched after this one to overlap it (a decode of the next layer) may start now: it reads what this
    // grid writes only after waiting for it
    grid_launch_dependents();
    grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pair = blockIdx.x;
    const int b = pair / p.Hq, hq = pair - b * p.Hq;
    const int G = p.Hq / p.Hkv;
    const int h = hq / G, g = hq - h * G;
    int S, base;
    if (p.variant == PKV_VARIANT_WORKQUEUE) {
        S = p.row_splits[b];
        base = p.row_off[b] + h * S;
    } else {
        S = p.num_splits;
        base = (b * p.Hkv + h) * S;
    }
    if (S < 0 || base < 0 || (int64_t)base + S > (int64_t)p.task_capacity) {  // row_off/row_splits not from
        if (tid == 0) atomicOr(p.status, PKV_STATUS_TASKS);                   // this plan: write nothing
        return;
    }
    const float2* mlp = reinterpret_cast<const float2*>(p.ml);
    const float4* accp = reinterpret_cast<const float4*>(p.acc);
    auto state = [&](int s) { return (size_t)(base + s) * G + g; };

    // first round of this warp's states, in flight during the max pass
    float2 ml[kRound];
    float4 v[kRound];
#pragma unroll
    for (int j = 0; j < kRound; ++j) {
        const int s = warp + kWarps * j;
        ml[j] = s < S ? __ldcg(mlp + state(s)) : make_float2(-INFINITY, 0.f);
        v[j] = s < S ? __ldcg(accp + state(s) * (kHeadDim / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float mx = -INFINITY;
    for (int s = tid; s < S; s += kWarps * 32) {
        const float2 t = __ldcg(mlp + state(s));
        if (t.y > 0.f) mx = fmaxf(mx, t.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_max[warp] = mx;
    __syncthreads();
    float M = s_max[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_max[w]);

    __half* out = static_cast<__half*>(p.out) + (size_t)pair * kHeadDim;
    if (M == -INFINITY) {
        if (warp == 0) *reinterpret_cast<uint2*>(out + lane * 4) = make_uint2(0u, 0u);
        return;
    }
    const float M2 = M * kLog2e;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    for (int r = 0;; ++r) {
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            if (ml[j].y > 0.f) {
                const float w = fast_exp2(ml[j].x * kLog2e - M2);
                den += w * ml[j].y;
                a.x += w * v[j].x;
                a.y += w * v[j].y;
                a.z += w * v[j].z;
                a.w += w * v[j].w;
            }
        }
        const int s0 = warp + kWarps * kRound * (r + 1);
        if (s0 >= S) break;
#pragma unroll
        for (int j = 0; j < kRound; ++j) {
            const int s = s0 + kWarps * j;
            ml[j] = s < S ? __ldcg(mlp + state(s)) : make_float2(-INFINITY, 0.f);
            v[j] = s < S ? __ldcg(accp + state(s) * (kHeadDim / 4) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    s_acc[warp][lane] = a;
    if (lane == 0) s_den[warp] = den;
    __syncthreads();
    if (warp == 0) {
        float4 t = s_acc[0][lane];
        float d = s_den[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            const float4 y = s_acc[w][lane];
            t.x += y.x;
            t.y += y.y;
            t.z += y.z;
            t.w += y.w;
            d += s_den[w];
        }
        const float inv = 1.f / d;
        uint2 pk;
        pk.x = pack_half2(t.x * inv, t.y * inv);
        pk.y = pack_half2(t.z * inv, t.w * inv);
        *reinterpret_cast<uint2*>(out + lane * 4) = pk;
    }
}

}  // namespace

int launch_merge(const MergeParams& p, void* stream) {
    const int pairs = p.B * p.Hq;
    if (pairs == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pairs);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

}  // namespace pkv
