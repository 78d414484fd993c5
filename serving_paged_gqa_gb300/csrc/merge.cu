// Log-sum-exp merge of split states.
//
// "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs", gist.science
// technical summary, "Methodologie" 1, "Sequentie Splitting": each split produces a partial online-softmax state
// and a separate merge kernel combines them exactly. For query head hq of row b with states (m_s, l_s, acc_s):
//   M = max_s m_s over states with l_s > 0,  out = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s.
// Neutral states (empty splits: m = -inf, l = 0) contribute nothing; a row with none gets 0.
// One CTA of 8 warps per (b, hq): the CTA reduces M, then warp w takes states w, w+8, ..., lane k the four
// dimensions 4k..4k+3 (one 16-byte load per state), and warp 0 adds the eight partial sums.
#include <cuda_fp16.h>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 8;
constexpr float kLog2e = 1.4426950408889634f;

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const MergeParams p) {
    __shared__ float s_max[kWarps];
    __shared__ float4 s_acc[kWarps][32];
    __shared__ float s_den[kWarps];
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
    const float2* ml = reinterpret_cast<const float2*>(p.ml);
    const float4* acc = reinterpret_cast<const float4*>(p.acc);

    float mx = -INFINITY;
    for (int s = tid; s < S; s += kWarps * 32) {
        const float2 v = ml[(size_t)(base + s) * G + g];
        if (v.y > 0.f) mx = fmaxf(mx, v.x);
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
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
#pragma unroll 4
    for (int s = warp; s < S; s += kWarps) {
        const size_t st = (size_t)(base + s) * G + g;
        const float2 v = ml[st];
        const float4 x = acc[st * (kHeadDim / 4) + lane];
        const float f = v.y > 0.f ? fast_exp2((v.x - M) * kLog2e) : 0.f;
        den += f * v.y;
        a.x += f * x.x;
        a.y += f * x.y;
        a.z += f * x.z;
        a.w += f * x.w;
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
    merge_kernel<<<pairs, kWarps * 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
