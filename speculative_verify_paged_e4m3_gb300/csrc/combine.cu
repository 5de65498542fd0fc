// combine.cu -- merge per-split FP32 state into FP16 output and FP32 log-sum-exp.
//
// The pages pair every grouped q8 attention kernel with one combine kernel ("[Perf] Reduce
// DFlash2 attention cost and screen exact QK reuse", Test Result). For query row r the active
// splits s carry (m_s, l_s, acc_s) with m in log2 units:
//   M = max_s m_s, L = sum_s 2^{m_s - M} l_s, out = sum_s 2^{m_s - M} acc_s / L,
//   lse = (M + log2 L) * ln 2.
// One CTA per (query row, sequence x KV head); each of its 64 threads owns four head-dim
// elements, so a split's numerator row is one coalesced 1 KB read.
#include <math.h>

#include "common.cuh"

namespace dflash {

constexpr int kCombineThreads = kHeadDim / 4;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    const int r = blockIdx.x;
    const int b = blockIdx.y / p.num_kv_heads, h = blockIdx.y % p.num_kv_heads;
    const int tid = threadIdx.x;
    int unused_flags;
    const int n = clamped_context(p.context_lens, b, p.max_context, &unused_flags);
    const int per = keys_per_split(n, p.num_splits, p.tile_keys, p.min_split_keys);
    const int active = n > 0 ? (n + per - 1) / per : 0;
    const int64_t base = ((int64_t)b * p.num_kv_heads + h) * p.num_splits;
    const int R = p.rows;

    float M = -INFINITY;
    for (int s = 0; s < active; ++s) M = fmaxf(M, p.ws_state[(base + s) * R + r].x);

    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        const float4* acc4 = reinterpret_cast<const float4*>(p.ws_acc);
        for (int s = 0; s < active; ++s) {
            const float2 st = p.ws_state[(base + s) * R + r];
            if (st.x == -INFINITY) continue;
            const float w = exp2f(st.x - M);
            L = fmaf(w, st.y, L);
            const float4 a = acc4[((base + s) * R + r) * (kHeadDim / 4) + tid];
            o.x = fmaf(w, a.x, o.x);
            o.y = fmaf(w, a.y, o.y);
            o.z = fmaf(w, a.z, o.z);
            o.w = fmaf(w, a.w, o.w);
        }
        o.x /= L;
        o.y /= L;
        o.z /= L;
        o.w /= L;
    }
    const int i = r / p.group, g = r % p.group;
    const int64_t orow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * p.group + g;
    __half2* out2 = reinterpret_cast<__half2*>(p.out + orow * kHeadDim + tid * 4);
    out2[0] = __floats2half2_rn(o.x, o.y);
    out2[1] = __floats2half2_rn(o.z, o.w);
    if (tid == 0) p.lse[orow] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    dim3 grid(p.rows, p.batch * p.num_kv_heads);
    combine_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
