// combine.cu -- merge per-split FP32 state into FP16 output and FP32 log-sum-exp.
//
// The pages pair every grouped q8 attention kernel with one combine kernel ("[Perf] Reduce
// DFlash2 attention cost and screen exact QK reuse", Test Result). For query row r the active
// splits s carry (m_s, l_s, acc_s) with m in log2 units:
//   M = max_s m_s, L = sum_s 2^{m_s - M} l_s, out = sum_s 2^{m_s - M} acc_s / L,
//   lse = (M + log2 L) * ln 2.
// One CTA per (query row, quarter of the head dim, sequence x KV head): 256 threads = 16 split
// lanes x 16 float4 columns, so the splits are read in parallel (16 at a time, each a coalesced
// 256-byte row segment) and reduced through shared memory.
#include <math.h>

#include "common.cuh"

namespace dflash {

constexpr int kCombineThreads = 256;
constexpr int kCombineSplitLanes = 16;  // splits in flight per CTA
constexpr int kCombineCols = 16;        // float4 columns per CTA (64 head-dim elements)

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    __shared__ float4 part[kCombineSplitLanes][kCombineCols];
    __shared__ float red[kCombineThreads / 32];
    __shared__ float lpart[kCombineSplitLanes];
    const int r = blockIdx.x, quarter = blockIdx.y;
    const int b = blockIdx.z / p.num_kv_heads, h = blockIdx.z % p.num_kv_heads;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = tid / kCombineCols, col = tid % kCombineCols;
    int unused_flags;
    const int n = clamped_context(p.context_lens, b, p.max_context, &unused_flags);
    const int per = keys_per_split(n, p.num_splits, p.tile_keys, p.min_split_keys);
    const int active = n > 0 ? (n + per - 1) / per : 0;
    const int64_t base = ((int64_t)b * p.num_kv_heads + h) * p.num_splits;
    const int R = p.rows;

    // M = max over the active splits
    float M = -INFINITY;
    for (int s = tid; s < active; s += kCombineThreads) M = fmaxf(M, p.ws_state[(base + s) * R + r].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, red[w]);

    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        const float4* acc4 = reinterpret_cast<const float4*>(p.ws_acc);
        for (int s = sl; s < active; s += kCombineSplitLanes) {
            const float2 st = p.ws_state[(base + s) * R + r];
            if (st.x == -INFINITY) continue;
            const float w = exp2f(st.x - M);
            L = fmaf(w, st.y, L);
            const float4 a = acc4[((base + s) * R + r) * (kHeadDim / 4) + quarter * kCombineCols + col];
            o.x = fmaf(w, a.x, o.x);
            o.y = fmaf(w, a.y, o.y);
            o.z = fmaf(w, a.z, o.z);
            o.w = fmaf(w, a.w, o.w);
        }
    }
    part[sl][col] = o;
    if (col == 0) lpart[sl] = L;
    __syncthreads();
    if (tid < kCombineCols) {
        float4 t = part[0][tid];
        float Lt = lpart[0];
#pragma unroll
        for (int k = 1; k < kCombineSplitLanes; ++k) {
            const float4 q = part[k][tid];
            t.x += q.x;
            t.y += q.y;
            t.z += q.z;
            t.w += q.w;
            Lt += lpart[k];
        }
        if (M != -INFINITY) {
            t.x /= Lt;
            t.y /= Lt;
            t.z /= Lt;
            t.w /= Lt;
        }
        const int i = r / p.group, g = r % p.group;
        const int64_t orow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * p.group + g;
        __half2* out2 =
            reinterpret_cast<__half2*>(p.out + orow * kHeadDim + (quarter * kCombineCols + tid) * 4);
        out2[0] = __floats2half2_rn(t.x, t.y);
        out2[1] = __floats2half2_rn(t.z, t.w);
        if (quarter == 0 && tid == 0)
            p.lse[orow] = (M == -INFINITY) ? -INFINITY : (M + log2f(Lt)) * kLn2;
    }
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    dim3 grid(p.rows, kHeadDim / (4 * kCombineCols), p.batch * p.num_kv_heads);
    combine_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
