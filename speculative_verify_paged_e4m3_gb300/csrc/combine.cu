// combine.cu -- standalone merge kernels: one CTA of 256 threads per (query row, quarter of the
// head dim, sequence x KV head); the merge itself is combine_item (combine_impl.cuh). A single
// sequence (every KV head owns num_splits slots) and a batch (slots shared out by length) have a
// kernel each, so that the one-sequence kernel carries no slot search.
#include "combine_impl.cuh"

namespace dflash {

// One sequence: every KV head owns num_splits slots, unit h at h * num_splits.
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    __shared__ CombineScratch sh;
    const int h = blockIdx.z;
    int n = p.context_lens[0];
    n = n > p.max_context ? p.max_context : (n < 0 ? 0 : n);
    combine_item(p, blockIdx.x, blockIdx.y, 0, h, threadIdx.x, 0, sh, h * p.num_splits,
                 p.num_splits, n);
}

// Several sequences: the unit's slots follow from every context length (locate_slots).
__global__ void __launch_bounds__(kCombineThreads) combine_batch_kernel(CombineParams p) {
    __shared__ CombineScratch sh;
    const int b = blockIdx.z / p.num_kv_heads, h = blockIdx.z % p.num_kv_heads;
    const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                      p.max_context, p.q_len, blockIdx.z, false);
    combine_item(p, blockIdx.x, blockIdx.y, b, h, threadIdx.x, 0, sh, us.first, us.count, us.n);
}

// Plans with few splits per unit (many units: a batch, whole-model heads) merge a whole row per
// 64 threads instead: one CTA per (4 query rows, unit), each thread one float4 column across
// all of the unit's splits. Same arithmetic as combine_item's final step (maximum, then weighted
// sums in split order), which is all of combine_item when no split lane holds more than one
// split: results are the same bits for up to 16 splits per unit.
constexpr int kRowCols = kHeadDim / 4;                 // 64 float4 columns per row
constexpr int kRowsPerCta = kCombineThreads / kRowCols;  // 4
constexpr int kRowKernelMaxSplits = kCombineSplitLanes;  // 16

template <bool kBatch>
__global__ void __launch_bounds__(kCombineThreads) combine_rows_kernel(CombineParams p) {
    const int unit = blockIdx.y;
    const int r = blockIdx.x * kRowsPerCta + threadIdx.x / kRowCols;
    const int col = threadIdx.x % kRowCols;
    const int b = unit / p.num_kv_heads, h = unit % p.num_kv_heads;
    int first, count, n;
    if constexpr (kBatch) {
        const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                          p.max_context, p.q_len, unit, false);
        first = us.first;
        count = us.count;
        n = us.count > 0 ? us.n : 0;
    } else {
        n = p.context_lens[0];
        n = n > p.max_context ? p.max_context : (n < 0 ? 0 : n);
        first = h * p.num_splits;
        count = p.num_splits;
    }
    if (r >= p.rows) return;  // whole warps: a row is two warps
    const int per = n > 0 ? keys_per_split(n, count, p.tile_keys, p.min_split_keys) : 1;
    const int active = n > 0 ? (n + per - 1) / per : 0;
    const int R = p.rows;
    const float4* acc4 = reinterpret_cast<const float4*>(p.ws_acc);
    float M = -INFINITY;
    for (int s = 0; s < active; ++s)
        M = fmaxf(M, __ldcg(&p.ws_state[(int64_t)(first + s) * R + r]).x);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float Lt = 0.f;
    if (M != -INFINITY) {
        constexpr int kBatchLoads = 8;  // splits whose loads are in flight together
        for (int s0 = 0; s0 < active; s0 += kBatchLoads) {
            float2 st[kBatchLoads];
            float4 a[kBatchLoads];
#pragma unroll
            for (int k = 0; k < kBatchLoads; ++k) {
                const int64_t slot = first + min(s0 + k, active - 1);
                st[k] = __ldcg(&p.ws_state[slot * R + r]);
                a[k] = __ldcg(&acc4[(slot * R + r) * kRowCols + col]);
            }
#pragma unroll
            for (int k = 0; k < kBatchLoads; ++k) {
                if (s0 + k >= active) break;
                const float w = st[k].x == -INFINITY ? 0.f : exp2f(st[k].x - M);
                t.x = fmaf(w, a[k].x, t.x);
                t.y = fmaf(w, a[k].y, t.y);
                t.z = fmaf(w, a[k].z, t.z);
                t.w = fmaf(w, a[k].w, t.w);
                Lt = fmaf(w, st[k].y, Lt);
            }
        }
        t.x /= Lt;
        t.y /= Lt;
        t.z /= Lt;
        t.w /= Lt;
    }
    const int i = r / p.group, g = r % p.group;
    const int64_t orow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * p.group + g;
    __half2* out2 = reinterpret_cast<__half2*>(p.out + orow * kHeadDim + col * 4);
    out2[0] = __floats2half2_rn(t.x, t.y);
    out2[1] = __floats2half2_rn(t.z, t.w);
    if (col == 0) p.lse[orow] = (M == -INFINITY) ? -INFINITY : (M + log2f(Lt)) * kLn2;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int units = p.batch * p.num_kv_heads;
    if (p.num_splits <= kRowKernelMaxSplits) {
        const dim3 grid((p.rows + kRowsPerCta - 1) / kRowsPerCta, units);
        if (p.batch == 1)
            combine_rows_kernel<false><<<grid, kCombineThreads, 0, stream>>>(p);
        else
            combine_rows_kernel<true><<<grid, kCombineThreads, 0, stream>>>(p);
        return cudaGetLastError();
    }
    dim3 grid(p.rows, kHeadDim / (4 * kCombineCols), units);
    if (p.batch == 1)
        combine_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    else
        combine_batch_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
