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

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    dim3 grid(p.rows, kHeadDim / (4 * kCombineCols), p.batch * p.num_kv_heads);
    if (p.batch == 1)
        combine_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    else
        combine_batch_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
