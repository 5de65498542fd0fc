// combine.cu -- standalone merge kernel: one CTA of 256 threads per (query row, quarter of the
// head dim, sequence x KV head); the merge itself is combine_item (combine_impl.cuh).
#include "combine_impl.cuh"

namespace dflash {

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(CombineParams p) {
    __shared__ CombineScratch sh;
    const int b = blockIdx.z / p.num_kv_heads, h = blockIdx.z % p.num_kv_heads;
    combine_item(p, blockIdx.x, blockIdx.y, b, h, threadIdx.x, 0, sh);
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    dim3 grid(p.rows, kHeadDim / (4 * kCombineCols), p.batch * p.num_kv_heads);
    combine_kernel<<<grid, kCombineThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
