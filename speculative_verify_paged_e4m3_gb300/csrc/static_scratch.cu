// static_scratch.cu -- forward pass (partial attention + combine) whose split workspace is a fixed
// device array compiled into this library, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- a plugin inside a host
// application whose device memory is all owned by another framework's allocator, a runtime that
// reserves its memory pool at start-up and forbids allocation afterwards, or a latency-critical
// loop that must never enter the driver's allocator. Such a caller still owns q, the page pools,
// the block table, context lengths, scales, out and lse; only the split workspace moves here.
//
// The array below is kStaticScratchBytes large and every GPU that loads this library keeps it
// until the process exits. Host code cannot use its name as a device address (on the host the
// name refers to a host-side stand-in), so the first call on each device, with that device
// current, looks the address up once with cudaGetSymbolAddress and caches it; make that first
// call before any stream capture. Every call shares the one array. At the start of each call the
// first 16 bytes of its header are cleared on the stream: the status word and the ticket counter
// of the fused merge's grid barrier, so that a call never inherits a count that an earlier,
// timed-out or overlapping fused call left behind. The split state is not cleared: when every
// wait of the kernels completes, each active split is written before the merge reads it. The
// status word is not reported on this path, so a wait that gives up (DFLASH_FLAG_KERNEL_TIMEOUT)
// goes unseen, and out and lse of that call are undefined. Two calls whose kernels overlap on
// the GPU -- on different streams, say -- race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;
// status word (offset 0) and the fused merge's 64-bit grid-barrier ticket counter (offset 8)
constexpr size_t kClearedHeaderBytes = 16;

static __device__ __align__(256) unsigned char g_verify_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices];  // device address of the array, per device ordinal

}  // namespace

extern "C" int dflash_verify_attn_forward_static_scratch(
    const dflash_verify_attn_plan_t* plan, const void* q, const void* k_pool, const void* v_pool,
    const int32_t* block_table, const int32_t* context_lens, const float* k_scale,
    const float* v_scale, void* out, float* lse, void* cuda_stream) {
    if (!plan || plan->version != DFLASH_VERIFY_ATTN_VERSION) return DFLASH_ERR_INVALID_ARGUMENT;
    if (plan->workspace_bytes > kStaticScratchBytes) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        if (!g_scratch_address[dev]) {
            void* p = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&p, g_verify_attn_scratch);
            if (e != cudaSuccess || !p) {
                cudaGetLastError();
                return DFLASH_ERR_CUDA;
            }
            g_scratch_address[dev] = p;
        }
        scratch = g_scratch_address[dev];
    }
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    if (cudaMemsetAsync(scratch, 0, kClearedHeaderBytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH_ERR_CUDA;
    }
    return dflash_verify_attn_forward(plan, q, k_pool, v_pool, block_table, context_lens,
                                      k_scale, v_scale, scratch, kStaticScratchBytes, out, lse,
                                      cuda_stream);
}
