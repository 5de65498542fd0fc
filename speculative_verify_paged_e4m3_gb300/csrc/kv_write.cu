// kv_write.cu -- the step before verification: the q_len drafted tokens' K and V rows written
// into the paged pools as E4M3 codes (the E4M3 target KV of "[Perf] Add opt-in DFlash2 schedules
// and numerical audits", Test Plan; the pages do not describe the write itself).
//
// Token i of sequence b sits at position n - q_len + i (n = context_lens[b] clamped to
// [0, max_context], as the attention reads it), in slot position % P of page
// block_table[b][position / P]. Each element becomes the E4M3FN code of x / scale: one correctly
// rounded FP32 division, then one conversion rounding to nearest even and saturating to +-448.
// One CTA per (token, KV head), two elements per thread: the work is a few kilobytes, bound by
// launch latency, not bandwidth.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace dflash {

struct KvWriteParams {
    const __half* k_new;  // [B, q_len, Hkv, D]
    const __half* v_new;
    const int32_t* block_table;
    const int32_t* context_lens;
    const float* k_scale;
    const float* v_scale;
    uint8_t* k_pool;  // [num_pages, P, Hkv, D]
    uint8_t* v_pool;
    int32_t* status;
    int q_len, num_kv_heads, page_size, max_pages_per_seq, num_pages, max_context;
};

constexpr int kKvWriteThreads = kHeadDim / 2;

__global__ void __launch_bounds__(kKvWriteThreads) kv_write_kernel(KvWriteParams p) {
    const int b = blockIdx.x / p.q_len, i = blockIdx.x % p.q_len, h = blockIdx.y;
    int n = p.context_lens[b];
    int flags = 0;
    if (n > p.max_context) {
        n = p.max_context;
        flags |= DFLASH_FLAG_CONTEXT_CLAMPED;
    }
    n = n < 0 ? 0 : n;
    const int pos = n - p.q_len + i;
    int page = -1;
    if (pos < 0) {
        flags |= DFLASH_FLAG_CONTEXT_SHORT;  // no slot before the sequence start: not written
    } else {
        page = p.block_table[(int64_t)b * p.max_pages_per_seq + pos / p.page_size];
        if (page < 0 || page >= p.num_pages) {
            flags |= DFLASH_FLAG_PAGE_CLAMPED;  // would land outside the pool: not written
            page = -1;
        }
    }
    if (flags && threadIdx.x == 0 && h == 0) atomicOr(p.status, flags);
    if (page < 0) return;
    const int64_t src = (((int64_t)b * p.q_len + i) * p.num_kv_heads + h) * kHeadDim;
    const int64_t dst =
        (((int64_t)page * p.page_size + pos % p.page_size) * p.num_kv_heads + h) * kHeadDim;
    const float ks = *p.k_scale, vs = *p.v_scale;
    const int t = threadIdx.x;
    const float2 kx = __half22float2(reinterpret_cast<const __half2*>(p.k_new + src)[t]);
    const float2 vx = __half22float2(reinterpret_cast<const __half2*>(p.v_new + src)[t]);
    reinterpret_cast<uint16_t*>(p.k_pool + dst)[t] =
        ptx::f32x2_to_e4m3x2(__fdiv_rn(kx.x, ks), __fdiv_rn(kx.y, ks));
    reinterpret_cast<uint16_t*>(p.v_pool + dst)[t] =
        ptx::f32x2_to_e4m3x2(__fdiv_rn(vx.x, vs), __fdiv_rn(vx.y, vs));
}

cudaError_t launch_kv_write(const dflash_verify_attn_plan_t* plan, const void* k_new,
                            const void* v_new, const int32_t* block_table,
                            const int32_t* context_lens, const float* k_scale,
                            const float* v_scale, void* k_pool, void* v_pool, int32_t* status,
                            cudaStream_t stream) {
    const dflash_verify_attn_problem& pr = plan->problem;
    KvWriteParams p;
    p.k_new = static_cast<const __half*>(k_new);
    p.v_new = static_cast<const __half*>(v_new);
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_pool = static_cast<uint8_t*>(k_pool);
    p.v_pool = static_cast<uint8_t*>(v_pool);
    p.status = status;
    p.q_len = pr.q_len;
    p.num_kv_heads = pr.num_kv_heads;
    p.page_size = pr.page_size;
    p.max_pages_per_seq = pr.max_pages_per_seq;
    p.num_pages = pr.num_pages;
    p.max_context = pr.max_context;
    const dim3 grid(pr.batch * pr.q_len, pr.num_kv_heads);
    kv_write_kernel<<<grid, kKvWriteThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dflash
