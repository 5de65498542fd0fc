// api.cu -- the C ABI: planner, argument checks, launches, debug export, status text.
//
// The split planner replaces the pages' fixed "80 logical splits" ("[Perf] Reduce DFlash2
// long-context verification decay", Implementation; 80 matched the V100's SM count) with a split
// count sized to this GPU's SMs, and a per-call rule that adapts the split length to the context
// length read on the device.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include <vector>

#include "common.cuh"
#include "e4m3.cuh"

namespace dflash {
cudaError_t launch_simt_partial(const PartialParams& p, cudaStream_t stream);
cudaError_t launch_tc_partial(const PartialParams& p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
cudaError_t launch_kv_write(const dflash_verify_attn_plan_t* plan, const void* k_new,
                            const void* v_new, const int32_t* block_table,
                            const int32_t* context_lens, const float* k_scale,
                            const float* v_scale, void* k_pool, void* v_pool, int32_t* status,
                            cudaStream_t stream);
size_t simt_smem_bytes();
size_t tc_smem_bytes(int rows);
int tc_threads(int rows);
bool tc_supports(int rows);
int tc_max_rows();
int simt_max_rows();
}  // namespace dflash

using namespace dflash;

namespace {

constexpr int kDefaultSmCount = 152;  // GB300
constexpr size_t kHeaderBytes = 256;
constexpr size_t kGridBarrierOffset = 8;  // 64-bit ticket counter of the fused merge's barrier

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int host_keys_per_split(int n, const dflash_verify_attn_plan_t* plan) {
    int64_t per = ceil_div(n, plan->num_splits);
    if (per < plan->min_split_keys) per = plan->min_split_keys;
    return (int)(ceil_div(per, plan->tile_keys) * plan->tile_keys);
}

int check_plan(const dflash_verify_attn_plan_t* plan) {
    if (!plan || plan->version != DFLASH_VERIFY_ATTN_VERSION) return DFLASH_ERR_INVALID_ARGUMENT;
    if (plan->num_splits < 1 || plan->tile_keys < 1 || plan->rows < 1 || plan->row_blocks < 1 ||
        plan->row_blocks > plan->rows)
        return DFLASH_ERR_INVALID_ARGUMENT;
    // slots: Hkv * num_splits for a single sequence (the grid (S, Hkv, 1)); at least one per
    // unit for a batch
    const int64_t units = (int64_t)plan->problem.batch * plan->problem.num_kv_heads;
    if (plan->problem.batch < 1 || plan->problem.num_kv_heads < 1)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (plan->problem.batch == 1 ? plan->num_slots != units * plan->num_splits
                                 : plan->num_slots < units)
        return DFLASH_ERR_INVALID_ARGUMENT;
    // the kernels' tile sizes are compile-time constants: split boundaries fall on their tiles
    if (plan->tile_keys != (plan->kernel == DFLASH_KERNEL_TCGEN05 ? 128 : 32) ||
        plan->min_split_keys % plan->tile_keys != 0)
        return DFLASH_ERR_INVALID_ARGUMENT;
    // every row block holds 1..capacity rows of the plan's kernel
    const int64_t block_rows = ceil_div(plan->rows, plan->row_blocks);
    const int capacity = plan->kernel == DFLASH_KERNEL_TCGEN05 ? tc_max_rows() : simt_max_rows();
    if (block_rows > capacity || (plan->row_blocks - 1) * block_rows >= plan->rows)
        return DFLASH_ERR_INVALID_ARGUMENT;
    return DFLASH_OK;
}

PartialParams partial_params(const dflash_verify_attn_plan_t* plan, const void* q,
                             const void* k_pool, const void* v_pool, const int32_t* block_table,
                             const int32_t* context_lens, const float* k_scale,
                             const float* v_scale, void* workspace) {
    const dflash_verify_attn_problem& pr = plan->problem;
    PartialParams p;
    p.q = static_cast<const __half*>(q);
    p.k_pool = static_cast<const uint8_t*>(k_pool);
    p.v_pool = static_cast<const uint8_t*>(v_pool);
    p.block_table = block_table;
    p.context_lens = context_lens;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    char* ws = static_cast<char*>(workspace);
    p.status = reinterpret_cast<int32_t*>(ws);
    p.ws_state = reinterpret_cast<float2*>(ws + plan->ws_state_offset);
    p.ws_acc = reinterpret_cast<float*>(ws + plan->ws_acc_offset);
    p.batch = pr.batch;
    p.q_len = pr.q_len;
    p.num_q_heads = pr.num_q_heads;
    p.num_kv_heads = pr.num_kv_heads;
    p.group = pr.num_q_heads / pr.num_kv_heads;
    p.rows = plan->rows;
    p.row_blocks = plan->row_blocks;
    p.block_rows = (int)ceil_div(plan->rows, plan->row_blocks);
    p.page_size = pr.page_size;
    p.max_pages_per_seq = pr.max_pages_per_seq;
    p.num_pages = pr.num_pages;
    p.max_context = pr.max_context;
    p.num_splits = plan->num_splits;
    p.num_slots = plan->num_slots;
    p.tile_keys = plan->tile_keys;
    p.min_split_keys = plan->min_split_keys;
    p.grid_bar = reinterpret_cast<unsigned long long*>(ws + kGridBarrierOffset);
    p.out = nullptr;  // partial state only; forward() sets these for a fused launch
    p.lse = nullptr;
    p.pdl = (pr.flags & DFLASH_PROBLEM_PDL) && !plan->combine_fused ? 1 : 0;
    p.per_max = host_keys_per_split(pr.max_context, plan);
    p.page_shift = -1;
    for (int s = 0; s < 31; ++s)
        if (pr.page_size == (1 << s)) p.page_shift = s;
    return p;
}

}  // namespace

extern "C" {

const char* dflash_verify_attn_status_string(int status) {
    switch (status) {
        case DFLASH_OK: return "ok";
        case DFLASH_ERR_INVALID_ARGUMENT: return "invalid argument";
        case DFLASH_ERR_UNSUPPORTED: return "unsupported shape or kernel";
        case DFLASH_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case DFLASH_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int dflash_verify_attn_plan(const dflash_verify_attn_problem* pr,
                            dflash_verify_attn_plan_t* plan) {
    if (!pr || !plan) return DFLASH_ERR_INVALID_ARGUMENT;
    if (pr->version != DFLASH_VERIFY_ATTN_VERSION) return DFLASH_ERR_INVALID_ARGUMENT;
    if (pr->batch < 1 || pr->q_len < 1 || pr->num_q_heads < 1 || pr->num_kv_heads < 1 ||
        pr->head_dim < 1 || pr->page_size < 1 || pr->max_pages_per_seq < 1 ||
        pr->num_pages < 1 || pr->max_context < 1 || pr->num_splits < 0)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (pr->num_q_heads % pr->num_kv_heads != 0) return DFLASH_ERR_INVALID_ARGUMENT;
    if ((int64_t)pr->max_pages_per_seq * pr->page_size < pr->max_context)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (pr->kernel < DFLASH_KERNEL_AUTO || pr->kernel > DFLASH_KERNEL_TCGEN05)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (pr->head_dim != kHeadDim) return DFLASH_ERR_UNSUPPORTED;
    if (pr->page_size % 16 != 0) return DFLASH_ERR_UNSUPPORTED;
    const int group = pr->num_q_heads / pr->num_kv_heads;
    const int64_t rows = (int64_t)pr->q_len * group;
    if (rows > kMaxRows) return DFLASH_ERR_UNSUPPORTED;
    // More rows than one CTA of the chosen kernel carries: the rows are dealt into row blocks of
    // ceil(R / blocks) each, every block a CTA of its own over the same split (the split count
    // shrinks by the same factor, so the grid stays one wave).
    const int tc_blocks = (int)ceil_div(rows, tc_max_rows());
    const int tc_block_rows = (int)ceil_div(rows, tc_blocks);
    const bool tc_ok = tc_supports(tc_block_rows);
    if (pr->kernel == DFLASH_KERNEL_TCGEN05 && !tc_ok) return DFLASH_ERR_UNSUPPORTED;
    const bool use_tc = tc_ok && pr->kernel != DFLASH_KERNEL_SIMT;
    const int row_blocks = use_tc ? tc_blocks : (int)ceil_div(rows, simt_max_rows());
    const int block_rows = (int)ceil_div(rows, row_blocks);

    int sm_count = kDefaultSmCount;
    if (pr->device >= 0) {
        if (cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, pr->device) !=
            cudaSuccess) {
            cudaGetLastError();
            return DFLASH_ERR_CUDA;
        }
    }

    memset(plan, 0, sizeof(*plan));
    plan->version = DFLASH_VERIFY_ATTN_VERSION;
    if (use_tc) {
        plan->kernel = DFLASH_KERNEL_TCGEN05;
        plan->tile_keys = 128;
        plan->min_split_keys = 256;
        plan->threads = tc_threads(block_rows);
        plan->smem_bytes = (int32_t)tc_smem_bytes(block_rows);
    } else {
        plan->kernel = DFLASH_KERNEL_SIMT;
        plan->tile_keys = 32;
        plan->min_split_keys = 256;
        plan->threads = 256;
        plan->smem_bytes = (int32_t)simt_smem_bytes();
    }
    const int64_t units = (int64_t)pr->batch * pr->num_kv_heads;
    const int64_t ctas_per_split = units * row_blocks;  // CTAs per split index
    // On request the tensor-core kernel merges the splits itself (one launch per forward), which
    // needs its whole grid on the GPU at once (one CTA per SM): the split count is then kept to
    // floor(SMs / (units * row blocks)).
    const bool fuse = use_tc && (pr->flags & DFLASH_PROBLEM_FUSED_COMBINE) &&
                      ctas_per_split <= sm_count &&
                      (pr->num_splits == 0 || ctas_per_split * pr->num_splits <= sm_count);
    int64_t S = pr->num_splits;
    if (S == 0 && fuse) {
        S = sm_count / ctas_per_split;
        const int64_t cap = ceil_div(pr->max_context, plan->min_split_keys);
        if (S > cap) S = cap;
    } else if (S == 0) {
        // one wave of single-CTA-per-SM work: units * row blocks * S <= SMs (a CTA past the SM
        // count would wait for a second wave and double the launch time)
        S = ctas_per_split < sm_count ? sm_count / ctas_per_split : 1;
        const int64_t cap = ceil_div(pr->max_context, plan->min_split_keys);
        if (S > cap) S = cap;
    }
    if (S < 1) S = 1;
    if (S > 65535) return DFLASH_ERR_UNSUPPORTED;
    // Workspace slots. A single sequence, or a forced split count: units * S, the grid
    // (S, Hkv, batch). A batch on the planner's split count: every SM's worth of slots (over the
    // row blocks), shared out among the units by length at run time, so that units * S rounding
    // leaves no SM idle.
    int64_t slots = units * S;
    if (pr->batch > 1 && pr->num_splits == 0) {
        int64_t all = sm_count / row_blocks;
        const int64_t cap = units * ceil_div(pr->max_context, plan->min_split_keys);
        if (all > cap) all = cap;
        if (all > slots) slots = all;
    }
    if (slots * row_blocks > 0x7FFFFFFF) return DFLASH_ERR_UNSUPPORTED;
    plan->num_splits = (int32_t)S;
    plan->num_slots = (int32_t)slots;
    plan->combine_fused = fuse ? 1 : 0;
    plan->rows = (int32_t)rows;
    plan->row_blocks = row_blocks;
    plan->sm_count = sm_count;
    const size_t state_bytes = (size_t)slots * rows * sizeof(float2);
    const size_t acc_bytes = (size_t)slots * rows * kHeadDim * sizeof(float);
    plan->ws_state_offset = kHeaderBytes;
    plan->ws_acc_offset = kHeaderBytes + align_up(state_bytes, 256);
    plan->workspace_bytes = plan->ws_acc_offset + acc_bytes;
    plan->problem = *pr;
    return DFLASH_OK;
}

int dflash_verify_attn_split_slots(const dflash_verify_attn_plan_t* plan,
                                   const int32_t* context_lens, int32_t* slot_start,
                                   int32_t* keys_per_split, int32_t* active) {
    int rc = check_plan(plan);
    if (rc != DFLASH_OK) return rc;
    if (!context_lens || !slot_start || !keys_per_split || !active)
        return DFLASH_ERR_INVALID_ARGUMENT;
    const dflash_verify_attn_problem& pr = plan->problem;
    const int B = pr.batch, Hkv = pr.num_kv_heads;
    const int64_t S = plan->num_splits;
    std::vector<int64_t> n(B), w(B);
    int64_t W = 0, wmax = 0;
    for (int b = 0; b < B; ++b) {
        int64_t nb = context_lens[b];
        nb = nb > pr.max_context ? pr.max_context : nb;
        nb = nb < 0 ? 0 : nb;
        n[b] = nb;
        w[b] = (nb + 127) / 128;
        W += w[b];
        wmax = w[b] > wmax ? w[b] : wmax;
    }
    // slots per KV head of each sequence (common.cuh, locate_slots): num_splits for a single
    // sequence; for a batch c_b = ceil(w_b / T), T the smallest tile count per split with
    // Hkv * sum_b ceil(w_b / T) <= num_slots
    std::vector<int64_t> c(B, 0);
    if (W > 0 && B == 1) {
        c[0] = S;
    } else if (W > 0) {
        const int64_t C = plan->num_slots;
        int64_t lo = 1, hi = wmax;  // T = wmax leaves one slot per non-empty unit: Hkv E <= C
        while (lo < hi) {
            const int64_t mid = (lo + hi) / 2;
            int64_t need = 0;
            for (int b = 0; b < B; ++b) need += ceil_div(w[b], mid);
            if (need * Hkv <= C)
                hi = mid;
            else
                lo = mid + 1;
        }
        for (int b = 0; b < B; ++b) c[b] = ceil_div(w[b], lo);
    }
    int64_t before = 0;
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) slot_start[b * Hkv + h] = (int32_t)(Hkv * before + h * c[b]);
        before += c[b];
    }
    slot_start[B * Hkv] = (int32_t)(Hkv * before);
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < Hkv; ++h) {
            const int u = b * Hkv + h;
            const int64_t cnt = slot_start[u + 1] - slot_start[u];
            if (n[b] == 0 || cnt == 0) {
                keys_per_split[u] = 0;
                active[u] = 0;
                continue;
            }
            int64_t per = ceil_div(n[b], cnt);
            if (per < plan->min_split_keys) per = plan->min_split_keys;
            per = ceil_div(per, plan->tile_keys) * plan->tile_keys;
            keys_per_split[u] = (int32_t)per;
            active[u] = (int32_t)ceil_div(n[b], per);
        }
    }
    return DFLASH_OK;
}

int dflash_verify_attn_split_bounds(const dflash_verify_attn_plan_t* plan, int32_t n,
                                    int32_t* starts, int32_t* active) {
    int rc = check_plan(plan);
    if (rc != DFLASH_OK) return rc;
    if (!starts || !active) return DFLASH_ERR_INVALID_ARGUMENT;
    if (n > plan->problem.max_context) n = plan->problem.max_context;
    if (n < 0) n = 0;
    const int per = host_keys_per_split(n, plan);
    for (int s = 0; s <= plan->num_splits; ++s) {
        int64_t st = (int64_t)s * per;
        starts[s] = (int32_t)(st < n ? st : n);
    }
    *active = n > 0 ? (int32_t)ceil_div(n, per) : 0;
    return DFLASH_OK;
}

int dflash_verify_attn_run(const dflash_verify_attn_plan_t* plan, const void* q,
                           const void* k_pool, const void* v_pool, const int32_t* block_table,
                           const int32_t* context_lens, const float* k_scale,
                           const float* v_scale, void* workspace, size_t workspace_bytes,
                           void* cuda_stream) {
    int rc = check_plan(plan);
    if (rc != DFLASH_OK) return rc;
    if (!q || !k_pool || !v_pool || !block_table || !context_lens || !k_scale || !v_scale ||
        !workspace)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
        !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(context_lens, 4))
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < plan->workspace_bytes) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
    const PartialParams p = partial_params(plan, q, k_pool, v_pool, block_table, context_lens,
                                           k_scale, v_scale, workspace);
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    cudaError_t e;
    if (plan->kernel == DFLASH_KERNEL_SIMT)
        e = launch_simt_partial(p, stream);
    else if (plan->kernel == DFLASH_KERNEL_TCGEN05)
        e = launch_tc_partial(p, stream);
    else
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return DFLASH_ERR_CUDA;
    }
    return DFLASH_OK;
}

int dflash_verify_attn_kv_write(const dflash_verify_attn_plan_t* plan, const void* k_new,
                                const void* v_new, const int32_t* block_table,
                                const int32_t* context_lens, const float* k_scale,
                                const float* v_scale, void* k_pool, void* v_pool,
                                void* workspace, size_t workspace_bytes, void* cuda_stream) {
    int rc = check_plan(plan);
    if (rc != DFLASH_OK) return rc;
    if (!k_new || !v_new || !block_table || !context_lens || !k_scale || !v_scale || !k_pool ||
        !v_pool || !workspace)
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (!aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(k_pool, 2) || !aligned(v_pool, 2) ||
        !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(context_lens, 4))
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < plan->workspace_bytes) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
    if (plan->problem.batch * plan->problem.q_len == 0) return DFLASH_OK;
    if (launch_kv_write(plan, k_new, v_new, block_table, context_lens, k_scale, v_scale, k_pool,
                        v_pool, static_cast<int32_t*>(workspace),
                        static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH_ERR_CUDA;
    }
    return DFLASH_OK;
}

int dflash_verify_attn_combine(const dflash_verify_attn_plan_t* plan, const void* workspace,
                               size_t workspace_bytes, const int32_t* context_lens, void* out,
                               float* lse, void* cuda_stream) {
    int rc = check_plan(plan);
    if (rc != DFLASH_OK) return rc;
    if (!workspace || !context_lens || !out || !lse) return DFLASH_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256) || !aligned(out, 8) || !aligned(lse, 4))
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (workspace_bytes < plan->workspace_bytes) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
    const dflash_verify_attn_problem& pr = plan->problem;
    const char* ws = static_cast<const char*>(workspace);
    CombineParams c;
    c.ws_state = reinterpret_cast<const float2*>(ws + plan->ws_state_offset);
    c.ws_acc = reinterpret_cast<const float*>(ws + plan->ws_acc_offset);
    c.context_lens = context_lens;
    c.out = static_cast<__half*>(out);
    c.lse = lse;
    c.batch = pr.batch;
    c.q_len = pr.q_len;
    c.num_q_heads = pr.num_q_heads;
    c.num_kv_heads = pr.num_kv_heads;
    c.group = pr.num_q_heads / pr.num_kv_heads;
    c.rows = plan->rows;
    c.max_context = pr.max_context;
    c.num_splits = plan->num_splits;
    c.num_slots = plan->num_slots;
    c.tile_keys = plan->tile_keys;
    c.min_split_keys = plan->min_split_keys;
    c.pdl = (pr.flags & DFLASH_PROBLEM_PDL) && !plan->combine_fused ? 1 : 0;
    if (launch_combine(c, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
        cudaGetLastError();
        return DFLASH_ERR_CUDA;
    }
    return DFLASH_OK;
}

int dflash_verify_attn_forward(const dflash_verify_attn_plan_t* plan, const void* q,
                               const void* k_pool, const void* v_pool,
                               const int32_t* block_table, const int32_t* context_lens,
                               const float* k_scale, const float* v_scale, void* workspace,
                               size_t workspace_bytes, void* out, float* lse, void* cuda_stream) {
    if (plan && plan->combine_fused) {
        int rc = check_plan(plan);
        if (rc != DFLASH_OK) return rc;
        if (plan->kernel != DFLASH_KERNEL_TCGEN05) return DFLASH_ERR_INVALID_ARGUMENT;
        if (!q || !k_pool || !v_pool || !block_table || !context_lens || !k_scale || !v_scale ||
            !workspace || !out || !lse)
            return DFLASH_ERR_INVALID_ARGUMENT;
        if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) ||
            !aligned(workspace, 256) || !aligned(block_table, 4) || !aligned(context_lens, 4) ||
            !aligned(out, 8) || !aligned(lse, 4))
            return DFLASH_ERR_INVALID_ARGUMENT;
        if (workspace_bytes < plan->workspace_bytes) return DFLASH_ERR_WORKSPACE_TOO_SMALL;
        PartialParams p = partial_params(plan, q, k_pool, v_pool, block_table, context_lens,
                                         k_scale, v_scale, workspace);
        p.pdl = 0;  // the cooperative fused launch is never a programmatic dependent
        p.out = static_cast<__half*>(out);
        p.lse = lse;
        if (launch_tc_partial(p, static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess) {
            cudaGetLastError();
            return DFLASH_ERR_CUDA;
        }
        return DFLASH_OK;
    }
    int rc = dflash_verify_attn_run(plan, q, k_pool, v_pool, block_table, context_lens, k_scale,
                                    v_scale, workspace, workspace_bytes, cuda_stream);
    if (rc != DFLASH_OK) return rc;
    return dflash_verify_attn_combine(plan, workspace, workspace_bytes, context_lens, out, lse,
                                      cuda_stream);
}

}  // extern "C"

namespace dflash {

__global__ void debug_dequant_kernel(const uint8_t* codes, int64_t n, const float* scale,
                                     float* decoded, float* scaled) {
    // pairs of consecutive codes go through the same two-code conversion the kernels use
    const float sc = scaled ? __ldg(scale) : 0.f;
    const int64_t pairs = (n + 1) / 2;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < pairs;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i0 = 2 * t;
        const bool two = i0 + 1 < n;
        const uint16_t c = static_cast<uint16_t>(codes[i0] | (two ? codes[i0 + 1] << 8 : 0));
        const uint32_t f = e4m3x2_to_f16x2(c);
        const float v0 = __half2float(__ushort_as_half(static_cast<unsigned short>(f & 0xFFFFu)));
        const float v1 = __half2float(__ushort_as_half(static_cast<unsigned short>(f >> 16)));
        decoded[i0] = v0;
        if (scaled) scaled[i0] = __fmul_rn(v0, sc);
        if (two) {
            decoded[i0 + 1] = v1;
            if (scaled) scaled[i0 + 1] = __fmul_rn(v1, sc);
        }
    }
}

}  // namespace dflash

extern "C" int dflash_verify_attn_debug_dequant(const uint8_t* codes, int64_t n,
                                                const float* scale, float* decoded,
                                                float* scaled, void* cuda_stream) {
    if (n < 0 || (n > 0 && (!codes || !decoded)) || (scaled && !scale))
        return DFLASH_ERR_INVALID_ARGUMENT;
    if (n == 0) return DFLASH_OK;
    int64_t blocks = ((n + 1) / 2 + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    debug_dequant_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
        codes, n, scale, decoded, scaled);
    if (cudaGetLastError() != cudaSuccess) return DFLASH_ERR_CUDA;
    return DFLASH_OK;
}

extern "C" int dflash_verify_attn_read_flags(const void* workspace, int32_t* flags_host,
                                             int clear, void* cuda_stream) {
    if (!workspace || !flags_host) return DFLASH_ERR_INVALID_ARGUMENT;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        goto fail;
    if (clear && cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(int32_t), stream) !=
                     cudaSuccess)
        goto fail;
    if (cudaStreamSynchronize(stream) != cudaSuccess) goto fail;
    *flags_host = v;
    return DFLASH_OK;
fail:
    cudaGetLastError();
    return DFLASH_ERR_CUDA;
}
