// combine.cu -- standalone merge kernels, 256 threads per CTA, shaped by the split count per
// (sequence, KV head) unit: up to 16 splits, 4 query rows per CTA with one thread per float4
// column (combine_rows_kernel); up to 64, one row per CTA with 4 split lanes; beyond, a quarter
// row per CTA with 16 split lanes (combine_lanes_kernel, merge in combine_item). A single
// sequence (every KV head owns num_splits slots) and a batch (slots shared out by length) get
// separate instances, so that the one-sequence kernels carry no slot search.
#include "combine_impl.cuh"

namespace dflash {

// Split-lane items: SL split lanes x 256 / SL float4 columns, one CTA per (query row, column
// block, unit), SL / 4 column blocks per row. 16 lanes (quarter rows) for long split lists
// (a single long sequence: about ten splits per lane); 4 lanes (whole rows) for 17..64 splits per
// unit (e.g. whole-model heads), so that each lane still folds about as many.
template <int SL, bool kBatch>
__global__ void __launch_bounds__(kCombineThreads) combine_lanes_kernel(CombineParams p) {
    __shared__ CombineScratch sh;
    griddep_launch_dependents();  // the next kernel may start launching (programmatic launch)
    const int unit = blockIdx.z;
    const int b = unit / p.num_kv_heads, h = unit % p.num_kv_heads;
    int first, count, n;
    if constexpr (kBatch) {  // several sequences: the unit's slots follow from every length
        const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                          p.num_slots, p.max_context, p.q_len, unit, false);
        first = us.first;
        count = us.count;
        n = us.n;
    } else {  // one sequence: every KV head owns num_splits slots, unit h at h * num_splits
        n = p.context_lens[0];
        n = n > p.max_context ? p.max_context : (n < 0 ? 0 : n);
        first = h * p.num_splits;
        count = p.num_splits;
    }
    combine_item<SL>(p, blockIdx.x, blockIdx.y, b, h, threadIdx.x, 0, sh, first, count, n);
}

// Plans with few splits per unit (many units: a batch, whole-model heads) merge a whole row per
// 64 threads instead: one CTA per (4 query rows, unit), each thread one float4 column across
// all of the unit's splits: the maximum, then one rounded product per split added in split
// order. That is combine_item's arithmetic when no split lane holds more than one split, so
// results are the same bits for up to 16 splits per unit.
constexpr int kRowCols = kHeadDim / 4;                 // 64 float4 columns per row
constexpr int kRowsPerCta = kCombineThreads / kRowCols;  // 4
constexpr int kRowKernelMaxSplits = kCombineSplitLanes;  // 16

template <bool kBatch>
__global__ void __launch_bounds__(kCombineThreads) combine_rows_kernel(CombineParams p) {
    griddep_launch_dependents();  // the next kernel may start launching (programmatic launch)
    const int unit = blockIdx.y;
    const int r = blockIdx.x * kRowsPerCta + threadIdx.x / kRowCols;
    const int col = threadIdx.x % kRowCols;
    const int b = unit / p.num_kv_heads, h = unit % p.num_kv_heads;
    int first, count, n;
    if constexpr (kBatch) {
        const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                          p.num_slots, p.max_context, p.q_len, unit, false);
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
    griddep_wait();  // the split state only after the partial kernel has completed
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
                const float w = st[k].x == -INFINITY ? 0.f : merge_ex2(st[k].x - M);
                t.x = __fadd_rn(t.x, __fmul_rn(w, a[k].x));
                t.y = __fadd_rn(t.y, __fmul_rn(w, a[k].y));
                t.z = __fadd_rn(t.z, __fmul_rn(w, a[k].z));
                t.w = __fadd_rn(t.w, __fmul_rn(w, a[k].w));
                Lt = __fadd_rn(Lt, __fmul_rn(w, st[k].y));
            }
        }
        const float inv = 1.f / Lt;
        t.x *= inv;
        t.y *= inv;
        t.z *= inv;
        t.w *= inv;
    }
    const int i = r / p.group, g = r % p.group;
    const int64_t orow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * p.group + g;
    __half2* out2 = reinterpret_cast<__half2*>(p.out + orow * kHeadDim + col * 4);
    out2[0] = __floats2half2_rn(t.x, t.y);
    out2[1] = __floats2half2_rn(t.z, t.w);
    if (col == 0) p.lse[orow] = (M == -INFINITY) ? -INFINITY : (M + log2f(Lt)) * kLn2;
}

// One launch of kernel over grid, 256 threads; with p.pdl a programmatic dependent of the
// preceding kernel on the stream.
static cudaError_t launch(void (*kernel)(CombineParams), dim3 grid, const CombineParams& p,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kCombineThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int SL>
static cudaError_t launch_lanes(const CombineParams& p, cudaStream_t stream) {
    const dim3 grid(p.rows, SL / 4, p.batch * p.num_kv_heads);
    return launch(p.batch == 1 ? combine_lanes_kernel<SL, false> : combine_lanes_kernel<SL, true>,
                  grid, p, stream);
}

constexpr int kMidKernelMaxSplits = 64;

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    cudaError_t e;
    if (p.num_splits <= kRowKernelMaxSplits) {
        const dim3 grid((p.rows + kRowsPerCta - 1) / kRowsPerCta, p.batch * p.num_kv_heads);
        e = launch(p.batch == 1 ? combine_rows_kernel<false> : combine_rows_kernel<true>, grid, p,
                   stream);
    } else if (p.num_splits <= kMidKernelMaxSplits) {
        e = launch_lanes<4>(p, stream);
    } else {
        e = launch_lanes<kCombineSplitLanes>(p, stream);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dflash
