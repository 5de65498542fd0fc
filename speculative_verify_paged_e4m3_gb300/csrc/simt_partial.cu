// simt_partial.cu -- CUDA-core FP32 split-KV partial attention (the correctness baseline kernel).
//
// One CTA per (split, KV head, sequence) and row block. It keeps the query rows of its block (up
// to 64; every row of the KV head, q_len x six heads, in the pages' q8 / Hq6 / Hkv1 shape) against
// each staged K/V tile, which is
// the "six-head KV reuse" of "[Perf] Reduce DFlash2 long-context verification decay",
// Implementation, and writes the split's FP32 max / sum / numerator ("complete FP32 workspace",
// "[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Purpose).
// Scores are kept in log2 units (Q is pre-multiplied by k_scale * D^-1/2 * log2 e), so the online
// softmax uses exp2.
#include <math.h>

#include "common.cuh"
#include "e4m3.cuh"

namespace dflash {

constexpr int kSimtThreads = 256;
constexpr int kSimtRows = 64;  // rows per row block this kernel carries
constexpr int kSimtTile = 32;
constexpr int kKStride = kHeadDim + 1;
constexpr int kPStride = kSimtTile + 1;

int simt_max_rows() { return kSimtRows; }

size_t simt_smem_bytes() {
    return sizeof(float) * (size_t)(kSimtRows * kHeadDim + kSimtTile * kKStride +
                                    kSimtTile * kHeadDim + kSimtRows * kPStride + kSimtRows);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kSimtThreads, 1) simt_partial_kernel(PartialParams p) {
    extern __shared__ float smem[];
    float* Qs = smem;                               // [kSimtRows][kHeadDim]
    float* Ks = Qs + kSimtRows * kHeadDim;           // [kSimtTile][kKStride]
    float* Vs = Ks + kSimtTile * kKStride;          // [kSimtTile][kHeadDim]
    float* Ps = Vs + kSimtTile * kHeadDim;          // [kSimtRows][kPStride]
    float* alpha_s = Ps + kSimtRows * kPStride;      // [kSimtRows]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();  // the next kernel may start launching (programmatic launch)
    // this CTA's workspace slot and rows, and the (sequence, KV head) unit owning the slot
    // (slots are shared out by context length; common.cuh)
    const RowBlock rb = row_block(p);
    const int G = p.group, R = rb.rows, row_lo = rb.row_lo, slot = rb.slot;
    const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                      p.num_slots, p.max_context, p.q_len, slot, true);
    if (slot == 0 && tid == 0 && us.flags) atomicOr(p.status, us.flags);
    const int b = us.b, h = us.h, split = slot - us.first, n = us.n;
    if (b < 0) return;
    const int per = keys_per_split(n, us.count, p.tile_keys, p.min_split_keys);
    const int start = split * per;
    if (start >= n) return;  // idle slot: the combine never reads it
    const int end = min(n, start + per);
    // Q, the scales, the pages and the workspace only after the preceding kernel has completed
    // (a no-op unless this grid is its programmatic dependent)
    griddep_wait();

    const float qscale = __ldg(p.k_scale) * 0.0625f * kLog2e;  // D = 256: D^-1/2 = 1/16
    for (int idx = tid; idx < kSimtRows * kHeadDim; idx += kSimtThreads) {
        const int r = idx / kHeadDim, d = idx % kHeadDim;
        float v = 0.f;
        if (r < R) {
            const int i = (row_lo + r) / G, g = (row_lo + r) % G;
            const int64_t qrow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * G + g;
            v = __half2float(p.q[qrow * kHeadDim + d]) * qscale;
        }
        Qs[idx] = v;
    }

    float m_run[kSimtRows / 8], l_run[kSimtRows / 8], acc[kSimtRows];
#pragma unroll
    for (int m = 0; m < kSimtRows / 8; ++m) {
        m_run[m] = -INFINITY;
        l_run[m] = 0.f;
    }
#pragma unroll
    for (int r = 0; r < kSimtRows; ++r) acc[r] = 0.f;

    bool page_clamped = false;
    for (int t0 = start; t0 < end; t0 += kSimtTile) {
        __syncthreads();  // previous tile's K/V/P fully consumed (and Q written, first time)
        {
            const int kk = tid >> 3, part = tid & 7;
            const int j = t0 + kk;
            float kf[32], vf[32];
            if (j < end) {
                const int phys = physical_page(p.block_table, b, p.max_pages_per_seq,
                                               j / p.page_size, p.num_pages, &page_clamped);
                const int64_t off =
                    (((int64_t)phys * p.page_size + j % p.page_size) * p.num_kv_heads + h) *
                        kHeadDim + part * 32;
                const uint4* kp = reinterpret_cast<const uint4*>(p.k_pool + off);
                const uint4* vp = reinterpret_cast<const uint4*>(p.v_pool + off);
                uint4 kw[2] = {__ldg(kp), __ldg(kp + 1)};
                uint4 vw[2] = {__ldg(vp), __ldg(vp + 1)};
                const uint32_t* kb = reinterpret_cast<const uint32_t*>(kw);
                const uint32_t* vb = reinterpret_cast<const uint32_t*>(vw);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    kf[e] = e4m3_to_float((kb[e >> 2] >> (8 * (e & 3))) & 0xFFu);
                    vf[e] = e4m3_to_float((vb[e >> 2] >> (8 * (e & 3))) & 0xFFu);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) kf[e] = vf[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                Ks[kk * kKStride + part * 32 + e] = kf[e];
                Vs[kk * kHeadDim + part * 32 + e] = vf[e];
            }
        }
        __syncthreads();

        // scores: lane = key of the tile, rows warp + 8m
        float s[kSimtRows / 8];
#pragma unroll
        for (int m = 0; m < kSimtRows / 8; ++m) s[m] = 0.f;
        for (int d = 0; d < kHeadDim; ++d) {
            const float kv = Ks[lane * kKStride + d];
#pragma unroll
            for (int m = 0; m < kSimtRows / 8; ++m)
                s[m] = fmaf(Qs[(warp + 8 * m) * kHeadDim + d], kv, s[m]);
        }
        const int j = t0 + lane;
#pragma unroll
        for (int m = 0; m < kSimtRows / 8; ++m) {
            const int r = warp + 8 * m;
            const int i = (row_lo + r) / G;
            const bool valid = (r < R) && (j < end) && (j <= n - p.q_len + i);
            const float sv = valid ? s[m] : -INFINITY;
            const float mn = fmaxf(m_run[m], warp_max(sv));
            float pj = 0.f, alpha = 1.f;
            if (mn != -INFINITY) {
                pj = valid ? exp2f(sv - mn) : 0.f;
                alpha = exp2f(m_run[m] - mn);  // 0 when nothing was seen before
            }
            l_run[m] = l_run[m] * alpha + warp_sum(pj);
            m_run[m] = mn;
            Ps[r * kPStride + lane] = pj;
            if (lane == 0) alpha_s[r] = alpha;
        }
        __syncthreads();

        // numerator: thread = head-dim element
#pragma unroll
        for (int r = 0; r < kSimtRows; ++r) acc[r] *= alpha_s[r];
        for (int kk = 0; kk < kSimtTile; ++kk) {
            const float v = Vs[kk * kHeadDim + tid];
#pragma unroll
            for (int r = 0; r < kSimtRows; ++r) acc[r] = fmaf(Ps[r * kPStride + kk], v, acc[r]);
        }
    }
    if (page_clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);

    const int64_t unit = slot;  // this split's workspace slot
#pragma unroll
    for (int m = 0; m < kSimtRows / 8; ++m) {
        const int r = warp + 8 * m;
        if (r < R && lane == 0)
            p.ws_state[unit * p.rows + row_lo + r] = make_float2(m_run[m], l_run[m]);
    }
    const float vs = __ldg(p.v_scale);
#pragma unroll
    for (int r = 0; r < kSimtRows; ++r)
        if (r < R) p.ws_acc[(unit * p.rows + row_lo + r) * kHeadDim + tid] = acc[r] * vs;
}

cudaError_t launch_simt_partial(const PartialParams& p, cudaStream_t stream) {
    const size_t smem = simt_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(simt_partial_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (!row_blocks_valid(p, kSimtRows)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = partial_grid(p);
    cfg.blockDim = dim3(kSimtThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.pdl) {  // a programmatic dependent of the preceding kernel on the stream
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, simt_partial_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dflash
