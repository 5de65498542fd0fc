// combine_impl.cuh -- the merge of per-split FP32 state into FP16 output and FP32 log-sum-exp,
// shared by the standalone combine kernel and the partial kernel's fused merge.
//
// The pages pair every grouped q8 attention kernel with one combine kernel ("[Perf] Reduce
// DFlash2 attention cost and screen exact QK reuse", Test Result). For query row r the active
// splits s carry (m_s, l_s, acc_s) with m in log2 units:
//   M = max_s m_s, L = sum_s 2^{m_s - M} l_s, out = sum_s 2^{m_s - M} acc_s / L,
//   lse = (M + log2 L) * ln 2.
// One work item is (query row, quarter of the head dim, sequence x KV head), done by 256 threads:
// 16 split lanes x 16 float4 columns, so the splits are read in parallel (16 at a time, each a
// coalesced 256-byte row segment) and reduced through shared memory. The merge is associative,
// so a lane may fold its splits in any grouping: out and lse are the same sums in another order.
#pragma once

#include <math.h>

#include "common.cuh"

namespace dflash {

constexpr int kCombineThreads = 256;
constexpr int kCombineSplitLanes = 16;  // splits in flight per item
constexpr int kCombineCols = 16;        // float4 columns per item (64 head-dim elements)
constexpr int kCombineFold = 10;        // splits per lane whose loads are in flight together

// Split lanes x float4 columns = the 256 threads of an item; kCombineSplitLanes lanes of
// kCombineCols columns (a quarter of the head dim) by default.
struct CombineScratch {
    float4 part[kCombineThreads];             // [split lane][column]
    float2 ml[kCombineSplitLanes];            // (running max, running sum) of each split lane
};

// 2^x for the merge weights (x <= 0): the hardware approximation, relative error about 2^-22;
// results below 2^-126 flush to zero (such a split's weight is below FP32 resolution anyway).
__device__ __forceinline__ float merge_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void combine_sync(int bar_id) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kCombineThreads) : "memory");
}

// Merge item (row r, column block cb of the head dim, sequence b, KV head h) with SL split lanes
// of 256 / SL float4 columns (block cb covers head-dim elements [cb, cb + 1) x 1024 / SL). tid
// in [0, 256) indexes the 256 threads that share named barrier bar_id and scratch sh. Each split
// lane folds its splits (sl, sl + SL, ...) into a running (max, sum, numerator) in one pass, so
// that all its loads can be in flight at once; the lanes are then merged the same way through
// shared memory. The split state is read through L2 (ld.global.cg), so that state written by
// other CTAs of the same launch is seen.
// The unit's splits sit in workspace slots [first, first + count) (common.cuh, locate_slots);
// n is its context length (clamped).
template <int SL = kCombineSplitLanes>
__device__ __forceinline__ void combine_item(const CombineParams& p, int r, int quarter, int b,
                                             int h, int tid, int bar_id, CombineScratch& sh,
                                             int first, int count, int n) {
    constexpr int kCols = kCombineThreads / SL;
    static_assert(SL <= kCombineSplitLanes && kCols * SL == kCombineThreads, "item shape");
    const int sl = tid / kCols, col = tid % kCols;
    const int64_t base = first;
    const int R = p.rows;
    const float4* acc4 = reinterpret_cast<const float4*>(p.ws_acc);
    // Each fold round loads kCombineFold splits of this lane at once (indices clamped into the
    // unit's slots, so no load needs the context length): the first round's loads go out
    // before the length is used, which for a single sequence (slots fixed by the plan) overlaps
    // the length's load. Splits at or past the active count are masked in the fold (their slots
    // are read, not used).
    float m = -INFINITY, L = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (count > 0) {
        int active = 0;
        int s0 = sl;
        do {
            float2 st[kCombineFold];
            float4 a[kCombineFold];
#pragma unroll
            for (int k = 0; k < kCombineFold; ++k) {
                const int s = min(s0 + k * SL, count - 1);
                st[k] = __ldcg(&p.ws_state[(base + s) * R + r]);
                a[k] = __ldcg(&acc4[((base + s) * R + r) * (kHeadDim / 4) + quarter * kCols + col]);
            }
            if (s0 == sl) {
                const int per = n > 0 ? keys_per_split(n, count, p.tile_keys, p.min_split_keys) : 1;
                active = n > 0 ? (n + per - 1) / per : 0;
            }
#pragma unroll
            for (int k = 0; k < kCombineFold; ++k) {
                if (s0 + k * SL >= active) {  // inactive split or clamped duplicate: no weight
                    st[k] = make_float2(-INFINITY, 0.f);
                    a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                const float mn = fmaxf(m, st[k].x);
                const float cr = mn == -INFINITY ? 1.f : merge_ex2(m - mn);
                const float cs = mn == -INFINITY ? 0.f : merge_ex2(st[k].x - mn);
                L = fmaf(cs, st[k].y, L * cr);
                o.x = fmaf(cs, a[k].x, o.x * cr);
                o.y = fmaf(cs, a[k].y, o.y * cr);
                o.z = fmaf(cs, a[k].z, o.z * cr);
                o.w = fmaf(cs, a[k].w, o.w * cr);
                m = mn;
            }
            s0 += SL * kCombineFold;
        } while (s0 < active);
    }
    sh.part[sl * kCols + col] = o;
    if (col == 0) sh.ml[sl] = make_float2(m, L);
    combine_sync(bar_id);
    if (tid < kCols) {
        float M = -INFINITY;
#pragma unroll 4
        for (int k = 0; k < SL; ++k) M = fmaxf(M, sh.ml[k].x);
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        float Lt = 0.f;
        if (M != -INFINITY) {
#pragma unroll 4
            for (int k = 0; k < SL; ++k) {
                const float2 ml = sh.ml[k];
                const float w = ml.x == -INFINITY ? 0.f : merge_ex2(ml.x - M);
                const float4 q = sh.part[k * kCols + tid];
                t.x = fmaf(w, q.x, t.x);
                t.y = fmaf(w, q.y, t.y);
                t.z = fmaf(w, q.z, t.z);
                t.w = fmaf(w, q.w, t.w);
                Lt = fmaf(w, ml.y, Lt);
            }
            const float inv = 1.f / Lt;
            t.x *= inv;
            t.y *= inv;
            t.z *= inv;
            t.w *= inv;
        }
        const int i = r / p.group, g = r % p.group;
        const int64_t orow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * p.group + g;
        __half2* out2 =
            reinterpret_cast<__half2*>(p.out + orow * kHeadDim + (quarter * kCols + tid) * 4);
        out2[0] = __floats2half2_rn(t.x, t.y);
        out2[1] = __floats2half2_rn(t.z, t.w);
        if (quarter == 0 && tid == 0)
            p.lse[orow] = (M == -INFINITY) ? -INFINITY : (M + log2f(Lt)) * kLn2;
    }
    combine_sync(bar_id);  // the scratch is reused by the next item
}

}  // namespace dflash
