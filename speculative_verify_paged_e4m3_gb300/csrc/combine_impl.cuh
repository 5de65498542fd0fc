// combine_impl.cuh -- the merge of per-split FP32 state into FP16 output and FP32 log-sum-exp,
// shared by the standalone combine kernel and the partial kernel's fused merge.
//
// The pages pair every grouped q8 attention kernel with one combine kernel ("[Perf] Reduce
// DFlash2 attention cost and screen exact QK reuse", Test Result). For query row r the active
// splits s carry (m_s, l_s, acc_s) with m in log2 units:
//   M = max_s m_s, w_s = 2^{m_s - M}, L = sum_s w_s l_s, out = sum_s w_s acc_s / L,
//   lse = (M + log2 L) * ln 2.
// One work item is (query row, quarter of the head dim, sequence x KV head), done by 256 threads:
// 16 split lanes x 16 float4 columns, so the splits are read in parallel (16 at a time, each a
// coalesced 256-byte row segment). The maximum comes first (lane maxima through shared memory),
// so every weight is independent of the others and the sums carry no rescaling chain; the lanes'
// partial sums are then added through shared memory in lane order.
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
    float4 part[kCombineThreads];  // [split lane][column]: weighted numerator sums
    float mx[kCombineSplitLanes];  // maximum m of each split lane
    float ls[kCombineSplitLanes];  // weighted sum of l of each split lane
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
// in [0, 256) indexes the 256 threads that share named barrier bar_id and scratch sh. Split lane
// sl holds splits sl, sl + SL, ...: first the maximum M over every lane, then each lane's
// weighted sums in split order (fmaf), then the lanes' sums added in lane order. With at most one
// split per lane that is exactly the row kernel's arithmetic (combine.cu): one product per split,
// added in split order. The split state is read through L2 (ld.global.cg), so that state
// written by other CTAs of the same launch is seen.
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
    const int64_t col4 = quarter * kCols + col;
    // the split state only after the partial kernel has completed (a no-op unless this grid is
    // its programmatic dependent, and inside the fused merge)
    griddep_wait();
    // The first kCombineFold splits of this lane are loaded at once (indices clamped into the
    // unit's slots, so no load needs the context length: for a single sequence they go out
    // while the length is in flight); splits at or past the active count get no weight. Lanes
    // of more than kCombineFold splits read the rest in further rounds.
    float2 st[kCombineFold];
    float4 a[kCombineFold];
    int active = 0;
    float mx = -INFINITY;
    if (count > 0) {
#pragma unroll
        for (int k = 0; k < kCombineFold; ++k) {
            const int s = min(sl + k * SL, count - 1);
            st[k] = __ldcg(&p.ws_state[(base + s) * R + r]);
            a[k] = __ldcg(&acc4[((base + s) * R + r) * (kHeadDim / 4) + col4]);
        }
        const int per = n > 0 ? keys_per_split(n, count, p.tile_keys, p.min_split_keys) : 1;
        active = n > 0 ? (n + per - 1) / per : 0;
#pragma unroll
        for (int k = 0; k < kCombineFold; ++k)
            if (sl + k * SL < active) mx = fmaxf(mx, st[k].x);
        for (int s = sl + kCombineFold * SL; s < active; s += SL)
            mx = fmaxf(mx, __ldcg(&p.ws_state[(base + s) * R + r]).x);
    }
    if (col == 0) sh.mx[sl] = mx;
    combine_sync(bar_id);
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < SL; ++k) M = fmaxf(M, sh.mx[k]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = 0.f;
    if (M != -INFINITY) {
        auto add = [&](float2 sv, float4 av) {
            const float w = sv.x == -INFINITY ? 0.f : merge_ex2(sv.x - M);
            o.x = fmaf(w, av.x, o.x);
            o.y = fmaf(w, av.y, o.y);
            o.z = fmaf(w, av.z, o.z);
            o.w = fmaf(w, av.w, o.w);
            L = fmaf(w, sv.y, L);
        };
#pragma unroll
        for (int k = 0; k < kCombineFold; ++k)
            if (sl + k * SL < active) add(st[k], a[k]);
        for (int s = sl + kCombineFold * SL; s < active; s += SL)
            add(__ldcg(&p.ws_state[(base + s) * R + r]),
                __ldcg(&acc4[((base + s) * R + r) * (kHeadDim / 4) + col4]));
    }
    sh.part[sl * kCols + col] = o;
    if (col == 0) sh.ls[sl] = L;
    combine_sync(bar_id);
    if (tid < kCols) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        float Lt = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int k = 0; k < SL; ++k) {
                const float4 q = sh.part[k * kCols + tid];
                t.x = __fadd_rn(t.x, q.x);
                t.y = __fadd_rn(t.y, q.y);
                t.z = __fadd_rn(t.z, q.z);
                t.w = __fadd_rn(t.w, q.w);
                Lt = __fadd_rn(Lt, sh.ls[k]);
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
