// tc_partial.cu -- tensor-core (tcgen05 + tensor memory) split-KV partial attention for sm_103a.
//
// Same contract as the CUDA-core kernel: one CTA per (split, KV head, sequence) carrying every
// query row of that KV head against each staged K/V tile ("six-head KV reuse", "[Perf] Reduce
// DFlash2 long-context verification decay", Implementation), writing the split's FP32 max / sum /
// numerator ("complete FP32 workspace", "[Perf] Reduce DFlash2 attention cost and screen exact QK
// reuse", Purpose). The GB300 design:
//
//  * Both products run on the raw E4M3 cache codes (kind::f8f6f4), so no K or V byte is ever
//    decoded or rewritten: K and V pages go from HBM into 128-byte-swizzled shared memory by TMA
//    and straight into the tensor core. Keys sit on the MMA's M dimension (M = 128 keys per tile)
//    and query rows on N: S^T = K Q^T (K K-major) and O^T = V^T P^T (V read MN-major from the very
//    same tile layout), so no MMA work is spent on padding rows.
//  * Q (FP16) is split exactly into three E4M3 terms q * 2^a = t0 + t1/16 + t2/256 (per-row
//    power-of-two a), stacked on N (N = 3 x rows); the score is (S0 + S1/16 + S2/256) * 2^-a *
//    k_scale / 16 * log2 e.
//  * The probabilities, taken as p = 2^(s - m) * 2^score with s = 4 and a reference max m (so
//    p <= 2^8, see below), are split the same way into three E4M3 terms p = h + m/16 + l/256
//    (Veltkamp splitting in FP32, relative error about 2^-12, finer than an FP16 P), stacked on N,
//    so O^T accumulates three FP32 terms that are summed at the end. The shift s keeps the leading
//    term out of E4M3's subnormal range down to p = 2^-10 of the reference: below 2^-6 the
//    leading term only has a 2^-9 grid, and over 10^5 keys those roundings add up.
//  * Softmax: keys on tensor-memory lanes (thread = key); RP/16 warpgroups of 16 query rows each.
//    Each keeps, per row, a reference max that only moves when a score exceeds it by more than
//    2^(8 - s) (then the warpgroup rescales its O columns in tensor memory), and FP32 row sums of
//    the unrounded (shifted) probabilities, reduced across the key lanes once per split. The
//    split state keeps m - s as its max, which makes the shift invisible to the combine.
//  * Warp roles: warp 0 copies K tiles (TMA, 2 stages of 128 keys); warp 1 owns tensor memory and
//    issues the MMAs; warp 2 copies V (TMA, 64-key stages) and zeroes the keys past the context
//    in the last one (a zero probability must not meet a NaN code); warps 4.. stage the Q terms
//    (while the first copies are in flight), then run the softmax and write O out. K and V copies
//    come from two different warps: one issuing warp tops out well below the HBM rate on this GPU
//    (measured), two reach it.
//    Every wait is bounded: on timeout the CTA sets DFLASH_FLAG_KERNEL_TIMEOUT, drains its copies
//    and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>

#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "e4m3.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace tc {

using namespace ptx;

constexpr int kTile = 128;    // keys per tile = MMA M
constexpr int kChunk = 16;    // keys per TMA box (pages are multiples of 16 tokens)
constexpr int kVKeys = 64;    // keys per V stage
constexpr int kTerms = 3;     // E4M3 terms of Q and of P
constexpr int kMaxRP = 48;    // padded rows per KV head this kernel carries
constexpr int kGroupRows = 16;
constexpr int kKStages = 2;
constexpr int kVStages = 5;
constexpr int kPStages = 2;

constexpr uint32_t kKStage = kTile * kHeadDim;   // 32768: two 128-byte column blocks of 128 keys
constexpr uint32_t kVStage = kVKeys * kHeadDim;  // 16384: two 128-byte column blocks of 64 keys
constexpr uint32_t kKHalf = kKStage / 2;
constexpr uint32_t kVHalf = kVStage / 2;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr int kRowCache = 512;  // 16-key chunks of a split whose source row is looked up up front
constexpr float kPShift = 4.f;         // s: probabilities are scaled by 2^s before the split
constexpr float kLazyThreshold = 8.f;  // largest shifted probability exponent, 8 - s above the max

// Per-row-count layout. Shared memory: Q terms | K stages | V stages | P stages | Small.
// Tensor memory: S^T (3 x RP columns) then O^T of the two head-dim halves (3 x RP columns each).
template <int RP>
struct Cfg {
    static constexpr int kGroups = RP / kGroupRows;
    static constexpr int kSoftWarps = 4 * kGroups;
    static constexpr int kThreads = 128 + 32 * kSoftWarps;
    static constexpr int SN = kTerms * RP;  // N of both MMAs
    static constexpr uint32_t kQBytes = SN * kHeadDim;
    static constexpr uint32_t kPStage = SN * kTile;
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQBytes;
    static constexpr uint32_t kOffV = kOffK + kKStages * kKStage;
    static constexpr uint32_t kOffP = kOffV + kVStages * kVStage;
    static constexpr uint32_t kOffSmall = kOffP + kPStages * kPStage;
    static constexpr uint32_t kColS = 0, kColO = SN;
    static constexpr uint32_t kTmemCols = 3 * SN <= 256 ? 256 : 512;
    static_assert(RP % kGroupRows == 0 && RP <= kMaxRP, "rows per CTA");
    static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzled stages need 1 KB alignment");
    static_assert(kOffSmall % 16 == 0, "Small must start 16-byte aligned");
    static_assert(3 * SN <= 512, "tensor memory budget");
};

struct Small {
    uint64_t kfull[kKStages], kempty[kKStages], sfull, sempty, pfull[kPStages], pempty[kPStages];
    uint64_t vfull[kVStages], vfree[kVStages], vtail;
    uint64_t odone, qready;
    uint32_t tmem_base;
    int abort;
    int flag[kMaxRP / kGroupRows][2][4];  // group barrier: [group][epoch parity][warp]
    alignas(16) float c0[kMaxRP];    // score scale of each row (log2 units per MMA unit), float4 reads
    alignas(16) float negm[kMaxRP];  // s minus the reference max of each row (+inf: none yet), float4
    float red[kMaxRP / kGroupRows][4][kGroupRows];  // per-group, per-warp partials (max, row sums)
    float alpha[kMaxRP];
    int rows[kRowCache];  // source row (physical page * page + slot) of chunk c of the split
};
static_assert(offsetof(Small, c0) % 16 == 0 && offsetof(Small, negm) % 16 == 0,
              "row constants are read as float4");

template <int RP>
constexpr uint32_t smem_bytes() {
    return Cfg<RP>::kOffSmall + sizeof(Small);
}
static_assert(smem_bytes<kMaxRP>() <= 227 * 1024, "shared memory budget");

// Byte offset of (row, byte k along K) in a K-major, 128-byte-swizzled operand with `rows` rows
// (8-row groups 1 KB apart, 128-byte K columns rows*128 bytes apart).
__device__ __forceinline__ uint32_t kmajor_off(int row, int kbyte, int rows) {
    const int col = kbyte >> 7, w = kbyte & 127;
    return col * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
           ((((w >> 4) ^ (row & 7)) << 4) | (w & 15));
}

// P stage: an MN-major, unswizzled 8-bit operand of N = 3*RP rows by 128 keys, made of 16-row x
// 8-key core matrices (128 bytes, key-major inside): key groups 128 bytes apart (the descriptor's
// leading offset), 16-row blocks 2 KB apart (its stride offset). Byte offset of the 16 rows
// [16*nb, 16*nb + 16) of key k.
__device__ __forceinline__ uint32_t p_chunk(int nb, int k) {
    return nb * 2048 + (k >> 3) * 128 + (k & 7) * 16;
}

__device__ __forceinline__ float f32(uint32_t x) { return __uint_as_float(x); }

__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Split two probabilities (0 <= x <= 2^8) into three E4M3 terms x = h + m/16 + l/256 and return
// the codes, two per 16-bit word (first value in the low byte). h and m are x and the scaled
// residual rounded to 4 significant bits by Veltkamp splitting (c = x(2^20 + 1), h = c - (c - x),
// exact in FP32 with round-to-nearest), so both are E4M3 values whenever they are at least 2^-6
// and the residuals are exact; l is the last residual rounded to nearest by the conversion.
__device__ __forceinline__ void split3_x2(float a, float b, uint32_t& h, uint32_t& m, uint32_t& l) {
    constexpr float kC = 1048577.f;  // 2^20 + 1
    const float ca = __fmul_rn(a, kC), cb = __fmul_rn(b, kC);
    const float ha = __fsub_rn(ca, __fsub_rn(ca, a)), hb = __fsub_rn(cb, __fsub_rn(cb, b));
    const float ra = __fmul_rn(__fsub_rn(a, ha), 16.f), rb = __fmul_rn(__fsub_rn(b, hb), 16.f);
    const float da = __fmul_rn(ra, kC), db = __fmul_rn(rb, kC);
    const float ma = __fsub_rn(da, __fsub_rn(da, ra)), mb = __fsub_rn(db, __fsub_rn(db, rb));
    const float la = __fmul_rn(__fsub_rn(ra, ma), 16.f), lb = __fmul_rn(__fsub_rn(rb, mb), 16.f);
    h = f32x2_to_e4m3x2(ha, hb);
    m = f32x2_to_e4m3x2(ma, mb);
    l = f32x2_to_e4m3x2(la, lb);
}

struct Ctx {
    Small* sm;
    int32_t* status;
    __device__ bool wait(uint64_t* bar, uint32_t parity) const {
        if (mbar_wait(smem_u32(bar), parity, &sm->abort, kWaitLimitNs)) return true;
        *reinterpret_cast<volatile int*>(&sm->abort) = 1;
        atomicOr(status, DFLASH_FLAG_KERNEL_TIMEOUT);
        return false;
    }
    // The same for code run by a whole warp: every lane waits, and the warp agrees on the result,
    // so that no later warp-synchronous instruction runs with part of the warp gone.
    __device__ bool wait_warp(uint64_t* bar, uint32_t parity) const {
        const bool ok = wait(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
    __device__ bool aborted() const { return *reinterpret_cast<volatile int*>(&sm->abort) != 0; }
};

// Barrier of one softmax warpgroup (4 warps) through per-warp flags in shared memory, with a
// bounded spin (a plain bar.sync could hang if one warp had given up). Each warp publishes
// (epoch << 1) | vote; returns whether the barrier completed and ORs the four votes into *any.
__device__ __forceinline__ bool wg_sync(const Ctx& ctx, int wg, int wq, int& epoch, bool vote,
                                        bool* any) {
    ++epoch;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        __threadfence_block();
        *reinterpret_cast<volatile int*>(&ctx.sm->flag[wg][epoch & 1][wq]) =
            (epoch << 1) | (vote ? 1 : 0);
    }
    // a warp can run at most one epoch ahead, so slot epoch & 1 holds this epoch or the one before
    volatile int* f = ctx.sm->flag[wg][epoch & 1];
    bool done = false, v = false;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        const int a = f[0], b = f[1], c = f[2], d = f[3];
        if ((a >> 1) >= epoch && (b >> 1) >= epoch && (c >> 1) >= epoch && (d >> 1) >= epoch) {
            v = ((a | b | c | d) & 1) != 0;
            done = true;
            break;
        }
        if ((it & 31) == 0 && (ctx.aborted() || globaltimer_ns() - t0 > kWaitLimitNs)) break;
    }
    __threadfence_block();
    if (!done) {
        *reinterpret_cast<volatile int*>(&ctx.sm->abort) = 1;
        atomicOr(ctx.status, DFLASH_FLAG_KERNEL_TIMEOUT);
    }
    if (any) *any = v;
    return __all_sync(0xffffffffu, done);
}

// Source row in the page pool of the 16-key chunk starting at key j0 of sequence b: read from the
// split's cache when the chunk is in it, else straight from the block table.
__device__ __forceinline__ int chunk_row(const PartialParams& p, const Small& sm, int b, int start,
                                         int j0, bool* clamped) {
    const int c = (j0 - start) / kChunk;
    if (c < kRowCache) return sm.rows[c];
    const int phys = physical_page(p.block_table, b, p.max_pages_per_seq, j0 / p.page_size,
                                   p.num_pages, clamped);
    return phys * p.page_size + (j0 % p.page_size);
}

// The three term slices (columns base, base + RP, base + 2RP) of this lane's 16 rows, combined
// as t0 + t1/16 + t2/256.
template <int RP>
__device__ __forceinline__ void load_terms16(uint32_t taddr, float (&y)[kGroupRows]) {
    uint32_t a[16];
    tmem_ld16(taddr, a);
    tmem_ld_wait(a);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = f32(a[i]);
    tmem_ld16(taddr + RP, a);
    tmem_ld_wait(a);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = fmaf(f32(a[i]), 0.0625f, y[i]);
    tmem_ld16(taddr + 2 * RP, a);
    tmem_ld_wait(a);
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = fmaf(f32(a[i]), 0.00390625f, y[i]);
}

template <int RP>
__global__ void __launch_bounds__(Cfg<RP>::kThreads, 1)
    tc_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PartialParams p) {
    using C = Cfg<RP>;
    extern __shared__ __align__(1024) uint8_t smem[];
    Small& sm = *reinterpret_cast<Small*>(smem + C::kOffSmall);
    constexpr int SN = C::SN;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int R = p.rows, G = p.group, P = p.page_size;

    int cflags;
    const int n = clamped_context(p.context_lens, b, p.max_context, &cflags);
    if (split == 0 && h == 0 && tid == 0) {
        if (n < p.q_len) cflags |= DFLASH_FLAG_CONTEXT_SHORT;
        if (cflags) atomicOr(p.status, cflags);
    }
    const int per = keys_per_split(n, p.num_splits, p.tile_keys, p.min_split_keys);
    const int start = split * per;
    if (start >= n) return;  // idle split: the combine never reads it
    const int end = min(n, start + per);
    const int ntiles = (end - start + kTile - 1) / kTile;
    const int nvst = (end - start + kVKeys - 1) / kVKeys;
    if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1 KB aligned base
        if (tid == 0) atomicOr(p.status, DFLASH_FLAG_KERNEL_TIMEOUT);
        return;
    }
    const Ctx ctx{&sm, p.status};

    // ---- set-up: barriers and tensor memory (Q terms are staged by the softmax warps while the
    // first copies are already in flight) ------------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(smem_u32(&sm.kfull[i]), 1);
            mbar_init(smem_u32(&sm.kempty[i]), 1);
        }
        mbar_init(smem_u32(&sm.sfull), 1);
        mbar_init(smem_u32(&sm.sempty), C::kSoftWarps);
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(smem_u32(&sm.pfull[i]), C::kSoftWarps);
            mbar_init(smem_u32(&sm.pempty[i]), 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(smem_u32(&sm.vfull[i]), 1);
            mbar_init(smem_u32(&sm.vfree[i]), 1);
        }
        mbar_init(smem_u32(&sm.vtail), 1);
        mbar_init(smem_u32(&sm.odone), 1);
        mbar_init(smem_u32(&sm.qready), C::kSoftWarps);
        sm.abort = 0;
        for (int i = 0; i < (int)(sizeof(sm.flag) / sizeof(int)); ++i) (&sm.flag[0][0][0])[i] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), C::kTmemCols);
        tmem_relinquish();
    }
    {
        // block-table lookups of the split's chunks, all in flight at once
        bool clamped = false;
        const int nchunks = min((end - start + kChunk - 1) / kChunk, kRowCache);
        for (int c = tid; c < nchunks; c += C::kThreads) {
            const int j0 = start + c * kChunk;
            const int phys = physical_page(p.block_table, b, p.max_pages_per_seq, j0 / P,
                                           p.num_pages, &clamped);
            sm.rows[c] = phys * P + (j0 % P);
        }
        if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------------- K copies (TMA)
        if (lane == 0) {
            bool clamped = false;
            int kdone = 0;
            for (int t = 0; t < ntiles; ++t) {
                const int s = t % kKStages;
                const int tile0 = start + t * kTile;
                int rows[kTile / kChunk];
                int nval = 0;
#pragma unroll
                for (int c = 0; c < kTile / kChunk; ++c) {
                    const int j0 = tile0 + kChunk * c;
                    rows[c] = -1;
                    if (j0 < end) {
                        rows[c] = chunk_row(p, sm, b, start, j0, &clamped);
                        ++nval;
                    }
                }
                if (!ctx.wait(&sm.kempty[s], ((t / kKStages) & 1) ^ 1)) break;
                mbar_arrive_expect_tx(smem_u32(&sm.kfull[s]), nval * kChunk * kHeadDim);
                const uint32_t dst = smem_u32(smem + C::kOffK + s * kKStage);
#pragma unroll
                for (int c = 0; c < kTile / kChunk; ++c) {
                    if (rows[c] < 0) continue;
                    tma_load_2d(dst + c * 2048, &kmap, h * kHeadDim, rows[c],
                                smem_u32(&sm.kfull[s]));
                    tma_load_2d(dst + c * 2048 + kKHalf, &kmap, h * kHeadDim + 128, rows[c],
                                smem_u32(&sm.kfull[s]));
                }
                kdone = t + 1;
            }
            if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
            // no copy may still be writing shared memory when the CTA retires
            for (int t = kdone - kKStages < 0 ? 0 : kdone - kKStages; t < kdone; ++t)
                mbar_wait(smem_u32(&sm.kfull[t % kKStages]), (t / kKStages) & 1, &sm.abort,
                          kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && ctx.wait(&sm.qready, 0)) {
            const uint32_t idesc_qk = idesc_f32acc(128, SN, 0, 0, 0, 0);
            const uint32_t idesc_pv = idesc_f32acc(128, SN, 0, 0, 1, 1);
            const uint32_t q_base = smem_u32(smem + C::kOffQ);
            // S^T = K Q^T for tile t into the single S buffer (free once the softmax has read
            // tile t-1's scores)
            auto issue_qk = [&](int t) -> bool {
                const int s = t % kKStages;
                if (!ctx.wait(&sm.kfull[s], (t / kKStages) & 1)) return false;
                if (!ctx.wait(&sm.sempty, (t & 1) ^ 1)) return false;
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + C::kOffK + s * kKStage);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad =
                        smem_desc(kb + (kk >> 2) * kKHalf + (kk & 3) * 32, 16, 1024, kSwizzle128B);
                    const uint64_t bd = smem_desc(q_base + (kk >> 2) * (SN * 128) + (kk & 3) * 32,
                                                  16, 1024, kSwizzle128B);
                    mma_f8_ss(tmem + C::kColS, ad, bd, idesc_qk, kk > 0);
                }
                mma_commit(smem_u32(&sm.kempty[s]));
                mma_commit(smem_u32(&sm.sfull));
                return true;
            };
            // O^T += V^T P^T for tile t: two V stages of 64 keys, two 32-key steps each, both
            // head-dim halves
            auto issue_pv = [&](int t) -> bool {
                const int pb = t % kPStages;
                if (!ctx.wait(&sm.pfull[pb], (t / kPStages) & 1)) return false;
                tc_fence_after();
                const uint32_t pbase = smem_u32(smem + C::kOffP + pb * C::kPStage);
#pragma unroll 1
                for (int hv = 0; hv < kTile / kVKeys; ++hv) {
                    const int u = (kTile / kVKeys) * t + hv;
                    if (u >= nvst) break;
                    const int vs = u % kVStages;
                    if (!ctx.wait(&sm.vfull[vs], (u / kVStages) & 1)) return false;
                    tc_fence_after();
                    const uint32_t vb = smem_u32(smem + C::kOffV + vs * kVStage);
#pragma unroll
                    for (int kq = 0; kq < kVKeys / 32; ++kq) {
                        const int kk = (kVKeys / 32) * hv + kq;  // 32-key step within the tile
                        const uint64_t bd = smem_desc(pbase + kk * 512, 128, 2048, kSwizzleNone);
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh) {
                            const uint64_t ad = smem_desc(vb + dh * kVHalf + kq * 4096, kVHalf,
                                                          1024, kSwizzle128B);
                            mma_f8_ss(tmem + C::kColO + dh * SN, ad, bd, idesc_pv, (t | kk) != 0);
                        }
                    }
                    mma_commit(smem_u32(&sm.vfree[vs]));
                }
                mma_commit(smem_u32(&sm.pempty[pb]));
                return true;
            };
            bool ok = issue_qk(0);
            for (int t = 0; ok && t < ntiles; ++t) {
                if (t + 1 < ntiles) ok = issue_qk(t + 1);
                if (ok) ok = issue_pv(t);
            }
        }
        if (lane == 0) mma_commit(smem_u32(&sm.odone));  // tracks every MMA issued above
    } else if (warp == 2) {
        // ------------------------------------------- V copies (TMA): 64-key stages, whole warp
        bool clamped = false;
        int vdone = 0;
        bool tail_pending = false;  // the ragged last stage's copies are issued but not awaited
        for (int u = 0; u < nvst; ++u) {
            const int vs = u % kVStages;
            const int h0 = start + u * kVKeys;
            const int nkeys = min(kVKeys, end - h0);
            const bool tail = nkeys < kVKeys;
            if (!ctx.wait_warp(&sm.vfree[vs], ((u / kVStages) & 1) ^ 1)) break;
            uint8_t* vstage = smem + C::kOffV + vs * kVStage;
            const uint32_t bar = smem_u32(tail ? &sm.vtail : &sm.vfull[vs]);
            if (lane == 0) {
                int rows[kVKeys / kChunk];
                int nval = 0;
#pragma unroll
                for (int c = 0; c < kVKeys / kChunk; ++c) {
                    const int j0 = h0 + kChunk * c;
                    rows[c] = -1;
                    if (j0 < end) {
                        rows[c] = chunk_row(p, sm, b, start, j0, &clamped);
                        ++nval;
                    }
                }
                mbar_arrive_expect_tx(bar, nval * kChunk * kHeadDim);
                const uint32_t dst = smem_u32(vstage);
#pragma unroll
                for (int c = 0; c < kVKeys / kChunk; ++c) {
                    if (rows[c] < 0) continue;
                    tma_load_2d(dst + c * 2048, &vmap, h * kHeadDim, rows[c], bar);
                    tma_load_2d(dst + c * 2048 + kVHalf, &vmap, h * kHeadDim + 128, rows[c], bar);
                }
            }
            vdone = u + 1;
            if (tail) {
                // keys nkeys..63 of this stage (page-tail slots or never-copied rows) are zeroed
                // once the copies have landed; a key's 128 bytes per half are contiguous
                tail_pending = true;
                if (!ctx.wait_warp(&sm.vtail, 0)) break;
                tail_pending = false;
                const int zero_chunks = (kVKeys - nkeys) * 8;  // 16-byte chunks per half
                for (int i = lane; i < 2 * zero_chunks; i += 32) {
                    const int dh = i / zero_chunks, c = i % zero_chunks;
                    *reinterpret_cast<uint4*>(vstage + dh * kVHalf + nkeys * 128 + c * 16) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.vfull[vs]));
            }
        }
        if (lane == 0) {
            if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
            // no copy may still be writing shared memory when the CTA retires
            for (int u = vdone - kVStages < 0 ? 0 : vdone - kVStages; u < vdone; ++u) {
                const bool is_tail = end - (start + u * kVKeys) < kVKeys;
                if (is_tail) {
                    if (tail_pending) mbar_wait(smem_u32(&sm.vtail), 0, &sm.abort, kWaitLimitNs);
                } else {
                    mbar_wait(smem_u32(&sm.vfull[u % kVStages]), (u / kVStages) & 1, &sm.abort,
                              kWaitLimitNs);
                }
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------- softmax (RP/16 groups)
        const int sw = warp - 4;          // 0 .. kSoftWarps - 1
        const int g = sw >> 2;            // rows [16 g, 16 g + 16)
        const int wq = warp & 3;          // tensor-memory lane quadrant
        const int st = (wq << 5) | lane;  // key of the tile = tensor-memory lane
        const int row0 = kGroupRows * g;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int qoff = n - p.q_len;  // row r sees keys j <= qoff + r / G

        // Q -> three E4M3 terms (one warp per row), row scales
        {
            constexpr int kRowsPerWarp = RP / C::kSoftWarps;  // 4
            const float qk_scale = __ldg(p.k_scale) * 0.0625f * kLog2e;  // D^-1/2 = 1/16
            uint4 qraw[kRowsPerWarp];  // this warp's rows: all loads in flight at once
#pragma unroll
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int r = sw + C::kSoftWarps * k;
                qraw[k] = make_uint4(0, 0, 0, 0);
                if (r < R) {
                    const int i = r / G, gg = r % G;
                    const int64_t qrow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * G + gg;
                    qraw[k] = *reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + lane * 8);
                }
            }
#pragma unroll
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int r = sw + C::kSoftWarps * k;
                float qv[8];
                const __half2* hh = reinterpret_cast<const __half2*>(&qraw[k]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(hh[e]);
                    qv[2 * e] = f.x;
                    qv[2 * e + 1] = f.y;
                }
                float amax = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(qv[e]));
                amax = warp_max(amax);
                // largest a with amax * 2^a <= 448 = 1.75 * 2^8 (amax >= 2^-24: a normal float)
                int a = 0;
                if (amax > 0.f) {
                    const int bits = __float_as_int(amax);
                    const int ex = ((bits >> 23) & 0xFF) - 127;
                    const float mant = __int_as_float((bits & 0x007FFFFF) | 0x3F800000);
                    a = (mant <= 1.75f ? 8 : 7) - ex;
                }
                const float up = __int_as_float((a + 127) << 23);
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[e] *= up;
#pragma unroll
                for (int term = 0; term < kTerms; ++term) {
                    uint32_t packed[2];
#pragma unroll
                    for (int w = 0; w < 2; ++w) {
                        const uint16_t c01 = f32x2_to_e4m3x2(qv[4 * w], qv[4 * w + 1]);
                        const uint16_t c23 = f32x2_to_e4m3x2(qv[4 * w + 2], qv[4 * w + 3]);
                        packed[w] = (uint32_t)c01 | ((uint32_t)c23 << 16);
                        uint32_t lo, hi;
                        e4m3x4_to_f16x4(packed[w], lo, hi);
                        const float2 d01 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
                        const float2 d23 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
                        qv[4 * w] = (qv[4 * w] - d01.x) * 16.f;
                        qv[4 * w + 1] = (qv[4 * w + 1] - d01.y) * 16.f;
                        qv[4 * w + 2] = (qv[4 * w + 2] - d23.x) * 16.f;
                        qv[4 * w + 3] = (qv[4 * w + 3] - d23.y) * 16.f;
                    }
                    *reinterpret_cast<uint2*>(smem + C::kOffQ +
                                              kmajor_off(term * RP + r, lane * 8, SN)) =
                        make_uint2(packed[0], packed[1]);
                }
                if (lane == 0) {
                    sm.c0[r] = qk_scale * __int_as_float((127 - a) << 23);
                    sm.negm[r] = INFINITY;  // no key seen yet
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.qready));
        }
        int epoch = 0;
        bool alive = ctx.wait_warp(&sm.qready, 0);
        // per-row scale and minus reference max live in shared memory (read as float4 vectors,
        // identical for every thread of the group); row sums stay in registers
        float lsum[kGroupRows];
        uint32_t rowmask = 0;
#pragma unroll
        for (int i = 0; i < kGroupRows; ++i) {
            lsum[i] = 0.f;
            rowmask |= (uint32_t)(row0 + i < R) << i;
        }
        const float4* c0v = reinterpret_cast<const float4*>(sm.c0 + row0);
        const float4* negmv = reinterpret_cast<const float4*>(sm.negm + row0);
        for (int t = 0; alive && t < ntiles; ++t) {
            const int tile0 = start + t * kTile;
            const int j = tile0 + st;
            if (!ctx.wait_warp(&sm.sfull, t & 1)) {
                alive = false;
                break;
            }
            tc_fence_after();
            // y = S0 + S1/16 + S2/256: the raw score in MMA units, kept in registers
            float y[kGroupRows];
            load_terms16<RP>(lane_base + C::kColS + row0, y);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.sempty));  // S free for QK(t+1)
            uint32_t validm = rowmask;  // bit i: key j visible to row row0 + i
            if (!((tile0 + kTile <= end) && (tile0 + kTile - 1 <= qoff))) {
#pragma unroll
                for (int i = 0; i < kGroupRows; ++i) {
                    const bool v = j < end && j <= qoff + (row0 + i) / G;
                    if (!v) validm &= ~(1u << i);
                }
            }
            // y <- score in log2 units; would any visible shifted probability 2^(y + negm) exceed
            // 2^8?
            bool need = false;
#pragma unroll
            for (int i4 = 0; i4 < kGroupRows / 4; ++i4) {
                const float4 c = c0v[i4], nm = negmv[i4];
                y[4 * i4 + 0] *= c.x;
                y[4 * i4 + 1] *= c.y;
                y[4 * i4 + 2] *= c.z;
                y[4 * i4 + 3] *= c.w;
                need |= ((validm >> (4 * i4 + 0)) & 1u) && y[4 * i4 + 0] + nm.x > kLazyThreshold;
                need |= ((validm >> (4 * i4 + 1)) & 1u) && y[4 * i4 + 1] + nm.y > kLazyThreshold;
                need |= ((validm >> (4 * i4 + 2)) & 1u) && y[4 * i4 + 2] + nm.z > kLazyThreshold;
                need |= ((validm >> (4 * i4 + 3)) & 1u) && y[4 * i4 + 3] + nm.w > kLazyThreshold;
            }
            bool need_any = false;
            if (!wg_sync(ctx, g, wq, epoch, __any_sync(0xffffffffu, need), &need_any)) {
                alive = false;
                break;
            }
            bool ok = true;
            if (need_any) {
                // exact tile maximum per row -> new reference max; rescale row sums and O
#pragma unroll
                for (int i = 0; i < kGroupRows; ++i) {
                    const float m = warp_max(((validm >> i) & 1u) ? y[i] : -INFINITY);
                    if (lane == 0) sm.red[g][wq][i] = m;
                }
                ok = wg_sync(ctx, g, wq, epoch, false, nullptr);
                float mnew_own = 0.f;
                bool own = false;
                if (ok) {
#pragma unroll
                    for (int i = 0; i < kGroupRows; ++i) {
                        const float mo = kPShift - sm.negm[row0 + i];
                        const float tm = fmaxf(fmaxf(sm.red[g][0][i], sm.red[g][1][i]),
                                               fmaxf(sm.red[g][2][i], sm.red[g][3][i]));
                        const float mn = fmaxf(mo, tm);
                        const float alpha = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
                        lsum[i] *= alpha;
                        if (i == st) {
                            sm.alpha[row0 + i] = alpha;
                            mnew_own = mn;
                            own = true;
                        }
                    }
                    ok = wg_sync(ctx, g, wq, epoch, false, nullptr);  // alphas visible, old m read
                    if (own) sm.negm[row0 + st] = kPShift - mnew_own;
                    ok = ok && wg_sync(ctx, g, wq, epoch, false, nullptr);  // new m visible
                }
                if (ok && t > 0) {
                    // O holds tiles < t: wait for their PV, then scale this group's row columns
                    // of all three terms in both head-dim halves
                    ok = ctx.wait_warp(&sm.pempty[(t - 1) % kPStages],
                                       ((t - 1) / kPStages) & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll 1
                        for (int sl = 0; sl < 2 * kTerms; ++sl) {
                            const int dh = sl / kTerms, term = sl % kTerms;
                            const uint32_t addr =
                                lane_base + C::kColO + dh * SN + term * RP + row0;
                            uint32_t o[16];
                            tmem_ld16(addr, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                o[i] = __float_as_uint(f32(o[i]) * sm.alpha[row0 + i]);
                            tmem_st16(addr, o);
                        }
                        tmem_st_wait();
                    }
                }
            }
            // pass 2: probabilities -> three E4M3 terms in P (this thread's 16 rows of each term
            // are one 16-byte chunk), row sums from the unrounded values
            const int ps = t % kPStages;
            if (ok) ok = ctx.wait_warp(&sm.pempty[ps], ((t / kPStages) & 1) ^ 1);
            if (!ok) {
                alive = false;
                break;
            }
            uint32_t code[kTerms][4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float4 nm = negmv[w];
                float pv[4];
                pv[0] = ((validm >> (4 * w + 0)) & 1u) ? ex2(y[4 * w + 0] + nm.x) : 0.f;
                pv[1] = ((validm >> (4 * w + 1)) & 1u) ? ex2(y[4 * w + 1] + nm.y) : 0.f;
                pv[2] = ((validm >> (4 * w + 2)) & 1u) ? ex2(y[4 * w + 2] + nm.z) : 0.f;
                pv[3] = ((validm >> (4 * w + 3)) & 1u) ? ex2(y[4 * w + 3] + nm.w) : 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) lsum[4 * w + e] += pv[e];
                uint32_t h01, m01, l01, h23, m23, l23;
                split3_x2(pv[0], pv[1], h01, m01, l01);
                split3_x2(pv[2], pv[3], h23, m23, l23);
                code[0][w] = h01 | (h23 << 16);
                code[1][w] = m01 | (m23 << 16);
                code[2][w] = l01 | (l23 << 16);
            }
            uint8_t* pbuf = smem + C::kOffP + ps * C::kPStage;
#pragma unroll
            for (int term = 0; term < kTerms; ++term)
                *reinterpret_cast<uint4*>(pbuf + p_chunk(term * C::kGroups + g, st)) =
                    make_uint4(code[term][0], code[term][1], code[term][2], code[term][3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.pfull[ps]));
        }
        // row sums over the 128 key lanes -> split state (max m - s, shifted sums and numerator)
#pragma unroll
        for (int i = 0; i < kGroupRows; ++i) {
            const float v = warp_sum(lsum[i]);
            if (lane == 0) sm.red[g][wq][i] = v;
        }
        if (alive) alive = wg_sync(ctx, g, wq, epoch, false, nullptr);
        const int64_t unit = ((int64_t)b * p.num_kv_heads + h) * p.num_splits + split;
        if (alive && !ctx.aborted()) {
#pragma unroll
            for (int i = 0; i < kGroupRows; ++i) {
                if (st == i && row0 + i < R) {
                    const float L = sm.red[g][0][i] + sm.red[g][1][i] + sm.red[g][2][i] +
                                    sm.red[g][3][i];
                    p.ws_state[unit * R + row0 + i] = make_float2(-sm.negm[row0 + i], L);
                }
            }
        }
        // O^T (tensor memory, lane = head-dim element) -> numerator rows: O = O_h + O_m/16 + O_l/256
        const bool ok = ctx.wait_warp(&sm.odone, 0);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok && !ctx.aborted())) {
            const float vs = __ldg(p.v_scale);
#pragma unroll 1
            for (int dh = 0; dh < 2; ++dh) {
                float o[kGroupRows];
                load_terms16<RP>(lane_base + C::kColO + dh * SN + row0, o);
                const int d = dh * 128 + st;
#pragma unroll
                for (int i = 0; i < kGroupRows; ++i) {
                    const int r = row0 + i;
                    if (r < R) p.ws_acc[(unit * R + r) * kHeadDim + d] = o[i] * vs;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace tc

int tc_rows_pad(int rows) { return (rows + tc::kGroupRows - 1) / tc::kGroupRows * tc::kGroupRows; }

bool tc_supports(int rows) { return tc_rows_pad(rows) <= tc::kMaxRP; }

size_t tc_smem_bytes(int rows) {
    switch (tc_rows_pad(rows)) {
        case 16: return tc::smem_bytes<16>();
        case 32: return tc::smem_bytes<32>();
        default: return tc::smem_bytes<48>();
    }
}

int tc_threads(int rows) {
    switch (tc_rows_pad(rows)) {
        case 16: return tc::Cfg<16>::kThreads;
        case 32: return tc::Cfg<32>::kThreads;
        default: return tc::Cfg<48>::kThreads;
    }
}

// The tensor-map encoder lives in the driver library; it is looked up at first use through the
// runtime (so the library itself loads on machines without a driver, e.g. to plan and test).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

template <int RP>
static cudaError_t launch_rp(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PartialParams& p, cudaStream_t stream) {
    constexpr uint32_t smem = tc::smem_bytes<RP>();
    cudaError_t e = cudaFuncSetAttribute(tc::tc_partial_kernel<RP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    tc::tc_partial_kernel<RP><<<grid, tc::Cfg<RP>::kThreads, smem, stream>>>(kmap, vmap, p);
    return cudaGetLastError();
}

cudaError_t launch_tc_partial(const PartialParams& p, cudaStream_t stream) {
    const int rp = tc_rows_pad(p.rows);
    if (rp > tc::kMaxRP) return cudaErrorInvalidValue;
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    // K and V pools viewed as [num_pages * page_size rows, Hkv * 256 bytes]; both copied in boxes
    // of 16 rows x 128 bytes into the 128-byte swizzle the MMA operands use
    CUtensorMap kmap, vmap;
    const cuuint64_t dims[2] = {(cuuint64_t)p.num_kv_heads * kHeadDim,
                                (cuuint64_t)p.num_pages * p.page_size};
    const cuuint64_t strides[1] = {(cuuint64_t)p.num_kv_heads * kHeadDim};
    const cuuint32_t box[2] = {128, tc::kChunk};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r1 = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.k_pool),
                         dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = encode(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.v_pool),
                         dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
    switch (rp) {
        case 16: return launch_rp<16>(kmap, vmap, p, stream);
        case 32: return launch_rp<32>(kmap, vmap, p, stream);
        default: return launch_rp<48>(kmap, vmap, p, stream);
    }
}

}  // namespace dflash
