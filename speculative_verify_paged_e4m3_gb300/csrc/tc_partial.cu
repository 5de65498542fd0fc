// tc_partial.cu -- tensor-core (tcgen05 + tensor memory) split-KV partial attention for sm_103a.
//
// Same contract as the CUDA-core kernel: one CTA per (split, KV head, sequence) carrying every
// query row of that KV head against each staged K/V tile ("six-head KV reuse", "[Perf] Reduce
// DFlash2 long-context verification decay", Implementation), writing the split's FP32 max / sum /
// numerator ("complete FP32 workspace", "[Perf] Reduce DFlash2 attention cost and screen exact QK
// reuse", Purpose). The GB300 design:
//
//  * keys on the MMA's M dimension (M = 128 keys per tile), query rows on N, so no MMA work is
//    spent on padding rows: S^T = K Q^T and O^T = V^T P^T, both with M = 128.
//  * QK^T runs on raw E4M3 K codes (kind::f8f6f4): K pages go from HBM to 128-byte-swizzled shared
//    memory by TMA and straight into the tensor core, with no decode. Q (FP16) is split exactly
//    into three E4M3 terms q * 2^a = t0 + t1/16 + t2/256 (per-row power-of-two a), stacked on N
//    (N = 3 x rows), and the score is (S0 + S1/16 + S2/256) * 2^-a * k_scale / 16 * log2 e.
//  * PV runs in FP16 (kind::f16): V codes are decoded exactly to FP16 with cvt.f16x2.e4m3x2 into
//    MN-major 32-key stages, P (<= 2^8) is rounded to FP16 into an MN-major tile (N padded to 64),
//    and O^T accumulates in tensor memory (FP32).
//  * Softmax: keys on tensor-memory lanes (thread = key); two warpgroups split the query rows.
//    Each keeps, per row, a reference max that only moves when a score exceeds it by more than 2^8
//    (then the warpgroup rescales its O columns in tensor memory), and FP32 row sums of the
//    unrounded probabilities, reduced across the key lanes once per split.
//  * Warp roles: warp 0 copies K tiles (TMA, 2 stages); warp 1 owns tensor memory and issues the
//    MMAs; warp 2 copies V in 64-key halves (TMA, 3 raw stages) and warps 2-3 decode them into
//    32-key FP16 stages (2 deep); warps 4-11 stage the Q terms (while the first
//    copies are in flight), then run the softmax (rows 0..RP/2-1 and RP/2..RP-1) and write O out.
//    K and V copies come from two different warps: one issuing warp tops out well below the HBM
//    rate on this GPU (measured), two reach it.
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

constexpr int kTile = 128;   // keys per tile = MMA M
constexpr int kChunk = 16;   // keys per TMA box (pages are multiples of 16 tokens)
constexpr int kVhKeys = 32;  // keys per decoded-V stage (two MMA K steps)
constexpr int kTerms = 3;    // E4M3 terms of Q
constexpr int kMaxRP = 48;   // padded rows per KV head this kernel carries
constexpr int kPN = 64;      // N of the PV MMA (rows padded to one 128-byte swizzle atom)
constexpr int kThreads = 512;
constexpr int kVWarps = 4;     // warps 12-15: V decode
constexpr int kVWarp0 = 12;
constexpr int kHalf = 64;      // keys per raw-V stage
constexpr int kVRawStages = 3;
constexpr int kPStages = 2;
constexpr int kVhStages = 2;

constexpr uint32_t kQBytes = kTerms * kMaxRP * kHeadDim;  // 36864
constexpr uint32_t kKStage = kTile * kHeadDim;            // 32768
constexpr uint32_t kVRawStage = kHalf * kHeadDim;         // 16384
constexpr uint32_t kVhStage = kVhKeys * kHeadDim * 2;     // 16384
constexpr uint32_t kPStage = kPN * kTile * 2;             // 16384
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffVRaw = kOffK + 2 * kKStage;
constexpr uint32_t kOffVh = kOffVRaw + kVRawStages * kVRawStage;
constexpr uint32_t kOffP = kOffVh + kVhStages * kVhStage;
constexpr uint32_t kOffSmall = kOffP + kPStages * kPStage;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kSStride = 192, kColO = 384, kOStride = 64;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr int kRowCache = 512;  // 16-key chunks of a split whose source row is looked up up front
constexpr float kLazyThreshold = 8.f;

struct Small {
    uint64_t kfull[2], kempty[2], sfull[2], sempty[2], pfull[kPStages], pempty[kPStages];
    uint64_t vfull[kVRawStages], vfree[kVRawStages], vhfull[kVhStages], vhempty[kVhStages];
    uint64_t odone, qready;
    uint32_t tmem_base;
    int abort;
    int flag[2][2][4];            // softmax group barrier: [group][epoch parity][warp]
    alignas(16) float c0[kMaxRP];    // score scale of each row (log2 units per MMA unit), read as float4
    alignas(16) float negm[kMaxRP];  // minus the reference max of each row (+inf: no key yet), float4
    float red[2][4][kMaxRP / 2];  // per-warpgroup, per-warp partials (tile max, row sums)
    float alpha[kMaxRP];
    int rows[kRowCache];          // source row (physical page * page + slot) of chunk c of the split
};
constexpr uint32_t kSmemBytes = kOffSmall + sizeof(Small);
static_assert(offsetof(Small, c0) % 16 == 0 && offsetof(Small, negm) % 16 == 0,
              "row constants are read as float4");
static_assert(kOffSmall % 16 == 0, "Small must start 16-byte aligned");
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Byte offset of (row, byte k along K) in a K-major, 128-byte-swizzled operand with `rows` rows
// (8-row groups 1 KB apart, 128-byte K columns rows*128 bytes apart).
__device__ __forceinline__ uint32_t kmajor_off(int row, int kbyte, int rows) {
    const int col = kbyte >> 7, w = kbyte & 127;
    return col * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
           ((((w >> 4) ^ (row & 7)) << 4) | (w & 15));
}

// Byte offset of the 16-byte chunk holding FP16 elements (mn .. mn+7, k) of an MN-major,
// 128-byte-swizzled operand: 64-element MN atoms `atom_stride` bytes apart, 8-k groups 1 KB apart.
__device__ __forceinline__ uint32_t mnmajor_chunk(int mn, int k, uint32_t atom_stride) {
    const int e = mn & 63, kr = k & 7;
    return (mn >> 6) * atom_stride + (k >> 3) * 1024 + kr * 128 + ((((e >> 3) ^ kr)) << 4);
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

// Loads / stores of N consecutive 32-bit tensor-memory columns of this thread's lane (N = 8k).
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* r) {
    if constexpr (N >= 16) {
        tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
        if constexpr (N > 16) tmem_load_cols<N - 16>(taddr + 16, r + 16);
    } else if constexpr (N == 8) {
        tmem_ld8(taddr, r);
    }
}
template <int N>
__device__ __forceinline__ void tmem_store_cols(uint32_t taddr, const uint32_t* r) {
    if constexpr (N >= 16) {
        tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(r));
        if constexpr (N > 16) tmem_store_cols<N - 16>(taddr + 16, r + 16);
    } else if constexpr (N == 8) {
        tmem_st8(taddr, r);
    }
}

template <int RP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PartialParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Small& sm = *reinterpret_cast<Small*>(smem + kOffSmall);
    constexpr int SN = kTerms * RP;
    constexpr int RH = RP / 2;  // rows per softmax warpgroup
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
    const int nhalves = (end - start + kHalf - 1) / kHalf;
    if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1 KB aligned base
        if (tid == 0) atomicOr(p.status, DFLASH_FLAG_KERNEL_TIMEOUT);
        return;
    }
    const Ctx ctx{&sm, p.status};

    // ---- set-up: barriers and tensor memory (Q terms are staged by the softmax warps while the
    // first copies are already in flight) ------------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.kfull[i]), 1);
            mbar_init(smem_u32(&sm.kempty[i]), 1);
            mbar_init(smem_u32(&sm.sfull[i]), 1);
            mbar_init(smem_u32(&sm.sempty[i]), 8);
        }
        for (int i = 0; i < kPStages; ++i) {
            mbar_init(smem_u32(&sm.pfull[i]), 8);
            mbar_init(smem_u32(&sm.pempty[i]), 1);
        }
        for (int i = 0; i < kVRawStages; ++i) {
            mbar_init(smem_u32(&sm.vfull[i]), 1);
            mbar_init(smem_u32(&sm.vfree[i]), kVWarps);
        }
        for (int i = 0; i < kVhStages; ++i) {
            mbar_init(smem_u32(&sm.vhfull[i]), kVWarps);
            mbar_init(smem_u32(&sm.vhempty[i]), 1);
        }
        mbar_init(smem_u32(&sm.odone), 1);
        mbar_init(smem_u32(&sm.qready), 8);
        sm.abort = 0;
        for (int i = 0; i < 16; ++i) (&sm.flag[0][0][0])[i] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    {
        // block-table lookups of the split's chunks, all in flight at once
        bool clamped = false;
        const int nchunks = min((end - start + kChunk - 1) / kChunk, kRowCache);
        for (int c = tid; c < nchunks; c += kThreads) {
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
                const int s = t & 1;
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
                if (!ctx.wait(&sm.kempty[s], ((t >> 1) & 1) ^ 1)) break;
                mbar_arrive_expect_tx(smem_u32(&sm.kfull[s]), nval * kChunk * kHeadDim);
                const uint32_t dst = smem_u32(smem + kOffK + s * kKStage);
#pragma unroll
                for (int c = 0; c < kTile / kChunk; ++c) {
                    if (rows[c] < 0) continue;
                    tma_load_2d(dst + c * 2048, &kmap, h * kHeadDim, rows[c],
                                smem_u32(&sm.kfull[s]));
                    tma_load_2d(dst + c * 2048 + kKStage / 2, &kmap, h * kHeadDim + 128, rows[c],
                                smem_u32(&sm.kfull[s]));
                }
                kdone = t + 1;
            }
            if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
            // no copy may still be writing shared memory when the CTA retires
            for (int t = kdone - 2 < 0 ? 0 : kdone - 2; t < kdone; ++t)
                mbar_wait(smem_u32(&sm.kfull[t & 1]), (t >> 1) & 1, &sm.abort, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && ctx.wait(&sm.qready, 0)) {
            const uint32_t idesc_qk = idesc_f32acc(128, SN, 0, 0, 0, 0);
            const uint32_t idesc_pv = idesc_f32acc(128, kPN, 0, 0, 1, 1);
            const uint32_t q_base = smem_u32(smem + kOffQ);
            auto issue_qk = [&](int u) -> bool {
                const int s = u & 1;
                const uint32_t ph = (u >> 1) & 1;
                if (!ctx.wait(&sm.kfull[s], ph)) return false;
                if (!ctx.wait(&sm.sempty[s], ph ^ 1)) return false;
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + kOffK + s * kKStage);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad =
                        smem_desc(kb + (kk >> 2) * (kKStage / 2) + (kk & 3) * 32, 16, 1024,
                                  kSwizzle128B);
                    const uint64_t bd = smem_desc(q_base + (kk >> 2) * (SN * 128) + (kk & 3) * 32,
                                                  16, 1024, kSwizzle128B);
                    mma_f8_ss(tmem + kColS + s * kSStride, ad, bd, idesc_qk, kk > 0);
                }
                mma_commit(smem_u32(&sm.kempty[s]));
                mma_commit(smem_u32(&sm.sfull[s]));
                return true;
            };
            auto issue_pv = [&](int t) -> bool {
                const int pb = t % kPStages;
                if (!ctx.wait(&sm.pfull[pb], (t / kPStages) & 1)) return false;
                tc_fence_after();
                const uint32_t pbase = smem_u32(smem + kOffP + pb * kPStage);
                const int halves = min(2, nhalves - 2 * t);
#pragma unroll 1
                for (int qq = 0; qq < 2 * halves; ++qq) {
                    const int e = 4 * t + qq;  // 32-key stage index
                    const int vs = e % kVhStages;
                    if (!ctx.wait(&sm.vhfull[vs], (e / kVhStages) & 1)) return false;
                    tc_fence_after();
                    const uint32_t vb = smem_u32(smem + kOffVh + vs * kVhStage);
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t bd = smem_desc(pbase + (4 * qq + 2 * ks) * 1024, kPStage,
                                                      1024, kSwizzle128B);
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh) {
                            const uint64_t ad = smem_desc(vb + dh * 2 * 4096 + ks * 2048, 4096,
                                                          1024, kSwizzle128B);
                            mma_f16_ss(tmem + kColO + dh * kOStride, ad, bd, idesc_pv,
                                       (t | qq | ks) != 0);
                        }
                    }
                    mma_commit(smem_u32(&sm.vhempty[vs]));
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
        // ------------------------------------------------- V copies (TMA): 64-key halves
        if (lane == 0) {
            bool clamped = false;
            int vdone = 0;
            for (int u = 0; u < nhalves; ++u) {
                const int st = u % kVRawStages;
                const int h0 = start + u * kHalf;
                int rows[kHalf / kChunk];
                int nval = 0;
#pragma unroll
                for (int c = 0; c < kHalf / kChunk; ++c) {
                    const int j0 = h0 + kChunk * c;
                    rows[c] = -1;
                    if (j0 < end) {
                        rows[c] = chunk_row(p, sm, b, start, j0, &clamped);
                        ++nval;
                    }
                }
                if (!ctx.wait(&sm.vfree[st], ((u / kVRawStages) & 1) ^ 1)) break;
                mbar_arrive_expect_tx(smem_u32(&sm.vfull[st]), nval * kChunk * kHeadDim);
                const uint32_t dst = smem_u32(smem + kOffVRaw + st * kVRawStage);
#pragma unroll
                for (int c = 0; c < kHalf / kChunk; ++c)
                    if (rows[c] >= 0)
                        tma_load_2d(dst + c * 4096, &vmap, h * kHeadDim, rows[c],
                                    smem_u32(&sm.vfull[st]));
                vdone = u + 1;
            }
            if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
            // no copy may still be writing shared memory when the CTA retires
            for (int u = vdone - kVRawStages < 0 ? 0 : vdone - kVRawStages; u < vdone; ++u)
                mbar_wait(smem_u32(&sm.vfull[u % kVRawStages]), (u / kVRawStages) & 1, &sm.abort,
                          kWaitLimitNs);
        }
    } else if (warp >= kVWarp0) {
        // ------------------------------------------------- V decode (warps 12-15)
        // All four warps decode every 32-key stage together into a 2-deep FP16 ring that the PV
        // MMAs consume in key order; a raw stage is released once all four have read it.
        const int vt = tid - kVWarp0 * 32;
        bool ok = true;
        for (int u = 0; ok && u < nhalves; ++u) {
            const int st = u % kVRawStages;
            if (!ctx.wait_warp(&sm.vfull[st], (u / kVRawStages) & 1)) break;
            const uint8_t* raw = smem + kOffVRaw + st * kVRawStage;
            const int h0 = start + u * kHalf;
#pragma unroll 1
            for (int q2 = 0; ok && q2 < kHalf / kVhKeys; ++q2) {
                const int e = 2 * u + q2;  // 32-key stage index
                const int vs = e % kVhStages;
                if (!ctx.wait_warp(&sm.vhempty[vs], ((e / kVhStages) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                uint8_t* vh = smem + kOffVh + vs * kVhStage;
                uint4 w[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int id = i * 128 + vt;
                    const int kk = q2 * kVhKeys + (id >> 4);  // key within the half
                    w[i] = h0 + kk < end ? *reinterpret_cast<const uint4*>(
                                               raw + kk * kHeadDim + (id & 15) * 16)
                                         : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int id = i * 128 + vt;
                    const int key = id >> 4, c = id & 15;
                    uint4 f0, f1;
                    e4m3x4_to_f16x4(w[i].x, f0.x, f0.y);
                    e4m3x4_to_f16x4(w[i].y, f0.z, f0.w);
                    e4m3x4_to_f16x4(w[i].z, f1.x, f1.y);
                    e4m3x4_to_f16x4(w[i].w, f1.z, f1.w);
                    *reinterpret_cast<uint4*>(vh + mnmajor_chunk(c * 16, key, 4096)) = f0;
                    *reinterpret_cast<uint4*>(vh + mnmajor_chunk(c * 16 + 8, key, 4096)) = f1;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.vhfull[vs]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.vfree[st]));
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- softmax (2 groups)
        const int sw = warp - 4;          // 0..7
        const int wg = sw >> 2;           // rows [wg * RH, wg * RH + RH)
        const int wq = warp & 3;          // tensor-memory lane quadrant
        const int st = (wq << 5) | lane;  // key of the tile = tensor-memory lane
        const int row0 = wg * RH;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int qoff = n - p.q_len;  // row r sees keys j <= qoff + r / G

        // Q -> three E4M3 terms (one warp per row), row scales, zero P padding rows
        {
            const float qk_scale = __ldg(p.k_scale) * 0.0625f * kLog2e;  // D^-1/2 = 1/16
            uint4 qraw[RP / 8];  // this warp's rows sw, sw + 8, ...: all loads in flight at once
#pragma unroll
            for (int k = 0; k < RP / 8; ++k) {
                const int r = sw + 8 * k;
                qraw[k] = make_uint4(0, 0, 0, 0);
                if (r < R) {
                    const int i = r / G, g = r % G;
                    const int64_t qrow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * G + g;
                    qraw[k] = *reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + lane * 8);
                }
            }
#pragma unroll
            for (int k = 0; k < RP / 8; ++k) {
                const int r = sw + 8 * k;
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
                    *reinterpret_cast<uint2*>(smem + kOffQ +
                                              kmajor_off(term * RP + r, lane * 8, SN)) =
                        make_uint2(packed[0], packed[1]);
                }
                if (lane == 0) {
                    sm.c0[r] = qk_scale * __int_as_float((127 - a) << 23);
                    sm.negm[r] = INFINITY;  // no key seen yet
                }
            }
            constexpr int kPadChunks = kTile * (kPN - RP) / 8;
            for (int i = tid - 128; i < kPStages * kPadChunks; i += 256) {
                const int stage = i / kPadChunks, rem = i % kPadChunks;
                const int key = rem % kTile, c = RP / 8 + rem / kTile;
                *reinterpret_cast<uint4*>(smem + kOffP + stage * kPStage +
                                          mnmajor_chunk(c * 8, key, kPStage)) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.qready));
        }
        int epoch = 0;
        bool alive = ctx.wait_warp(&sm.qready, 0);
        // per-row scale and minus reference max live in shared memory (read as float4 vectors,
        // identical for every thread of the group); row sums stay in registers
        float lsum[RH];
        uint32_t rowmask = 0;
#pragma unroll
        for (int i = 0; i < RH; ++i) {
            lsum[i] = 0.f;
            rowmask |= (uint32_t)(row0 + i < R) << i;
        }
        const float4* c0v = reinterpret_cast<const float4*>(sm.c0 + row0);
        float4* negmv = reinterpret_cast<float4*>(sm.negm + row0);
        for (int t = 0; alive && t < ntiles; ++t) {
            const int s = t & 1;
            const uint32_t ph = (t >> 1) & 1;
            const int tile0 = start + t * kTile;
            const int j = tile0 + st;
            if (!ctx.wait_warp(&sm.sfull[s], ph)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const uint32_t sbase = lane_base + kColS + s * kSStride + row0;
            // y = S0 + S1/16 + S2/256: the raw score in MMA units, kept in registers
            float y[RH];
            {
                uint32_t a[RH];
                tmem_load_cols<RH>(sbase, a);
                tmem_ld_wait_n<RH>(a);
#pragma unroll
                for (int i = 0; i < RH; ++i) y[i] = f32(a[i]);
                tmem_load_cols<RH>(sbase + RP, a);
                tmem_ld_wait_n<RH>(a);
#pragma unroll
                for (int i = 0; i < RH; ++i) y[i] = fmaf(f32(a[i]), 0.0625f, y[i]);
                tmem_load_cols<RH>(sbase + 2 * RP, a);
                tmem_ld_wait_n<RH>(a);
#pragma unroll
                for (int i = 0; i < RH; ++i) y[i] = fmaf(f32(a[i]), 0.00390625f, y[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.sempty[s]));  // S buffer free for QK(t+2)
            uint32_t validm = rowmask;  // bit i: key j visible to row row0 + i
            if (!((tile0 + kTile <= end) && (tile0 + kTile - 1 <= qoff))) {
#pragma unroll
                for (int i = 0; i < RH; ++i) {
                    const bool v = j < end && j <= qoff + (row0 + i) / G;
                    if (!v) validm &= ~(1u << i);
                }
            }
            // y <- score in log2 units; does any visible score exceed its row's reference max by
            // more than 2^8?
            bool need = false;
#pragma unroll
            for (int i4 = 0; i4 < RH / 4; ++i4) {
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
            if (!wg_sync(ctx, wg, wq, epoch, __any_sync(0xffffffffu, need), &need_any)) {
                alive = false;
                break;
            }
            bool ok = true;
            if (need_any) {
                // exact tile maximum per row -> new reference max; rescale row sums and O
#pragma unroll
                for (int i = 0; i < RH; ++i) {
                    const float m = warp_max(((validm >> i) & 1u) ? y[i] : -INFINITY);
                    if (lane == 0) sm.red[wg][wq][i] = m;
                }
                ok = wg_sync(ctx, wg, wq, epoch, false, nullptr);
                float mnew_own = 0.f;
                bool own = false;
                if (ok) {
#pragma unroll
                    for (int i = 0; i < RH; ++i) {
                        const float mo = -sm.negm[row0 + i];
                        const float tm = fmaxf(fmaxf(sm.red[wg][0][i], sm.red[wg][1][i]),
                                               fmaxf(sm.red[wg][2][i], sm.red[wg][3][i]));
                        const float mn = fmaxf(mo, tm);
                        const float alpha = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
                        lsum[i] *= alpha;
                        if (i == st) {
                            sm.alpha[row0 + i] = alpha;
                            mnew_own = mn;
                            own = true;
                        }
                    }
                    ok = wg_sync(ctx, wg, wq, epoch, false, nullptr);  // alphas visible, old m read
                    if (own) sm.negm[row0 + st] = -mnew_own;
                    ok = ok && wg_sync(ctx, wg, wq, epoch, false, nullptr);  // new m visible
                }
                if (ok && t > 0) {
                    // O holds tiles < t: wait for their PV, then scale this group's row columns
                    ok = ctx.wait_warp(&sm.pempty[(t - 1) % kPStages], ((t - 1) / kPStages) & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh) {
                            uint32_t o[RH];
                            const uint32_t oaddr = lane_base + kColO + dh * kOStride + row0;
                            tmem_load_cols<RH>(oaddr, o);
                            tmem_ld_wait_n<RH>(o);
#pragma unroll
                            for (int i = 0; i < RH; ++i)
                                o[i] = __float_as_uint(f32(o[i]) * sm.alpha[row0 + i]);
                            tmem_store_cols<RH>(oaddr, o);
                        }
                        tmem_st_wait();
                    }
                }
            }
            // pass 2: probabilities -> FP16 P (MN-major: this thread's rows, contiguous), row sums
            const int ps = t % kPStages;
            if (ok) ok = ctx.wait_warp(&sm.pempty[ps], ((t / kPStages) & 1) ^ 1);
            if (!ok) {
                alive = false;
                break;
            }
            uint8_t* pbuf = smem + kOffP + ps * kPStage;
#pragma unroll
            for (int c = 0; c < RH / 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                    const int i0 = c * 8 + 2 * q2, i1 = i0 + 1;
                    const float p0 = ((validm >> i0) & 1u) ? ex2(y[i0] + sm.negm[row0 + i0]) : 0.f;
                    const float p1 = ((validm >> i1) & 1u) ? ex2(y[i1] + sm.negm[row0 + i1]) : 0.f;
                    lsum[i0] += p0;
                    lsum[i1] += p1;
                    const __half2 hp = __floats2half2_rn(p0, p1);
                    w[q2] = *reinterpret_cast<const uint32_t*>(&hp);
                }
                *reinterpret_cast<uint4*>(pbuf + mnmajor_chunk(row0 + c * 8, st, kPStage)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.pfull[ps]));
        }
        // row sums over the 128 key lanes -> split state
#pragma unroll
        for (int i = 0; i < RH; ++i) {
            const float v = warp_sum(lsum[i]);
            if (lane == 0) sm.red[wg][wq][i] = v;
        }
        if (alive) alive = wg_sync(ctx, wg, wq, epoch, false, nullptr);
        const int64_t unit = ((int64_t)b * p.num_kv_heads + h) * p.num_splits + split;
        if (alive && !ctx.aborted()) {
#pragma unroll
            for (int i = 0; i < RH; ++i) {
                if (st == i && row0 + i < R) {
                    const float L = sm.red[wg][0][i] + sm.red[wg][1][i] + sm.red[wg][2][i] +
                                    sm.red[wg][3][i];
                    p.ws_state[unit * R + row0 + i] = make_float2(-sm.negm[row0 + i], L);
                }
            }
        }
        // O^T (tensor memory, lane = head-dim element) -> numerator rows; group wg writes half wg
        const bool ok = ctx.wait_warp(&sm.odone, 0);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok && !ctx.aborted())) {
            const float vs = __ldg(p.v_scale);
            const int d = wg * 128 + st;
            const uint32_t base = lane_base + kColO + wg * kOStride;
#pragma unroll
            for (int rc = 0; rc < RP / 8; ++rc) {
                uint32_t o[8];
                tmem_ld8(base + rc * 8, o);
                tmem_ld_wait_n<8>(o);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = rc * 8 + e;
                    if (r < R) p.ws_acc[(unit * R + r) * kHeadDim + d] = f32(o[e]) * vs;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace tc

int tc_rows_pad(int rows) { return (rows + 15) / 16 * 16; }

bool tc_supports(int rows) { return tc_rows_pad(rows) <= tc::kMaxRP; }

size_t tc_smem_bytes() { return tc::kSmemBytes; }

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
    cudaError_t e = cudaFuncSetAttribute(tc::tc_partial_kernel<RP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    tc::tc_partial_kernel<RP><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(kmap, vmap, p);
    return cudaGetLastError();
}

cudaError_t launch_tc_partial(const PartialParams& p, cudaStream_t stream) {
    const int rp = tc_rows_pad(p.rows);
    if (rp > tc::kMaxRP) return cudaErrorInvalidValue;
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap kmap, vmap;
    const cuuint64_t dims[2] = {(cuuint64_t)p.num_kv_heads * kHeadDim,
                                (cuuint64_t)p.num_pages * p.page_size};
    const cuuint64_t strides[1] = {(cuuint64_t)p.num_kv_heads * kHeadDim};
    const cuuint32_t kbox[2] = {128, tc::kChunk};
    const cuuint32_t vbox[2] = {kHeadDim, tc::kChunk};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r1 = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.k_pool),
                         dims, strides, kbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = encode(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.v_pool),
                         dims, strides, vbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
    switch (rp) {
        case 16: return launch_rp<16>(kmap, vmap, p, stream);
        case 32: return launch_rp<32>(kmap, vmap, p, stream);
        default: return launch_rp<48>(kmap, vmap, p, stream);
    }
}

}  // namespace dflash
