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
//    an MN-major tile, P (<= 2^8) is rounded to FP16, O^T accumulates in tensor memory (FP32).
//  * Softmax with keys on tensor-memory lanes (thread = key) keeps a per-row reference max that
//    only moves when a score exceeds it by more than 2^8 (then O is rescaled in tensor memory);
//    row sums are kept per thread in FP32 from the unrounded probabilities and reduced once.
//  * Warp roles: warp 0 TMA producer, warp 1 MMA issuer, warp 2 tensor-memory allocator, warps 4-7
//    V decode (and O half 1 write-out), warps 8-11 softmax (and O half 0 write-out). Every wait is
//    bounded: on timeout the CTA sets DFLASH_FLAG_KERNEL_TIMEOUT, drains its copies and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "e4m3.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace tc {

using namespace ptx;

constexpr int kTile = 128;    // keys per tile = MMA M
constexpr int kChunk = 16;    // keys per TMA box (pages are multiples of 16 tokens)
constexpr int kQuarter = 32;  // keys per decoded-V stage
constexpr int kTerms = 3;     // E4M3 terms of Q
constexpr int kMaxRP = 48;    // padded rows per KV head this kernel carries
constexpr int kThreads = 384;

constexpr uint32_t kQBytes = kTerms * kMaxRP * kHeadDim;  // 36864
constexpr uint32_t kKStage = kTile * kHeadDim;            // 32768
constexpr uint32_t kVRawStage = kTile * kHeadDim;         // 32768
constexpr uint32_t kVhStage = kQuarter * kHeadDim * 2;    // 16384
constexpr uint32_t kPStage = kMaxRP * kTile * 2;          // 12288
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffVRaw = kOffK + 2 * kKStage;
constexpr uint32_t kOffVh = kOffVRaw + 2 * kVRawStage;
constexpr uint32_t kOffP = kOffVh + 2 * kVhStage;
constexpr uint32_t kOffSmall = kOffP + 2 * kPStage;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kSStride = 192, kColO = 384, kOStride = 64;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr float kLazyThreshold = 8.f;

struct Small {
    uint64_t kfull[2], kempty[2], vfull[2], vempty[2], sfull[2], sempty[2], pfull[2], pempty[2];
    uint64_t vhfull[2], vhempty[2], odone, wgbar;
    uint32_t tmem_base;
    int abort;
    float2 rowp[kMaxRP];      // (score scale c0 of the row, reference max m in log2 units)
    float red[4][kMaxRP];     // per-warp partials (tile max, row sums)
    float alpha[kMaxRP];
    int vote[2][4];
};
constexpr uint32_t kSmemBytes = kOffSmall + sizeof(Small);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// Byte offset of (row, byte k along K) in a K-major, 128-byte-swizzled operand with `rows` rows
// (8-row groups 1 KB apart, 128-byte K columns rows*128 bytes apart).
__device__ __forceinline__ uint32_t kmajor_off(int row, int kbyte, int rows) {
    const int col = kbyte >> 7, w = kbyte & 127;
    return col * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
           ((((w >> 4) ^ (row & 7)) << 4) | (w & 15));
}

// Byte offset of FP16 element (d, key) in a decoded-V stage: MN-major (d contiguous),
// 128-byte swizzle, 64-d atoms 4 KB apart (LBO), 8-key groups 1 KB apart (SBO).
__device__ __forceinline__ uint32_t vh_off(int d, int key) {
    const int e = d & 63, kr = key & 7;
    return (d >> 6) * 4096 + (key >> 3) * 1024 + kr * 128 + ((((e >> 3) ^ kr)) << 4) +
           ((e & 7) << 1);
}

__device__ __forceinline__ float f32(uint32_t x) { return __uint_as_float(x); }

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
};

// Barrier of the 128 softmax threads on an mbarrier, so that it is bounded like every other
// wait (a plain bar.sync would hang if one thread had given up). Returns false on abort.
__device__ __forceinline__ bool wg_sync(const Ctx& ctx, uint32_t& phase) {
    __syncwarp();
    mbar_arrive(smem_u32(&ctx.sm->wgbar));
    const bool ok = ctx.wait_warp(&ctx.sm->wgbar, phase & 1);
    ++phase;
    return ok;
}

// Load the three term columns of 16 rows for this thread's key.
__device__ __forceinline__ void load_s(uint32_t base, int RP, int rc, uint32_t (&a0)[16],
                                       uint32_t (&a1)[16], uint32_t (&a2)[16]) {
    tmem_ld16(base + rc * 16, a0);
    tmem_ld16(base + RP + rc * 16, a1);
    tmem_ld16(base + 2 * RP + rc * 16, a2);
    tmem_ld_wait(a0);
    tmem_ld_wait(a1);
    tmem_ld_wait(a2);
}

template <int RP>
__global__ void __launch_bounds__(kThreads, 1)
    tc_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PartialParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Small& sm = *reinterpret_cast<Small*>(smem + kOffSmall);
    constexpr int SN = kTerms * RP;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int R = p.rows, G = p.group;

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
    if (smem_u32(smem) & 1023u) {  // the swizzled layouts need a 1 KB aligned base
        if (tid == 0) atomicOr(p.status, DFLASH_FLAG_KERNEL_TIMEOUT);
        return;
    }
    const Ctx ctx{&sm, p.status};

    // ---- set-up: barriers, tensor memory, Q terms -------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&sm.kfull[i]), 1);
            mbar_init(smem_u32(&sm.kempty[i]), 1);
            mbar_init(smem_u32(&sm.vfull[i]), 1);
            mbar_init(smem_u32(&sm.vempty[i]), 4);
            mbar_init(smem_u32(&sm.sfull[i]), 1);
            mbar_init(smem_u32(&sm.sempty[i]), 4);
            mbar_init(smem_u32(&sm.pfull[i]), 4);
            mbar_init(smem_u32(&sm.pempty[i]), 1);
            mbar_init(smem_u32(&sm.vhfull[i]), 4);
            mbar_init(smem_u32(&sm.vhempty[i]), 1);
        }
        mbar_init(smem_u32(&sm.odone), 1);
        mbar_init(smem_u32(&sm.wgbar), 128);
        sm.abort = 0;
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    {
        const float qk_scale = __ldg(p.k_scale) * 0.0625f * kLog2e;  // D^-1/2 = 1/16
        for (int r = warp; r < RP; r += kThreads / 32) {
            float qv[8];
            if (r < R) {
                const int i = r / G, g = r % G;
                const int64_t qrow = ((int64_t)b * p.q_len + i) * p.num_q_heads + h * G + g;
                const uint4 raw = *reinterpret_cast<const uint4*>(p.q + qrow * kHeadDim + lane * 8);
                const __half2* hh = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = __half22float2(hh[e]);
                    qv[2 * e] = f.x;
                    qv[2 * e + 1] = f.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[e] = 0.f;
            }
            float amax = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(qv[e]));
            amax = warp_max(amax);
            int a = 0;
            if (amax > 0.f) {
                a = (int)floorf(log2f(448.f / amax));
                while (amax * ldexpf(1.f, a) > 448.f) --a;
            }
            const float up = ldexpf(1.f, a);
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
                *reinterpret_cast<uint2*>(smem + kOffQ + kmajor_off(term * RP + r, lane * 8, SN)) =
                    make_uint2(packed[0], packed[1]);
            }
            if (lane == 0) sm.rowp[r] = make_float2(ldexpf(qk_scale, -a), -INFINITY);
        }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        const int P = p.page_size;
        bool clamped = false;
        int issued = 0;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t & 1;
            const uint32_t ph = (t >> 1) & 1;
            const int tile0 = start + t * kTile;
            int row = 0;
            bool valid = false;
            if (lane < kTile / kChunk) {
                const int j0 = tile0 + kChunk * lane;
                if (j0 < end) {
                    valid = true;
                    const int phys = physical_page(p.block_table, b, p.max_pages_per_seq, j0 / P,
                                                   p.num_pages, &clamped);
                    row = phys * P + (j0 % P);
                }
            }
            const uint32_t bytes = __popc(__ballot_sync(0xffffffffu, valid)) * kChunk * kHeadDim;
            int ok = 1;
            if (lane == 0) {
                ok = ctx.wait(&sm.kempty[s], ph ^ 1);
                if (ok) mbar_arrive_expect_tx(smem_u32(&sm.kfull[s]), bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            if (valid) {
                const uint32_t dst = smem_u32(smem + kOffK + s * kKStage) + lane * 2048;
                tma_load_2d(dst, &kmap, h * kHeadDim, row, smem_u32(&sm.kfull[s]));
                tma_load_2d(dst + kKStage / 2, &kmap, h * kHeadDim + 128, row,
                            smem_u32(&sm.kfull[s]));
            }
            if (lane == 0) {
                ok = ctx.wait(&sm.vempty[s], ph ^ 1);
                if (ok) mbar_arrive_expect_tx(smem_u32(&sm.vfull[s]), bytes);
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                issued = -(t + 1);  // K of tile t is in flight, V is not
                break;
            }
            if (valid) {
                tma_load_2d(smem_u32(smem + kOffVRaw + s * kVRawStage) + lane * 4096, &vmap,
                            h * kHeadDim, row, smem_u32(&sm.vfull[s]));
            }
            issued = t + 1;
        }
        if (__any_sync(0xffffffffu, clamped) && lane == 0)
            atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
        if (lane == 0) {
            // no copy may still be writing shared memory when the CTA retires
            const int kdone = issued < 0 ? -issued : issued;
            const int vdone = issued < 0 ? -issued - 1 : issued;
            for (int t = kdone - 2 < 0 ? 0 : kdone - 2; t < kdone; ++t)
                mbar_wait(smem_u32(&sm.kfull[t & 1]), (t >> 1) & 1, &sm.abort, kWaitLimitNs);
            for (int t = vdone - 2 < 0 ? 0 : vdone - 2; t < vdone; ++t)
                mbar_wait(smem_u32(&sm.vfull[t & 1]), (t >> 1) & 1, &sm.abort, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_f32acc(128, SN, 0, 0, 0, 0);
            const uint32_t idesc_pv = idesc_f32acc(128, RP, 0, 0, 1, 0);
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
                const int pb = t & 1;
                if (!ctx.wait(&sm.pfull[pb], (t >> 1) & 1)) return false;
                tc_fence_after();
                const uint32_t pbase = smem_u32(smem + kOffP + pb * kPStage);
#pragma unroll 1
                for (int qq = 0; qq < kTile / kQuarter; ++qq) {
                    const int u = 4 * t + qq;
                    const int vs = u & 1;
                    if (!ctx.wait(&sm.vhfull[vs], (u >> 1) & 1)) return false;
                    tc_fence_after();
                    const uint32_t vb = smem_u32(smem + kOffVh + vs * kVhStage);
#pragma unroll
                    for (int dh = 0; dh < 2; ++dh) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            const uint64_t ad =
                                smem_desc(vb + dh * 8192 + ks * 2048, 4096, 1024, kSwizzle128B);
                            const uint64_t bd = smem_desc(
                                pbase + (qq >> 1) * (RP * 128) + (qq & 1) * 64 + ks * 32, 16,
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
            mma_commit(smem_u32(&sm.odone));  // tracks every MMA issued above
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------------------------------------------------------- V decode
        const int dt = tid - 128;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t & 1;
            if (!ctx.wait_warp(&sm.vfull[s], (t >> 1) & 1)) break;
            const uint8_t* raw = smem + kOffVRaw + s * kVRawStage;
            const int tile0 = start + t * kTile;
            bool ok = true;
#pragma unroll 1
            for (int qq = 0; qq < kTile / kQuarter; ++qq) {
                const int u = 4 * t + qq;
                const int vs = u & 1;
                if (!ctx.wait_warp(&sm.vhempty[vs], ((u >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                uint8_t* vh = smem + kOffVh + vs * kVhStage;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int id = i * 128 + dt;
                    const int key = id >> 4, c = id & 15;
                    const int kk = qq * kQuarter + key;
                    uint4 f0 = make_uint4(0, 0, 0, 0), f1 = make_uint4(0, 0, 0, 0);
                    if (tile0 + kk < end) {
                        const uint4 w = *reinterpret_cast<const uint4*>(raw + kk * kHeadDim + c * 16);
                        e4m3x4_to_f16x4(w.x, f0.x, f0.y);
                        e4m3x4_to_f16x4(w.y, f0.z, f0.w);
                        e4m3x4_to_f16x4(w.z, f1.x, f1.y);
                        e4m3x4_to_f16x4(w.w, f1.z, f1.w);
                    }
                    *reinterpret_cast<uint4*>(vh + vh_off(c * 16, key)) = f0;
                    *reinterpret_cast<uint4*>(vh + vh_off(c * 16 + 8, key)) = f1;
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.vhfull[vs]));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.vempty[s]));
            if (!ok) break;
        }
    } else if (warp >= 8) {
        // ---------------------------------------------------------------- softmax
        const int st = tid - 256;  // key of the tile = tensor-memory lane
        const int wq = warp - 8;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int qoff = n - p.q_len;  // row r sees keys j <= qoff + r / G
        uint32_t wg_phase = 0;
        bool alive = true;
        float lsum[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) lsum[r] = 0.f;
        for (int t = 0; t < ntiles; ++t) {
            const int s = t & 1;
            const uint32_t ph = (t >> 1) & 1;
            const int tile0 = start + t * kTile;
            const int j = tile0 + st;
            if (!ctx.wait_warp(&sm.sfull[s], ph)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const uint32_t sbase = lane_base + kColS + s * kSStride;
            const bool tile_all = (tile0 + kTile <= end) && (tile0 + kTile - 1 <= qoff);
            // pass 1: does any score exceed its row's reference max by more than 2^8?
            bool need = false;
#pragma unroll
            for (int rc = 0; rc < RP / 16; ++rc) {
                uint32_t a0[16], a1[16], a2[16];
                load_s(sbase, RP, rc, a0, a1, a2);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = rc * 16 + e;
                    const float2 rp = sm.rowp[r];
                    const float x =
                        (f32(a0[e]) + f32(a1[e]) * 0.0625f + f32(a2[e]) * 0.00390625f) * rp.x;
                    const bool valid =
                        r < R && (tile_all || (j < end && j <= qoff + r / G));
                    need |= valid && (x > rp.y + kLazyThreshold);
                }
            }
            const unsigned any = __ballot_sync(0xffffffffu, need);
            if (lane == 0) sm.vote[t & 1][wq] = any != 0;
            if (!wg_sync(ctx, wg_phase)) {
                alive = false;
                break;
            }
            const bool need_any =
                sm.vote[t & 1][0] | sm.vote[t & 1][1] | sm.vote[t & 1][2] | sm.vote[t & 1][3];
            bool ok = true;
            if (need_any) {
                // exact tile maximum per row, new reference max, rescale of row sums and O
#pragma unroll
                for (int rc = 0; rc < RP / 16; ++rc) {
                    uint32_t a0[16], a1[16], a2[16];
                    load_s(sbase, RP, rc, a0, a1, a2);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int r = rc * 16 + e;
                        const float x = (f32(a0[e]) + f32(a1[e]) * 0.0625f +
                                         f32(a2[e]) * 0.00390625f) * sm.rowp[r].x;
                        const bool valid =
                            r < R && (tile_all || (j < end && j <= qoff + r / G));
                        const float m = warp_max(valid ? x : -INFINITY);
                        if (lane == 0) sm.red[wq][r] = m;
                    }
                }
                ok = wg_sync(ctx, wg_phase);
                float mnew_own = -INFINITY;
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    const float mo = sm.rowp[r].y;
                    const float tm = fmaxf(fmaxf(sm.red[0][r], sm.red[1][r]),
                                           fmaxf(sm.red[2][r], sm.red[3][r]));
                    const float mn = fmaxf(mo, tm);
                    const float alpha = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
                    lsum[r] *= alpha;
                    if (r == st) {
                        mnew_own = mn;
                        sm.alpha[r] = alpha;
                    }
                }
                ok = ok && wg_sync(ctx, wg_phase);
                if (st < RP) sm.rowp[st].y = mnew_own;
                if (ok && t > 0) {
                    // O holds tiles < t: wait for their PV, then scale its row columns
                    ok = ctx.wait_warp(&sm.pempty[(t - 1) & 1], ((t - 1) >> 1) & 1);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh) {
#pragma unroll
                            for (int rc = 0; rc < RP / 16; ++rc) {
                                uint32_t o[16];
                                const uint32_t oaddr = lane_base + kColO + dh * kOStride + rc * 16;
                                tmem_ld16(oaddr, o);
                                tmem_ld_wait(o);
#pragma unroll
                                for (int e = 0; e < 16; ++e)
                                    o[e] = __float_as_uint(f32(o[e]) * sm.alpha[rc * 16 + e]);
                                tmem_st16(oaddr, o);
                            }
                        }
                        tmem_st_wait();
                    }
                }
                ok = ok && wg_sync(ctx, wg_phase);
            }
            // pass 2: probabilities -> FP16 P tile (K-major, 128-byte swizzle), row sums in FP32
            if (ok) ok = ctx.wait_warp(&sm.pempty[s], ph ^ 1);
            if (!ok) {
                alive = false;
                break;
            }
            uint8_t* pbuf = smem + kOffP + s * kPStage;
            const int pcol = st >> 6, pw = (st & 63) * 2;
#pragma unroll
            for (int rc = 0; rc < RP / 16; ++rc) {
                uint32_t a0[16], a1[16], a2[16];
                load_s(sbase, RP, rc, a0, a1, a2);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = rc * 16 + e;
                    const float2 rp = sm.rowp[r];
                    const float x =
                        (f32(a0[e]) + f32(a1[e]) * 0.0625f + f32(a2[e]) * 0.00390625f) * rp.x;
                    const bool valid =
                        r < R && (tile_all || (j < end && j <= qoff + r / G));
                    const float pj = valid ? ex2(x - rp.y) : 0.f;
                    lsum[r] += pj;
                    const uint32_t off = pcol * (RP * 128) + (r >> 3) * 1024 + (r & 7) * 128 +
                                         ((((pw >> 4) ^ (r & 7))) << 4) + (pw & 15);
                    *reinterpret_cast<__half*>(pbuf + off) = __float2half_rn(pj);
                }
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(smem_u32(&sm.sempty[s]));
                mbar_arrive(smem_u32(&sm.pfull[s]));
            }
        }
        // row sums over the 128 key lanes -> split state
#pragma unroll
        for (int r = 0; r < RP; ++r) {
            const float v = warp_sum(lsum[r]);
            if (lane == 0) sm.red[wq][r] = v;
        }
        if (alive) alive = wg_sync(ctx, wg_phase);
        if (alive && st < R && !sm.abort) {
            const int64_t unit = ((int64_t)b * p.num_kv_heads + h) * p.num_splits + split;
            const float L = sm.red[0][st] + sm.red[1][st] + sm.red[2][st] + sm.red[3][st];
            p.ws_state[unit * R + st] = make_float2(sm.rowp[st].y, L);
        }
    }

    // ---- epilogue: O^T (tensor memory, lane = head-dim element) -> numerator rows -----------
    if (warp >= 4) {
        const int dh = warp >= 8 ? 0 : 1;
        const int wq = warp & 3;
        const bool ok = ctx.wait_warp(&sm.odone, 0);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok && !*reinterpret_cast<volatile int*>(&sm.abort))) {
            const float vs = __ldg(p.v_scale);
            const int d = dh * 128 + wq * 32 + lane;
            const int64_t unit = ((int64_t)b * p.num_kv_heads + h) * p.num_splits + split;
            const uint32_t base = tmem + ((uint32_t)(wq * 32) << 16) + kColO + dh * kOStride;
#pragma unroll
            for (int rc = 0; rc < RP / 16; ++rc) {
                uint32_t o[16];
                tmem_ld16(base + rc * 16, o);
                tmem_ld_wait(o);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = rc * 16 + e;
                    if (r < R) p.ws_acc[(unit * R + r) * kHeadDim + d] = f32(o[e]) * vs;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
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
    CUresult r1 = encode(
        &kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.k_pool), dims, strides,
        kbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = encode(
        &vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.v_pool), dims, strides,
        vbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
    dim3 grid(p.num_splits, p.num_kv_heads, p.batch);
    cudaError_t e = cudaSuccess;
    switch (rp) {
        case 16:
            e = cudaFuncSetAttribute(tc::tc_partial_kernel<16>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
            if (e == cudaSuccess)
                tc::tc_partial_kernel<16><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(kmap, vmap, p);
            break;
        case 32:
            e = cudaFuncSetAttribute(tc::tc_partial_kernel<32>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
            if (e == cudaSuccess)
                tc::tc_partial_kernel<32><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(kmap, vmap, p);
            break;
        default:
            e = cudaFuncSetAttribute(tc::tc_partial_kernel<48>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
            if (e == cudaSuccess)
                tc::tc_partial_kernel<48><<<grid, tc::kThreads, tc::kSmemBytes, stream>>>(kmap, vmap, p);
            break;
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dflash
