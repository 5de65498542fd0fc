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
//  * Q (FP16) is split into three E4M3 terms q * 2^a = t0 + t1/16 + t2/256 (per-row power-of-two
//    a, which puts the row's largest magnitude in (224, 448]), stacked on N (N = 3 x rows); the
//    score is (S0 + S1/16 + S2/256) * 2^-a * k_scale / 16 * log2 e. Each residual is exact, so
//    the split is exact for every element of at least 2^-7 after scaling (2^-15 of the row
//    maximum): three 4-bit significands cover FP16's 11 bits. Smaller elements lose low bits to
//    the third term's subnormal grid, an absolute error of at most 2^-18 after scaling, below
//    2^-25 of the row maximum.
//  * The probabilities, taken as p = 2^(s - m) * 2^score with s = 4 and a reference max m (so
//    p <= 2^8, see below), are split the same way into three E4M3 terms p = h + m/16 + l/256
//    (h and m truncated to 4 significant bits, residuals exact, l rounded: relative error about
//    2^-12, finer than an FP16 P), stacked on N, so O^T accumulates three FP32 terms that are
//    summed at the end. The shift s keeps the leading
//    term out of E4M3's subnormal range down to p = 2^-10 of the reference: below 2^-6 the
//    leading term only has a 2^-9 grid, and over 10^5 keys those roundings add up.
//  * Softmax: keys on tensor-memory lanes (thread = key); RP/16 warpgroups of 16 query rows each.
//    Each keeps, per row, a reference max that only moves when a score exceeds it by more than
//    2^(8 - s) (then the warpgroup rescales its O columns in tensor memory), and FP32 row sums of
//    the unrounded (shifted) probabilities, reduced across the key lanes once per split. The
//    split state keeps m - s as its max, which makes the shift invisible to the combine.
//  * Warp roles: warps 0, 2 and 3 share the copies of K (TMA, 3 stages of 128 keys) and V (2
//    stages), each a fixed third of every tile's 16-key page chunks; the last ragged V stage is
//    copied whole by one of them, which zeroes its keys past the context (a zero probability must
//    not meet a NaN code). Three K stages against two V stages: a K copy lands about 2 us after
//    it is issued under load and tile t+3's copy waits for QK of tile t, while V of a tile is
//    needed only after its softmax (at 48 rows the softmax warpgroups and the V ring together
//    set the tile period: V of tile t, copied once PV of tile t-2 is done, lands about as P of
//    tile t is written; the other split, 2 K + 3 V, makes K late instead). Warp 1 owns tensor
//    memory and issues the MMAs from one thread that polls both streams (QK of the next tile, PV
//    of the next V stage) without blocking on either; warps 4.. stage the Q terms (while the
//    first copies are in flight), then run the softmax and write O out. The copies come from
//    three warps: on this GPU the copy throughput of one SM grows with the number of warps
//    issuing them (4.4, 6.2 and 6.6 TB/s over the whole GPU for one, two and three warps; two
//    warps measured slower in this kernel too).
//  * One P buffer: the softmax warp of lane quadrant q writes keys [32q, 32q + 32) of every
//    tile once the PV of the previous tile has read them; the PV of a tile waits for one
//    barrier that every softmax warp arrives on (one test for the MMA thread to poll).
//  * The softmax math runs on FP32 pairs (f32x2 instructions). A warpgroup synchronises on a
//    hardware named barrier (one per group), whose reduction also carries the vote on moving the
//    reference max.
//  * Optionally (fused combine) the CTAs of one launch meet at a grid barrier once every split
//    state is written and merge the splits themselves.
//    Every wait on another warp's or the copy engine's progress is bounded: on timeout the CTA
//    sets DFLASH_FLAG_KERNEL_TIMEOUT, drains its copies and returns. A softmax warp whose wait
//    gave up still runs the rest of its tiles without work, so the four warps of a group always
//    reach the same named barriers.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>

#include <cstddef>
#include <mutex>
#include <type_traits>

#include "combine_impl.cuh"
#include "common.cuh"
#include "e4m3.cuh"
#include "tc_ptx.cuh"

namespace dflash {
namespace tc {

using namespace ptx;

constexpr int kTile = 128;    // keys per tile = MMA M
constexpr int kChunk = 16;    // keys per TMA box (pages are multiples of 16 tokens)
constexpr int kVKeys = 128;   // keys per V stage (a whole tile: four 32-key MMA steps)
constexpr int kTerms = 3;     // E4M3 terms of Q and of P
constexpr int kMaxRP = 48;    // padded rows per KV head this kernel carries
constexpr int kGroupRows = 16;
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSteps = kVKeys / 32;  // 32-key MMA steps of a V stage (one per lane quadrant)

// K and V stages hold their 16-key chunks (one 4 KB page box each) back to back; inside a chunk,
// [8-key group i][head-dim half h][key e][128 bytes] with the 128-byte swizzle, so the 8-key group
// g of the stage (keys 8g..8g+7) of half h starts at g * kGroupStride + h * kHalfOffset: one
// uniform group stride for the MMA descriptors, keys in their natural order.
constexpr uint32_t kKStage = kTile * kHeadDim;   // 32768
constexpr uint32_t kVStage = kVKeys * kHeadDim;  // 32768
constexpr uint32_t kChunkBytes = kChunk * kHeadDim;  // 4096
constexpr uint32_t kGroupStride = 2048;              // 8 keys x both halves
constexpr uint32_t kHalfOffset = 1024;               // 8 keys x 128 bytes
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
    static constexpr uint32_t kOffSmall = kOffP + kPStage;  // one P buffer, reused per tile
    static constexpr uint32_t kColS = 0, kColO = SN;
    static constexpr uint32_t kTmemCols = 3 * SN <= 256 ? 256 : 512;
    static_assert(RP % kGroupRows == 0 && RP <= kMaxRP, "rows per CTA");
    static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0, "swizzled stages need 1 KB alignment");
    static_assert(kOffSmall % 16 == 0, "Small must start 16-byte aligned");
    static_assert(3 * SN <= 512, "tensor memory budget");
};

struct Small {
    uint64_t kfull[kKStages], kempty[kKStages], sfull, sempty;
    uint64_t pfull;  // P of the current tile written (one arrival per softmax warp)
    uint64_t vfull[kVStages], vfree[kVStages], vtail;
    uint64_t odone, qready;
    uint32_t tmem_base;
    int abort;
    float vscale;  // v_scale, loaded while Q is staged (read after the last PV)
    alignas(16) float c0[kMaxRP];  // score scale of each row (log2 units per MMA unit), as float4
    float rmax[kMaxRP / kGroupRows][4][kGroupRows];  // per-group, per-warp row maxima of a tile
    float rsum[kMaxRP / kGroupRows][4][kGroupRows];  // per-group, per-warp row sums of the split
    float mref[kMaxRP / kGroupRows][kGroupRows];     // the split state's max (m - s) of each row
    float nmcur[kMaxRP / kGroupRows][4][kGroupRows];  // each warp's copy of s - reference max
    int rows[kRowCache];  // source row (physical page * page + slot) of chunk c of the split
};
static_assert(offsetof(Small, c0) % 16 == 0, "row constants are read as float4");

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

// Bounded wait on an mbarrier phase (try_wait lets the hardware suspend the thread meanwhile):
// gives up when the CTA's abort flag is raised or after kWaitLimitNs.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, const volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 7) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

struct Ctx {
    Small* sm;
    int32_t* status;
    __device__ bool wait(uint64_t* bar, uint32_t parity) const {
        if (bar_wait(smem_u32(bar), parity, &sm->abort)) return true;
        *reinterpret_cast<volatile int*>(&sm->abort) = 1;
        atomicOr(status, DFLASH_FLAG_KERNEL_TIMEOUT);
        return false;
    }
    // The same for code run by a whole warp: every lane waits (the hardware suspends and wakes
    // the warp as one; a wait by lane 0 with the others held at a shuffle measured slower), and
    // the warp agrees on the result, so that no later warp-synchronous instruction runs with part
    // of the warp gone.
    __device__ bool wait_warp(uint64_t* bar, uint32_t parity) const {
        const bool ok = wait(bar, parity);
        return __all_sync(0xffffffffu, ok);
    }
    __device__ bool aborted() const { return *reinterpret_cast<volatile int*>(&sm->abort) != 0; }
};

// Hardware barrier of one softmax warpgroup (named barrier 1 + g, its 128 threads), optionally
// OR-reducing a predicate over them. Every warp of the group runs every tile (a failed wait
// skips work, never the loop), so each barrier is always reached by all four warps.
__device__ __forceinline__ bool group_vote(int g, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pv, pr;\n\t"
        "setp.ne.u32 pv, %1, 0;\n\t"
        "bar.red.or.pred pr, %2, 128, pv;\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(1 + g)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void group_bar(int g) {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
}

// (pool row, clamped?) of key j0 of sequence b from the block table, for splits longer than the
// row cache (out of line: the copiers' common path stays compact)
__device__ __noinline__ int2 table_row(const int32_t* block_table, int b, int max_pages_per_seq,
                                       int page_size, int num_pages, int j0) {
    bool clamped = false;
    const int phys = physical_page(block_table, b, max_pages_per_seq, j0 / page_size, num_pages,
                                   &clamped);
    return make_int2(phys * page_size + (j0 % page_size), clamped ? 1 : 0);
}

// Source row in the page pool of the 16-key chunk starting at key j0 of sequence b: read from the
// split's cache when the chunk is in it, else straight from the block table.
__device__ __forceinline__ int chunk_row(const PartialParams& p, const Small& sm, int b, int start,
                                         int j0, bool* clamped) {
    const int c = (j0 - start) / kChunk;
    if (c < kRowCache) return sm.rows[c];
    const int2 r = table_row(p.block_table, b, p.max_pages_per_seq, p.page_size, p.num_pages, j0);
    if (r.y) *clamped = true;
    return r.x;
}

// The three term slices (columns base, base + RP, base + 2RP) of this lane's 16 rows, combined
// as t0 + t1/16 + t2/256 (the three loads in flight together, one wait).
template <int RP>
__device__ __forceinline__ void load_terms16(uint32_t taddr, float (&y)[kGroupRows]) {
    uint32_t a0[16], a1[16], a2[16];
    tmem_ld16(taddr, a0);
    tmem_ld16(taddr + RP, a1);
    tmem_ld16(taddr + 2 * RP, a2);
    tmem_ld_wait(a0);
    tmem_ld_wait(a1);
    tmem_ld_wait(a2);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        y[i] = fmaf(f32(a2[i]), 0.00390625f, fmaf(f32(a1[i]), 0.0625f, f32(a0[i])));
}

// Grid-wide barrier of one launch (thread 0 of every CTA) on a 64-bit ticket counter: CTA tickets
// of one launch fall in one block of 2^20 values, the barrier opens when the counter reaches the
// block base + the CTA count, and the last arrival moves the counter to the next block (so plans
// of any grid size can share a workspace). One atomic per CTA and no reset on the critical path.
// Bounded: on timeout the status word gets DFLASH_FLAG_KERNEL_TIMEOUT and false is returned (the
// counter is then off until the caller zeroes the workspace header). Every CTA must be resident,
// which the cooperative launch guarantees.
__device__ __forceinline__ bool grid_barrier(unsigned long long* ctr, uint32_t num_ctas,
                                             int32_t* status) {
    constexpr unsigned long long kBlock = 1ull << 20;
    __threadfence();  // this CTA's split state is written before it arrives
    const unsigned long long t = atomicAdd(ctr, 1ull);
    const unsigned long long base = t & ~(kBlock - 1);
    if (t - base == num_ctas - 1) {  // last arrival: every state is written
        atomicAdd(ctr, kBlock - num_ctas);
        __threadfence();
        return true;
    }
    const unsigned long long target = base + num_ctas;
    const volatile unsigned long long* vctr = ctr;
    const uint64_t t0 = globaltimer_ns();
    while (*vctr < target) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, DFLASH_FLAG_KERNEL_TIMEOUT);
            return false;
        }
        __nanosleep(32);
    }
    __threadfence();
    return true;
}

// The merge of a fused launch: once every CTA has written its split state, the CTAs share the
// (query row, head-dim quarter, sequence x KV head) items of the combine, 256 threads per item
// (each 256-thread half of the CTA has its own named barrier and scratch at the base of the
// CTA's shared memory, unused by then).
template <int NT>
__device__ __forceinline__ void fused_merge(const PartialParams& p, uint8_t* smem) {
    constexpr int kHalves = NT / kCombineThreads;
    constexpr int kQuarters = kHeadDim / (4 * kCombineCols);
    volatile int* barrier_ok =
        reinterpret_cast<volatile int*>(smem + kHalves * sizeof(CombineScratch));
    const int half = threadIdx.x / kCombineThreads;
    const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const int workers = gridDim.x * gridDim.y * gridDim.z * kHalves;
    const int items = p.batch * p.num_kv_heads * p.rows * kQuarters;
    const int first = cta * kHalves + half;
    __syncthreads();
    if (threadIdx.x == 0)
        *barrier_ok = grid_barrier(p.grid_bar, gridDim.x * gridDim.y * gridDim.z, p.status);
    __syncthreads();
    if (!*barrier_ok) return;
    if (half >= kHalves) return;
    CombineParams c;
    c.ws_state = p.ws_state;
    c.ws_acc = p.ws_acc;
    c.context_lens = p.context_lens;
    c.out = p.out;
    c.lse = p.lse;
    c.batch = p.batch;
    c.q_len = p.q_len;
    c.num_q_heads = p.num_q_heads;
    c.num_kv_heads = p.num_kv_heads;
    c.group = p.group;
    c.rows = p.rows;
    c.max_context = p.max_context;
    c.num_splits = p.num_splits;
    c.num_slots = p.num_slots;
    c.tile_keys = p.tile_keys;
    c.min_split_keys = p.min_split_keys;
    CombineScratch& sh = reinterpret_cast<CombineScratch*>(smem)[half];
    for (int it = first; it < items; it += workers) {
        const int quarter = it % kQuarters, r = (it / kQuarters) % p.rows;
        const int unit = it / (kQuarters * p.rows);
        const UnitSlots us = locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                          p.num_slots, p.max_context, p.q_len, unit, false);
        combine_item(c, r, quarter, unit / p.num_kv_heads, unit % p.num_kv_heads,
                     threadIdx.x % kCombineThreads, 1 + half, sh, us.first, us.count, us.n);
    }
}

// kFused: the instance that merges the splits after the grid barrier (p.out set); the other
// carries no merge code at all.
template <int RP, bool kFused>
__global__ void __launch_bounds__(Cfg<RP>::kThreads, 1)
    tc_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PartialParams p) {
    using C = Cfg<RP>;
    extern __shared__ __align__(1024) uint8_t smem[];
    Small& sm = *reinterpret_cast<Small*>(smem + C::kOffSmall);
    constexpr int SN = C::SN;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // rows [row_lo, row_lo + R) of the slot: all of them unless R > 48 (row blocks)
    const RowBlock rblk = row_block(p);
    const int R = rblk.rows, row_lo = rblk.row_lo, G = p.group, P = p.page_size;
    // With programmatic dependent launch the next kernel's CTAs may be scheduled from here on
    // (onto SMs this grid leaves free); it waits for this grid's completion before it reads the
    // workspace.
    griddep_launch_dependents();

    // This CTA's workspace slot, and which (sequence, KV head) unit owns it, follow from every
    // context length (slots are shared out by length), a load away. For a batch of equal lengths
    // slot (x, y, z) belongs to split x of KV head y of sequence z, and the split's key range is
    // the one a context of max_context keys gives whenever the split size comes out the same
    // (split sizes are whole tiles, so any context close to max_context): thread c looks up
    // chunk c of that range while the lengths are in flight, and the row cache below takes it if
    // the guess holds.
    // (divisions by the page size become shifts for power-of-two pages, and the tile size is
    // this kernel's constant: the set-up's dependent chain is short)
    const int per_max = p.per_max;
    int page_max = 0;
    if (tid < kRowCache && rblk.xs * per_max + tid * kChunk < p.max_context) {
        const int j = rblk.xs * per_max + tid * kChunk;
        page_max = p.block_table[(int64_t)blockIdx.z * p.max_pages_per_seq +
                                 (p.page_shift >= 0 ? j >> p.page_shift : j / P)];
    }
    const int slot = rblk.slot;
    // a single sequence's unit is the grid row (KV head): no search, no division
    const UnitSlots us =
        p.batch == 1 ? locate_slots_single(p.context_lens, p.num_kv_heads, p.num_splits,
                                           p.max_context, p.q_len, blockIdx.y, false)
                     : locate_slots(p.context_lens, p.batch, p.num_kv_heads, p.num_splits,
                                    p.num_slots, p.max_context, p.q_len, slot, true);
    if (slot == 0 && tid == 0 && us.flags) atomicOr(p.status, us.flags);
    const int b = us.b, h = us.h, split = slot - us.first, n = us.n;
    int per = 1;
    if (b >= 0) {  // keys_per_split with this kernel's tile size
        per = max((n + us.count - 1) / us.count, p.min_split_keys);
        per = (per + kTile - 1) / kTile * kTile;
    }
    const int start = split * per;
    if (b < 0 || start >= n) {  // idle slot: the combine never reads it
        if constexpr (kFused) fused_merge<C::kThreads>(p, smem);
        return;
    }
    const bool guessed = b == (int)blockIdx.z && split == rblk.xs && per == per_max;
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
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(smem_u32(&sm.kfull[i]), 3);  // one arrival per copying warp
            mbar_init(smem_u32(&sm.kempty[i]), 1);
        }
        mbar_init(smem_u32(&sm.sfull), 1);
        mbar_init(smem_u32(&sm.sempty), C::kSoftWarps);
        mbar_init(smem_u32(&sm.pfull), C::kSoftWarps);
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(smem_u32(&sm.vfull[i]), 3);  // one arrival per copying warp
            mbar_init(smem_u32(&sm.vfree[i]), 1);
        }
        mbar_init(smem_u32(&sm.vtail), 1);
        mbar_init(smem_u32(&sm.odone), 1);
        mbar_init(smem_u32(&sm.qready), C::kSoftWarps);
        sm.abort = 0;
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
            const int lp = p.page_shift >= 0 ? j0 >> p.page_shift : j0 / P;
            const int phys = (guessed && c == tid)
                                 ? clamp_page(page_max, p.num_pages, &clamped)
                                 : physical_page(p.block_table, b, p.max_pages_per_seq, lp,
                                                 p.num_pages, &clamped);
            sm.rows[c] = phys * P + (j0 - lp * P);
        }
        if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0 || warp == 2 || warp == 3) {
        // --------------------------------------------------------- K and V copies (TMA)
        // Three warps share the copies of every tile: one warp's TMA instruction stream issues
        // about 15 boxes a microsecond, an SM about 22, and a tile takes 32 (16-key chunks, two
        // 128-byte halves, K and V). Copier ci owns the K chunks c with c % 3 == ci and the V
        // chunks with c % 3 == (ci + 1) % 3, and arrives once per K tile and per V stage with the
        // bytes of its own copies. The copiers take the stages in the order in which the MMAs
        // release them: K tiles 0-2 and V stages 0-1 at once, then K tile t + 2 before V stage t
        // (QK of tile t - 1 is issued, and so completes, before PV of tile t - 2). Each waits for
        // its next stage with the hardware-suspended mbarrier wait instead of polling: the copier
        // warps share their SM sub-partitions with softmax warps, whose issue slots polling
        // takes, and a copy has more than a tile of slack. A ragged last V stage is copied whole
        // by copier 1, which zeroes its keys past the split's end once they have landed (P is
        // zero there, but a stale NaN code times zero is NaN); the others only arrive on it.
        const int ci = warp == 0 ? 0 : (warp == 2 ? 1 : 2);
        const uint64_t stream = l2_evict_first_policy();  // every page is read once
        constexpr int kChunks = kTile / kChunk;          // 8 per K tile and per V stage
        constexpr int kOwn = (kChunks + 2) / 3;           // at most 3 chunks per copier
        static_assert(kVKeys == kTile, "one V stage per tile");
        bool clamped = false;
        // the pool rows of this copier's chunks of K tile tk and V stage tv, looked up ahead
        auto own_rows = [&](int tile0, int first, int (&rows)[kOwn]) {
#pragma unroll
            for (int k = 0; k < kOwn; ++k) {
                const int c = first + 3 * k;
                const int j0 = tile0 + kChunk * c;
                rows[k] = (c < kChunks && j0 < end) ? chunk_row(p, sm, b, start, j0, &clamped) : -1;
            }
        };
        const int kfirst = ci, vfirst = (ci + 1) % 3;
        // Keys from n - q_len on (the drafted tokens) may be written by the kernel just before
        // this one (their KV write): tiles reaching them are copied only after griddep_wait,
        // which returns at once unless this grid is a programmatic dependent.
        const int drafted = n - p.q_len;
        bool dep_done = false;
        int krows[kOwn], vrows[kOwn];
        if (lane == 0) {
            own_rows(start, kfirst, krows);
            own_rows(start, vfirst, vrows);
        }
        int tk = 0, tv = 0;
        bool tail_pending = false;  // the ragged stage's copies are issued but not awaited
        while (tk < ntiles || tv < nvst) {
            // K tile tk next, or V stage tv (every lane waits for the stage's release, which
            // also orders the tail's zeroing stores below after the MMAs that read the stage)
            const bool k_next = tk < ntiles && (tv >= nvst || tk < kKStages ||
                                                (tv >= kVStages && tk <= tv + 2));
            if (k_next) {
                if (!ctx.wait_warp(&sm.kempty[tk % kKStages], ((tk / kKStages) & 1) ^ 1)) break;
            } else if (!ctx.wait_warp(&sm.vfree[tv % kVStages], ((tv / kVStages) & 1) ^ 1)) {
                break;
            }
            if (k_next) {
                if (lane == 0) {
                    if (!dep_done && start + (tk + 1) * kTile > drafted) {
                        griddep_wait();
                        dep_done = true;
                    }
                    const int s = tk % kKStages;
                    const uint32_t bar = smem_u32(&sm.kfull[s]);
                    int nval = 0;
#pragma unroll
                    for (int k = 0; k < kOwn; ++k) nval += krows[k] >= 0;
                    mbar_arrive_expect_tx(bar, nval * kChunk * kHeadDim);
                    const uint32_t dst = smem_u32(smem + C::kOffK + s * kKStage);
#pragma unroll
                    for (int k = 0; k < kOwn; ++k) {
                        if (krows[k] < 0) continue;
                        tma_load_4d(dst + (kfirst + 3 * k) * kChunkBytes, &kmap, 0, 0, 2 * h,
                                    krows[k] / 8, bar, stream);
                    }
                    if (tk + 1 < ntiles) own_rows(start + (tk + 1) * kTile, kfirst, krows);
                }
                ++tk;
            } else {
                const int vs = tv % kVStages;
                const int h0 = start + tv * kVKeys;
                const int nkeys = min(kVKeys, end - h0);
                uint8_t* vstage = smem + C::kOffV + vs * kVStage;
                if (lane == 0 && !dep_done && h0 + kVKeys > drafted) {
                    griddep_wait();
                    dep_done = true;
                }
                if (nkeys == kVKeys) {
                    if (lane == 0) {
                        const uint32_t bar = smem_u32(&sm.vfull[vs]);
                        int nval = 0;
#pragma unroll
                        for (int k = 0; k < kOwn; ++k) nval += vrows[k] >= 0;
                        mbar_arrive_expect_tx(bar, nval * kChunk * kHeadDim);
                        const uint32_t dst = smem_u32(vstage);
#pragma unroll
                        for (int k = 0; k < kOwn; ++k) {
                            if (vrows[k] < 0) continue;
                            tma_load_4d(dst + (vfirst + 3 * k) * kChunkBytes, &vmap, 0, 0, 2 * h,
                                        vrows[k] / 8, bar, stream);
                        }
                    }
                } else if (ci == 1) {
                    if (lane == 0) {
                        const int nval = (nkeys + kChunk - 1) / kChunk;  // chunks holding a key
                        const uint32_t bar = smem_u32(&sm.vtail);
                        mbar_arrive_expect_tx(bar, nval * kChunk * kHeadDim);
                        const uint32_t dst = smem_u32(vstage);
#pragma unroll 1
                        for (int c = 0; c < nval; ++c) {
                            const int row = chunk_row(p, sm, b, start, h0 + kChunk * c, &clamped);
                            tma_load_4d(dst + c * kChunkBytes, &vmap, 0, 0, 2 * h, row / 8, bar,
                                        stream);
                        }
                    }
                    tail_pending = true;
                    if (!ctx.wait_warp(&sm.vtail, 0)) break;
                    tail_pending = false;
                    // keys nkeys..127 (page-tail slots or never-copied rows); a key's 128 bytes
                    // per half are contiguous (the swizzle permutes 16-byte units inside them)
                    const int zero_units = (kVKeys - nkeys) * 16;  // 16-byte units, both halves
                    for (int i = lane; i < zero_units; i += 32) {
                        const int key = nkeys + i / 16, dh = (i / 8) & 1, u = i & 7;
                        *reinterpret_cast<uint4*>(vstage + (key / 8) * kGroupStride +
                                                  dh * kHalfOffset + (key % 8) * 128 + u * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sm.vfull[vs]));
                } else {
                    if (lane == 0) mbar_arrive(smem_u32(&sm.vfull[vs]));
                }
                if (lane == 0 && tv + 1 < nvst) own_rows(h0 + kVKeys, vfirst, vrows);
                ++tv;
            }
        }
        if (lane == 0) {
            if (clamped) atomicOr(p.status, DFLASH_FLAG_PAGE_CLAMPED);
            // no copy of this warp may still be writing shared memory when the CTA retires
            for (int t = tk - kKStages < 0 ? 0 : tk - kKStages; t < tk; ++t)
                mbar_wait(smem_u32(&sm.kfull[t % kKStages]), (t / kKStages) & 1, &sm.abort,
                          kWaitLimitNs);
            for (int u = tv - kVStages < 0 ? 0 : tv - kVStages; u < tv; ++u) {
                if (end - (start + u * kVKeys) < kVKeys) {
                    if (tail_pending) mbar_wait(smem_u32(&sm.vtail), 0, &sm.abort, kWaitLimitNs);
                } else {
                    mbar_wait(smem_u32(&sm.vfull[u % kVStages]), (u / kVStages) & 1, &sm.abort,
                              kWaitLimitNs);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // One thread, one event loop over two streams: QK of tile tq (its K copies landed and the
        // softmax has read the previous scores) and PV of V stage up (its copies and the tile's
        // probabilities are written). Polling both without blocking keeps a QK from queueing behind
        // a PV whose V copies are late, and vice versa. When both are ready PV goes first: it
        // frees the P buffer the softmax writes next and the V stage the next copy fills, while
        // the scores of QK are needed only once the softmax is through the current tile (issuing
        // eight MMAs blocks this thread while the tensor pipe drains the ones before them).
        if (lane == 0 && ctx.wait(&sm.qready, 0)) {
            const uint32_t idesc_qk = idesc_f32acc(128, SN, 0, 0, 0, 0);
            const uint32_t idesc_pv = idesc_f32acc(128, SN, 0, 0, 1, 1);
            const uint32_t q_base = smem_u32(smem + C::kOffQ);
            const uint32_t pbase = smem_u32(smem + C::kOffP);
            constexpr int kStagesPerTile = kTile / kVKeys;
            int tq = 0, up = 0;
            uint64_t last = globaltimer_ns();
            uint32_t idle = 0;
            while (tq < ntiles || up < nvst) {
                bool progressed = false;
                if (up < nvst) {
                    const int t = up / kStagesPerTile, hv = up % kStagesPerTile;
                    const int vs = up % kVStages;
                    // both tests issued back to back (no short circuit): their shared-memory
                    // round trips overlap
                    const bool ready =
                        mbar_test_wait(smem_u32(&sm.vfull[vs]), (up / kVStages) & 1) &
                        mbar_test_wait(smem_u32(&sm.pfull), t & 1);
                    if (ready) {
                        // O^T += V^T P^T over this stage's keys, both head-dim halves (the two
                        // MMAs of a 32-key step back to back: they read the same P columns)
                        tc_fence_after();
                        const uint32_t vb = smem_u32(smem + C::kOffV + vs * kVStage);
#pragma unroll
                        for (int kq = 0; kq < kSteps; ++kq) {
                            const int kk = kSteps * hv + kq;  // 32-key step of the tile
                            const uint64_t bd =
                                smem_desc(pbase + kk * 512, 128, 2048, kSwizzleNone);
#pragma unroll
                            for (int dh = 0; dh < 2; ++dh) {
                                // 32 keys = four 8-key groups from group 4 kq on
                                const uint64_t ad =
                                    smem_desc(vb + dh * kHalfOffset + kq * 4 * kGroupStride,
                                              kVStage, kGroupStride, kSwizzle128B);
                                mma_f8_ss(tmem + C::kColO + dh * SN, ad, bd, idesc_pv,
                                          (t | kk) != 0);
                            }
                        }
                        mma_commit(smem_u32(&sm.vfree[vs]));  // V stage and P buffer reusable
                        ++up;
                        progressed = true;
                    }
                }
                if (tq < ntiles &&
                    (mbar_test_wait(smem_u32(&sm.kfull[tq % kKStages]), (tq / kKStages) & 1) &
                     mbar_test_wait(smem_u32(&sm.sempty), (tq & 1) ^ 1))) {
                    // S^T = K Q^T into the single S buffer
                    tc_fence_after();
                    const int s = tq % kKStages;
                    const uint32_t kb = smem_u32(smem + C::kOffK + s * kKStage);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = smem_desc(kb + (kk >> 2) * kHalfOffset + (kk & 3) * 32,
                                                      16, kGroupStride, kSwizzle128B);
                        const uint64_t bd = smem_desc(
                            q_base + (kk >> 2) * (SN * 128) + (kk & 3) * 32, 16, 1024,
                            kSwizzle128B);
                        mma_f8_ss(tmem + C::kColS, ad, bd, idesc_qk, kk > 0);
                    }
                    mma_commit(smem_u32(&sm.kempty[s]));
                    mma_commit(smem_u32(&sm.sfull));
                    ++tq;
                    progressed = true;
                }
                if (progressed) {
                    idle = 0;
                    last = globaltimer_ns();
                } else if ((++idle & 15) == 0) {
                    if (ctx.aborted()) break;
                    if (globaltimer_ns() - last > kWaitLimitNs) {
                        *reinterpret_cast<volatile int*>(&sm.abort) = 1;
                        atomicOr(p.status, DFLASH_FLAG_KERNEL_TIMEOUT);
                        break;
                    }
                }
            }
        }
        if (lane == 0) mma_commit(smem_u32(&sm.odone));  // tracks every MMA issued above
    } else if (warp >= 4) {
        // ------------------------------------------------------------- softmax (RP/16 groups)
        const int sw = warp - 4;          // 0 .. kSoftWarps - 1
        const int g = sw >> 2;            // rows [16 g, 16 g + 16)
        const int wq = warp & 3;          // tensor-memory lane quadrant
        const int st = (wq << 5) | lane;  // key of the tile = tensor-memory lane
        const int row0 = kGroupRows * g;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const int qoff = n - p.q_len;  // row r of the slot sees keys j <= qoff + r / G

        // Q -> three E4M3 terms (one warp per row), row scales. Q and the scales, and every
        // workspace write below, come after the preceding kernel's completion (a no-op unless
        // this grid is its programmatic dependent).
        griddep_wait();
        {
            constexpr int kRowsPerWarp = RP / C::kSoftWarps;  // 4
            const float qk_scale = __ldg(p.k_scale) * 0.0625f * kLog2e;  // D^-1/2 = 1/16
            if (sw == 0 && lane == 0) sm.vscale = __ldg(p.v_scale);  // seen by all after qready
            uint4 qraw[kRowsPerWarp];  // this warp's rows: all loads in flight at once
#pragma unroll
            for (int k = 0; k < kRowsPerWarp; ++k) {
                const int r = sw + C::kSoftWarps * k;
                qraw[k] = make_uint4(0, 0, 0, 0);
                if (r < R) {
                    const int i = (row_lo + r) / G, gg = (row_lo + r) % G;
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
                if (lane == 0) sm.c0[r] = qk_scale * __int_as_float((127 - a) << 23);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.qready));
        }
        bool alive = ctx.wait_warp(&sm.qready, 0);
        // Per-row score scale and s minus the reference max live in shared memory (read as pairs
        // of 64-bit words, identical for every thread of the group). Scores, exponents, row sums
        // and probabilities are handled as FP32 pairs (element i of a 16-row block is word i / 2,
        // half i % 2).
        uint64_t lsum[kGroupRows / 2];
        uint32_t rowmask = 0;
#pragma unroll
        for (int i = 0; i < kGroupRows; ++i) rowmask |= (uint32_t)(row0 + i < R) << i;
#pragma unroll
        for (int i = 0; i < kGroupRows / 2; ++i) lsum[i] = 0;
        const ulonglong2* c0v = reinterpret_cast<const ulonglong2*>(sm.c0 + row0);
        // s minus the reference max of each of the group's rows (+inf: none yet), in pairs; every
        // thread of the group holds the same values (they are computed from shared partials)
        uint64_t nm[kGroupRows / 2];
#pragma unroll
        for (int q = 0; q < kGroupRows / 2; ++q) nm[q] = pk2(INFINITY, INFINITY);
        if (lane < kGroupRows) sm.nmcur[g][wq][lane] = INFINITY;
        __syncwarp();
        const uint64_t k16th = pk2(0.0625f, 0.0625f), k256th = pk2(0.00390625f, 0.00390625f);
        const uint64_t k16 = pk2(16.f, 16.f);
        constexpr uint64_t kTrunc4 = 0xFFF00000FFF00000ull;  // sign, exponent, 3 mantissa bits
        for (int t = 0; t < ntiles; ++t) {
            const int tile0 = start + t * kTile;
            const int j = tile0 + st;
            if (alive && !ctx.wait_warp(&sm.sfull, t & 1)) alive = false;
            tc_fence_after();
            // y = (S0 + S1/16 + S2/256) * c0: the score in log2 units
            uint64_t y[kGroupRows / 2];
            {
                uint32_t a0[16], a1[16], a2[16];
                const uint32_t sbase = lane_base + C::kColS + row0;
                tmem_ld16(sbase, a0);
                tmem_ld16(sbase + RP, a1);
                tmem_ld16(sbase + 2 * RP, a2);
                tmem_ld_wait(a0);
                tmem_ld_wait(a1);
                tmem_ld_wait(a2);
#pragma unroll
                for (int q = 0; q < kGroupRows / 2; ++q)
                    y[q] = fma2(pk2(f32(a2[2 * q]), f32(a2[2 * q + 1])), k256th,
                                fma2(pk2(f32(a1[2 * q]), f32(a1[2 * q + 1])), k16th,
                                     pk2(f32(a0[2 * q]), f32(a0[2 * q + 1]))));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && alive) mbar_arrive(smem_u32(&sm.sempty));  // S free for QK(t+1)
            uint32_t validm = rowmask;  // bit i: key j visible to row row0 + i
            if (!((tile0 + kTile <= end) && (tile0 + kTile - 1 <= qoff))) {
                // row r of the slot (query token r / G) sees key j iff r / G >= j - qoff, that is
                // r >= (j - qoff) G: the group's rows from `first` on
                const int first = (j - qoff) * G - row_lo - row0;
                if (j >= end)
                    validm = 0;
                else if (first > 0)
                    validm &= first >= kGroupRows ? 0u : (0xFFFFFFFFu << first);
            }
            // e = y c0 + (s - m): the exponent of the shifted probability, one fused multiply-add
            // (the scaled score y c0 itself is formed only on the reference-max path); would any
            // visible one exceed 2^8?
            uint64_t e[kGroupRows / 2];
            bool need = false;
#pragma unroll
            for (int i4 = 0; i4 < kGroupRows / 4; ++i4) {
                const ulonglong2 c = c0v[i4];
                e[2 * i4] = fma2(y[2 * i4], c.x, nm[2 * i4]);
                e[2 * i4 + 1] = fma2(y[2 * i4 + 1], c.y, nm[2 * i4 + 1]);
            }
            // Every row of the group sees this key (all but the causal-window and ragged tiles):
            // the per-row visibility tests are skipped below.
            const bool all_rows = validm == 0xFFFFu;
            if (all_rows) {
#pragma unroll
                for (int q = 0; q < kGroupRows / 2; ++q)
                    need |= (lo2(e[q]) > kLazyThreshold) | (hi2(e[q]) > kLazyThreshold);
            } else {
#pragma unroll
                for (int q = 0; q < kGroupRows / 2; ++q) {
                    need |= ((validm >> (2 * q)) & 1u) && lo2(e[q]) > kLazyThreshold;
                    need |= ((validm >> (2 * q + 1)) & 1u) && hi2(e[q]) > kLazyThreshold;
                }
            }
            // shifted probabilities -> three E4M3 terms (this thread's 16 rows of each term are one
            // 16-byte chunk of P); row sums take the unrounded values
            uint64_t pv[kGroupRows / 2];
            uint32_t code[kTerms][4];
            // kAll: every row visible (no per-row tests)
            auto make_p = [&](auto all) {
                constexpr bool kAll = decltype(all)::value;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t ch[2], cm[2], cl[2];
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const int jj = 2 * w + q;
                        const float p0 = (kAll || ((validm >> (2 * jj)) & 1u)) ? ex2(lo2(e[jj]))
                                                                               : 0.f;
                        const float p1 = (kAll || ((validm >> (2 * jj + 1)) & 1u))
                                             ? ex2(hi2(e[jj]))
                                             : 0.f;
                        pv[jj] = pk2(p0, p1);
                        // h, m: truncations to 4 significant bits (mantissa masked), so p - h and
                        // r - m are exact and the three terms sum to p up to l's final rounding
                        const uint64_t hv = pv[jj] & kTrunc4;
                        const uint64_t r = mul2(sub2(pv[jj], hv), k16);
                        const uint64_t mv = r & kTrunc4;
                        const uint64_t lv = mul2(sub2(r, mv), k16);
                        ch[q] = f32x2_to_e4m3x2(hv);
                        cm[q] = f32x2_to_e4m3x2(mv);
                        cl[q] = f32x2_to_e4m3x2(lv);
                    }
                    code[0][w] = ch[0] | (ch[1] << 16);
                    code[1][w] = cm[0] | (cm[1] << 16);
                    code[2][w] = cl[0] | (cl[1] << 16);
                }
            };
            // tile 0 always sets the reference max; later tiles vote on whether to move it
            bool need_any = true;
            if (t > 0) need_any = group_vote(g, need);
            bool ok = true;
            if (need_any) {
                // exact tile maximum per row -> new reference max; rescale row sums and O. The
                // warp's row maxima by a transposed butterfly (lane l ends with row (l >> 1) & 15),
                // the group's through shared memory; lanes 2i and 2i + 1 then derive row i's new
                // reference and weight, which the shuffles below hand to every lane (compact code:
                // tile 0 runs it cold, later tiles rarely)
#pragma unroll
                for (int i4 = 0; i4 < kGroupRows / 4; ++i4) {  // the scaled scores
                    const ulonglong2 c = c0v[i4];
                    y[2 * i4] = mul2(y[2 * i4], c.x);
                    y[2 * i4 + 1] = mul2(y[2 * i4 + 1], c.y);
                }
                {
                    float v[kGroupRows];
#pragma unroll
                    for (int q = 0; q < kGroupRows / 2; ++q) {
                        v[2 * q] = ((validm >> (2 * q)) & 1u) ? lo2(y[q]) : -INFINITY;
                        v[2 * q + 1] = ((validm >> (2 * q + 1)) & 1u) ? hi2(y[q]) : -INFINITY;
                    }
#pragma unroll
                    for (int half = kGroupRows / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
                        const bool upper = (lane & off) != 0;
#pragma unroll
                        for (int j = 0; j < half; ++j) {
                            const float keep = upper ? v[j + half] : v[j];
                            const float send = upper ? v[j] : v[j + half];
                            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, off));
                        }
                    }
                    v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
                    if ((lane & 1) == 0) sm.rmax[g][wq][lane >> 1] = v[0];
                }
                group_bar(g);
                const int ri = (lane >> 1) & (kGroupRows - 1);
                const float mo = kPShift - sm.nmcur[g][wq][ri];
                const float tm = fmaxf(fmaxf(sm.rmax[g][0][ri], sm.rmax[g][1][ri]),
                                       fmaxf(sm.rmax[g][2][ri], sm.rmax[g][3][ri]));
                const float mn = fmaxf(mo, tm);
                const float alpha_r = (mn == -INFINITY) ? 1.f : ex2(mo - mn);
                const float nm_r = (mn == -INFINITY) ? INFINITY : kPShift - mn;
                __syncwarp();  // every lane has read its row's old reference
                if ((lane & 1) == 0) sm.nmcur[g][wq][ri] = nm_r;
                float alpha[kGroupRows];
#pragma unroll
                for (int q = 0; q < kGroupRows / 2; ++q) {
                    alpha[2 * q] = __shfl_sync(0xffffffffu, alpha_r, 4 * q);
                    alpha[2 * q + 1] = __shfl_sync(0xffffffffu, alpha_r, 4 * q + 2);
                    nm[q] = pk2(__shfl_sync(0xffffffffu, nm_r, 4 * q),
                                __shfl_sync(0xffffffffu, nm_r, 4 * q + 2));
                    lsum[q] = mul2(lsum[q], pk2(alpha[2 * q], alpha[2 * q + 1]));
                    e[q] = add2(y[q], nm[q]);
                }
                if (t > 0) {
                    // O holds tiles < t: wait for their PV (MMAs complete in issue order, so
                    // the last V stage of tile t-1 done means all of it), then scale this
                    // group's row columns of all three terms in both head-dim halves
                    const int ul = (kTile / kVKeys) * t - 1;
                    ok = alive && ctx.wait_warp(&sm.vfree[ul % kVStages], (ul / kVStages) & 1);
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
                                o[i] = __float_as_uint(f32(o[i]) * alpha[i]);
                            tmem_st16(addr, o);
                        }
                        tmem_st_wait();
                    }
                }
            }
            if (all_rows)
                make_p(std::true_type{});
            else
                make_p(std::false_type{});
#pragma unroll
            for (int q = 0; q < kGroupRows / 2; ++q) lsum[q] = add2(lsum[q], pv[q]);
            // this warp's keys of P are free once the V stage that consumed them in tile t-1
            // is done
            if (alive && ok && t > 0) {
                const int u = (kTile / kVKeys) * (t - 1);
                ok = ctx.wait_warp(&sm.vfree[u % kVStages], (u / kVStages) & 1);
            }
            if (!ok) alive = false;
            if (!alive) continue;  // every warp still runs the remaining tiles' barriers
            uint8_t* pbuf = smem + C::kOffP;
#pragma unroll
            for (int term = 0; term < kTerms; ++term)
                *reinterpret_cast<uint4*>(pbuf + p_chunk(term * C::kGroups + g, st)) =
                    make_uint4(code[term][0], code[term][1], code[term][2], code[term][3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.pfull));
        }
        // row sums over the 128 key lanes -> split state (max m - s, shifted sums and numerator).
        // A transposed butterfly over the warp: each step trades half of the rows with the lane
        // `off` away, so lane l ends with row (l >> 1) & 15 after 16 shuffles, each sum taken in
        // the order of a plain xor reduction of that row (same bits, far less code).
        {
            float v[kGroupRows];
#pragma unroll
            for (int q = 0; q < kGroupRows / 2; ++q) {
                v[2 * q] = lo2(lsum[q]);
                v[2 * q + 1] = hi2(lsum[q]);
            }
#pragma unroll
            for (int half = kGroupRows / 2, off = 16; half >= 1; half >>= 1, off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int j = 0; j < half; ++j) {
                    const float keep = upper ? v[j + half] : v[j];
                    const float send = upper ? v[j] : v[j + half];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
            if ((lane & 1) == 0) sm.rsum[g][wq][lane >> 1] = v[0];
            if (lane == 0 && wq == 0) {
#pragma unroll
                for (int q = 0; q < kGroupRows / 2; ++q) {
                    sm.mref[g][2 * q] = -lo2(nm[q]);
                    sm.mref[g][2 * q + 1] = -hi2(nm[q]);
                }
            }
        }
        group_bar(g);
        const int64_t unit = slot;  // this split's workspace slot
        // lane i of the group's first warp writes row i (a compact block: this code runs once per
        // CTA, from a cold instruction cache)
        if (alive && !ctx.aborted() && wq == 0 && lane < kGroupRows && row0 + lane < R) {
            const float L = sm.rsum[g][0][lane] + sm.rsum[g][1][lane] + sm.rsum[g][2][lane] +
                            sm.rsum[g][3][lane];
            p.ws_state[unit * p.rows + row_lo + row0 + lane] = make_float2(sm.mref[g][lane], L);
        }
        // O^T (tensor memory, lane = head-dim element) -> numerator rows:
        // O = O_h + O_m/16 + O_l/256
        const bool ok = ctx.wait_warp(&sm.odone, 0);
        tc_fence_after();
        if (__all_sync(0xffffffffu, ok && !ctx.aborted())) {
            const float vs = sm.vscale;
#pragma unroll 1
            for (int dh = 0; dh < 2; ++dh) {
                float o[kGroupRows];
                load_terms16<RP>(lane_base + C::kColO + dh * SN + row0, o);
                const int d = dh * 128 + st;
#pragma unroll
                for (int i = 0; i < kGroupRows; ++i) {
                    const int r = row0 + i;
                    if (r < R) p.ws_acc[(unit * p.rows + row_lo + r) * kHeadDim + d] = o[i] * vs;
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
    if constexpr (kFused) fused_merge<C::kThreads>(p, smem);
}

}  // namespace tc

int tc_rows_pad(int rows) { return (rows + tc::kGroupRows - 1) / tc::kGroupRows * tc::kGroupRows; }

bool tc_supports(int rows) { return tc_rows_pad(rows) <= tc::kMaxRP; }

int tc_max_rows() { return tc::kMaxRP; }

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

template <int RP, bool kFused>
static cudaError_t launch_rp(const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const PartialParams& p, cudaStream_t stream) {
    constexpr uint32_t smem = tc::smem_bytes<RP>();
    cudaError_t e = cudaFuncSetAttribute(tc::tc_partial_kernel<RP, kFused>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = partial_grid(p);
    cfg.blockDim = dim3(tc::Cfg<RP>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p.out) {  // the fused merge waits for every CTA: they must all be resident at once
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    } else if (p.pdl) {  // a programmatic dependent of the preceding kernel on the stream
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, tc::tc_partial_kernel<RP, kFused>, kmap, vmap, p);
}

cudaError_t launch_tc_partial(const PartialParams& p, cudaStream_t stream) {
    if (!row_blocks_valid(p, tc::kMaxRP)) return cudaErrorInvalidValue;
    const int rp = tc_rows_pad(p.block_rows);
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    // K and V pools (rows of Hkv * 256 bytes, num_pages * page_size of them) viewed as 4-D:
    // (byte within a 128-byte head-dim half, row within an 8-row group, half index 2 h + half,
    // 8-row group). A box (128, 8, 2, 2) is one 16-row chunk of one head, both halves, landing as
    // [group][half][row][128 bytes] in the 128-byte swizzle the MMA operands use: one copy
    // instruction per 4 KB page chunk. Rows of a chunk start at a multiple of 16 (pages are).
    CUtensorMap kmap, vmap;
    const cuuint64_t row = (cuuint64_t)p.num_kv_heads * kHeadDim;
    const cuuint64_t dims[4] = {128, 8, 2 * (cuuint64_t)p.num_kv_heads,
                                (cuuint64_t)p.num_pages * p.page_size / 8};
    const cuuint64_t strides[3] = {row, 128, 8 * row};
    const cuuint32_t box[4] = {128, 8, 2, 2};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r1 = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(p.k_pool),
                         dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult r2 = encode(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(p.v_pool),
                         dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
    switch (rp) {
        case 16: return p.out ? launch_rp<16, true>(kmap, vmap, p, stream)
                              : launch_rp<16, false>(kmap, vmap, p, stream);
        case 32: return p.out ? launch_rp<32, true>(kmap, vmap, p, stream)
                              : launch_rp<32, false>(kmap, vmap, p, stream);
        default: return p.out ? launch_rp<48, true>(kmap, vmap, p, stream)
                              : launch_rp<48, false>(kmap, vmap, p, stream);
    }
}

}  // namespace dflash
