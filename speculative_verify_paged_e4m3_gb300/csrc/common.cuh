// common.cuh -- device-side parameter blocks and helpers shared by the partial and combine kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "dflash_verify_attn.h"

namespace dflash {

constexpr int kHeadDim = 256;  // the only head dim the kernels are built for
constexpr int kMaxRows = 256;  // q_len * Hq / Hkv rows per KV head (split over row blocks)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct PartialParams {
    const __half* q;
    const uint8_t* k_pool;
    const uint8_t* v_pool;
    const int32_t* block_table;
    const int32_t* context_lens;
    const float* k_scale;
    const float* v_scale;
    int32_t* status;   // workspace status word
    float2* ws_state;  // (m, l) [B, Hkv, S, R]
    float* ws_acc;     // [B, Hkv, S, R, D]
    int batch, q_len, num_q_heads, num_kv_heads, group, rows;
    int page_size, max_pages_per_seq, num_pages, max_context;
    int num_splits, tile_keys, min_split_keys;
    int num_slots;  // workspace split slots: Hkv * num_splits for one sequence, else the plan's
    // Row blocks: the grid's x extent is num_splits * row_blocks; CTA x = split * row_blocks + k
    // carries rows [k * block_rows, min(rows, (k + 1) * block_rows)) of that split's slot.
    int row_blocks, block_rows;
    // keys per split of a max_context-long context (the split size the kernels guess while the
    // context length is in flight), and log2 of page_size when it is a power of two (else -1)
    int per_max, page_shift;
    // merge of the splits inside the same launch (every CTA resident): grid barrier words in the
    // workspace header, then FP16 output and FP32 log-sum-exp; null out when not fused
    unsigned long long* grid_bar;  // ticket counter of the grid barrier (workspace header)
    __half* out;
    float* lse;
    int pdl;  // host side: launch as a programmatic dependent of the preceding kernel
};

struct CombineParams {
    const float2* ws_state;
    const float* ws_acc;
    const int32_t* context_lens;
    __half* out;
    float* lse;
    int batch, q_len, num_q_heads, num_kv_heads, group, rows;
    int max_context, num_splits, tile_keys, min_split_keys;
    int num_slots;
    int pdl;  // host side: launch as a programmatic dependent of the preceding kernel
};

// This CTA's place in a row-blocked grid: the split position x / row_blocks (the workspace slot
// is that position plus one grid row's worth per (y, z) grid row: a single sequence launches
// (num_splits, Hkv, 1) slots, a batch (num_slots, 1, 1)) and its row range.
struct RowBlock {
    int xs;      // split position within the grid row
    int slot;    // workspace slot
    int row_lo;  // first row (of R) this CTA carries
    int rows;    // rows it carries, >= 1
};

// Host check of a launch's row blocks: every block carries 1..capacity rows and together they
// cover the R rows exactly once.
inline bool row_blocks_valid(const PartialParams& p, int capacity) {
    return p.row_blocks >= 1 && p.block_rows >= 1 && p.block_rows <= capacity &&
           (int64_t)p.row_blocks * p.block_rows >= p.rows &&
           (int64_t)(p.row_blocks - 1) * p.block_rows < p.rows;
}

__device__ __forceinline__ RowBlock row_block(const PartialParams& p) {
    RowBlock rb;
    if (p.row_blocks == 1) {  // one CTA per split: no division
        rb.xs = blockIdx.x;
        rb.row_lo = 0;
        rb.rows = p.rows;
        rb.slot = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        return rb;
    }
    rb.xs = blockIdx.x / p.row_blocks;
    rb.row_lo = (blockIdx.x - rb.xs * p.row_blocks) * p.block_rows;
    rb.rows = min(p.block_rows, p.rows - rb.row_lo);
    rb.slot = rb.xs + (gridDim.x / p.row_blocks) * (blockIdx.y + gridDim.y * blockIdx.z);
    return rb;
}

// ---- programmatic dependent launch -------------------------------------------------------------
// Let the next kernel on the stream, if it was launched as this one's programmatic dependent,
// start launching its CTAs (it still waits for this grid's completion where it calls
// griddep_wait). Issued by every thread of a CTA; idempotent.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grid this one depends on programmatically (the preceding kernel on the stream)
// has completed and its memory writes are visible; returns at once when this grid was launched
// without the programmatic attribute. The wait ends because that grid's CTAs are all resident
// or done by the time this grid starts.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Context length of sequence b as the kernels see it: clamped into [0, max_context].
__device__ __forceinline__ int clamped_context(const int32_t* context_lens, int b, int max_context,
                                              int* flags) {
    int n = context_lens[b];
    int f = 0;
    if (n > max_context) {
        n = max_context;
        f |= DFLASH_FLAG_CONTEXT_CLAMPED;
    }
    if (n < 0) {
        n = 0;
    }
    *flags = f;
    return n;
}

// Keys per split for context n (the rule dflash_verify_attn_split_bounds restates on the host).
__device__ __forceinline__ int keys_per_split(int n, int num_splits, int tile_keys,
                                              int min_split_keys) {
    int per = (n + num_splits - 1) / num_splits;
    per = per > min_split_keys ? per : min_split_keys;
    return (per + tile_keys - 1) / tile_keys * tile_keys;
}

// A block-table entry clamped into the pool of num_pages pages.
__device__ __forceinline__ int clamp_page(int phys, int num_pages, bool* clamped) {
    if (phys < 0 || phys >= num_pages) {
        *clamped = true;
        phys = phys < 0 ? 0 : num_pages - 1;
    }
    return phys;
}

// Physical page of logical page lp of sequence b, clamped into the pool.
__device__ __forceinline__ int physical_page(const int32_t* block_table, int b,
                                             int max_pages_per_seq, int lp, int num_pages,
                                             bool* clamped) {
    return clamp_page(block_table[(int64_t)b * max_pages_per_seq + lp], num_pages, clamped);
}

// ---- split slots of a batch -------------------------------------------------------------------
// The plan's C split slots (one CTA each; as many as the GPU runs at once unless the split
// count is forced, then batch * Hkv * S) are shared out among the (sequence, KV head) units so
// that the busiest slot has as few 128-key tiles as possible. With w_b = ceil(n_b / 128) tiles
// in sequence b, T is the smallest tile count with
//   Hkv * sum_b ceil(w_b / T) <= C,
// and each KV head of sequence b owns c_b = ceil(w_b / T) contiguous slots, unit u = b * Hkv + h
// from slot Hkv * (c of the sequences before b) + h * c_b; the slots past all units stay idle.
// A unit's splits then hold at most T tiles each (the least any split of the units into
// contiguous pieces achieves), an empty unit owns no slot. A single sequence keeps num_splits
// slots per KV head (the same splits: its units are equal). dflash_verify_attn_split_slots does
// the same integer arithmetic on the host.
struct UnitSlots {
    int b, h;    // the unit (b = -1: no unit owns the slot)
    int first;   // its first slot
    int count;   // its slot count (its split count)
    int n;       // context length of sequence b, clamped to [0, max_context]
    int flags;   // DFLASH_FLAG_CONTEXT_* of the whole batch
};

__device__ __forceinline__ int slot_granules(int n) { return (n + 127) >> 7; }

// The clamped length of sequence b; sets the batch's context flags.
__device__ __forceinline__ int slot_length(const int32_t* context_lens, int b, int max_context,
                                           int q_len, int* flags) {
    int n = context_lens[b];
    if (n > max_context) {
        n = max_context;
        *flags |= DFLASH_FLAG_CONTEXT_CLAMPED;
    }
    n = n < 0 ? 0 : n;
    if (n < q_len) *flags |= DFLASH_FLAG_CONTEXT_SHORT;
    return n;
}

// Slots of a single sequence: its units are equal, S slots each.
__device__ __forceinline__ UnitSlots locate_slots_single(const int32_t* context_lens, int Hkv,
                                                         int S, int max_context, int q_len,
                                                         int key, bool by_slot) {
    UnitSlots r = {-1, 0, 0, 0, 0, 0};
    int flags = 0;
    const int n = slot_length(context_lens, 0, max_context, q_len, &flags);
    const int u = by_slot ? key / S : key;
    r.flags = flags;
    if (n == 0 || u >= Hkv) return r;
    r.b = 0;
    r.h = u;
    r.first = u * S;
    r.count = S;
    r.n = n;
    return r;
}

// Slots of a batch of several sequences. Warp-cooperative: every lane of the warp calls it with
// the same arguments and gets the same result. by_slot: the unit owning slot key; else the slots
// of unit key.
__device__ __forceinline__ UnitSlots locate_slots_batch_body(const int32_t* context_lens,
                                                             int B, int Hkv, int num_slots,
                                                             int max_context, int q_len,
                                                             int key, bool by_slot) {
    const int lane = threadIdx.x & 31;
    UnitSlots r = {-1, 0, 0, 0, 0, 0};
    int unused = 0;
    auto tiles = [&](int b) {  // w_b (0 past the batch)
        return b < B ? slot_granules(slot_length(context_lens, b, max_context, q_len, &unused)) : 0;
    };
    // tiles in all (W), the longest sequence, non-empty sequences, the batch's context flags
    long long W = 0;
    int wmax = 0, E = 0, flags = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        const int w =
            b < B ? slot_granules(slot_length(context_lens, b, max_context, q_len, &flags)) : 0;
        W += w;
        wmax = max(wmax, w);
        E += w > 0;
    }
    for (int o = 16; o > 0; o >>= 1) {
        W += __shfl_xor_sync(0xffffffffu, W, o);
        wmax = max(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
        E += __shfl_xor_sync(0xffffffffu, E, o);
        flags |= __shfl_xor_sync(0xffffffffu, flags, o);
    }
    r.flags = flags;
    if (W == 0) return r;
    // T: binary search between W Hkv / C (no split can do better) and the first count that is
    // surely enough, W Hkv / (C - U) (U = Hkv E: each unit's last split may be short), or wmax
    const long long C = num_slots, U = (long long)Hkv * E;
    long long lo = (W * Hkv + C - 1) / C;
    long long hi = wmax;
    if (C > U) hi = min(hi, (W * Hkv + (C - U) - 1) / (C - U));
    lo = max(1ll, min(lo, hi));
    while (lo < hi) {
        const long long mid = (lo + hi) >> 1;
        long long need = 0;
        for (int b0 = 0; b0 < B; b0 += 32) need += (tiles(b0 + lane) + mid - 1) / mid;
        for (int o = 16; o > 0; o >>= 1) need += __shfl_xor_sync(0xffffffffu, need, o);
        if (need * Hkv <= C)
            hi = mid;
        else
            lo = mid + 1;
    }
    const int T = (int)lo;
    // slots per KV head of each sequence, scanned over the batch
    int c_carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        const int b = b0 + lane;
        const int n = b < B ? slot_length(context_lens, b, max_context, q_len, &unused) : 0;
        const int c = (slot_granules(n) + T - 1) / T;
        int sc = c;  // inclusive scan over the chunk
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, sc, o);
            if (lane >= o) sc += t;
        }
        const int c_before = c_carry + sc - c;  // per KV head, sequences before b
        const bool mine = by_slot ? (b < B && c > 0 && key >= Hkv * c_before &&
                                     key < Hkv * (c_before + c))
                                  : b == key / Hkv;
        const unsigned m = __ballot_sync(0xffffffffu, mine);
        if (m) {
            const int src = __ffs(m) - 1;
            const int cb0 = __shfl_sync(0xffffffffu, c_before, src);
            const int cb = __shfl_sync(0xffffffffu, c, src);
            const int nb = __shfl_sync(0xffffffffu, n, src);
            const int hh = by_slot ? (key - Hkv * cb0) / cb : key % Hkv;
            r.b = b0 + src;
            r.h = hh;
            r.first = Hkv * cb0 + hh * cb;
            r.count = cb;
            r.n = nb;
            return r;
        }
        c_carry += __shfl_sync(0xffffffffu, sc, 31);
    }
    return r;
}

static __device__ __noinline__ UnitSlots locate_slots_batch(const int32_t* context_lens, int B,
                                                            int Hkv, int num_slots,
                                                            int max_context, int q_len, int key,
                                                            bool by_slot) {
    return locate_slots_batch_body(context_lens, B, Hkv, num_slots, max_context, q_len, key,
                                   by_slot);
}

// The slots of a unit or the unit of a slot (see above). Warp-cooperative. The several-sequence
// search is called out of line: it runs once per CTA, and the kernels' hot code stays compact.
__device__ __forceinline__ UnitSlots locate_slots(const int32_t* context_lens, int B, int Hkv,
                                                  int S, int num_slots, int max_context,
                                                  int q_len, int key, bool by_slot) {
    if (B == 1) return locate_slots_single(context_lens, Hkv, S, max_context, q_len, key, by_slot);
    return locate_slots_batch(context_lens, B, Hkv, num_slots, max_context, q_len, key, by_slot);
}

// Grid of a partial launch: (splits x row blocks, Hkv, 1) for a single sequence, (slots x row
// blocks, 1, 1) for a batch.
inline dim3 partial_grid(const PartialParams& p) {
    return p.batch == 1 ? dim3(p.num_splits * p.row_blocks, p.num_kv_heads, 1)
                        : dim3(p.num_slots * p.row_blocks, 1, 1);
}

}  // namespace dflash
