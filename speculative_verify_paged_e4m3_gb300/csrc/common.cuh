// common.cuh -- device-side parameter blocks and helpers shared by the partial and combine kernels.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "dflash_verify_attn.h"

namespace dflash {

constexpr int kHeadDim = 256;  // the only head dim the kernels are built for
constexpr int kMaxRows = 64;   // q_len * Hq / Hkv rows per KV head a CTA carries
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
    // merge of the splits inside the same launch (every CTA resident): grid barrier words in the
    // workspace header, then FP16 output and FP32 log-sum-exp; null out when not fused
    unsigned long long* grid_bar;  // ticket counter of the grid barrier (workspace header)
    __half* out;
    float* lse;
};

struct CombineParams {
    const float2* ws_state;
    const float* ws_acc;
    const int32_t* context_lens;
    __half* out;
    float* lse;
    int batch, q_len, num_q_heads, num_kv_heads, group, rows;
    int max_context, num_splits, tile_keys, min_split_keys;
};

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

}  // namespace dflash
