/*
 * dflash_verify_attn.h -- C ABI of the GB300 (sm_103a) DFlash2 speculative-verification attention.
 *
 * What the operation is. A block of q_len drafted query tokens (FP16 Q) attends causally over a
 * paged KV cache stored as E4M3 codes with one FP32 scale per layer for K and one for V. The
 * context is cut into logical splits; each split keeps an FP32 running max, sum and numerator per
 * query row, and a combine pass merges them into an FP16 output and an FP32 log-sum-exp.
 * Sources, by page and section:
 *   - "[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Test Plan: shape
 *     q8 / Hq6 / Hkv1 / D256 per tensor-parallel rank, FP16 activations, E4M3 KV, FP32 state,
 *     sixteen distinct layer KV allocations timed under CUDA-graph replay; Test Result: each layer
 *     runs one grouped q8 attention kernel followed by one combine kernel.
 *   - "[Perf] Reduce DFlash2 long-context verification decay", Implementation: six-head KV reuse,
 *     vector loads, page specialisation, logical context splits with FP32 state; Purpose:
 *     capacity 262144 tokens.
 *   - "[Perf] Add opt-in DFlash2 schedules and numerical audits", Test Plan: E4M3 target KV,
 *     FP32 logits/state.
 *
 * The math (the pages leave it implicit; this is the plain reading):
 *   k^ = e4m3(code) * k_scale, v^ = e4m3(code) * v_scale  (OCP E4M3FN: bias 7, max 448)
 *   query token i (0 <= i < q_len) of sequence b sits at position N - q_len + i, N = context_lens[b]
 *   s_j = (q . k^_j) / sqrt(head_dim), visible iff 0 <= j <= N - q_len + i
 *   lse = ln sum_visible e^{s_j}  (natural log),  out = sum_visible e^{s_j - lse} v^_j
 *   A row with no visible key gets out = 0 and lse = -inf.
 * Query head hq uses KV head hq / (num_q_heads / num_kv_heads).
 *
 * Layouts (row-major, no padding, device memory unless stated):
 *   q            FP16  [batch, q_len, num_q_heads, head_dim]
 *   k_pool       uint8 [num_pages, page_size, num_kv_heads, head_dim]  E4M3FN codes
 *   v_pool       uint8 same layout as k_pool
 *   block_table  int32 [batch, max_pages_per_seq]; logical page p of sequence b lives in
 *                physical page block_table[b][p]; only the first ceil(N / page_size) entries of a
 *                row are read
 *   context_lens int32 [batch]; N, counting the q_len drafted tokens
 *   k_scale, v_scale  one FP32 each (device scalars, so one captured graph serves every layer's
 *                scale and a growing context)
 *   out          FP16  [batch, q_len, num_q_heads, head_dim]
 *   lse          FP32  [batch, q_len, num_q_heads]
 *   workspace    caller-allocated, plan.workspace_bytes, 256-byte aligned; private layout
 *                described by the plan (offsets below) so tests can read the split state.
 *
 * Conventions.
 *   - Every call returns a dflash_status. Nothing allocates, throws, or synchronises, except
 *     dflash_verify_attn_read_flags, which is documented as synchronous.
 *   - run and combine are stream-ordered and capturable in a CUDA graph; they read
 *     context_lens, k_scale and v_scale on the device.
 *   - Host-checkable preconditions are checked in plan (shape support) and in run / combine
 *     (null pointers, alignment, workspace size) and return DFLASH_ERR_INVALID_ARGUMENT or
 *     DFLASH_ERR_WORKSPACE_TOO_SMALL without launching anything.
 *   - Device-only conditions never fault. A context above plan.problem.max_context is clamped to
 *     it, a block-table entry outside [0, num_pages) is clamped into range, and each sets a bit in
 *     the sticky status word at the head of the workspace (DFLASH_FLAG_*). The caller zeroes the
 *     first 16 bytes of the workspace once when allocating it: the status word (offset 0,
 *     dflash_verify_attn_read_flags can clear it) and the 64-bit grid-barrier counter of the
 *     fused merge (offset 8; it needs no reset between calls, but zero it again after a
 *     DFLASH_FLAG_KERNEL_TIMEOUT).
 *   - Launch failures map to DFLASH_ERR_CUDA (cudaGetLastError, which does not synchronise).
 */
#ifndef DFLASH_VERIFY_ATTN_H
#define DFLASH_VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_VERIFY_ATTN_VERSION 3

typedef enum {
    DFLASH_OK = 0,
    DFLASH_ERR_INVALID_ARGUMENT = -1,
    DFLASH_ERR_UNSUPPORTED = -2,
    DFLASH_ERR_WORKSPACE_TOO_SMALL = -3,
    DFLASH_ERR_CUDA = -4
} dflash_status;

/* Bits of the device status word (workspace offset 0, int32, sticky). */
#define DFLASH_FLAG_CONTEXT_CLAMPED 0x1  /* some context_lens[b] > max_context: clamped     */
#define DFLASH_FLAG_CONTEXT_SHORT 0x2    /* some context_lens[b] < q_len: early rows see no key */
#define DFLASH_FLAG_PAGE_CLAMPED 0x4     /* a block-table entry outside [0, num_pages): clamped */
#define DFLASH_FLAG_KERNEL_TIMEOUT 0x8   /* a tensor-core kernel wait gave up; outputs invalid */

/* Bits of dflash_verify_attn_problem.flags. */
#define DFLASH_PROBLEM_FUSED_COMBINE 0x1 /* forward merges the splits inside the partial launch */
/* Launch the partial and combine kernels as programmatic dependents of the preceding kernel on
 * the stream (CUDA programmatic dependent launch), so that each starts while its predecessor
 * drains. A partial kernel then reads context_lens, the block table and the K/V pages of the
 * positions before N - q_len while the preceding kernel may still be running; Q, k_scale,
 * v_scale and the pages of the q_len drafted positions are read, and the split state in the
 * workspace is written, only once it has completed (status flags are OR-ed into the status word
 * at any time). The combine reads the workspace only once the partial kernel has completed.
 * So set this bit only when the kernel launched just before run / forward writes none of
 * context_lens, the block table or the pages of earlier positions (the drafted tokens' KV write,
 * dflash_verify_attn_kv_write, writes only the drafted positions). Ignored with
 * DFLASH_PROBLEM_FUSED_COMBINE. Results are the same bits with and without it. */
#define DFLASH_PROBLEM_PDL 0x2

/* Partial-attention kernel variants a plan can select. */
#define DFLASH_KERNEL_AUTO 0
#define DFLASH_KERNEL_SIMT 1     /* CUDA-core FP32 kernel: any supported shape */
#define DFLASH_KERNEL_TCGEN05 2  /* tensor-core (tcgen05, TMEM) kernel */

/* Shape of one layer's problem. Host struct, filled by the caller. */
typedef struct {
    int32_t version;           /* DFLASH_VERIFY_ATTN_VERSION */
    int32_t batch;             /* sequences, >= 1 */
    int32_t q_len;             /* drafted tokens per sequence, >= 1 (8 in the pages' runs) */
    int32_t num_q_heads;       /* Hq */
    int32_t num_kv_heads;      /* Hkv; Hq % Hkv == 0 and R = q_len * Hq / Hkv <= 256 */
    int32_t head_dim;          /* 256 */
    int32_t page_size;         /* tokens per page; a multiple of 16 */
    int32_t max_pages_per_seq; /* block-table row stride; >= ceil(max_context / page_size) */
    int32_t num_pages;         /* pages in each pool (bounds for block-table entries) */
    int32_t max_context;       /* largest N any call of this plan sees, >= 1 */
    int32_t device;            /* CUDA ordinal whose SM count sizes the plan */
    int32_t num_splits;        /* 0: planner's choice; > 0 forces the split count */
    int32_t kernel;            /* DFLASH_KERNEL_*; AUTO picks the fastest supported */
    int32_t flags;             /* DFLASH_PROBLEM_* bits; 0 for the defaults */
} dflash_verify_attn_problem;

/* Written by dflash_verify_attn_plan, read-only afterwards. Host POD; copy freely. */
typedef struct {
    int32_t version;
    int32_t kernel;           /* DFLASH_KERNEL_SIMT or DFLASH_KERNEL_TCGEN05 */
    int32_t num_splits;       /* S: splits per (sequence, KV head) */
    int32_t tile_keys;        /* keys per pipeline tile; split boundaries are multiples of it */
    int32_t min_split_keys;   /* lower bound on keys per split (a multiple of tile_keys) */
    int32_t rows;             /* R = q_len * Hq / Hkv query rows per KV head */
    int32_t threads;          /* partial-kernel block size */
    int32_t smem_bytes;       /* partial-kernel dynamic shared memory */
    int32_t sm_count;         /* SMs of plan.problem.device */
    int32_t combine_fused;    /* 1: forward merges the splits inside the partial-kernel launch */
    int32_t row_blocks;       /* CTAs per split, each carrying ceil(R / row_blocks) consecutive
                                 rows (1 unless R exceeds what one CTA of the kernel holds: 48
                                 rows for TCGEN05, 64 for SIMT) */
    int32_t num_slots;        /* split slots of the workspace, one partial-kernel CTA (per row
                                 block) each: batch * Hkv * num_splits for a single sequence or a
                                 forced split count; for a batch on the planner's split count, the
                                 SMs' worth (sm_count / row_blocks, at least batch * Hkv), shared
                                 out by length at run time (dflash_verify_attn_split_slots) */
    size_t workspace_bytes;   /* caller allocates at least this many bytes */
    size_t ws_state_offset;   /* float2 (m, l) [slots, R]; m in log2 units (slots below) */
    size_t ws_acc_offset;     /* float numerator [slots, R, head_dim], v_scale applied */
    dflash_verify_attn_problem problem;
} dflash_verify_attn_plan_t;

/*
 * Check the problem and choose the split count, tile and kernel for it. The context is cut into
 * logical splits ("[Perf] Reduce DFlash2 long-context verification decay", Implementation: 80
 * logical splits, sized there to the V100's 80 SMs); here the split count follows this GPU's SM
 * count and the keys per split follow the live context length. Host only; queries the
 * device's SM count (cudaDeviceGetAttribute) unless problem->device < 0, in which case a
 * 152-SM part is assumed (lets plans be built and checked without a GPU).
 * Returns DFLASH_ERR_INVALID_ARGUMENT for a malformed problem, DFLASH_ERR_UNSUPPORTED for a
 * well-formed shape this build has no kernel for.
 */
int dflash_verify_attn_plan(const dflash_verify_attn_problem* problem,
                            dflash_verify_attn_plan_t* plan);

/*
 * Split slots (host restatement of the device rule). The workspace holds slots = num_slots split
 * states, one per partial-kernel CTA (and row block). They are shared out among the
 * (sequence, KV head) units u = b * Hkv + h so that the busiest slot holds as few 128-key tiles
 * as possible. With w_b = ceil(n_b / 128) tiles in sequence b (n_b = context_lens[b] clamped to
 * [0, max_context]), T is the smallest tile count with
 *   Hkv * sum_b ceil(w_b / T) <= slots,
 * and each KV head of sequence b owns c_b = ceil(w_b / T) contiguous slots:
 *   slot_start[b * Hkv + h] = Hkv * (c of the sequences before b) + h * c_b.
 * Slots past slot_start[batch * Hkv] stay idle. A single sequence (batch 1) keeps num_splits
 * slots per KV head. Every non-empty unit owns at least one slot, an empty unit none. Unit u
 * splits its n_b keys into pieces of
 * keys_per_split[u] = roundup(max(ceil(n_b / S_u), min_split_keys), tile_keys) keys, S_u =
 * slot_start[u + 1] - slot_start[u]; its first active[u] = ceil(n_b / keys_per_split[u]) slots
 * hold state (0 for an empty unit). context_lens: batch entries (host memory); slot_start:
 * batch * Hkv + 1 entries; keys_per_split and active: batch * Hkv entries.
 */
int dflash_verify_attn_split_slots(const dflash_verify_attn_plan_t* plan,
                                   const int32_t* context_lens, int32_t* slot_start,
                                   int32_t* keys_per_split, int32_t* active);

/*
 * Split boundaries the kernels use for a single sequence of context length n, whose KV heads
 * own num_splits slots each (for a batch, dflash_verify_attn_split_slots): keys_per_split =
 * roundup(max(ceil(n / S), min_split_keys), tile_keys), split s covers
 * [s * keys_per_split, min(n, (s + 1) * keys_per_split)), and the first
 * *active = ceil(n / keys_per_split) splits are non-empty (0 when n == 0). n is clamped to
 * [0, max_context] first. starts[] receives S + 1 entries (host memory); empty splits start and
 * end at n.
 */
int dflash_verify_attn_split_bounds(const dflash_verify_attn_plan_t* plan, int32_t n,
                                    int32_t* starts, int32_t* active);

/*
 * Partial attention: for every (sequence, KV head, active split) write the split's FP32 state
 * (m, l, numerator) into the workspace ("[Perf] Reduce DFlash2 attention cost and screen exact QK
 * reuse", Purpose: the complete FP32 numerator / max / sum workspace; "[Perf] Reduce DFlash2
 * long-context verification decay", Implementation: one CTA carries every query head of its KV
 * head, so each K/V page is read once). Inputs as in the layout table above. workspace_bytes must
 * be >= plan->workspace_bytes and the workspace 256-byte aligned; q, k_pool and v_pool must be
 * 16-byte aligned. cuda_stream is a cudaStream_t (NULL: legacy default stream).
 */
int dflash_verify_attn_run(const dflash_verify_attn_plan_t* plan, const void* q,
                           const void* k_pool, const void* v_pool, const int32_t* block_table,
                           const int32_t* context_lens, const float* k_scale,
                           const float* v_scale, void* workspace, size_t workspace_bytes,
                           void* cuda_stream);

/*
 * Combine: merge the active splits' state of every query row into out (FP16, round to nearest
 * even) and lse (FP32, natural log): M = max_s m_s, L = sum_s e^{m_s - M} l_s,
 * out = sum_s e^{m_s - M} acc_s / L, lse = M + ln L ("[Perf] Reduce DFlash2 attention cost and
 * screen exact QK reuse", Test Result: each grouped q8 attention kernel is followed by one
 * combine kernel). Must follow dflash_verify_attn_run on the same stream with the same plan,
 * workspace and context_lens.
 */
int dflash_verify_attn_combine(const dflash_verify_attn_plan_t* plan, const void* workspace,
                               size_t workspace_bytes, const int32_t* context_lens, void* out,
                               float* lse, void* cuda_stream);

/*
 * run followed by combine on one stream: the per-layer pair of "[Perf] Reduce DFlash2 attention
 * cost and screen exact QK reuse", Test Result. With DFLASH_PROBLEM_FUSED_COMBINE in problem.flags
 * (tensor-core kernel, batch * num_kv_heads * row_blocks <= the SM count; plan->combine_fused
 * tells), both happen in a single cooperative launch of the
 * partial kernel instead: after every CTA has written its split state (a bounded grid-wide
 * barrier on the workspace header), the CTAs share out the combine's work and write out and lse
 * themselves. Results match run + combine within the output tolerance, and are the same bits
 * when each (sequence, KV head) has at most 16 or more than 64 splits (the separate combine then
 * groups the splits as the fused merge does).
 */
int dflash_verify_attn_forward(const dflash_verify_attn_plan_t* plan, const void* q,
                               const void* k_pool, const void* v_pool,
                               const int32_t* block_table, const int32_t* context_lens,
                               const float* k_scale, const float* v_scale, void* workspace,
                               size_t workspace_bytes, void* out, float* lse, void* cuda_stream);

/*
 * The step before verification: write the q_len drafted tokens' K and V rows (FP16) into the
 * paged pools as E4M3FN codes (the E4M3 target KV of "[Perf] Add opt-in DFlash2 schedules and
 * numerical audits", Test Plan; the pages do not describe the write itself).
 *   k_new, v_new  fp16 [batch, q_len, Hkv, head_dim], 4-byte aligned (device)
 *   k_pool, v_pool  E4M3 [num_pages, page_size, Hkv, head_dim] (device), written in place
 *   block_table, context_lens, k_scale, v_scale  as for run (device)
 * Token i of sequence b goes to position n - q_len + i, n = context_lens[b] clamped to
 * [0, max_context] (the position the attention's causal rule gives it): slot position %
 * page_size of page block_table[b][position / page_size]. Each element is stored as the E4M3FN
 * code of x / scale (one correctly rounded FP32 division, then round to nearest even, magnitudes
 * beyond 448 saturated to 448, NaN to a NaN code). A token whose position is negative
 * (DFLASH_FLAG_CONTEXT_SHORT) or whose page entry lies outside [0, num_pages)
 * (DFLASH_FLAG_PAGE_CLAMPED) is not written; a clamped context sets DFLASH_FLAG_CONTEXT_CLAMPED.
 * The flags go to the status word of workspace (>= plan->workspace_bytes, 256-byte aligned, the
 * one run uses). No allocation, no synchronisation; capture-safe.
 */
int dflash_verify_attn_kv_write(const dflash_verify_attn_plan_t* plan, const void* k_new,
                                const void* v_new, const int32_t* block_table,
                                const int32_t* context_lens, const float* k_scale,
                                const float* v_scale, void* k_pool, void* v_pool,
                                void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Debug export of an E4M3 decode: the two-code hardware conversion (cvt.rn.f16x2.e4m3x2) that the
 * CUDA-core kernel uses for K and V and the tensor-core kernel uses for the residuals of its Q
 * split. (The tensor-core kernel hands K and V codes to the tensor core undecoded; its decode is
 * checked through the attention outputs of one-key problems instead.) decoded[t] = exact value
 * of codes[t] (NaN for S.1111.111), scaled[t] = decoded[t] * *scale rounded once to FP32
 * ("[Perf] Add opt-in DFlash2 schedules and numerical audits", Test Plan: E4M3 target KV).
 * n >= 0 elements; all pointers device memory; scaled may be NULL.
 */
int dflash_verify_attn_debug_dequant(const uint8_t* codes, int64_t n, const float* scale,
                                     float* decoded, float* scaled, void* cuda_stream);

/*
 * Copy the workspace status word (DFLASH_FLAG_* bits) to *flags_host, optionally zeroing it.
 * Synchronises cuda_stream; not for use inside graph capture.
 */
int dflash_verify_attn_read_flags(const void* workspace, int32_t* flags_host, int clear,
                                  void* cuda_stream);

/*
 * run followed by combine with the split workspace taken from a 16 MiB device array built into
 * the library instead of caller memory. The pages have no counterpart: this entry point exists
 * for callers that may not allocate device memory (a plugin whose device memory belongs to a host
 * framework's allocator, a runtime that freezes its memory pool after start-up, a loop that must
 * never enter the allocator). They still pass every input and output; nothing here allocates.
 * Limits and behaviour: plan->workspace_bytes must be <= 16 MiB, else
 * DFLASH_ERR_WORKSPACE_TOO_SMALL and nothing is launched. The first call on a device (with that
 * device current) looks up the array's device address once; make it before any stream capture.
 * All calls share the array. The first 16 bytes of its header (the status word and the fused
 * merge's grid-barrier counter) are zeroed on the stream at the start of each call, so no call
 * inherits a barrier count from an earlier one. The status word is not reported on this path:
 * a clamped context or page entry goes unseen, and after a kernel wait that gave up
 * (DFLASH_FLAG_KERNEL_TIMEOUT on the ordinary entry points) out and lse are undefined. Calls
 * whose kernels overlap on the GPU race on the array. The array stays allocated on every device
 * that loaded the library until the process exits.
 */
int dflash_verify_attn_forward_static_scratch(const dflash_verify_attn_plan_t* plan,
                                              const void* q, const void* k_pool,
                                              const void* v_pool, const int32_t* block_table,
                                              const int32_t* context_lens, const float* k_scale,
                                              const float* v_scale, void* out, float* lse,
                                              void* cuda_stream);

/* Static text for a dflash_status value. */
const char* dflash_verify_attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_VERIFY_ATTN_H */
