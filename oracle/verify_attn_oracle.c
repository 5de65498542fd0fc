/*
 * verify_attn_oracle.c -- plain, slow, FP64 CPU oracle for DFlash2 speculative-verification
 * attention over a paged E4M3 KV cache.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this code. It shares nothing with the CUDA path (no headers, no tables, no helpers).
 *
 * What it computes (sources):
 *   - "[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Test Plan: a q8 block of
 *     query tokens, 6 query heads sharing 1 KV head, head dim 256, FP16 activations, E4M3 KV
 *     cache, FP32 state; output bytes plus the split numerator/max/sum state are what is checked.
 *   - "[Perf] Reduce DFlash2 long-context verification decay", Implementation: the context is cut
 *     into logical splits that each keep FP32 state (running max, sum, numerator) and are merged
 *     afterwards by a combine pass.
 *   - "[Perf] Add opt-in DFlash2 schedules and numerical audits", Test Plan: E4M3 target KV, FP32
 *     logits/state.
 * The pages do not write the formula down. The oracle is the plain definition of causal softmax
 * attention, evaluated in FP64 with no blocking or reordering:
 *   k^[j,d] = e4m3(k_code) * k_scale,   v^[j,d] = e4m3(v_code) * v_scale
 *   s_j     = D^-1/2 * sum_d q[d] * k^[j,d]                 (query row: token i, query head hq)
 *   visible = { j : 0 <= j <= N - q_len + i }              (token i sits at position N-q_len+i)
 *   lse     = ln sum_{j visible} e^{s_j}   (computed as max + ln sum e^{s - max})
 *   out[d]  = sum_{j visible} e^{s_j - lse} v^[j,d]
 * A row with no visible key has out = 0 and lse = -inf.
 *
 * E4M3 is the OCP 8-bit floating-point format "E4M3FN": 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits, exponent field 0 encodes subnormals m/8 * 2^-6, no infinities, and S.1111.111
 * is NaN (largest finite magnitude 448).
 *
 * Data layouts (all row-major):
 *   q            [B, q_len, Hq, D]      doubles holding the exact FP16 values
 *   k_pool/v_pool[num_pages, P, Hkv, D] E4M3 codes
 *   block_table  [B, max_pages_per_seq] physical page of logical page j / P
 *   context_lens [B]                    N, which counts the q_len drafted tokens
 *   out          [B, q_len, Hq, D],  lse [B, q_len, Hq]
 *   query head hq reads KV head hq / (Hq / Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_SHAPE -1
#define ORACLE_BAD_PAGE -2
#define ORACLE_NO_MEMORY -3

/* Exact value of one E4M3FN code, from the format's definition. */
double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);             /* (m / 8) * 2^(1 - 7) */
    else
        mag = ldexp((double)(8 + mant), expo - 10); /* (1 + m / 8) * 2^(e - 7) */
    return sign ? -mag : mag;
}

void oracle_e4m3_decode(const uint8_t* codes, int64_t n, double* out)
{
    for (int64_t t = 0; t < n; ++t)
        out[t] = oracle_e4m3_value(codes[t]);
}

typedef struct {
    int B, q_len, Hq, Hkv, D, P, max_pages_per_seq, num_pages;
    const double* q;
    const uint8_t* k_pool;
    const uint8_t* v_pool;
    const int32_t* block_table;
    const int32_t* context_lens;
    double k_scale, v_scale;
} oracle_problem;

static int check_problem(const oracle_problem* p)
{
    if (p->B < 1 || p->q_len < 1 || p->Hq < 1 || p->Hkv < 1 || p->D < 1 || p->P < 1)
        return ORACLE_BAD_SHAPE;
    if (p->Hq % p->Hkv != 0)
        return ORACLE_BAD_SHAPE;
    for (int b = 0; b < p->B; ++b) {
        int n = p->context_lens[b];
        if (n < 0 || (int64_t)n > (int64_t)p->max_pages_per_seq * p->P)
            return ORACLE_BAD_SHAPE;
        for (int lp = 0; lp * p->P < n; ++lp) {
            int32_t phys = p->block_table[(int64_t)b * p->max_pages_per_seq + lp];
            if (phys < 0 || phys >= p->num_pages)
                return ORACLE_BAD_PAGE;
        }
    }
    return ORACLE_OK;
}

/* Byte offset of (logical token j, KV head h, dim 0) of sequence b in a page pool. */
static int64_t kv_offset(const oracle_problem* p, int b, int j, int h)
{
    int32_t phys = p->block_table[(int64_t)b * p->max_pages_per_seq + j / p->P];
    int slot = j % p->P;
    return (((int64_t)phys * p->P + slot) * p->Hkv + h) * p->D;
}

/* s_j for one query row (b, i, hq) against logical key j. */
static double score(const oracle_problem* p, const double* e4m3, int b, int i, int hq, int j)
{
    int h = hq / (p->Hq / p->Hkv);
    const double* qrow = p->q + (((int64_t)b * p->q_len + i) * p->Hq + hq) * p->D;
    const uint8_t* krow = p->k_pool + kv_offset(p, b, j, h);
    double dot = 0.0;
    for (int d = 0; d < p->D; ++d)
        dot += qrow[d] * (e4m3[krow[d]] * p->k_scale);
    return dot / sqrt((double)p->D);
}

static double vhat(const oracle_problem* p, const double* e4m3, int b, int j, int h, int d)
{
    return e4m3[p->v_pool[kv_offset(p, b, j, h) + d]] * p->v_scale;
}

/* Last logical key index that query token i may see: its own position N - q_len + i. */
static int last_visible(const oracle_problem* p, int b, int i)
{
    return p->context_lens[b] - p->q_len + i;
}

/* The unsplit definition: out and lse for every query row. */
int oracle_verify_attn(int B, int q_len, int Hq, int Hkv, int D, int P, int max_pages_per_seq,
                       int num_pages, const double* q, const uint8_t* k_pool,
                       const uint8_t* v_pool, const int32_t* block_table,
                       const int32_t* context_lens, double k_scale, double v_scale, double* out,
                       double* lse)
{
    oracle_problem p = {B, q_len, Hq, Hkv, D, P, max_pages_per_seq, num_pages, q, k_pool,
                        v_pool, block_table, context_lens, k_scale, v_scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK)
        return rc;
    double e4m3[256];
    for (int c = 0; c < 256; ++c)
        e4m3[c] = oracle_e4m3_value((uint8_t)c);
    int rows = B * q_len * Hq;
    int failed = 0;

#pragma omp parallel for schedule(dynamic, 1)
    for (int row = 0; row < rows; ++row) {
        int hq = row % Hq;
        int i = (row / Hq) % q_len;
        int b = row / (Hq * q_len);
        int h = hq / (Hq / Hkv);
        double* o = out + (int64_t)row * D;
        int last = last_visible(&p, b, i);
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (last < 0) {
            lse[row] = -INFINITY;
            continue;
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)(last + 1));
        if (!s) {
#pragma omp atomic write
            failed = 1;
            continue;
        }
        double mx = -INFINITY;
        for (int j = 0; j <= last; ++j) {
            s[j] = score(&p, e4m3, b, i, hq, j);
            if (s[j] > mx)
                mx = s[j];
        }
        double sum = 0.0;
        for (int j = 0; j <= last; ++j)
            sum += exp(s[j] - mx);
        double l = mx + log(sum);
        lse[row] = l;
        for (int j = 0; j <= last; ++j) {
            double w = exp(s[j] - l);
            for (int d = 0; d < D; ++d)
                o[d] += w * vhat(&p, e4m3, b, j, h, d);
        }
        free(s);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Split state, as the pages keep it per logical split: for split s = [start_s, end_s) of the
 * context and each query row, m = max visible score in the split, l = sum e^{s_j - m} and
 * acc[d] = sum e^{s_j - m} v^[j,d] over the split's visible keys (numerator not normalised).
 * A split with no visible key for a row has m = -inf, l = 0, acc = 0.
 * split_bounds is [B, S + 1] (start of every split, then the end of the last one).
 * m, l are [B, Hkv, S, R] and acc is [B, Hkv, S, R, D] with R = q_len * (Hq / Hkv) rows per KV
 * head, row r = i * G + g for token i and group member g (query head h * G + g).
 */
int oracle_verify_attn_partials(int B, int q_len, int Hq, int Hkv, int D, int P,
                                int max_pages_per_seq, int num_pages, const double* q,
                                const uint8_t* k_pool, const uint8_t* v_pool,
                                const int32_t* block_table, const int32_t* context_lens,
                                double k_scale, double v_scale, int S,
                                const int32_t* split_bounds, double* m, double* l, double* acc)
{
    oracle_problem p = {B, q_len, Hq, Hkv, D, P, max_pages_per_seq, num_pages, q, k_pool,
                        v_pool, block_table, context_lens, k_scale, v_scale};
    int rc = check_problem(&p);
    if (rc != ORACLE_OK)
        return rc;
    if (S < 1)
        return ORACLE_BAD_SHAPE;
    double e4m3[256];
    for (int c = 0; c < 256; ++c)
        e4m3[c] = oracle_e4m3_value((uint8_t)c);
    int G = Hq / Hkv;
    int R = q_len * G;
    int64_t units = (int64_t)B * Hkv * S * R;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int r = (int)(u % R);
        int s = (int)((u / R) % S);
        int h = (int)((u / ((int64_t)R * S)) % Hkv);
        int b = (int)(u / ((int64_t)R * S * Hkv));
        int i = r / G, g = r % G;
        int hq = h * G + g;
        int start = split_bounds[(int64_t)b * (S + 1) + s];
        int end = split_bounds[(int64_t)b * (S + 1) + s + 1];
        int last = last_visible(&p, b, i);
        if (end > last + 1)
            end = last + 1;
        double* a = acc + u * D;
        for (int d = 0; d < D; ++d)
            a[d] = 0.0;
        double mx = -INFINITY;
        for (int j = start; j < end; ++j) {
            double sj = score(&p, e4m3, b, i, hq, j);
            if (sj > mx)
                mx = sj;
        }
        double sum = 0.0;
        for (int j = start; j < end; ++j) {
            double w = exp(score(&p, e4m3, b, i, hq, j) - mx);
            sum += w;
            for (int d = 0; d < D; ++d)
                a[d] += w * vhat(&p, e4m3, b, j, h, d);
        }
        m[u] = mx;
        l[u] = sum;
    }
    return ORACLE_OK;
}

/*
 * The combine pass ("[Perf] Reduce DFlash2 attention cost and screen exact QK reuse", Test
 * Result: every full-q8 kernel is followed by a combine kernel), written as its definition:
 *   M = max_s m_s,  L = sum_s e^{m_s - M} l_s,  out = sum_s e^{m_s - M} acc_s / L,  lse = M + ln L.
 * m, l are [rows, S]; acc is [rows, S, D]; out is [rows, D]; lse is [rows].
 */
void oracle_merge_partials(int64_t rows, int S, int D, const double* m, const double* l,
                           const double* acc, double* out, double* lse)
{
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (m[r * S + s] > M)
                M = m[r * S + s];
        double* o = out + r * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double L = 0.0;
        for (int s = 0; s < S; ++s) {
            if (m[r * S + s] == -INFINITY)
                continue;
            double w = exp(m[r * S + s] - M);
            L += w * l[r * S + s];
            for (int d = 0; d < D; ++d)
                o[d] += w * acc[(r * S + s) * D + d];
        }
        for (int d = 0; d < D; ++d)
            o[d] /= L;
        lse[r] = M + log(L);
    }
}

/* Number of host threads the oracle's parallel loops use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * E4M3FN code of a real value v, from the format's definition: the finite code whose value is
 * nearest to v, ties going to the code with the even mantissa (round to nearest even), magnitudes
 * of 448 and above saturated to 448 (the saturating conversion: S.1111.111 is NaN, not a larger
 * number), NaN to the NaN code 0x7F. The sign bit follows v, so -0 gives 0x80. A search over the
 * 127 non-negative finite codes: slow and plainly the definition.
 */
uint8_t oracle_e4m3_encode(double v)
{
    if (isnan(v))
        return 0x7F;
    const int neg = signbit(v) ? 1 : 0;
    const double a = fabs(v);
    int best = 0x7E;
    if (a < 448.0) {
        double best_err = INFINITY;
        for (int c = 0; c <= 0x7E; ++c) {
            const double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
            /* a tie is between neighbours c - 1 and c: keep the even one */
            if (err < best_err || (err == best_err && (c & 1) == 0)) {
                best = c;
                best_err = err;
            }
        }
    }
    return (uint8_t)(best | (neg << 7));
}

void oracle_e4m3_encode_array(const double* v, int64_t n, uint8_t* codes)
{
    for (int64_t t = 0; t < n; ++t)
        codes[t] = oracle_e4m3_encode(v[t]);
}

/*
 * The step before verification: the q_len drafted tokens' K and V rows written into the paged
 * pools as E4M3 codes. The pages imply it ("[Perf] Add opt-in DFlash2 schedules and numerical
 * audits", Test Plan: E4M3 target KV) without describing it; this is the plain reading, the
 * inverse of the decode above:
 *   n    = context_lens[b] clamped to [0, max_context]       (as the attention clamps it)
 *   pos  = n - q_len + i             (drafted token i sits where the causal rule places it)
 *   page = block_table[b][pos / P],  slot = pos % P
 *   code = oracle_e4m3_encode(x / scale), the quotient taken in FP32 (single precision, one
 *          correctly rounded division: the precision the kernel decides the byte in)
 * A token with pos < 0, or whose page entry lies outside [0, num_pages), is not written.
 * k_new, v_new: [B, q_len, Hkv, D] holding exact FP16 values. Returns a bit set: 1 = a token had
 * pos < 0, 2 = a page entry was out of range, 4 = context_lens[b] exceeded max_context.
 */
int oracle_kv_write(int B, int q_len, int Hkv, int D, int P, int max_pages_per_seq, int num_pages,
                    int max_context, const float* k_new, const float* v_new,
                    const int32_t* block_table, const int32_t* context_lens, float k_scale,
                    float v_scale, uint8_t* k_pool, uint8_t* v_pool)
{
    int flags = 0;
    for (int b = 0; b < B; ++b) {
        int n = context_lens[b];
        if (n > max_context) {
            n = max_context;
            flags |= 4;
        }
        if (n < 0)
            n = 0;
        for (int i = 0; i < q_len; ++i) {
            const int pos = n - q_len + i;
            if (pos < 0) {
                flags |= 1;
                continue;
            }
            const int page = block_table[(int64_t)b * max_pages_per_seq + pos / P];
            if (page < 0 || page >= num_pages) {
                flags |= 2;
                continue;
            }
            for (int h = 0; h < Hkv; ++h) {
                const int64_t src = (((int64_t)b * q_len + i) * Hkv + h) * D;
                const int64_t dst = (((int64_t)page * P + pos % P) * Hkv + h) * D;
                for (int d = 0; d < D; ++d) {
                    const float kq = k_new[src + d] / k_scale;
                    const float vq = v_new[src + d] / v_scale;
                    k_pool[dst + d] = oracle_e4m3_encode((double)kq);
                    v_pool[dst + d] = oracle_e4m3_encode((double)vq);
                }
            }
        }
    }
    return flags;
}
