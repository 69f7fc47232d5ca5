/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the paged KV
 * cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * under paged_kv_cache_303_gb300/) may include, link or call this file; only
 * the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * Sources (page title + section):
 *   [P2] "L17: Qwen3 attention sub-layer" (nano-vllm series, yeyulingfeng.com)
 *        §3 QKV projection and GQA, §5.1 store_kvcache, §5.2 FlashAttention
 *        (naive definition and online softmax), §5.3 prefill/decode calls,
 *        §7 integration check.
 *   [P3] "Lesson 04: where exactly does the KV go" (diomchen.github.io)
 *        §2 how slot_mapping is built, §3 the write kernel, §4 two
 *        FlashAttention calls, §7 Exercise A, §9 code hunt item 1.
 *   [P1] "Nano-VLLM full-code notes (5): layernorm & attention"
 *        (m.demingchina.com), the RMSNorm module (layernorm.py).
 *   [P2] §4 applies a rotary position embedding after QK-Norm but does
 *        not print it (it defers to an earlier lesson that is not among the
 *        pages).  The reading taken is the split-halves ("rotate-half")
 *        pairing used by the engine's model family: element e < d/2 pairs
 *        with e + d/2.  (RoFormer, Su et al. 2021, §3.2, writes the same
 *        rotation over adjacent pairs (x_2i, x_2i+1); that interleaved form is
 *        a different permutation of the dimensions and is not computed here.)
 *
 * Arithmetic: bf16 inputs are widened exactly (bits << 16) to float and then
 * to double; every score, exponential, sum and output is computed in double
 * (fp64).  Attention follows the three-step naive definition of [P2] §5.2:
 * S = scale * Q K^T, P = row softmax(S), O = P V, with the row maximum
 * subtracted before exponentiation (shift invariance, same section).
 *
 * Every function returns 0 on success or a negative ORC_E* code on invalid
 * input; it never reads or writes out of the bounds its arguments describe.
 *
 * ORC_PLANT_* macros (never defined in normal builds) each plant one
 * plausible mistake; tests/test_oracle_planted.py rebuilds the oracle with
 * each of them and checks that the pins catch it.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EARG (-1)      /* malformed sizes / null pointers            */
#define ORC_ESLOT (-2)     /* slot out of range (other than -1)          */
#define ORC_EDUP (-3)      /* the same slot written twice in one call    */
#define ORC_ETABLE (-4)    /* block table entry missing / out of range   */
#define ORC_ELEN (-5)      /* inconsistent sequence lengths              */
#define ORC_ENOMEM (-6)

/* exact bf16 -> double widening: a bf16 value is the top half of a float */
static double bf16_to_f64(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_version(void) { return 1; }

/* ------------------------------------------------------------------------
 * slot_mapping, prefill / chunked prefill.
 *
 * [P3] §2: for a sequence whose first `start` tokens are already cached and
 * which computes tokens [start, end) this step, walk the logical blocks
 * start_block = start / bs ... end_block = ceil(end / bs) - 1; the first
 * block begins at start % bs, the last one stops at end - i*bs, every other
 * block is covered entirely.  The slots of one sequence follow each other in
 * token order; sequences are concatenated in cu_seqlens_q order ([P3] §1).
 * A physical slot is block_id * block_size + offset ([P3] §2, the flat
 * kv_cache tensor).
 * ---------------------------------------------------------------------- */
int orc_slot_mapping_blockwalk(const int32_t *block_tables, int64_t bt_stride,
                               int32_t max_blocks, const int32_t *start,
                               const int32_t *cu_seqlens_q, int32_t num_seqs,
                               int32_t block_size, int32_t *slot_mapping,
                               int64_t num_tokens)
{
    if (num_seqs < 0 || block_size <= 0 || max_blocks < 0 || num_tokens < 0)
        return ORC_EARG;
    if (cu_seqlens_q[0] != 0 || cu_seqlens_q[num_seqs] != num_tokens)
        return ORC_ELEN;
    int64_t w = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int64_t len = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int64_t s = start[i];
        if (len < 0 || s < 0)
            return ORC_ELEN;
        int64_t e = s + len;
        const int32_t *row = block_tables + (int64_t)i * bt_stride;
        int64_t start_block = s / block_size;
        int64_t end_block = (e + block_size - 1) / block_size;
        for (int64_t b = start_block; b < end_block; ++b) {
            if (b >= max_blocks || row[b] < 0)
                return ORC_ETABLE;
            int64_t base = (int64_t)row[b] * block_size;
            int64_t lo = base;
            if (b == start_block)
                lo += s % block_size;               /* first block: mid-block start */
            int64_t hi;
            if (b != end_block - 1)
                hi = base + block_size;             /* full block */
            else
                hi = base + (e - b * block_size);   /* last block: stop at end */
            for (int64_t x = lo; x < hi; ++x) {
                if (w >= num_tokens)
                    return ORC_ELEN;
                slot_mapping[w++] = (int32_t)x;
            }
        }
    }
    return w == num_tokens ? ORC_OK : ORC_ELEN;
}

/* The same mapping written token by token: logical position p of sequence i
 * lives in logical block p / bs at offset p % bs, so its slot is
 * table[i][p / bs] * bs + p % bs ([P3] §2 and §7, the worked answer).
 * Kept as a second, independent statement so that the two can be checked
 * against each other. */
int orc_slot_mapping_per_token(const int32_t *block_tables, int64_t bt_stride,
                               int32_t max_blocks, const int32_t *start,
                               const int32_t *cu_seqlens_q, int32_t num_seqs,
                               int32_t block_size, int32_t *slot_mapping,
                               int64_t num_tokens)
{
    if (num_seqs < 0 || block_size <= 0 || max_blocks < 0 || num_tokens < 0)
        return ORC_EARG;
    if (cu_seqlens_q[0] != 0 || cu_seqlens_q[num_seqs] != num_tokens)
        return ORC_ELEN;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int64_t len = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        if (len < 0 || start[i] < 0)
            return ORC_ELEN;
        const int32_t *row = block_tables + (int64_t)i * bt_stride;
        for (int64_t t = 0; t < len; ++t) {
            int64_t p = (int64_t)start[i] + t;
            int64_t lb = p / block_size;
            if (lb >= max_blocks || row[lb] < 0)
                return ORC_ETABLE;
#ifdef ORC_PLANT_SLOT_OFFSET
            slot_mapping[cu_seqlens_q[i] + t] =
                (int32_t)((int64_t)row[lb] * block_size + (p + 1) % block_size);
#else
            slot_mapping[cu_seqlens_q[i] + t] =
                (int32_t)((int64_t)row[lb] * block_size + p % block_size);
#endif
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Decode slot: one new token per sequence ([P3] §9 item 1):
 *   slot = block_table[-1] * block_size + last_block_num_tokens - 1
 * where the sequence already counts the new token (context_len includes it,
 * [P2] §7: slot N written, context length N + 1).  "block_table[-1]" is the
 * table entry that holds position context_len - 1, i.e. entry
 * (context_len - 1) / bs, and last_block_num_tokens is the number of tokens
 * in that block.  A row with context_len == 0 is a padding row of a
 * CUDA-graph batch ([P2] §5.1) and gets slot -1.
 * ---------------------------------------------------------------------- */
int orc_decode_slots(const int32_t *block_tables, int64_t bt_stride,
                     int32_t max_blocks, const int32_t *context_lens,
                     int32_t batch, int32_t block_size, int32_t *slot_mapping)
{
    if (batch < 0 || block_size <= 0 || max_blocks < 0)
        return ORC_EARG;
    for (int32_t b = 0; b < batch; ++b) {
        int64_t ctx = context_lens[b];
        if (ctx < 0)
            return ORC_ELEN;
        if (ctx == 0) {
            slot_mapping[b] = -1;
            continue;
        }
        int64_t last = (ctx - 1) / block_size;          /* index of the last used entry */
        if (last >= max_blocks)
            return ORC_ETABLE;
        int32_t blk = block_tables[(int64_t)b * bt_stride + last];
        if (blk < 0)
            return ORC_ETABLE;
        int64_t last_block_num_tokens = ctx - last * block_size;
        slot_mapping[b] = (int32_t)((int64_t)blk * block_size + last_block_num_tokens - 1);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * store_kvcache ([P2] §5.1, [P3] §3): for every token n whose slot is not
 * -1, copy the D = num_kv_heads * head_dim contiguous elements of key row n
 * (found at n * key_row_stride) into k_cache at slot * D, and the value row
 * into v_cache likewise.  A -1 slot leaves the cache untouched.  Any other
 * slot outside [0, num_slots), or a slot written twice in the same call, is
 * rejected before anything is written.
 * ---------------------------------------------------------------------- */
int orc_kv_store(const uint16_t *key, int64_t key_row_stride,
                 const uint16_t *value, int64_t value_row_stride,
                 uint16_t *k_cache, uint16_t *v_cache,
                 const int32_t *slot_mapping, int64_t num_tokens,
                 int64_t D, int64_t num_slots)
{
    if (num_tokens < 0 || D <= 0 || num_slots < 0)
        return ORC_EARG;
    unsigned char *seen = (unsigned char *)calloc((size_t)(num_slots > 0 ? num_slots : 1), 1);
    if (!seen)
        return ORC_ENOMEM;
    for (int64_t n = 0; n < num_tokens; ++n) {
        int64_t s = slot_mapping[n];
        if (s == -1)
            continue;
        if (s < 0 || s >= num_slots) {
            free(seen);
            return ORC_ESLOT;
        }
        if (seen[s]) {
            free(seen);
            return ORC_EDUP;
        }
        seen[s] = 1;
    }
    free(seen);
    for (int64_t n = 0; n < num_tokens; ++n) {
        int64_t s = slot_mapping[n];
#ifdef ORC_PLANT_KEEP_PADDING
        if (s == -1)
            s = num_slots - 1;
#else
        if (s == -1)
            continue;
#endif
        for (int64_t e = 0; e < D; ++e) {
            k_cache[s * D + e] = key[n * key_row_stride + e];
            v_cache[s * D + e] = value[n * value_row_stride + e];
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Attention core.
 *
 * One query row attends to keys 0 .. n_keys-1 of its sequence; row t of a
 * sequence with Lq queries and Lk keys sees n_keys = Lk - Lq + t + 1 keys
 * (causal, aligned so that the last query sees every key: the prefix-cache
 * prefill of [P2] §5.3 has k longer than q, the prefix is not recomputed,
 * and decode at step t sees position t itself, [P3] §4).  With Lk == Lq
 * this is the ordinary block-diagonal causal mask of varlen prefill.
 *
 * Query head h reads kv head h / (Hq / Hkv): the Hq/Hkv query heads of one
 * group are consecutive and share one kv head ([P2] §3).
 *
 * Key j of the sequence is found either in the packed k/v tensors (row
 * cu_seqlens_k[i] + j) or, when a block table is given, in the paged cache
 * at slot table[i][j / bs] * bs + j % bs ([P3] §2, §4).
 * ---------------------------------------------------------------------- */
typedef struct {
    const uint16_t *q; int64_t q_rs;
    const uint16_t *k; int64_t k_rs;
    const uint16_t *v; int64_t v_rs;
    const uint16_t *kc; const uint16_t *vc; int64_t num_blocks;
    const int32_t *bt; int64_t bt_stride; int32_t max_blocks;
    int32_t Hq, Hkv, d, bs;
    double scale;
} orc_attn_args;

/* address of key/value row j of sequence i, kv head kvh; NULL if the table
 * does not cover it */
static const uint16_t *kv_row(const orc_attn_args *a, const uint16_t *packed,
                              int64_t packed_rs, const uint16_t *cache,
                              int32_t i, int64_t k_begin, int64_t j, int32_t kvh)
{
    if (!a->bt)
        return packed + (k_begin + j) * packed_rs + (int64_t)kvh * a->d;
    int64_t lb = j / a->bs;
    if (lb >= a->max_blocks)
        return NULL;
    int64_t blk = a->bt[(int64_t)i * a->bt_stride + lb];
    if (blk < 0 || blk >= a->num_blocks)
        return NULL;
    int64_t slot = blk * a->bs + j % a->bs;
    return cache + (slot * a->Hkv + kvh) * a->d;
}

/* one (sequence, query head, query row): naive softmax attention, fp64 */
static int attend_row(const orc_attn_args *a, int32_t i, int64_t k_begin,
                      int64_t q_row, int32_t h, int64_t n_keys,
                      double *s, double *o, double *lse_out)
{
    const int32_t g = a->Hq / a->Hkv;
#ifdef ORC_PLANT_GQA_MODULO
    const int32_t kvh = h % a->Hkv;
#else
    const int32_t kvh = h / g;
#endif
    const uint16_t *qr = a->q + q_row * a->q_rs + (int64_t)h * a->d;
    for (int32_t e = 0; e < a->d; ++e)
        o[e] = 0.0;
    if (n_keys <= 0) {              /* nothing to attend to: zero output */
        *lse_out = -INFINITY;
        return ORC_OK;
    }
    /* step 1: scaled scores s_j = scale * <q, k_j> */
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *kr = kv_row(a, a->k, a->k_rs, a->kc, i, k_begin, j, kvh);
        if (!kr)
            return ORC_ETABLE;
        double dot = 0.0;
        for (int32_t e = 0; e < a->d; ++e)
            dot += bf16_to_f64(qr[e]) * bf16_to_f64(kr[e]);
#ifdef ORC_PLANT_NO_SCALE
        s[j] = dot;
#else
        s[j] = a->scale * dot;
#endif
    }
    /* step 2: row softmax, shifted by the row maximum */
    double m = s[0];
    for (int64_t j = 1; j < n_keys; ++j)
        if (s[j] > m)
            m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* step 3: O = P V */
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *vr = kv_row(a, a->v, a->v_rs, a->vc, i, k_begin, j, kvh);
        if (!vr)
            return ORC_ETABLE;
        double p = s[j] / l;
#ifdef ORC_PLANT_V_REVERSED
        for (int32_t e = 0; e < a->d; ++e)
            o[e] += p * bf16_to_f64(vr[a->d - 1 - e]);
#else
        for (int32_t e = 0; e < a->d; ++e)
            o[e] += p * bf16_to_f64(vr[e]);
#endif
    }
    *lse_out = m + log(l);
    return ORC_OK;
}

static int check_heads(int32_t Hq, int32_t Hkv, int32_t d)
{
    if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0)
        return ORC_EARG;
    return ORC_OK;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int orc_num_threads(int nthreads)
{
#ifdef _OPENMP
    set_threads(nthreads);
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
#else
    (void)nthreads;
    return 1;
#endif
}

/* Varlen causal prefill, with or without a prefix in the paged cache
 * ([P2] §5.3, [P3] §4).  q is [total_q, Hq, d] with row stride q_rs; out is
 * [total_q, Hq, d] doubles; lse (optional) is [total_q, Hq].  When bt is
 * NULL keys come from the packed k/v (row strides k_rs / v_rs), else from
 * the paged caches [num_blocks, bs, Hkv, d]. */
int orc_prefill(const uint16_t *q, int64_t q_rs,
                const uint16_t *k, int64_t k_rs, const uint16_t *v, int64_t v_rs,
                const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks,
                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t d,
                int32_t block_size, double scale, double *out, double *lse,
                int nthreads)
{
    if (check_heads(Hq, Hkv, d) || num_seqs < 0)
        return ORC_EARG;
    if (block_tables && (block_size <= 0 || !k_cache || !v_cache))
        return ORC_EARG;
    if (!block_tables && (!k || !v))
        return ORC_EARG;
    orc_attn_args a = {q, q_rs, k, k_rs, v, v_rs, k_cache, v_cache, num_blocks,
                       block_tables, bt_stride, max_blocks, Hq, Hkv, d, block_size, scale};
    int64_t max_lk = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int64_t lq = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int64_t lk = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
        if (lq < 0 || lk < lq)
            return ORC_ELEN;
        if (lk > max_lk)
            max_lk = lk;
    }
    int rc = ORC_OK;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(max_lk > 0 ? max_lk : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !o) {
#pragma omp atomic write
            rc = ORC_ENOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int32_t i = 0; i < num_seqs; ++i) {
            for (int32_t h = 0; h < Hq; ++h) {
                if (!s || !o)
                    continue;
                int64_t lq = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
                int64_t lk = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
                for (int64_t t = 0; t < lq; ++t) {
                    int64_t row = cu_seqlens_q[i] + t;
                    double l;
#ifdef ORC_PLANT_CAUSAL_OFF_BY_ONE
                    int r = attend_row(&a, i, cu_seqlens_k[i], row, h, lk - lq + t, s, o, &l);
#else
                    int r = attend_row(&a, i, cu_seqlens_k[i], row, h, lk - lq + t + 1, s, o, &l);
#endif
                    if (r) {
#pragma omp atomic write
                        rc = r;
                        break;
                    }
                    memcpy(out + (row * Hq + h) * (int64_t)d, o, sizeof(double) * (size_t)d);
                    if (lse)
                        lse[row * Hq + h] = l;
                }
            }
        }
        free(s);
        free(o);
    }
    return rc;
}

/* Single-token decode ([P2] §5.3, [P3] §4): query b attends to the
 * context_lens[b] tokens in the paged cache, the one written this step
 * included.  context_len 0 (a padding row) yields a zero output. */
int orc_decode(const uint16_t *q, int64_t q_rs,
               const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
               const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks,
               const int32_t *context_lens, int32_t batch,
               int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
               double scale, double *out, double *lse, int nthreads)
{
    if (check_heads(Hq, Hkv, d) || batch < 0 || block_size <= 0)
        return ORC_EARG;
    orc_attn_args a = {q, q_rs, NULL, 0, NULL, 0, k_cache, v_cache, num_blocks,
                       block_tables, bt_stride, max_blocks, Hq, Hkv, d, block_size, scale};
    int64_t max_ctx = 1;
    for (int32_t b = 0; b < batch; ++b) {
        if (context_lens[b] < 0)
            return ORC_ELEN;
        if (context_lens[b] > max_ctx)
            max_ctx = context_lens[b];
    }
    int rc = ORC_OK;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)max_ctx);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !o) {
#pragma omp atomic write
            rc = ORC_ENOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int32_t b = 0; b < batch; ++b) {
            for (int32_t h = 0; h < Hq; ++h) {
                if (!s || !o)
                    continue;
                double l;
                int r = attend_row(&a, b, 0, b, h, context_lens[b], s, o, &l);
                if (r) {
#pragma omp atomic write
                    rc = r;
                    continue;
                }
                memcpy(out + ((int64_t)b * Hq + h) * d, o, sizeof(double) * (size_t)d);
                if (lse)
                    lse[(int64_t)b * Hq + h] = l;
            }
        }
        free(s);
        free(o);
    }
    return rc;
}

/* ------------------------------------------------------------------------
 * Online (blocked) softmax, [P2] §5.2.  One row of already-scaled scores
 * s[0..n) with value vectors v[j][0..w) is consumed `block` entries at a
 * time while three accumulators are kept: the running maximum m, the
 * running denominator l and the unnormalised output acc.  When a block
 * raises the maximum from m to m', the old l and acc are multiplied by
 * exp(m - m') (the factorisation exp(x - m') = exp(x - m) exp(m - m')); the
 * block's own terms exp(s_j - m') and exp(s_j - m') v_j are then added.
 * After the last block the output is acc / l.
 *
 * For every block b the trace receives 3 + 2w doubles:
 *   m after the block, l and acc[0..w) after rescaling (before the block's
 *   terms are added), l and acc[0..w) after the block.
 * trace may be NULL.
 * ---------------------------------------------------------------------- */
int orc_online_softmax(const double *s, const double *v, int64_t n, int64_t w,
                       int64_t block, double *out, double *out_m, double *out_l,
                       double *trace)
{
    if (n <= 0 || w <= 0 || block <= 0)
        return ORC_EARG;
    double *acc = (double *)calloc((size_t)w, sizeof(double));
    if (!acc)
        return ORC_ENOMEM;
    double m = -INFINITY, l = 0.0;
    int64_t nb = 0;
    for (int64_t j0 = 0; j0 < n; j0 += block, ++nb) {
        int64_t j1 = j0 + block < n ? j0 + block : n;
        double mb = s[j0];
        for (int64_t j = j0 + 1; j < j1; ++j)
            if (s[j] > mb)
                mb = s[j];
        double m_new = mb > m ? mb : m;
#ifdef ORC_PLANT_NO_RESCALE
        double f = 1.0;
#else
        double f = (m == -INFINITY) ? 0.0 : exp(m - m_new);
#endif
        l *= f;
        for (int64_t e = 0; e < w; ++e)
            acc[e] *= f;
        double *tr = trace ? trace + nb * (3 + 2 * w) : NULL;
        if (tr) {
            tr[0] = m_new;
            tr[1] = l;
            for (int64_t e = 0; e < w; ++e)
                tr[2 + e] = acc[e];
        }
        for (int64_t j = j0; j < j1; ++j) {
            double p = exp(s[j] - m_new);
            l += p;
            for (int64_t e = 0; e < w; ++e)
                acc[e] += p * v[j * w + e];
        }
        if (tr) {
            tr[2 + w] = l;
            for (int64_t e = 0; e < w; ++e)
                tr[3 + w + e] = acc[e];
        }
        m = m_new;
    }
    for (int64_t e = 0; e < w; ++e)
        out[e] = acc[e] / l;
    if (out_m)
        *out_m = m;
    if (out_l)
        *out_l = l;
    free(acc);
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * Split-K decode, the decomposition used to spread one long context over
 * many workers.  The keys of each (sequence, head) are cut into consecutive
 * splits of `split` tokens; each split is reduced on its own to the triple
 * (m_s, l_s, acc_s) by the naive definition (its maximum, its sum of
 * exp(s_j - m_s), and its sum of exp(s_j - m_s) v_j), and the triples are
 * merged with the rescaling identity of [P2] §5.2:
 *   m = max_s m_s,  l = sum_s exp(m_s - m) l_s,
 *   O = sum_s exp(m_s - m) acc_s / l.
 * The result must equal orc_decode up to rounding.
 * ---------------------------------------------------------------------- */
int orc_decode_split(const uint16_t *q, int64_t q_rs,
                     const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                     const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks,
                     const int32_t *context_lens, int32_t batch,
                     int32_t Hq, int32_t Hkv, int32_t d, int32_t block_size,
                     double scale, int64_t split, double *out, double *lse)
{
    if (check_heads(Hq, Hkv, d) || batch < 0 || block_size <= 0 || split <= 0)
        return ORC_EARG;
    orc_attn_args a = {q, q_rs, NULL, 0, NULL, 0, k_cache, v_cache, num_blocks,
                       block_tables, bt_stride, max_blocks, Hq, Hkv, d, block_size, scale};
    const int32_t g = Hq / Hkv;
    int64_t max_ctx = 1;
    for (int32_t b = 0; b < batch; ++b) {
        if (context_lens[b] < 0)
            return ORC_ELEN;
        if (context_lens[b] > max_ctx)
            max_ctx = context_lens[b];
    }
    int64_t max_splits = (max_ctx + split - 1) / split;
    double *sm = (double *)malloc(sizeof(double) * (size_t)max_splits);
    double *sl = (double *)malloc(sizeof(double) * (size_t)max_splits);
    double *sacc = (double *)malloc(sizeof(double) * (size_t)(max_splits * d));
    double *s = (double *)malloc(sizeof(double) * (size_t)split);
    if (!sm || !sl || !sacc || !s) {
        free(sm); free(sl); free(sacc); free(s);
        return ORC_ENOMEM;
    }
    int rc = ORC_OK;
    for (int32_t b = 0; b < batch && rc == ORC_OK; ++b) {
        int64_t ctx = context_lens[b];
        int64_t ns = (ctx + split - 1) / split;
        for (int32_t h = 0; h < Hq && rc == ORC_OK; ++h) {
            const uint16_t *qr = q + (int64_t)b * q_rs + (int64_t)h * d;
            double *o = out + ((int64_t)b * Hq + h) * d;
            for (int32_t e = 0; e < d; ++e)
                o[e] = 0.0;
            if (ns == 0) {
                if (lse)
                    lse[(int64_t)b * Hq + h] = -INFINITY;
                continue;
            }
            for (int64_t sp = 0; sp < ns && rc == ORC_OK; ++sp) {
                int64_t j0 = sp * split, j1 = j0 + split < ctx ? j0 + split : ctx;
                for (int64_t j = j0; j < j1; ++j) {
                    const uint16_t *kr = kv_row(&a, NULL, 0, k_cache, b, 0, j, h / g);
                    if (!kr) { rc = ORC_ETABLE; break; }
                    double dot = 0.0;
                    for (int32_t e = 0; e < d; ++e)
                        dot += bf16_to_f64(qr[e]) * bf16_to_f64(kr[e]);
                    s[j - j0] = scale * dot;
                }
                if (rc)
                    break;
                double m = s[0];
                for (int64_t j = 1; j < j1 - j0; ++j)
                    if (s[j] > m)
                        m = s[j];
                double l = 0.0;
                double *acc = sacc + sp * d;
                for (int32_t e = 0; e < d; ++e)
                    acc[e] = 0.0;
                for (int64_t j = j0; j < j1; ++j) {
                    const uint16_t *vr = kv_row(&a, NULL, 0, v_cache, b, 0, j, h / g);
                    if (!vr) { rc = ORC_ETABLE; break; }
                    double p = exp(s[j - j0] - m);
                    l += p;
                    for (int32_t e = 0; e < d; ++e)
                        acc[e] += p * bf16_to_f64(vr[e]);
                }
                sm[sp] = m;
                sl[sp] = l;
            }
            if (rc)
                break;
            double M = sm[0];
            for (int64_t sp = 1; sp < ns; ++sp)
                if (sm[sp] > M)
                    M = sm[sp];
            double L = 0.0;
            for (int64_t sp = 0; sp < ns; ++sp)
                L += exp(sm[sp] - M) * sl[sp];
            for (int64_t sp = 0; sp < ns; ++sp) {
                double f = exp(sm[sp] - M) / L;
                for (int32_t e = 0; e < d; ++e)
                    o[e] += f * sacc[sp * d + e];
            }
            if (lse)
                lse[(int64_t)b * Hq + h] = M + log(L);
        }
    }
    free(sm); free(sl); free(sacc); free(s);
    return rc;
}

/* Prefill restricted to selected query rows (global row indices into q),
 * for checking full-size launches on a sample: rows[r] is looked up in
 * cu_seqlens_q, then computed exactly as orc_prefill computes it.
 * out is [n_rows, Hq, d], lse [n_rows, Hq] (optional). */
int orc_prefill_rows(const uint16_t *q, int64_t q_rs,
                     const uint16_t *k, int64_t k_rs, const uint16_t *v, int64_t v_rs,
                     const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                     const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks,
                     const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                     int32_t num_seqs, int32_t Hq, int32_t Hkv, int32_t d,
                     int32_t block_size, double scale, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, int nthreads)
{
    if (check_heads(Hq, Hkv, d) || num_seqs < 0 || n_rows < 0)
        return ORC_EARG;
    if (block_tables && (block_size <= 0 || !k_cache || !v_cache))
        return ORC_EARG;
    if (!block_tables && (!k || !v))
        return ORC_EARG;
    orc_attn_args a = {q, q_rs, k, k_rs, v, v_rs, k_cache, v_cache, num_blocks,
                       block_tables, bt_stride, max_blocks, Hq, Hkv, d, block_size, scale};
    int64_t max_lk = 1;
    for (int32_t i = 0; i < num_seqs; ++i) {
        int64_t lq = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        int64_t lk = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
        if (lq < 0 || lk < lq)
            return ORC_ELEN;
        if (lk > max_lk)
            max_lk = lk;
    }
    int rc = ORC_OK;
    set_threads(nthreads);
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)max_lk);
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
        if (!s || !o) {
#pragma omp atomic write
            rc = ORC_ENOMEM;
        }
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            for (int32_t h = 0; h < Hq; ++h) {
                if (!s || !o)
                    continue;
                int64_t row = rows[r];
                int32_t i = 0;
                while (i < num_seqs && cu_seqlens_q[i + 1] <= row)
                    ++i;
                if (i >= num_seqs || row < cu_seqlens_q[i]) {
#pragma omp atomic write
                    rc = ORC_EARG;
                    continue;
                }
                int64_t lq = (int64_t)cu_seqlens_q[i + 1] - cu_seqlens_q[i];
                int64_t lk = (int64_t)cu_seqlens_k[i + 1] - cu_seqlens_k[i];
                int64_t t = row - cu_seqlens_q[i];
                double l;
                int e = attend_row(&a, i, cu_seqlens_k[i], row, h, lk - lq + t + 1, s, o, &l);
                if (e) {
#pragma omp atomic write
                    rc = e;
                    continue;
                }
                memcpy(out + (r * Hq + h) * (int64_t)d, o, sizeof(double) * (size_t)d);
                if (lse)
                    lse[r * Hq + h] = l;
            }
        }
        free(s);
        free(o);
    }
    return rc;
}

/* ------------------------------------------------------------------------
 * Round a double to the nearest bf16 (ties to even), returned as its bit
 * pattern.  bf16 keeps 8 significant bits: for |x| = m * 2^k with m in
 * [0.5, 1), x is rounded to a multiple of 2^(k-8).  Values here are far
 * from the bf16 overflow and subnormal ranges; those, NaN and infinities go
 * through float, whose rounding there is the same.
 * ---------------------------------------------------------------------- */
uint16_t orc_round_bf16(double x)
{
    double ax = fabs(x);
    uint32_t u;
    float f;
    if (ax >= 0x1p-126 && ax < 0x1p127) {
        int k;
        double m = frexp(x, &k);      /* x = m * 2^k, 0.5 <= |m| < 1 */
#ifdef ORC_PLANT_ROUND_TRUNC
        f = (float)ldexp(trunc(ldexp(m, 8)), k - 8);
#else
        f = (float)ldexp(nearbyint(ldexp(m, 8)), k - 8);   /* exact in float */
#endif
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    /* zero, subnormal range, huge, inf, NaN: through float */
    f = (float)x;
    memcpy(&u, &f, sizeof u);
    if (f != f)
        return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------
 * QK-Norm then RoPE on one row of head_dim elements ([P2] §4: q and k of
 * every head are RMS-normalised over head_dim, then rotated by position; v
 * is left alone).
 *
 * RMSNorm ([P1], layernorm.py): widen to float, divide by
 * sqrt(mean(x^2) + eps), convert back to the input dtype (bf16), and only
 * then multiply by the bf16 weight (a bf16 product, rounded).  The oracle
 * keeps the two roundings to bf16 where the module has them and computes
 * everything else in double.
 *
 * RoPE (a reading: [P2] §4 applies it without printing it; the
 * split-halves "rotate-half" pairing of the engine's model family, not the
 * adjacent pairs of RoFormer §3.2): element e < d/2 pairs with e + d/2;
 * pair i turns by the angle pos * theta^(-2i/d):
 *     y[i]       = x[i] cos(a_i) - x[i + d/2] sin(a_i)
 *     y[i + d/2] = x[i + d/2] cos(a_i) + x[i] sin(a_i)
 * computed in double from the bf16 QK-Norm output and rounded to bf16 once.
 * ---------------------------------------------------------------------- */
static void norm_rope_row(const uint16_t *x, const uint16_t *w, int32_t d, double eps,
                          double pos, double theta, uint16_t *out, double *tmp)
{
    double ss = 0.0;
    for (int32_t e = 0; e < d; ++e) {
        double v = bf16_to_f64(x[e]);
        ss += v * v;
    }
#if defined(ORC_PLANT_NORM_SUM)
    double inv = 1.0 / sqrt(ss + eps);
#elif defined(ORC_PLANT_EPS_OUTSIDE)
    double inv = 1.0 / (sqrt(ss / d) + eps);
#else
    double inv = 1.0 / sqrt(ss / d + eps);
#endif
    for (int32_t e = 0; e < d; ++e) {
        double n = bf16_to_f64(orc_round_bf16(bf16_to_f64(x[e]) * inv));
        tmp[e] = bf16_to_f64(orc_round_bf16(n * bf16_to_f64(w[e])));
    }
    int32_t h = d / 2;
#ifdef ORC_PLANT_ROPE_INTERLEAVED
    for (int32_t i = 0; i < h; ++i) {
        double a = pos * pow(theta, -2.0 * i / d);
        double c = cos(a), sn = sin(a);
        out[2 * i] = orc_round_bf16(tmp[2 * i] * c - tmp[2 * i + 1] * sn);
        out[2 * i + 1] = orc_round_bf16(tmp[2 * i + 1] * c + tmp[2 * i] * sn);
    }
    return;
#endif
    for (int32_t i = 0; i < h; ++i) {
#ifdef ORC_PLANT_ROPE_FREQ
        double a = pos * pow(theta, -1.0 * i / d);
#else
        double a = pos * pow(theta, -2.0 * i / d);
#endif
        double c = cos(a), sn = sin(a);
#ifdef ORC_PLANT_ROPE_SIGN
        sn = -sn;
#endif
        out[i] = orc_round_bf16(tmp[i] * c - tmp[i + h] * sn);
        out[i + h] = orc_round_bf16(tmp[i + h] * c + tmp[i] * sn);
    }
}

/* q [N, Hq, d] and k [N, Hkv, d] (bf16 bits, row strides q_rs / k_rs in
 * elements, heads contiguous) -> q_out [N, Hq, d], k_out [N, Hkv, d]
 * (contiguous).  positions[n] is token n's absolute position; q_w and k_w
 * are the d-element bf16 weights of the two norms. */
int orc_qk_norm_rope(const uint16_t *q, int64_t q_rs, const uint16_t *k, int64_t k_rs,
                     const int64_t *positions, const uint16_t *q_w, const uint16_t *k_w,
                     double eps, double theta, int64_t num_tokens, int32_t Hq, int32_t Hkv,
                     int32_t d, uint16_t *q_out, uint16_t *k_out)
{
    if (num_tokens < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || (d & 1) || eps < 0 || theta <= 0 ||
        q_rs < (int64_t)Hq * d || k_rs < (int64_t)Hkv * d)
        return ORC_EARG;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    if (!tmp)
        return ORC_ENOMEM;
    for (int64_t n = 0; n < num_tokens; ++n) {
        double pos = (double)positions[n];
        for (int32_t h = 0; h < Hq; ++h)
            norm_rope_row(q + n * q_rs + (int64_t)h * d, q_w, d, eps, pos, theta,
                          q_out + (n * Hq + h) * d, tmp);
        for (int32_t h = 0; h < Hkv; ++h)
            norm_rope_row(k + n * k_rs + (int64_t)h * d, k_w, d, eps, pos, theta,
                          k_out + (n * Hkv + h) * d, tmp);
    }
    free(tmp);
    return ORC_OK;
}
