/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV cache hot path.
 *
 * The operations follow the attention layer of the nano-vllm engine as the
 * pages describe it:
 *   - "L17: Qwen3 attention sub-layer" (nano-vllm series), §3 (GQA), §5.1
 *     (store_kvcache), §5.2 (FlashAttention / online softmax), §5.3 (the
 *     prefill, prefix-cache and decode calls), §7 (integration check);
 *   - "Lesson 04: where exactly does the KV go", §1 (the five forward
 *     inputs), §2 (slot_mapping), §3 (the write kernel), §4 (two
 *     FlashAttention calls), §9 (decode slot).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *    library never allocates, frees or keeps a pointer past the call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream) and never synchronises, except in validate mode
 *    (pkv_set_validate), which synchronises the stream after the launch and
 *    reports device-side checks.
 *  - bf16 tensors are passed as pkv_bf16 (the raw 16-bit pattern).
 *  - Strides are in ELEMENTS.  "Row" means one token (or one decode
 *    sequence).  Inside a row, heads are contiguous and each head's head_dim
 *    elements are contiguous (head stride == head_dim, element stride 1), as
 *    store_kvcache asserts in §5.1; the row stride itself is free (k and v
 *    may be views of a fused qkv projection output, §3).
 *  - The cache of one layer is two tensors k_cache, v_cache, each
 *    [num_blocks, block_size, num_kv_heads, head_dim] contiguous bf16; slot
 *    s = block_id * block_size + offset addresses the num_kv_heads*head_dim
 *    elements at s * num_kv_heads * head_dim (Lesson 04, §2).
 *  - block_tables is [num_seqs, bt_stride] int32; row i lists the physical
 *    blocks of sequence i in logical order, padded with -1 (Lesson 04, §1).
 *    max_blocks_per_seq <= bt_stride is the number of usable columns.
 *  - Query head h uses kv head h / (num_heads / num_kv_heads) (§3).
 *  - Return value: PKV_OK or a PKV_ERR_* code; pkv_last_error() describes the
 *    last failure on the calling host thread.  Invalid arguments are
 *    rejected before anything is launched.  Data-dependent problems that
 *    only the device can see (a slot or block id out of range, a -1 inside
 *    the used part of a block table, a length above the stated maximum) never
 *    cause an out-of-bounds access: the offending row/token is skipped or
 *    clamped and a sticky bit is set in the device status word
 *    (pkv_device_status).
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;                 /* raw bf16 bits */
typedef struct CUstream_st *pkv_stream_t;  /* same type as cudaStream_t */

enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shapes */
    PKV_ERR_UNSUPPORTED = 2,   /* a valid request the library does not handle (e.g. head_dim) */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than the *_workspace_size() */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
    PKV_ERR_DEVICE_CHECK = 5,  /* validate mode: the device flagged invalid data */
    PKV_ERR_DEVICE_TIMEOUT = 6 /* validate mode: a bounded device wait gave up */
};

/* device status bits (sticky until cleared) */
enum {
    PKV_STATUS_BAD_SLOT = 1u << 0,    /* kv_store: slot < -1 or >= num_slots        */
    PKV_STATUS_BAD_BLOCK = 1u << 1,   /* block table entry < 0 or >= num_blocks     */
    PKV_STATUS_BAD_LENGTH = 1u << 2,  /* length above its declared maximum / table   */
    PKV_STATUS_TIMEOUT = 1u << 3,     /* a bounded wait on an mbarrier expired        */
    PKV_STATUS_DUP_SLOT = 1u << 4     /* validate mode: two tokens of one call write
                                         the same slot (a write race, L17 §5.1)     */
};

/* Message describing the last error returned on this host thread ("" if none). */
const char *pkv_last_error(void);

/* ABI version (increments on any signature change). */
int pkv_version(void);

/* Validate mode: when on, every entry point synchronises `stream` after its
 * launches and turns a non-zero device status into PKV_ERR_DEVICE_CHECK or
 * PKV_ERR_DEVICE_TIMEOUT (clearing it).  The entry points that write the
 * cache (kv_store, qk_norm_rope_store, paged_attn_decode_store) also check,
 * in validate mode only, that no two tokens of the call write the same slot
 * (PKV_STATUS_DUP_SLOT); the check compares every pair of slots on the device
 * and is meant for debugging, not for the hot path.  Off by default; the
 * environment variable PKV_VALIDATE=1 turns it on at load time. */
void pkv_set_validate(int on);

/* Synchronise `stream`, then OR together the status words of every kernel
 * family of the current device into *status; clear them when `clear` != 0. */
int pkv_device_status(pkv_stream_t stream, uint32_t *status, int clear);

/* Tuning and test control of the decode split (no counterpart in the pages):
 * with tiles > 0 every later decode launch splits each sequence's keys into
 * chunks of tiles * 32 keys instead of the automatic plan (tiles == 0, the
 * default).  The chunk size changes paged_attn_decode_workspace_size(), so
 * set it before sizing workspaces.  Process-wide; returns PKV_ERR_INVALID_ARG
 * outside [0, 4096]. */
int pkv_set_decode_chunk_tiles(int tiles);

/* ------------------------------------------------------------------------
 * kv_build_slot_mapping -- Lesson 04, §2 (and §7, Exercise A).
 *
 * For sequence i with start[i] tokens already cached and
 * cu_seqlens_q[i+1] - cu_seqlens_q[i] new tokens, token t of the step
 * (logical position p = start[i] + t) is assigned
 *     slot_mapping[cu_seqlens_q[i] + t] = block_tables[i][p / block_size] * block_size
 *                                         + p % block_size.
 * The first block may start mid-block (chunked prefill), the last may end
 * mid-block.
 *   block_tables  [num_seqs, bt_stride] int32 (device)
 *   start         [num_seqs] int32 (device), cached tokens per sequence
 *   cu_seqlens_q  [num_seqs+1] int32 (device), prefix sums of new tokens
 *   slot_mapping  [num_tokens] int32 (device, output); num_tokens is the
 *                 capacity, cu_seqlens_q[num_seqs] must not exceed it.
 * A table entry that is missing (-1 or beyond max_blocks_per_seq) yields
 * slot -1 and sets PKV_STATUS_BAD_BLOCK.
 * ---------------------------------------------------------------------- */
int kv_build_slot_mapping(const int32_t *block_tables, int64_t bt_stride,
                          int32_t max_blocks_per_seq, const int32_t *start,
                          const int32_t *cu_seqlens_q, int32_t num_seqs,
                          int32_t block_size, int32_t *slot_mapping,
                          int32_t num_tokens, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * kv_build_decode_slots -- Lesson 04, §9 item 1; L17 §7.
 *
 * One new token per row: with context_lens[b] counting that token,
 *     slot_mapping[b] = block_tables[b][(ctx-1) / block_size] * block_size
 *                       + (ctx-1) % block_size
 * (the page's block_table[-1] * block_size + last_block_num_tokens - 1).
 * context_lens[b] == 0 marks a padding row of a CUDA-graph batch (L17,
 * §5.1) and yields slot -1.
 * ---------------------------------------------------------------------- */
int kv_build_decode_slots(const int32_t *block_tables, int64_t bt_stride,
                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                          int32_t batch, int32_t block_size, int32_t *slot_mapping,
                          pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * kv_store -- L17 §5.1 (store_kvcache), Lesson 04 §3.
 *
 * For every token n in [0, num_tokens) whose slot s = slot_mapping[n] is not
 * -1, copy the D = num_kv_heads * head_dim elements of key row n into
 * k_cache[s*D .. s*D+D) and of value row n into v_cache likewise.  A -1 slot
 * (a padding token) leaves the cache untouched.  Bit-exact copy.
 *   key, value  [num_tokens, num_kv_heads, head_dim] bf16, row strides
 *               key_row_stride / value_row_stride (>= D)
 *   k_cache, v_cache  num_slots * D bf16 each
 *   slot_mapping [num_tokens] int32
 * Two tokens with the same slot in one call race (invalid input; validate
 * mode flags it with PKV_STATUS_DUP_SLOT).  A slot outside [-1, num_slots)
 * is skipped and sets PKV_STATUS_BAD_SLOT.
 * ---------------------------------------------------------------------- */
int kv_store(const pkv_bf16 *key, int64_t key_row_stride,
             const pkv_bf16 *value, int64_t value_row_stride,
             pkv_bf16 *k_cache, pkv_bf16 *v_cache,
             const int32_t *slot_mapping, int32_t num_tokens,
             int32_t num_kv_heads, int32_t head_dim, int64_t num_slots,
             pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * qk_norm_rope_store -- L17 §4 (QK-Norm, then RoPE, on q and k; v as is)
 * fused with the store of §5.1 / Lesson 04 §3.
 *
 * For every token n and head h (q: num_heads heads, k: num_kv_heads):
 *   RMSNorm (layernorm module of "Nano-VLLM full-code notes (5)"):
 *     y = bf16( bf16( x / sqrt(mean(x^2) + rms_eps) ) * w )   (fp32 inside)
 *     with w = q_norm_weight or k_norm_weight [head_dim] bf16;
 *   RoPE (the pages apply it, L17 §4, but do not print it; read as the
 *   split-halves "rotate-half" pairing of the engine's model family, not the
 *   adjacent pairs of RoFormer §3.2): element e < head_dim/2 pairs with
 *   e + head_dim/2, pair i turns by a_i = positions[n] * rope_theta^(-2i/head_dim):
 *     out[i]       = y[i] cos a_i - y[i + d/2] sin a_i
 *     out[i + d/2] = y[i + d/2] cos a_i + y[i] sin a_i      (fp32, then bf16)
 * Rotated q goes to q_out; rotated k goes to k_out when k_out != NULL, and,
 * with v unchanged, to the caches at slot_mapping[n] exactly as kv_store
 * does (-1 skips the cache write; any other slot outside [0, num_slots) is
 * skipped and sets PKV_STATUS_BAD_SLOT).
 *   q [num_tokens, num_heads, head_dim], k and v [num_tokens, num_kv_heads,
 *   head_dim], all bf16 with free row strides (multiples of 8 elements,
 *   16-byte aligned), for example views into one fused qkv projection.
 *   positions [num_tokens] int64 (absolute positions; int64 as in Lesson 04
 *   §1).
 *   q_out may be q itself (same row stride), k_out may be k; otherwise the
 *   outputs must not overlap the inputs.
 * Supported: head_dim 64 or 128.  Positions are exact up to 2^24.
 * ---------------------------------------------------------------------- */
int qk_norm_rope_store(const pkv_bf16 *q, int64_t q_row_stride,
                       const pkv_bf16 *k, int64_t k_row_stride,
                       const pkv_bf16 *v, int64_t v_row_stride,
                       const int64_t *positions,
                       const pkv_bf16 *q_norm_weight, const pkv_bf16 *k_norm_weight,
                       float rms_eps, float rope_theta,
                       pkv_bf16 *q_out, int64_t q_out_row_stride,
                       pkv_bf16 *k_out, int64_t k_out_row_stride,
                       pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *slot_mapping,
                       int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int64_t num_slots, pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * paged_attn_prefill -- L17 §5.2/§5.3 (flash_attn_varlen_func with
 * causal=True), Lesson 04 §4.
 *
 * Varlen causal attention over packed sequences.  Sequence i owns query rows
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) (Lq_i rows) and Lk_i =
 * cu_seqlens_k[i+1] - cu_seqlens_k[i] >= Lq_i keys.  Query row t of the
 * sequence (0 <= t < Lq_i) attends to keys j <= Lk_i - Lq_i + t (causal mask
 * aligned to the last key: the cached prefix is seen by every new token):
 *     out[row, h] = sum_j softmax_j(softmax_scale * q[row,h] . k_j) v_j
 *     lse[row, h] = log sum_j exp(softmax_scale * q[row,h] . k_j)
 * Keys and values come from
 *   - the packed k, v [total_k, num_kv_heads, head_dim] when
 *     block_tables == NULL (plain prefill; key j of sequence i is row
 *     cu_seqlens_k[i] + j), or
 *   - the paged caches when block_tables != NULL (prefix-cache hit, §5.3:
 *     the prefix plus the chunk that kv_store has just written; key j lives
 *     at slot block_tables[i][j / block_size] * block_size + j % block_size).
 *   q    [total_q, num_heads, head_dim] bf16, row stride q_row_stride
 *   out  [total_q, num_heads, head_dim] bf16, row stride out_row_stride
 *   lse  [total_q, num_heads] fp32 or NULL
 * Supported: head_dim 128 (and 64); any num_heads / num_kv_heads; with
 * block_tables, any power-of-two block_size (blocks of 1, 2 or 4 slots are
 * gathered row by row, larger ones by TMA boxes); row strides multiples of 8
 * elements, pointers 16-byte aligned.
 * workspace: device scratch of at least paged_attn_prefill_workspace_size()
 * bytes (may be NULL when that is 0); its content need not be initialised.
 * ---------------------------------------------------------------------- */
int paged_attn_prefill(const pkv_bf16 *q, int64_t q_row_stride,
                       const pkv_bf16 *k, int64_t k_row_stride,
                       const pkv_bf16 *v, int64_t v_row_stride,
                       const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, int64_t num_blocks,
                       const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks_per_seq,
                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_seqs,
                       int32_t total_q, int32_t total_k,
                       int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, float softmax_scale,
                       pkv_bf16 *out, int64_t out_row_stride, float *lse,
                       void *workspace, size_t workspace_bytes, pkv_stream_t stream);

size_t paged_attn_prefill_workspace_size(int32_t num_seqs, int32_t total_q,
                                         int32_t max_seqlen_q, int32_t num_heads);

/* ------------------------------------------------------------------------
 * paged_attn_decode -- L17 §5.3 (flash_attn_with_kvcache), Lesson 04 §4.
 *
 * One query per sequence: row b attends to the context_lens[b] tokens of its
 * paged cache, the token kv_store wrote this step included (§4: the write
 * comes first, so step t sees position t):
 *     out[b, h] = sum_{j < ctx_b} softmax_j(softmax_scale * q[b,h] . k_j) v_j
 * with k_j at slot block_tables[b][j / block_size] * block_size + j % block_size.
 * A row with context_len 0 (padding) gets out = 0 and lse = -inf.
 * The keys of a (row, kv head) are split into chunks processed in parallel
 * and merged with the online-softmax rescaling of §5.2.
 *   q    [batch, num_heads, head_dim] bf16, row stride q_row_stride
 *   out  [batch, num_heads, head_dim] bf16, row stride out_row_stride
 *   lse  [batch, num_heads] fp32 or NULL
 *   max_context_len >= every context_lens[b] (host-side bound used to size
 *   the launch; a larger device value is clamped and flagged).
 * workspace: at least paged_attn_decode_workspace_size() bytes of device
 * scratch (256 bytes or more for any batch > 0: it holds the counter from
 * which the kernel's resident CTAs claim chunks, zeroed by the call in stream
 * order, and the chunk partials); content need not be initialised.  Calls
 * that share a workspace must be ordered on the device.
 * Supported: head_dim 64 or 128; any num_heads / num_kv_heads; block_size a
 * power of two.  A GQA group of G > 8 query heads runs as r sub-groups of
 * G / r heads (r the smallest divisor of G with G / r <= 8), each reading
 * the group's keys and values: such a call reads them r times.
 * ---------------------------------------------------------------------- */
int paged_attn_decode(const pkv_bf16 *q, int64_t q_row_stride,
                      const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, int64_t num_blocks,
                      const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t batch,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_context_len, float softmax_scale,
                      pkv_bf16 *out, int64_t out_row_stride, float *lse,
                      void *workspace, size_t workspace_bytes, pkv_stream_t stream);

size_t paged_attn_decode_workspace_size(int32_t batch, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_context_len);

/* ------------------------------------------------------------------------
 * paged_attn_decode_store -- the write-then-attend order of Lesson 04 §4
 * (store_kvcache, then flash_attn_with_kvcache) and the decode slot of
 * §4/L17 §5.3, in one launch (for a GQA group of more than 8 query heads,
 * whose sub-groups read each kv head from several CTAs, the rows are stored
 * by a launch of their own just before the decode).
 *
 * For every row b with context_lens[b] >= 1 it writes key[b] and value[b]
 * ([num_kv_heads, head_dim] each) to the decode slot of position
 * ctx_b - 1,
 *     slot_b = block_tables[b][(ctx_b-1) / block_size] * block_size
 *              + (ctx_b-1) % block_size,
 * and then computes exactly what paged_attn_decode computes over the
 * context_lens[b] tokens, the new one included.  On return (in stream order)
 * the caches hold the same bytes that kv_build_decode_slots + kv_store would
 * have written, and out/lse equal paged_attn_decode's bit for bit.
 *   key, value  [batch, num_kv_heads, head_dim] bf16, row strides in
 *               elements (multiples of 8; 16-byte aligned pointers).
 *   k_cache, v_cache are written (only the batch slots above).
 * Padding rows (context_lens[b] == 0) write nothing.  A block-table entry
 * outside [0, num_blocks) at the new position skips the write and sets
 * PKV_STATUS_BAD_BLOCK.  Two rows whose new positions map to the same slot
 * race (invalid input; validate mode flags it with PKV_STATUS_DUP_SLOT).  All other arguments, the workspace and the
 * supported shapes are those of paged_attn_decode.
 * ---------------------------------------------------------------------- */
int paged_attn_decode_store(const pkv_bf16 *q, int64_t q_row_stride,
                            const pkv_bf16 *key, int64_t key_row_stride,
                            const pkv_bf16 *value, int64_t value_row_stride,
                            pkv_bf16 *k_cache, pkv_bf16 *v_cache, int64_t num_blocks,
                            const int32_t *block_tables, int64_t bt_stride,
                            int32_t max_blocks_per_seq, const int32_t *context_lens,
                            int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int32_t max_context_len,
                            float softmax_scale, pkv_bf16 *out, int64_t out_row_stride,
                            float *lse, void *workspace, size_t workspace_bytes,
                            pkv_stream_t stream);

/* ------------------------------------------------------------------------
 * paged_attn_decode_noalloc -- the pages have no counterpart: this entry
 * point exists for callers of this library that cannot allocate device
 * memory, such as a plugin inside a host framework that owns every device
 * allocation and only passes tensors in, or a runtime that forbids
 * allocations after start-up.  It computes exactly what paged_attn_decode
 * computes, with the same arguments minus the workspace: its scratch (the
 * chunk counter and the split partials) goes to a static device array of
 * PKV_DECODE_STATIC_SCRATCH_BYTES owned by the library, which every GPU
 * that loads the library keeps resident until the process exits.  The
 * caller still passes inputs and outputs.  It calls no cudaMalloc, cudaFree
 * or allocating library routine.
 *   - A launch whose paged_attn_decode_workspace_size() exceeds
 *     PKV_DECODE_STATIC_SCRATCH_BYTES is rejected with PKV_ERR_WORKSPACE and
 *     a message saying so; nothing is launched.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture on the device.  The address is kept for the life of the
 *     process: it assumes the device's primary context, in which the CUDA
 *     runtime loaded the library, is not destroyed while the library is in
 *     use (no cudaDeviceReset between calls).
 *   - Every call shares the one array, which keeps the last call's contents
 *     (nothing in it needs to start at zero).  Calls that can overlap on the
 *     GPU (different streams, or several host threads, without ordering
 *     between them) race on it and give wrong results; order them.
 * ---------------------------------------------------------------------- */
#define PKV_DECODE_STATIC_SCRATCH_BYTES (16u << 20)

int paged_attn_decode_noalloc(const pkv_bf16 *q, int64_t q_row_stride,
                              const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, int64_t num_blocks,
                              const int32_t *block_tables, int64_t bt_stride,
                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t block_size, int32_t max_context_len,
                              float softmax_scale, pkv_bf16 *out, int64_t out_row_stride,
                              float *lse, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
