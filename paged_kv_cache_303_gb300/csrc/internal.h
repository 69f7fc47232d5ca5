// internal.h -- host-side interface between the C ABI layer (api.cu) and the
// kernel translation units.  Arguments arriving here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr int kMaxDevices = 64;

// One-time set-up per device (kernel attributes, occupancy queries) that is
// safe when several host threads make their first call on a device at the
// same time: the first caller runs `fn` under a lock, the others wait for it;
// a failed set-up is retried by the next call.  Values `fn` writes are
// visible to every caller that sees run() return cudaSuccess.
class PerDeviceOnce {
  public:
    template <class F>
    cudaError_t run(int dev, F &&fn) {
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        const cudaError_t e = fn();
        if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
        return e;
    }

  private:
    std::mutex mu_;
    std::atomic<bool> done_[kMaxDevices] = {};
};

// Each kernel translation unit keeps its own sticky device status word
// (PKV_STATUS_* bits).  These read (and optionally clear) it on `stream`.
cudaError_t store_status(cudaStream_t stream, uint32_t *host, bool clear);
cudaError_t decode_status(cudaStream_t stream, uint32_t *host, bool clear);
cudaError_t prefill_status(cudaStream_t stream, uint32_t *host, bool clear);

// ---- kv_store.cu ----------------------------------------------------------
cudaError_t launch_slot_mapping(const int32_t *bt, int64_t bt_stride, int32_t max_blocks,
                                const int32_t *start, const int32_t *cu_q, int32_t num_seqs,
                                int32_t block_size, int32_t *slots, int32_t num_tokens,
                                cudaStream_t stream);
cudaError_t launch_decode_slots(const int32_t *bt, int64_t bt_stride, int32_t max_blocks,
                                const int32_t *ctx, int32_t batch, int32_t block_size,
                                int32_t *slots, cudaStream_t stream);
cudaError_t launch_kv_store(const uint16_t *key, int64_t key_rs, const uint16_t *value,
                            int64_t value_rs, uint16_t *kc, uint16_t *vc, const int32_t *slots,
                            int32_t n, int64_t D, int64_t num_slots, cudaStream_t stream);

// Validate mode: flag PKV_STATUS_DUP_SLOT when two of the n tokens write the
// same slot.  The slots are slots[i] when `slots` is given, else the decode
// slot of row i (position ctx[i]-1 through the block table; none for ctx 0).
cudaError_t launch_check_duplicate_slots(const int32_t *slots, const int32_t *bt, int64_t bt_stride,
                                         int32_t max_blocks, const int32_t *ctx,
                                         int32_t block_size, int64_t num_blocks, int32_t n,
                                         cudaStream_t stream);

struct PrologueArgs {
    const uint16_t *q;
    int64_t q_rs;
    const uint16_t *k;
    int64_t k_rs;
    const uint16_t *v;
    int64_t v_rs;
    const int64_t *positions;
    const uint16_t *q_weight, *k_weight;
    float eps, theta;
    uint16_t *q_out;
    int64_t q_out_rs;
    uint16_t *k_out;
    int64_t k_out_rs;
    uint16_t *k_cache, *v_cache;
    const int32_t *slots;
    int64_t num_slots;
    int32_t num_tokens, num_heads, num_kv_heads, head_dim;
};
cudaError_t launch_qk_norm_rope_store(const PrologueArgs &a, cudaStream_t stream);

// ---- decode.cu ------------------------------------------------------------
struct DecodeArgs {
    const uint16_t *q;
    int64_t q_rs;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    int64_t num_blocks;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t max_blocks;
    const int32_t *ctx;
    int32_t batch, num_heads, num_kv_heads, head_dim, block_size, max_context_len;
    float scale;
    uint16_t *out;
    int64_t out_rs;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    // fused store of the step's new token (paged_attn_decode_store); null
    // new_k means the caches are only read
    const uint16_t *new_k, *new_v;
    int64_t new_k_rs, new_v_rs;
};
// keys per split chunk forced by pkv_set_decode_chunk_tiles (0: automatic)
extern std::atomic<int> g_decode_chunk_tiles;
// chunk of keys per split and number of splits for a decode launch
void decode_plan(int32_t batch, int32_t num_kv_heads, int32_t head_dim, int32_t max_context_len,
                 int32_t *chunk, int32_t *max_splits);
size_t decode_workspace_bytes(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_context_len);
// returns a PKV_* code; message in *err when not PKV_OK
int launch_decode(const DecodeArgs &a, cudaStream_t stream, const char **err);

// ---- prefill.cu -----------------------------------------------------------
struct PrefillArgs {
    const uint16_t *q;
    int64_t q_rs;
    const uint16_t *k;
    int64_t k_rs;
    const uint16_t *v;
    int64_t v_rs;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    int64_t num_blocks;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t max_blocks;
    const int32_t *cu_q;
    const int32_t *cu_k;
    int32_t max_seqlen_q, max_seqlen_k, num_seqs, total_q, total_k;
    int32_t num_heads, num_kv_heads, head_dim, block_size;
    float scale;
    uint16_t *out;
    int64_t out_rs;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
};
size_t prefill_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                               int32_t num_heads);
int launch_prefill(const PrefillArgs &a, cudaStream_t stream, const char **err);

// ---- tensor maps (api.cu) -------------------------------------------------
// Encodes a tiled map over a [rows, heads, head_dim] bf16 tensor with the given
// row / head strides (elements) and box (box_d, 1, box_rows).
int encode_rows_heads_map(CUtensorMap *map, const void *base, int64_t rows, int32_t heads,
                          int32_t head_dim, int64_t row_stride, int64_t head_stride,
                          int32_t box_d, int32_t box_rows, bool swizzle128, const char **err);

int num_sms();

// record an error for pkv_last_error() and return `code`
int report(int code, const char *fmt, ...);

}  // namespace pkv
