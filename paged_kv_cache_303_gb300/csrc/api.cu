// api.cu -- the extern "C" boundary of libpagedkv (declared in
// include/pagedkv.h).  Host code only: it validates every argument before
// anything is launched, encodes TMA tensor maps, dispatches to the kernel
// translation units, and implements validate mode and the device status
// query.  No entry point allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "internal.h"

namespace {

thread_local char g_err[512];
std::atomic<int> g_validate{-1};   // -1: not read from the environment yet

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return PKV_OK;
}

bool validate_on() {
    int v = g_validate.load(std::memory_order_relaxed);
    if (v < 0) {
        const char *e = getenv("PKV_VALIDATE");
        int expected = -1;
        // an explicit pkv_set_validate() wins over the environment
        g_validate.compare_exchange_strong(expected, (e && e[0] == '1') ? 1 : 0);
        v = g_validate.load(std::memory_order_relaxed);
    }
    return v == 1;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_fail(cudaError_t e, const char *what) {
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// validate mode: synchronise and turn device status bits into an error code
int post_launch(cudaStream_t stream, const char *what) {
    if (!validate_on()) return ok();
    uint32_t st = 0;
    cudaError_t e = pkv::store_status(stream, &st, true);
    if (e == cudaSuccess) e = pkv::decode_status(stream, &st, true);
    if (e == cudaSuccess) e = pkv::prefill_status(stream, &st, true);
    if (e != cudaSuccess) return cuda_fail(e, what);
    if (st & PKV_STATUS_TIMEOUT)
        return fail(PKV_ERR_DEVICE_TIMEOUT, "%s: a bounded device wait expired (status 0x%x)", what, st);
    if (st)
        return fail(PKV_ERR_DEVICE_CHECK, "%s: device flagged invalid data (status 0x%x)", what, st);
    return ok();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn(const char **err) {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!fn) *err = "cuTensorMapEncodeTiled is not available from the driver";
    return fn;
}

}  // namespace

namespace pkv {

int report(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int num_sms() {
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int encode_rows_heads_map(CUtensorMap *map, const void *base, int64_t rows, int32_t heads,
                          int32_t head_dim, int64_t row_stride, int64_t head_stride,
                          int32_t box_d, int32_t box_rows, bool swizzle128, const char **err) {
    EncodeTiledFn fn = encode_fn(err);
    if (!fn) return PKV_ERR_CUDA;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_stride * 2, (cuuint64_t)row_stride * 2};
    const cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *err = "cuTensorMapEncodeTiled rejected the tensor (alignment or size)";
        return PKV_ERR_INVALID_ARG;
    }
    return PKV_OK;
}

}  // namespace pkv

extern "C" {

const char *pkv_last_error(void) { return g_err; }

int pkv_version(void) { return 1; }

void pkv_set_validate(int on) { g_validate.store(on ? 1 : 0, std::memory_order_relaxed); }

int pkv_set_decode_chunk_tiles(int tiles) {
    if (tiles < 0 || tiles > 4096)
        return fail(PKV_ERR_INVALID_ARG, "pkv_set_decode_chunk_tiles: tiles must be in [0, 4096]");
    pkv::g_decode_chunk_tiles.store(tiles, std::memory_order_relaxed);
    return ok();
}

int pkv_device_status(pkv_stream_t stream, uint32_t *status, int clear) {
    if (!status) return fail(PKV_ERR_INVALID_ARG, "pkv_device_status: status is NULL");
    *status = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::store_status(s, status, clear != 0);
    if (e == cudaSuccess) e = pkv::decode_status(s, status, clear != 0);
    if (e == cudaSuccess) e = pkv::prefill_status(s, status, clear != 0);
    if (e != cudaSuccess) return cuda_fail(e, "pkv_device_status");
    return ok();
}

int kv_build_slot_mapping(const int32_t *block_tables, int64_t bt_stride,
                          int32_t max_blocks_per_seq, const int32_t *start,
                          const int32_t *cu_seqlens_q, int32_t num_seqs, int32_t block_size,
                          int32_t *slot_mapping, int32_t num_tokens, pkv_stream_t stream) {
    if (num_seqs < 0 || num_tokens < 0 || block_size <= 0 || max_blocks_per_seq < 0 ||
        bt_stride < max_blocks_per_seq)
        return fail(PKV_ERR_INVALID_ARG,
                    "kv_build_slot_mapping: need num_seqs, num_tokens >= 0, block_size > 0, "
                    "0 <= max_blocks_per_seq <= bt_stride");
    if (num_seqs > 0 && (!start || !cu_seqlens_q || (max_blocks_per_seq > 0 && !block_tables)))
        return fail(PKV_ERR_INVALID_ARG, "kv_build_slot_mapping: null pointer");
    if (num_tokens > 0 && !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "kv_build_slot_mapping: slot_mapping is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::launch_slot_mapping(block_tables, bt_stride, max_blocks_per_seq, start,
                                             cu_seqlens_q, num_seqs, block_size, slot_mapping,
                                             num_tokens, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_build_slot_mapping");
    return post_launch(s, "kv_build_slot_mapping");
}

int kv_build_decode_slots(const int32_t *block_tables, int64_t bt_stride,
                          int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                          int32_t block_size, int32_t *slot_mapping, pkv_stream_t stream) {
    if (batch < 0 || block_size <= 0 || max_blocks_per_seq < 0 || bt_stride < max_blocks_per_seq)
        return fail(PKV_ERR_INVALID_ARG,
                    "kv_build_decode_slots: need batch >= 0, block_size > 0, "
                    "0 <= max_blocks_per_seq <= bt_stride");
    if (batch > 0 && (!context_lens || !slot_mapping || (max_blocks_per_seq > 0 && !block_tables)))
        return fail(PKV_ERR_INVALID_ARG, "kv_build_decode_slots: null pointer");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::launch_decode_slots(block_tables, bt_stride, max_blocks_per_seq,
                                             context_lens, batch, block_size, slot_mapping, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_build_decode_slots");
    return post_launch(s, "kv_build_decode_slots");
}

int kv_store(const pkv_bf16 *key, int64_t key_row_stride, const pkv_bf16 *value,
             int64_t value_row_stride, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
             const int32_t *slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
             int32_t head_dim, int64_t num_slots, pkv_stream_t stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_slots < 0)
        return fail(PKV_ERR_INVALID_ARG,
                    "kv_store: need num_tokens >= 0, num_kv_heads > 0, head_dim > 0, num_slots >= 0");
    const int64_t D = (int64_t)num_kv_heads * head_dim;
    if (num_tokens > 0) {
        if (!key || !value || !k_cache || !v_cache || !slot_mapping)
            return fail(PKV_ERR_INVALID_ARG, "kv_store: null pointer");
        if (key_row_stride < D || value_row_stride < D)
            return fail(PKV_ERR_INVALID_ARG,
                        "kv_store: row strides (%lld, %lld) must be >= num_kv_heads*head_dim (%lld)",
                        (long long)key_row_stride, (long long)value_row_stride, (long long)D);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::launch_kv_store(key, key_row_stride, value, value_row_stride, k_cache,
                                         v_cache, slot_mapping, num_tokens, D, num_slots, s);
    if (e == cudaSuccess && validate_on())
        e = pkv::launch_check_duplicate_slots(slot_mapping, nullptr, 0, 0, nullptr, 1, 0, num_tokens, s);
    if (e != cudaSuccess) return cuda_fail(e, "kv_store");
    return post_launch(s, "kv_store");
}

int qk_norm_rope_store(const pkv_bf16 *q, int64_t q_row_stride, const pkv_bf16 *k,
                       int64_t k_row_stride, const pkv_bf16 *v, int64_t v_row_stride,
                       const int64_t *positions, const pkv_bf16 *q_norm_weight,
                       const pkv_bf16 *k_norm_weight, float rms_eps, float rope_theta,
                       pkv_bf16 *q_out, int64_t q_out_row_stride, pkv_bf16 *k_out,
                       int64_t k_out_row_stride, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                       const int32_t *slot_mapping, int32_t num_tokens, int32_t num_heads,
                       int32_t num_kv_heads, int32_t head_dim, int64_t num_slots,
                       pkv_stream_t stream) {
    const char *what = "qk_norm_rope_store";
    if (num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_slots < 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: negative or zero sizes", what);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128", what);
    if (!(rms_eps >= 0.f) || !(rope_theta > 0.f) || !(rope_theta < HUGE_VALF))
        return fail(PKV_ERR_INVALID_ARG, "%s: need rms_eps >= 0 and a finite rope_theta > 0", what);
    if (num_tokens == 0) return ok();
    if (!q || !k || !v || !positions || !q_norm_weight || !k_norm_weight || !q_out || !k_cache ||
        !v_cache || !slot_mapping)
        return fail(PKV_ERR_INVALID_ARG, "%s: null pointer", what);
    const int64_t qrow = (int64_t)num_heads * head_dim, kvrow = (int64_t)num_kv_heads * head_dim;
    if (q_row_stride < qrow || q_out_row_stride < qrow || k_row_stride < kvrow ||
        v_row_stride < kvrow || (k_out && k_out_row_stride < kvrow))
        return fail(PKV_ERR_INVALID_ARG, "%s: a row stride is below heads*head_dim", what);
    if (q_row_stride % 8 || q_out_row_stride % 8 || k_row_stride % 8 || v_row_stride % 8 ||
        (k_out && k_out_row_stride % 8) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
        !aligned16(q_out) || (k_out && !aligned16(k_out)) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(q_norm_weight) || !aligned16(k_norm_weight))
        return fail(PKV_ERR_UNSUPPORTED,
                    "%s: tensors must be 16-byte aligned with row strides a multiple of 8", what);
    if ((q_out == q && q_out_row_stride != q_row_stride) ||
        (k_out && k_out == k && k_out_row_stride != k_row_stride))
        return fail(PKV_ERR_INVALID_ARG, "%s: an in-place output must keep its input's row stride",
                    what);
    pkv::PrologueArgs a{};
    a.q = q;
    a.q_rs = q_row_stride;
    a.k = k;
    a.k_rs = k_row_stride;
    a.v = v;
    a.v_rs = v_row_stride;
    a.positions = positions;
    a.q_weight = q_norm_weight;
    a.k_weight = k_norm_weight;
    a.eps = rms_eps;
    a.theta = rope_theta;
    a.q_out = q_out;
    a.q_out_rs = q_out_row_stride;
    a.k_out = k_out;
    a.k_out_rs = k_out_row_stride;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.slots = slot_mapping;
    a.num_slots = num_slots;
    a.num_tokens = num_tokens;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::launch_qk_norm_rope_store(a, s);
    if (e == cudaSuccess && validate_on())
        e = pkv::launch_check_duplicate_slots(slot_mapping, nullptr, 0, 0, nullptr, 1, 0, num_tokens, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return post_launch(s, what);
}

size_t paged_attn_decode_workspace_size(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t max_context_len) {
    if (batch <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len <= 0)
        return 0;
    return pkv::decode_workspace_bytes(batch, num_heads, num_kv_heads, head_dim, max_context_len);
}

static int check_heads(const char *what, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size) {
    if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: head counts, head_dim and block_size must be > 0", what);
    if (num_heads % num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: num_heads %% num_kv_heads != 0", what);
    if (head_dim != 64 && head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "%s: head_dim must be 64 or 128", what);
    return PKV_OK;
}

}  // extern "C"

// shared by paged_attn_decode and paged_attn_decode_store (key == NULL: the
// caches are only read)
static int decode_entry(const char *what, const pkv_bf16 *q, int64_t q_row_stride,
                        const pkv_bf16 *key, int64_t key_row_stride, const pkv_bf16 *value,
                        int64_t value_row_stride, const pkv_bf16 *k_cache,
                        const pkv_bf16 *v_cache, int64_t num_blocks, const int32_t *block_tables,
                        int64_t bt_stride, int32_t max_blocks_per_seq,
                        const int32_t *context_lens, int32_t batch, int32_t num_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                        int32_t max_context_len, float softmax_scale, pkv_bf16 *out,
                        int64_t out_row_stride, float *lse, void *workspace,
                        size_t workspace_bytes, pkv_stream_t stream) {
    if (int rc = check_heads(what, num_heads, num_kv_heads, head_dim, block_size)) return rc;
    if (batch < 0 || max_context_len < 0 || num_blocks < 0 || max_blocks_per_seq < 0 ||
        bt_stride < max_blocks_per_seq)
        return fail(PKV_ERR_INVALID_ARG, "%s: negative size or bt_stride < max_blocks_per_seq", what);
    if (batch == 0) return ok();
    if (block_size & (block_size - 1))
        return fail(PKV_ERR_UNSUPPORTED, "%s: block_size must be a power of two", what);
    const int G = num_heads / num_kv_heads;
    if (G < 1)
        return fail(PKV_ERR_INVALID_ARG, "%s: num_heads / num_kv_heads must be at least 1", what);
    if (!q || !k_cache || !v_cache || !context_lens || !out || (max_blocks_per_seq > 0 && !block_tables))
        return fail(PKV_ERR_INVALID_ARG, "%s: null pointer", what);
    const int64_t row = (int64_t)num_heads * head_dim;
    if (q_row_stride < row || out_row_stride < row)
        return fail(PKV_ERR_INVALID_ARG, "%s: q/out row stride below num_heads*head_dim", what);
    if (q_row_stride % 8 || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        out_row_stride % 2 || (reinterpret_cast<uintptr_t>(out) & 3u))
        return fail(PKV_ERR_UNSUPPORTED,
                    "%s: q rows and caches must be 16-byte aligned (row stride multiple of 8), "
                    "out 4-byte aligned with an even row stride", what);
    if ((int64_t)max_blocks_per_seq * block_size < max_context_len)
        return fail(PKV_ERR_INVALID_ARG, "%s: max_context_len %d exceeds the block table capacity",
                    what, max_context_len);
    if (num_blocks * block_size > INT32_MAX)
        return fail(PKV_ERR_UNSUPPORTED, "%s: more than 2^31 slots per cache", what);
    if (key || value) {
        const int64_t kv_row = (int64_t)num_kv_heads * head_dim;
        if (!key || !value)
            return fail(PKV_ERR_INVALID_ARG, "%s: null key or value", what);
        if (key_row_stride < kv_row || value_row_stride < kv_row)
            return fail(PKV_ERR_INVALID_ARG,
                        "%s: key/value row strides below num_kv_heads*head_dim", what);
        if (key_row_stride % 8 || value_row_stride % 8 || !aligned16(key) || !aligned16(value))
            return fail(PKV_ERR_UNSUPPORTED,
                        "%s: key/value must be 16-byte aligned with row strides a multiple of 8",
                        what);
    }
    pkv::DecodeArgs a{};
    a.q = q;
    a.q_rs = q_row_stride;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_blocks = num_blocks;
    a.bt = block_tables;
    a.bt_stride = bt_stride;
    a.max_blocks = max_blocks_per_seq;
    a.ctx = context_lens;
    a.batch = batch;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.max_context_len = max_context_len;
    a.scale = softmax_scale;
    a.out = out;
    a.out_rs = out_row_stride;
    a.lse = lse;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.new_k = key;
    a.new_v = value;
    a.new_k_rs = key_row_stride;
    a.new_v_rs = value_row_stride;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const char *err = "";
    int rc = pkv::launch_decode(a, s, &err);
    if (rc) return fail(rc, "%s: %s", what, err);
    if (key && validate_on()) {
        cudaError_t e = pkv::launch_check_duplicate_slots(nullptr, block_tables, bt_stride,
                                                          max_blocks_per_seq, context_lens,
                                                          block_size, num_blocks, batch, s);
        if (e != cudaSuccess) return cuda_fail(e, what);
    }
    return post_launch(s, what);
}

extern "C" {

int paged_attn_decode(const pkv_bf16 *q, int64_t q_row_stride, const pkv_bf16 *k_cache,
                      const pkv_bf16 *v_cache, int64_t num_blocks, const int32_t *block_tables,
                      int64_t bt_stride, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      int32_t batch, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_context_len, float softmax_scale,
                      pkv_bf16 *out, int64_t out_row_stride, float *lse, void *workspace,
                      size_t workspace_bytes, pkv_stream_t stream) {
    return decode_entry("paged_attn_decode", q, q_row_stride, nullptr, 0, nullptr, 0, k_cache,
                        v_cache, num_blocks, block_tables, bt_stride, max_blocks_per_seq,
                        context_lens, batch, num_heads, num_kv_heads, head_dim, block_size,
                        max_context_len, softmax_scale, out, out_row_stride, lse, workspace,
                        workspace_bytes, stream);
}

int paged_attn_decode_store(const pkv_bf16 *q, int64_t q_row_stride, const pkv_bf16 *key,
                            int64_t key_row_stride, const pkv_bf16 *value,
                            int64_t value_row_stride, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                            int64_t num_blocks, const int32_t *block_tables, int64_t bt_stride,
                            int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t batch,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t max_context_len, float softmax_scale,
                            pkv_bf16 *out, int64_t out_row_stride, float *lse, void *workspace,
                            size_t workspace_bytes, pkv_stream_t stream) {
    if (batch > 0 && (!key || !value))
        return fail(PKV_ERR_INVALID_ARG, "paged_attn_decode_store: null key or value");
    return decode_entry("paged_attn_decode_store", q, q_row_stride, key, key_row_stride, value,
                        value_row_stride, k_cache, v_cache, num_blocks, block_tables, bt_stride,
                        max_blocks_per_seq, context_lens, batch, num_heads, num_kv_heads, head_dim,
                        block_size, max_context_len, softmax_scale, out, out_row_stride, lse,
                        workspace, workspace_bytes, stream);
}

size_t paged_attn_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                                         int32_t num_heads) {
    if (num_seqs <= 0 || total_q <= 0 || num_heads <= 0) return 0;
    return pkv::prefill_workspace_bytes(num_seqs, total_q, max_seqlen_q, num_heads);
}

int paged_attn_prefill(const pkv_bf16 *q, int64_t q_row_stride, const pkv_bf16 *k,
                       int64_t k_row_stride, const pkv_bf16 *v, int64_t v_row_stride,
                       const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, int64_t num_blocks,
                       const int32_t *block_tables, int64_t bt_stride, int32_t max_blocks_per_seq,
                       const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, int32_t num_seqs,
                       int32_t total_q, int32_t total_k, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, float softmax_scale, pkv_bf16 *out,
                       int64_t out_row_stride, float *lse, void *workspace,
                       size_t workspace_bytes, pkv_stream_t stream) {
    const char *what = "paged_attn_prefill";
    const bool paged = block_tables != nullptr;
    if (int rc = check_heads(what, num_heads, num_kv_heads, head_dim, paged ? block_size : 1)) return rc;
    if (num_seqs < 0 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
        return fail(PKV_ERR_INVALID_ARG, "%s: negative size", what);
    if (num_seqs == 0 || total_q == 0) return ok();
    if (!q || !cu_seqlens_q || !cu_seqlens_k || !out)
        return fail(PKV_ERR_INVALID_ARG, "%s: null pointer", what);
    const int64_t qrow = (int64_t)num_heads * head_dim;
    const int64_t kvrow = (int64_t)num_kv_heads * head_dim;
    if (q_row_stride < qrow || out_row_stride < qrow)
        return fail(PKV_ERR_INVALID_ARG, "%s: q/out row stride below num_heads*head_dim", what);
    if (q_row_stride % 8 || out_row_stride % 8 || !aligned16(q) || !aligned16(out))
        return fail(PKV_ERR_UNSUPPORTED, "%s: q/out must be 16-byte aligned with row strides "
                                         "that are multiples of 8", what);
    if (paged) {
        if (!k_cache || !v_cache || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
            bt_stride < max_blocks_per_seq)
            return fail(PKV_ERR_INVALID_ARG, "%s: paged mode needs caches and a block table", what);
        if (!aligned16(k_cache) || !aligned16(v_cache))
            return fail(PKV_ERR_UNSUPPORTED, "%s: caches must be 16-byte aligned", what);
        if ((int64_t)max_blocks_per_seq * block_size < max_seqlen_k)
            return fail(PKV_ERR_INVALID_ARG, "%s: max_seqlen_k exceeds the block table capacity", what);
        if (num_blocks * block_size > INT32_MAX)
            return fail(PKV_ERR_UNSUPPORTED, "%s: more than 2^31 slots per cache", what);
    } else {
        if (!k || !v || total_k <= 0)
            return fail(PKV_ERR_INVALID_ARG, "%s: packed mode needs k and v", what);
        if (k_row_stride < kvrow || v_row_stride < kvrow)
            return fail(PKV_ERR_INVALID_ARG, "%s: k/v row stride below num_kv_heads*head_dim", what);
        if (k_row_stride % 8 || v_row_stride % 8 || !aligned16(k) || !aligned16(v))
            return fail(PKV_ERR_UNSUPPORTED, "%s: k/v must be 16-byte aligned with row strides "
                                             "that are multiples of 8", what);
    }
    pkv::PrefillArgs a{};
    a.q = q;
    a.q_rs = q_row_stride;
    a.k = k;
    a.k_rs = k_row_stride;
    a.v = v;
    a.v_rs = v_row_stride;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_blocks = num_blocks;
    a.bt = block_tables;
    a.bt_stride = bt_stride;
    a.max_blocks = max_blocks_per_seq;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.total_k = total_k;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.scale = softmax_scale;
    a.out = out;
    a.out_rs = out_row_stride;
    a.lse = lse;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const char *err = "";
    int rc = pkv::launch_prefill(a, s, &err);
    if (rc) return fail(rc, "%s: %s", what, err);
    return post_launch(s, what);
}

}  // extern "C"

#if PKV_TEST_HOOKS
// Only in the test-only build (never in libpagedkv.so): see decode.cu and
// prefill.cu.
namespace pkv {
int test_withhold_decode_ready(int on);
int test_withhold_prefill_unit(int on);
}
extern "C" int pkv_test_withhold_decode_ready(int on) { return pkv::test_withhold_decode_ready(on); }
extern "C" int pkv_test_withhold_prefill_unit(int on) { return pkv::test_withhold_prefill_unit(on); }
#endif
