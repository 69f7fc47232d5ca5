// kv_store.cu -- the write side of the paged KV cache:
//   * slot_mapping for a prefill / chunked-prefill step (Lesson 04, §2),
//   * the decode slot of each sequence (Lesson 04, §9 item 1),
//   * store_kvcache, the slot-addressed scatter of new K/V rows
//     (L17: Qwen3 attention sub-layer, §5.1; Lesson 04, §3).
//
// The pages' write kernel runs one program per token and moves D elements
// with one vector load/store.  Here one WARP owns one token: the 32 lanes
// move the token's K row and V row as 16-byte vectors (D = 1024 bf16 = 2 KiB
// per row is 4 vectors per lane per tensor), all loads of a lane are issued
// before its stores so that each warp keeps 8 x 512 B in flight, and eight
// tokens share a 256-thread CTA.  The copy is HBM-bound: per live token it
// reads 2*D*2 bytes + 4 bytes of slot and writes 2*D*2 bytes.
#include "common.cuh"
#include "internal.h"

namespace pkv {

static __device__ unsigned int g_store_status;

__device__ __forceinline__ void flag(unsigned int bits) { atomicOr(&g_store_status, bits); }

cudaError_t store_status(cudaStream_t stream, uint32_t *host, bool clear) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_store_status, sizeof v, 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && clear && v) {
        unsigned int z = 0;
        e = cudaMemcpyToSymbolAsync(g_store_status, &z, sizeof z, 0, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    *host |= v;
    return e;
}

// ---------------------------------------------------------------------------
// slot_mapping: one CTA per sequence, threads stride over its new tokens.
// slot = table[i][p / bs] * bs + p % bs for logical position p = start + t.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) slot_mapping_kernel(
    const int32_t *__restrict__ bt, int64_t bt_stride, int32_t max_blocks,
    const int32_t *__restrict__ start, const int32_t *__restrict__ cu_q, int32_t block_size,
    int32_t *__restrict__ slots, int32_t num_tokens) {
    const int32_t i = blockIdx.x;
    const int32_t q0 = cu_q[i];
    const int32_t q1 = cu_q[i + 1];
    const int64_t s0 = start[i];
    if (q0 < 0 || q1 < q0 || q1 > num_tokens || s0 < 0) {
        if (threadIdx.x == 0) flag(PKV_STATUS_BAD_LENGTH);
        return;
    }
    const int32_t *row = bt + (int64_t)i * bt_stride;
    for (int32_t t = threadIdx.x; t < q1 - q0; t += blockDim.x) {
        const int64_t p = s0 + t;
        const int64_t lb = p / block_size;
        int32_t blk = lb < max_blocks ? row[lb] : -1;
        int32_t slot = -1;
        if (blk >= 0)
            slot = (int32_t)((int64_t)blk * block_size + p % block_size);
        else
            flag(PKV_STATUS_BAD_BLOCK);
        slots[q0 + t] = slot;
    }
}

// decode slot: one thread per row; context 0 (padding) -> -1
__global__ void __launch_bounds__(256) decode_slots_kernel(
    const int32_t *__restrict__ bt, int64_t bt_stride, int32_t max_blocks,
    const int32_t *__restrict__ ctx, int32_t batch, int32_t block_size,
    int32_t *__restrict__ slots) {
    const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int64_t c = ctx[b];
    int32_t slot = -1;
    if (c > 0) {
        const int64_t p = c - 1;
        const int64_t lb = p / block_size;
        const int32_t blk = lb < max_blocks ? bt[(int64_t)b * bt_stride + lb] : -1;
        if (blk >= 0)
            slot = (int32_t)((int64_t)blk * block_size + p % block_size);
        else
            flag(PKV_STATUS_BAD_BLOCK);
    } else if (c < 0) {
        flag(PKV_STATUS_BAD_LENGTH);
    }
    slots[b] = slot;
}

// ---------------------------------------------------------------------------
// kv_store, 16-byte vector path: a warp per token.
// D, both row strides and all four base pointers are multiples of 8 elements
// (16 bytes) -- checked on the host.
// ---------------------------------------------------------------------------
constexpr int kStoreWarps = 8;
constexpr int kStoreUnroll = 4;   // 16-byte vectors per lane per tensor per pass

__global__ void __launch_bounds__(kStoreWarps * 32) kv_store_v16_kernel(
    const uint16_t *__restrict__ key, int64_t key_rs, const uint16_t *__restrict__ value,
    int64_t value_rs, uint16_t *__restrict__ kc, uint16_t *__restrict__ vc,
    const int32_t *__restrict__ slots, int32_t n, int64_t D, int64_t num_slots) {
    const int32_t tok = blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= n) return;
    const int64_t slot = slots[tok];
    if (slot == -1) return;                     // padding token: leave the cache alone
    if (slot < 0 || slot >= num_slots) {
        if (lane == 0) flag(PKV_STATUS_BAD_SLOT);
        return;
    }
    const uint16_t *ksrc = key + (int64_t)tok * key_rs;
    const uint16_t *vsrc = value + (int64_t)tok * value_rs;
    uint16_t *kdst = kc + slot * D;
    uint16_t *vdst = vc + slot * D;
    constexpr int64_t kStep = 32 * 8;           // elements per warp-wide vector pass
    for (int64_t base = (int64_t)lane * 8; base < D; base += kStep * kStoreUnroll) {
        uint4 kr[kStoreUnroll], vr[kStoreUnroll];
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t e = base + u * kStep;
            if (e < D) {
                kr[u] = ld_stream_v4(ksrc + e);
                vr[u] = ld_stream_v4(vsrc + e);
            }
        }
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t e = base + u * kStep;
            if (e < D) {
                st_v4(kdst + e, kr[u]);
                st_v4(vdst + e, vr[u]);
            }
        }
    }
}

// element-wise path for shapes or alignments the vector path cannot take
__global__ void __launch_bounds__(kStoreWarps * 32) kv_store_scalar_kernel(
    const uint16_t *__restrict__ key, int64_t key_rs, const uint16_t *__restrict__ value,
    int64_t value_rs, uint16_t *__restrict__ kc, uint16_t *__restrict__ vc,
    const int32_t *__restrict__ slots, int32_t n, int64_t D, int64_t num_slots) {
    const int32_t tok = blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= n) return;
    const int64_t slot = slots[tok];
    if (slot == -1) return;
    if (slot < 0 || slot >= num_slots) {
        if (lane == 0) flag(PKV_STATUS_BAD_SLOT);
        return;
    }
    for (int64_t e = lane; e < D; e += 32) {
        kc[slot * D + e] = key[(int64_t)tok * key_rs + e];
        vc[slot * D + e] = value[(int64_t)tok * value_rs + e];
    }
}

cudaError_t launch_slot_mapping(const int32_t *bt, int64_t bt_stride, int32_t max_blocks,
                                const int32_t *start, const int32_t *cu_q, int32_t num_seqs,
                                int32_t block_size, int32_t *slots, int32_t num_tokens,
                                cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    slot_mapping_kernel<<<num_seqs, 256, 0, stream>>>(bt, bt_stride, max_blocks, start, cu_q,
                                                      block_size, slots, num_tokens);
    return cudaGetLastError();
}

cudaError_t launch_decode_slots(const int32_t *bt, int64_t bt_stride, int32_t max_blocks,
                                const int32_t *ctx, int32_t batch, int32_t block_size,
                                int32_t *slots, cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    decode_slots_kernel<<<(batch + 255) / 256, 256, 0, stream>>>(bt, bt_stride, max_blocks, ctx,
                                                                 batch, block_size, slots);
    return cudaGetLastError();
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaError_t launch_kv_store(const uint16_t *key, int64_t key_rs, const uint16_t *value,
                            int64_t value_rs, uint16_t *kc, uint16_t *vc, const int32_t *slots,
                            int32_t n, int64_t D, int64_t num_slots, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    const dim3 grid((n + kStoreWarps - 1) / kStoreWarps);
    const bool vec = D % 8 == 0 && key_rs % 8 == 0 && value_rs % 8 == 0 && aligned16(key) &&
                     aligned16(value) && aligned16(kc) && aligned16(vc);
    if (vec)
        kv_store_v16_kernel<<<grid, kStoreWarps * 32, 0, stream>>>(key, key_rs, value, value_rs,
                                                                  kc, vc, slots, n, D, num_slots);
    else
        kv_store_scalar_kernel<<<grid, kStoreWarps * 32, 0, stream>>>(
            key, key_rs, value, value_rs, kc, vc, slots, n, D, num_slots);
    return cudaGetLastError();
}

}  // namespace pkv
