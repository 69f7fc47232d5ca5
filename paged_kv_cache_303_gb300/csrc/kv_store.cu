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
//
// qk_norm_rope_store_kernel fuses the two steps that precede the store in
// the attention sub-layer (L17, §4: QK-Norm, then RoPE on q and k; v as is)
// with the store itself: one pass over the projected q/k/v rows writes the
// rotated q, the rotated k (optionally back to the caller) and the k/v
// cache rows.
#include <math.h>

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

// ---------------------------------------------------------------------------
// QK-Norm + RoPE + store.
//
// RMSNorm as the layernorm module of "Nano-VLLM full-code notes (5)" does
// it: x / sqrt(mean(x^2) + eps) in fp32, rounded to bf16, then the bf16
// product with the weight (rounded to bf16).  RoPE (RoFormer, rotate-half
// pairing): element e < d/2 pairs with e + d/2 and pair i turns by
// pos * theta^(-2i/d); the rotation is computed in fp32 from the bf16 norm
// output and rounded to bf16 once.
//
// A warp owns a token: a row of head_dim bf16 is HD/8 lanes x 16 bytes, so a
// warp-wide vector load covers 32/(HD/8) rows and all of the token's
// Hq + 2*Hkv rows take a few passes of kProUnroll loads per lane, issued
// before any arithmetic.  Each lane holds the same 8 element positions of
// every row, so it computes the 8 (cos, sin) pairs of those positions once
// per token; the RMS sum is reduced over the row's lanes and the rotation
// partner (element e +- d/2) is HD/16 lanes away (one xor shuffle).
// The angle pos * f_i is formed as pos * f_hi + (error of that product +
// pos * f_lo) with f_hi + f_lo = theta^(-2i/d) computed on the host in
// double, so the angle carries no fp32 rounding of f_i or of the product;
// sincosf of the rounded part is then corrected to first order by the rest.
// HBM-bound: per token it reads (Hq + 2*Hkv) * d * 2 bytes and writes
// (Hq + 2*Hkv) * d * 2 bytes (+ Hkv * d * 2 when k is also written back).
// ---------------------------------------------------------------------------
constexpr int kProWarps = 8;
constexpr int kProUnroll = 4;

struct PrologueParams {
    const uint16_t *q;
    int64_t q_rs;
    const uint16_t *k;
    int64_t k_rs;
    const uint16_t *v;
    int64_t v_rs;
    const int64_t *pos;
    const uint16_t *qw, *kw;
    float eps;
    uint16_t *q_out;
    int64_t q_out_rs;
    uint16_t *k_out;             // null: rotated k only goes to the cache
    int64_t k_out_rs;
    uint16_t *kc, *vc;
    const int32_t *slots;
    int64_t num_slots;
    int32_t n, hq, hkv;
    float inv_hi[64], inv_lo[64];
};

__device__ __forceinline__ float round_bf16(float x) {
    return bf16lo_to_f32(pack_bf16x2(x, 0.f));
}

template <int HD>
__global__ void __launch_bounds__(kProWarps * 32)
qk_norm_rope_store_kernel(const __grid_constant__ PrologueParams p) {
    constexpr int LPR = HD / 8;                 // lanes per row
    constexpr int RPW = 32 / LPR;               // rows per warp-wide pass
    constexpr int HALF = HD / 2;
    const int lane = threadIdx.x & 31;
    const int sub = lane / LPR;
    const int e0 = (lane % LPR) * 8;            // this lane's elements e0 .. e0+7
    const bool first = e0 < HALF;
    const int i0 = e0 % HALF;                   // and their pair indices

    float wq[8], wk[8];
    {
        const uint4 a = *reinterpret_cast<const uint4 *>(p.qw + e0);
        const uint4 b = *reinterpret_cast<const uint4 *>(p.kw + e0);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            wq[2 * j] = bf16lo_to_f32(av[j]);
            wq[2 * j + 1] = bf16hi_to_f32(av[j]);
            wk[2 * j] = bf16lo_to_f32(bv[j]);
            wk[2 * j + 1] = bf16hi_to_f32(bv[j]);
        }
    }
    const int rows = p.hq + 2 * p.hkv;
    const int64_t D = (int64_t)p.hkv * HD;

    for (int64_t t = (int64_t)blockIdx.x * kProWarps + (threadIdx.x >> 5); t < p.n;
         t += (int64_t)gridDim.x * kProWarps) {
        const float pos = (float)p.pos[t];      // exact for positions below 2^24
        float cs[8], sn[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float fh = p.inv_hi[i0 + j], fl = p.inv_lo[i0 + j];
            const float ah = pos * fh;
            const float al = fmaf(pos, fl, fmaf(pos, fh, -ah));
            float s0, c0;
            sincosf(ah, &s0, &c0);
            sn[j] = fmaf(al, c0, s0);
            cs[j] = fmaf(-al, s0, c0);
        }
        const int64_t slot = p.slots[t];
        const bool store = slot >= 0 && slot < p.num_slots;
        if (lane == 0 && !store && slot != -1) flag(PKV_STATUS_BAD_SLOT);

        for (int r0 = 0; r0 < rows; r0 += RPW * kProUnroll) {
            uint4 x[kProUnroll];
#pragma unroll
            for (int u = 0; u < kProUnroll; ++u) {
                const int r = r0 + u * RPW + sub;
                const uint16_t *src = nullptr;
                if (r < p.hq)
                    src = p.q + t * p.q_rs + (int64_t)r * HD;
                else if (r < p.hq + p.hkv)
                    src = p.k + t * p.k_rs + (int64_t)(r - p.hq) * HD;
                else if (r < rows)
                    src = p.v + t * p.v_rs + (int64_t)(r - p.hq - p.hkv) * HD;
                x[u] = src ? ld_stream_v4(src + e0) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kProUnroll; ++u) {
                const int r = r0 + u * RPW + sub;
                const bool is_q = r < p.hq;
                const bool is_k = !is_q && r < p.hq + p.hkv;
                const uint32_t xv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                float xf[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    xf[2 * j] = bf16lo_to_f32(xv[j]);
                    xf[2 * j + 1] = bf16hi_to_f32(xv[j]);
                }
                // every lane takes part in the shuffles, whatever its row is
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) ss = fmaf(xf[j], xf[j], ss);
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float inv = rsqrtf(ss * (1.f / HD) + p.eps);
                uint32_t yp[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float w0 = is_q ? wq[2 * j] : wk[2 * j];
                    const float w1 = is_q ? wq[2 * j + 1] : wk[2 * j + 1];
                    yp[j] = pack_bf16x2(round_bf16(xf[2 * j] * inv) * w0,
                                        round_bf16(xf[2 * j + 1] * inv) * w1);
                }
                uint32_t pp[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) pp[j] = __shfl_xor_sync(0xffffffffu, yp[j], LPR / 2);
                uint32_t ov[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float y0 = bf16lo_to_f32(yp[j]), y1 = bf16hi_to_f32(yp[j]);
                    const float q0 = bf16lo_to_f32(pp[j]), q1 = bf16hi_to_f32(pp[j]);
                    // first half: y cos - partner sin; second half: y cos + partner sin
                    const float s0 = first ? -sn[2 * j] : sn[2 * j];
                    const float s1 = first ? -sn[2 * j + 1] : sn[2 * j + 1];
                    ov[j] = pack_bf16x2(fmaf(q0, s0, y0 * cs[2 * j]), fmaf(q1, s1, y1 * cs[2 * j + 1]));
                }
                const uint4 o = make_uint4(ov[0], ov[1], ov[2], ov[3]);
                if (is_q) {
                    st_v4(p.q_out + t * p.q_out_rs + (int64_t)r * HD + e0, o);
                } else if (is_k) {
                    const int h = r - p.hq;
                    if (p.k_out) st_v4(p.k_out + t * p.k_out_rs + (int64_t)h * HD + e0, o);
                    if (store) st_v4(p.kc + slot * D + (int64_t)h * HD + e0, o);
                } else if (r < rows && store) {
                    st_v4(p.vc + slot * D + (int64_t)(r - p.hq - p.hkv) * HD + e0, x[u]);
                }
            }
        }
    }
}

cudaError_t launch_qk_norm_rope_store(const PrologueArgs &a, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    PrologueParams p{};
    p.q = a.q;
    p.q_rs = a.q_rs;
    p.k = a.k;
    p.k_rs = a.k_rs;
    p.v = a.v;
    p.v_rs = a.v_rs;
    p.pos = a.positions;
    p.qw = a.q_weight;
    p.kw = a.k_weight;
    p.eps = a.eps;
    p.q_out = a.q_out;
    p.q_out_rs = a.q_out_rs;
    p.k_out = a.k_out;
    p.k_out_rs = a.k_out_rs;
    p.kc = a.k_cache;
    p.vc = a.v_cache;
    p.slots = a.slots;
    p.num_slots = a.num_slots;
    p.n = a.num_tokens;
    p.hq = a.num_heads;
    p.hkv = a.num_kv_heads;
    const int half = a.head_dim / 2;
    for (int i = 0; i < half; ++i) {
        const double f = pow((double)a.theta, -2.0 * i / a.head_dim);
        p.inv_hi[i] = (float)f;
        p.inv_lo[i] = (float)(f - (double)p.inv_hi[i]);
    }
    const dim3 grid((a.num_tokens + kProWarps - 1) / kProWarps);
    if (a.head_dim == 128)
        qk_norm_rope_store_kernel<128><<<grid, kProWarps * 32, 0, stream>>>(p);
    else
        qk_norm_rope_store_kernel<64><<<grid, kProWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
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
