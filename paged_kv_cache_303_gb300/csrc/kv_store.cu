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
#ifndef PKV_STORE_CS
#define PKV_STORE_CS 1            // cache rows written with the streaming hint
#endif
#ifndef PKV_STORE_EARLY
#define PKV_STORE_EARLY 1         // row loads issued before the slot is known
#endif
#ifndef PKV_STORE_WARPS
#define PKV_STORE_WARPS 8         // tokens (warps) per CTA
#endif
constexpr int kStoreWarps = PKV_STORE_WARPS;
constexpr int kStoreUnroll = 4;   // 16-byte vectors per lane per tensor per pass

__global__ void __launch_bounds__(kStoreWarps * 32) kv_store_v16_kernel(
    const uint16_t *__restrict__ key, int64_t key_rs, const uint16_t *__restrict__ value,
    int64_t value_rs, uint16_t *__restrict__ kc, uint16_t *__restrict__ vc,
    const int32_t *__restrict__ slots, int32_t n, int64_t D, int64_t num_slots) {
    const int32_t tok = blockIdx.x * kStoreWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (tok >= n) return;
    const uint16_t *ksrc = key + (int64_t)tok * key_rs;
    const uint16_t *vsrc = value + (int64_t)tok * value_rs;
    constexpr int64_t kStep = 32 * 8;           // elements per warp-wide vector pass
    // The first pass's row loads go out together with the slot load (they do
    // not depend on it), so a token costs one memory round trip, not two.
    uint4 kr[kStoreUnroll], vr[kStoreUnroll];
    auto load_pass = [&](int64_t base) {
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t e = base + u * kStep;
            if (e < D) {
                kr[u] = ld_stream_v4(ksrc + e);
                vr[u] = ld_stream_v4(vsrc + e);
            }
        }
    };
    if (PKV_STORE_EARLY) load_pass((int64_t)lane * 8);
    const int64_t slot = slots[tok];
    if (slot == -1) return;                     // padding token: leave the cache alone
    if (slot < 0 || slot >= num_slots) {
        if (lane == 0) flag(PKV_STATUS_BAD_SLOT);
        return;
    }
    uint16_t *kdst = kc + slot * D;
    uint16_t *vdst = vc + slot * D;
    for (int64_t base = (int64_t)lane * 8; base < D; base += kStep * kStoreUnroll) {
        if (!PKV_STORE_EARLY || base != (int64_t)lane * 8) load_pass(base);
#pragma unroll
        for (int u = 0; u < kStoreUnroll; ++u) {
            const int64_t e = base + u * kStep;
            if (e < D) {
                if (PKV_STORE_CS) {
                    st_cs_v4(kdst + e, kr[u]);
                    st_cs_v4(vdst + e, vr[u]);
                } else {
                    st_v4(kdst + e, kr[u]);
                    st_v4(vdst + e, vr[u]);
                }
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
// product with the weight (rounded to bf16).  RoPE (applied by L17 §4 but
// not printed there; read as the split-halves "rotate-half" pairing of the
// engine's model family, not RoFormer's adjacent pairs): element e < d/2
// pairs with e + d/2 and pair i turns by
// pos * theta^(-2i/d); the rotation is computed in fp32 from the bf16 norm
// output and rounded to bf16 once.
//
// Lane layout: a lane holds 8 elements e .. e+7 of the first half of a row
// and their rotation partners e+d/2 .. (two 16-byte pieces), so a row is
// d/16 lanes, the RMS sum is reduced over d/16 lanes by xor shuffles, and
// the rotation needs no exchange between lanes.
// Work unit: one warp takes kProUnroll warp-wide passes of one token's rows
// (a pass covers 32/(d/16) rows): 12 rows at head_dim 128, so a Qwen3 token
// (16 q + 8 k + 8 v rows) is three units.  One resident wave of CTAs; each
// warp walks its units with kProStages of them in flight: their rows are
// copied into the warp's shared-memory stages by cp.async, so the loads
// hold no registers while a unit is computed.
// The unit's (cos, sin) of the d/2 pair angles are computed two per lane
// and handed to the lanes that need them by shuffles.  The angle pos * f_i
// is formed as pos * f_hi + (error of that product + pos * f_lo) with
// f_hi + f_lo = theta^(-2i/d) computed on the host in double, so the angle
// carries no fp32 rounding of f_i or of the product; it is reduced by 2*pi
// (Cody and Waite) and finished by the hardware sine / cosine.  Value rows
// are copied as they are.
// HBM-bound: per token it reads (Hq + 2*Hkv) * d * 2 bytes and writes
// (Hq + 2*Hkv) * d * 2 bytes (+ Hkv * d * 2 when k is also written back).
// ---------------------------------------------------------------------------
#ifndef PKV_PRO_UNROLL
#define PKV_PRO_UNROLL 3      // warp-wide passes per work unit
#endif
#ifndef PKV_PRO_MIN_CTAS
#define PKV_PRO_MIN_CTAS 2
#endif
#ifndef PKV_PRO_STAGES
#define PKV_PRO_STAGES 2      // units in flight per warp
#endif
#ifndef PKV_PRO_WARPS
#define PKV_PRO_WARPS 8       // warps per CTA
#endif
constexpr int kProWarps = PKV_PRO_WARPS;
constexpr int kProUnroll = PKV_PRO_UNROLL;

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
    int32_t chunks;              // units per token
    float inv_hi[64], inv_lo[64];
};

// bf16 x bf16 -> bf16 for a packed pair (the exact product, rounded once)
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
}

// cos and sin of the angle ah + al (al: the rounding error of ah and the
// low part of the frequency).  Cody and Waite's additive range reduction
// with 2*pi split in two floats: k*P1 is subtracted exactly (ah and k*P1 are
// multiples of 2^-22 once |ah| >= pi and the difference is below 4), k*P2
// with one rounding, then al is added to the small remainder; the hardware
// sine and cosine (absolute error about 2^-21 on [-pi, pi]) finish it.  The
// split leaves 7e-15 * k of 2*pi unaccounted, 2e-8 rad at positions near 2^24.
__device__ __forceinline__ void rope_cos_sin(float ah, float al, float &c, float &s) {
    constexpr float kInv2Pi = 0x1.45f306p-3f;   // 1 / (2 pi), rounded to float
    constexpr float kP1 = 0x1.921fb6p+2f;       // 2 pi rounded to float
    constexpr float kP2 = -0x1.777a5cp-23f;     // 2 pi - kP1, rounded to float
    const float k = rintf(ah * kInv2Pi);
    float r = fmaf(-k, kP1, ah);
    r = fmaf(-k, kP2, r) + al;
    __sincosf(r, &s, &c);
}

// Norm, rotation and stores of one work unit whose rows are in xa / xb
// (this lane's two 16-byte pieces of each pass).
template <int HD>
__device__ __forceinline__ void prologue_unit(const PrologueParams &p, int64_t unit, int lane,
                                              const uint4 (&xa)[kProUnroll],
                                              const uint4 (&xb)[kProUnroll], int64_t slot, float pos,
                                              uint4 wqa, uint4 wqb, uint4 wka, uint4 wkb) {
    constexpr int HALF = HD / 2;
    constexpr int LPR = HD / 16;                // lanes per row
    constexpr int RPW = 32 / LPR;               // rows per warp-wide pass
    const int sub = lane / LPR;
    const int ea = (lane % LPR) * 8;
    const int rows = p.hq + 2 * p.hkv;
    const int64_t D = (int64_t)p.hkv * HD;
    const int64_t t = unit / p.chunks;
    const int r0 = (int)(unit % p.chunks) * (RPW * kProUnroll);
    const bool store = slot >= 0 && slot < p.num_slots;
    if (lane == 0 && r0 == 0 && !store && slot != -1) flag(PKV_STATUS_BAD_SLOT);

    float cs[8], sn[8];
    if (r0 < p.hq + p.hkv) {                    // the unit rotates rows (warp-uniform)
        // pairs 2*lane and 2*lane+1 (mod d/2) of the angle table
        float c2[2], s2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = (2 * lane + h) % HALF;
            const float fh = p.inv_hi[i], fl = p.inv_lo[i];
            const float ah = pos * fh;
            const float al = fmaf(pos, fl, fmaf(pos, fh, -ah));
            rope_cos_sin(ah, al, c2[h], s2[h]);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int src = ea / 2 + jj;        // lane holding pairs ea + 2jj, ea + 2jj + 1
            cs[2 * jj] = __shfl_sync(0xffffffffu, c2[0], src);
            cs[2 * jj + 1] = __shfl_sync(0xffffffffu, c2[1], src);
            sn[2 * jj] = __shfl_sync(0xffffffffu, s2[0], src);
            sn[2 * jj + 1] = __shfl_sync(0xffffffffu, s2[1], src);
        }
    }

#pragma unroll
    for (int u = 0; u < kProUnroll; ++u) {
        const int r = r0 + u * RPW + sub;
        const bool is_q = r < p.hq;
        const bool is_k = !is_q && r < p.hq + p.hkv;
        if (r0 + u * RPW < p.hq + p.hkv) {      // some row of this pass rotates (warp-uniform)
            const uint32_t av[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w};
            const uint32_t bv[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
            float2 fa[4], fb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                fa[j] = unpack_bf16x2(av[j]);
                fb[j] = unpack_bf16x2(bv[j]);
            }
            // every lane takes part in the shuffles, whatever its row is
            float2 ss2 = fmul2(fa[0], fa[0]);
#pragma unroll
            for (int j = 1; j < 4; ++j) ss2 = ffma2(fa[j], fa[j], ss2);
#pragma unroll
            for (int j = 0; j < 4; ++j) ss2 = ffma2(fb[j], fb[j], ss2);
            float ss = ss2.x + ss2.y;
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float inv = rsqrtf(ss * (1.f / HD) + p.eps);
            const float2 inv2 = make_float2(inv, inv);
            const uint4 wa = is_q ? wqa : wka, wb = is_q ? wqb : wkb;
            const uint32_t wav[4] = {wa.x, wa.y, wa.z, wa.w}, wbv[4] = {wb.x, wb.y, wb.z, wb.w};
            uint32_t oa[4], ob[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // y = bf16(bf16(x * inv) * w), the two roundings of the norm
                const float2 na2 = fmul2(fa[j], inv2), nb2 = fmul2(fb[j], inv2);
                const float2 ya = unpack_bf16x2(mul_bf16x2(pack_bf16x2(na2.x, na2.y), wav[j]));
                const float2 yb = unpack_bf16x2(mul_bf16x2(pack_bf16x2(nb2.x, nb2.y), wbv[j]));
                const float2 c = make_float2(cs[2 * j], cs[2 * j + 1]);
                const float2 sv = make_float2(sn[2 * j], sn[2 * j + 1]);
                // first half: y cos - partner sin; second half: y cos + partner sin
                const float2 ra = ffma2(yb, make_float2(-sv.x, -sv.y), fmul2(ya, c));
                const float2 rb = ffma2(ya, sv, fmul2(yb, c));
                oa[j] = pack_bf16x2(ra.x, ra.y);
                ob[j] = pack_bf16x2(rb.x, rb.y);
            }
            const uint4 oA = make_uint4(oa[0], oa[1], oa[2], oa[3]);
            const uint4 oB = make_uint4(ob[0], ob[1], ob[2], ob[3]);
            uint16_t *dst = nullptr, *dst2 = nullptr;
            if (is_q) {
                dst = p.q_out + t * p.q_out_rs + (int64_t)r * HD;
            } else if (is_k) {
                const int h = r - p.hq;
                if (p.k_out) dst = p.k_out + t * p.k_out_rs + (int64_t)h * HD;
                if (store) dst2 = p.kc + slot * D + (int64_t)h * HD;
            }
            if (dst) {
                st_v4(dst + ea, oA);
                st_v4(dst + HALF + ea, oB);
            }
            if (dst2) {                         // cache row: streaming hint, as kv_store
                st_cs_v4(dst2 + ea, oA);
                st_cs_v4(dst2 + HALF + ea, oB);
            }
        }
        if (!is_q && !is_k && r < rows && store) {
            uint16_t *dst = p.vc + slot * D + (int64_t)(r - p.hq - p.hkv) * HD;
            st_cs_v4(dst + ea, xa[u]);
            st_cs_v4(dst + HALF + ea, xb[u]);
        }
    }
}

// source row of pass u of a unit for this lane, or null past the last row
template <int HD>
__device__ __forceinline__ const uint16_t *prologue_row(const PrologueParams &p, int64_t t, int r) {
    if (r < p.hq) return p.q + t * p.q_rs + (int64_t)r * HD;
    if (r < p.hq + p.hkv) return p.k + t * p.k_rs + (int64_t)(r - p.hq) * HD;
    if (r < p.hq + 2 * p.hkv) return p.v + t * p.v_rs + (int64_t)(r - p.hq - p.hkv) * HD;
    return nullptr;
}

// Each warp keeps kProStages units in flight with cp.async (16-byte pieces,
// zero-filled past the last row, plus the token's slot and position).
constexpr int kProStages = PKV_PRO_STAGES;
template <int HD>
struct ProStage {
    static constexpr int kPieceBytes = 32 * 16;                    // one piece of a pass, all lanes
    static constexpr int kRowBytes = 2 * kProUnroll * kPieceBytes; // the unit's rows
    static constexpr int kBytes = kRowBytes + 16;                  // + slot (4 B) and position (8 B)
    static constexpr int kWarpBytes = kProStages * kBytes;
};

__device__ __forceinline__ void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kProWarps * 32, PKV_PRO_MIN_CTAS)
qk_norm_rope_store_kernel(const __grid_constant__ PrologueParams p) {
    using S = ProStage<HD>;
    constexpr int HALF = HD / 2;
    constexpr int LPR = HD / 16;
    constexpr int RPW = 32 / LPR;
    extern __shared__ __align__(16) unsigned char pro_smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane / LPR;
    const int ea = (lane % LPR) * 8;
    const int64_t total = (int64_t)p.n * p.chunks;
    const int64_t stride = (int64_t)gridDim.x * kProWarps;
    int64_t unit = (int64_t)blockIdx.x * kProWarps + warp;
    if (unit >= total) return;                  // uniform per warp
    const uint4 wqa = ld_stream_v4(p.qw + ea), wqb = ld_stream_v4(p.qw + HALF + ea);
    const uint4 wka = ld_stream_v4(p.kw + ea), wkb = ld_stream_v4(p.kw + HALF + ea);
    unsigned char *wbase = pro_smem + warp * S::kWarpBytes;
    const uint32_t wbase_s = smem_u32(wbase);

    // start the copies of unit u_id into stage st (one commit group per unit,
    // also when there is no such unit, so that group counting stays uniform)
    auto issue = [&](int64_t u_id, int st) {
        if (u_id < total) {
            const int64_t t = u_id / p.chunks;
            const int r0 = (int)(u_id % p.chunks) * (RPW * kProUnroll);
            const uint32_t sb = wbase_s + st * S::kBytes;
#pragma unroll
            for (int u = 0; u < kProUnroll; ++u) {
                const uint16_t *src = prologue_row<HD>(p, t, r0 + u * RPW + sub);
                const uint32_t nbytes = src ? 16u : 0u;
                const uint16_t *s0 = src ? src + ea : p.qw;
                const uint16_t *s1 = src ? src + HALF + ea : p.qw;
                cp_async16(sb + (2 * u) * S::kPieceBytes + lane * 16, s0, nbytes);
                cp_async16(sb + (2 * u + 1) * S::kPieceBytes + lane * 16, s1, nbytes);
            }
            if (lane == 0) {
                cp_async4(sb + S::kRowBytes, p.slots + t);
                cp_async8(sb + S::kRowBytes + 8, p.pos + t);
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int k = 0; k < kProStages; ++k) issue(unit + k * stride, k);
    int st = 0;
    for (; unit < total; unit += stride) {
        cp_async_wait<kProStages - 1>();       // this lane's copies of the unit have landed
        __syncwarp();                           // ... and lane 0's slot / position
        const unsigned char *sp = wbase + st * S::kBytes;
        uint4 xa[kProUnroll], xb[kProUnroll];
#pragma unroll
        for (int u = 0; u < kProUnroll; ++u) {
            xa[u] = *reinterpret_cast<const uint4 *>(sp + (2 * u) * S::kPieceBytes + lane * 16);
            xb[u] = *reinterpret_cast<const uint4 *>(sp + (2 * u + 1) * S::kPieceBytes + lane * 16);
        }
        const int64_t slot = *reinterpret_cast<const int32_t *>(sp + S::kRowBytes);
        const int64_t pos64 = *reinterpret_cast<const int64_t *>(sp + S::kRowBytes + 8);
        __syncwarp();                           // every lane has read the stage before it is refilled
        issue(unit + kProStages * stride, st);
        const int r0 = (int)(unit % p.chunks) * (RPW * kProUnroll);
        const float pos = r0 < p.hq + p.hkv ? (float)pos64 : 0.f;   // exact below 2^24
        prologue_unit<HD>(p, unit, lane, xa, xb, slot, pos, wqa, wqb, wka, wkb);
        st = st + 1 == kProStages ? 0 : st + 1;
    }
    cp_async_wait<0>();                         // no copy may land after the warp has left
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
    const int rows_per_unit = (32 / (a.head_dim / 16)) * kProUnroll;
    p.chunks = (a.num_heads + 2 * a.num_kv_heads + rows_per_unit - 1) / rows_per_unit;
    // one resident wave of CTAs; each warp walks its units with the next
    // unit's loads in flight
    const int64_t units = (int64_t)a.num_tokens * p.chunks;
    const int64_t need = (units + kProWarps - 1) / kProWarps;
    const int64_t wave = (int64_t)num_sms() * PKV_PRO_MIN_CTAS;
    const dim3 grid((unsigned)(need < wave ? need : wave));
    const int smem = kProWarps * (a.head_dim == 128 ? ProStage<128>::kWarpBytes : ProStage<64>::kWarpBytes);
    static PerDeviceOnce once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = once.run(dev, []() {
            cudaError_t r = cudaFuncSetAttribute(qk_norm_rope_store_kernel<128>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kProWarps * ProStage<128>::kWarpBytes);
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(qk_norm_rope_store_kernel<64>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kProWarps * ProStage<64>::kWarpBytes);
            return r;
        });
    if (e != cudaSuccess) return e;
    if (a.head_dim == 128)
        qk_norm_rope_store_kernel<128><<<grid, kProWarps * 32, smem, stream>>>(p);
    else
        qk_norm_rope_store_kernel<64><<<grid, kProWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Duplicate-slot check (validate mode only): every pair (i, j), i < j, of the
// call's written slots is compared; a CTA holds 256 tokens' slots in
// registers and streams the later tokens' slots through shared memory.
// ---------------------------------------------------------------------------
struct SlotSource {
    const int32_t *slots;       // given slots, or null: derive decode slots
    const int32_t *bt;
    int64_t bt_stride;
    int32_t max_blocks;
    const int32_t *ctx;
    int32_t block_size;
    int64_t num_blocks;
};

// the slot token i writes, -1 when it writes nothing
__device__ __forceinline__ int32_t written_slot(const SlotSource &s, int32_t i) {
    if (s.slots) return s.slots[i];
    const int64_t c = s.ctx[i];
    if (c <= 0) return -1;
    const int64_t p = c - 1;
    const int64_t lb = p / s.block_size;
    const int32_t blk = lb < s.max_blocks ? s.bt[(int64_t)i * s.bt_stride + lb] : -1;
    if (blk < 0 || blk >= s.num_blocks) return -1;
    return (int32_t)((int64_t)blk * s.block_size + p % s.block_size);
}

constexpr int kDupThreads = 256;

__global__ void __launch_bounds__(kDupThreads) duplicate_slots_kernel(SlotSource src, int32_t n) {
    __shared__ int32_t later[kDupThreads];
    const int32_t i = blockIdx.x * kDupThreads + threadIdx.x;
    const int32_t mine = i < n ? written_slot(src, i) : -1;
    bool dup = false;
    for (int32_t j0 = blockIdx.x * kDupThreads; j0 < n; j0 += kDupThreads) {
        __syncthreads();
        later[threadIdx.x] = j0 + (int32_t)threadIdx.x < n ? written_slot(src, j0 + threadIdx.x) : -1;
        __syncthreads();
        if (mine >= 0) {
            for (int t = 0; t < kDupThreads; ++t)
                dup |= j0 + t > i && later[t] == mine;
        }
    }
    if (dup) flag(PKV_STATUS_DUP_SLOT);
}

cudaError_t launch_check_duplicate_slots(const int32_t *slots, const int32_t *bt, int64_t bt_stride,
                                         int32_t max_blocks, const int32_t *ctx,
                                         int32_t block_size, int64_t num_blocks, int32_t n,
                                         cudaStream_t stream) {
    if (n <= 1) return cudaSuccess;
    SlotSource s{slots, bt, bt_stride, max_blocks, ctx, block_size, num_blocks};
    duplicate_slots_kernel<<<(n + kDupThreads - 1) / kDupThreads, kDupThreads, 0, stream>>>(s, n);
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
