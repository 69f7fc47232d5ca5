// decode.cu -- single-token paged GQA attention over the paged KV cache
// (L17: Qwen3 attention sub-layer, §5.3 decode call; Lesson 04, §4), with
// the keys of a sequence split into chunks that are reduced independently
// and merged by the online-softmax rescaling of §5.2.
//
// Work unit: one CTA per (kv head, chunk of keys, sequence).  The CTA holds
// the GQA group's G query vectors (all query heads that share the kv head,
// §3) in registers, so every K/V byte it reads serves G heads.
//
// Data path:
//   * K and V of 64 tokens at a time ("tile") are staged into shared memory
//     by 3-D TMA over the cache viewed as [num_slots, num_kv_heads, head_dim]
//     (box: 64 head_dim elements x 1 head x min(block_size, 64) slots).  A
//     tile of a block_size >= 64 cache is one box per 64-element half of the
//     head_dim; smaller blocks take one box per block segment.  With
//     block_size >= 8 the boxes use the 128-byte swizzle so that the
//     row-per-thread reads below are bank-conflict free.
//   * A 3-stage mbarrier pipeline keeps two tiles in flight while one is
//     consumed; thread 0 refills a stage as soon as the whole CTA has left it.
//   * Scores: each token is owned by TPT consecutive threads that each dot a
//     slice of head_dim with the G queries (packed fp32x2 FMAs) and combine
//     by shuffles.  Scores carry scale*log2(e) so the softmax uses exp2.
//   * Softmax: the CTA-wide tile maximum updates the running maximum m; the
//     running sum l and output accumulators are rescaled by 2^(m_old-m_new)
//     (§5.2's exact rescaling).  Probabilities go to shared memory.
//   * P.V: each thread owns 8 head_dim elements of a group of tokens; tokens
//     whose probabilities are all zero (masked tail, invalid block) are
//     skipped, so garbage in unwritten cache slots never reaches the sum.
//   * Epilogue: a single-chunk launch writes bf16 out and lse directly;
//     otherwise each CTA writes (m, l, unnormalised o) in fp32 to the
//     workspace and decode_combine_kernel merges the chunks of each
//     (sequence, head).
//
// Bound: HBM.  Algorithmic bytes per launch = sum_b ctx_b * Hkv * d * 2 * 2
// (K and V, bf16) + q and out; arithmetic intensity about G FLOP/byte.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static __device__ unsigned int g_decode_status;

cudaError_t decode_status(cudaStream_t stream, uint32_t *host, bool clear) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_decode_status, sizeof v, 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && clear && v) {
        unsigned int z = 0;
        e = cudaMemcpyToSymbolAsync(g_decode_status, &z, sizeof z, 0, cudaMemcpyHostToDevice,
                                    stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    *host |= v;
    return e;
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 64;      // tokens per pipeline stage
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
    const uint16_t *q;
    int64_t q_rs;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t max_blocks;
    int64_t num_blocks;
    const int32_t *ctx;
    int32_t num_heads, num_kv_heads, block_size, max_context_len;
    int32_t chunk, max_splits;
    float scale_log2;          // softmax_scale * log2(e)
    uint16_t *out;
    int64_t out_rs;
    float *lse;
    float *part_o;             // [B, Hq, S, HD] fp32 (split mode)
    float *part_ml;            // [B, Hq, S, 2]  fp32 (split mode)
};

template <int HD>
struct Layout {
    static constexpr int kHalves = HD / 64;                      // 128-byte rows per head_dim
    static constexpr int kTileBytes = kHalves * kTile * 128;     // one of K or V
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kStages * kStageBytes;
};

template <bool SW>
__device__ __forceinline__ uint32_t chunk_off(int row, int chunk) {
    return row * 128 + ((SW ? (chunk ^ (row & 7)) : chunk) << 4);
}

template <int HD, int G, bool SW>
__global__ void __launch_bounds__(kThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using L = Layout<HD>;
    constexpr int TPT = (G <= 2) ? 4 : 8;           // threads per token in the score phase
    constexpr int E = HD / TPT;                     // head_dim elements per score thread
    constexpr int EC = E / 8;                       // 16-byte chunks per score thread
    constexpr int TOK_PASS = kThreads / TPT;        // tokens per score pass
    constexpr int PASSES = kTile / TOK_PASS;
    constexpr int CPR = HD / 8;                     // 16-byte chunks per row (P.V phase)
    constexpr int GROUPS = kThreads / CPR;          // token groups in the P.V phase
    constexpr int TPG = kTile / GROUPS;             // tokens per group per tile
    static_assert(PASSES >= 1 && TPG >= 1 && EC >= 1, "shape");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *pipe = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kPipeBytes);
    float *probs = reinterpret_cast<float *>(smem + L::kPipeBytes + 64);      // [G][kTile]
    float *red = probs + G * kTile;                                           // [kWarps][G]
    float *lred = red + kWarps * G;                                           // [kWarps][G]

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int kvh = blockIdx.x;
    const int split = blockIdx.y;
    const int b = blockIdx.z;
    const int hq0 = kvh * G;
    const int S = p.max_splits;
    const bool direct = (S == 1);

    int ctx = p.ctx[b];
    if (ctx < 0 || ctx > p.max_context_len) {
        if (tid == 0 && split == 0) atomicOr(&g_decode_status, PKV_STATUS_BAD_LENGTH);
        ctx = ctx < 0 ? 0 : p.max_context_len;
    }
    const int tok_begin = split * p.chunk;
    if (tok_begin >= ctx) {
        // nothing to read; a padding row (ctx == 0) still owns its output
        if (direct && split == 0) {
            for (int i = tid; i < G * HD; i += kThreads) {
                const int h = i / HD, e = i % HD;
                p.out[(int64_t)b * p.out_rs + (int64_t)(hq0 + h) * HD + e] = 0;
            }
            if (p.lse && tid < G) p.lse[(int64_t)b * p.num_heads + hq0 + tid] = -INFINITY;
        }
        return;
    }
    const int tok_end = min(ctx, tok_begin + p.chunk);
    const int ntiles = (tok_end - tok_begin + kTile - 1) / kTile;
    const int32_t *bt_row = p.bt + (int64_t)b * p.bt_stride;
    const int bs = p.block_size;
    const int TB = bs < kTile ? bs : kTile;          // slots per TMA box
    const uint32_t box_bytes = (uint32_t)TB * 128u;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    __syncthreads();

    const uint64_t policy = policy_evict_first();
    // thread 0: stage tile `i` into its stage
    auto issue = [&](int i) {
        const int stage = i % kStages;
        const int p0 = tok_begin + i * kTile;
        const int nv = min(kTile, tok_end - p0);
        const int nseg = (nv + TB - 1) / TB;
        int ok = 0;
        for (int sg = 0; sg < nseg; ++sg) {
            const int pos = p0 + sg * TB;
            const int lb = pos / bs;
            const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
            if (blk >= 0 && blk < p.num_blocks) ++ok;
        }
        mbar_arrive_expect_tx(&full[stage], (uint32_t)ok * L::kHalves * 2u * box_bytes);
        unsigned char *kdst = pipe + stage * L::kStageBytes;
        unsigned char *vdst = kdst + L::kTileBytes;
        for (int sg = 0; sg < nseg; ++sg) {
            const int pos = p0 + sg * TB;
            const int lb = pos / bs;
            const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
            if (blk < 0 || blk >= p.num_blocks) {
                atomicOr(&g_decode_status, PKV_STATUS_BAD_BLOCK);
                continue;
            }
            const int z = (int)((int64_t)blk * bs + pos % bs);
#pragma unroll
            for (int hf = 0; hf < L::kHalves; ++hf) {
                const int off = hf * kTile * 128 + sg * TB * 128;
                tma_load_3d(kdst + off, &kmap, &full[stage], hf * 64, kvh, z, policy);
                tma_load_3d(vdst + off, &vmap, &full[stage], hf * 64, kvh, z, policy);
            }
        }
    };
    if (tid == 0) {
        for (int i = 0; i < kStages && i < ntiles; ++i) issue(i);
    }

    // ---- this thread's query slice, pre-scaled by scale*log2(e) ----
    const int qd = tid % TPT;                       // slice of head_dim in the score phase
    const int e0 = qd * E;
    float2 q2[G][E / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint16_t *qrow = p.q + (int64_t)b * p.q_rs + (int64_t)(hq0 + h) * HD + e0;
#pragma unroll
        for (int c = 0; c < EC; ++c) {
            const uint4 w = *reinterpret_cast<const uint4 *>(qrow + c * 8);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                q2[h][c * 4 + k] = make_float2(bf16lo_to_f32(ws[k]) * p.scale_log2,
                                               bf16hi_to_f32(ws[k]) * p.scale_log2);
        }
    }

    // P.V role of this thread
    const int pv_chunk = tid % CPR;                 // 8-element chunk of head_dim
    const int pv_group = tid / CPR;                 // token group
    const int pv_half = pv_chunk / 8;
    const int pv_c = pv_chunk % 8;

    float m_run[G], l_part[G];
    float2 o2[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m_run[h] = -INFINITY;
        l_part[h] = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) o2[h][k] = make_float2(0.f, 0.f);
    }

    bool aborted = false;
    for (int i = 0; i < ntiles; ++i) {
        const int stage = i % kStages;
        const uint32_t parity = (uint32_t)(i / kStages) & 1u;
        const bool ok = mbar_wait(&full[stage], parity);
        const unsigned char *ktile = pipe + stage * L::kStageBytes;
        const unsigned char *vtile = ktile + L::kTileBytes;
        const int p0 = tok_begin + i * kTile;

        // ---- scores for this thread's token(s) ----
        float s_tok[PASSES][G];
        float tmax[G];
#pragma unroll
        for (int h = 0; h < G; ++h) tmax[h] = -INFINITY;
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int r = ps * TOK_PASS + tid / TPT;
            float2 acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < EC; ++c) {
                const int gchunk = (e0 / 8) + c;                 // chunk index within the row
                const int hf = gchunk / 8;
                const uint4 w = *reinterpret_cast<const uint4 *>(
                    ktile + hf * kTile * 128 + chunk_off<SW>(r, gchunk % 8));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 kf = make_float2(bf16lo_to_f32(ws[k]), bf16hi_to_f32(ws[k]));
#pragma unroll
                    for (int h = 0; h < G; ++h) acc[h] = ffma2(q2[h][c * 4 + k], kf, acc[h]);
                }
            }
            const int pos = p0 + r;
            bool valid = pos < tok_end;
            if (valid) {
                const int lb = pos / bs;
                const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                valid = blk >= 0 && blk < p.num_blocks;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s = acc[h].x + acc[h].y;
#pragma unroll
                for (int off = 1; off < TPT; off <<= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                s = valid ? s : -INFINITY;
                s_tok[ps][h] = s;
                tmax[h] = fmaxf(tmax[h], s);
            }
        }
        // CTA-wide tile maximum
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float v = tmax[h];
#pragma unroll
            for (int off = TPT; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            if (lane == 0) red[warp * G + h] = v;
        }
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        // every thread has left tile i-1: refill its stage
        if (tid == 0 && i >= 1 && i - 1 + kStages < ntiles) issue(i - 1 + kStages);

        float alpha[G], m_use[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float v = red[h];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) v = fmaxf(v, red[w * G + h]);
            const float m_new = fmaxf(m_run[h], v);
            m_use[h] = (m_new == -INFINITY) ? 0.f : m_new;
            alpha[h] = fast_exp2(m_run[h] - m_use[h]);     // 0 when m_run is -inf
            m_run[h] = m_new;
            l_part[h] *= alpha[h];
        }
        if (qd == 0) {
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) {
                const int r = ps * TOK_PASS + tid / TPT;
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float pr = fast_exp2(s_tok[ps][h] - m_use[h]);
                    probs[h * kTile + r] = pr;
                    l_part[h] += pr;
                }
            }
        }
        __syncthreads();

        // ---- P.V ----
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float2 a2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
            for (int k = 0; k < 4; ++k) o2[h][k] = make_float2(o2[h][k].x * a2.x, o2[h][k].y * a2.y);
        }
        const unsigned char *vbase = vtile + pv_half * kTile * 128;
#pragma unroll
        for (int t = 0; t < TPG; ++t) {
            const int r = pv_group * TPG + t;
            float pr[G];
            bool any = false;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                pr[h] = probs[h * kTile + r];
                any |= pr[h] != 0.f;
            }
            if (!any) continue;
            const uint4 w = *reinterpret_cast<const uint4 *>(vbase + chunk_off<SW>(r, pv_c));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 vf = make_float2(bf16lo_to_f32(ws[k]), bf16hi_to_f32(ws[k]));
#pragma unroll
                for (int h = 0; h < G; ++h) o2[h][k] = ffma2(make_float2(pr[h], pr[h]), vf, o2[h][k]);
            }
        }
    }

    if (aborted) {
        if (tid == 0) {
            atomicOr(&g_decode_status, PKV_STATUS_TIMEOUT);
            // let copies already in flight land before the CTA's shared memory is released
            for (int i = 0; i < ntiles && i < kStages; ++i) {
                (void)mbar_wait(&full[i % kStages], 0);
            }
        }
        return;
    }

    // ---- reduce accumulators over token groups ----
    __syncthreads();                                 // all P.V reads of the pipeline are done
    float *ored = reinterpret_cast<float *>(pipe);   // [kWarps][G][HD], reuses the pipeline
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 v = o2[h][k];
#pragma unroll
            for (int off = CPR; off < 32; off <<= 1) {
                v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
                v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
            }
            o2[h][k] = v;
        }
        float l = l_part[h];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        if (lane == 0) lred[warp * G + h] = l;
    }
    if (lane < CPR) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float *dst = ored + (warp * G + h) * HD + pv_chunk * 8;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dst[2 * k] = o2[h][k].x;
                dst[2 * k + 1] = o2[h][k].y;
            }
        }
    }
    __syncthreads();
    for (int idx = tid; idx < G * HD; idx += kThreads) {
        const int h = idx / HD, e = idx % HD;
        float o = 0.f, l = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            o += ored[(w * G + h) * HD + e];
            l += lred[w * G + h];
        }
        const int hq = hq0 + h;
        if (direct) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float r = o * inv;
            p.out[(int64_t)b * p.out_rs + (int64_t)hq * HD + e] =
                (uint16_t)(pack_bf16x2(r, 0.f) & 0xffffu);
            if (p.lse && e == 0)
                p.lse[(int64_t)b * p.num_heads + hq] =
                    l > 0.f ? (m_run[h] + log2f(l)) * kLn2 : -INFINITY;
        } else {
            const int64_t part = ((int64_t)b * p.num_heads + hq) * S + split;
            p.part_o[part * HD + e] = o;
            if (e == 0) {
                p.part_ml[part * 2] = m_run[h];
                p.part_ml[part * 2 + 1] = l;
            }
        }
    }
}

// Merge the chunks of each (sequence, head): one warp per pair.
//   m = max_s m_s, l = sum_s 2^(m_s - m) l_s, o = sum_s 2^(m_s - m) o_s / l
template <int HD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
    constexpr int EPL = HD / 32;                     // elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.x * 4 + warp;
    const int b = blockIdx.y;
    if (hq >= p.num_heads) return;
    int ctx = p.ctx[b];
    ctx = ctx < 0 ? 0 : (ctx > p.max_context_len ? p.max_context_len : ctx);
    const int ns = (ctx + p.chunk - 1) / p.chunk;
    uint16_t *orow = p.out + (int64_t)b * p.out_rs + (int64_t)hq * HD + lane * EPL;
    const int64_t part0 = ((int64_t)b * p.num_heads + hq) * p.max_splits;
    float m = -INFINITY;
    for (int s = 0; s < ns; ++s) m = fmaxf(m, p.part_ml[(part0 + s) * 2]);
    const float mu = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
    float o[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) o[k] = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float f = fast_exp2(p.part_ml[(part0 + s) * 2] - mu);
        l += f * p.part_ml[(part0 + s) * 2 + 1];
        const float *src = p.part_o + (part0 + s) * HD + lane * EPL;
#pragma unroll
        for (int k = 0; k < EPL; ++k) o[k] += f * src[k];
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int k = 0; k < EPL; k += 2) {
        const uint32_t w = pack_bf16x2(o[k] * inv, o[k + 1] * inv);
        *reinterpret_cast<uint32_t *>(orow + k) = w;
    }
    if (p.lse && lane == 0)
        p.lse[(int64_t)b * p.num_heads + hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

template <int HD>
constexpr size_t split_smem_bytes(int G) {
    return 1024 /*alignment slack*/ + Layout<HD>::kPipeBytes + 64 +
           sizeof(float) * (G * kTile + 2 * kWarps * G);
}

template <int HD, int G, bool SW>
int launch_split(const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p, int batch,
                 int num_kv_heads, cudaStream_t stream, const char **err) {
    auto kern = decode_split_kernel<HD, G, SW>;
    const size_t smem = split_smem_bytes<HD>(G);
    static_assert(Layout<HD>::kPipeBytes >= kWarps * 8 * HD * 4, "reduction buffer must fit");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    dim3 grid(num_kv_heads, p.max_splits, batch);
    kern<<<grid, kThreads, smem, stream>>>(km, vm, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    return PKV_OK;
}

template <int HD, bool SW>
int dispatch_group(int G, const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p,
                   int batch, int hkv, cudaStream_t s, const char **err) {
    switch (G) {
        case 1: return launch_split<HD, 1, SW>(km, vm, p, batch, hkv, s, err);
        case 2: return launch_split<HD, 2, SW>(km, vm, p, batch, hkv, s, err);
        case 4: return launch_split<HD, 4, SW>(km, vm, p, batch, hkv, s, err);
        case 8: return launch_split<HD, 8, SW>(km, vm, p, batch, hkv, s, err);
        default: *err = "num_heads / num_kv_heads must be 1, 2, 4 or 8"; return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace

void decode_plan(int32_t batch, int32_t num_kv_heads, int32_t head_dim, int32_t max_context_len,
                 int32_t *chunk, int32_t *max_splits) {
    (void)head_dim;
    const int64_t tiles = (int64_t)batch * num_kv_heads * ((max_context_len + kTile - 1) / kTile);
    // aim for about four waves of two CTAs per SM, assuming contexts average
    // about half of the maximum
    const int64_t target = (int64_t)num_sms() * 2 * 4;
    int64_t per = (tiles / 2 + target - 1) / (target > 0 ? target : 1);
    if (per < 4) per = 4;
    if (per > 64) per = 64;
    if (const char *env = getenv("PKV_DECODE_CHUNK_TILES")) {
        const int v = atoi(env);
        if (v >= 1 && v <= 4096) per = v;
    }
    *chunk = (int32_t)(per * kTile);
    *max_splits = max_context_len <= 0 ? 1 : (int32_t)((max_context_len + *chunk - 1) / *chunk);
}

size_t decode_workspace_bytes(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_context_len) {
    int32_t chunk, splits;
    decode_plan(batch, num_kv_heads, head_dim, max_context_len, &chunk, &splits);
    if (splits <= 1) return 0;
    const size_t parts = (size_t)batch * num_heads * splits;
    return parts * head_dim * sizeof(float) + parts * 2 * sizeof(float) + 256;
}

int launch_decode(const DecodeArgs &a, cudaStream_t stream, const char **err) {
    if (a.batch == 0) return PKV_OK;
    if (a.head_dim != 64 && a.head_dim != 128) {
        *err = "paged_attn_decode supports head_dim 64 and 128";
        return PKV_ERR_UNSUPPORTED;
    }
    int32_t chunk, splits;
    decode_plan(a.batch, a.num_kv_heads, a.head_dim, a.max_context_len, &chunk, &splits);
    DecodeParams p{};
    p.q = a.q;
    p.q_rs = a.q_rs;
    p.bt = a.bt;
    p.bt_stride = a.bt_stride;
    p.max_blocks = a.max_blocks;
    p.num_blocks = a.num_blocks;
    p.ctx = a.ctx;
    p.num_heads = a.num_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.block_size = a.block_size;
    p.max_context_len = a.max_context_len;
    p.chunk = chunk;
    p.max_splits = splits;
    p.scale_log2 = a.scale * kLog2e;
    p.out = a.out;
    p.out_rs = a.out_rs;
    p.lse = a.lse;
    if (splits > 1) {
        const size_t need = decode_workspace_bytes(a.batch, a.num_heads, a.num_kv_heads,
                                                   a.head_dim, a.max_context_len);
        if (!a.workspace || a.workspace_bytes < need) {
            *err = "paged_attn_decode: workspace smaller than paged_attn_decode_workspace_size()";
            return PKV_ERR_WORKSPACE;
        }
        uintptr_t w = (reinterpret_cast<uintptr_t>(a.workspace) + 255) & ~uintptr_t(255);
        p.part_o = reinterpret_cast<float *>(w);
        p.part_ml = p.part_o + (size_t)a.batch * a.num_heads * splits * a.head_dim;
    }
    const int tb = a.block_size < kTile ? a.block_size : kTile;
    const bool sw = tb >= 8;
    const int64_t num_slots = a.num_blocks * a.block_size;
    CUtensorMap km, vm;
    int rc = encode_rows_heads_map(&km, a.k_cache, num_slots, a.num_kv_heads, a.head_dim,
                                   (int64_t)a.num_kv_heads * a.head_dim, a.head_dim, 64, tb, sw, err);
    if (rc) return rc;
    rc = encode_rows_heads_map(&vm, a.v_cache, num_slots, a.num_kv_heads, a.head_dim,
                               (int64_t)a.num_kv_heads * a.head_dim, a.head_dim, 64, tb, sw, err);
    if (rc) return rc;
    const int G = a.num_heads / a.num_kv_heads;
    if (a.head_dim == 128)
        rc = sw ? dispatch_group<128, true>(G, km, vm, p, a.batch, a.num_kv_heads, stream, err)
                : dispatch_group<128, false>(G, km, vm, p, a.batch, a.num_kv_heads, stream, err);
    else
        rc = sw ? dispatch_group<64, true>(G, km, vm, p, a.batch, a.num_kv_heads, stream, err)
                : dispatch_group<64, false>(G, km, vm, p, a.batch, a.num_kv_heads, stream, err);
    if (rc) return rc;
    if (splits > 1) {
        dim3 grid((a.num_heads + 3) / 4, a.batch);
        if (a.head_dim == 128)
            decode_combine_kernel<128><<<grid, 128, 0, stream>>>(p);
        else
            decode_combine_kernel<64><<<grid, 128, 0, stream>>>(p);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    }
    return PKV_OK;
}

}  // namespace pkv

// ---------------------------------------------------------------------------
// Decode without any allocation by the caller.
//
// Some callers cannot obtain device memory for the split partials: a plugin
// running inside a host framework that owns every device allocation and only
// hands over tensors, or a runtime that forbids allocations after start-up.
// For them the partials live in a fixed array that belongs to this library
// and stays resident on every GPU that loads it, until the process exits.
// Nothing in the array has to start at zero: every partial the merge kernel
// reads is written earlier in the same call.
// ---------------------------------------------------------------------------
namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)PKV_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_static_scratch[kStaticScratchBytes];

// Device address of the array, looked up once per device with that device
// current (in host code the array's name is only a host-side stand-in, never
// a device address).
void *static_scratch_address(const char **err) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return nullptr; }
    if (dev < 0 || dev >= 64) { *err = "device ordinal out of range"; return nullptr; }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_static_scratch);
        if (e != cudaSuccess) { *err = cudaGetErrorString(e); return nullptr; }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" int paged_attn_decode_noalloc(const pkv_bf16 *q, int64_t q_row_stride,
                                         const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                         int64_t num_blocks, const int32_t *block_tables,
                                         int64_t bt_stride, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t batch,
                                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t block_size, int32_t max_context_len,
                                         float softmax_scale, pkv_bf16 *out,
                                         int64_t out_row_stride, float *lse, pkv_stream_t stream) {
    const size_t need = paged_attn_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                                         max_context_len);
    if (need > pkv::kStaticScratchBytes)
        return pkv::report(PKV_ERR_WORKSPACE,
                           "paged_attn_decode_noalloc: this launch needs %zu bytes of split "
                           "scratch, more than the %zu-byte static array; use paged_attn_decode "
                           "with a caller workspace, or a smaller batch*num_heads or "
                           "max_context_len",
                           need, pkv::kStaticScratchBytes);
    void *scratch = nullptr;
    if (need > 0) {
        const char *err = "";
        scratch = pkv::static_scratch_address(&err);
        if (!scratch)
            return pkv::report(PKV_ERR_CUDA,
                               "paged_attn_decode_noalloc: cudaGetSymbolAddress failed: %s", err);
    }
    return paged_attn_decode(q, q_row_stride, k_cache, v_cache, num_blocks, block_tables, bt_stride,
                             max_blocks_per_seq, context_lens, batch, num_heads, num_kv_heads,
                             head_dim, block_size, max_context_len, softmax_scale, out,
                             out_row_stride, lse, scratch, scratch ? pkv::kStaticScratchBytes : 0,
                             stream);
}
