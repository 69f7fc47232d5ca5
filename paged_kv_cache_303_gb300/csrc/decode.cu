// decode.cu -- single-token paged GQA attention over the paged KV cache
// (L17: Qwen3 attention sub-layer, §5.3 decode call; Lesson 04, §4), with
// the keys of a sequence split into chunks that are reduced independently
// and merged by the online-softmax rescaling of §5.2.
//
// Work items: (chunk of keys, sequence, kv head).  A CTA works on one item
// at a time with the GQA group's G query vectors (all query heads that share
// the kv head, §3) in shared memory, so every K/V byte it reads serves G
// heads.  The CTAs are persistent -- one resident wave, six per SM (shared
// memory the limit) -- and claim items from a counter in the workspace,
// chunk index outermost, so the full chunks are taken before the short last
// chunks of each sequence.
//
// Data path:
//   * K and V of 32 tokens at a time ("tile") are staged into shared memory
//     by 3-D TMA over the cache viewed as [num_slots, num_kv_heads, head_dim]
//     (box: 64 head_dim elements x 1 head x min(block_size, 32) slots).  With
//     block_size >= 8 the boxes use the 128-byte swizzle so that the
//     ldmatrix fragment reads below (8 rows of 16 bytes each) are
//     bank-conflict free.
//   * One producer warp claims items, writes each item's record and query
//     vectors into a two-entry item queue, and keeps a 2-stage tile ring
//     full (an mbarrier pair per stage) across item boundaries, so the next
//     item's first tile is in flight while the consumer merges the current
//     one.  kConsumers consumer warps (one by default) take the queue's items
//     in order; tile i of an item goes to warp i % kConsumers, with no
//     CTA-wide barrier inside the tile loop.
//   * Scores and P.V are warp-wide tensor-core products (mma.sync, bf16
//     inputs, fp32 accumulators): S = q K^T with the group's heads as rows,
//     then O^T += V^T P^T with the probabilities kept in the registers the
//     scores came out in.  The fp32 scores are multiplied by
//     scale*log2(e) so the softmax uses exp2.  (The two products are small -- G heads by 32 tokens -- and the
//     kernel stays HBM-bound; the tensor cores take the instruction count per
//     tile from about 1800 to about 200, which is what limited it.)
//   * Softmax: per warp and head, the tile maximum (shuffles) updates the
//     warp's running maximum m; its running sum l and output accumulators are
//     rescaled by 2^(m_old-m_new) (§5.2's exact rescaling).
//   * In a tile that is not complete (sequence tail, missing block) tokens
//     that are not valid get probability 0 and their value rows are zeroed
//     in registers, so garbage in unwritten cache slots never reaches the
//     sum.
//   * Fused store (paged_attn_decode_store): for the item whose chunk holds
//     position ctx-1 the producer warp first writes the step's new K/V row
//     of its kv head to that slot (the decode slot of Lesson 04 §4) with
//     generic stores, then orders them before its TMA reads with a proxy
//     fence; the tile that holds the new token then loads it like any other.
//     Exactly one item per (sequence, kv head) writes; a padding row writes
//     nothing.
//   * The consumer warps' (m, l, o) are merged in warp order at the end of
//     each item (the result does not depend on which CTA took the item); a
//     single-chunk launch writes bf16 out and lse directly, otherwise the
//     item's (m, l, unnormalised o) go to the workspace in fp32 and
//     decode_combine_kernel merges the chunks of each (sequence, head).
//   * How it was reached (kernel GB/s, qwen3-decode-b64): one CTA per item
//     with 3 stages x 4 CTAs/SM 5.21, 4 x 3 5.08, 6 x 2 4.26; the persistent
//     form 5.33 (per-item start-up hidden behind the previous item); on it,
//     two consumer warps per CTA instead of three (cheaper merges, more
//     CTAs' producers in flight) 5.36 -> 5.52, and 4.93 -> 5.08 on the
//     large batch-256 workload.  The CUDA-core products were issue-bound
//     (ncu on the group-4 workload: 45 % issue-active, 51 % DRAM-active);
//     with the tensor-core products the step (CUDA graph) went from 5.66 to
//     6.02 TB/s and the group-4 decode from 4.98 to 6.90 TB/s; consumers x
//     stages x CTAs/SM then: 2x3x5 6.02 / 6.90, 1x3x8 5.97 / 6.91, 1x4x6
//     5.89 / 6.82, 2x4x4 5.78 / 6.76, 1x2x8 6.06 / 6.92 (kept), 2x2x6 5.45 /
//     6.79.
//
// Bound: HBM.  Algorithmic bytes per launch = sum_b ctx_b * Hkv * d * 2 * 2
// (K and V, bf16) + q and out; arithmetic intensity about G FLOP/byte.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static __device__ unsigned int g_decode_status;

#if PKV_TEST_HOOKS
// Test-only build: while set, every CTA's producer withholds its arrival on
// the first item's ready barrier, so the consumers' bounded wait runs out
// (no bulk copy is ever pending on that barrier).
static __device__ int g_test_withhold_ready;

int test_withhold_decode_ready(int on) {
    return cudaMemcpyToSymbol(g_test_withhold_ready, &on, sizeof on) == cudaSuccess ? 0 : -1;
}
#endif

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

// Tunables (compile-time): consumer warps per CTA, ring depth, CTAs per SM.
#ifndef PKV_DEC_CONSUMERS
#define PKV_DEC_CONSUMERS 1
#endif
#ifndef PKV_DEC_STAGES
#define PKV_DEC_STAGES 2
#endif
#ifndef PKV_DEC_MIN_CTAS
#define PKV_DEC_MIN_CTAS 8
#endif
constexpr int kConsumers = PKV_DEC_CONSUMERS;    // consumer warps per CTA
constexpr int kThreads = (kConsumers + 1) * 32;  // + one TMA producer warp
constexpr int kTile = 32;                        // tokens per pipeline stage (one per lane)
constexpr int kStages = PKV_DEC_STAGES;
// Ring protocol.  Tile gt of the ring (counted across items) lives in stage
// gt % kStages and is that stage's phase K = gt / kStages.  A parity wait
// for phase K also passes while phase K-1 is still open (its parity is the
// one before), so a consumer may wait on full[stage] for tile gt only once
// phase K-1 -- tile gt - kStages -- has completed.  That tile may belong to
// the other consumer warp and TMA completions are unordered, so nothing in
// the consumer's own history implies it.  The consumer therefore first waits
// on empty[stage] for the release of tile gt - kStages: its consumer waited
// for that tile's phase before releasing it, so after this wait phase K-1 of
// full[stage] is complete, and phase K+1 cannot complete before this warp
// releases tile gt, which makes the parity wait for K exact.  The empty wait
// is itself exact when phase K-2 of empty[stage] (the release of tile
// gt - 2 kStages) has completed: that tile is either in an earlier item (all
// of whose tiles are released before the consumers' merge barrier) or this
// warp's own tile of the current item, which holds when kConsumers divides
// 2 kStages (tiles of an item go round-robin to the warps).  The producer
// needs the same release before it loads tile gt, so the extra wait costs a
// shared-memory poll, not time.
static_assert((2 * kStages) % kConsumers == 0,
              "tile gt - 2*kStages must be the waiting warp's own tile");
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
    unsigned int *work_counter; // items handed out so far (zeroed before the launch)
    int32_t batch;
    // fused store: this step's key/value rows [B, Hkv, HD] (null: no store)
    const uint16_t *new_k, *new_v;
    int64_t new_k_rs, new_v_rs;
    uint16_t *k_cache, *v_cache;
    // a GQA group larger than the kernel's 8 rows runs as kv_rep sub-groups
    // of G / kv_rep heads: work items name a virtual kv head v (num_kv_heads *
    // kv_rep of them) whose keys and values are those of kv head v / kv_rep
    int32_t kv_rep, num_vheads;   // num_vheads = num_kv_heads * kv_rep
};

template <bool SW>
__device__ __forceinline__ uint32_t chunk_off(int row, int chunk) {
    return row * 128 + ((SW ? (chunk ^ (row & 7)) : chunk) << 4);
}

// Merge the chunks of one (sequence, query head) with one warp:
//   m = max_s m_s, l = sum_s 2^(m_s - m) l_s, o = sum_s 2^(m_s - m) o_s / l
// The lanes read the (m, l) pairs of 32 chunks at once and the partial
// outputs eight chunks at a time (independent loads in flight), each chunk's
// factor passed by shuffle from the lane that computed it.  The partials are
// read through L2 only (they were written by other SMs and are read once).
template <int HD>
__device__ __forceinline__ void merge_head(const DecodeParams &p, int b, int hq, int ns, int lane) {
    constexpr int EPL = HD / 32;                     // elements per lane
    constexpr int kAhead = 8;
    const int64_t part0 = ((int64_t)b * p.num_heads + hq) * p.max_splits;
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml) + part0;
    float2 ml0 = lane < ns ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
    float m = ml0.x;
    for (int s = lane + 32; s < ns; s += 32) m = fmaxf(m, __ldcg(ml + s).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float mu = (m == -INFINITY) ? 0.f : m;
    float l = 0.f;
    float o[EPL];
#pragma unroll
    for (int k = 0; k < EPL; ++k) o[k] = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 32) {
        const int cnt = ns - s0 < 32 ? ns - s0 : 32;          // warp-uniform
        float f = 0.f;
        if (lane < cnt) {
            const float2 v = s0 == 0 ? ml0 : __ldcg(ml + s0 + lane);
            f = fast_exp2(v.x - mu);
            l += f * v.y;
        }
        for (int t = 0; t < cnt; t += kAhead) {
            float fs[kAhead];
            float src[kAhead][EPL];
#pragma unroll
            for (int u = 0; u < kAhead; ++u) {
                fs[u] = __shfl_sync(0xffffffffu, f, (t + u) & 31);
                if (t + u < cnt) {
                    const float *ps = p.part_o + (part0 + s0 + t + u) * HD + lane * EPL;
#pragma unroll
                    for (int k = 0; k < EPL; ++k) src[u][k] = __ldcg(ps + k);
                } else {
                    fs[u] = 0.f;
#pragma unroll
                    for (int k = 0; k < EPL; ++k) src[u][k] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kAhead; ++u)
#pragma unroll
                for (int k = 0; k < EPL; ++k) o[k] += fs[u] * src[u][k];
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint16_t *orow = p.out + (int64_t)b * p.out_rs + (int64_t)hq * HD + lane * EPL;
#pragma unroll
    for (int k = 0; k < EPL; k += 2) {
        const uint32_t w = pack_bf16x2(o[k] * inv, o[k + 1] * inv);
        *reinterpret_cast<uint32_t *>(orow + k) = w;
    }
    if (p.lse && lane == 0)
        p.lse[(int64_t)b * p.num_heads + hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers * 32) : "memory");
}

// Wait that gives up when another warp has aborted, or after the time bound
// (then it raises the abort flag itself).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            atomicOr(&g_decode_status, PKV_STATUS_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// The split kernel.  One resident wave of CTAs; the producer of each CTA
// claims work items -- (chunk, sequence, kv head), chunk index outermost, so
// the full chunks come before the short last chunks -- from a counter, loads
// the item's G query vectors into a two-entry item queue in shared memory and
// streams the item's tiles through the ring; consumers take the items from
// the queue in order.  Tile i of an item goes to consumer warp i % kConsumers
// and the warps' states are merged in warp order, so the result does not
// depend on which CTA claimed which item.  The next item's query vectors and
// first tiles are loaded while the consumers merge the current item.
// ---------------------------------------------------------------------------
constexpr int kQ = 2;                               // item queue entries

struct ItemRec {
    int b, kvh, split, tok_begin, tok_end, ntiles, kv, pad1;   // kv: the kv head whose K/V are read
};

template <int HD, int G>
struct Layout {
    static constexpr int kHalves = HD / 64;
    static constexpr int kTileBytes = kHalves * kTile * 128;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kStages * kStageBytes;
    static constexpr int kOffBar = kPipeBytes;      // full[S] empty[S] ready[Q] free[Q] masks abort
    static constexpr int kOffItems = kOffBar + 256; // ItemRec[kQ], then two decision words
    // per queue entry: q as bf16 [G][HD] in the first half, later the fp32
    // merge buffer [G][HD]
    static constexpr int kOffQ = kOffItems + 128;
    static constexpr int kOffML = kOffQ + kQ * G * HD * 4;           // [warp][G][2]
    static constexpr int kBytes = kOffML + kConsumers * G * 2 * 4;
    static_assert(2 * kStages * 8 + 2 * kQ * 8 + kStages * 4 + 4 <= 256, "barrier area");
    static_assert(kQ * (int)sizeof(ItemRec) + 8 <= 128, "item area");
};

template <int HD, int G, bool SW>
__global__ void __launch_bounds__(kThreads, PKV_DEC_MIN_CTAS)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using L = Layout<HD, G>;
    constexpr int DPL = HD / 32;                    // head_dim elements per lane of the fused store

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem =
        reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *pipe = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *empty = full + kStages;
    uint64_t *ready = empty + kStages;              // [kQ] item entry written
    uint64_t *freed = ready + kQ;                   // [kQ] item merged, entry reusable
    uint32_t *seg_valid = reinterpret_cast<uint32_t *>(freed + kQ);   // [kStages]
    volatile int *abort_flag = reinterpret_cast<volatile int *>(seg_valid + kStages);
    ItemRec *items = reinterpret_cast<ItemRec *>(smem + L::kOffItems);
    // consumer-wide decisions, published by one thread before a barrier so
    // that every consumer warp takes the same path through the barriers
    int *decide = reinterpret_cast<int *>(smem + L::kOffItems + kQ * sizeof(ItemRec));
    float *qring = reinterpret_cast<float *>(smem + L::kOffQ);
    float *mml = reinterpret_cast<float *>(smem + L::kOffML);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool direct = (p.max_splits == 1);
    const int bs = p.block_size;
    const int TB = bs < kTile ? bs : kTile;          // slots per TMA box
    const int per_split = p.batch * p.num_vheads;
    const int total = per_split * p.max_splits;

    if (warp == kConsumers && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int e = 0; e < kQ; ++e) {
            mbar_init(&ready[e], 1);
            mbar_init(&freed[e], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumers) {
        // ------------------------------------------------------------------
        // producer warp: claim items, fill the item queue, stream the tiles
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
        const uint64_t policy = policy_evict_first();
        const uint32_t box_bytes = (uint32_t)TB * 128u;
        int seq = 0, g = 0;
        bool live = true;
        while (live) {
            int idx = 0;
            if (lane == 0) idx = (int)atomicAdd(p.work_counter, 1u);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            ItemRec it{};
            const bool have = idx < total;
            if (have) {
                it.split = idx / per_split;
                const int rem = idx % per_split;
                it.b = rem / p.num_vheads;
                it.kvh = rem % p.num_vheads;
                it.kv = it.kvh / p.kv_rep;
                int ctx = p.ctx[it.b];
                if (ctx < 0 || ctx > p.max_context_len) {
                    if (lane == 0 && it.split == 0 && it.kvh == 0)
                        atomicOr(&g_decode_status, PKV_STATUS_BAD_LENGTH);
                    ctx = ctx < 0 ? 0 : p.max_context_len;
                }
                it.tok_begin = it.split * p.chunk;
                it.tok_end = min(ctx, it.tok_begin + p.chunk);
                it.ntiles = it.tok_begin < ctx ? (it.tok_end - it.tok_begin + kTile - 1) / kTile : 0;
                if (it.ntiles == 0) {
                    // nothing to read; a padding row still owns its output
                    if (direct && it.split == 0) {
                        const int hq0 = it.kvh * G;
                        for (int i = lane; i < G * HD; i += 32) {
                            const int h = i / HD, e = i % HD;
                            p.out[(int64_t)it.b * p.out_rs + (int64_t)(hq0 + h) * HD + e] = 0;
                        }
                        if (p.lse && lane < G) p.lse[(int64_t)it.b * p.num_heads + hq0 + lane] = -INFINITY;
                    }
                    continue;
                }
                // fused store: the chunk that holds position ctx-1 writes the
                // new token's row of its kv head before requesting any tile
                const bool ctx_ok = p.ctx[it.b] >= 0 && p.ctx[it.b] <= p.max_context_len;
                if (p.new_k != nullptr && ctx_ok && ctx - 1 >= it.tok_begin && ctx - 1 < it.tok_end) {
                    const int pos = ctx - 1;
                    const int lb = pos / bs;
                    const int32_t *bt_row = p.bt + (int64_t)it.b * p.bt_stride;
                    const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                    if (blk >= 0 && blk < p.num_blocks) {
                        // (the host stores the rows in a launch of their own when
                        // kv_rep > 1, so that every sub-group's reads see them)
                        const int64_t dst = ((int64_t)blk * bs + pos % bs) * p.num_kv_heads * HD +
                                            (int64_t)it.kvh * HD + lane * DPL;
                        const uint16_t *ks = p.new_k + (int64_t)it.b * p.new_k_rs + (int64_t)it.kvh * HD + lane * DPL;
                        const uint16_t *vs = p.new_v + (int64_t)it.b * p.new_v_rs + (int64_t)it.kvh * HD + lane * DPL;
                        if constexpr (DPL == 4) {
                            *reinterpret_cast<uint2 *>(p.k_cache + dst) = *reinterpret_cast<const uint2 *>(ks);
                            *reinterpret_cast<uint2 *>(p.v_cache + dst) = *reinterpret_cast<const uint2 *>(vs);
                        } else {
                            *reinterpret_cast<uint32_t *>(p.k_cache + dst) = *reinterpret_cast<const uint32_t *>(ks);
                            *reinterpret_cast<uint32_t *>(p.v_cache + dst) = *reinterpret_cast<const uint32_t *>(vs);
                        }
                        // the row is read back below by TMA (the async proxy)
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                }
            }
            // the queue entry of this item was last used two items ago
            const int e = seq % kQ;
            bool ok = true;
            if (lane == 0 && seq >= kQ) ok = wait_or_abort(&freed[e], (uint32_t)((seq / kQ) - 1) & 1u, abort_flag);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (!have) {
                if (lane == 0) {
                    items[e].ntiles = -1;               // end of the queue
                    mbar_arrive(&ready[e]);
                }
                break;
            }
            // the item's G query vectors (bf16, as given) into the queue entry
            uint4 *qd = reinterpret_cast<uint4 *>(qring + e * G * HD);
            for (int c = lane; c < G * HD / 8; c += 32) {
                const int h = c / (HD / 8), cc = c % (HD / 8);
                qd[c] = *reinterpret_cast<const uint4 *>(p.q + (int64_t)it.b * p.q_rs +
                                                         (int64_t)(it.kvh * G + h) * HD + cc * 8);
            }
            __syncwarp();
            if (lane == 0) {
                items[e] = it;
#if PKV_TEST_HOOKS
                if (!(seq == 0 && g_test_withhold_ready))
#endif
                mbar_arrive(&ready[e]);                 // releases q and the record
                // the item's tiles, tile i -> ring position g
                const int32_t *bt_row = p.bt + (int64_t)it.b * p.bt_stride;
                for (int i = 0; i < it.ntiles; ++i, ++g) {
                    const int stage = g % kStages;
                    if (g >= kStages &&
                        !wait_or_abort(&empty[stage], (uint32_t)((g / kStages) - 1) & 1u, abort_flag)) {
                        live = false;
                        break;
                    }
                    const int p0 = it.tok_begin + i * kTile;
                    const int nv = min(kTile, it.tok_end - p0);
                    const int nseg = (nv + TB - 1) / TB;
                    int okc = 0;
                    uint32_t mask = 0;                  // bit sg: segment sg was loaded
                    for (int sg = 0; sg < nseg; ++sg) {
                        const int pos = p0 + sg * TB;
                        const int lb = pos / bs;
                        const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                        if (blk >= 0 && blk < p.num_blocks) {
                            ++okc;
                            mask |= 1u << sg;
                        }
                    }
                    seg_valid[stage] = mask;            // released by the arrive below
                    mbar_arrive_expect_tx(&full[stage], (uint32_t)okc * L::kHalves * 2u * box_bytes);
                    unsigned char *kdst = pipe + stage * L::kStageBytes;
                    unsigned char *vdst = kdst + L::kTileBytes;
                    for (int sg = 0; sg < nseg; ++sg) {
                        if (!((mask >> sg) & 1u)) {
                            atomicOr(&g_decode_status, PKV_STATUS_BAD_BLOCK);
                            continue;
                        }
                        const int pos = p0 + sg * TB;
                        const int blk = bt_row[pos / bs];
                        const int z = (int)((int64_t)blk * bs + pos % bs);
#pragma unroll
                        for (int hf = 0; hf < L::kHalves; ++hf) {
                            const int off = hf * kTile * 128 + sg * TB * 128;
                            tma_load_3d(kdst + off, &kmap, &full[stage], hf * 64, it.kv, z, policy);
                            tma_load_3d(vdst + off, &vmap, &full[stage], hf * 64, it.kv, z, policy);
                        }
                    }
                }
            }
            live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
            ++seq;
        }
        if (lane == 0) {
            // no copy may still be landing when the CTA exits
            for (int j = g > kStages ? g - kStages : 0; j < g; ++j)
                (void)mbar_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1u);
        }
        return;
    }

    // ----------------------------------------------------------------------
    // consumer warps: items in queue order.  The two products of a tile run
    // on the tensor cores as warp-wide mma.sync (m16n8k16, bf16 inputs, fp32
    // accumulators); a lane holds fragments, g = lane / 4, t = lane % 4:
    //   S = q K^T    M = query heads of the group (G <= 8 real rows of 16),
    //                N = 8 tokens per product, K = 16 head_dim elements;
    //                q (A) stays in registers for the item, K (B) comes from
    //                the ring by ldmatrix.  Lane (g, t) holds the scores of
    //                head g for tokens 8n + 2t, 8n + 2t + 1 (n = 0..3).
    //   O^T += V^T P^T   M = 16 head_dim elements, N = 8 heads, K = 16
    //                tokens; V^T (A) comes from the ring by ldmatrix.trans,
    //                and the score fragments, turned into bf16 probabilities,
    //                are exactly the B fragments (P^T), so P never leaves
    //                registers.  Lane (g, t) accumulates O of heads 2t, 2t+1
    //                at head_dim elements 16m + g and 16m + g + 8.
    // Softmax per head over the tile: the 4 lanes of a group hold the head's
    // 32 scores (8 each); two xor shuffles give the tile maximum.  Tokens
    // that are not valid (sequence tail, missing block) get probability 0
    // and their value rows are zeroed in registers, so unwritten cache slots
    // never reach the sum.  The running sum l adds the probabilities as
    // rounded to bf16 for the product, so numerator and denominator use the
    // same weights.
    // ----------------------------------------------------------------------
    constexpr int KS = HD / 16;                    // 16-element steps over head_dim
    const int gq = lane >> 2, tq = lane & 3;
    const bool real_head = gq < G;
    // ldmatrix: lane 8i + r addresses row r of matrix i; matrices 0,1 cover
    // tokens 0..7 and 2,3 tokens 8..15 of a 16-token block, even / odd
    // 16-byte chunks
    const int lm_row = ((lane >> 4) << 3) + (lane & 7);
    const int lm_odd = (lane >> 3) & 1;
    const uint32_t all_segs = kTile / TB >= 32 ? 0xffffffffu : ((1u << (kTile / TB)) - 1u);
    auto frag_addr = [&](uint32_t tile_base, int row, int chunk) -> uint32_t {
        return tile_base + (uint32_t)((chunk >> 3) * kTile * 128) + chunk_off<SW>(row, chunk & 7);
    };
    int g0 = 0;
    for (int seq = 0;; ++seq) {
        const int e = seq % kQ;
        if (tid == 0) {
            const bool ok = wait_or_abort(&ready[e], (uint32_t)(seq / kQ) & 1u, abort_flag);
            decide[0] = ok ? 1 : 0;
        }
        consumer_sync();
        if (!decide[0]) break;                      // uniform
        const ItemRec it = items[e];
        if (it.ntiles < 0) break;                   // uniform
        const float *qs = qring + e * G * HD;
        const int hq0 = it.kvh * G;

        // q fragments of head gq (rows gq + 8 are zero)
        uint32_t qa[KS][2];
        {
            const uint16_t *qrow = reinterpret_cast<const uint16_t *>(qs) + gq * HD + 2 * tq;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                qa[kk][0] = real_head ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16) : 0u;
                qa[kk][1] = real_head ? *reinterpret_cast<const uint32_t *>(qrow + kk * 16 + 8) : 0u;
            }
        }
        float m_run = -INFINITY, l_part = 0.f;      // head gq
        float o[KS][4];                             // O^T fragments
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        bool live = true;
        for (int i = warp; i < it.ntiles; i += kConsumers) {
            const int gt = g0 + i;
            const int stage = gt % kStages;
            // the previous tile of this stage has been released (so it had
            // landed) before this tile's phase is awaited; see kStages above
            if (gt >= kStages &&
                !wait_or_abort(&empty[stage], (uint32_t)((gt / kStages) - 1) & 1u, abort_flag)) {
                live = false;
                break;
            }
            if (!wait_or_abort(&full[stage], (uint32_t)(gt / kStages) & 1u, abort_flag)) {
                live = false;
                break;
            }
            const uint32_t kbase = smem_u32(pipe + stage * L::kStageBytes);
            const uint32_t vbase = kbase + L::kTileBytes;
            const int p0 = it.tok_begin + i * kTile;
            const uint32_t mask = seg_valid[stage];
            const bool full_tile = (p0 + kTile <= it.tok_end) && mask == all_segs;

            // ---- S = q K^T ----
            float s[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                for (int np = 0; np < 2; ++np) {
                    uint32_t b[4];
                    ldmatrix_x4(b, frag_addr(kbase, np * 16 + lm_row, 2 * kk + lm_odd));
                    mma_bf16_16816(s[2 * np], qa[kk][0], 0u, qa[kk][1], 0u, b[0], b[1]);
                    mma_bf16_16816(s[2 * np + 1], qa[kk][0], 0u, qa[kk][1], 0u, b[2], b[3]);
                }
            }
            // scores in exp2 units; padding heads keep 0 (finite, unused)
            float sc[8];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                sc[2 * nt] = real_head ? s[nt][0] * p.scale_log2 : 0.f;
                sc[2 * nt + 1] = real_head ? s[nt][1] * p.scale_log2 : 0.f;
            }
            if (!full_tile && real_head) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int tk = (u >> 1) * 8 + 2 * tq + (u & 1);
                    const bool ok = (p0 + tk < it.tok_end) && ((mask >> (tk / TB)) & 1u);
                    if (!ok) sc[u] = -INFINITY;
                }
            }
            // ---- online softmax of head gq over the tile ----
            float mt = fmax3(fmax3(sc[0], sc[1], sc[2]), fmax3(sc[3], sc[4], sc[5]), fmaxf(sc[6], sc[7]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const float m_new = fmaxf(m_run, mt);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = fast_exp2(m_run - m_use);
            m_run = m_new;
            uint32_t pb[2][2];                      // P^T fragments, 16-token steps
            float lsum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const uint32_t pk = pack_bf16x2(fast_exp2(sc[2 * nt] - m_use), fast_exp2(sc[2 * nt + 1] - m_use));
                pb[nt >> 1][nt & 1] = pk;
                lsum += bf16lo_to_f32(pk) + bf16hi_to_f32(pk);
            }
            l_part = l_part * alpha + lsum;
            // rescale the accumulators of heads 2t, 2t+1
            const float a0 = __shfl_sync(0xffffffffu, alpha, (2 * tq) * 4);
            const float a1 = __shfl_sync(0xffffffffu, alpha, (2 * tq + 1) * 4);
#pragma unroll
            for (int m2 = 0; m2 < KS; ++m2) {
                o[m2][0] *= a0;
                o[m2][1] *= a1;
                o[m2][2] *= a0;
                o[m2][3] *= a1;
            }
            // ---- O^T += V^T P^T ----
            // value rows of tokens that are not valid: zeroed in the fragments
            uint32_t vmask[2][2] = {{0xffffffffu, 0xffffffffu}, {0xffffffffu, 0xffffffffu}};
            if (!full_tile) {
#pragma unroll
                for (int kt = 0; kt < 2; ++kt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t m2 = 0u;
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int tk = kt * 16 + hh * 8 + 2 * tq + u;
                            const bool ok = (p0 + tk < it.tok_end) && ((mask >> (tk / TB)) & 1u);
                            if (ok) m2 |= 0xffffu << (16 * u);
                        }
                        vmask[kt][hh] = m2;
                    }
            }
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
#pragma unroll
                for (int m2 = 0; m2 < KS; ++m2) {
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, frag_addr(vbase, kt * 16 + lm_row, 2 * m2 + lm_odd));
                    mma_bf16_16816(o[m2], a[0] & vmask[kt][0], a[1] & vmask[kt][0], a[2] & vmask[kt][1],
                                   a[3] & vmask[kt][1], pb[kt][0], pb[kt][1]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }

        // ---- merge the consumer warps' states, in warp order ----
        // (the item's q is in registers: its smem takes the merged output)
        consumer_sync();
        (void)live;
        if (tid == 0) decide[1] = *abort_flag;      // read once, seen by all after the barrier
        float *ob = const_cast<float *>(qs);        // [G][HD]
        {
            float l = l_part;
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (tq == 0 && real_head) {
                mml[(warp * G + gq) * 2] = m_run;
                mml[(warp * G + gq) * 2 + 1] = l;
            }
        }
        consumer_sync();
        const bool aborted = decide[1] != 0;        // uniform
        // this warp's factor for the heads 2t, 2t+1 of its fragments
        float f_own[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int h = 2 * tq + u;
            f_own[u] = 0.f;
            if (h < G) {
                float m = -INFINITY;
#pragma unroll
                for (int w = 0; w < kConsumers; ++w) m = fmaxf(m, mml[(w * G + h) * 2]);
                const float mu = (m == -INFINITY) ? 0.f : m;
                f_own[u] = fast_exp2(mml[(warp * G + h) * 2] - mu);
            }
        }
#pragma unroll 1
        for (int w = 0; w < kConsumers; ++w) {
            if (warp == w) {
#pragma unroll
                for (int m2 = 0; m2 < KS; ++m2)
#pragma unroll
                    for (int r = 0; r < 2; ++r)
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int h = 2 * tq + u;
                            if (h < G) {
                                float *dst = ob + h * HD + m2 * 16 + gq + 8 * r;
                                const float v = f_own[u] * o[m2][2 * r + u];
                                *dst = (w == 0 ? 0.f : *dst) + v;
                            }
                        }
            }
            consumer_sync();
        }
        for (int idx = tid; idx < G * HD && !aborted; idx += kConsumers * 32) {
            const int h = idx / HD, ee = idx % HD;
            float m = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) m = fmaxf(m, mml[(w * G + h) * 2]);
            const float mu = (m == -INFINITY) ? 0.f : m;
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w)
                l += fast_exp2(mml[(w * G + h) * 2] - mu) * mml[(w * G + h) * 2 + 1];
            const float o = ob[h * HD + ee];
            const int hq = hq0 + h;
            if (direct) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                p.out[(int64_t)it.b * p.out_rs + (int64_t)hq * HD + ee] =
                    (uint16_t)(pack_bf16x2(o * inv, 0.f) & 0xffffu);
                if (p.lse && ee == 0)
                    p.lse[(int64_t)it.b * p.num_heads + hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            } else {
                const int64_t part = ((int64_t)it.b * p.num_heads + hq) * p.max_splits + it.split;
                p.part_o[part * HD + ee] = o;
                if (ee == 0) {
                    p.part_ml[part * 2] = m;
                    p.part_ml[part * 2 + 1] = l;
                }
            }
        }
        // the entry (record, q / merge buffer) may be refilled
        consumer_sync();
        if (tid == 0) mbar_arrive(&freed[e]);
        if (aborted) break;                         // uniform, after the last barrier
        g0 += it.ntiles;
    }
    // the merge kernel (a programmatic dependent) may be scheduled once every
    // CTA of this one resident wave has got here; it waits for this grid's
    // completion before it reads the partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Merge the chunks of each (sequence, head): one warp per pair.
template <int HD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
    // launched as the split kernel's programmatic dependent: its partials
    // are complete and visible after this wait
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hq = blockIdx.x * 4 + warp;
    const int b = blockIdx.y;
    if (hq >= p.num_heads) return;
    int ctx = p.ctx[b];
    ctx = ctx < 0 ? 0 : (ctx > p.max_context_len ? p.max_context_len : ctx);
    merge_head<HD>(p, b, hq, (ctx + p.chunk - 1) / p.chunk, lane);
}

// The new K/V rows of a decode step written on their own (a GQA group split
// into sub-groups reads each kv head from several CTAs, which must all see
// the row): one warp per (row, kv head), the slot of position ctx - 1.
template <int HD>
__global__ void __launch_bounds__(128) decode_store_rows_kernel(const DecodeParams p) {
    constexpr int DPL = HD / 32;
    const int w = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (w >= p.batch * p.num_kv_heads) return;
    const int b = w / p.num_kv_heads, kvh = w % p.num_kv_heads;
    const int ctx = p.ctx[b];
    if (ctx <= 0 || ctx > p.max_context_len) return;      // padding row, or flagged by the decode
    const int pos = ctx - 1, bs = p.block_size, lb = pos / bs;
    const int32_t *bt_row = p.bt + (int64_t)b * p.bt_stride;
    const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
    if (blk < 0 || blk >= p.num_blocks) return;             // flagged by the decode's loads
    const int64_t dst = ((int64_t)blk * bs + pos % bs) * p.num_kv_heads * HD + (int64_t)kvh * HD + lane * DPL;
    const uint16_t *ks = p.new_k + (int64_t)b * p.new_k_rs + (int64_t)kvh * HD + lane * DPL;
    const uint16_t *vs = p.new_v + (int64_t)b * p.new_v_rs + (int64_t)kvh * HD + lane * DPL;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
        p.k_cache[dst + i] = ks[i];
        p.v_cache[dst + i] = vs[i];
    }
}

template <int HD, int G, bool SW>
int launch_split(const CUtensorMap &km, const CUtensorMap &vm, const DecodeParams &p, int batch,
                 int num_kv_heads, cudaStream_t stream, const char **err) {
    auto kern = decode_split_kernel<HD, G, SW>;
    const size_t smem = 1024 /*alignment slack*/ + Layout<HD, G>::kBytes;
    static PerDeviceOnce once;
    static int resident[kMaxDevices];                  // CTAs of this kernel per SM
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = once.run(dev, [&]() -> cudaError_t {
            cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            int nb = 0;
            if (r == cudaSuccess)
                r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kThreads, smem);
            if (r == cudaSuccess) resident[dev] = nb > 0 ? nb : 1;
            return r;
        });
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    // one resident wave; the CTAs claim the items
    const int64_t items = (int64_t)batch * num_kv_heads * p.max_splits;
    const int64_t wave = (int64_t)num_sms() * resident[dev];
    const dim3 grid((unsigned)(items < wave ? items : wave));
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
        case 3: return launch_split<HD, 3, SW>(km, vm, p, batch, hkv, s, err);
        case 4: return launch_split<HD, 4, SW>(km, vm, p, batch, hkv, s, err);
        case 5: return launch_split<HD, 5, SW>(km, vm, p, batch, hkv, s, err);
        case 6: return launch_split<HD, 6, SW>(km, vm, p, batch, hkv, s, err);
        case 7: return launch_split<HD, 7, SW>(km, vm, p, batch, hkv, s, err);
        case 8: return launch_split<HD, 8, SW>(km, vm, p, batch, hkv, s, err);
        default: *err = "GQA sub-group of more than 8 heads"; return PKV_ERR_UNSUPPORTED;
    }
}

}  // namespace

std::atomic<int> g_decode_chunk_tiles{0};

int decode_kv_rep(int32_t num_heads, int32_t num_kv_heads) {
    const int G = num_heads / num_kv_heads;
    int r = 1;
    while (G / r > 8 || G % r != 0) ++r;
    return r;
}

void decode_plan(int32_t batch, int32_t num_kv_heads, int32_t head_dim, int32_t max_context_len,
                 int32_t *chunk, int32_t *max_splits) {
    (void)head_dim;
    // about one and a half waves of resident CTAs, assuming contexts average
    // half of the maximum; chunks of 256 .. 2048 keys.  (Chunks per sweep on
    // qwen3-decode-b64, step GB/s: 288 keys 6.13, 384 6.26, 512 6.36, 768
    // 6.28; the group-4 large decode is best at the 2048-key cap.)
    const int64_t keys = (int64_t)batch * num_kv_heads * max_context_len / 2;
    const int64_t target = (int64_t)num_sms() * PKV_DEC_MIN_CTAS * 3 / 2;
    int64_t per = (keys + target * kTile - 1) / (target * kTile);
    if (per < 8) per = 8;
    if (per > 64) per = 64;
    // a power of two of tiles, the nearer one (chunks of 512 keys beat 576
    // on qwen3-decode-b64: 6.25-6.36 against 6.08 TB/s)
    {
        int64_t lo = 8;
        while (lo * 2 <= per) lo *= 2;
        per = (per - lo <= lo * 2 - per) ? lo : lo * 2;
        if (per > 64) per = 64;
    }
    const int forced = g_decode_chunk_tiles.load(std::memory_order_relaxed);
    if (forced > 0) per = forced;
    *chunk = (int32_t)(per * kTile);
    *max_splits = max_context_len <= 0 ? 1 : (int32_t)((max_context_len + *chunk - 1) / *chunk);
}

size_t decode_workspace_bytes(int32_t batch, int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t max_context_len) {
    int32_t chunk, splits;
    decode_plan(batch, num_kv_heads * decode_kv_rep(num_heads, num_kv_heads), head_dim, max_context_len,
                &chunk, &splits);
    // a work counter (256 bytes, first), then the chunk partials
    const size_t counter = 256;
    if (splits <= 1) return counter;
    const size_t parts = (size_t)batch * num_heads * splits;
    return counter + parts * head_dim * sizeof(float) + parts * 2 * sizeof(float) + 256;
}

int launch_decode(const DecodeArgs &a, cudaStream_t stream, const char **err) {
    if (a.batch == 0) return PKV_OK;
    if (a.head_dim != 64 && a.head_dim != 128) {
        *err = "paged_attn_decode supports head_dim 64 and 128";
        return PKV_ERR_UNSUPPORTED;
    }
    const int rep = decode_kv_rep(a.num_heads, a.num_kv_heads);
    int32_t chunk, splits;
    decode_plan(a.batch, a.num_kv_heads * rep, a.head_dim, a.max_context_len, &chunk, &splits);
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
    p.new_k = a.new_k;
    p.new_v = a.new_v;
    p.new_k_rs = a.new_k_rs;
    p.new_v_rs = a.new_v_rs;
    p.k_cache = const_cast<uint16_t *>(a.k_cache);
    p.v_cache = const_cast<uint16_t *>(a.v_cache);
    p.batch = a.batch;
    p.kv_rep = rep;
    p.num_vheads = a.num_kv_heads * rep;
    // workspace: the item counter (zeroed here, in stream order), then the
    // chunk partials when there is more than one chunk
    const size_t need = decode_workspace_bytes(a.batch, a.num_heads, a.num_kv_heads, a.head_dim,
                                               a.max_context_len);
    if (!a.workspace || a.workspace_bytes < need) {
        *err = "paged_attn_decode: workspace smaller than paged_attn_decode_workspace_size()";
        return PKV_ERR_WORKSPACE;
    }
    uintptr_t w = (reinterpret_cast<uintptr_t>(a.workspace) + 255) & ~uintptr_t(255);
    p.work_counter = reinterpret_cast<unsigned int *>(w);
    cudaError_t me = cudaMemsetAsync(p.work_counter, 0, sizeof(unsigned int), stream);
    if (me != cudaSuccess) { *err = cudaGetErrorString(me); return PKV_ERR_CUDA; }
    w += 256;
    if (splits > 1) {
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
    if (rep > 1 && p.new_k != nullptr) {
        // the step's rows first, then the decode without its fused store
        const int warps = a.batch * a.num_kv_heads;
        if (a.head_dim == 128)
            decode_store_rows_kernel<128><<<(warps + 3) / 4, 128, 0, stream>>>(p);
        else
            decode_store_rows_kernel<64><<<(warps + 3) / 4, 128, 0, stream>>>(p);
        cudaError_t se = cudaGetLastError();
        if (se != cudaSuccess) { *err = cudaGetErrorString(se); return PKV_ERR_CUDA; }
        p.new_k = p.new_v = nullptr;
    }
    const int G = a.num_heads / a.num_kv_heads / rep;        // heads per (sub-)group
    const int nvh = a.num_kv_heads * rep;
    if (a.head_dim == 128)
        rc = sw ? dispatch_group<128, true>(G, km, vm, p, a.batch, nvh, stream, err)
                : dispatch_group<128, false>(G, km, vm, p, a.batch, nvh, stream, err);
    else
        rc = sw ? dispatch_group<64, true>(G, km, vm, p, a.batch, nvh, stream, err)
                : dispatch_group<64, false>(G, km, vm, p, a.batch, nvh, stream, err);
    if (rc) return rc;
    if (splits > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((a.num_heads + 3) / 4, a.batch);
        cfg.blockDim = dim3(128);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = a.head_dim == 128 ? cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, p)
                                          : cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, p);
        if (e == cudaSuccess) e = cudaGetLastError();
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
// a device address).  The address stays valid while the device's primary
// context lives; a cudaDeviceReset would make the kept address stale, so the
// entry point's documentation rules that out.
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
