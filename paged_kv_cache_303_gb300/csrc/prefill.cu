// prefill.cu -- varlen causal paged prefill on the 5th-generation tensor
// cores (tcgen05 + tensor memory), for plain prefill (keys from the packed
// k/v of the step) and prefix-cache prefill (keys through block_tables from
// the paged cache).  L17: Qwen3 attention sub-layer, §5.2 (blocked softmax
// with exact rescaling) and §5.3 (the varlen call, causal=True, and its
// prefix-cache branch); Lesson 04, §4.
//
// Work unit: one CTA per (128 query rows of one sequence, two query heads of
// one GQA group).  The two heads share every K/V tile the CTA loads, which
// halves K/V traffic per FLOP compared with one head per CTA.
//
// Roles (320 threads):
//   warps 0-3  softmax warpgroup of query head A, thread = query row = TMEM lane
//   warps 4-7  softmax warpgroup of query head B
//   warp 8     TMA producer: Q once, then K and V tiles of 64 keys through a
//              3-stage ring (packed k/v: one box per half of head_dim; paged
//              cache: one box per block segment, addressed via block_tables)
//   warp 9     MMA issuer: S = Q K^T (M=128, N=64, K=head_dim) into TMEM, and
//              O += P V (M=128, N=head_dim, K=64) with O resident in TMEM
//
// Tensor memory (fp32 accumulators, lane = query row):
//   S_A cols [0,64), S_B [64,128), O_A [128,128+d), O_B [128+d,128+2d)
//
// Shared-memory operands use the 128-byte swizzle written by TMA: Q, K and P
// are K-major, V is read as an MN-major B operand (keys are K, head_dim N).
//
// Softmax: per row, scores are scaled by scale*log2(e) and exponentiated
// with exp2.  The running maximum is only moved when a tile's maximum
// exceeds it by more than 8 (a factor 256): then l and the O accumulator
// in TMEM are rescaled by 2^(m_old - m_new) (§5.2's identity).  Otherwise
// the stale maximum is kept; every p is then <= 2^8, and the final O / l
// uses the same maximum for numerator and denominator, so the result is the
// same softmax.
//
// Causality: query row t of a sequence with Lq queries and Lk keys sees keys
// j <= Lk - Lq + t.  KV tiles past the last row's bound are never loaded;
// only tiles that cross a row's bound are masked.  In paged mode the value
// rows past Lk of the last tile are zeroed in shared memory before P V, so
// unwritten cache slots (possibly NaN) never meet a zero probability.
//
// A one-CTA planning kernel lists the (sequence, 128-row block) work items
// in decreasing order of key tiles (longest first) in the workspace.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static __device__ unsigned int g_prefill_status;

cudaError_t prefill_status(cudaStream_t stream, uint32_t *host, bool clear) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_prefill_status, sizeof v, 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && clear && v) {
        unsigned int z = 0;
        e = cudaMemcpyToSymbolAsync(g_prefill_status, &z, sizeof z, 0, cudaMemcpyHostToDevice,
                                    stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    *host |= v;
    return e;
}

namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 64;           // keys per KV tile
constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kCostBins = 2048;

// ---------------------------------------------------------------------------
// tcgen05 / tensor-memory wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;          // descriptor version of the 5th-generation tensor core
    d |= (uint64_t)2 << 61;          // 128-byte swizzle
    return d;
}

// instruction descriptor: bf16 x bf16 -> fp32, A K-major, B K- or MN-major
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers (waits)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 registers -> 32 consecutive TMEM columns of this warp's lanes (waits)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Wait that gives up when another role has aborted, or after the time bound
// (then it raises the abort flag itself).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            atomicOr(&g_prefill_status, PKV_STATUS_TIMEOUT);
            return false;
        }
    }
}

struct PrefillParams {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t max_blocks;
    int64_t num_blocks;
    int32_t block_size;
    int32_t num_seqs;
    int32_t num_heads, num_kv_heads;
    int32_t paged;
    float scale_log2;
    uint16_t *out;
    int64_t out_rs;
    float *lse;
    const int32_t *work_count;   // [1]
    const int2 *work;            // [max_items] (sequence, 128-row block)
    int32_t max_items;
};

__device__ __forceinline__ int kv_tiles_for(int Lq, int Lk, int mb) {
    const int t_last = min(Lq, (mb + 1) * kBM) - 1;
    const int keys = Lk - Lq + t_last + 1;
    return (keys + kBN - 1) / kBN;
}

// Work list: every (sequence, 128-row block), ordered by decreasing number
// of key tiles (a counting sort on the cost).  One CTA.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(PrefillParams p, int32_t *work_count,
                                                            int2 *work) {
    __shared__ int hist[kCostBins];
    __shared__ int total;
    for (int i = threadIdx.x; i < kCostBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
        const int Lq = p.cu_q[s + 1] - p.cu_q[s];
        const int Lk = p.cu_k[s + 1] - p.cu_k[s];
        if (Lq <= 0) continue;
        if (Lk < Lq) { atomicOr(&g_prefill_status, PKV_STATUS_BAD_LENGTH); continue; }
        const int nmb = (Lq + kBM - 1) / kBM;
        for (int mb = 0; mb < nmb; ++mb)
            atomicAdd(&hist[min(kv_tiles_for(Lq, Lk, mb), kCostBins - 1)], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;   // descending cost: bins from high to low
        for (int c = kCostBins - 1; c >= 0; --c) {
            const int h = hist[c];
            hist[c] = run;
            run += h;
        }
        total = min(run, p.max_items);
        if (run > p.max_items) atomicOr(&g_prefill_status, PKV_STATUS_BAD_LENGTH);
        *work_count = total;
    }
    __syncthreads();
    for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
        const int Lq = p.cu_q[s + 1] - p.cu_q[s];
        const int Lk = p.cu_k[s + 1] - p.cu_k[s];
        if (Lq <= 0 || Lk < Lq) continue;
        const int nmb = (Lq + kBM - 1) / kBM;
        for (int mb = 0; mb < nmb; ++mb) {
            const int pos = atomicAdd(&hist[min(kv_tiles_for(Lq, Lk, mb), kCostBins - 1)], 1);
            if (pos < p.max_items) work[pos] = make_int2(s, mb);
        }
    }
}

template <int HD>
struct PLayout {
    static constexpr int H = HD / 64;                       // 128-byte halves of a row
    static constexpr int kQTile = H * kBM * 128;            // one query head's tile
    static constexpr int kKTile = H * kBN * 128;            // K or V tile
    static constexpr int kStage = 2 * kKTile;
    static constexpr int kPTile = kBM * 128;                // 128 rows x 64 keys bf16
    static constexpr int kOffKV = 2 * kQTile;
    static constexpr int kOffP = kOffKV + kStages * kStage;
    static constexpr int kOffBar = kOffP + 2 * kPTile;
    static constexpr int kBytes = kOffBar + 256;
    static constexpr int kTmemCols = (2 * kBN + 2 * HD) <= 256 ? 256 : 512;
    static constexpr int kColS = 0;                         // + t * kBN
    static constexpr int kColO = 2 * kBN;                   // + t * HD
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using L = PLayout<HD>;
    constexpr int H = L::H;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int item = blockIdx.y;
    if (item >= p.max_items || item >= *p.work_count) return;     // uniform for the CTA
    const int2 w = p.work[item];
    const int seq = w.x, mb = w.y;
    const int q0 = p.cu_q[seq];
    const int Lq = p.cu_q[seq + 1] - q0;
    const int k0 = p.cu_k[seq];
    const int Lk = p.cu_k[seq + 1] - k0;
    const int off = Lk - Lq;
    const int r0 = mb * kBM;
    const int n_kv = kv_tiles_for(Lq, Lk, mb);
    const int G = p.num_heads / p.num_kv_heads;
    const int ntile = G >= 2 ? 2 : 1;
    const int h0 = blockIdx.x * ntile;
    const int kvh = h0 / G;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;      // [kStages]
    uint64_t *kv_empty = bars + 4;     // [kStages]
    uint64_t *s_full = bars + 7;       // [2]
    uint64_t *s_free = bars + 9;       // [2]
    uint64_t *p_full = bars + 11;      // [2]
    uint64_t *o_ready = bars + 13;     // [2]
    uint64_t *drain = bars + 15;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 17);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&s_free[t], kBM);
            mbar_init(&p_full[t], kBM);
            mbar_init(&o_ready[t], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensormap(&qmap);
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
            const uint64_t pol_stream = policy_evict_first();
            mbar_arrive_expect_tx(q_full, (uint32_t)(ntile * L::kQTile));
            for (int t = 0; t < ntile; ++t)
                for (int hf = 0; hf < H; ++hf)
                    tma_load_3d(smem + t * L::kQTile + hf * kBM * 128, &qmap, q_full, hf * 64, h0 + t,
                                q0 + r0, pol_stream);
            const int bs = p.block_size;
            const int TB = p.paged ? (bs < kBN ? bs : kBN) : kBN;
            const int32_t *bt_row = p.paged ? p.bt + (int64_t)seq * p.bt_stride : nullptr;
            int issued = 0;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % kStages;
                if (j >= kStages &&
                    !wait_or_abort(&kv_empty[s], (uint32_t)((j / kStages) - 1) & 1u, abort_flag))
                    break;
                unsigned char *kdst = smem + L::kOffKV + s * L::kStage;
                unsigned char *vdst = kdst + L::kKTile;
                if (!p.paged) {
                    mbar_arrive_expect_tx(&kv_full[s], (uint32_t)(2 * L::kKTile));
                    for (int hf = 0; hf < H; ++hf) {
                        tma_load_3d(kdst + hf * kBN * 128, &kmap, &kv_full[s], hf * 64, kvh,
                                    k0 + j * kBN, pol_stream);
                        tma_load_3d(vdst + hf * kBN * 128, &vmap, &kv_full[s], hf * 64, kvh,
                                    k0 + j * kBN, pol_stream);
                    }
                } else {
                    const int nseg = kBN / TB;
                    int ok = 0;
                    for (int sg = 0; sg < nseg; ++sg) {
                        const int pos = j * kBN + sg * TB;
                        if (pos >= Lk) break;
                        const int lb = pos / bs;
                        const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                        if (blk >= 0 && blk < p.num_blocks) ++ok;
                    }
                    mbar_arrive_expect_tx(&kv_full[s], (uint32_t)(ok * H * 2 * TB * 128));
                    for (int sg = 0; sg < nseg; ++sg) {
                        const int pos = j * kBN + sg * TB;
                        if (pos >= Lk) break;
                        const int lb = pos / bs;
                        const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                        if (blk < 0 || blk >= p.num_blocks) {
                            atomicOr(&g_prefill_status, PKV_STATUS_BAD_BLOCK);
                            continue;
                        }
                        const int z = (int)((int64_t)blk * bs + pos % bs);
                        for (int hf = 0; hf < H; ++hf) {
                            const int o = hf * kBN * 128 + sg * TB * 128;
                            tma_load_3d(kdst + o, &kmap, &kv_full[s], hf * 64, kvh, z, pol_stream);
                            tma_load_3d(vdst + o, &vmap, &kv_full[s], hf * 64, kvh, z, pol_stream);
                        }
                    }
                }
                ++issued;
            }
            // no copy may still be landing when the CTA leaves
            for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
                (void)mbar_wait(&kv_full[j % kStages], (uint32_t)(j / kStages) & 1u);
            (void)mbar_wait(q_full, 0);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------
        // MMA issuer (lane 0); the whole warp zeroes value rows past the
        // keys of a paged sequence
        // ------------------------------------------------------------------
        constexpr uint32_t kIdS = idesc_bf16(kBM, kBN, false);
        constexpr uint32_t kIdO = idesc_bf16(kBM, HD, true);
        const uint32_t sbase = smem_u32(smem);
        auto issue_S = [&](int j, int t) {
            const uint32_t kb = sbase + L::kOffKV + (j % kStages) * L::kStage;
            const uint32_t qb = sbase + t * L::kQTile;
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const int hf = kk / 4;
                const uint32_t ko = (kk % 4) * 32;
                const uint64_t a = sdesc_sw128(qb + hf * kBM * 128 + ko, 16, 1024);
                const uint64_t b = sdesc_sw128(kb + hf * kBN * 128 + ko, 16, 1024);
                umma_bf16(tmem + L::kColS + t * kBN, a, b, kIdS, kk > 0 ? 1u : 0u);
            }
            umma_commit(&s_full[t]);
        };
        auto issue_PV = [&](int j, int t) {
            const uint32_t vb = sbase + L::kOffKV + (j % kStages) * L::kStage + L::kKTile;
            const uint32_t pb = sbase + L::kOffP + t * L::kPTile;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                const uint64_t a = sdesc_sw128(pb + kk * 32, 16, 1024);
                const uint64_t b = sdesc_sw128(vb + kk * 16 * 128, kBN * 128, 1024);
                umma_bf16(tmem + L::kColO + t * HD, a, b, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&o_ready[t]);
        };
        bool live = true;
        if (lane == 0) {
            live = wait_or_abort(q_full, 0, abort_flag) && wait_or_abort(&kv_full[0], 0, abort_flag);
            if (live) {
                tc_fence_after();
                for (int t = 0; t < ntile; ++t) issue_S(0, t);
            }
        }
        live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
        for (int j = 0; j < n_kv && live; ++j) {
            if (lane == 0) {
                if (j + 1 < n_kv) {
                    const int s1 = (j + 1) % kStages;
                    live = wait_or_abort(&kv_full[s1], (uint32_t)((j + 1) / kStages) & 1u, abort_flag);
                    for (int t = 0; t < ntile && live; ++t) {
                        live = wait_or_abort(&s_free[t], (uint32_t)j & 1u, abort_flag);
                        if (live) {
                            tc_fence_after();
                            issue_S(j + 1, t);
                        }
                    }
                }
            }
            live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
            if (!live) break;
            if (p.paged && j == n_kv - 1 && (j + 1) * kBN > Lk) {
                // the tile landed (every lane observes the barrier), then zero rows >= Lk
                const int s = j % kStages;
                live = wait_or_abort(&kv_full[s], (uint32_t)(j / kStages) & 1u, abort_flag);
                if (__shfl_sync(0xffffffffu, live ? 1 : 0, 0) == 0 || !__all_sync(0xffffffffu, live)) {
                    live = false;
                    break;
                }
                unsigned char *vt = smem + L::kOffKV + s * L::kStage + L::kKTile;
                const int first = Lk - j * kBN;
                for (int r = first; r < kBN; ++r)
                    for (int hf = 0; hf < H; ++hf)
                        *reinterpret_cast<uint32_t *>(vt + hf * kBN * 128 + r * 128 + lane * 4) = 0u;
                fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                for (int t = 0; t < ntile && live; ++t) {
                    live = wait_or_abort(&p_full[t], (uint32_t)j & 1u, abort_flag);
                    if (live) {
                        tc_fence_after();
                        issue_PV(j, t);
                    }
                }
                if (live) umma_commit(&kv_empty[j % kStages]);
            }
            live = __shfl_sync(0xffffffffu, live ? 1 : 0, 0) != 0;
        }
        if (lane == 0) {
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(drain);
            (void)mbar_wait(drain, 0);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------------------
        // softmax warpgroups: thread = query row = TMEM lane
        // ------------------------------------------------------------------
        const int t = warp >> 2;
        if (t < ntile) {
            const int row = tid & (kBM - 1);
            const int qi = r0 + row;                    // query index within the sequence
            const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + lane_base + L::kColS + t * kBN;
            const uint32_t tO = tmem + lane_base + L::kColO + t * HD;
            const uint32_t prow = smem_u32(smem + L::kOffP + t * L::kPTile + row * 128);
            const int sw = row & 7;
            float m = -INFINITY, l = 0.f;
            bool live = true;
            for (int j = 0; j < n_kv; ++j) {
                live = wait_or_abort(&s_full[t], (uint32_t)j & 1u, abort_flag);
                if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                tc_fence_after();
                float s[kBN];
                {
                    float a[32], b[32];
                    tmem_ld32(tS, a);
                    tmem_ld32(tS + 32, b);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        s[c] = a[c];
                        s[32 + c] = b[c];
                    }
                }
                tc_fence_before();
                mbar_arrive(&s_free[t]);
                // scale, causal mask, row maximum
                const int limit = off + qi - j * kBN;   // columns <= limit are visible
                float rmax = -INFINITY;
                if (limit >= kBN - 1) {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        s[c] *= p.scale_log2;
                        rmax = fmaxf(rmax, s[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kBN; ++c) {
                        s[c] = c <= limit ? s[c] * p.scale_log2 : -INFINITY;
                        rmax = fmaxf(rmax, s[c]);
                    }
                }
                const float m_new = fmaxf(m, rmax);
                const bool rescale = (m == -INFINITY) ? (m_new != -INFINITY)
                                                      : (m_new > m + kRescaleThreshold);
                float alpha = 1.f;
                if (rescale) {
                    alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - m_new);
                    m = m_new;
                }
                const float mu = (m == -INFINITY) ? 0.f : m;
                l *= alpha;
                uint32_t pk[kBN / 2];
#pragma unroll
                for (int c = 0; c < kBN; c += 2) {
                    const float e0 = fast_exp2(s[c] - mu);
                    const float e1 = fast_exp2(s[c + 1] - mu);
                    l += e0 + e1;
                    pk[c / 2] = pack_bf16x2(e0, e1);
                }
                // P V of the previous tile must be complete: O is stable and the P buffer is free
                if (j > 0) {
                    live = wait_or_abort(&o_ready[t], (uint32_t)(j - 1) & 1u, abort_flag);
                    if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                    tc_fence_after();
                    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
                        for (int cc = 0; cc < HD / 32; ++cc) {
                            float o[32];
                            tmem_ld32(tO + cc * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(tO + cc * 32, o);
                        }
                    }
                }
#pragma unroll
                for (int c8 = 0; c8 < kBN / 8; ++c8)
                    st_shared_v4(prow + ((c8 ^ sw) << 4), pk[c8 * 4], pk[c8 * 4 + 1], pk[c8 * 4 + 2],
                                 pk[c8 * 4 + 3]);
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&p_full[t]);
            }
            // epilogue: O / l -> bf16 rows, lse
            if (live) live = wait_or_abort(&o_ready[t], (uint32_t)(n_kv - 1) & 1u, abort_flag);
            if (__all_sync(0xffffffffu, live)) {
                tc_fence_after();
                const bool row_ok = qi < Lq;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int hq = h0 + t;
                uint16_t *orow = p.out + (int64_t)(q0 + (row_ok ? qi : 0)) * p.out_rs + (int64_t)hq * HD;
#pragma unroll
                for (int cc = 0; cc < HD / 32; ++cc) {
                    float o[32];
                    tmem_ld32(tO + cc * 32, o);
                    if (row_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint4 pkt;
                            pkt.x = pack_bf16x2(o[v * 8 + 0] * inv, o[v * 8 + 1] * inv);
                            pkt.y = pack_bf16x2(o[v * 8 + 2] * inv, o[v * 8 + 3] * inv);
                            pkt.z = pack_bf16x2(o[v * 8 + 4] * inv, o[v * 8 + 5] * inv);
                            pkt.w = pack_bf16x2(o[v * 8 + 6] * inv, o[v * 8 + 7] * inv);
                            *reinterpret_cast<uint4 *>(orow + cc * 32 + v * 8) = pkt;
                        }
                    }
                }
                if (row_ok && p.lse)
                    p.lse[(int64_t)(q0 + qi) * p.num_heads + hq] =
                        l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int HD>
int launch_hd(const PrefillArgs &a, const PrefillParams &pp, int2 *work, int32_t *count,
              int max_items, cudaStream_t stream, const char **err) {
    using L = PLayout<HD>;
    CUtensorMap qm, km, vm;
    int rc = encode_rows_heads_map(&qm, a.q, a.total_q, a.num_heads, HD, a.q_rs, HD, 64, kBM, true, err);
    if (rc) return rc;
    if (pp.paged) {
        const int64_t slots = a.num_blocks * a.block_size;
        const int tb = a.block_size < kBN ? a.block_size : kBN;
        const int64_t D = (int64_t)a.num_kv_heads * HD;
        rc = encode_rows_heads_map(&km, a.k_cache, slots, a.num_kv_heads, HD, D, HD, 64, tb, true, err);
        if (!rc) rc = encode_rows_heads_map(&vm, a.v_cache, slots, a.num_kv_heads, HD, D, HD, 64, tb, true, err);
    } else {
        rc = encode_rows_heads_map(&km, a.k, a.total_k, a.num_kv_heads, HD, a.k_rs, HD, 64, kBN, true, err);
        if (!rc) rc = encode_rows_heads_map(&vm, a.v, a.total_k, a.num_kv_heads, HD, a.v_rs, HD, 64, kBN, true, err);
    }
    if (rc) return rc;
    prefill_plan_kernel<<<1, 1024, 0, stream>>>(pp, count, work);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    const int smem = L::kBytes + 1024;
    auto kern = prefill_kernel<HD>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    const int G = a.num_heads / a.num_kv_heads;
    const int ntile = G >= 2 ? 2 : 1;
    dim3 grid(a.num_heads / ntile, max_items);
    kern<<<grid, kThreads, smem, stream>>>(qm, km, vm, pp);
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    return PKV_OK;
}

int max_work_items(int32_t num_seqs, int32_t total_q) {
    return num_seqs + (total_q + kBM - 1) / kBM;
}

}  // namespace

size_t prefill_workspace_bytes(int32_t num_seqs, int32_t total_q, int32_t max_seqlen_q,
                               int32_t num_heads) {
    (void)max_seqlen_q;
    (void)num_heads;
    return 256 + sizeof(int2) * (size_t)max_work_items(num_seqs, total_q);
}

int launch_prefill(const PrefillArgs &a, cudaStream_t stream, const char **err) {
    if (a.head_dim != 64 && a.head_dim != 128) {
        *err = "head_dim must be 64 or 128";
        return PKV_ERR_UNSUPPORTED;
    }
    const int G = a.num_heads / a.num_kv_heads;
    if (G > 1 && G % 2) {
        *err = "num_heads / num_kv_heads must be 1 or even";
        return PKV_ERR_UNSUPPORTED;
    }
    const bool paged = a.bt != nullptr;
    if (paged && (a.block_size < 8 || (a.block_size & (a.block_size - 1)))) {
        *err = "paged prefill needs a power-of-two block_size >= 8";
        return PKV_ERR_UNSUPPORTED;
    }
    const size_t need = prefill_workspace_bytes(a.num_seqs, a.total_q, a.max_seqlen_q, a.num_heads);
    if (!a.workspace || a.workspace_bytes < need) {
        *err = "workspace smaller than paged_attn_prefill_workspace_size()";
        return PKV_ERR_WORKSPACE;
    }
    const int max_items = max_work_items(a.num_seqs, a.total_q);
    if (max_items > 65535) {
        *err = "too many 128-row query blocks for one launch";
        return PKV_ERR_UNSUPPORTED;
    }
    int32_t *count = reinterpret_cast<int32_t *>(a.workspace);
    int2 *work = reinterpret_cast<int2 *>(reinterpret_cast<unsigned char *>(a.workspace) + 256);
    PrefillParams pp{};
    pp.cu_q = a.cu_q;
    pp.cu_k = a.cu_k;
    pp.bt = a.bt;
    pp.bt_stride = a.bt_stride;
    pp.max_blocks = a.max_blocks;
    pp.num_blocks = a.num_blocks;
    pp.block_size = paged ? a.block_size : 1;
    pp.num_seqs = a.num_seqs;
    pp.num_heads = a.num_heads;
    pp.num_kv_heads = a.num_kv_heads;
    pp.paged = paged ? 1 : 0;
    pp.scale_log2 = a.scale * kLog2e;
    pp.out = a.out;
    pp.out_rs = a.out_rs;
    pp.lse = a.lse;
    pp.work_count = count;
    pp.work = work;
    pp.max_items = max_items;
    if (a.head_dim == 128) return launch_hd<128>(a, pp, work, count, max_items, stream, err);
    return launch_hd<64>(a, pp, work, count, max_items, stream, err);
}

}  // namespace pkv
