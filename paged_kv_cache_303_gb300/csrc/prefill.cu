// prefill.cu -- varlen causal paged prefill on the 5th-generation tensor
// cores (tcgen05 + tensor memory), for plain prefill (keys from the packed
// k/v of the step) and prefix-cache prefill (keys through block_tables from
// the paged cache).  L17: Qwen3 attention sub-layer, §5.2 (blocked softmax
// with exact rescaling) and §5.3 (the varlen call, causal=True, and its
// prefix-cache branch); Lesson 04, §4.
//
// Work unit: (128 query rows of one sequence, two query heads of one GQA
// group).  The two heads share every K/V tile the unit loads, which halves
// K/V traffic per FLOP compared with one head per unit.  When the group size
// is odd a unit takes one head (the second softmax warpgroup idles).  A block
// of at most 64 rows (a sequence's last block, or a short sequence) carries
// both heads in one 128-row tile, 64 rows each, so its half-empty rows are
// not computed twice.
//
// Persistent CTAs, one per SM, each running units until none is left: a
// unit's set-up (Q and first K/V loads, first S products) overlaps the
// previous unit's last tiles and epilogue, and TMEM, barriers and tensor-map
// prefetches are set up once per SM instead of once per unit.
//
// Roles (384 threads; the softmax warpgroups run with 208 registers a thread,
// the other four warps with 80, by setmaxnreg):
//   warps 0-3  softmax warpgroup of query head A, thread = query row = TMEM lane
//   warps 4-7  softmax warpgroup of query head B
//   warp 8     producer: per unit K_0, V_0, Q, K_1, V_1, ... (128 keys a
//              tile) through a ring of kSlots tiles numbered across units
//              (packed k/v: one TMA box per 64 columns of head_dim; paged
//              cache: one box per block segment, addressed via block_tables;
//              blocks shorter than 8 rows are copied row by row with cp.async
//              into the same layout)
//   warp 9     MMA issuer (one lane): S_A(0), S_B(0), then per key tile j
//              P_A(j) V_j, S_A(j+1), P_B(j) V_j, S_B(j+1), so the tensor core
//              works on one head while the other head's softmax runs
//   warp 10    idle (completes the third warpgroup for the register split)
//   warp 11    scheduler (one lane): claims the next unit once the producer
//              has issued the current one's loads, and publishes units to the
//              other roles through two shared-memory records
//
// Tensor memory (fp32 accumulators, lane = query row), 512 columns: S of
// head t at 128 t (P, bf16 pairs, written over its upper 64 columns and
// read from there as the A operand of P V), O of head t at 256 + d t.
//
// Shared-memory operands use the 128-byte swizzle written by TMA: Q and K
// are K-major, V is read as an MN-major B operand (keys are K, head_dim N).
//
// Softmax: per row, scores are scaled by scale*log2(e) and exponentiated
// with exp2.  The running maximum is only moved when a tile's maximum
// exceeds it by more than 8 (a factor 256): then l and the O accumulator
// in TMEM are rescaled by 2^(m_old - m_new) (§5.2's identity), after the
// earlier P V products have landed.  Otherwise the stale maximum is kept;
// every p is then <= 2^8, and the final O / l uses the same maximum for
// numerator and denominator, so the result is the same softmax.
//
// Causality: query row t of a sequence with Lq queries and Lk keys sees keys
// j <= Lk - Lq + t.  KV tiles past the last row's bound are never loaded;
// only tiles that cross a row's bound are masked.  In paged mode the value
// rows past Lk of the last tile are zeroed in shared memory before P V, so
// unwritten cache slots (possibly NaN) never meet a zero probability.
//
// A one-CTA planning kernel lists the (sequence, 128-row block) work items
// in decreasing order of key tiles (longest first) in the workspace, each as
// a record of everything a unit needs to start (offsets, lengths, key
// tiles), and zeroes the claim counter; the prefill kernel is its
// programmatic dependent and reads the list after griddepcontrol.wait, its
// set-up overlapping the planning.  Units are items x head pairs, item-major.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace pkv {

static __device__ unsigned int g_prefill_status;

#if PKV_TEST_HOOKS
// Test-only build: while set, the scheduler of CTA 0 publishes no unit at
// all, so that CTA's other roles wait on the first unit record until the
// bound runs out.  Nothing has been issued by then (no copy, no tensor-core
// product), so every role leaves with nothing in flight.
static __device__ int g_test_withhold_prefill_unit;

int test_withhold_prefill_unit(int on) {
    return cudaMemcpyToSymbol(g_test_withhold_prefill_unit, &on, sizeof on) == cudaSuccess ? 0 : -1;
}
#endif

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
constexpr int kBN = 128;          // keys per KV tile
constexpr int kSlots = 5;         // ring of K / V tiles (K_j, V_j, K_j+1, ...)
constexpr int kThreads = 384;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSchedWarp = 11;   // warp 10 only fills the register-split warpgroup
constexpr int kUnitSlots = 2;     // published work units (double-buffered)
constexpr int kUnitUsers = 10;    // roles done with a unit: 8 softmax warps, producer, MMA
// registers per thread after the split: softmax warpgroups / the other four warps
// (8*32*208 + 4*32*80 = 63488 <= 384 threads * 168 at launch)
constexpr int kRegsSoftmax = 208;
constexpr int kRegsOther = 80;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr int kCostBins = 2048;
constexpr int kPlanThreads = 1024;
constexpr int kPlanSeqs = 1024;   // sequences whose lengths the planning kernel keeps on chip
constexpr int kColP = kBN / 2;
#ifndef PKV_PF_PDL
#define PKV_PF_PDL 1   // prefill kernel launched as a programmatic dependent of the planning kernel
#endif
#ifndef PKV_PF_OUT_V8
#define PKV_PF_OUT_V8 1   // 32-byte output stores when the output rows are 32-byte aligned
#endif
#ifndef PKV_PF_PACK
#define PKV_PF_PACK 1   // blocks of at most 64 rows carry both heads of a pair in one tile
#endif    // P (bf16 pairs) over the upper half of a head's S columns

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

// 128 consecutive TMEM columns of this warp's 32 lanes -> 128 registers (waits)
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr), "r"(taddr + 64u)
        : "memory");
}

// 64 consecutive TMEM columns of this warp's lanes -> 64 registers (waits)
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr)
        : "memory");
}

// a row's HD output columns in one go (one wait instead of one per 32)
template <int HD>
__device__ __forceinline__ void tmem_ld_row(uint32_t taddr, uint32_t (&r)[HD]) {
    if constexpr (HD == 128) {
        tmem_ld128(taddr, r);
    } else {
        tmem_ld64(taddr, r);
    }
}

// 32 registers -> 32 consecutive TMEM columns of this warp's lanes (no wait)
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// One softmax pass over a row's 128 scores: p = 2^(s*sc - mu) as bf16 pairs
// stored over the row's upper 64 S columns (not waited for), and the row sum
// of p in acc.
__device__ __forceinline__ void exp_pack_store(const uint32_t (&sr)[kBN], float sc, float mu,
                                               uint32_t tS, float2 (&acc)[2]) {
    const float2 sc2 = make_float2(sc, sc);
    const float2 nm2 = make_float2(-mu, -mu);
    acc[0] = acc[1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int hpart = 0; hpart < 2; ++hpart) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int col = hpart * 64 + 2 * c;
            const float2 x = ffma2(make_float2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])),
                                   sc2, nm2);
            const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            acc[c & 1] = fadd2(acc[c & 1], e);
            pk[c] = pack_bf16x2(e.x, e.y);
        }
        tmem_st32_nowait(tS + kColP + hpart * 32, pk);
    }
}

// D (TMEM) += A (TMEM, K-major) * B (shared memory descriptor)
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Wait that gives up when another role has aborted, or after the time bound
// (then it raises the abort flag itself).
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
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
    int32_t *claim;              // [1] next unit to claim, less the grid size (zeroed by the plan)
    // [max_items][2]: {sequence, 128-row block, first query row, query rows},
    // {first key row, keys, key tiles, 0} -- everything a CTA needs to start
    const int4 *work;
    int32_t max_items;
    // paged mode with blocks shorter than the 8-row swizzle atom: K/V tiles
    // are copied row by row from the caches instead of by TMA boxes
    int32_t row_copy;
    const uint16_t *k_cache, *v_cache;
    int32_t out_v8;              // out and its row stride allow 32-byte stores
};

__device__ __forceinline__ int kv_tiles_for(int Lq, int Lk, int mb) {
    const int t_last = min(Lq, (mb + 1) * kBM) - 1;
    const int keys = Lk - Lq + t_last + 1;
    return (keys + kBN - 1) / kBN;
}

// Work list: every (sequence, 128-row block), ordered by decreasing number
// of key tiles (a counting sort on the cost).  One CTA: a warp per sequence,
// lanes over its row blocks; one warp scans the bins in use, 32 at a time.
__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(PrefillParams p, int32_t *work_count,
                                                            int4 *work) {
    __shared__ int hist[kCostBins];
    __shared__ int top;                         // highest cost bin in use
    __shared__ int4 seqs[kPlanSeqs];            // {first query row, query rows, first key row, keys}
#if PKV_PF_PDL
    // the prefill kernel may start its set-up now; it waits for this grid
    // (and its writes) before reading the work list
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int i = threadIdx.x; i < kCostBins; i += blockDim.x) hist[i] = 0;
    if (threadIdx.x == 0) top = 0;
    __syncthreads();
    // pass 1: cost histogram; each sequence's offsets and lengths are kept
    // for pass 2 (in shared memory for the first kPlanSeqs sequences)
    for (int s = warp; s < p.num_seqs; s += nwarps) {
        const int q0 = p.cu_q[s], k0 = p.cu_k[s];
        const int Lq = p.cu_q[s + 1] - q0, Lk = p.cu_k[s + 1] - k0;
        if (s < kPlanSeqs && lane == 0) seqs[s] = make_int4(q0, Lq, k0, Lk);
        if (Lq <= 0) continue;
        if (Lk < Lq) {
            if (lane == 0) atomicOr(&g_prefill_status, PKV_STATUS_BAD_LENGTH);
            continue;
        }
        const int nmb = (Lq + kBM - 1) / kBM;
        for (int mb = lane; mb < nmb; mb += 32)
            atomicAdd(&hist[min(kv_tiles_for(Lq, Lk, mb), kCostBins - 1)], 1);
        if (lane == 0) atomicMax(&top, min(kv_tiles_for(Lq, Lk, nmb - 1), kCostBins - 1));
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive prefix sums in descending cost: each bin's first position
        int run = 0;
        for (int hi = top; hi >= 0; hi -= 32) {
            const int c = hi - lane;                    // lane 0: the chunk's highest bin
            const int h = c >= 0 ? hist[c] : 0;
            int x = h;                                  // inclusive scan over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (c >= 0) hist[c] = run + x - h;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            if (run > p.max_items) atomicOr(&g_prefill_status, PKV_STATUS_BAD_LENGTH);
            *work_count = min(run, p.max_items);
            *p.claim = 0;
        }
    }
    __syncthreads();
    // pass 2: each item's record at the next position of its cost bin
    for (int s = warp; s < p.num_seqs; s += nwarps) {
        int4 sq;
        if (s < kPlanSeqs) {
            sq = seqs[s];
        } else {
            const int q0 = p.cu_q[s], k0 = p.cu_k[s];
            sq = make_int4(q0, p.cu_q[s + 1] - q0, k0, p.cu_k[s + 1] - k0);
        }
        const int q0 = sq.x, Lq = sq.y, k0 = sq.z, Lk = sq.w;
        if (Lq <= 0 || Lk < Lq) continue;
        const int nmb = (Lq + kBM - 1) / kBM;
        for (int mb = lane; mb < nmb; mb += 32) {
            const int nkv = kv_tiles_for(Lq, Lk, mb);
            const int pos = atomicAdd(&hist[min(nkv, kCostBins - 1)], 1);
            if (pos < p.max_items) {
                work[2 * pos] = make_int4(s, mb, q0, Lq);
                work[2 * pos + 1] = make_int4(k0, Lk, nkv, 0);
            }
        }
    }
}

template <int HD>
struct PLayout {
    static constexpr int H = HD / 64;                       // 128-byte halves of a row
    static constexpr int kQTile = H * kBM * 128;            // one query head's tile
    static constexpr int kKVTile = H * kBN * 128;           // one K or V tile (a ring slot)
    static constexpr int kOffRing = 2 * kQTile;
    static constexpr int kOffBar = kOffRing + kSlots * kKVTile;
    static constexpr int kOffUnits = kOffBar + 256;         // kUnitSlots work units, 32 bytes each
    static constexpr int kBytes = kOffBar + 512;
    static constexpr int kTmemCols = 512;
    static constexpr int kColS = 0;                         // S/P of head t at t * kBN
    static constexpr int kColO = 2 * kBN;                   // O of head t at kColO + t * HD
    static_assert(kColO + 2 * HD <= kTmemCols, "tensor memory");
};

// A work unit as the scheduler warp publishes it: the item's record (see the
// planning kernel) with the head pair in the last field; a negative head pair
// ends the CTA's loop.
struct Unit {
    int seq, mb, q0, Lq, k0, Lk, n_kv, hp;
};
__device__ __forceinline__ Unit read_unit(const int4 *units, int slot) {
    const int4 a = units[2 * slot], b = units[2 * slot + 1];
    return Unit{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
}

// Q of a unit: both heads' 128-row tiles, or (packed) both heads' 64 rows in
// one tile
template <int HD>
__device__ __forceinline__ void load_q_tiles(unsigned char *smem, const CUtensorMap *qmap,
                                             const CUtensorMap *qmap64, uint64_t *q_full, bool packed,
                                             int pair, int h0, int row0, uint64_t pol) {
    using L = PLayout<HD>;
    const int ntile = packed ? 1 : pair;
    mbar_arrive_expect_tx(q_full, (uint32_t)(ntile * L::kQTile));
    if (packed) {
        for (int t = 0; t < 2; ++t)
            for (int hf = 0; hf < L::H; ++hf)
                tma_load_3d(smem + hf * kBM * 128 + t * (kBM / 2) * 128, qmap64, q_full, hf * 64, h0 + t,
                            row0, pol);
    } else {
        for (int t = 0; t < ntile; ++t)
            for (int hf = 0; hf < L::H; ++hf)
                tma_load_3d(smem + t * L::kQTile + hf * kBM * 128, qmap, q_full, hf * 64, h0 + t, row0, pol);
    }
}

// L2 policy of the K/V tile loads: every later block of the sequence reads
// the same tiles (Q, read once, keeps evict_first)
__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 32 bytes to global memory, streaming (written once)
__device__ __forceinline__ void st_cs_v8(void *p, const uint32_t (&w)[8]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

template <int N>
__device__ __forceinline__ void regs_raise() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_lower() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap qmap64,
               const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const PrefillParams p) {
    using L = PLayout<HD>;
    constexpr int H = L::H;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *q_full = bars + 0;               // Q of the current unit landed
    uint64_t *q_free = q_full + 1;             // the unit's last S products have read Q
    uint64_t *slot_full = q_free + 1;          // [kSlots] a K or V tile landed
    uint64_t *slot_free = slot_full + kSlots;  // [kSlots] its MMAs are done with it
    uint64_t *s_full = slot_free + kSlots;     // [2] S of head t in TMEM
    uint64_t *p_full = s_full + 2;             // [2] P of head t in TMEM (4 warp arrivals)
    uint64_t *o_done = p_full + 2;             // [2] P V of head t complete
    uint64_t *unit_full = o_done + 2;          // [kUnitSlots] a unit published
    uint64_t *unit_empty = unit_full + kUnitSlots;   // [kUnitSlots] every role is done with it
    uint64_t *loads_done = unit_empty + kUnitSlots;  // the producer issued a unit's last load
    uint64_t *drain = loads_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int4 *units = reinterpret_cast<int4 *>(smem + L::kOffUnits);
    static_assert((2 * kSlots + 10 + 2 * kUnitSlots) * 8 + 8 <= L::kOffUnits - L::kOffBar,
                  "barriers run into the unit records");

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, L::kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_free, 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(&slot_full[s], 1);
            mbar_init(&slot_free[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 4);
            mbar_init(&o_done[t], 1);
        }
        for (int s = 0; s < kUnitSlots; ++s) {
            mbar_init(&unit_full[s], 1);
            mbar_init(&unit_empty[s], kUnitUsers);
        }
        mbar_init(loads_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&qmap64);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
#if PKV_PF_PDL
    // the work list is written by the planning kernel launched just before
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int G = p.num_heads / p.num_kv_heads;
    const int pair = G % 2 == 0 ? 2 : 1;         // two heads of one group, or one head
    // A block with at most 64 query rows (the last block of a sequence, or a
    // short one) holds both heads in one 128-row tile: head h0 in rows 0..63,
    // head h0+1 in rows 64..127.  The two heads share every K/V tile, so one
    // S and one P V stream cover both and the half-empty rows are not
    // computed twice.
    auto is_packed = [&](const Unit &U) {
        return PKV_PF_PACK && pair == 2 && U.Lq - U.mb * kBM <= kBM / 2;
    };

    if (warp >= 8) {
        // the four single-lane roles give registers to the softmax warpgroups
        // (one setmaxnreg per warpgroup, executed by all its warps)
        regs_lower<kRegsOther>();
        if (warp == kSchedWarp) {
            // ------------------------------------------------------------------
            // Scheduler (one lane): the CTA's first unit is its index; each later
            // one is claimed from a counter once the producer has issued the
            // current unit's last load (a few tiles before the SM runs out of
            // work), so units run longest first in about the order the SMs
            // become free.  A unit is (work item, head pair), items in the
            // planning kernel's order.
            // ------------------------------------------------------------------
            if (lane == 0) {
                const int npairs = p.num_heads / pair;
                const int total = *p.work_count * npairs;
                int unit = blockIdx.x;
                for (int u = 0;; ++u) {
                    const int slot = u % kUnitSlots;
                    if (u > 0) {
                        if (!wait_or_abort(loads_done, (uint32_t)(u - 1) & 1u, abort_flag)) break;
                        unit = atomicAdd(p.claim, 1) + (int)gridDim.x;
                    }
                    int4 a = make_int4(0, 0, 0, 0), b = make_int4(0, 0, 0, -1);
                    if (unit < total) {
                        const int item = unit / npairs;
                        a = p.work[2 * item];
                        b = p.work[2 * item + 1];
                        b.w = unit - item * npairs;
                    }
                    if (u >= kUnitSlots &&
                        !wait_or_abort(&unit_empty[slot], (uint32_t)((u / kUnitSlots) - 1) & 1u, abort_flag))
                        break;
#if PKV_TEST_HOOKS
                    if (u == 0 && blockIdx.x == 0 && g_test_withhold_prefill_unit) break;
#endif
                    units[2 * slot] = a;
                    units[2 * slot + 1] = b;
                    mbar_arrive(&unit_full[slot]);
                    if (b.w < 0) break;
                }
            }
        } else if (warp == kProducerWarp && p.row_copy) {
            // ------------------------------------------------------------------
            // Producer for paged caches whose blocks are shorter than the 8-row
            // swizzle atom (block_size 1, 2, 4): Q by TMA as usual; each K / V
            // tile is copied by the whole warp in 16-byte pieces with cp.async,
            // row by row through block_tables, into the same 128-byte-swizzled
            // layout a TMA box writes.  Rows past the last key and rows of
            // missing blocks are zero-filled, so the final tile needs no fix-up.
            // A tile is published (slot_full) once the next one is in flight:
            // every lane waits for its own pieces, fences them into the async
            // proxy that the tensor core reads through, then lane 0 arrives.
            // Loads are numbered across the CTA's units (load n -> slot n % kSlots).
            // ------------------------------------------------------------------
            constexpr int CPR = HD / 8;                  // 16-byte pieces per row
            const int bs = p.block_size;
            const int64_t row_elems = (int64_t)p.num_kv_heads * HD;
            const uint64_t pol = policy_evict_first();
            bool live = true;
            int n = 0, nq = 0;
            for (int u = 0; live; ++u) {
                const int slot = u % kUnitSlots;
                live = wait_or_abort(&unit_full[slot], (uint32_t)(u / kUnitSlots) & 1u, abort_flag);
                if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                const Unit U = read_unit(units, slot);
                if (U.hp < 0) break;
                const int h0 = U.hp * pair, kvh = h0 / G;
                const bool packed = is_packed(U);
                const int32_t *bt_row = p.bt + (int64_t)U.seq * p.bt_stride;
                // Q after the unit's first K (and V) tile: it waits for the
                // previous unit's last S products
                const int q_at = u == 0 ? 0 : min(2, 2 * U.n_kv - 1);
                for (int i = 0; i < 2 * U.n_kv; ++i, ++n) {
                    if (i == q_at) {
                        int ok = 1;
                        if (lane == 0) {
                            ok = (u == 0 || wait_or_abort(q_free, (uint32_t)(u - 1) & 1u, abort_flag)) ? 1 : 0;
                            if (ok) load_q_tiles<HD>(smem, &qmap, &qmap64, q_full, packed, pair, h0, U.q0 + U.mb * kBM, pol);
                        }
                        if (!__shfl_sync(0xffffffffu, ok, 0)) { live = false; break; }
                        ++nq;
                    }
                    const int s = n % kSlots;
                    const int j = i >> 1;
                    const uint16_t *cache = (i & 1) ? p.v_cache : p.k_cache;
                    if (n >= kSlots) {
                        int ok = 1;
                        if (lane == 0)
                            ok = wait_or_abort(&slot_free[s], (uint32_t)((n / kSlots) - 1) & 1u, abort_flag) ? 1 : 0;
                        if (!__shfl_sync(0xffffffffu, ok, 0)) { live = false; break; }
                    }
                    const uint32_t dst = smem_u32(smem + L::kOffRing + s * L::kKVTile);
                    bool missing = false;
                    for (int pc = lane; pc < kBN * CPR; pc += 32) {
                        const int r = pc / CPR, cc = pc % CPR;
                        const int pos = j * kBN + r;
                        const uint16_t *src = cache;
                        uint32_t nbytes = 0;
                        if (pos < U.Lk) {
                            const int lb = pos / bs;
                            const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                            if (blk >= 0 && blk < p.num_blocks) {
                                src = cache + ((int64_t)blk * bs + pos % bs) * row_elems + (int64_t)kvh * HD + cc * 8;
                                nbytes = 16;
                            } else {
                                missing = true;
                            }
                        }
                        cp_async16(dst + (uint32_t)((cc / 8) * (kBN * 128) + r * 128 + (((cc % 8) ^ (r & 7)) << 4)),
                                   src, nbytes);
                    }
                    cp_async_commit();
                    if (missing && !(i & 1)) atomicOr(&g_prefill_status, PKV_STATUS_BAD_BLOCK);
                    if (n > 0) {
                        cp_async_wait<1>();              // this lane's pieces of load n-1 landed
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&slot_full[(n - 1) % kSlots]);
                    }
                }
                if (!live) break;
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(loads_done);
                    mbar_arrive(&unit_empty[slot]);
                }
            }
            cp_async_wait<0>();                          // nothing may land after the CTA leaves
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (live && n > 0) mbar_arrive(&slot_full[(n - 1) % kSlots]);
                if (nq > 0) (void)mbar_wait(q_full, (uint32_t)(nq - 1) & 1u);
            }
        } else if (warp == kProducerWarp) {
            // ------------------------------------------------------------------
            // TMA producer (one lane): per unit the loads K_0, V_0, K_1, V_1, ...
            // into a ring of kSlots tiles, numbered across the CTA's units (load
            // n -> slot n % kSlots); Q of a unit after its first K/V pair, once
            // the previous unit's last S products have read the Q buffer.
            // ------------------------------------------------------------------
            if (lane == 0) {
                const uint64_t pol = policy_evict_first();
                const uint64_t kvpol = policy_evict_normal();
                const int bs = p.block_size;
                const int TB = p.paged ? (bs < kBN ? bs : kBN) : kBN;
                bool live = true;
                int n = 0, nq = 0;
                for (int u = 0; live; ++u) {
                    const int slot = u % kUnitSlots;
                    if (!wait_or_abort(&unit_full[slot], (uint32_t)(u / kUnitSlots) & 1u, abort_flag)) break;
                    const Unit U = read_unit(units, slot);
                    if (U.hp < 0) break;
                    const int h0 = U.hp * pair, kvh = h0 / G;
                    const bool packed = is_packed(U);
                    const int32_t *bt_row = p.paged ? p.bt + (int64_t)U.seq * p.bt_stride : nullptr;
                    const int q_at = u == 0 ? 0 : min(2, 2 * U.n_kv - 1);
                    for (int i = 0; i < 2 * U.n_kv; ++i, ++n) {
                        if (i == q_at) {
                            if (u > 0 && !wait_or_abort(q_free, (uint32_t)(u - 1) & 1u, abort_flag)) {
                                live = false;
                                break;
                            }
                            load_q_tiles<HD>(smem, &qmap, &qmap64, q_full, packed, pair, h0, U.q0 + U.mb * kBM, pol);
                            ++nq;
                        }
                        const int s = n % kSlots;
                        const int j = i >> 1;
                        const CUtensorMap *map = (i & 1) ? &vmap : &kmap;
                        if (n >= kSlots &&
                            !wait_or_abort(&slot_free[s], (uint32_t)((n / kSlots) - 1) & 1u, abort_flag)) {
                            live = false;
                            break;
                        }
                        unsigned char *dst = smem + L::kOffRing + s * L::kKVTile;
                        if (!p.paged) {
                            mbar_arrive_expect_tx(&slot_full[s], (uint32_t)L::kKVTile);
                            for (int hf = 0; hf < H; ++hf)
                                tma_load_3d(dst + hf * kBN * 128, map, &slot_full[s], hf * 64, kvh,
                                            U.k0 + j * kBN, kvpol);
                        } else {
                            const int nseg = kBN / TB;
                            int ok = 0;
                            for (int sg = 0; sg < nseg; ++sg) {
                                const int pos = j * kBN + sg * TB;
                                if (pos >= U.Lk) break;
                                const int lb = pos / bs;
                                const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                                if (blk >= 0 && blk < p.num_blocks) ++ok;
                            }
                            mbar_arrive_expect_tx(&slot_full[s], (uint32_t)(ok * H * TB * 128));
                            for (int sg = 0; sg < nseg; ++sg) {
                                const int pos = j * kBN + sg * TB;
                                if (pos >= U.Lk) break;
                                const int lb = pos / bs;
                                const int blk = lb < p.max_blocks ? bt_row[lb] : -1;
                                if (blk < 0 || blk >= p.num_blocks) {
                                    if (!(i & 1)) atomicOr(&g_prefill_status, PKV_STATUS_BAD_BLOCK);
                                    continue;
                                }
                                const int z = (int)((int64_t)blk * bs + pos % bs);
                                for (int hf = 0; hf < H; ++hf)
                                    tma_load_3d(dst + hf * kBN * 128 + sg * TB * 128, map, &slot_full[s],
                                                hf * 64, kvh, z, kvpol);
                            }
                        }
                    }
                    if (!live) break;
                    mbar_arrive(loads_done);
                    mbar_arrive(&unit_empty[slot]);
                }
                // no copy may still be landing when the CTA leaves: every load
                // before the last kSlots was waited for by the MMA thread before
                // its slot was released, and every Q before the last one before
                // q_free
                for (int m = n - kSlots < 0 ? 0 : n - kSlots; m < n; ++m)
                    (void)mbar_wait(&slot_full[m % kSlots], (uint32_t)(m / kSlots) & 1u);
                if (nq > 0) (void)mbar_wait(q_full, (uint32_t)(nq - 1) & 1u);
            }
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------------
            // MMA issuer (lane 0).  Per unit: S_A(0), S_B(0), then per tile j:
            // P_A(j) V_j, S_A(j+1), P_B(j) V_j, S_B(j+1) -- the tensor core works
            // on one head while the other head's softmax runs.  P is read from
            // tensor memory (it overwrites the head's S columns), V and K/Q from
            // shared memory.  The next unit's first S products follow the last
            // P V products in the tensor pipe, which has then read every P.
            // ------------------------------------------------------------------
            constexpr uint32_t kIdS = idesc_bf16(kBM, kBN, false);
            constexpr uint32_t kIdO = idesc_bf16(kBM, HD, true);
            const uint32_t sbase = smem_u32(smem);
            const uint32_t ring = sbase + L::kOffRing;
            auto issue_S = [&](int s, int t) {
                const uint64_t a0 = sdesc_sw128(sbase + t * L::kQTile, 16, 1024);
                const uint64_t b0 = sdesc_sw128(ring + s * L::kKVTile, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t step = (uint32_t)(((kk / 4) * kBN * 128 + (kk % 4) * 32) >> 4);
                    const uint32_t astep = (uint32_t)(((kk / 4) * kBM * 128 + (kk % 4) * 32) >> 4);
                    umma_bf16(tmem + L::kColS + t * kBN, a0 + astep, b0 + step, kIdS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[t]);
            };
            auto issue_PV = [&](int s, int t, bool first) {
                const uint64_t b0 = sdesc_sw128(ring + s * L::kKVTile, kBN * 128, 1024);
                const uint32_t a_tm = tmem + L::kColS + t * kBN + kColP;   // P: kBN/2 columns
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    umma_bf16_ts(tmem + L::kColO + t * HD, a_tm + kk * 8, b0 + (uint32_t)((kk * 16 * 128) >> 4),
                                 kIdO, (!first || kk > 0) ? 1u : 0u);
                umma_commit(&o_done[t]);
            };
            if (lane == 0) {
                bool live = true;
                int n0 = 0;                  // load index of the unit's K_0
                uint32_t ppar = 0;           // bit t: parity of head slot t's tile count
                for (int u = 0; live; ++u) {
                    const int slot = u % kUnitSlots;
                    if (!wait_or_abort(&unit_full[slot], (uint32_t)(u / kUnitSlots) & 1u, abort_flag)) break;
                    const Unit U = read_unit(units, slot);
                    if (U.hp < 0) break;
                    const int ntile = is_packed(U) ? 1 : pair;
                    live = wait_or_abort(q_full, (uint32_t)u & 1u, abort_flag) &&
                           wait_or_abort(&slot_full[n0 % kSlots], (uint32_t)(n0 / kSlots) & 1u, abort_flag);
                    if (!live) break;
                    tc_fence_after();
                    for (int t = 0; t < ntile; ++t) issue_S(n0 % kSlots, t);
                    if (U.n_kv == 1) umma_commit(q_free);
                    umma_commit(&slot_free[n0 % kSlots]);
                    for (int j = 0; j < U.n_kv && live; ++j) {
                        const int nv = n0 + 2 * j + 1;              // load index of V_j
                        const int sv = nv % kSlots;
                        const bool next = j + 1 < U.n_kv;
                        const int nk = nv + 1;                      // load index of K_{j+1}
                        // (a paged unit's last V tile has its rows past the
                        // last key zeroed by softmax warpgroup 0 before its
                        // P arrival, which P_A V waits for)
                        live = wait_or_abort(&slot_full[sv], (uint32_t)(nv / kSlots) & 1u, abort_flag);
                        // K_{j+1} too, while the tensor pipe still works through
                        // the previous tile's last S products
                        if (live && next)
                            live = wait_or_abort(&slot_full[nk % kSlots], (uint32_t)(nk / kSlots) & 1u, abort_flag);
                        for (int t = 0; t < ntile && live; ++t) {
                            live = wait_or_abort(&p_full[t], (ppar >> t) & 1u, abort_flag);
                            if (!live) break;
                            ppar ^= 1u << t;
                            tc_fence_after();
                            issue_PV(sv, t, j == 0);
                            if (next) issue_S(nk % kSlots, t);
                        }
                        if (live) {
                            if (j + 2 == U.n_kv) umma_commit(q_free);       // the unit's last S products
                            umma_commit(&slot_free[sv]);                    // V_j
                            if (next) umma_commit(&slot_free[nk % kSlots]); // K_{j+1}
                        }
                    }
                    n0 += 2 * U.n_kv;
                    if (live) mbar_arrive(&unit_empty[slot]);
                }
                // every MMA issued by this thread has completed before TMEM is released
                umma_commit(drain);
                (void)mbar_wait(drain, 0);
            }
            __syncwarp();
        }
    } else {
        regs_raise<kRegsSoftmax>();
        // ------------------------------------------------------------------
        // softmax warpgroups: thread = query row = TMEM lane; warpgroup t
        // takes head h0 + t of each unit (both heads of a packed unit in
        // warpgroup 0)
        // ------------------------------------------------------------------
        const int t = warp >> 2;
        const int row = tid & (kBM - 1);
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + L::kColS + t * kBN;
        const uint32_t tO = tmem + lane_base + L::kColO + t * HD;
        const float sc = p.scale_log2;
        uint32_t jpar = 0;              // parity of this head slot's tile count
        int n0 = 0;                     // load index of the unit's K_0
        bool live = true;
        for (int u = 0; live; ++u) {
            const int slot = u % kUnitSlots;
            live = wait_or_abort(&unit_full[slot], (uint32_t)(u / kUnitSlots) & 1u, abort_flag);
            if (!__all_sync(0xffffffffu, live)) { live = false; break; }
            const Unit U = read_unit(units, slot);
            if (U.hp < 0) break;
            const bool packed = is_packed(U);
            const int ntile = packed ? 1 : pair;
            const int nv_last = n0 + 2 * U.n_kv - 1;      // load index of the unit's last V tile
            n0 += 2 * U.n_kv;
            if (t < ntile) {
                const int r0 = U.mb * kBM;
                const int off = U.Lk - U.Lq;
                // query index within the sequence (packed: rows 64.. are head h0+1)
                const int qi = r0 + (packed ? (row & (kBM / 2 - 1)) : row);
                float m = -INFINITY, l = 0.f;
                for (int j = 0; j < U.n_kv; ++j) {
                    live = wait_or_abort(&s_full[t], jpar, abort_flag);
                    if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                    jpar ^= 1u;
                    tc_fence_after();
                    // scores of the tile, with the causal mask on the tiles
                    // that cross the row's bound
                    const int limit = off + qi - j * kBN;   // columns <= limit are visible
                    uint32_t sr[kBN];
                    tmem_ld128(tS, sr);
                    if (limit < kBN - 1) {
#pragma unroll
                        for (int c = 0; c < kBN; ++c)
                            if (c > limit) sr[c] = __float_as_uint(-INFINITY);
                    }
                    // row maximum of the raw scores (scale > 0), in four
                    // independent partial maxima; three-input max takes two
                    // new scores per instruction
                    float pm[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        pm[i] = fmaxf(__uint_as_float(sr[i]), __uint_as_float(sr[4 + i]));
#pragma unroll
                    for (int c = 8; c < kBN; c += 8)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            pm[i] = fmax3(pm[i], __uint_as_float(sr[c + i]), __uint_as_float(sr[c + 4 + i]));
                    const float rmax = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
                    const float m_new = fmaxf(m, rmax * sc);
                    const bool rescale = (m == -INFINITY) ? (m_new != -INFINITY)
                                                          : (m_new > m + kRescaleThreshold);
                    float alpha = 1.f;
                    if (rescale) {
                        alpha = (m == -INFINITY) ? 0.f : fast_exp2(m - m_new);
                        m = m_new;
                    }
                    const float mu = (m == -INFINITY) ? 0.f : m;
                    const bool any_rescale = __any_sync(0xffffffffu, rescale);
                    // p = 2^(s*scale - m), bf16 pairs written over the upper S columns
                    float2 acc[2];
                    exp_pack_store(sr, sc, mu, tS, acc);
                    // S_t(j) follows P_t(j-1) V_{j-1} on the tensor core, so O
                    // is final for the earlier tiles: rescale it in place if needed
                    if (j > 0 && any_rescale) {
#pragma unroll 1
                        for (int cc = 0; cc < HD / 32; ++cc) {
                            float o[32];
                            tmem_ld32(tO + cc * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(tO + cc * 32, o);
                        }
                    }
                    l *= alpha;
                    tmem_wait_st();
                    l += (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
                    if (t == 0 && j + 1 == U.n_kv && p.paged && !p.row_copy && U.n_kv * kBN > U.Lk) {
                        // paged cache by TMA boxes: zero the value rows past the
                        // last key of the final V tile once it has landed, so
                        // unwritten cache slots (possibly NaN) never meet a zero
                        // probability.  S of this tile has landed, so every
                        // earlier load of the slot was waited for by the MMA
                        // thread, and the slot is not refilled before the P V
                        // products that follow this arrival: the parity below
                        // names this load's phase.
                        const int sv = nv_last % kSlots;
                        live = wait_or_abort(&slot_full[sv], (uint32_t)(nv_last / kSlots) & 1u, abort_flag);
                        if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                        unsigned char *vt = smem + L::kOffRing + sv * L::kKVTile;
                        const int first = U.Lk - (U.n_kv - 1) * kBN;
                        const int pieces = (kBN - first) * 8;      // 16-byte pieces per 128-byte half
                        for (int c = row; c < H * pieces; c += kBM) {
                            const int hf = c / pieces, rc = c % pieces;
                            *reinterpret_cast<uint4 *>(vt + hf * kBN * 128 + (first + rc / 8) * 128 + (rc % 8) * 16) =
                                make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&p_full[t]);
                }
                if (!live) break;
                // epilogue: O / l -> bf16 rows, lse.  The tensor memory read
                // here is complete before this warp's next P arrival, which
                // the next unit's first P V product (overwriting O) waits for.
                live = wait_or_abort(&o_done[t], jpar ^ 1u, abort_flag);
                if (!__all_sync(0xffffffffu, live)) { live = false; break; }
                tc_fence_after();
                const bool row_ok = qi < U.Lq;
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const int hq = U.hp * pair + (packed ? (row >> 6) : t);
                uint16_t *orow = p.out + (int64_t)(U.q0 + (row_ok ? qi : 0)) * p.out_rs + (int64_t)hq * HD;
                uint32_t ov[HD];
                tmem_ld_row<HD>(tO, ov);
                if (row_ok && PKV_PF_OUT_V8 && p.out_v8) {
#pragma unroll
                    for (int v = 0; v < HD / 16; ++v) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(ov[v * 16 + 2 * e]) * inv,
                                               __uint_as_float(ov[v * 16 + 2 * e + 1]) * inv);
                        st_cs_v8(orow + v * 16, w);   // written once
                    }
                } else if (row_ok) {
#pragma unroll
                    for (int v = 0; v < HD / 8; ++v) {
                        uint4 pkt;
                        pkt.x = pack_bf16x2(__uint_as_float(ov[v * 8 + 0]) * inv, __uint_as_float(ov[v * 8 + 1]) * inv);
                        pkt.y = pack_bf16x2(__uint_as_float(ov[v * 8 + 2]) * inv, __uint_as_float(ov[v * 8 + 3]) * inv);
                        pkt.z = pack_bf16x2(__uint_as_float(ov[v * 8 + 4]) * inv, __uint_as_float(ov[v * 8 + 5]) * inv);
                        pkt.w = pack_bf16x2(__uint_as_float(ov[v * 8 + 6]) * inv, __uint_as_float(ov[v * 8 + 7]) * inv);
                        st_cs_v4(orow + v * 8, pkt);   // written once
                    }
                }
                if (row_ok && p.lse)
                    p.lse[(int64_t)(U.q0 + qi) * p.num_heads + hq] =
                        l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&unit_empty[slot]);
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
int launch_hd(const PrefillArgs &a, const PrefillParams &pp, int4 *work, int32_t *count,
              int max_items, cudaStream_t stream, const char **err) {
    using L = PLayout<HD>;
    CUtensorMap qm, qm64, km, vm;
    int rc = encode_rows_heads_map(&qm, a.q, a.total_q, a.num_heads, HD, a.q_rs, HD, 64, kBM, true, err);
    if (!rc) rc = encode_rows_heads_map(&qm64, a.q, a.total_q, a.num_heads, HD, a.q_rs, HD, 64, kBM / 2, true, err);
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
    const int smem = L::kBytes + 1024;
    auto kern = prefill_kernel<HD>;
    static PerDeviceOnce once;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    bool regs_ok = true;
    if (e == cudaSuccess)
        e = once.run(dev, [&]() {
            // the register split (setmaxnreg) redistributes the registers the
            // CTA is launched with; it must not ask for more than that
            cudaFuncAttributes fa;
            cudaError_t r = cudaFuncGetAttributes(&fa, kern);
            if (r == cudaSuccess &&
                fa.numRegs * kThreads < 8 * 32 * kRegsSoftmax + 4 * 32 * kRegsOther)
                return cudaErrorInvalidConfiguration;
            if (r == cudaSuccess)
                r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            return r;
        });
    if (e == cudaErrorInvalidConfiguration) regs_ok = false;
    if (!regs_ok) { *err = "prefill kernel compiled with fewer registers than its register split needs"; return PKV_ERR_CUDA; }
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(pp, count, work);
    e = cudaGetLastError();
    if (e != cudaSuccess) { *err = cudaGetErrorString(e); return PKV_ERR_CUDA; }
    const int G = a.num_heads / a.num_kv_heads;
    const int pair = G % 2 == 0 ? 2 : 1;
    const int64_t max_units = (int64_t)max_items * (a.num_heads / pair);
    const int grid = (int)(max_units < num_sms() ? max_units : num_sms());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = PKV_PF_PDL ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, qm, qm64, km, vm, pp);
    if (e == cudaSuccess) e = cudaGetLastError();
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
    return 256 + 2 * sizeof(int4) * (size_t)max_work_items(num_seqs, total_q);
}

int launch_prefill(const PrefillArgs &a, cudaStream_t stream, const char **err) {
    if (a.head_dim != 64 && a.head_dim != 128) {
        *err = "head_dim must be 64 or 128";
        return PKV_ERR_UNSUPPORTED;
    }
    const bool paged = a.bt != nullptr;
    if (paged && (a.block_size < 1 || (a.block_size & (a.block_size - 1)))) {
        *err = "paged prefill needs a power-of-two block_size";
        return PKV_ERR_UNSUPPORTED;
    }
    const size_t need = prefill_workspace_bytes(a.num_seqs, a.total_q, a.max_seqlen_q, a.num_heads);
    if (!a.workspace || a.workspace_bytes < need) {
        *err = "workspace smaller than paged_attn_prefill_workspace_size()";
        return PKV_ERR_WORKSPACE;
    }
    const int max_items = max_work_items(a.num_seqs, a.total_q);
    if ((int64_t)max_items * a.num_heads > (int64_t)1 << 30) {
        *err = "too many 128-row query blocks for one launch";
        return PKV_ERR_UNSUPPORTED;
    }
    int32_t *count = reinterpret_cast<int32_t *>(a.workspace);
    int4 *work = reinterpret_cast<int4 *>(reinterpret_cast<unsigned char *>(a.workspace) + 256);
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
    pp.claim = count + 1;
    pp.work = work;
    pp.max_items = max_items;
    pp.row_copy = paged && a.block_size < 8 ? 1 : 0;
    pp.out_v8 = (reinterpret_cast<uintptr_t>(a.out) % 32 == 0 && a.out_rs % 16 == 0) ? 1 : 0;
    pp.k_cache = a.k_cache;
    pp.v_cache = a.v_cache;
    if (a.head_dim == 128) return launch_hd<128>(a, pp, work, count, max_items, stream, err);
    return launch_hd<64>(a, pp, work, count, max_items, stream, err);
}

}  // namespace pkv
