// Grouped GEMM over routed experts on the 5th-generation tensor cores, with
// the Q4 dequantisation done in shared memory on the way to the MMA.
//
// BaseRT: optimal LLM inference on Apple Silicon with native Metal, §3.4
// "Prefill": prompts run as GEMMs whose arithmetic intensity grows with the
// sequence length; §3.3: every matmul kernel dequantises in its inner loop
// (never materialising dequantised weights in global memory); abstract and
// Fig. 1: MoE prefill (Qwen3-30B-A3B, 4-bit) is where BaseRT's lead is largest.
//
// Shape: for expert e and its routed rows r in offsets[e] .. offsets[e+1]-1,
// Y[r][n] = sum_k w_e[n][k] * X[r][k].  GLU mode: W_e holds 2N rows (gate then
// up) and Y = fp16(SiLU(gate) * up).
//
// GB300 design (one CTA per SM, persistent):
// * Work unit = (expert, token tile of up to 128 rows, 128-row output tile),
//   decoded on the device from `offsets` (no host readback).  The weight rows
//   of a unit fill the MMA's M = 128; the tokens are its N (16..128, padded to
//   a multiple of 16): small token counts per expert still use the tensor core.
// * Warp 0 (TMA): per 64-wide K step, the packed codes of the unit's 128 rows
//   (one 2-D tensor-map copy per matrix, 128 rows x 32 bytes) and the X tile
//   (128 rows x 64 fp16, 128-byte swizzle = the canonical K-major UMMA layout).
// * Warp 0 also bulk-copies each unit's scale and bias block (the unit's 128
//   rows are contiguous in both arrays) into a staging buffer; the dequant
//   threads move their row's values into private shared slots at unit start.
// * Warps 2..9 (dequant): codes -> fp16 w = s*q + b with the code OR-ed into
//   the mantissa of 1024.0/64.0 (exact), one fp16 subtract and one fp16 FMA per
//   pair (w rounded once to fp16).  Units of up to 64 tokens: the row's values
//   go to its TMEM lane with tcgen05.st (A read by the MMA from tensor memory);
//   larger units: written as the A tile in the swizzled K-major shared-memory
//   layout, fenced to the async proxy.
// * Warp 15 (dispatch): one thread waits for each K step's input stage and
//   free A stage and releases the step to the dequant warps with one mbarrier
//   arrival (each completed-phase wait costs ~80 ns of the step).
// * Warp 1 (MMA) and warp 14: two issuing threads (GLU: one per matrix;
//   plain: alternate K steps into two accumulators, added in the epilogue)
//   issue tcgen05.mma kind::f16 (fp16 x fp16 -> fp32) into double-buffered
//   TMEM accumulators, committing to mbarriers to release input stages and
//   hand the accumulator to the epilogue.  With few tokens per unit an MMA is
//   small and its issue, not its arithmetic, sets the pace (a per-role
//   timestamp trace: ~40-100 ns per 128 x 16..32 x 16 MMA).
// * Warps 10..13 (epilogue): tcgen05.ld of the accumulator, SiLU*up or plain,
//   coalesced stores.
// * Every mbarrier wait is bounded; on expiry the CTA latches an error bit,
//   winds down, and still frees its tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <climits>

#include "q4_device.cuh"

#include "q4_internal.h"

namespace q4g {

constexpr int kTN = 128;          // tokens per unit at most (MMA N, max; the launch may take fewer)
constexpr int kRows = 128;        // weight rows per unit (MMA M)
constexpr int kKS = 64;           // K per step (one swizzle atom row of fp16, one Q4 group)
constexpr int kMaxInStages = 16;  // codes + X ring (stage count set per launch)
constexpr int kMaxAStages = 4;    // dequantised A ring (stage count set per launch)
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kUpMmaWarp = 2 + kDeqWarps + kEpiWarps;  // 14
// Epilogue staging: per epilogue warp 16 columns x 32 rows of fp32, turned
// from one value per lane and column into 8 consecutive outputs per lane
constexpr uint32_t kEpiStageBytes = kEpiWarps * 16 * 32 * 4;
constexpr int kMaxSeg = 3;  // weight matrices one dense launch may cover
constexpr int kDispWarp = kUpMmaWarp + 1;               // 15: releases each K step to the dequant warps
constexpr int kThreads = (kDispWarp + 1) * 32;
constexpr int kMaxExperts = 256;
constexpr uint32_t kTmemCols = 512;   // 2 accumulator buffers x 2 accumulators x 128 columns; with
                                      // units of <= 64 tokens: 2 x 2 x tn, and A stages from column 256

constexpr uint32_t kCodesBytes = kRows * 32;         // one matrix, one K step
constexpr uint32_t kATileBytes = kRows * kKS * 2;    // 16 KB
// An input stage holds one K step's codes of each matrix, then X (at a
// 1024-byte multiple, as the 128-byte swizzle needs): tn x 128 bytes of X, so
// 20 KB plain and 24 KB GLU with 128-token units.
// An A stage holds one dequantised tile per matrix: 16 KB plain, 32 KB GLU.

struct Params {
    const int32_t* expert_ids;  // routed launches: checked against offsets by the epilogue warps
    const uint16_t* scales;
    const uint16_t* biases;
    const uint16_t* scales_u;  // the up matrix's scales and biases (GLU): its rows are
    const uint16_t* biases_u;  // e * rows_e + up_off + n of these arrays
    const uint16_t* residual;  // PLAIN, fp16 out: Y = fp16(residual + acc); may alias Y
    const int32_t* offsets;    // NULL: dense, one expert holding rows 0..R-1
    void* Y;
    int E, N, K, R, rows_e, up_off, nmat, glu, out_f16;
    int n_tiles, nK, G;
    int tn;               // tokens per unit (32, 64 or 128): the X box rows
    uint32_t x_bytes;     // X bytes per input stage (tn x 64 fp16)
    int a_tmem;           // dequantised A tiles in tensor memory (units of <= 64 tokens) instead of shared memory
    uint32_t acc_cols;    // TMEM columns of one accumulator (tn in TMEM-A mode, else 128)
    uint32_t a_col0;      // TMEM column of the first A stage (TMEM-A mode)
    int kparts, ksteps;   // split of K over units (dense, few units): K steps per part
    float* part;          // kparts > 1: fp32 partials [kparts][nmat][R][N], reduced by reduce_parts_kernel
    int in_stages, a_stages;       // ring depths (the rest of shared memory, see launch_grouped)
    uint32_t in_bytes, a_bytes;    // bytes per input / A stage
    uint32_t x_off;                // X's offset in an input stage
    uint32_t sb_bytes;   // private per-thread scale/bias slots
    uint32_t stg_bytes;  // staging buffer: the unit's scale and bias blocks
    // Dense PLAIN launches over several weight matrices of one input (q, k, v):
    // segment i owns the global weight tiles from seg_t0[i] (INT_MAX for a
    // matrix the launch does not have) to the next segment's first, its own
    // tensor map (tmW, tmWu, tmW2), scales, biases, output and width.
    int nseg;
    int seg_t0[kMaxSeg];
    const uint16_t* seg_s[kMaxSeg];
    const uint16_t* seg_b[kMaxSeg];
    void* seg_Y[kMaxSeg];
    int seg_N[kMaxSeg];
    int sb_global;       // the dequant warps read scales and biases from global memory (no staging;
                         // the kernel instantiation with kSbGlobal)
    int vec_out;         // epilogue staging tiles present (Y and residual 16-byte aligned, room left)
    int* err;
};

struct Smem {
    uint64_t in_full[kMaxInStages], in_empty[kMaxInStages];
    uint64_t a_full[kMaxAStages], a_empty[kMaxAStages];
    uint64_t go[kMaxAStages];    // K step ready for the dequant warps: its input landed, its A stage is free
    uint64_t acc_full[2], acc_empty[2];
    uint64_t sb_full, sb_empty;  // staging buffer of the unit's scales and biases
    uint64_t drain;  // completion probe for in-flight MMAs on the abort path
    uint32_t tmem_base;
    volatile int abort;
    int total_units;
    int prefix[kMaxExperts + 1];  // token tiles before expert e
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// UMMA shared-memory descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride byte offset), version 1 (sm_100 family).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
    d |= (uint64_t)1 << 46;                    // descriptor version
    d |= (uint64_t)2 << 61;                    // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(
            d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with A in tensor memory (M = 128 lanes, two fp16 K values per
// 32-bit column) and B by descriptor.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                               uint32_t acc) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(
            d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 16 / 32 consecutive 32-bit TMEM columns of this thread's lane (the warp's
// lane quarter is in taddr).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-wide forms: the whole (converged) warp executes them and one elected
// lane issues (the warp's values stay uniform, which a clean issue loop
// measured ~13 % cheaper per MMA than one lane issuing alone).
__device__ __forceinline__ void mma_f16_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{ .reg .pred p, e; elect.sync _|e, 0xffffffff; setp.ne.b32 p, %4, 0;\n"
        "  @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_f16_tmem_a_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 uint32_t acc) {
    asm volatile(
        "{ .reg .pred p, e; elect.sync _|e, 0xffffffff; setp.ne.b32 p, %4, 0;\n"
        "  @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar) {
    asm volatile(
        "{ .reg .pred e; elect.sync _|e, 0xffffffff;\n"
        "  @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0]; }" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Position in a ring of n stages: the stage index and how often the ring has
// wrapped (whose low bit is the mbarrier phase parity), advanced without a
// division (the stage counts are launch parameters).
struct RingPos {
    int s = 0, r = 0;
    __device__ __forceinline__ void next(int n) {
        if (++s == n) {
            s = 0;
            ++r;
        }
    }
};

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_bar(Smem& sm, uint64_t& bar, uint32_t parity, int* err) {
    if (sm.abort) return false;
    if (!q4d::mbar_wait(q4d::smem_addr(&bar), parity, err)) {
        sm.abort = 1;
        return false;
    }
    return true;
}

struct Unit {
    int e, r0, tn, nt, kp;  // expert, first token row, valid tokens, output tile index, K part
    int seg;                // weight matrix of a several-matrix launch (nt counts within it)
};

__device__ __forceinline__ Unit decode_unit(const Smem& sm, const Params& p, int u) {
    const int kp = u % p.kparts;
    u /= p.kparts;
    const int tt = u / p.n_tiles;
    int lo = 0, hi = p.E;  // largest e with prefix[e] <= tt
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.prefix[mid] <= tt) lo = mid;
        else hi = mid;
    }
    Unit un;
    un.e = lo;
    const int j = tt - sm.prefix[lo];
    int a = p.offsets ? p.offsets[lo] : 0, b = p.offsets ? p.offsets[lo + 1] : p.R;
    a = max(0, min(a, p.R));
    b = max(a, min(b, p.R));
    un.r0 = a + j * p.tn;
    un.tn = min(p.tn, b - un.r0);
    un.nt = u % p.n_tiles;
    un.seg = 0;
    un.kp = kp;
    return un;
}

// The weight matrix of a several-matrix launch that owns the unit's output
// tile, the tile made relative to it (only the roles that address weights,
// scales or outputs need it).
__device__ __forceinline__ void unit_seg(const Params& p, Unit& un) {
    // seg_t0[i] of a matrix the launch does not have is INT_MAX
    un.seg = (un.nt >= p.seg_t0[1] ? 1 : 0) + (un.nt >= p.seg_t0[2] ? 1 : 0);
    un.nt -= un.seg == 0 ? 0 : un.seg == 1 ? p.seg_t0[1] : p.seg_t0[2];
}

// SiLU(y) = y / (1 + e^-y) with the fast exponential and division (a few
// ulp of fp32, far below the fp16 rounding of the result; y -> -inf gives 0).
__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.0f + __expf(-y)); }

// Bulk prefetch of global memory into L2; bytes a multiple of 16, address
// 16-byte aligned.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// A weight row's scale (low half) and bias (high half) of Q4 group g.
__device__ __forceinline__ uint32_t load_sb(const uint16_t* s, const uint16_t* b, int g) {
    return (uint32_t)__ldg(s + g) | ((uint32_t)__ldg(b + g) << 16);
}

// The scales (qs) and biases (qb) of groups g .. g + 3 of a weight row whose
// group count G is a multiple of 4 (8-byte loads); left as they are when g is
// past the row's end.
__device__ __forceinline__ void load_quad(const uint16_t* s, const uint16_t* b, int g, int G, uint2& qs, uint2& qb) {
    if (g < G) {
        qs = __ldg(reinterpret_cast<const uint2*>(s + g));
        qb = __ldg(reinterpret_cast<const uint2*>(b + g));
    }
}

// Dequantise one word of 8 codes to 8 fp16 weights in k order.
__device__ __forceinline__ uint4 dequant_word(uint32_t q, __half2 s2, __half2 b2) {
    const __half2 m1024 = __float2half2_rn(-1024.f), m64 = __float2half2_rn(-64.f);
    const uint32_t q8 = q >> 8;
    uint32_t v0 = q4d::and_or(q, 0x000F000Fu, 0x64006400u);   // 1024+q0, 1024+q4
    uint32_t v1 = q4d::and_or(q, 0x00F000F0u, 0x54005400u);   // 64+q1,   64+q5
    uint32_t v2 = q4d::and_or(q8, 0x000F000Fu, 0x64006400u);  // 1024+q2, 1024+q6
    uint32_t v3 = q4d::and_or(q8, 0x00F000F0u, 0x54005400u);  // 64+q3,   64+q7
    __half2 h0 = __hfma2(__hadd2(*reinterpret_cast<__half2*>(&v0), m1024), s2, b2);  // w0, w4
    __half2 h1 = __hfma2(__hadd2(*reinterpret_cast<__half2*>(&v1), m64), s2, b2);    // w1, w5
    __half2 h2 = __hfma2(__hadd2(*reinterpret_cast<__half2*>(&v2), m1024), s2, b2);  // w2, w6
    __half2 h3 = __hfma2(__hadd2(*reinterpret_cast<__half2*>(&v3), m64), s2, b2);    // w3, w7
    const uint32_t a0 = *reinterpret_cast<uint32_t*>(&h0), a1 = *reinterpret_cast<uint32_t*>(&h1);
    const uint32_t a2 = *reinterpret_cast<uint32_t*>(&h2), a3 = *reinterpret_cast<uint32_t*>(&h3);
    return make_uint4(prmt(a0, a1, 0x5410), prmt(a2, a3, 0x5410), prmt(a0, a1, 0x7632), prmt(a2, a3, 0x7632));
}

// kATmem: the dequantised A tiles live in tensor memory (units of <= 64
// tokens), else in shared memory.  kSbGlobal (A in shared memory only): the
// dequant warps read the scales and biases from global memory instead of a
// per-unit staging copy.  kMulti: a dense launch over several weight
// matrices of one input (each unit finds its matrix from its output tile).  One instantiation per mode keeps each role's loop
// free of the other's code and registers (a runtime choice between the two
// scale sources measured slower than either).
template <bool kATmem, bool kSbGlobal, bool kMulti>
__global__ void __launch_bounds__(kThreads, 1)
    q4_moe_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWu,
                       const __grid_constant__ CUtensorMap tmW2,
                       const __grid_constant__ CUtensorMap tmX, const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles.
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* in_ring = base;
    uint8_t* a_ring = in_ring + (size_t)p.in_stages * p.in_bytes;
    uint32_t* sb = reinterpret_cast<uint32_t*>(a_ring + (size_t)p.a_stages * p.a_bytes);
    const int IS = p.in_stages, AS = p.a_stages;
    // Plain mode, A in shared memory, staged scales: each half of the
    // dequant warps takes every other K step whole (all 8 words of its rows)
    // instead of half of every step, so a warp waits once per two steps;
    // elsewhere all 8 warps take every step (with A in tensor memory this
    // measured no faster and cost the GLU launches of the same kernel 5 %).
    const bool step_split = !kATmem && !p.glu && !kSbGlobal;
    const int deq_per_step = step_split ? kDeqWarps / 2 : kDeqWarps;  // dequant arrivals per K step
    uint8_t* stg = reinterpret_cast<uint8_t*>(sb) + p.sb_bytes;
    float* epi_st = reinterpret_cast<float*>(stg + p.stg_bytes);  // vec_out only
    Smem& sm = *reinterpret_cast<Smem*>(stg + p.stg_bytes + (p.vec_out ? kEpiStageBytes : 0u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < IS; ++i) {
            q4d::mbar_init(q4d::smem_addr(&sm.in_full[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&sm.in_empty[i]), deq_per_step + p.nmat);
        }
        for (int i = 0; i < AS; ++i) {
            q4d::mbar_init(q4d::smem_addr(&sm.a_full[i]), deq_per_step);
            q4d::mbar_init(q4d::smem_addr(&sm.a_empty[i]), p.nmat);
            q4d::mbar_init(q4d::smem_addr(&sm.go[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            q4d::mbar_init(q4d::smem_addr(&sm.acc_full[i]), 2);  // both issuers commit
            q4d::mbar_init(q4d::smem_addr(&sm.acc_empty[i]), kEpiWarps);
        }
        q4d::mbar_init(q4d::smem_addr(&sm.sb_full), 1);
        q4d::mbar_init(q4d::smem_addr(&sm.sb_empty), kDeqWarps);
        q4d::mbar_init(q4d::smem_addr(&sm.drain), 2);
        sm.abort = 0;
        q4d::fence_mbar_init();
    }
    if (warp == 0) {
        // token tiles per expert -> prefix sums (offsets clamped to [0, R])
        if (lane == 0) {
            int run = 0;
            for (int e = 0; e < p.E; ++e) {
                sm.prefix[e] = run;
                int a = p.offsets ? max(0, min(p.offsets[e], p.R)) : 0;
                int b = p.offsets ? max(a, min(p.offsets[e + 1], p.R)) : p.R;
                run += (b - a + p.tn - 1) / p.tn;
            }
            sm.prefix[p.E] = run;
            sm.total_units = run * p.n_tiles * p.kparts;
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         q4d::smem_addr(&sm.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    const int U = sm.total_units;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            int it = 0, uu = 0, staged = 0;
            RingPos ip;
            const uint32_t blk = (uint32_t)kRows * (uint32_t)p.G * 2u;  // one matrix's scales (or biases) of a unit
            for (int u = blockIdx.x; u < U && !sm.abort; u += gridDim.x, ++uu) {
                Unit un = decode_unit(sm, p, u);
                if constexpr (kMulti) unit_seg(p, un);
                const int wrow = un.e * p.rows_e + un.nt * kRows;
                const int wrow_u = un.e * p.rows_e + p.up_off + un.nt * kRows;
                const CUtensorMap* mw = !kMulti || un.seg == 0 ? &tmW : un.seg == 1 ? &tmWu : &tmW2;
                if constexpr (kSbGlobal) {
                    // the dequant warps read the scales and biases from global
                    // memory: bring the unit's rows into L2
                    for (int m = 0; m < p.nmat; ++m) {
                        const size_t r = (size_t)(m ? wrow_u : wrow) * p.G;
                        bulk_prefetch_l2((m ? p.scales_u : kMulti ? p.seg_s[un.seg] : p.scales) + r, blk);
                        bulk_prefetch_l2((m ? p.biases_u : kMulti ? p.seg_b[un.seg] : p.biases) + r, blk);
                    }
                } else {
                    // the staging buffer is free once every dequant warp has read the previous unit's values
                    if (uu > 0 && !wait_bar(sm, sm.sb_empty, (uu - 1) & 1, p.err)) break;
                    const uint32_t fb = q4d::smem_addr(&sm.sb_full);
                    q4d::mbar_arrive_expect_tx(fb, (uint32_t)p.nmat * 2u * blk);
                    for (int m = 0; m < p.nmat; ++m) {
                        const size_t r = (size_t)(m ? wrow_u : wrow) * p.G;
                        q4d::bulk_g2s(q4d::smem_addr(stg + (2 * m) * blk), (m ? p.scales_u : kMulti ? p.seg_s[un.seg] : p.scales) + r,
                                      blk, fb);
                        q4d::bulk_g2s(q4d::smem_addr(stg + (2 * m + 1) * blk), (m ? p.biases_u : kMulti ? p.seg_b[un.seg] : p.biases) + r, blk,
                                      fb);
                    }
                    ++staged;
                }
                const int ks0 = un.kp * p.ksteps, ks1 = ks0 + p.ksteps;
                for (int ks = ks0; ks < ks1; ++ks, ++it) {
                    const int s = ip.s;
                    if (ip.r > 0 && !wait_bar(sm, sm.in_empty[s], (ip.r - 1) & 1, p.err)) break;
                    uint8_t* st = in_ring + (size_t)s * p.in_bytes;
                    const uint32_t fb = q4d::smem_addr(&sm.in_full[s]);
                    q4d::mbar_arrive_expect_tx(fb, p.nmat * kCodesBytes + p.x_bytes);
                    tma_load_2d(q4d::smem_addr(st), mw, ks * 32, wrow, fb);
                    if (p.glu) tma_load_2d(q4d::smem_addr(st + kCodesBytes), &tmWu, ks * 32, wrow_u, fb);
                    tma_load_2d(q4d::smem_addr(st + p.x_off), &tmX, ks * kKS, un.r0, fb);
                    ip.next(IS);
                }
            }
            if (sm.abort) {
                // let this thread's last copies land before the CTA can exit
                for (int j = (it > IS ? it - IS : 0); j < it; ++j)
                    q4d::mbar_wait(q4d::smem_addr(&sm.in_full[j % IS]), (j / IS) & 1, nullptr);
                if (staged > 0) q4d::mbar_wait(q4d::smem_addr(&sm.sb_full), (staged - 1) & 1, nullptr);
            }
        }
    } else if (warp == 1 || warp == kUpMmaWarp) {
        // ------------------------------------------------------------ MMA
        // Two issuing threads (a thread issues a tcgen05.mma of N <= 64 in
        // ~46 cycles at best, more beside the dequant warps on its SMSP,
        // while the SM accepts them faster, so one thread would set the
        // pace).  GLU: issuer r owns matrix r (gate, up) for every K step.
        // Plain: both own the one matrix, issuer r the K steps of parity r of
        // each unit, into an accumulator of its own (the columns the up
        // matrix has in GLU mode); the epilogue adds the two.
        const int r = warp == 1 ? 0 : 1;
        const int mi = p.glu ? r : 0;
        // the whole warp runs the loop (uniform values); one elected lane issues
        {
            int acc_it = 0;
            RingPos ip, ap;
            for (int u = blockIdx.x; u < U && !sm.abort; u += gridDim.x, ++acc_it) {
                const Unit un = decode_unit(sm, p, u);
                const int npad = ((un.tn + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(npad);
                const int buf = acc_it & 1;
                if (acc_it >= 2 &&
                    !__all_sync(0xffffffffu, wait_bar(sm, sm.acc_empty[buf], ((acc_it >> 1) - 1) & 1, p.err)))
                    break;
                tc_fence_after();
                const uint32_t dm = tmem + (uint32_t)(buf * 2 + r) * p.acc_cols;
                bool ok = true, first = true;
                const int ks0 = un.kp * p.ksteps, ks1 = ks0 + p.ksteps;
                // One K step's MMAs (4 of K = 16) on input stage s, A stage a,
                // then the commits that release both.
                auto issue = [&](int s, int a) {
                    const uint32_t xs = q4d::smem_addr(in_ring + (size_t)s * p.in_bytes + p.x_off);
                    // K-chunk kk advances the X descriptor's start address by 32 bytes
                    const uint64_t xd = sw128_desc(xs);
                    if constexpr (kATmem) {
                        // 16 fp16 of K = 8 TMEM columns
                        const uint32_t at = tmem + p.a_col0 + (uint32_t)(a * 2 + mi) * 32u;
#pragma unroll
                        for (int kk = 0; kk < kKS / 16; ++kk)
                            mma_f16_tmem_a_w(dm, at + 8 * kk, xd + 2 * kk, idesc, (!first || kk > 0) ? 1u : 0u);
                    } else {
                        const uint32_t as = q4d::smem_addr(a_ring + (size_t)a * p.a_bytes);
                        const uint64_t ad = sw128_desc(as + mi * kATileBytes);
#pragma unroll
                        for (int kk = 0; kk < kKS / 16; ++kk)
                            mma_f16_w(dm, ad + 2 * kk, xd + 2 * kk, idesc, (!first || kk > 0) ? 1u : 0u);
                    }
                    first = false;
                    mma_commit_w(q4d::smem_addr(&sm.in_empty[s]));
                    mma_commit_w(q4d::smem_addr(&sm.a_empty[a]));
                };
                // With A in tensor memory (4 A stages) this issuer's steps go
                // in pairs behind one wait: every dequant warp arrives on the
                // A stages in step order, so the second step's a_full phase
                // completes after the first's.  A completed-phase wait costs
                // ~80 ns of the issuer's step.  In plain mode a deferred step
                // holds its input stage until the issuer's next step (two
                // steps on) is dequantised, whose codes need a stage of their
                // own, and the A stage two steps on must be free: pairs only
                // with 4 A stages and, in plain mode, 3 or more input stages
                // (a model of the rings' hand-offs finds no deadlock then, and
                // one with 2 input or 2 A stages).
                const bool pairs = kATmem && AS >= 4 && (p.glu || IS >= 3);
                int pend_s = -1, pend_a = 0;
                for (int ks = ks0; ks < ks1; ++ks) {
                    const int s = ip.s, a = ap.s;
                    if (p.glu || ((ks - ks0) & 1) == r) {
                        const bool more = ks + (p.glu ? 1 : 2) < ks1;  // another step of this issuer follows
                        if (pairs && pend_s < 0 && more) {
                            pend_s = s;
                            pend_a = a;
                        } else {
                            // A stage a is complete only after every dequant
                            // warp was released for input stage s (codes and X
                            // land together on in_full), so that one wait also
                            // covers the X tile.
                            if (!__all_sync(0xffffffffu, wait_bar(sm, sm.a_full[a], ap.r & 1, p.err))) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (pend_s >= 0) {
                                issue(pend_s, pend_a);
                                pend_s = -1;
                            }
                            issue(s, a);
                        }
                    }
                    ip.next(IS);
                    ap.next(AS);
                }
                if (!ok) break;
                mma_commit_w(q4d::smem_addr(&sm.acc_full[buf]));
            }
        }
    } else if (warp == kDispWarp) {
        // ------------------------------------------------------------ dispatch
        // One thread waits, for every K step, on the two barriers the dequant
        // warps would otherwise each wait on (the input stage landed, the A
        // stage's previous MMAs done) and releases the step with one arrival:
        // a completed-phase wait costs ~80 ns, and this takes one of the two
        // off the dequant warps' step.  It arrives on go[a] for round r only
        // after a_empty[a] of round r - 1, which needs every dequant warp's
        // a_full arrival of that round, so the dequant warps have consumed
        // the previous phase of go[a] by then.
        if (lane == 0) {
            RingPos ip, ap;
            for (int u = blockIdx.x; u < U && !sm.abort; u += gridDim.x) {
                bool ok = true;
                for (int j = 0; j < p.ksteps; ++j) {
                    const int s = ip.s, a = ap.s;
                    if (!wait_bar(sm, sm.in_full[s], ip.r & 1, p.err) ||
                        (ap.r > 0 && !wait_bar(sm, sm.a_empty[a], (ap.r - 1) & 1, p.err))) {
                        ok = false;
                        break;
                    }
                    q4d::mbar_arrive(q4d::smem_addr(&sm.go[a]));
                    ip.next(IS);
                    ap.next(AS);
                }
                if (!ok) break;
            }
        }
    } else if (warp < 2 + kDeqWarps) {
        // ------------------------------------------------------------ dequant
        // Thread dt owns weight row `row` of the tile -- the TMEM lane its warp
        // may write, 32 (warp % 4) + lane -- and half `part` of the row's 16
        // (GLU: gate then up) or 8 (plain) words of a K step: in GLU mode all
        // 8 words of matrix `part` of every step; in plain mode with staged
        // scales all 8 words of the steps of parity `part` (step_split), else
        // words 4 part .. 4 part + 3 of every step.
        // Its scales/biases live in private shared slots (no cross-thread
        // sharing, so no barrier that an aborting warp could leave the others
        // waiting on).
        const int dt = threadIdx.x - 64;          // 0 .. 255
        const int row = 32 * (warp & 3) + lane;
        const int part = (warp - 2) >> 2;         // 0 or 1
        const int m = p.glu ? part : 0;
        const int G = p.G, Gp = G + 1;
        uint32_t* my_sb = sb + (size_t)dt * Gp;
        const uint32_t blk = (uint32_t)kRows * (uint32_t)G * 2u;
        const uint16_t* sp = reinterpret_cast<const uint16_t*>(stg + (2 * m) * blk) + (size_t)row * G;
        const uint16_t* bp = reinterpret_cast<const uint16_t*>(stg + (2 * m + 1) * blk) + (size_t)row * G;
        int it = 0, uu = 0;
        RingPos ip, ap;
        const bool quads = (G & 3) == 0;
        for (int u = blockIdx.x; u < U && !sm.abort; u += gridDim.x, ++uu) {
            // sb_global: this thread's row of scales and biases in global
            // memory, read ahead of their use four groups to a load
            // (G % 4 == 0) or two steps ahead one group at a time
            Unit un = decode_unit(sm, p, u);
            if constexpr (kSbGlobal && kMulti) unit_seg(p, un);  // (the staged scales need no weight row)
            const size_t gr = (size_t)(un.e * p.rows_e + (m ? p.up_off : 0) + un.nt * kRows + row) * G;
            const uint16_t* sr = (m ? p.scales_u : kMulti ? p.seg_s[un.seg] : p.scales) + gr;
            const uint16_t* br = (m ? p.biases_u : kMulti ? p.seg_b[un.seg] : p.biases) + gr;
            if constexpr (!kSbGlobal) {
            // this unit's scales and biases, from the staging buffer into private slots
            if (!__all_sync(0xffffffffu, wait_bar(sm, sm.sb_full, uu & 1, p.err))) {
                sm.abort = 1;
                break;
            }
            if (quads) {
                for (int g = 0; g < G; g += 4) {  // 8-byte loads: 4 values of a row
                    const uint2 s4 = *reinterpret_cast<const uint2*>(sp + g);
                    const uint2 b4 = *reinterpret_cast<const uint2*>(bp + g);
                    my_sb[g] = prmt(s4.x, b4.x, 0x5410);
                    my_sb[g + 1] = prmt(s4.x, b4.x, 0x7632);
                    my_sb[g + 2] = prmt(s4.y, b4.y, 0x5410);
                    my_sb[g + 3] = prmt(s4.y, b4.y, 0x7632);
                }
            } else {
                for (int g = 0; g < G; ++g) my_sb[g] = (uint32_t)sp[g] | ((uint32_t)bp[g] << 16);
            }
            __syncwarp();
            if (lane == 0) q4d::mbar_arrive(q4d::smem_addr(&sm.sb_empty));
            }
            bool ok = true;
            const int ks0 = un.kp * p.ksteps, ks1 = ks0 + p.ksteps;
            uint2 qs[2] = {}, qb[2] = {};  // [0] the four groups holding step ks, [1] the next four
            uint32_t sb0 = 0, sb1 = 0;     // G % 4 != 0: steps ks and ks + 1
            if constexpr (kSbGlobal) {
                if (quads) {
                    load_quad(sr, br, ks0 & ~3, G, qs[0], qb[0]);
                    load_quad(sr, br, (ks0 & ~3) + 4, G, qs[1], qb[1]);
                } else {
                    sb0 = load_sb(sr, br, ks0);
                    sb1 = ks0 + 1 < ks1 ? load_sb(sr, br, ks0 + 1) : 0u;
                }
            }
            for (int ks = ks0; ks < ks1; ++ks, ++it) {
                const int s = ip.s, a = ap.s;
                if (step_split && ((ks - ks0) & 1) != part) {  // the other half's step
                    ip.next(IS);
                    ap.next(AS);
                    continue;
                }
                // released by the dispatch thread: input stage s landed and A stage a is free
                const bool w = wait_bar(sm, sm.go[a], ap.r & 1, p.err);
                if (!__all_sync(0xffffffffu, w)) {
                    sm.abort = 1;
                    ok = false;
                    break;
                }
                // (the next scale loads go out after the wait: an outstanding
                // global load held the acquire wait up by its latency)
                uint32_t sbv;
                if constexpr (!kSbGlobal) {
                    sbv = my_sb[ks];
                } else if (quads) {
                    if ((ks & 3) == 0 && ks != ks0) {
                        qs[0] = qs[1];
                        qb[0] = qb[1];
                        load_quad(sr, br, ks + 4, G, qs[1], qb[1]);
                    }
                    const int j = ks & 3;
                    const uint32_t sw = j < 2 ? qs[0].x : qs[0].y, bw = j < 2 ? qb[0].x : qb[0].y;
                    sbv = (j & 1) ? prmt(sw, bw, 0x7632) : prmt(sw, bw, 0x5410);
                } else {
                    sbv = sb0;
                    sb0 = sb1;
                    sb1 = ks + 2 < ks1 ? load_sb(sr, br, ks + 2) : 0u;
                }
                const uint8_t* st = in_ring + (size_t)s * p.in_bytes;
                uint8_t* at = a_ring + (size_t)a * p.a_bytes;
                const int w0 = p.glu || step_split ? 0 : 4 * part, nw = p.glu || step_split ? 8 : 4;
                const __half sh = __ushort_as_half((uint16_t)(sbv & 0xFFFF));
                const __half bh = __ushort_as_half((uint16_t)(sbv >> 16));
                const __half2 s2 = __halves2half2(sh, sh), b2 = __halves2half2(bh, bh);
                const uint4* cw = reinterpret_cast<const uint4*>(st + m * kCodesBytes + row * 32);
                if constexpr (kATmem) {
                    // the row's fp16 weights in k order, two per 32-bit column
                    // of its TMEM lane: matrix m of A stage a
                    tc_fence_after();  // the MMAs that read this A stage before are complete
                    uint32_t v[32];
                    const uint32_t* cw32 = reinterpret_cast<const uint32_t*>(cw) + w0;
                    uint32_t words[8];
                    {
                        const uint4 c = *reinterpret_cast<const uint4*>(cw32);
                        words[0] = c.x; words[1] = c.y; words[2] = c.z; words[3] = c.w;
                    }
                    if (nw == 8) {
                        const uint4 c = *reinterpret_cast<const uint4*>(cw32 + 4);
                        words[4] = c.x; words[5] = c.y; words[6] = c.z; words[7] = c.w;
                    } else {
                        words[4] = words[5] = words[6] = words[7] = 0;
                    }
#pragma unroll
                    for (int wi = 0; wi < 8; ++wi) {
                        if (wi < nw) {
                            const uint4 d = dequant_word(words[wi], s2, b2);
                            v[4 * wi + 0] = d.x;
                            v[4 * wi + 1] = d.y;
                            v[4 * wi + 2] = d.z;
                            v[4 * wi + 3] = d.w;
                        }
                    }
                    const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + p.a_col0 +
                                        (uint32_t)(a * 2 + m) * 32u + (uint32_t)(w0 * 4);
                    if (nw == 8) tmem_st32(ta, v);
                    else tmem_st16(ta, v);
                    tmem_st_wait();
                    tc_fence_before();
                } else {
                    uint8_t* arow = at + m * kATileBytes + (row >> 3) * 1024 + (row & 7) * 128;
                    for (int h = 0; h < nw / 4; ++h) {
                        const uint4 c = cw[(w0 >> 2) + h];
                        const uint32_t words[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int wi = 0; wi < 4; ++wi) {
                            const int j = w0 + h * 4 + wi;   // 16-byte chunk = 8 consecutive k
                            *reinterpret_cast<uint4*>(arow + ((j ^ (row & 7)) << 4)) = dequant_word(words[wi], s2, b2);
                        }
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                }
                __syncwarp();
                if (lane == 0) {
                    q4d::mbar_arrive(q4d::smem_addr(&sm.in_empty[s]));
                    q4d::mbar_arrive(q4d::smem_addr(&sm.a_full[a]));
                }
                ip.next(IS);
                ap.next(AS);
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Routed launches: the device check that expert_ids agrees with
        // offsets (and that offsets are a monotone partition of 0..R-1), one
        // thread per check over the grid's epilogue threads, while the first
        // units' main loops run; a mismatch latches kErrDeviceCheck.
        if (p.offsets && p.expert_ids) {
            const int nthr = (int)gridDim.x * 32 * kEpiWarps;
            const int t = (int)blockIdx.x * 32 * kEpiWarps + ((int)threadIdx.x - 32 * (2 + kDeqWarps));
            if (t == 0 && (p.offsets[0] != 0 || p.offsets[p.E] != p.R)) atomicOr(p.err, q4d::kErrDeviceCheck);
            for (int e = t; e < p.E; e += nthr)
                if (p.offsets[e] > p.offsets[e + 1]) atomicOr(p.err, q4d::kErrDeviceCheck);
            for (int r = t; r < p.R; r += nthr) {
                const int e = p.expert_ids[r];
                if (e < 0 || e >= p.E || r < p.offsets[e] || r >= p.offsets[e + 1]) atomicOr(p.err, q4d::kErrDeviceCheck);
            }
        }
        const int q = warp & 3;                   // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;            // accumulator lane = weight row in the tile
        int acc_it = 0;
        for (int u = blockIdx.x; u < U && !sm.abort; u += gridDim.x, ++acc_it) {
            Unit un = decode_unit(sm, p, u);
            if constexpr (kMulti) unit_seg(p, un);
            const int buf = acc_it & 1;
            if (!__all_sync(0xffffffffu, wait_bar(sm, sm.acc_full[buf], (acc_it >> 1) & 1, p.err))) {
                sm.abort = 1;
                break;
            }
            tc_fence_after();
            const int n = un.nt * kRows + row;
            const uint32_t t0 = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * 2) * p.acc_cols;
            // plain mode: the second issuer's accumulator holds the odd K steps
            const bool two = p.glu || p.ksteps >= 2;
            // this unit's output: its row width and base
#define yN (kMulti ? p.seg_N[un.seg] : p.N)
#define Yp (kMulti ? p.seg_Y[un.seg] : p.Y)
            if (p.kparts > 1) {
                // one K part: raw fp32 sums, reduced (and finished) by reduce_parts_kernel
                const size_t pr = (size_t)p.R * p.N;
                for (int c0 = 0; c0 < un.tn; c0 += 16) {
                    uint32_t g[16], v[16];
                    tmem_ld16(t0 + c0, g);
                    if (two) tmem_ld16(t0 + p.acc_cols + c0, v);
                    tmem_ld_wait();
                    if (!p.glu && two) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) g[c] = __float_as_uint(__uint_as_float(g[c]) + __uint_as_float(v[c]));
                    }
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        if (c0 + c < un.tn) {
                            const size_t o = (size_t)(un.r0 + c0 + c) * p.N + n;
                            p.part[(size_t)(un.kp * p.nmat) * pr + o] = __uint_as_float(g[c]);
                            if (p.glu) p.part[(size_t)(un.kp * p.nmat + 1) * pr + o] = __uint_as_float(v[c]);
                        }
                    }
                }
            } else {
                // 16 columns (tokens) at a time; the next 16 columns' tensor-memory
                // loads are in flight while these are finished and stored.  With
                // an aligned Y the values go through this warp's staging tile, so
                // that each lane stores runs of 8 consecutive outputs (16 or 32
                // bytes) instead of one 2- or 4-byte value per column.
                float* ws = epi_st + q * (16 * 32);
                const int nb = un.nt * kRows + q * 32;  // this warp's first weight row
                uint32_t g[16], v[16] = {};
                tmem_ld16(t0, g);
                if (two) tmem_ld16(t0 + p.acc_cols, v);
                for (int c0 = 0; c0 < un.tn; c0 += 16) {
                    // the residuals this lane adds, loaded before the wait (runs j: column
                    // (lane + 32 j) / 4, outputs 8 ((lane + 32 j) % 4) ..; scalar: column c)
                    uint4 rv[2] = {};
                    float rs[16];
                    if (p.residual) {
                        if (p.vec_out) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int k = lane + 32 * j, c = k >> 2;
                                if (c0 + c < un.tn)
                                    rv[j] = *reinterpret_cast<const uint4*>(
                                        p.residual + (size_t)(un.r0 + c0 + c) * yN + nb + (k & 3) * 8);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 16; ++c)
                                rs[c] = c0 + c < un.tn
                                            ? __half2float(__ushort_as_half(p.residual[(size_t)(un.r0 + c0 + c) * yN + n]))
                                            : 0.f;
                        }
                    }
                    tmem_ld_wait();
                    float y[16], w[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        y[c] = __uint_as_float(g[c]);
                        w[c] = __uint_as_float(v[c]);
                        if (!p.glu && two) y[c] += w[c];
                    }
                    if (c0 + 16 < un.tn) {
                        tmem_ld16(t0 + c0 + 16, g);
                        if (two) tmem_ld16(t0 + p.acc_cols + c0 + 16, v);
                    }
                    if (p.glu) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) y[c] = silu(y[c]) * w[c];
                    }
                    if (p.vec_out) {
#pragma unroll
                        for (int c = 0; c < 16; ++c) ws[c * 32 + lane] = y[c];
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int k = lane + 32 * j, c = k >> 2;
                            if (c0 + c >= un.tn) continue;
                            const float4 e0 = *reinterpret_cast<const float4*>(ws + c * 32 + (k & 3) * 8);
                            const float4 e1 = *reinterpret_cast<const float4*>(ws + c * 32 + (k & 3) * 8 + 4);
                            const size_t o = (size_t)(un.r0 + c0 + c) * yN + nb + (k & 3) * 8;
                            float e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                            if (p.residual) {
                                const uint32_t rw[4] = {rv[j].x, rv[j].y, rv[j].z, rv[j].w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&rw[i]));
                                    e[2 * i] += f.x;
                                    e[2 * i + 1] += f.y;
                                }
                            }
                            if (p.out_f16) {
                                uint32_t h[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const __half2 t = __floats2half2_rn(e[2 * i], e[2 * i + 1]);
                                    h[i] = *reinterpret_cast<const uint32_t*>(&t);
                                }
                                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(Yp) + o) = make_uint4(h[0], h[1], h[2], h[3]);
                            } else {
                                float4* d = reinterpret_cast<float4*>(static_cast<float*>(Yp) + o);
                                d[0] = make_float4(e[0], e[1], e[2], e[3]);
                                d[1] = make_float4(e[4], e[5], e[6], e[7]);
                            }
                        }
                        __syncwarp();  // the staging tile is read before the next group writes it
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {
                            if (c0 + c >= un.tn) continue;
                            const size_t o = (size_t)(un.r0 + c0 + c) * yN + n;
                            float yy = y[c];
                            if (p.residual) yy += rs[c];
                            if (p.out_f16)
                                static_cast<uint16_t*>(Yp)[o] = __half_as_ushort(__float2half_rn(yy));
                            else
                                static_cast<float*>(Yp)[o] = yy;
                        }
                    }
                }
            }
#undef yN
#undef Yp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) q4d::mbar_arrive(q4d::smem_addr(&sm.acc_empty[buf]));
        }
    }

    // Wind down: every role has left its loop (all waits are bounded).  The
    // last accumulator hand-off already waited for all issued MMAs; on abort
    // give in-flight tensor-core work a bounded moment via one more commit
    // from each issuer.
    tc_fence_before();
    __syncthreads();
    if (warp == kUpMmaWarp && sm.abort) {
        if (lane == 0) {
            // completes once every MMA of both issuers has finished
            mma_commit(q4d::smem_addr(&sm.drain));
            q4d::mbar_wait(q4d::smem_addr(&sm.drain), 0, nullptr);
        }
        __syncwarp();
    }
    if (warp == 1) {
        if (sm.abort) {
            if (lane == 0) {
                // completes once every MMA this thread issued has finished
                mma_commit(q4d::smem_addr(&sm.drain));
                q4d::mbar_wait(q4d::smem_addr(&sm.drain), 0, nullptr);
            }
            __syncwarp();
        }
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// Sum of the K parts of a split launch, then the epilogue the unsplit kernel
// applies: SiLU(g) * u in GLU mode, + residual, fp16 or fp32 store.  Four
// outputs per thread (N is a multiple of 128).
__global__ void reduce_parts_kernel(const float* __restrict__ part, int kparts, int nmat, int R, int N, int glu,
                                    const uint16_t* residual, void* Y, int out_f16) {
    const size_t pr = (size_t)R * N;
    const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= pr) return;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int k = 0; k < kparts; ++k) {
        const float4 a = *reinterpret_cast<const float4*>(part + (size_t)(k * nmat) * pr + i);
        g = make_float4(g.x + a.x, g.y + a.y, g.z + a.z, g.w + a.w);
        if (glu) {
            const float4 b = *reinterpret_cast<const float4*>(part + (size_t)(k * nmat + 1) * pr + i);
            u = make_float4(u.x + b.x, u.y + b.y, u.z + b.z, u.w + b.w);
        }
    }
    float y[4] = {g.x, g.y, g.z, g.w};
    const float uu[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        if (glu) y[e] = y[e] / (1.0f + expf(-y[e])) * uu[e];
        if (residual) y[e] += __half2float(__ushort_as_half(residual[i + e]));
    }
    if (out_f16) {
        uint16_t* o = static_cast<uint16_t*>(Y) + i;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = __half_as_ushort(__float2half_rn(y[e]));
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(Y) + i) = make_float4(y[0], y[1], y[2], y[3]);
    }
}

}  // namespace q4g

namespace q4i {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    // looked up once (thread-safe initialisation of a function-local static)
    static const EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}

q4_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(Q4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return Q4_OK;
}

namespace {


// One launch of the grouped GEMM.  Routed (offsets != NULL): E experts, rows
// of W_e at e * rows_e, the up matrix at + N rows of the same arrays.  Dense
// (offsets == NULL): one expert over rows 0..R-1, the up matrix given apart.
struct GroupedArgs {
    const uint32_t* Wq;
    const uint16_t *scales, *biases;
    const uint32_t* Wq_u;  // GLU: the up matrix (may be Wq)
    const uint16_t *scales_u, *biases_u;
    int up_off;            // row of the up matrix's first row within Wq_u's expert block
    const uint16_t* X;
    const int32_t *expert_ids, *offsets;
    void* Y;
    const uint16_t* residual;
    int E, N, K, R;
    q4_gemv_mode mode;
    q4_dtype out_dtype;
    int kparts = 1;        // split K over this many units (dense only); 1 = no split
    float* part = nullptr; // kparts > 1: fp32 [kparts][nmat][R][N]
    bool skip_reduce = false;  // kparts > 1: leave the partials for the caller to add
    // Several weight matrices of one input (dense PLAIN, no residual, no
    // split): matrix 0 is Wq / scales / biases / Y with N = seg_N[0], the
    // others follow; N is then their total.
    int nseg = 1;
    const uint32_t* seg_Wq[q4g::kMaxSeg] = {};
    const uint16_t* seg_s[q4g::kMaxSeg] = {};
    const uint16_t* seg_b[q4g::kMaxSeg] = {};
    void* seg_Y[q4g::kMaxSeg] = {};
    int seg_N[q4g::kMaxSeg] = {};
};

q4_status launch_grouped(const GroupedArgs& a, q4_stream_t stream) {
    if (a.E < 1 || a.E > q4g::kMaxExperts) return fail(Q4_ERR_INVALID_ARG, "E=%d outside 1..%d", a.E, q4g::kMaxExperts);
    if (a.K < 64 || a.K % 64) return fail(Q4_ERR_INVALID_ARG, "K=%d is not a positive multiple of 64", a.K);
    if (a.N < 1) return fail(Q4_ERR_INVALID_ARG, "N=%d", a.N);
    if (a.N % 128) return fail(Q4_ERR_UNSUPPORTED, "N=%d is not a multiple of 128", a.N);
    if (a.R < 0) return fail(Q4_ERR_INVALID_ARG, "R=%d", a.R);
    if (a.mode != Q4_GEMV_PLAIN && a.mode != Q4_GEMV_GLU) return fail(Q4_ERR_INVALID_ARG, "bad mode");
    if (a.out_dtype != Q4_F32 && a.out_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "bad out_dtype");
    if (a.mode == Q4_GEMV_GLU && a.out_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "GLU mode writes fp16");
    if (a.residual && (a.mode != Q4_GEMV_PLAIN || a.out_dtype != Q4_F16))
        return fail(Q4_ERR_INVALID_ARG, "a residual needs PLAIN mode and fp16 output");
    const bool glu = a.mode == Q4_GEMV_GLU;
    if (!aligned16(a.Wq) || !aligned16(a.X) || !aligned16(a.scales) || !aligned16(a.biases) ||
        (glu && (!aligned16(a.Wq_u) || !aligned16(a.scales_u) || !aligned16(a.biases_u))))
        return fail(Q4_ERR_MISALIGNED, "Wq, X, scales and biases must be 16-byte aligned");
    if (a.nseg < 1 || a.nseg > q4g::kMaxSeg) return fail(Q4_ERR_INVALID_ARG, "nseg=%d", a.nseg);
    if (a.nseg > 1) {
        if (glu || a.offsets || a.residual || a.kparts > 1)
            return fail(Q4_ERR_INVALID_ARG, "several matrices need dense PLAIN mode without residual or split");
        int total = 0;
        for (int i = 0; i < a.nseg; ++i) {
            if (!a.seg_Wq[i] || !a.seg_s[i] || !a.seg_b[i] || !a.seg_Y[i])
                return fail(Q4_ERR_INVALID_ARG, "NULL pointer of matrix %d", i);
            if (a.seg_N[i] < 128 || a.seg_N[i] % 128)
                return fail(Q4_ERR_UNSUPPORTED, "N=%d of matrix %d is not a multiple of 128", a.seg_N[i], i);
            if (!aligned16(a.seg_Wq[i]) || !aligned16(a.seg_s[i]) || !aligned16(a.seg_b[i]))
                return fail(Q4_ERR_MISALIGNED, "matrix %d: Wq, scales and biases must be 16-byte aligned", i);
            total += a.seg_N[i];
        }
        if (total != a.N) return fail(Q4_ERR_INVALID_ARG, "N=%d is not the matrices' total %d", a.N, total);
    }
    const int rows_e = a.offsets ? (glu ? 2 : 1) * a.N : a.N;
    if ((long long)a.E * rows_e > (1ll << 31)) return fail(Q4_ERR_UNSUPPORTED, "too many weight rows");
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    if (a.R == 0) return Q4_OK;

    q4g::Params p = {};
    p.expert_ids = a.expert_ids;
    p.scales = a.scales;
    p.biases = a.biases;
    p.scales_u = a.scales_u;
    p.biases_u = a.biases_u;
    p.residual = a.residual;
    p.vec_out = aligned16(a.Y) && (!a.residual || aligned16(a.residual)) ? 1 : 0;
    p.nseg = a.nseg;
    for (int i = 0; i < q4g::kMaxSeg; ++i) p.seg_t0[i] = i == 0 ? 0 : INT_MAX;
    if (a.nseg == 1) {
        p.seg_s[0] = a.scales;
        p.seg_b[0] = a.biases;
        p.seg_Y[0] = a.Y;
        p.seg_N[0] = a.N;
    } else {
        for (int i = 0; i < a.nseg; ++i) {
            p.seg_s[i] = a.seg_s[i];
            p.seg_b[i] = a.seg_b[i];
            p.seg_Y[i] = a.seg_Y[i];
            p.seg_N[i] = a.seg_N[i];
            if (i > 0) p.seg_t0[i] = p.seg_t0[i - 1] + a.seg_N[i - 1] / q4g::kRows;
            if (!aligned16(a.seg_Y[i])) p.vec_out = 0;
        }
    }
    p.offsets = a.offsets;
    p.Y = a.Y;
    p.E = a.E;
    p.N = a.N;
    p.K = a.K;
    p.R = a.R;
    p.glu = glu;
    p.nmat = glu ? 2 : 1;
    p.rows_e = rows_e;
    p.up_off = a.up_off;
    p.out_f16 = a.out_dtype == Q4_F16;
    p.n_tiles = a.N / q4g::kRows;
    p.nK = a.K / q4g::kKS;
    p.G = a.K / 64;
    p.kparts = a.kparts > 1 ? a.kparts : 1;
    p.ksteps = p.nK / p.kparts;
    p.part = a.part;
    p.err = dev->err_word;

    // Rings: an A ring of up to 4 stages (4 in tensor memory; in shared
    // memory 4 when the scales come from global memory, else 3, or 2 in GLU
    // mode, whose stages are twice the size), giving up stages until the
    // input ring has 4, and an input ring as deep as the rest of shared
    // memory allows (up to 16): an input stage waits ~1 us for its codes,
    // so its depth sets the K-step rate; at least 2 of each.
    // Tokens per unit: a routed launch with few rows per expert takes a
    // smaller X box, so its input stages are smaller and the ring deeper (an
    // expert with more rows than that takes more units).
    p.tn = q4g::kTN;
    if (a.offsets) {
        const long long avg = ((long long)a.R + a.E - 1) / a.E;
        p.tn = avg <= 16 ? 32 : avg <= 48 ? 64 : q4g::kTN;
    }
    p.x_bytes = (uint32_t)p.tn * q4g::kKS * 2u;
    p.x_off = (uint32_t)p.nmat * q4g::kCodesBytes;
    p.in_bytes = p.x_off + p.x_bytes;
    // Units of at most 64 tokens leave half the 512 TMEM columns free of
    // accumulators (2 buffers x 2 accumulators x tn): the dequantised A
    // stages go there (4 stages x 2 matrices x 32 columns), not into shared
    // memory, which then holds only the input ring.
    p.a_tmem = p.tn <= 64 ? 1 : 0;
    if (p.a_tmem && p.nseg > 1) return fail(Q4_ERR_UNSUPPORTED, "several matrices need 128-token units");
    p.acc_cols = p.a_tmem ? (uint32_t)p.tn : (uint32_t)q4g::kTN;
    p.a_col0 = 256;
    p.a_bytes = p.a_tmem ? 0u : (uint32_t)p.nmat * q4g::kATileBytes;
    // The dequant warps keep each unit's scales and biases in shared memory
    // (a staging block the TMA thread fills, copied into private per-thread
    // slots), except with A in shared memory when that would take more than
    // 32 KB: then they read them from global memory (four groups to a load,
    // the unit's rows prefetched into L2), which leaves the room to the A
    // and input rings.  Staged values cost nothing at a unit's start, which
    // counts for units of few K steps.
    const size_t stg_need = ((size_t)p.nmat * 2 * q4g::kRows * p.G * 2 + 127) & ~size_t(127);
    const size_t sb_need = ((size_t)q4g::kDeqWarps * 32 * (p.G + 1) * 4 + 127) & ~size_t(127);
    p.sb_global = !p.a_tmem && stg_need + sb_need > 32768 ? 1 : 0;
    p.stg_bytes = p.sb_global ? 0u : (uint32_t)stg_need;
    p.sb_bytes = p.sb_global ? 0u : (uint32_t)sb_need;
    // The epilogue's staging tiles when Y (and the residual) are 16-byte
    // aligned and the rings keep their depth without them (else the
    // epilogue stores one value per lane and column).
    int as = 0, is = 0;
    for (int stage_tiles = p.vec_out; stage_tiles >= 0; --stage_tiles) {
        const size_t fixed = 1024 + (size_t)p.sb_bytes + p.stg_bytes + (stage_tiles ? q4g::kEpiStageBytes : 0u) +
                             sizeof(q4g::Smem);
        const size_t avail = (size_t)dev->smem_optin > fixed ? (size_t)dev->smem_optin - fixed : 0;
        as = p.a_tmem || p.sb_global ? q4g::kMaxAStages : glu ? 2 : 3;
        is = 0;
        if (p.a_tmem) {
            // the A stages live in TMEM: all of shared memory past the fixed
            // part goes to the input ring
            is = (int)(avail / p.in_bytes);
            if (is > q4g::kMaxInStages) is = q4g::kMaxInStages;
        } else {
            for (; as >= 2; --as) {
                const size_t left = avail > (size_t)as * p.a_bytes ? avail - (size_t)as * p.a_bytes : 0;
                is = (int)(left / p.in_bytes);
                if (is > q4g::kMaxInStages) is = q4g::kMaxInStages;
                if (is >= 4 || as == 2) break;
            }
        }
        p.vec_out = stage_tiles;
        if (as >= 2 && is >= 2) break;
    }
    if (as < 2 || is < 2)
        return fail(Q4_ERR_UNSUPPORTED, "K=%d: its scale/bias buffers leave no room for two pipeline stages", a.K);
    p.in_stages = is;
    p.a_stages = as;
    const size_t smem = 1024 + (size_t)p.sb_bytes + p.stg_bytes + (p.vec_out ? q4g::kEpiStageBytes : 0u) +
                        sizeof(q4g::Smem) + (size_t)is * p.in_bytes + (size_t)as * p.a_bytes;

    CUtensorMap tmW, tmWu, tmW2, tmX;
    const uint64_t wrows = a.nseg > 1 ? (uint64_t)a.seg_N[0] : (uint64_t)a.E * rows_e;
    st = make_map(&tmW, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.nseg > 1 ? a.seg_Wq[0] : a.Wq, (uint64_t)a.K / 2, wrows,
                  (uint64_t)a.K / 2, 32, q4g::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != Q4_OK) return st;
    tmWu = tmW;
    tmW2 = tmW;
    // several matrices: each its own map over its own rows (tmWu, tmW2)
    for (int i = 1; i < a.nseg; ++i) {
        st = make_map(i == 1 ? &tmWu : &tmW2, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.seg_Wq[i], (uint64_t)a.K / 2,
                      (uint64_t)a.seg_N[i], (uint64_t)a.K / 2, 32, q4g::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != Q4_OK) return st;
    }
    if (glu && a.Wq_u != a.Wq) {
        st = make_map(&tmWu, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.Wq_u, (uint64_t)a.K / 2, wrows, (uint64_t)a.K / 2, 32,
                      q4g::kRows, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != Q4_OK) return st;
    }
    st = make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.X, (uint64_t)a.K, (uint64_t)a.R, (uint64_t)a.K * 2,
                  q4g::kKS, (uint32_t)p.tn, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != Q4_OK) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    static std::atomic<int> smem_marks[5][64];
    // instantiation: A in TMEM; A in shared memory with staged / global
    // scales; the same two over several weight matrices
    const int inst = p.a_tmem ? 0 : (p.sb_global ? 2 : 1) + (p.nseg > 1 ? 2 : 0);
    const void* kern = inst == 0   ? reinterpret_cast<const void*>(q4g::q4_moe_gemm_kernel<true, false, false>)
                       : inst == 1 ? reinterpret_cast<const void*>(q4g::q4_moe_gemm_kernel<false, false, false>)
                       : inst == 2 ? reinterpret_cast<const void*>(q4g::q4_moe_gemm_kernel<false, true, false>)
                       : inst == 3 ? reinterpret_cast<const void*>(q4g::q4_moe_gemm_kernel<false, false, true>)
                                   : reinterpret_cast<const void*>(q4g::q4_moe_gemm_kernel<false, true, true>);
    cudaError_t e = ensure_smem_attr(kern, smem_marks[inst], (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(q4_moe_gemm_kernel)");
    const unsigned nb = dev->sms;
    if (inst == 0) q4g::q4_moe_gemm_kernel<true, false, false><<<nb, q4g::kThreads, smem, s>>>(tmW, tmWu, tmW2, tmX, p);
    else if (inst == 1)
        q4g::q4_moe_gemm_kernel<false, false, false><<<nb, q4g::kThreads, smem, s>>>(tmW, tmWu, tmW2, tmX, p);
    else if (inst == 2)
        q4g::q4_moe_gemm_kernel<false, true, false><<<nb, q4g::kThreads, smem, s>>>(tmW, tmWu, tmW2, tmX, p);
    else if (inst == 3)
        q4g::q4_moe_gemm_kernel<false, false, true><<<nb, q4g::kThreads, smem, s>>>(tmW, tmWu, tmW2, tmX, p);
    else
        q4g::q4_moe_gemm_kernel<false, true, true><<<nb, q4g::kThreads, smem, s>>>(tmW, tmWu, tmW2, tmX, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "grouped GEMM launch");
    if (p.kparts > 1 && !a.skip_reduce) {
        const size_t quads = (size_t)a.R * a.N / 4;
        q4g::reduce_parts_kernel<<<(unsigned)((quads + 255) / 256), 256, 0, s>>>(
            p.part, p.kparts, p.nmat, a.R, a.N, p.glu, a.residual, a.Y, p.out_f16);
        e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "split reduction launch");
    }
    return Q4_OK;
}

}  // namespace

// K parts for a dense GEMM whose output tiles do not fill the GPU: the
// largest divisor of the K steps whose units still fit one wave of 152 (one
// per SM of a GB300; a fixed target keeps workspace sizes computable without
// a device), with at least 4 K steps per unit.  Only for K of 2048 or more:
// with fewer K steps the partial sums' round trip and the reduction launch
// cost more than the idle SMs.  CUDA-event timings of the Qwen3-0.6B shapes
// at 512 tokens: K = 1024 is faster unsplit; o (K = 2048) takes 17.9 us in
// 4 parts against 22.7 us in 8 (two waves) and 24.8 us unsplit, down
// (K = 3072) 19.3 us in 4 parts against 22.8 us in 6 and 31.8 us unsplit.
constexpr int kSplitTargetUnits = 152;
constexpr int kSplitMinKSteps = 32;

int gemm_split_parts(int M, int N, int K) {
    if (M < 1 || N < 128 || K < 64) return 1;
    const int units = ((M + q4g::kTN - 1) / q4g::kTN) * (N / q4g::kRows);
    const int nK = K / q4g::kKS;
    const int sms = kSplitTargetUnits;
    if (units >= sms || nK < kSplitMinKSteps) return 1;
    int best = 1;
    for (int d = 2; d <= nK / 4; ++d) {
        if (nK % d) continue;
        if (units * d > sms) break;
        best = d;
    }
    return best;
}

size_t gemm_split_bytes(int M, int N, int K, bool glu) {
    const int kp = gemm_split_parts(M, N, K);
    return kp > 1 ? (size_t)kp * (glu ? 2 : 1) * (size_t)M * N * 4 : 0;
}

q4_status gemm_launch_multi(const q4_linear* w, void* const* Y, int nseg, const uint16_t* X, int M,
                            q4_stream_t stream) {
    if (!w || !Y || !X) return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (nseg < 1 || nseg > q4g::kMaxSeg) return fail(Q4_ERR_INVALID_ARG, "nseg=%d outside 1..%d", nseg, q4g::kMaxSeg);
    if (M < 0) return fail(Q4_ERR_INVALID_ARG, "M=%d", M);
    GroupedArgs a = {};
    a.nseg = nseg;
    a.N = 0;
    for (int i = 0; i < nseg; ++i) {
        if (w[i].K != w[0].K) return fail(Q4_ERR_INVALID_ARG, "matrix %d: K=%d, matrix 0: K=%d", i, w[i].K, w[0].K);
        a.seg_Wq[i] = w[i].Wq;
        a.seg_s[i] = w[i].scales;
        a.seg_b[i] = w[i].biases;
        a.seg_Y[i] = Y[i];
        a.seg_N[i] = w[i].N;
        a.N += w[i].N;
    }
    a.Wq = a.Wq_u = w[0].Wq;
    a.scales = a.scales_u = w[0].scales;
    a.biases = a.biases_u = w[0].biases;
    a.X = X;
    a.Y = Y[0];
    a.E = 1;
    a.K = w[0].K;
    a.R = M;
    a.mode = Q4_GEMV_PLAIN;
    a.out_dtype = Q4_F16;
    return launch_grouped(a, stream);
}

namespace {
q4_status gemm_launch_impl(const q4_gemm_desc* d, q4_stream_t stream, bool skip_reduce, int* kparts);
}  // namespace

q4_status gemm_launch(const q4_gemm_desc* d, q4_stream_t stream) {
    return gemm_launch_impl(d, stream, false, nullptr);
}

q4_status gemm_launch_parts(const q4_gemm_desc* d, q4_stream_t stream, int* kparts) {
    return gemm_launch_impl(d, stream, true, kparts);
}

namespace {
q4_status gemm_launch_impl(const q4_gemm_desc* d, q4_stream_t stream, bool skip_reduce, int* kparts) {
    if (kparts) *kparts = 1;
    if (!d) return fail(Q4_ERR_INVALID_ARG, "desc is NULL");
    const bool glu = d->mode == Q4_GEMV_GLU;
    if (!d->w.Wq || !d->w.scales || !d->w.biases || !d->X || !d->Y)
        return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (glu && (!d->up.Wq || !d->up.scales || !d->up.biases))
        return fail(Q4_ERR_INVALID_ARG, "GLU mode needs the up matrix");
    if (glu && (d->up.N != d->w.N || d->up.K != d->w.K))
        return fail(Q4_ERR_INVALID_ARG, "gate %dx%d and up %dx%d differ", d->w.N, d->w.K, d->up.N, d->up.K);
    if (d->M < 0) return fail(Q4_ERR_INVALID_ARG, "M=%d", d->M);
    GroupedArgs a = {};
    a.Wq = d->w.Wq;
    a.scales = d->w.scales;
    a.biases = d->w.biases;
    a.Wq_u = glu ? d->up.Wq : d->w.Wq;
    a.scales_u = glu ? d->up.scales : d->w.scales;
    a.biases_u = glu ? d->up.biases : d->w.biases;
    a.up_off = 0;
    a.X = d->X;
    a.Y = d->Y;
    a.residual = d->residual;
    a.E = 1;
    a.N = d->w.N;
    a.K = d->w.K;
    a.R = d->M;
    a.mode = d->mode;
    a.out_dtype = d->out_dtype;
    if (d->workspace && d->M > 0 && d->w.N % 128 == 0 && d->w.K % 64 == 0) {
        const size_t need = gemm_split_bytes(d->M, d->w.N, d->w.K, glu);
        if (need > 0 && d->workspace_bytes >= need && (reinterpret_cast<uintptr_t>(d->workspace) & 15u) == 0) {
            a.kparts = gemm_split_parts(d->M, d->w.N, d->w.K);
            a.part = static_cast<float*>(d->workspace);
        }
    }
    a.skip_reduce = skip_reduce && a.kparts > 1;
    if (kparts) *kparts = a.kparts;
    return launch_grouped(a, stream);
}
}  // namespace

}  // namespace q4i

using namespace q4i;

extern "C" q4_status q4_moe_gemm(const uint32_t* Wq, const uint16_t* scales, const uint16_t* biases,
                                 const uint16_t* X, const int32_t* expert_ids, const int32_t* offsets, void* Y,
                                 const q4_moe_desc* d, q4_stream_t stream) {
    clear_error();
    if (!d) return fail(Q4_ERR_INVALID_ARG, "desc is NULL");
    if (!Wq || !scales || !biases || !X || !expert_ids || !offsets || !Y)
        return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    GroupedArgs a = {};
    a.Wq = a.Wq_u = Wq;
    a.scales = a.scales_u = scales;
    a.biases = a.biases_u = biases;
    a.up_off = d->N;
    a.X = X;
    a.expert_ids = expert_ids;
    a.offsets = offsets;
    a.Y = Y;
    a.E = d->E;
    a.N = d->N;
    a.K = d->K;
    a.R = d->R;
    a.mode = d->mode;
    a.out_dtype = d->out_dtype;
    return launch_grouped(a, stream);
}

extern "C" size_t q4_gemm_workspace_bytes(int M, int N, int K, q4_gemv_mode mode) {
    clear_error();
    return gemm_split_bytes(M, N, K, mode == Q4_GEMV_GLU);
}

extern "C" q4_status q4_gemm(const q4_gemm_desc* desc, q4_stream_t stream) {
    clear_error();
    return gemm_launch(desc, stream);
}
