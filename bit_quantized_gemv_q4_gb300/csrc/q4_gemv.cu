// Group-64 GEMV for decode (M = 1) and batched decode (M = 2..8), with the
// dequantisation inside the dot product (BaseRT: optimal LLM inference on
// Apple Silicon with native Metal, §3.3 "Kernel fusion and specialisation"),
// several matrices sharing one x per launch (same section: fused operator
// sequences; "Mac on-device AI performance breakthrough" §2.2: Q, K, V merged
// into one product) and fused prologue/epilogues (RMSNorm of x, fp16 store,
// residual add, SiLU*up).  The code width is a template parameter: 4 bits
// (the main path) and 8 bits at M = 1..8, 2, 3, 5 and 6 bits at M = 1 (BaseRT
// §3.3 and §4.1: a kernel per quantisation format).
//
// GB300 design
// ------------
// * The output rows are cut into tiles of TR rows.  The rows of a tile are
//   contiguous in all three arrays (Wq row n is K/2 bytes, its scales and
//   biases K/32 bytes each), so one tile is three 1-D bulk copies
//   (cp.async.bulk) into shared memory, completed on an mbarrier.  One
//   producer warp keeps `stages` tiles in flight per CTA; the grid is at most
//   (SMs x CTAs per SM) persistent CTAs that walk the tiles round-robin.
// * Eight consumer warps dequantise and accumulate from shared memory.  A
//   uint32 of 8 codes becomes four fp16 pairs with one AND-OR each (the code
//   is OR-ed into the mantissa of 1024.0 or 64.0, giving 1024+q or 64+q
//   exactly); w = s*(M+q) + (b - M*s) is then one mixed-precision FMA
//   (fp16 x fp16 products are exact in fp32), and w*x is accumulated with the
//   packed fp32x2 FMA, two weights per instruction, in fp32.
// * x is converted once per CTA to fp32 (optionally RMS-normalised: the first
//   operation of a pre-norm sublayer, fused into the load -- the norm weights
//   are staged before the dependency wait, the sum of squares is reduced as x
//   streams in, and the scalar 1/rms multiplies the dot products), laid out so
//   each lane's operands are conflict-free 16-byte shared loads,
//   and reused across the rows a warp handles together.  A warp reduces all
//   the totals of its row batch at once with a transposing shuffle butterfly
//   (fixed order, so results are bit-reproducible); the lane that stores an
//   output fetches its residual before the dot products.
// * Under programmatic dependent launch the weight copies start before the
//   wait on the previous kernel (weights never depend on it); only the x load
//   and the epilogue wait.  Inside a decode step x may instead arrive as
//   tagged words that are polled (no wait for the previous grid), and the
//   whole step may run as one persistent cooperative launch whose stages
//   start on a completion counter (end of file).
// * Every wait is bounded; on expiry the kernel latches an error bit and
//   leaves.
#include <cuda_fp16.h>
#include <stdio.h>

#include <utility>

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4k {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 8;
// Barriers (full + empty per stage) and the RMSNorm reduction scratch.
constexpr uint32_t kBarBytes = 2 * kMaxStages * 8 + kConsumerWarps * 8 * 4;

struct Seg {
    const uint32_t* Wq;
    const uint16_t* s;
    const uint16_t* b;
    void* y;
    const uint16_t* res;
    uint32_t* y_tag;          // tagged copy of y (decode step), or nullptr
    const uint32_t* res_tag;  // tagged residual (decode step), or nullptr
    int N, ldy, tile_begin, tiles;
};

struct alignas(16) Params {
    Seg seg[Q4_MAX_SEGMENTS];
    const uint16_t* x;
    const uint32_t* x_tag;    // tagged x (decode step), or nullptr
    int nseg, K, ldx, TR, rows_per_tile, total_tiles, stages;
    int out_f16, glu, early_prefetch;
    int norm;                // RMSNorm of each x row on load
    const uint16_t* norm_w;  // fp16 [K] or nullptr (ones)
    float norm_eps;
    uint32_t stage_bytes, x_bytes;
    // decode-step tags: tag(stage) = 1 + (step * n_stages + stage) mod 65535
    const uint32_t* step_ctr;
    uint32_t* done_ctr;
    int stage, n_stages, x_stage, res_stage, last;
    int tile_base;  // persistent step: tiles of all earlier stages (round-robin origin)
    int bits;       // code width: 4 (8 codes per word) or 8 (4 codes per word)
    int* err;
};

__device__ __forceinline__ uint32_t tag_of(uint32_t step, int stage, int n_stages) {
    return 1u + (uint32_t)(((unsigned long long)step * (unsigned)n_stages + (unsigned)stage) % 65535ull);
}

// Poll tagged words until every tag equals `tag` (bounded; on expiry the
// error word is latched, whatever was read is used and false is returned).
template <int NW>
__device__ __forceinline__ bool poll_tagged(const uint32_t* src, uint32_t tag, uint32_t* w, int* err) {
    unsigned long long t0 = 0;
    while (true) {
        bool ok = true;
        if constexpr (NW == 8) {
            const uint4 a = q4d::ld_relaxed_v4(src), b = q4d::ld_relaxed_v4(src + 4);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        } else {
            w[0] = q4d::ld_relaxed(src);
        }
#pragma unroll
        for (int i = 0; i < NW; ++i) ok &= (w[i] >> 16) == tag;
        if (ok) return true;
        if (t0 == 0) {
            t0 = q4d::globaltimer();
        } else if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
            atomicOr(err, q4d::kErrTimeout);
            return false;
        }
        __nanosleep(100);  // let the producing kernel use the issue slots and L2
    }
}

// One warp waits for a sample of a tagged x (the last word of each 32nd of
// every row) before the whole CTA reads it: a poll then moves 128 bytes per
// row instead of the whole vector, which leaves L2 to the producing grid.
template <int M>
__device__ __forceinline__ void gate_tagged_x(const Params& p, uint32_t tag, int lane) {
    const int W = p.K / 32;  // words per 32nd of a row (K is a multiple of 64)
#pragma unroll
    for (int m = 0; m < M; ++m) {
        uint32_t w;
        if (!poll_tagged<1>(p.x_tag + (size_t)m * p.ldx + (size_t)(lane + 1) * W - 1, tag, &w, p.err)) break;
    }
    __syncwarp();
}

// Lane words (LW): how many uint32 (8 codes each) one lane handles per chunk.
template <int M>
struct Cfg {
    static constexpr int LW = (M == 1) ? 4 : (M == 2 ? 2 : 1);
    static constexpr int RB = (M == 1) ? 8 : (M <= 4 ? 4 : 2);  // rows processed together per warp
    static constexpr int XV = LW * 2 * M;        // float4 of x per lane per chunk
};

__device__ __forceinline__ void find_tile(const Params& p, int t, int& si, int& n0, int& nrows) {
    si = 0;
    if (!p.glu) {
#pragma unroll
        for (int i = 1; i < Q4_MAX_SEGMENTS; ++i)
            if (i < p.nseg && t >= p.seg[i].tile_begin) si = i;
    }
    n0 = (t - p.seg[si].tile_begin) * p.TR;
    nrows = min(p.TR, p.seg[si].N - n0);
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ void issue_rows(const Params& p, const Seg& sg, int n0, int nrows, int row_off,
                                           uint8_t* stage, uint32_t full_bar, int lane, uint64_t pol) {
    const int K = p.K, G = K / 64, R = p.rows_per_tile;
    const int crb = K * p.bits / 8;  // code bytes per row
    const uint32_t wq_bytes = (uint32_t)nrows * (uint32_t)crb;
    const uint32_t sb_bytes = (uint32_t)nrows * (uint32_t)G * 2u;
    uint8_t* wq_dst = stage + (size_t)row_off * crb;
    uint8_t* s_dst = stage + (size_t)R * crb + (size_t)row_off * G * 2;
    uint8_t* b_dst = s_dst + (size_t)R * G * 2;
    const uint32_t* wq_src = sg.Wq + (size_t)n0 * (crb / 4);
    const uint16_t* s_src = sg.s + (size_t)n0 * G;
    const uint16_t* b_src = sg.b + (size_t)n0 * G;
    if ((wq_bytes & 15u) == 0) {
        if (lane == 0) q4d::bulk_g2s_evict_first(q4d::smem_addr(wq_dst), wq_src, wq_bytes, full_bar, pol);
    } else {
        // A ragged last tile of 3- or 5-bit codes whose code block is not a
        // 16-byte multiple: the producer lanes copy it word by word.
        uint32_t* wd = reinterpret_cast<uint32_t*>(wq_dst);
        for (uint32_t i = lane; i < wq_bytes / 4; i += 32) wd[i] = __ldg(wq_src + i);
    }
    if ((sb_bytes & 15u) == 0) {
        if (lane == 0) {
            q4d::bulk_g2s(q4d::smem_addr(s_dst), s_src, sb_bytes, full_bar);
            q4d::bulk_g2s(q4d::smem_addr(b_dst), b_src, sb_bytes, full_bar);
        }
    } else {
        // Ragged last tile whose scale block is not a 16-byte multiple: the
        // producer lanes copy it with ordinary loads.
        uint16_t* sd = reinterpret_cast<uint16_t*>(s_dst);
        uint16_t* bd = reinterpret_cast<uint16_t*>(b_dst);
        for (uint32_t i = lane; i < sb_bytes / 2; i += 32) {
            sd[i] = __ldg(s_src + i);
            bd[i] = __ldg(b_src + i);
        }
    }
}

// Bytes the bulk copies of one segment's rows bring in (the expect-tx count).
__device__ __forceinline__ uint32_t bulk_bytes(const Params& p, int nrows) {
    const uint32_t wq_b = (uint32_t)nrows * (uint32_t)(p.K * p.bits / 8);
    const uint32_t sb_b = (uint32_t)nrows * (uint32_t)(p.K / 64) * 2u;
    return (((wq_b & 15u) == 0) ? wq_b : 0) + (((sb_b & 15u) == 0) ? 2 * sb_b : 0);
}

// ------------------------------------------------------------------ consumer
// The same for 8-bit codes: two words a, b hold the 8 codes of one octet
// (codes 0-3 in a, 4-7 in b, lowest byte first).  Masking every other byte
// and OR-ing it into the mantissa of 1024.0 gives 1024+q exactly (q <= 255);
// the pairs are (q0,q2), (q1,q3), (q4,q6), (q5,q7) and x is staged in that
// pairing for 8-bit matrices (see load_x).
template <int M>
__device__ __forceinline__ void word_mac8(uint32_t a, uint32_t b, uint16_t sh, float c1024, const float4* xa,
                                          const float4* xb, float2* acc) {
    const uint32_t v0 = q4d::and_or(a, 0x00FF00FFu, 0x64006400u);       // 1024+q0, 1024+q2
    const uint32_t v1 = q4d::and_or(a >> 8, 0x00FF00FFu, 0x64006400u);  // 1024+q1, 1024+q3
    const uint32_t v2 = q4d::and_or(b, 0x00FF00FFu, 0x64006400u);       // 1024+q4, 1024+q6
    const uint32_t v3 = q4d::and_or(b >> 8, 0x00FF00FFu, 0x64006400u);  // 1024+q5, 1024+q7
    const float2 d0 = q4d::fma_h2_s_f32(v0, sh, c1024);
    const float2 d1 = q4d::fma_h2_s_f32(v1, sh, c1024);
    const float2 d2 = q4d::fma_h2_s_f32(v2, sh, c1024);
    const float2 d3 = q4d::fma_h2_s_f32(v3, sh, c1024);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        acc[m] = __ffma2_rn(d0, make_float2(xa[m].x, xa[m].y), acc[m]);
        acc[m] = __ffma2_rn(d1, make_float2(xa[m].z, xa[m].w), acc[m]);
        acc[m] = __ffma2_rn(d2, make_float2(xb[m].x, xb[m].y), acc[m]);
        acc[m] = __ffma2_rn(d3, make_float2(xb[m].z, xb[m].w), acc[m]);
    }
}

// 2-, 3-, 5- and 6-bit codes (M = 1): a lane's 32 codes are exactly BITS
// words of the row's little-endian bit stream.  Code c sits at bit BITS*c;
// one funnel shift brings it to the bottom of a register and one AND-OR puts
// it under the mantissa of 1024.0 in the low half (1024+q, exact), so each
// code is dequantised by one mixed-precision FMA on a low half, and pairs of
// codes meet their x in the packed fp32x2 FMA.
template <int BITS, int C>
__device__ __forceinline__ uint32_t code_at(const uint32_t* w) {
    constexpr int P = BITS * C, W = P >> 5, S = P & 31;
    uint32_t v;
    if constexpr (S == 0) {
        v = w[W];
    } else if constexpr (S + BITS <= 32) {
        v = w[W] >> S;
    } else {
        v = __funnelshift_r(w[W], w[W + 1], S);
    }
    return q4d::and_or(v, (1u << BITS) - 1u, 0x6400u);
}

__device__ __forceinline__ float fma_lo_s_f32(uint32_t v, uint16_t s, float c) {
    float r;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; fma.rn.f32.f16 %0, l, %2, %3; }" : "=f"(r) : "r"(v), "h"(s), "f"(c));
    return r;
}

template <int BITS, int C>
__device__ __forceinline__ void pair_mac(const uint32_t* w, uint16_t sh, float c1024, const float4* xr, float2& acc) {
    const float wa = fma_lo_s_f32(code_at<BITS, C>(w), sh, c1024);
    const float wb = fma_lo_s_f32(code_at<BITS, C + 1>(w), sh, c1024);
    const float4 xq = xr[C / 4];
    const float2 xp = (C % 4 == 0) ? make_float2(xq.x, xq.y) : make_float2(xq.z, xq.w);
    acc = __ffma2_rn(make_float2(wa, wb), xp, acc);
}

template <int BITS, int... Cs>
__device__ __forceinline__ void chunk_mac(const uint32_t* w, uint16_t sh, float c1024, const float4* xr, float2& acc,
                                          std::integer_sequence<int, Cs...>) {
    (pair_mac<BITS, 2 * Cs>(w, sh, c1024, xr, acc), ...);
}

template <int LW>
__device__ __forceinline__ void load_words(const uint32_t* src, uint32_t* w) {
    if constexpr (LW == 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        const uint4 u = *reinterpret_cast<const uint4*>(src + 4);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
        w[4] = u.x;
        w[5] = u.y;
        w[6] = u.z;
        w[7] = u.w;
    } else if constexpr (LW == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(src);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else if constexpr (LW == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(src);
        w[0] = v.x;
        w[1] = v.y;
    } else {
        w[0] = *src;
    }
}

// Dot products of RB tile rows (shared-memory row indices `rows`) with all M
// x vectors; every lane ends with all RB*M totals.  A lane handles LW octets
// (8 codes each: one 4-bit word or two 8-bit words) per chunk.
template <int M, int RB, int BITS>
__device__ __forceinline__ void dot_rows(const Params& p, const uint32_t* wq, const uint16_t* ss,
                                         const uint16_t* bs, const float4* xs, const int* rows, int lane,
                                         float (*out)[M]) {
    constexpr int LW = Cfg<M>::LW, XV = Cfg<M>::XV;
    const int W8 = p.K / 8, G = p.K / 64;
    const int chunk_words = 32 * LW;
    const int nchunks = (W8 + chunk_words - 1) / chunk_words;
    float2 acc[RB][M];
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = make_float2(0.f, 0.f);

    if constexpr (BITS != 4 && BITS != 8) {
        static_assert(M == 1 && LW == 4, "2/3/5/6-bit codes: M = 1 (32 codes per lane chunk)");
        const int words_row = W8 * BITS / 4;
        for (int c = 0; c < nchunks; ++c) {
            const int j0 = c * chunk_words + lane * LW;
            if (j0 < W8) {
                float4 xr[XV];
                const float4* xc = xs + (size_t)c * XV * 32 + lane;
#pragma unroll
                for (int i = 0; i < XV; ++i) xr[i] = xc[i * 32];
                const int g = j0 >> 3;
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const uint32_t* src = wq + (size_t)rows[r] * words_row + j0 * BITS / 4;
                    uint32_t w[BITS];
#pragma unroll
                    for (int i = 0; i < BITS; ++i) w[i] = src[i];
                    const uint16_t sh = ss[rows[r] * G + g];
                    const float sf = __half2float(__ushort_as_half(sh));
                    const float c1024 = fmaf(-1024.f, sf, __half2float(__ushort_as_half(bs[rows[r] * G + g])));
                    chunk_mac<BITS>(w, sh, c1024, xr, acc[r][0], std::make_integer_sequence<int, 16>{});
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) out[r][0] = acc[r][0].x + acc[r][0].y;
    } else {
        for (int c = 0; c < nchunks; ++c) {
            const int j0 = c * chunk_words + lane * LW;
            if (j0 < W8) {
                float4 xr[XV];
                const float4* xc = xs + (size_t)c * XV * 32 + lane;
#pragma unroll
                for (int i = 0; i < XV; ++i) xr[i] = xc[i * 32];
                const int g = j0 >> 3;
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    constexpr int WPO = BITS / 4;  // words per octet
                    uint32_t w[LW * WPO];
                    load_words<LW * WPO>(wq + ((size_t)rows[r] * W8 + j0) * WPO, w);
                    const uint16_t sh = ss[rows[r] * G + g];
                    const uint16_t bh = bs[rows[r] * G + g];
                    const float sf = __half2float(__ushort_as_half(sh));
                    const float bf = __half2float(__ushort_as_half(bh));
                    const float c1024 = fmaf(-1024.f, sf, bf);
                    const float c64 = fmaf(-64.f, sf, bf);
#pragma unroll
                    for (int wi = 0; wi < LW; ++wi) {
                        if constexpr (BITS == 4)
                            q4d::word_mac<M>(w[wi], sh, c1024, c64, &xr[(wi * 2 + 0) * M], &xr[(wi * 2 + 1) * M], acc[r]);
                        else
                            word_mac8<M>(w[2 * wi], w[2 * wi + 1], sh, c1024, &xr[(wi * 2 + 0) * M],
                                         &xr[(wi * 2 + 1) * M], acc[r]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) out[r][m] = acc[r][m].x + acc[r][m].y;
    }
}

// Sum V values (power of two, V <= 32) across the 32 lanes of a warp with a
// transposing butterfly: each halving round exchanges half of the values
// still held, so V values cost about 4*(V-1) + 2*(5 - log2 V) instructions
// instead of 10*V.  On return lane L holds the total of value index
// (L >> (5 - log2 V)) in v[0]; the order of additions is fixed.
template <int V>
__device__ __forceinline__ void warp_sum_transpose(float* v, int lane) {
    constexpr int LOGV = (V >= 32) ? 5 : (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
    int n = V;
#pragma unroll
    for (int r = 0; r < LOGV; ++r) {
        const int o = 16 >> r;
        const bool upper = (lane & o) != 0;
        const int half = n >> 1;
#pragma unroll
        for (int i = 0; i < V / 2; ++i) {
            if (i < half) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        n = half;
    }
#pragma unroll
    for (int o = 16 >> LOGV; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

// fp16 store of one output, plus its tagged copy when the stage publishes one.
__device__ __forceinline__ void store_f16(const Seg& sg, size_t i, float v, uint32_t tag) {
    const uint16_t h = __half_as_ushort(__float2half_rn(v));
    reinterpret_cast<uint16_t*>(sg.y)[i] = h;
    if (sg.y_tag) q4d::st_relaxed(sg.y_tag + i, (tag << 16) | h);
}

// The residual word of output i, read before the dot products so its latency
// overlaps them: a tagged word (checked, and polled again if not yet current,
// by add_residual) or a plain fp16 value.
__device__ __forceinline__ uint32_t prefetch_residual(const Seg& sg, size_t i) {
    if (sg.res_tag) return q4d::ld_relaxed(sg.res_tag + i);
    if (sg.res) return sg.res[i];
    return 0;
}

__device__ __forceinline__ bool store_out(const Params& p, const Seg& sg, int m, int n, float v, uint32_t ytag,
                                          uint32_t rtag, uint32_t resw) {
    const size_t i = (size_t)m * sg.ldy + n;
    bool ok = true;
    if (p.out_f16) {
        if (sg.res_tag) {
            if ((resw >> 16) != rtag) ok = poll_tagged<1>(sg.res_tag + i, rtag, &resw, p.err);
            v += __half2float(__ushort_as_half((uint16_t)(resw & 0xFFFFu)));
        } else if (sg.res) {
            v += __half2float(__ushort_as_half((uint16_t)resw));
        }
        store_f16(sg, i, v, ytag);
    } else {
        reinterpret_cast<float*>(sg.y)[i] = v;
    }
    return ok;
}

template <int M, int RB, int BITS>
__device__ __forceinline__ bool tile_batch(const Params& p, const uint32_t* wq, const uint16_t* ss,
                                           const uint16_t* bs, const float4* xs, const float* scale, int warp,
                                           int lane, int j_begin, int rpw, int si, int n0, int nrows,
                                           uint32_t ytag, uint32_t rtag) {
    int rows[RB];
    int locals[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const int j = j_begin + r;
        if (p.glu) {
            // gate row and up row of the same output interleave: (g0, u0, g1, u1, ...)
            const int local = warp * (rpw / 2) + (j >> 1);
            locals[r] = local;
            rows[r] = (j & 1) ? p.TR + local : local;
        } else {
            locals[r] = warp * rpw + j;
            rows[r] = locals[r];
        }
    }
    // After the reduction below lane L holds value index idx = L >> SH
    // (idx = r*M + m), and the lanes with L % 2^SH == 0 store it.  Which
    // output a lane stores is known now, so its residual is fetched first.
    constexpr int V = RB * M;
    constexpr int VP = (V > 16) ? 32 : (V > 8) ? 16 : (V > 4) ? 8 : (V > 2) ? 4 : (V > 1) ? 2 : 1;  // power of two
    constexpr int SH = 5 - ((VP >= 32) ? 5 : (VP >= 16) ? 4 : (VP >= 8) ? 3 : (VP >= 4) ? 2 : (VP >= 2) ? 1 : 0);
    const int idx_raw = lane >> SH;
    const bool holds = idx_raw < V;   // lanes past V hold padding
    const int idx = holds ? idx_raw : 0;
    const int r_l = idx / M, m_l = idx - r_l * M;
    int local = 0;
    float sc = 1.0f;
#pragma unroll
    for (int r = 0; r < RB; ++r)
        if (r == r_l) local = locals[r];
#pragma unroll
    for (int m = 0; m < M; ++m)
        if (m == m_l) sc = scale[m];
    const bool storer = holds && (lane & ((1 << SH) - 1)) == 0 && local < nrows;
    uint32_t resw = 0;
    if (!p.glu && storer && p.out_f16) {
        const Seg& sg = p.seg[si];
        resw = prefetch_residual(sg, (size_t)m_l * sg.ldy + n0 + local);
    }

    float out[RB][M];
    dot_rows<M, RB, BITS>(p, wq, ss, bs, xs, rows, lane, out);
    // Reduce all RB*M values at once.
    float v[VP];
#pragma unroll
    for (int i = V; i < VP; ++i) v[i] = 0.f;
#pragma unroll
    for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) v[r * M + m] = out[r][m];
    warp_sum_transpose<VP>(v, lane);
    const float y = v[0] * sc;
    if (p.glu) {
        // gate (even r) and up (odd r) of one output row: the up total sits M
        // value indices further on
        const float u = __shfl_down_sync(0xffffffffu, y, M << SH);
        if (storer && (r_l & 1) == 0) {
            const float a = y / (1.0f + expf(-y)) * u;
            const Seg& sg = p.seg[0];
            store_f16(sg, (size_t)m_l * sg.ldy + n0 + local, a, ytag);
        }
    } else if (storer) {
        return store_out(p, p.seg[si], m_l, n0 + local, y, ytag, rtag, resw);
    }
    return true;
}

// 8 consecutive fp16 values (16 bytes) as fp32.
__device__ __forceinline__ void load8_f32(const uint16_t* src, float* f) {
    const uint4 raw = *reinterpret_cast<const uint4*>(src);
    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&wv[h]));
        f[2 * h] = t.x;
        f[2 * h + 1] = t.y;
    }
}

// Shared-memory float4 slots of x word j (8 values) for row m, in the
// lane-interleaved pair layout the dot product reads.
template <int M>
__device__ __forceinline__ float4* x_slot(float4* xs, int j, int m, int half) {
    constexpr int LW = Cfg<M>::LW, XV = Cfg<M>::XV;
    const int c = j / (32 * LW), rem = j % (32 * LW), l = rem / LW, wi = rem % LW;
    return xs + ((size_t)c * XV + (wi * 2 + half) * M + m) * 32 + l;
}

// Consumers, before the dependency wait: the RMSNorm weights (a weight, not
// an activation) are staged into the x slots so the post-wait pass only
// multiplies.
// Shared-memory order of one octet's 8 values: the pairing the dequantised
// pairs meet (4-bit: (0,4) (1,5) | (2,6) (3,7); 8-bit: (0,2) (1,3) | (4,6) (5,7)).
template <int BITS>
__device__ __forceinline__ void octet_halves(const float* f, float4& a, float4& b) {
    if constexpr (BITS == 4) {
        a = make_float4(f[0], f[4], f[1], f[5]);
        b = make_float4(f[2], f[6], f[3], f[7]);
    } else if constexpr (BITS == 8) {
        a = make_float4(f[0], f[2], f[1], f[3]);
        b = make_float4(f[4], f[6], f[5], f[7]);
    } else {  // 2, 3, 5, 6 bits: codes are dequantised one by one, pairs in order
        a = make_float4(f[0], f[1], f[2], f[3]);
        b = make_float4(f[4], f[5], f[6], f[7]);
    }
}

template <int M, int BITS>
__device__ __forceinline__ void stage_norm_weight(const Params& p, float4* xs) {
    constexpr int kCT = kConsumerWarps * 32;
    const int W8 = p.K / 8;
    for (int j = threadIdx.x; j < W8; j += kCT) {
        float g[8];
        load8_f32(p.norm_w + 8 * j, g);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float4 a, b;
            octet_halves<BITS>(g, a, b);
            *x_slot<M>(xs, j, m, 0) = a;
            *x_slot<M>(xs, j, m, 1) = b;
        }
    }
}

// Consumers, after the dependency wait: x (times the staged norm weights, if
// any) into shared memory as fp32 in one pass over global memory.  With the
// RMSNorm the per-row sum of squares is reduced on the way (thread partials,
// warp xor tree; the warps' partials are added in index order by
// norm_scales); the scalar 1/rms is applied to the dot products in the
// epilogue, so x is read once.
template <int M, int BITS>
__device__ __forceinline__ bool load_x(const Params& p, float4* xs, float* red, int warp, int lane, uint32_t xtag,
                                       const uint16_t* gamma_sm = nullptr) {
    constexpr int kCT = kConsumerWarps * 32;
    const int W8 = p.K / 8;
    const bool gw = p.norm && p.norm_w;
    bool ok = true;
    float ss[M];
#pragma unroll
    for (int m = 0; m < M; ++m) ss[m] = 0.f;
    for (int j = threadIdx.x; j < W8; j += kCT) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float f[8];
            if (p.x_tag) {
                uint32_t w[8];
                if (ok) {
                    ok = poll_tagged<8>(p.x_tag + (size_t)m * p.ldx + 8 * j, xtag, w, p.err);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) w[e] = 0;  // after a timeout: no further waits
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = __half2float(__ushort_as_half((uint16_t)(w[e] & 0xFFFFu)));
            } else {
                load8_f32(p.x + (size_t)m * p.ldx + 8 * j, f);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) ss[m] = fmaf(f[e], f[e], ss[m]);
            float4* d0 = x_slot<M>(xs, j, m, 0);
            float4* d1 = x_slot<M>(xs, j, m, 1);
            float4 a, b;
            octet_halves<BITS>(f, a, b);
            if (gamma_sm) {
                float g[8];
                load8_f32(gamma_sm + 8 * j, g);
                float4 ga, gb;
                octet_halves<BITS>(g, ga, gb);
                a = make_float4(a.x * ga.x, a.y * ga.y, a.z * ga.z, a.w * ga.w);
                b = make_float4(b.x * gb.x, b.y * gb.y, b.z * gb.z, b.w * gb.w);
            } else if (gw) {
                const float4 ga = *d0, gb = *d1;
                a = make_float4(a.x * ga.x, a.y * ga.y, a.z * ga.z, a.w * ga.w);
                b = make_float4(b.x * gb.x, b.y * gb.y, b.z * gb.z, b.w * gb.w);
            }
            *d0 = a;
            *d1 = b;
        }
    }
    if (p.norm) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss[m] += __shfl_xor_sync(0xffffffffu, ss[m], o);
            if (lane == 0) red[warp * M + m] = ss[m];
        }
    }
    return ok;
}

// 1/sqrt(mean(x^2) + eps) per row (after the barrier that follows load_x).
template <int M>
__device__ __forceinline__ void norm_scales(const Params& p, const float* red, float* scale) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
        float t = 0.f;
        if (p.norm) {
            for (int w = 0; w < kConsumerWarps; ++w) t += red[w * M + m];
            scale[m] = rsqrtf(t / (float)p.K + p.norm_eps);
        } else {
            scale[m] = 1.0f;
        }
    }
}

// One consumer warp's share of tile t (its rows, all M vectors), read from the
// shared-memory stage that holds the tile.  False if a residual wait expired.
template <int M, int BITS>
__device__ __forceinline__ bool consume_tile(const Params& p, const uint8_t* stage, const float4* xs,
                                             const float* scale, int warp, int lane, int t, uint32_t ytag,
                                             uint32_t rtag) {
    constexpr int RB = Cfg<M>::RB;
    const int K = p.K, G = K / 64, R = p.rows_per_tile;
    const int rpw = R / kConsumerWarps;  // rows per warp per tile (1, 2, 4, 8)
    const uint32_t* wq = reinterpret_cast<const uint32_t*>(stage);
    const uint16_t* ss = reinterpret_cast<const uint16_t*>(stage + (size_t)R * (K * BITS / 8));
    const uint16_t* bs = ss + (size_t)R * G;
    int si, n0, nrows;
    find_tile(p, t, si, n0, nrows);
    bool ok = true;
    if (rpw >= RB) {
        for (int j = 0; j < rpw; j += RB)
            ok &= tile_batch<M, RB, BITS>(p, wq, ss, bs, xs, scale, warp, lane, j, rpw, si, n0, nrows, ytag, rtag);
    } else if (rpw == 4) {
        ok = tile_batch<M, (RB < 4 ? RB : 4), BITS>(p, wq, ss, bs, xs, scale, warp, lane, 0, rpw, si, n0, nrows,
                                                    ytag, rtag);
    } else if (rpw == 2) {
        ok = tile_batch<M, 2, BITS>(p, wq, ss, bs, xs, scale, warp, lane, 0, rpw, si, n0, nrows, ytag, rtag);
    } else {
        ok = tile_batch<M, 1, BITS>(p, wq, ss, bs, xs, scale, warp, lane, 0, rpw, si, n0, nrows, ytag, rtag);
    }
    return ok;
}

template <int M, int BITS>
__global__ void __launch_bounds__(kThreads, 2) q4_gemv_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages;
    float4* xs = reinterpret_cast<float4*>(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.x_bytes);
    float* red = reinterpret_cast<float*>(bars + 2 * kMaxStages);
    uint8_t* stages = smem + p.x_bytes + kBarBytes;
    const uint32_t full0 = q4d::smem_addr(bars), empty0 = q4d::smem_addr(bars + kMaxStages);

    __shared__ uint32_t step_sh;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            q4d::mbar_init(full0 + 8 * i, 32);               // every producer lane arrives
            q4d::mbar_init(empty0 + 8 * i, kConsumerWarps);  // one arrival per consumer warp
        }
        q4d::fence_mbar_init();
        // decode-step counter, read at launch (off the critical path when the
        // kernel was launched early)
        step_sh = p.step_ctr ? q4d::ld_relaxed(p.step_ctr) : 0u;
    }
    __syncthreads();
    // With a plain x the dependents may launch at once (they only stream
    // weights until this grid completes); with a tagged x they launch once
    // this grid holds its x, so at most one grid polls at a time.
    if (!p.x_tag) q4d::pdl_trigger();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer warp
        if (!p.early_prefetch) q4d::pdl_wait();
        const uint64_t pol = q4d::policy_evict_first();
        int i = 0;
        for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++i) {
            const int st = i % S, k = i / S;
            if (k > 0) {
                // lane 0 waits (suspended in hardware); the others park at the shuffle
                int ok = 1;
                if (lane == 0) ok = q4d::mbar_wait(empty0 + 8 * st, (k - 1) & 1, p.err) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) return;
            }
            int si, n0, nrows;
            find_tile(p, t, si, n0, nrows);
            uint8_t* stage = stages + (size_t)st * p.stage_bytes;
            const uint32_t fb = full0 + 8 * st;
            // Expected bytes first, then the copies; the phase completes only
            // when all 32 lanes have arrived and every byte has landed.
            const uint32_t expect = (p.glu ? 2u : 1u) * bulk_bytes(p, nrows);
            if (lane == 0)
                asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(expect)
                             : "memory");
            __syncwarp();
            issue_rows(p, p.seg[si], n0, nrows, 0, stage, fb, lane, pol);
            if (p.glu) issue_rows(p, p.seg[1], n0, nrows, p.TR, stage, fb, lane, pol);
            q4d::mbar_arrive(fb);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    if (p.norm && p.norm_w) stage_norm_weight<M, BITS>(p, xs);
    uint32_t xtag = 0, ytag = 0, rtag = 0;
    if (p.step_ctr) {
        const uint32_t step = step_sh;
        xtag = tag_of(step, p.x_stage, p.n_stages);
        ytag = tag_of(step, p.stage, p.n_stages);
        rtag = tag_of(step, p.res_stage, p.n_stages);
    }
    // A tagged x is polled directly (its producer may still be running); a
    // plain x and plain residuals wait for the previous grid to complete.
    if (!p.x_tag) {
        q4d::pdl_wait();
    } else {
        if (warp == 0) gate_tagged_x<M>(p, xtag, lane);
        q4d::named_bar(1, kConsumerWarps * 32);
    }
    load_x<M, BITS>(p, xs, red, warp, lane, xtag);
    q4d::named_bar(1, kConsumerWarps * 32);
    if (p.x_tag) q4d::pdl_trigger();
    float scale[M];
    norm_scales<M>(p, red, scale);

    int i = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++i) {
        const int st = i % S, k = i / S;
        // on a timeout leave the loop (not the kernel): every consumer warp
        // must still reach the barrier below
        if (!q4d::mbar_wait(full0 + 8 * st, k & 1, p.err)) break;
        consume_tile<M, BITS>(p, stages + (size_t)st * p.stage_bytes, xs, scale, warp, lane, t, ytag, rtag);
        __syncwarp();
        if (lane == 0) q4d::mbar_arrive(empty0 + 8 * st);
    }
    if (p.last) {
        // The last stage of a decode step: the last CTA to finish advances the
        // step counter (every CTA of this launch read it at its start).
        q4d::named_bar(1, kConsumerWarps * 32);
        if (threadIdx.x == 0) {
            __threadfence();
            if (atomicAdd(p.done_ctr, 1u) == gridDim.x - 1) {
                *p.done_ctr = 0;
                atomicAdd(const_cast<uint32_t*>(p.step_ctr), 1u);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Persistent decode step.  One CTA per SM (a cooperative launch, so all CTAs
// are resident together) walks every stage of the step in order, which
// removes the per-stage kernel launch and grid-completion wait.  The tiles of
// all stages are numbered one after another and dealt round-robin to the
// CTAs.  Because weights never depend on activations, the producer warp
// streams a CTA's tiles through one shared-memory ring across stage
// boundaries, as far ahead as the ring allows; the consumers of stage s wait
// only for their x.  Hand-off: a CTA that owns tiles of a stage adds one to a
// stage-completion counter after its last tile of that stage (release); the
// consumers of stage s poll that one word until it reaches the number of CTAs
// owning tiles of stages 0..s-1.  Every stage reads only what earlier stages
// wrote, so a CTA of stage s can add to the counter only after all of stages
// 0..s-1 have, and the count therefore means that every earlier stage is
// complete (which also covers residuals and the reuse of buffers).  The x
// words are then read once; they still carry a tag (fp16 value | tag of step
// and stage), which is checked.  The last CTA of the step resets the counter.  Stage parameters live in a device table; the
// consumers copy the next stage's entry into shared memory while they work on
// the current one.  Every wait is bounded; an expired wait is OR-ed over the
// consumers at the end of the stage and the CTA then stops, waits (bounded)
// for its copies in flight and leaves.
constexpr int kMaxSlots = 16;
constexpr uint32_t kStepBarBytes = 2 * kMaxSlots * 8 + kConsumerWarps * 8 * 4;
constexpr int kParamWords = (int)(sizeof(Params) / 16);
static_assert(sizeof(Params) % 16 == 0 && kParamWords <= kConsumerWarps * 32, "Params size");

struct StepParams {
    const Params* stages;  // device table [n]
    int n;
    int slots;             // ring slots
    uint32_t slot_bytes;   // bytes per slot
    uint32_t meta_off;     // offset in a slot of the stage parameters (then the norm weights)
    uint32_t ring_off;     // offset of the ring in shared memory
    uint32_t x_bytes;      // x region (largest K)
    const uint32_t* step_ctr;
    uint32_t* done_ctr;
    uint32_t* stage_ctr;   // CTA-stage completions in this step
    int* err;
};

// Bounded wait until the completion counter reaches `need` (acquire).
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t need, int* err) {
    unsigned long long t0 = 0;
    while (true) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= need) return true;
        if (t0 == 0) {
            t0 = q4d::globaltimer();
        } else if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
            atomicOr(err, q4d::kErrTimeout);
            return false;
        }
    }
}

// First tile of a stage that CTA c owns: tile t goes to CTA (tile_base + t) mod G.
__device__ __forceinline__ int first_tile(int tile_base, int G, int c) {
    const int r = tile_base % G;
    return c >= r ? c - r : c - r + G;
}

// Bytes of stage metadata that travel with a CTA's first tile of a stage: the
// stage's parameter block and, for a normalised x, its norm weights.
__device__ __forceinline__ uint32_t meta_bytes(const Params& p) {
    return (uint32_t)sizeof(Params) + ((p.norm && p.norm_w) ? (uint32_t)p.K * 2u : 0u);
}

template <int M>
__global__ void __launch_bounds__(kThreads, 1) q4_decode_persistent_kernel(const __grid_constant__ StepParams sp) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = sp.slots, G = gridDim.x, c = blockIdx.x;
    float4* xs = reinterpret_cast<float4*>(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sp.x_bytes);
    float* red = reinterpret_cast<float*>(bars + 2 * kMaxSlots);
    Params* prm = reinterpret_cast<Params*>(smem + sp.x_bytes + kStepBarBytes);
    int2* tt = reinterpret_cast<int2*>(smem + sp.x_bytes + kStepBarBytes + sizeof(Params));
    uint8_t* ring = smem + sp.ring_off;
    const uint32_t full0 = q4d::smem_addr(bars), empty0 = q4d::smem_addr(bars + kMaxSlots);

    __shared__ uint32_t step_sh;
    __shared__ int issued_sh, consumed_sh;
    __shared__ volatile int abort_sh;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            q4d::mbar_init(full0 + 8 * i, 32);
            q4d::mbar_init(empty0 + 8 * i, kConsumerWarps);
        }
        q4d::fence_mbar_init();
        step_sh = q4d::ld_relaxed(sp.step_ctr);
        issued_sh = 0;
        consumed_sh = 0x7fffffff;
        abort_sh = 0;
    }
    // (tile origin, tile count) of every stage, for the consumers
    for (int s = threadIdx.x; s < sp.n; s += blockDim.x)
        tt[s] = make_int2(sp.stages[s].tile_base, sp.stages[s].total_tiles);
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer warp
        const uint64_t pol = q4d::policy_evict_first();
        int i = 0;
        bool ok = true;
        for (int s = 0; s < sp.n && ok; ++s) {
            const Params& p = sp.stages[s];
            const int t0 = first_tile(p.tile_base, G, c);
            for (int t = t0; t < p.total_tiles; t += G, ++i) {
                const int st = i % S, k = i / S;
                if (k > 0) {
                    int w_ok = 1;
                    if (lane == 0) w_ok = (q4d::mbar_wait(empty0 + 8 * st, (k - 1) & 1, sp.err) && !abort_sh) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, w_ok, 0)) {
                        ok = false;
                        break;
                    }
                }
                int si, n0, nrows;
                find_tile(p, t, si, n0, nrows);
                uint8_t* stage = ring + (size_t)st * sp.slot_bytes;
                const uint32_t fb = full0 + 8 * st;
                const uint32_t expect = (p.glu ? 2u : 1u) * bulk_bytes(p, nrows) + (t == t0 ? meta_bytes(p) : 0u);
                if (lane == 0)
                    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(expect)
                                 : "memory");
                __syncwarp();
                issue_rows(p, p.seg[si], n0, nrows, 0, stage, fb, lane, pol);
                if (p.glu) issue_rows(p, p.seg[1], n0, nrows, p.TR, stage, fb, lane, pol);
                if (t == t0 && lane == 0) {
                    q4d::bulk_g2s(q4d::smem_addr(stage + sp.meta_off), &sp.stages[s], (uint32_t)sizeof(Params), fb);
                    if (p.norm && p.norm_w)
                        q4d::bulk_g2s(q4d::smem_addr(stage + sp.meta_off + sizeof(Params)), p.norm_w,
                                      (uint32_t)p.K * 2u, fb);
                }
                q4d::mbar_arrive(fb);
            }
        }
        if (lane == 0) issued_sh = i;
    } else {
        // ---------------------------------------------------------- consumers
        constexpr uint32_t kCT = kConsumerWarps * 32;
        const int tid = threadIdx.x;
        const uint32_t step = step_sh;
        int i = 0;
        bool bad = false;
        uint32_t done_before = 0;  // CTAs owning tiles of the stages before s
        for (int s = 0; s < sp.n; ++s) {
            const int2 st_ = tt[s];
            const int t0 = first_tile(st_.x, G, c), T = st_.y;
            if (t0 < T) {
                // The first tile's slot also holds the stage's parameters and
                // norm weights; they are read from there until the x barrier
                // (the slot is released only after that tile is consumed).
                const int sl = i % S;
                if (!q4d::mbar_wait(full0 + 8 * sl, (i / S) & 1, sp.err)) bad = true;
                const uint8_t* slot = ring + (size_t)sl * sp.slot_bytes;
                const Params& ps = *reinterpret_cast<const Params*>(slot + sp.meta_off);
                if (tid < kParamWords)
                    reinterpret_cast<uint4*>(prm)[tid] = reinterpret_cast<const uint4*>(&ps)[tid];
                const uint32_t xtag = tag_of(step, ps.x_stage, ps.n_stages);
                const uint16_t* gam =
                    (ps.norm && ps.norm_w) ? reinterpret_cast<const uint16_t*>(slot + sp.meta_off + sizeof(Params))
                                           : nullptr;
                if (s > 0) {
                    // every earlier stage complete (one poller, then the CTA)
                    bool w_bad = bad;
                    if (tid == 0 && !w_bad) w_bad = !wait_count(sp.stage_ctr, done_before, sp.err);
                    if (q4d::named_bar_or(2, kCT, w_bad)) bad = true;
                }
                if (!bad && !load_x<M, 4>(ps, xs, red, warp, lane, xtag, gam)) bad = true;
                q4d::named_bar(1, kCT);
                const Params& p = *prm;
                const uint32_t ytag = tag_of(step, p.stage, p.n_stages);
                const uint32_t rtag = tag_of(step, p.res_stage, p.n_stages);
                float scale[M];
                norm_scales<M>(p, red, scale);
                if (!bad) {
                    for (int t = t0; t < T; t += G, ++i) {
                        const int st = i % S, k = i / S;
                        if (!q4d::mbar_wait(full0 + 8 * st, k & 1, sp.err)) {
                            bad = true;
                            break;
                        }
                        if (!consume_tile<M, 4>(p, ring + (size_t)st * sp.slot_bytes, xs, scale, warp, lane, t, ytag,
                                             rtag))
                            bad = true;
                        __syncwarp();
                        if (lane == 0) q4d::mbar_arrive(empty0 + 8 * st);
                    }
                }
            }
            if (q4d::named_bar_or(1, kCT, bad)) {
                if (tid == 0) abort_sh = 1;
                break;
            }
            if (t0 < T && tid == 0) {
                // the consumers' stores of this stage precede the barrier above
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(sp.stage_ctr) : "memory");
            }
            done_before += (uint32_t)(T < G ? T : G);
        }
        if (lane == 0) atomicMin(&consumed_sh, i);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // After an abort, copies may still be landing in slots nobody will
        // read: wait for them (bounded) before the CTA's shared memory goes.
        for (int j = consumed_sh; j < issued_sh; ++j) q4d::mbar_wait(full0 + 8 * (j % S), (j / S) & 1, nullptr);
        // The last CTA to finish advances the step counter (every CTA read it
        // at its start).
        __threadfence();
        if (atomicAdd(sp.done_ctr, 1u) == gridDim.x - 1) {
            *sp.done_ctr = 0;
            *sp.stage_ctr = 0;
            atomicAdd(const_cast<uint32_t*>(sp.step_ctr), 1u);
        }
    }
}

// Failure-detection self-test: both bounded waits against conditions that
// never come true; each latches kErrTimeout into the error word and returns.
__device__ uint32_t g_never_written_tagged_word;  // stays 0: tag 0 is never a valid tag

__global__ void expired_wait_kernel(int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        uint32_t w;
        poll_tagged<1>(&g_never_written_tagged_word, 1u, &w, err);
        q4d::mbar_init(q4d::smem_addr(&bar), 1);
        q4d::fence_mbar_init();
        q4d::mbar_wait(q4d::smem_addr(&bar), 0, err);  // nothing arrives
    }
}

}  // namespace q4k

extern "C" q4_status q4_selftest_expired_wait(q4_stream_t stream) {
    q4i::clear_error();
    const q4i::DeviceInfo* dev = nullptr;
    q4_status st = q4i::current_device(&dev);
    if (st != Q4_OK) return st;
    q4k::expired_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev->err_word);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return q4i::cuda_fail(e, "self-test kernel launch");
    return Q4_OK;
}

namespace q4i {

using q4k::Params;

q4_status validate_gemv(const q4_gemv_desc& d) {
    if (d.M < 1 || d.M > 8) return fail(d.M < 1 ? Q4_ERR_INVALID_ARG : Q4_ERR_UNSUPPORTED, "M=%d outside 1..8", d.M);
    if (d.K < 64 || d.K % 64) return fail(Q4_ERR_INVALID_ARG, "K=%d is not a positive multiple of 64", d.K);
    if (d.K > (1 << 20)) return fail(Q4_ERR_UNSUPPORTED, "K=%d above 1048576", d.K);
    if (!d.x) return fail(Q4_ERR_INVALID_ARG, "x is NULL");
    const int ldx = d.ldx ? d.ldx : d.K;
    if (ldx < d.K) return fail(Q4_ERR_INVALID_ARG, "ldx=%d < K=%d", ldx, d.K);
    if (!aligned16(d.x) || ldx % 8) return fail(Q4_ERR_MISALIGNED, "x must be 16-byte aligned with ldx %% 8 == 0");
    if (d.n_segments < 1 || d.n_segments > Q4_MAX_SEGMENTS)
        return fail(Q4_ERR_INVALID_ARG, "n_segments=%d outside 1..%d", d.n_segments, Q4_MAX_SEGMENTS);
    if (d.out_dtype != Q4_F32 && d.out_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "bad out_dtype");
    if (d.mode != Q4_GEMV_PLAIN && d.mode != Q4_GEMV_GLU) return fail(Q4_ERR_INVALID_ARG, "bad mode");
    if (d.mode == Q4_GEMV_GLU) {
        if (d.n_segments != 2) return fail(Q4_ERR_INVALID_ARG, "GLU mode needs exactly 2 segments");
        if (d.seg[0].N != d.seg[1].N) return fail(Q4_ERR_INVALID_ARG, "GLU gate/up widths differ");
        if (d.out_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "GLU mode writes fp16");
        if (d.seg[0].residual || d.seg[1].residual) return fail(Q4_ERR_INVALID_ARG, "GLU mode takes no residual");
    }
    if (d.x_rmsnorm != 0 && d.x_rmsnorm != 1) return fail(Q4_ERR_INVALID_ARG, "x_rmsnorm must be 0 or 1");
    if (d.x_rmsnorm && !(d.norm_eps >= 0.f)) return fail(Q4_ERR_INVALID_ARG, "norm_eps must be >= 0");
    if (d.x_rmsnorm && d.norm_weight && !aligned16(d.norm_weight))
        return fail(Q4_ERR_MISALIGNED, "norm_weight must be 16-byte aligned");
    if (d.flags & ~Q4_GEMV_EARLY_WEIGHTS) return fail(Q4_ERR_INVALID_ARG, "unknown flags 0x%x", d.flags);
    for (int i = 0; i < d.n_segments; ++i) {
        const q4_segment& s = d.seg[i];
        if (!s.Wq || !s.scales || !s.biases) return fail(Q4_ERR_INVALID_ARG, "segment %d: NULL weights", i);
        if (s.N < 1) return fail(Q4_ERR_INVALID_ARG, "segment %d: N=%d", i, s.N);
        if (!(d.mode == Q4_GEMV_GLU && i == 1) && !s.y) return fail(Q4_ERR_INVALID_ARG, "segment %d: y is NULL", i);
        const int ldy = s.ldy ? s.ldy : s.N;
        if (ldy < s.N) return fail(Q4_ERR_INVALID_ARG, "segment %d: ldy < N", i);
        if (!aligned16(s.Wq) || !aligned16(s.scales) || !aligned16(s.biases))
            return fail(Q4_ERR_MISALIGNED, "segment %d: Wq/scales/biases must be 16-byte aligned", i);
        if (s.residual && d.out_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "segment %d: residual needs fp16 output", i);
    }
    return Q4_OK;
}

namespace {

int lane_words_rt(int M) { return M == 1 ? 4 : (M == 2 ? 2 : 1); }

uint32_t x_smem_bytes(int M, int K) {
    const int LW = lane_words_rt(M);
    const int chunk_words = 32 * LW;
    const int nchunks = (K / 8 + chunk_words - 1) / chunk_words;
    return (uint32_t)nchunks * (uint32_t)(LW * 2 * M) * 32u * 16u;
}

template <int M, int BITS>
cudaError_t launch_m(const Params& p, dim3 grid, size_t smem, cudaStream_t stream, bool pdl) {
    auto kern = q4k::q4_gemv_kernel<M, BITS>;
    static std::atomic<int> smem_marks[64];
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem_marks, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(q4k::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// Kernel parameters of one fused GEMV (everything but the shared-memory
// geometry).
void fill_params(const q4_gemv_desc& d, const GemvTagged* tg, bool early_prefetch, int min_tiles,
                 uint32_t max_stage, int* err, Params& p, int bits = 4) {
    p = {};
    p.bits = bits;
    const int K = d.K, G = K / 64;
    const bool glu = d.mode == Q4_GEMV_GLU;
    p.x = d.x;
    p.K = K;
    p.ldx = d.ldx ? d.ldx : K;
    p.nseg = d.n_segments;
    p.out_f16 = d.out_dtype == Q4_F16;
    p.glu = glu;
    p.early_prefetch = early_prefetch ? 1 : 0;
    p.norm = d.x_rmsnorm ? 1 : 0;
    p.norm_w = d.norm_weight;
    p.norm_eps = d.norm_eps;
    p.err = err;
    p.n_stages = 1;
    if (tg) {
        p.x_tag = tg->x;
        p.x_stage = tg->x_stage;
        p.res_stage = tg->res_stage;
        p.step_ctr = tg->step_ctr;
        p.done_ctr = tg->done_ctr;
        p.stage = tg->stage;
        p.n_stages = tg->n_stages;
        p.last = tg->last ? 1 : 0;
    }

    // Tile rows: largest of 64/32/16/8 (per matrix) whose tile count still
    // reaches min_tiles, with a stage of at most max_stage bytes.
    const uint32_t row_bytes = (uint32_t)(K * bits / 8 + G * 4);
    int TR = 64;
    while (TR > 8) {
        const uint32_t stage = (uint32_t)(glu ? 2 * TR : TR) * row_bytes;
        long tiles = 0;
        for (int i = 0; i < (glu ? 1 : d.n_segments); ++i) tiles += (d.seg[i].N + TR - 1) / TR;
        if (stage <= max_stage && tiles >= min_tiles) break;
        TR /= 2;
    }
    p.TR = TR;
    p.rows_per_tile = glu ? 2 * TR : TR;
    int tiles = 0;
    for (int i = 0; i < (glu ? 2 : d.n_segments); ++i) {
        const q4_segment& s = d.seg[i];
        q4k::Seg& g = p.seg[i];
        g.Wq = s.Wq;
        g.s = s.scales;
        g.b = s.biases;
        g.y = s.y;
        g.res = s.residual;
        g.y_tag = tg ? tg->y[i] : nullptr;
        g.res_tag = tg ? tg->res[i] : nullptr;
        g.N = s.N;
        g.ldy = s.ldy ? s.ldy : s.N;
        g.tile_begin = glu ? 0 : tiles;
        g.tiles = (s.N + TR - 1) / TR;
        if (!glu) tiles += g.tiles;
    }
    if (glu) tiles = p.seg[0].tiles;
    p.total_tiles = tiles;

    p.stage_bytes = ((uint32_t)p.rows_per_tile * row_bytes + 127u) & ~127u;
}

}  // namespace

bool gemv_fits_unsplit(int M, int K) {
    const DeviceInfo* dev = nullptr;
    if (current_device(&dev) != Q4_OK) return false;
    const uint32_t row_bytes = (uint32_t)(K / 2 + (K / 64) * 4);
    const uint32_t stage = ((uint32_t)(2 * 8) * row_bytes + 127u) & ~127u;  // smallest GLU tile
    const uint32_t fixed = ((x_smem_bytes(M, K) + 127u) & ~127u) + q4k::kBarBytes;
    return fixed + 2 * stage <= (uint32_t)dev->smem_optin - 256u;
}

q4_status launch_gemv(const q4_gemv_desc& d, cudaStream_t stream, bool pdl, bool early_prefetch,
                      const GemvTagged* tg, int bits) {
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    if (bits < 2 || bits > 8 || bits == 7) return fail(Q4_ERR_INVALID_ARG, "bits=%d", bits);
    if (bits != 4 && bits != 8 && d.M != 1) return fail(Q4_ERR_UNSUPPORTED, "%d-bit codes need M = 1", bits);

    Params p;
    fill_params(d, tg, early_prefetch, dev->sms, 48u * 1024u, dev->err_word, p, bits);
    const int M = d.M, K = d.K;
    p.x_bytes = (x_smem_bytes(M, K) + 127u) & ~127u;
    const uint32_t fixed = p.x_bytes + q4k::kBarBytes;
    // Two CTAs per SM when they fit (lets the next kernel's CTAs start
    // streaming their weights under programmatic dependent launch).
    const uint32_t budget_two = (uint32_t)dev->smem_per_sm / 2 - 1024u;
    uint32_t budget = budget_two;
    int ctas_per_sm = 2;
    if (fixed + 2 * p.stage_bytes > budget_two) {
        budget = (uint32_t)dev->smem_optin - 256u;  // the kernel's static shared variables
        ctas_per_sm = 1;
    }
    if (fixed + 2 * p.stage_bytes > budget) {
        // x for all M rows does not fit next to two weight stages: run the
        // rows of x in two halves (the weights are then streamed twice).
        if (M == 1) return fail(Q4_ERR_UNSUPPORTED, "K=%d needs more shared memory than the device has", K);
        if (tg) return fail(Q4_ERR_UNSUPPORTED, "M=%d, K=%d does not fit one launch of a decode stage", M, K);
        q4_gemv_desc lo = d, hi = d;
        lo.M = (M + 1) / 2;
        hi.M = M - lo.M;
        const int ldx = d.ldx ? d.ldx : K;
        hi.x = d.x + (size_t)lo.M * ldx;
        lo.ldx = hi.ldx = ldx;
        const size_t esz = d.out_dtype == Q4_F16 ? 2 : 4;
        for (int i = 0; i < d.n_segments; ++i) {
            const int ldy = d.seg[i].ldy ? d.seg[i].ldy : d.seg[i].N;
            lo.seg[i].ldy = hi.seg[i].ldy = ldy;
            if (d.seg[i].y) hi.seg[i].y = static_cast<uint8_t*>(d.seg[i].y) + (size_t)lo.M * ldy * esz;
            if (d.seg[i].residual) hi.seg[i].residual = d.seg[i].residual + (size_t)lo.M * ldy;
        }
        st = launch_gemv(lo, stream, pdl, early_prefetch, nullptr, bits);
        if (st != Q4_OK) return st;
        return launch_gemv(hi, stream, pdl, early_prefetch, nullptr, bits);
    }
    int S = (int)((budget - fixed) / p.stage_bytes);
    if (S > q4k::kMaxStages) S = q4k::kMaxStages;
    p.stages = S;
    const size_t smem = fixed + (size_t)S * p.stage_bytes;
    const int tiles = p.total_tiles;
    const int grid = tiles < dev->sms * ctas_per_sm ? tiles : dev->sms * ctas_per_sm;

    cudaError_t e = cudaSuccess;
#define Q4_LAUNCH_M(MM)                                                                          \
    case MM:                                                                                     \
        e = bits == 4 ? launch_m<MM, 4>(p, dim3(grid), smem, stream, pdl)                        \
                      : launch_m<MM, 8>(p, dim3(grid), smem, stream, pdl);                       \
        break;
    if (bits != 4 && bits != 8) {
        switch (bits) {
            case 2: e = launch_m<1, 2>(p, dim3(grid), smem, stream, pdl); break;
            case 3: e = launch_m<1, 3>(p, dim3(grid), smem, stream, pdl); break;
            case 5: e = launch_m<1, 5>(p, dim3(grid), smem, stream, pdl); break;
            default: e = launch_m<1, 6>(p, dim3(grid), smem, stream, pdl); break;
        }
        if (e != cudaSuccess) return cuda_fail(e, "q4_gemv kernel launch");
        return Q4_OK;
    }
    switch (M) {
        Q4_LAUNCH_M(1)
        Q4_LAUNCH_M(2)
        Q4_LAUNCH_M(3)
        Q4_LAUNCH_M(4)
        Q4_LAUNCH_M(5)
        Q4_LAUNCH_M(6)
        Q4_LAUNCH_M(7)
        Q4_LAUNCH_M(8)
    }
#undef Q4_LAUNCH_M
    if (e != cudaSuccess) return cuda_fail(e, "q4_gemv kernel launch");
    return Q4_OK;
}


size_t gemv_params_bytes() { return sizeof(Params); }

q4_status persistent_plan(const q4_gemv_desc* d, const GemvTagged* tg, int n, void* host_params,
                          PersistentGeom* g, bool* fits) {
    *fits = false;
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    if (n < 1) return fail(Q4_ERR_INVALID_ARG, "no stages");
    const int M = d[0].M;
    Params* P = static_cast<Params*>(host_params);
    uint32_t tile_max = 0, gamma_max = 0, xb = 0;
    int base = 0;
    for (int s = 0; s < n; ++s) {
        if (d[s].M != M) return Q4_OK;
        // Tiles of at most 24 KB, and at least one per SM where the matrix allows.
        fill_params(d[s], &tg[s], true, dev->sms, 24u * 1024u, dev->err_word, P[s]);
        P[s].tile_base = base;
        base += P[s].total_tiles;
        if (P[s].stage_bytes > tile_max) tile_max = P[s].stage_bytes;
        if (P[s].norm && P[s].norm_w && (uint32_t)d[s].K * 2u > gamma_max) gamma_max = (uint32_t)d[s].K * 2u;
        const uint32_t x = (x_smem_bytes(M, d[s].K) + 127u) & ~127u;
        if (x > xb) xb = x;
    }
    // A slot: tile data, then (first tile of a stage only) the parameter block
    // and the norm weights at a fixed offset.
    const uint32_t slot = (tile_max + (uint32_t)sizeof(Params) + gamma_max + 127u) & ~127u;
    const size_t fixed =
        ((size_t)xb + q4k::kStepBarBytes + sizeof(Params) + (((size_t)n * 8 + 15) & ~(size_t)15) + 127) & ~(size_t)127;
    const size_t avail = (size_t)dev->smem_optin - 256;  // the kernel's static shared variables
    if (fixed + 2 * (size_t)slot > avail) return Q4_OK;  // does not fit: the caller plans launches
    int slots = (int)((avail - fixed) / slot);
    if (slots > q4k::kMaxSlots) slots = q4k::kMaxSlots;
    for (int s = 0; s < n; ++s) {
        P[s].x_bytes = xb;
        P[s].stages = slots;
    }
    g->M = M;
    g->n = n;
    g->grid = dev->sms;
    g->slots = slots;
    g->slot_bytes = slot;
    g->meta_off = slot - (uint32_t)sizeof(Params) - gamma_max;
    g->ring_off = (uint32_t)fixed;
    g->x_bytes = xb;
    g->smem = fixed + (size_t)slots * slot;
    g->step_ctr = tg[0].step_ctr;
    g->done_ctr = tg[0].done_ctr;
    *fits = true;
    return Q4_OK;
}

namespace {
template <int M>
cudaError_t launch_persistent_m(const q4k::StepParams& sp, const PersistentGeom& g, cudaStream_t stream) {
    auto kern = q4k::q4_decode_persistent_kernel<M>;
    static std::atomic<int> smem_marks[64];
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), smem_marks, (int)g.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.grid);
    cfg.blockDim = dim3(q4k::kThreads);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    // cooperative: the launch fails unless every CTA can be resident at once,
    // which the waits between CTAs rely on
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sp);
}
}  // namespace

q4_status persistent_launch(const PersistentGeom& g, const void* dev_params, cudaStream_t stream) {
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    q4k::StepParams sp = {};
    sp.stages = static_cast<const Params*>(dev_params);
    sp.n = g.n;
    sp.slots = g.slots;
    sp.slot_bytes = g.slot_bytes;
    sp.meta_off = g.meta_off;
    sp.ring_off = g.ring_off;
    sp.x_bytes = g.x_bytes;
    sp.step_ctr = g.step_ctr;
    sp.done_ctr = g.done_ctr;
    sp.stage_ctr = g.done_ctr + 1;
    sp.err = dev->err_word;
    cudaError_t e = cudaSuccess;
    switch (g.M) {
        case 1: e = launch_persistent_m<1>(sp, g, stream); break;
        case 2: e = launch_persistent_m<2>(sp, g, stream); break;
        case 3: e = launch_persistent_m<3>(sp, g, stream); break;
        case 4: e = launch_persistent_m<4>(sp, g, stream); break;
        case 5: e = launch_persistent_m<5>(sp, g, stream); break;
        case 6: e = launch_persistent_m<6>(sp, g, stream); break;
        case 7: e = launch_persistent_m<7>(sp, g, stream); break;
        case 8: e = launch_persistent_m<8>(sp, g, stream); break;
        default: return fail(Q4_ERR_UNSUPPORTED, "M=%d", g.M);
    }
    if (e != cudaSuccess) return cuda_fail(e, "persistent decode kernel launch");
    return Q4_OK;
}

}  // namespace q4i
