// The layer stack of a decode step (M = 1) as ONE persistent launch of
// thread-block clusters, with two grid-wide hand-offs per layer instead of
// four dependent kernel launches (BaseRT: optimal LLM inference on Apple
// Silicon with native Metal, §3 "BaseRT runtime design": a decode loop that
// amortises dispatch and synchronisation; §3.3 "Kernel fusion and
// specialisation": fused operator sequences in the attention block and FFN).
//
// Dataflow of a layer (the pre-norm layer of the decode stream):
//   q = fp16(Wq n(h)),  k, v likewise,  h' = fp16(h + Wo q),
//   act = fp16(SiLU(Wg n(h')) * (Wu n(h'))),  h = fp16(h' + Wd act).
// A GEMV whose input is produced by the GEMV before it needs all of that
// input; but the o and down products can be split along K instead of N:
//   * cluster c owns a block of q rows (whole 64-row groups) and the matching
//     column block of Wo; its CTAs compute their share of those q rows,
//     broadcast them to every CTA of the cluster through distributed shared
//     memory (st.async onto each peer's mbarrier), and then CTA i of the
//     cluster multiplies its 64 (hidden / cluster size) rows of the column
//     block: a partial h' over the cluster's columns;
//   * the partials of all clusters meet in global memory as 64-bit words
//     (fp32 value | 32-bit tag naming the step and the exchange), so a reader
//     polls the data itself; CTA i of every cluster sums block i over the
//     clusters in a fixed order (every cluster computes identical bits),
//     rounds h' = fp16(h + sum) and broadcasts its block to its cluster;
//   * the FFN half does the same with act and Wd.
// So a layer costs two global hand-offs and two in-cluster ones, and every
// CTA holds the whole h (or h') in shared memory at each layer boundary,
// where it also computes the RMS norm itself.  lm_head follows as its own
// launch (the ordinary fused-dequant GEMV over all SMs).
//
// Weights never depend on activations, so one producer warp per CTA streams
// the CTA's pieces of every layer through a ring of shared-memory slots as
// far ahead as the ring allows: whole rows by 1-D bulk copies, the o / down
// column blocks by 2-D tensor-map copies.  The dot products are the
// CUDA-core fused dequantisation of the GEMV kernel (one fp16 x fp16 -> fp32
// FMA per weight, packed fp32 multiply-accumulate).
//
// Every wait is bounded (2 s); an expired wait latches an error bit, and the
// CTA stops working but still meets its cluster at the final barrier, waits
// for its copies in flight and leaves.
#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4s {

// Per-phase timestamps (%globaltimer) of the first and the last CTA, for the
// step-latency breakdown; compiled in only with -DQ4_STEP_TRACE (a separate
// diagnostic build, bit_quantized_gemv_q4_gb300/trace_step.py).
#ifdef Q4_STEP_TRACE
__device__ unsigned long long g_step_trace[2 * 4096];
#define Q4_TRACE_T(k, t)                                                                             \
    do {                                                                                             \
        if (tid == (t) && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1) && l < 128)                \
            g_step_trace[(blockIdx.x ? 4096 : 0) + l * 32 + (k)] = q4d::globaltimer();                \
    } while (0)
#else
#define Q4_TRACE_T(k, t) \
    do {                 \
    } while (0)
#endif
#define Q4_TRACE(k) Q4_TRACE_T(k, 0)  // the consumers' points (0..14)

constexpr int kWarps = 11;                       // consumer warps (the layer's critical path)
constexpr int kCT = kWarps * 32;                 // consumer threads
constexpr int kProducerWarp = kWarps;            // streams the weight pieces
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kKvThreads = 256;                  // the k / v kernel's CTA
constexpr int kMaxSlots = 16;
constexpr int kItems = 4;                        // ring pieces per layer and CTA: q, o, gate/up, down

struct Lin {
    const uint32_t* Wq;
    const uint16_t* s;
    const uint16_t* b;
};

struct LayerDesc {
    Lin q, k, v, gate, up;
    const uint16_t* attn_norm;  // nullptr: ones
    const uint16_t* ffn_norm;
};

struct Params {
    const LayerDesc* layers;   // device [L]
    const CUtensorMap* maps;   // device [L][6]: o codes, o scales, o biases, down codes, scales, biases
    const uint16_t* x;         // fp16 [H], input of layer 0
    uint16_t *h, *h_mid, *q, *k, *v, *act;  // fp16 outputs (the last layer's values remain)
    uint32_t* htag;            // [L][H]: every layer's input h, tagged (fp16 | tag << 16), for the k / v kernel
    unsigned long long* xch;   // [2L][C][H]: (tag << 32) | fp32 partial
    uint32_t* ctr;             // [0] step counter, [1] CTAs finished
    int* err;
    int L, H, QN, KVN, F, C, S;
    float eps;
    int ro;                    // output rows per CTA in the o / down partials (H / S)
    int qspan, fspan;          // column-block widths in groups (largest cluster share)
    int qspan_s, fspan_s;      // scale / bias box widths in groups (multiples of 8)
    int slots;
    uint32_t slot_bytes;
    // shared memory: x of the two halves (fp32, lane-interleaved), the
    // cluster's block sums of squares of both halves ([2][S]), this CTA's
    // octet sums of squares (layer 0's input: all of them), this CTA's h
    // block and norm weights, row totals, q / act blocks, partials (ro, then
    // span x ro per group), barriers, the ring
    uint32_t off_xs, xs_bytes, off_bsum, off_nss, off_hown, off_gown, off_rows, off_qx, off_ax, off_red, off_bar,
        off_ring;
};

// The k / v kernel: the k and v rows of every layer on the SMs the clusters
// leave free.  It reads each layer's input h from the clustered kernel's
// tagged copy and normalises it in that kernel's order, so its k and v are
// the bits the clustered kernel would compute.
struct KvParams {
    const LayerDesc* layers;             // device [L]
    const uint16_t* x;                   // fp16 [H], input of layer 0
    uint16_t *k, *v;                     // fp16 outputs (the last layer's values remain)
    const uint32_t* htag;                // the clustered kernel's tagged layer inputs [L][H]
    uint32_t* ctr;                       // [0] clustered steps done, [3] k / v steps done, [4] k / v CTAs done
    int* err;
    int L, H, KVN, S, ro;
    float eps;
    uint32_t slot_bytes, xs_bytes;
    // shared memory: h (fp16), x (fp32, lane-interleaved), octet sums of
    // squares, row totals, barriers, a ring of two slots
    uint32_t off_h, off_xs, off_nss, off_rows, off_bar, off_ring;
};

// [a, b) = part i of n split into `parts` nearly equal pieces.
__host__ __device__ inline void split(int n, int parts, int i, int& a, int& b) {
    a = (int)((long long)n * i / parts);
    b = (int)((long long)n * (i + 1) / parts);
}

__host__ __device__ inline uint32_t align128(uint32_t v) { return (v + 127u) & ~127u; }

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Store into a peer CTA's shared memory; the byte count completes on the
// peer's mbarrier (both addresses are shared::cluster addresses).
__device__ __forceinline__ void st_async_b32(uint32_t raddr, uint32_t v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr), "r"(v),
                 "r"(rbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v4(uint32_t raddr, uint4 v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     raddr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rbar)
                 : "memory");
}
// Wait on a barrier that peers complete (acquire at cluster scope).  The
// clock is read every 16th attempt only (a read costs about as much as the
// attempt), which bounds the wait all the same.
__device__ __forceinline__ bool wait_cluster_bar(uint32_t bar, uint32_t parity, int* err) {
    unsigned long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
            "selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (it & 15u) continue;
        if (t0 == 0) {
            t0 = q4d::globaltimer();
        } else if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
            atomicOr(err, q4d::kErrTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 64-bit exchange words: single-copy atomic, coherent at L2.
__device__ __forceinline__ void st_xch(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_xch(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// ---------------------------------------------------------------- work split
struct Work {
    int qg0, qg1;   // the cluster's q groups
    int qa, qb;     // this CTA's q rows
    int k0, k1, v0, v1;  // this CTA's k and v rows
    int fg0, fg1;   // the cluster's ffn groups
    int fa, fb;     // this CTA's act rows
};

__host__ __device__ inline Work work_of(int QN, int KVN, int F, int C, int S, int c, int i) {
    Work w;
    split(QN / 64, C, c, w.qg0, w.qg1);
    split(64 * (w.qg1 - w.qg0), S, i, w.qa, w.qb);
    w.qa += 64 * w.qg0;
    w.qb += 64 * w.qg0;
    int a, b;
    split(2 * KVN, C * S, c * S + i, a, b);
    w.k0 = a < KVN ? a : KVN;
    w.k1 = b < KVN ? b : KVN;
    w.v0 = (a > KVN ? a : KVN) - KVN;
    w.v1 = (b > KVN ? b : KVN) - KVN;
    split(F / 64, C, c, w.fg0, w.fg1);
    split(64 * (w.fg1 - w.fg0), S, i, w.fa, w.fb);
    w.fa += 64 * w.fg0;
    w.fb += 64 * w.fg0;
    return w;
}

// Byte layout of a row item in a slot: two row blocks (codes, scales,
// biases); `gam` marks the end.
struct RowItem {
    uint32_t cA, cB, sA, bA, sB, bB, gam;
};
__host__ __device__ inline RowItem row_item(int H, int nA, int nB) {
    const uint32_t rc = (uint32_t)H / 2, rs = (uint32_t)H / 32;  // code / scale bytes per row
    RowItem r;
    r.cA = 0;
    r.cB = align128((uint32_t)nA * rc);
    r.sA = align128(r.cB + (uint32_t)nB * rc);
    r.bA = r.sA + (uint32_t)nA * rs;
    r.sB = r.bA + (uint32_t)nA * rs;
    r.bB = r.sB + (uint32_t)nB * rs;
    r.gam = align128(r.bB + (uint32_t)nB * rs);
    return r;
}
// Layout of a column-block item: codes [ro][span * 8 words], scales and
// biases [ro][span_s].
struct ColItem {
    uint32_t s, b, end;
};
__host__ __device__ inline ColItem col_item(int ro, int span, int span_s) {
    ColItem c;
    c.s = align128((uint32_t)ro * (uint32_t)span * 32u);
    c.b = c.s + align128((uint32_t)ro * (uint32_t)span_s * 2u);
    c.end = c.b + align128((uint32_t)ro * (uint32_t)span_s * 2u);
    return c;
}

// ---------------------------------------------------------------- producer
__device__ __forceinline__ void issue_rows(const Lin& m, int r0, int n, int H, uint8_t* dst_c, uint8_t* dst_s,
                                           uint8_t* dst_b, uint32_t bar, uint64_t pol) {
    if (n <= 0) return;
    const uint32_t rc = (uint32_t)H / 2, rs = (uint32_t)H / 32;
    q4d::bulk_g2s_evict_first(q4d::smem_addr(dst_c), reinterpret_cast<const uint8_t*>(m.Wq) + (size_t)r0 * rc,
                              (uint32_t)n * rc, bar, pol);
    q4d::bulk_g2s(q4d::smem_addr(dst_s), reinterpret_cast<const uint8_t*>(m.s) + (size_t)r0 * rs, (uint32_t)n * rs, bar);
    q4d::bulk_g2s(q4d::smem_addr(dst_b), reinterpret_cast<const uint8_t*>(m.b) + (size_t)r0 * rs, (uint32_t)n * rs, bar);
}

// Bytes item `it` brings into a slot, and the copies (lane 0 only).
__device__ uint32_t issue_item(const Params& p, const LayerDesc& L, const CUtensorMap* maps, const Work& w, int it,
                               int i, uint8_t* slot, uint32_t bar, bool do_issue, uint64_t pol) {
    const int H = p.H;
    const uint32_t rc = (uint32_t)H / 2, rs = (uint32_t)H / 32;
    if (it == 0 || it == 2 || it == 3) {
        // row items: q rows (0), k and v rows (2), gate and up rows (3)
        const Lin& A = it == 0 ? L.q : it == 2 ? L.k : L.gate;
        const int a0 = it == 0 ? w.qa : it == 2 ? w.k0 : w.fa;
        const int nA = it == 0 ? w.qb - w.qa : it == 2 ? w.k1 - w.k0 : w.fb - w.fa;
        const int nB = it == 0 ? 0 : it == 2 ? w.v1 - w.v0 : w.fb - w.fa;
        const int b0 = it == 2 ? w.v0 : w.fa;
        const RowItem r = row_item(H, nA, nB);
        if (do_issue) {
            issue_rows(A, a0, nA, H, slot + r.cA, slot + r.sA, slot + r.bA, bar, pol);
            if (it != 0) issue_rows(it == 2 ? L.v : L.up, b0, nB, H, slot + r.cB, slot + r.sB, slot + r.bB, bar, pol);
        }
        return (uint32_t)(nA + nB) * (rc + 2 * rs);
    }
    // column blocks: o (item 1) and down (item 4)
    const bool o = it == 1;
    const int span = o ? p.qspan : p.fspan, span_s = o ? p.qspan_s : p.fspan_s;
    const int g0 = o ? w.qg0 : w.fg0;
    const ColItem c = col_item(p.ro, span, span_s);
    const CUtensorMap* m = maps + (o ? 0 : 3);
    if (do_issue) {
        const uint32_t d = q4d::smem_addr(slot);
        tma_load_2d(d, m, g0 * 8, i * p.ro, bar);
        tma_load_2d(d + c.s, m + 1, g0 & ~7, i * p.ro, bar);
        tma_load_2d(d + c.b, m + 2, g0 & ~7, i * p.ro, bar);
    }
    return (uint32_t)p.ro * ((uint32_t)span * 32u + 2u * (uint32_t)span_s * 2u);
}

// ---------------------------------------------------------------- consumers
// x layout of dot_rows (fp32): octet j (8 inputs) sits in two float4 slots,
// (x0, x4, x1, x5) and (x2, x6, x3, x7), of lane l = (j % 128) / 4, word
// wi = j % 4 of chunk c = j / 128: slot (c * 8 + 2 wi + half) * 32 + l, so a
// lane's 16-byte loads over its 4 words are conflict-free across the warp.
__device__ __forceinline__ uint32_t xs_slot(int j) {
    const int c = j >> 7, l = (j & 127) >> 2, wi = j & 3;
    return (uint32_t)((c * 8 + wi * 2) * 32 + l);
}

// 1/rms from the per-octet sums of squares of the vector (nss[H/8]), the
// same bits in every warp and every CTA (fixed order, then an xor tree).
__device__ __forceinline__ float rms_inv(const float* nss, int H, float eps, int lane) {
    float t = 0.f;
    for (int j = lane; j < H / 8; j += 32) t += nss[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return rsqrtf(t / (float)H + eps);
}

// Dequantise one word and accumulate against 8 inputs in natural order
// (A = x0..x3, B = x4..x7): the nibble pairs (0,4) (1,5) (2,6) (3,7) meet
// (A.x, B.x) ... (A.w, B.w); one accumulator per pair.
__device__ __forceinline__ void word_mac_nat(uint32_t q, uint16_t sh, float c1024, float c64, const float4& A,
                                             const float4& B, float2* acc) {
    const uint32_t q8 = q >> 8;
    const uint32_t v0 = q4d::and_or(q, 0x000F000Fu, 0x64006400u);
    const uint32_t v1 = q4d::and_or(q, 0x00F000F0u, 0x54005400u);
    const uint32_t v2 = q4d::and_or(q8, 0x000F000Fu, 0x64006400u);
    const uint32_t v3 = q4d::and_or(q8, 0x00F000F0u, 0x54005400u);
    acc[0] = __ffma2_rn(q4d::fma_h2_s_f32(v0, sh, c1024), make_float2(A.x, B.x), acc[0]);
    acc[1] = __ffma2_rn(q4d::fma_h2_s_f32(v1, sh, c64), make_float2(A.y, B.y), acc[1]);
    acc[2] = __ffma2_rn(q4d::fma_h2_s_f32(v2, sh, c1024), make_float2(A.z, B.z), acc[2]);
    acc[3] = __ffma2_rn(q4d::fma_h2_s_f32(v3, sh, c64), make_float2(A.w, B.w), acc[3]);
}

// Dot products of the rows of a row item (block A rows, then block B rows)
// with x (K = H), by NW warps.  In each pass warp w takes rows w, w + NW, ...,
// w + 7 NW of the next 8 NW (those that exist); a lane covers 4 words (32
// inputs) of each 128-word chunk, x is loaded once per chunk for all the
// warp's rows, and the rows' totals are reduced together by a transposing
// butterfly.  Totals go to out[row].
template <int NW>
__device__ __forceinline__ void dot_rows(const uint8_t* slot, RowItem ri, int nA, int nB, int H, const float4* xs,
                                         int warp, int lane, float* out) {
    constexpr int RB = 8;
    const int W8 = H / 8, G = H / 64, n = nA + nB;
    const int nchunks = (W8 + 127) / 128;
    for (int base = 0; base < n; base += RB * NW) {
        int nr = (n - base - warp + NW - 1) / NW;  // rows of this warp in the pass
        nr = nr < 0 ? 0 : (nr > RB ? RB : nr);
        if (nr == 0) continue;
        float2 acc[RB];
#pragma unroll
        for (int k = 0; k < RB; ++k) acc[k] = make_float2(0.f, 0.f);
        for (int c = 0; c < nchunks; ++c) {
            const int j0 = c * 128 + lane * 4;
            if (j0 >= W8) continue;
            float4 xr[8];
            const float4* xc = xs + (size_t)c * 8 * 32 + lane;
#pragma unroll
            for (int e = 0; e < 8; ++e) xr[e] = xc[e * 32];
            const int g = j0 >> 3;
#pragma unroll
            for (int k = 0; k < RB; ++k) {
                if (k < nr) {
                    const int r = base + warp + k * NW;
                    const bool b = r >= nA;
                    const int q = b ? r - nA : r;
                    const uint4 v = *reinterpret_cast<const uint4*>(
                        reinterpret_cast<const uint32_t*>(slot + (b ? ri.cB : ri.cA)) + (size_t)q * W8 + j0);
                    const uint16_t sh = reinterpret_cast<const uint16_t*>(slot + (b ? ri.sB : ri.sA))[(size_t)q * G + g];
                    const uint16_t bh = reinterpret_cast<const uint16_t*>(slot + (b ? ri.bB : ri.bA))[(size_t)q * G + g];
                    const float sf = __half2float(__ushort_as_half(sh)), bf = __half2float(__ushort_as_half(bh));
                    const float ca = fmaf(-1024.f, sf, bf), cb = fmaf(-64.f, sf, bf);
                    q4d::word_mac<1>(v.x, sh, ca, cb, &xr[0], &xr[1], &acc[k]);
                    q4d::word_mac<1>(v.y, sh, ca, cb, &xr[2], &xr[3], &acc[k]);
                    q4d::word_mac<1>(v.z, sh, ca, cb, &xr[4], &xr[5], &acc[k]);
                    q4d::word_mac<1>(v.w, sh, ca, cb, &xr[6], &xr[7], &acc[k]);
                }
            }
        }
        // transposing butterfly over the 8 totals: after three rounds lanes
        // 4k .. 4k+3 hold row k's partials, two more rounds finish them
        float v[RB];
#pragma unroll
        for (int k = 0; k < RB; ++k) v[k] = acc[k].x + acc[k].y;
        int m = RB;
#pragma unroll
        for (int rnd = 0; rnd < 3; ++rnd) {
            const int o = 16 >> rnd;
            const bool upper = (lane & o) != 0;
            const int half = m >> 1;
#pragma unroll
            for (int k = 0; k < RB / 2; ++k) {
                if (k < half) {
                    const float send = upper ? v[k] : v[k + half];
                    const float keep = upper ? v[k + half] : v[k];
                    v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            m = half;
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        const int k = lane >> 2;
        if ((lane & 3) == 0 && k < nr) out[base + warp + k * NW] = v[0];
    }
}

// The o / down column-block product of this CTA: partial[rr] = sum over the
// cluster's columns of W[row oa + rr][col] * x[col], x (fp32, natural order)
// being the cluster's q or act block.  Work unit = (group g, row rr): one
// thread, 8 words, the group's 64 inputs read as a broadcast by the warp
// (consecutive lanes take consecutive rows of one group).  The units' sums
// meet in pg[g][rr] and are added over g in order.  Every consumer thread
// calls this (it holds a barrier); slot == nullptr (after a failed wait)
// skips the arithmetic.
__device__ __forceinline__ void col_partial(const uint8_t* slot, ColItem ci, int span, int span_s, int g0,
                                         const float* xb, int ro, float* pg, float* part) {
    const int tid = threadIdx.x;
    const float4* x4 = reinterpret_cast<const float4*>(xb);
    for (int u = tid; slot && u < span * ro; u += kCT) {
        const int g = u / ro, rr = u - g * ro;
        const uint4* cw = reinterpret_cast<const uint4*>(slot + (size_t)rr * span * 32 + (size_t)g * 32);
        const uint4 va = cw[0], vb = cw[1];
        const size_t si = (size_t)rr * span_s + (g0 & 7) + g;
        const uint16_t sh = reinterpret_cast<const uint16_t*>(slot + ci.s)[si];
        const float sf = __half2float(__ushort_as_half(sh));
        const float bf = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(slot + ci.b)[si]));
        const float ca = fmaf(-1024.f, sf, bf), cb = fmaf(-64.f, sf, bf);
        const float4* xg = x4 + 16 * g;
        float2 a[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) a[k] = make_float2(0.f, 0.f);
        word_mac_nat(va.x, sh, ca, cb, xg[0], xg[1], a);
        word_mac_nat(va.y, sh, ca, cb, xg[2], xg[3], a);
        word_mac_nat(va.z, sh, ca, cb, xg[4], xg[5], a);
        word_mac_nat(va.w, sh, ca, cb, xg[6], xg[7], a);
        word_mac_nat(vb.x, sh, ca, cb, xg[8], xg[9], a);
        word_mac_nat(vb.y, sh, ca, cb, xg[10], xg[11], a);
        word_mac_nat(vb.z, sh, ca, cb, xg[12], xg[13], a);
        word_mac_nat(vb.w, sh, ca, cb, xg[14], xg[15], a);
        pg[u] = ((a[0].x + a[0].y) + (a[1].x + a[1].y)) + ((a[2].x + a[2].y) + (a[3].x + a[3].y));
    }
    q4d::named_bar(1, kCT);
    for (int rr = tid; rr < ro; rr += kCT) {
        float t = 0.f;
        for (int g = 0; g < span; ++g) t += pg[g * ro + rr];
        part[rr] = t;
    }
}

// Publish this CTA's partials of rows oa .. oa + ro - 1 (thread r holds part[r]).
__device__ __forceinline__ void publish(unsigned long long* X, const float* part, int c, int H, int oa, int ro,
                                       uint32_t tag) {
    for (int r = threadIdx.x; r < ro; r += kCT)
        st_xch(X + (size_t)c * H + oa + r, ((unsigned long long)tag << 32) | __float_as_uint(part[r]));
}

// Collect every cluster's partials of this CTA's rows, add them in a fixed
// order to the residual (this CTA's block of h, hown), round to fp16 -- the
// new block, kept in hown and written to `out` (and tagged to `htag`) from
// cluster 0 -- and, when a next phase exists (gnext != nullptr), send every
// CTA of the cluster that phase's input for these rows: x = h * norm weight
// in the dot_rows layout (xs_next), and this block's sum of squares (octets
// in order, each octet's squares in order) into bsum_next[rank].  Warp w
// takes row octets w, w + 8, ...; in an octet, lane = 8 rs + cc polls cluster
// cc (cc + 8, ... when there are more than 8 clusters) of rows rs and rs + 4,
// the 8 lanes of each row add by an xor tree.  Every consumer thread calls
// this (it holds a barrier when gnext is set); `skip` (after a failed wait)
// leaves out the polls, the writes and the sends.  Returns false when a poll
// expired.
__device__ __forceinline__ bool collect(const unsigned long long* X, uint16_t* hown, const uint16_t* gnext,
                                        float4* xs_next, float* bsum_next, float* octss, uint16_t* out,
                                        uint32_t* htag, uint32_t htag_tag, int C, int H, int S, int oa, int ro,
                                        int rank, uint32_t tag, uint32_t hbar, int* err, bool skip) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cc = lane & 7, rs = lane >> 3;
    bool ok = true;
    for (int oc = warp; !skip && oc < ro / 8; oc += kWarps) {
        const int rA = 8 * oc + rs, rB = rA + 4;
        float vA = 0.f, vB = 0.f;
        for (int k = cc; k < C; k += 8) {
            const unsigned long long* pa = X + (size_t)k * H + oa + rA;
            const unsigned long long* pb = pa + 4;
            unsigned long long a = ld_xch(pa), b = ld_xch(pb);
            unsigned long long t0 = 0;
            for (uint32_t it = 1; ok && ((uint32_t)(a >> 32) != tag || (uint32_t)(b >> 32) != tag); ++it) {
                if ((it & 15u) == 0) {  // the clock every 16th poll (a read costs about a poll)
                    if (t0 == 0) {
                        t0 = q4d::globaltimer();
                    } else if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
                        atomicOr(err, q4d::kErrTimeout);
                        ok = false;
                    }
                }
                a = ld_xch(pa);
                b = ld_xch(pb);
            }
            vA += __uint_as_float((uint32_t)a);
            vB += __uint_as_float((uint32_t)b);
        }
        vA += __shfl_xor_sync(0xffffffffu, vA, 1);
        vB += __shfl_xor_sync(0xffffffffu, vB, 1);
        vA += __shfl_xor_sync(0xffffffffu, vA, 2);
        vB += __shfl_xor_sync(0xffffffffu, vB, 2);
        vA += __shfl_xor_sync(0xffffffffu, vA, 4);
        vB += __shfl_xor_sync(0xffffffffu, vB, 4);
        const __half hA = __float2half_rn(vA + __half2float(__ushort_as_half(hown[rA])));
        const __half hB = __float2half_rn(vB + __half2float(__ushort_as_half(hown[rB])));
        __syncwarp();
        if (cc == 0) {
            hown[rA] = __half_as_ushort(hA);
            hown[rB] = __half_as_ushort(hB);
            if (out) {
                out[oa + rA] = __half_as_ushort(hA);
                out[oa + rB] = __half_as_ushort(hB);
            }
            if (htag) {
                q4d::st_relaxed(htag + oa + rA, (htag_tag << 16) | __half_as_ushort(hA));
                q4d::st_relaxed(htag + oa + rB, (htag_tag << 16) | __half_as_ushort(hB));
            }
        }
        if (gnext) {
            // the octet's 8 values on every lane: rows 0..3 from lanes 0, 8, 16,
            // 24 (hA), rows 4..7 likewise (hB)
            float f[8];
            const float fA = __half2float(hA), fB = __half2float(hB);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[e] = __shfl_sync(0xffffffffu, fA, 8 * e);
                f[4 + e] = __shfl_sync(0xffffffffu, fB, 8 * e);
            }
            if (lane == 0) {
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                octss[oc] = ss;
            }
            if (lane < S) {
                float gm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) gm[e] = __half2float(__ushort_as_half(gnext[8 * oc + e]));
                const int j = (oa >> 3) + oc;
                const uint32_t xs0 = q4d::smem_addr(xs_next + xs_slot(j));
                const uint32_t rb = peer_addr(hbar, (uint32_t)lane);
                const float4 p0 = make_float4(f[0] * gm[0], f[4] * gm[4], f[1] * gm[1], f[5] * gm[5]);
                const float4 p1 = make_float4(f[2] * gm[2], f[6] * gm[6], f[3] * gm[3], f[7] * gm[7]);
                st_async_v4(peer_addr(xs0, (uint32_t)lane),
                            make_uint4(__float_as_uint(p0.x), __float_as_uint(p0.y), __float_as_uint(p0.z),
                                       __float_as_uint(p0.w)),
                            rb);
                st_async_v4(peer_addr(xs0 + 32 * 16, (uint32_t)lane),
                            make_uint4(__float_as_uint(p1.x), __float_as_uint(p1.y), __float_as_uint(p1.z),
                                       __float_as_uint(p1.w)),
                            rb);
            }
        }
    }
    if (gnext) {
        // the block's sum of squares, to every CTA of the cluster
        q4d::named_bar(1, kCT);
        if (!skip && warp == 0 && lane < S) {
            float t = 0.f;
            for (int oc = 0; oc < ro / 8; ++oc) t += octss[oc];
            st_async_b32(peer_addr(q4d::smem_addr(bsum_next + rank), (uint32_t)lane), __float_as_uint(t),
                         peer_addr(hbar, (uint32_t)lane));
        }
    }
    return ok;
}

// 1/rms from the S block sums of squares (the same order in every CTA).
__device__ __forceinline__ float rinv_from(const float* bsum, int S, int H, float eps) {
    float t = 0.f;
    for (int b = 0; b < S; ++b) t += bsum[b];
    return rsqrtf(t / (float)H + eps);
}

// 16-bit tag of layer l's input h in step `step` (never 0, so zeroed words
// never look current).
__host__ __device__ inline uint32_t htag_of(uint32_t step, int L, int l) {
    return 1u + (uint32_t)(((unsigned long long)step * (unsigned)L + (unsigned)l) % 65535ull);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// x * norm weight of one octet (8 inputs) in the dot_rows layout, and its sum
// of squares: the one formula both kernels use for every layer's input.
__device__ __forceinline__ void stage_octet(const float* f, const float* g, float4* xs, float* nss, int j) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    nss[j] = ss;
    float4* d = xs + xs_slot(j);
    d[0] = make_float4(f[0] * g[0], f[4] * g[4], f[1] * g[1], f[5] * g[5]);
    d[32] = make_float4(f[2] * g[2], f[6] * g[6], f[3] * g[3], f[7] * g[7]);
}

// Block sums of squares from all octet sums (block b = octets b ro/8 ..
// (b+1) ro/8 - 1, in order), by threads 0 .. S-1: the order collect() uses.
__device__ __forceinline__ void block_sums(const float* nss, float* bsum, int S, int ro) {
    const int b = threadIdx.x;
    if (b < S) {
        float t = 0.f;
        for (int oc = 0; oc < ro / 8; ++oc) t += nss[b * (ro / 8) + oc];
        bsum[b] = t;
    }
}

__global__ void __launch_bounds__(kThreads, 1) q4_step_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int c = (int)cluster_index(), i = (int)cluster_rank();
    const int S = p.S, C = p.C, H = p.H, ro = p.ro, L = p.L;
    // the k / v kernel may start once every CTA of this grid runs
    q4d::pdl_trigger();
    float4* xs0 = reinterpret_cast<float4*>(smem + p.off_xs);                 // attention half input
    float4* xs1 = reinterpret_cast<float4*>(smem + p.off_xs + p.xs_bytes);    // FFN half input
    float* bsum0 = reinterpret_cast<float*>(smem + p.off_bsum);               // their block sums of squares
    float* bsum1 = bsum0 + S;
    float* nss = reinterpret_cast<float*>(smem + p.off_nss);                  // octet sums of squares
    uint16_t* hown = reinterpret_cast<uint16_t*>(smem + p.off_hown);          // this CTA's block of h / h'
    uint16_t* gown = reinterpret_cast<uint16_t*>(smem + p.off_gown);          // [2L][ro] norm weights of that block
    float* rowout = reinterpret_cast<float*>(smem + p.off_rows);              // row totals of a row item
    float* qx = reinterpret_cast<float*>(smem + p.off_qx);                    // the cluster's q block
    float* ax = reinterpret_cast<float*>(smem + p.off_ax);                    // the cluster's act block
    float* red = reinterpret_cast<float*>(smem + p.off_red);                  // [0, ro): this CTA's partials
    float* pg = red + ro;                                                     // per-group partials
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint8_t* ring = smem + p.off_ring;
    const uint32_t full0 = q4d::smem_addr(bars), empty0 = q4d::smem_addr(bars + kMaxSlots);
    const uint32_t qbar = q4d::smem_addr(bars + 2 * kMaxSlots), abar = qbar + 8, hbar = qbar + 16;
    const Work w = work_of(p.QN, p.KVN, p.F, C, S, c, i);
    const int oa = i * ro;
    const uint32_t q_bytes = 64u * (uint32_t)(w.qg1 - w.qg0) * 4u, a_bytes = 64u * (uint32_t)(w.fg1 - w.fg0) * 4u;
    // per broadcast: two float4 of x per octet and every peer's block sum of squares
    const uint32_t h_bytes = (uint32_t)(H / 8) * 32u + (uint32_t)S * 4u;

    __shared__ uint32_t step_sh;
    __shared__ int issued_sh, consumed_sh;
    __shared__ volatile int abort_sh;
    if (tid == 0) {
        for (int s = 0; s < p.slots; ++s) {
            q4d::mbar_init(full0 + 8 * s, 32);
            q4d::mbar_init(empty0 + 8 * s, kWarps);
        }
        q4d::mbar_init(qbar, 1);
        q4d::mbar_init(abar, 1);
        q4d::mbar_init(hbar, 1);
        q4d::fence_mbar_init();
        step_sh = q4d::ld_relaxed(p.ctr);
        issued_sh = 0;
        consumed_sh = 0x7fffffff;
        abort_sh = 0;
    }
    // q / act blocks zeroed (their tails past the cluster's share stay zero,
    // so padded columns contribute nothing); the norm weights of this CTA's
    // rows for every layer (ones where a layer has none); this CTA's block of
    // x; layer 0's input x * attn_norm and its block sums of squares
    for (int e = tid; e < p.qspan * 64; e += kThreads) qx[e] = 0.f;
    for (int e = tid; e < p.fspan * 64; e += kThreads) ax[e] = 0.f;
    for (int e = tid; e < 2 * L * ro; e += kThreads) {
        const int l = e / (2 * ro), which = (e / ro) & 1, r = e - (e / ro) * ro;
        const uint16_t* g = which ? p.layers[l].ffn_norm : p.layers[l].attn_norm;
        gown[e] = g ? g[oa + r] : (uint16_t)0x3C00;
    }
    for (int r = tid; r < ro; r += kThreads) hown[r] = p.x[oa + r];
    {
        const uint16_t* g0 = p.layers[0].attn_norm;
        for (int j = tid; j < H / 8; j += kThreads) {
            float f[8], g[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                f[e] = __half2float(__ushort_as_half(p.x[8 * j + e]));
                g[e] = g0 ? __half2float(__ushort_as_half(g0[8 * j + e])) : 1.f;
            }
            stage_octet(f, g, xs0, nss, j);
        }
    }
    __syncthreads();
    block_sums(nss, bsum0, S, ro);
    if (tid == 0) {
        // phase 0 of each exchange barrier: this thread's arrival plus the bytes peers send
        q4d::mbar_arrive_expect_tx(qbar, q_bytes);
        q4d::mbar_arrive_expect_tx(abar, a_bytes);
        q4d::mbar_arrive_expect_tx(hbar, h_bytes);
    }
    cluster_sync();  // every peer's barriers are initialised before anything is sent (and bsum0 is complete)

    if (warp == kProducerWarp) {
        // ------------------------------------------------------ producer warp
        // q rows, o column block, gate/up rows, down column block of every layer
        const uint64_t pol = q4d::policy_evict_first();
        int n = 0;
        for (int l = 0; l < L && !abort_sh; ++l) {
            const LayerDesc& Ld = p.layers[l];
            for (int ii = 0; ii < kItems; ++ii, ++n) {
                const int it = ii < 2 ? ii : ii + 1;  // item kinds 0, 1, 3, 4 (2, the k / v rows, is not streamed here)
                const int st = n % p.slots, k = n / p.slots;
                if (k > 0) {
                    int ok = 1;
                    if (lane == 0) ok = (q4d::mbar_wait(empty0 + 8 * st, (k - 1) & 1, p.err) && !abort_sh) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, ok, 0)) {
                        l = L;
                        break;
                    }
                }
                uint8_t* slot = ring + (size_t)st * p.slot_bytes;
                const uint32_t fb = full0 + 8 * st;
                if (lane == 0) {
                    const uint32_t bytes = issue_item(p, Ld, p.maps + 6 * l, w, it, i, slot, fb, false, pol);
                    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(fb), "r"(bytes)
                                 : "memory");
                    issue_item(p, Ld, p.maps + 6 * l, w, it, i, slot, fb, true, pol);
                }
                __syncwarp();
                q4d::mbar_arrive(fb);
            }
        }
        if (lane == 0) issued_sh = n;
    } else {
        // ---------------------------------------------------------- consumers
        const uint32_t step = step_sh;
        bool bad = false;
        int n = 0;  // items consumed
        // The next weight item: lane 0 waits and the warp shares the outcome,
        // so `bad` stays uniform within a warp (the warp-wide shuffles need
        // every lane); named_bar_or makes it uniform across the CTA.  A failed
        // or skipped wait returns nullptr and the item is not released (its
        // copies may still be in flight).  Items are waited for behind the
        // hand-off waits (a completed-phase wait still costs a few hundred
        // cycles), so that cost overlaps them.
        auto item_wait = [&](int& slot_idx) -> const uint8_t* {
            slot_idx = n % p.slots;
            int ok = 0;
            if (lane == 0 && !bad) ok = q4d::mbar_wait(full0 + 8 * slot_idx, (n / p.slots) & 1, p.err) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                bad = true;
                return nullptr;
            }
            return ring + (size_t)slot_idx * p.slot_bytes;
        };
        auto item_done = [&](int slot_idx) {
            __syncwarp();
            if (lane == 0) q4d::mbar_arrive(empty0 + 8 * slot_idx);
            ++n;
        };
        auto tag_of = [&](int e) {
            return (uint32_t)((unsigned long long)step * (unsigned)(2 * L) + (unsigned)e + 1u);
        };
        // wait for a phase of the cluster's broadcasts (the next half's
        // input), then arm the barrier's next phase
        auto wait_h = [&](uint32_t par) {
            if (!bad && !wait_cluster_bar(hbar, par, p.err)) bad = true;
            if (tid == 0) q4d::mbar_arrive_expect_tx(hbar, h_bytes);
            bad = q4d::named_bar_or(1, kCT, bad);
        };

        int sl = 0;
        const uint8_t* slot = item_wait(sl);  // layer 0's q rows
        for (int l = 0; l < L && !bad; ++l) {
            unsigned long long* Xa = p.xch + (size_t)(2 * l) * C * H;
            unsigned long long* Xf = Xa + (size_t)C * H;
            // ---------------- attention half: q rows (sent to the cluster),
            // the o partial, published; the next half's input collected
            Q4_TRACE(0);
            const int nq = w.qb - w.qa;
            RowItem ri = row_item(H, nq, 0);
            if (slot) dot_rows<kWarps>(slot, ri, nq, 0, H, xs0, warp, lane, rowout);
            const float rinv = rinv_from(bsum0, S, H, p.eps);
            q4d::named_bar(1, kCT);
            Q4_TRACE(1);
            if (slot) item_done(sl);
            // four rows per 16-byte store (a CTA's share of a cluster's rows is
            // a multiple of 4, starting at a multiple of 4)
            for (int idx = tid; idx < (nq / 4) * S; idx += kCT) {
                const int r4 = idx / S, peer = idx - r4 * S;
                uint16_t qh[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) qh[e] = __half_as_ushort(__float2half_rn(rowout[4 * r4 + e] * rinv));
                if (peer == 0)
                    *reinterpret_cast<uint2*>(p.q + w.qa + 4 * r4) =
                        make_uint2(qh[0] | ((uint32_t)qh[1] << 16), qh[2] | ((uint32_t)qh[3] << 16));
                st_async_v4(peer_addr(q4d::smem_addr(qx + (w.qa + 4 * r4 - 64 * w.qg0)), (uint32_t)peer),
                            make_uint4(__float_as_uint(__half2float(__ushort_as_half(qh[0]))),
                                       __float_as_uint(__half2float(__ushort_as_half(qh[1]))),
                                       __float_as_uint(__half2float(__ushort_as_half(qh[2]))),
                                       __float_as_uint(__half2float(__ushort_as_half(qh[3])))),
                            peer_addr(qbar, (uint32_t)peer));
            }
            Q4_TRACE(2);
            slot = item_wait(sl);  // the o column block
            // the cluster's q block is complete once every peer's share arrived
            if (!bad && !wait_cluster_bar(qbar, l & 1, p.err)) bad = true;
            Q4_TRACE(3);
            if (tid == 0) q4d::mbar_arrive_expect_tx(qbar, q_bytes);  // the next layer's phase
            col_partial(slot, col_item(ro, p.qspan, p.qspan_s), p.qspan, p.qspan_s, w.qg0, qx, ro, pg, red);
            if (slot) item_done(sl);
            Q4_TRACE(4);
            publish(Xa, red, c, H, oa, ro, tag_of(2 * l));
            Q4_TRACE(5);
            if (!collect(Xa, hown, gown + (size_t)(2 * l + 1) * ro, xs1, bsum1, nss, c == 0 ? p.h_mid : nullptr,
                         nullptr, 0, C, H, S, oa, ro, i, tag_of(2 * l), hbar, p.err, bad))
                bad = true;
            Q4_TRACE(6);
            slot = item_wait(sl);  // gate / up rows
            wait_h(0);
            Q4_TRACE(7);
            if (bad) break;
            // ---------------- FFN half: act = SiLU(gate) * up (sent to the
            // cluster), the down partial, published; the next layer's input
            // collected
            const int nf = w.fb - w.fa;
            ri = row_item(H, nf, nf);
            if (slot) dot_rows<kWarps>(slot, ri, nf, nf, H, xs1, warp, lane, rowout);
            const float rinv2 = rinv_from(bsum1, S, H, p.eps);
            q4d::named_bar(1, kCT);
            Q4_TRACE(8);
            if (slot) item_done(sl);
            for (int idx = tid; idx < (nf / 4) * S; idx += kCT) {
                const int r4 = idx / S, peer = idx - r4 * S;
                uint16_t ah[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 4 * r4 + e;
                    const float g = rowout[r] * rinv2, u = rowout[nf + r] * rinv2;
                    ah[e] = __half_as_ushort(__float2half_rn(g / (1.0f + expf(-g)) * u));
                }
                if (peer == 0)
                    *reinterpret_cast<uint2*>(p.act + w.fa + 4 * r4) =
                        make_uint2(ah[0] | ((uint32_t)ah[1] << 16), ah[2] | ((uint32_t)ah[3] << 16));
                st_async_v4(peer_addr(q4d::smem_addr(ax + (w.fa + 4 * r4 - 64 * w.fg0)), (uint32_t)peer),
                            make_uint4(__float_as_uint(__half2float(__ushort_as_half(ah[0]))),
                                       __float_as_uint(__half2float(__ushort_as_half(ah[1]))),
                                       __float_as_uint(__half2float(__ushort_as_half(ah[2]))),
                                       __float_as_uint(__half2float(__ushort_as_half(ah[3])))),
                            peer_addr(abar, (uint32_t)peer));
            }
            Q4_TRACE(9);
            slot = item_wait(sl);  // the down column block
            if (!bad && !wait_cluster_bar(abar, l & 1, p.err)) bad = true;
            Q4_TRACE(10);
            if (tid == 0) q4d::mbar_arrive_expect_tx(abar, a_bytes);
            col_partial(slot, col_item(ro, p.fspan, p.fspan_s), p.fspan, p.fspan_s, w.fg0, ax, ro, pg, red);
            if (slot) item_done(sl);
            Q4_TRACE(11);
            publish(Xf, red, c, H, oa, ro, tag_of(2 * l + 1));
            const bool next = l + 1 < L;
            Q4_TRACE(12);
            if (!collect(Xf, hown, next ? gown + (size_t)(2 * l + 2) * ro : nullptr, xs0, bsum0, nss,
                         c == 0 ? p.h : nullptr, (c == 0 && next) ? p.htag + (size_t)(l + 1) * H : nullptr,
                         htag_of(step, L, l + 1), C, H, S, oa, ro, i, tag_of(2 * l + 1), hbar, p.err, bad))
                bad = true;
            Q4_TRACE(13);
            if (next) {
                slot = item_wait(sl);  // the next layer's q rows
                wait_h(1);
            }
            Q4_TRACE(14);
        }
        if (bad && tid == 0) abort_sh = 1;
        if (lane == 0) atomicMin(&consumed_sh, n);
    }
    __syncthreads();
    if (tid == 0) {
        // copies still landing in slots nobody will read (after an abort)
        for (int j = consumed_sh; j < issued_sh; ++j)
            q4d::mbar_wait(full0 + 8 * (j % p.slots), (j / p.slots) & 1, nullptr);
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(p.ctr + 1, 1u) == gridDim.x - 1) {
            p.ctr[1] = 0;
            __threadfence();
            atomicAdd(p.ctr, 1u);
        }
    }
}

// ---------------------------------------------------------------- k / v kernel
__global__ void __launch_bounds__(kKvThreads, 1) q4_step_kv_kernel(const __grid_constant__ KvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int H = p.H, L = p.L, S = p.S;
    constexpr int NW = kKvThreads / 32;
    uint16_t* h = reinterpret_cast<uint16_t*>(smem + p.off_h);  // the layer's input h
    float4* xs = reinterpret_cast<float4*>(smem + p.off_xs);
    float* nss = reinterpret_cast<float*>(smem + p.off_nss);
    float* bsum = nss + H / 8;
    float* rows = reinterpret_cast<float*>(smem + p.off_rows);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint8_t* ring = smem + p.off_ring;
    const uint32_t full0 = q4d::smem_addr(bars);
    // this CTA's rows of the k and v rows taken as one list
    int a, b;
    split(2 * p.KVN, (int)gridDim.x, (int)blockIdx.x, a, b);
    const int k0 = a < p.KVN ? a : p.KVN, k1 = b < p.KVN ? b : p.KVN;
    const int v0 = (a > p.KVN ? a : p.KVN) - p.KVN, v1 = (b > p.KVN ? b : p.KVN) - p.KVN;
    const int nk = k1 - k0, nv = v1 - v0;
    const RowItem ri = row_item(H, nk, nv);
    __shared__ uint32_t step_sh;
    if (tid == 0) {
        q4d::mbar_init(full0, 1);
        q4d::mbar_init(full0 + 8, 1);
        q4d::fence_mbar_init();
        step_sh = q4d::ld_relaxed(p.ctr + 3);  // this kernel's steps so far = the clustered kernel's step
    }
    __syncthreads();
    const uint32_t step = step_sh;
    const uint64_t pol = q4d::policy_evict_first();
    auto issue = [&](int l) {  // one thread
        const LayerDesc& Ld = p.layers[l];
        uint8_t* slot = ring + (size_t)(l & 1) * p.slot_bytes;
        const uint32_t fb = full0 + 8 * (l & 1);
        const uint32_t bytes = (uint32_t)(nk + nv) * ((uint32_t)H / 2 + 2u * ((uint32_t)H / 32));
        q4d::mbar_arrive_expect_tx(fb, bytes);
        issue_rows(Ld.k, k0, nk, H, slot + ri.cA, slot + ri.sA, slot + ri.bA, fb, pol);
        issue_rows(Ld.v, v0, nv, H, slot + ri.cB, slot + ri.sB, slot + ri.bB, fb, pol);
    };
    const int first = L < 2 ? L : 2;
    if (tid == 0)
        for (int l = 0; l < first; ++l) issue(l);
    int issued = first, consumed = 0;
    for (int l = 0; l < L; ++l) {
        // layer l's input: the step's x, else the clustered kernel's tagged copy
        if (l == 0) {
            for (int j = tid; j < H; j += kKvThreads) h[j] = p.x[j];
        } else {
            const uint32_t tg = htag_of(step, L, l);
            const uint32_t* src = p.htag + (size_t)l * H;
            bool ok = true;
            for (int j = 4 * tid; ok && j < H; j += 4 * kKvThreads) {
                uint4 v = q4d::ld_relaxed_v4(src + j);
                unsigned long long t0 = 0;
                for (uint32_t it = 1; (v.x >> 16) != tg || (v.y >> 16) != tg || (v.z >> 16) != tg ||
                                      (v.w >> 16) != tg;
                     ++it) {
                    if ((it & 15u) == 0) {
                        if (t0 == 0) {
                            t0 = q4d::globaltimer();
                        } else if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
                            atomicOr(p.err, q4d::kErrTimeout);
                            ok = false;
                            break;
                        }
                    }
                    __nanosleep(256);  // this kernel trails the clusters: poll gently
                    v = q4d::ld_relaxed_v4(src + j);
                }
                *reinterpret_cast<uint2*>(h + j) =
                    make_uint2((v.x & 0xFFFFu) | (v.y << 16), (v.z & 0xFFFFu) | (v.w << 16));
            }
            if (__syncthreads_or(!ok)) break;
        }
        __syncthreads();
        {
            // x * attn_norm and the sums of squares, in the clustered kernel's order
            const uint16_t* g = p.layers[l].attn_norm;
            for (int j = tid; j < H / 8; j += kKvThreads) {
                float f[8], gm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    f[e] = __half2float(__ushort_as_half(h[8 * j + e]));
                    gm[e] = g ? __half2float(__ushort_as_half(g[8 * j + e])) : 1.f;
                }
                stage_octet(f, gm, xs, nss, j);
            }
        }
        __syncthreads();
        block_sums(nss, bsum, S, p.ro);
        __syncthreads();
        Q4_TRACE_T(20, 0);
        const float rinv = rinv_from(bsum, S, H, p.eps);
        int ok = 0;
        if (lane == 0) ok = q4d::mbar_wait(full0 + 8 * (l & 1), (l >> 1) & 1, p.err) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (__syncthreads_or(!ok)) break;
        dot_rows<NW>(ring + (size_t)(l & 1) * p.slot_bytes, ri, nk, nv, H, xs, warp, lane, rows);
        __syncthreads();  // the slot and x are read
        ++consumed;
        if (tid == 0 && l + 2 < L) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(l + 2);
        }
        if (l + 2 < L) ++issued;
        for (int r = tid; r < nk + nv; r += kKvThreads) {
            const uint16_t hv = __half_as_ushort(__float2half_rn(rows[r] * rinv));
            if (r < nk) p.k[k0 + r] = hv;
            else p.v[v0 + r - nk] = hv;
        }
        Q4_TRACE_T(21, 0);
    }
    __syncthreads();
    if (tid == 0) {
        // copies still landing in slots nobody will read (after an abort)
        for (int j = consumed; j < issued; ++j) q4d::mbar_wait(full0 + 8 * (j & 1), (j >> 1) & 1, nullptr);
        // The step ends when both kernels have: wait for the clustered kernel
        // (it counts its finished steps), then count this CTA.
        const unsigned long long t0 = q4d::globaltimer();
        while (ld_acquire_gpu(p.ctr) < step + 1u) {
            __nanosleep(256);
            if (q4d::globaltimer() - t0 > q4d::kWaitLimitNs) {
                atomicOr(p.err, q4d::kErrTimeout);
                break;
            }
        }
        __threadfence();
        if (atomicAdd(p.ctr + 4, 1u) == gridDim.x - 1) {
            p.ctr[4] = 0;
            __threadfence();
            atomicAdd(p.ctr + 3, 1u);
        }
    }
}

}  // namespace q4s

namespace q4i {

size_t step_layer_desc_bytes() { return sizeof(q4s::LayerDesc); }

// Plans the clustered step for the given dims; false (with Q4_OK) when the
// shapes or the device do not allow it.
q4_status step_plan(const StepArgs& a, StepPlan* out, bool* ok) {
    *ok = false;
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    const int H = a.H, QN = a.QN, KVN = a.KVN, F = a.F, L = a.L;
    if (L < 1 || H % 512 || QN % 512 || F % 512 || KVN % 64 || KVN < 64) return Q4_OK;
    auto kern = q4s::q4_step_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return Q4_OK;
    }
    const int smem_max = dev->smem_optin - 1024;  // static shared variables and slack
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(q4_step_kernel)");
    for (int S : {16, 8}) {
        if (H % S || H / S > 256 || (H / S) % 8) continue;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = (unsigned)S;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.blockDim = dim3(q4s::kThreads);
        cfg.dynamicSmemBytes = (size_t)smem_max;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3((unsigned)S);
        int ncl = 0;
        e = cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg);
        if (e != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        int C = ncl < kStepMaxClusters ? ncl : kStepMaxClusters;
        if (C < 2) continue;
        q4s::Params p = {};
        p.L = L;
        p.H = H;
        p.QN = QN;
        p.KVN = KVN;
        p.F = F;
        p.C = C;
        p.S = S;
        p.eps = a.eps;
        p.ro = H / S;
        // column-block widths: the largest cluster share, and its scale box
        int qs = 0, fs = 0;
        for (int cc = 0; cc < C; ++cc) {
            int g0, g1;
            q4s::split(QN / 64, C, cc, g0, g1);
            qs = g1 - g0 > qs ? g1 - g0 : qs;
            q4s::split(F / 64, C, cc, g0, g1);
            fs = g1 - g0 > fs ? g1 - g0 : fs;
        }
        if (qs < 1 || fs < 1 || qs > 32 || fs > 32) continue;
        p.qspan = qs;
        p.fspan = fs;
        p.qspan_s = (qs + 7 + 7) & ~7;
        p.fspan_s = (fs + 7 + 7) & ~7;
        // slot size: the largest ring item of any CTA (q rows, gate/up rows,
        // the column blocks); the most rows a row item has
        uint32_t slot = 0;
        int max_rows = 0;
        for (int cc = 0; cc < C; ++cc)
            for (int ii = 0; ii < S; ++ii) {
                const q4s::Work w = q4s::work_of(QN, KVN, F, C, S, cc, ii);
                const int nr[2][2] = {{w.qb - w.qa, 0}, {w.fb - w.fa, w.fb - w.fa}};
                for (const auto& r : nr) {
                    const uint32_t b = q4s::row_item(H, r[0], r[1]).gam;
                    slot = b > slot ? b : slot;
                    max_rows = r[0] + r[1] > max_rows ? r[0] + r[1] : max_rows;
                }
            }
        const uint32_t co = q4s::col_item(p.ro, qs, p.qspan_s).end, cd = q4s::col_item(p.ro, fs, p.fspan_s).end;
        slot = co > slot ? co : slot;
        slot = cd > slot ? cd : slot;
        slot = q4s::align128(slot);
        // fixed shared memory: x of both halves (fp32, lane-interleaved) and
        // their block sums of squares, the octet sums of squares, this CTA's
        // h block and norm weights, the row totals, the q / act blocks, the
        // partials, barriers
        uint32_t off = 0;
        p.off_xs = off;
        p.xs_bytes = q4s::align128((uint32_t)((H / 8 + 127) / 128) * 8u * 32u * 16u);
        off += 2 * p.xs_bytes;
        p.off_bsum = off;
        off += q4s::align128(2u * (uint32_t)S * 4u);
        p.off_nss = off;
        off += q4s::align128((uint32_t)(H / 8) * 4u);
        p.off_hown = off;
        off += q4s::align128((uint32_t)p.ro * 2u);
        p.off_gown = off;
        off += q4s::align128(2u * (uint32_t)L * (uint32_t)p.ro * 2u);
        p.off_rows = off;
        off += q4s::align128((uint32_t)max_rows * 4u);
        p.off_qx = off;
        off += q4s::align128((uint32_t)qs * 64u * 4u);
        p.off_ax = off;
        off += q4s::align128((uint32_t)fs * 64u * 4u);
        p.off_red = off;
        off += q4s::align128((uint32_t)(1 + (qs > fs ? qs : fs)) * (uint32_t)p.ro * 4u);
        p.off_bar = off;
        off += q4s::align128((2 * q4s::kMaxSlots + 3) * 8u);
        p.off_ring = off;
        if ((uint32_t)smem_max < off + 2 * slot) continue;
        int slots = (int)(((uint32_t)smem_max - off) / slot);
        if (slots > q4s::kMaxSlots) slots = q4s::kMaxSlots;
        p.slots = slots;
        p.slot_bytes = slot;

        // the k / v launch: one CTA on each SM the clusters leave free (at
        // least 8; any that do not fit beside the clusters run after them)
        q4s::KvParams kp = {};
        kp.L = L;
        kp.H = H;
        kp.KVN = KVN;
        kp.S = S;
        kp.ro = p.ro;
        kp.eps = a.eps;
        const int G2 = dev->sms - C * S > 8 ? dev->sms - C * S : 8;
        uint32_t kslot = 0;
        int kmax = 0;
        for (int bb = 0; bb < G2; ++bb) {
            int ra, rb;
            q4s::split(2 * KVN, G2, bb, ra, rb);
            const int nk = (rb < KVN ? rb : KVN) - (ra < KVN ? ra : KVN);
            const int nv = (rb > KVN ? rb : KVN) - (ra > KVN ? ra : KVN);
            const uint32_t b2 = q4s::row_item(H, nk, nv).gam;
            kslot = b2 > kslot ? b2 : kslot;
            kmax = nk + nv > kmax ? nk + nv : kmax;
        }
        kp.slot_bytes = q4s::align128(kslot);
        kp.xs_bytes = p.xs_bytes;
        uint32_t ko = 0;
        kp.off_h = ko;
        ko += q4s::align128((uint32_t)H * 2u);
        kp.off_xs = ko;
        ko += kp.xs_bytes;
        kp.off_nss = ko;  // the octet sums of squares, then the block sums
        ko += q4s::align128((uint32_t)(H / 8 + S) * 4u);
        kp.off_rows = ko;
        ko += q4s::align128((uint32_t)(kmax > 0 ? kmax : 1) * 4u);
        kp.off_bar = ko;
        ko += 128;
        kp.off_ring = ko;
        ko += 2 * kp.slot_bytes;
        if (ko > (uint32_t)smem_max) continue;
        e = cudaFuncSetAttribute(q4s::q4_step_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ko);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(q4_step_kv_kernel)");
        out->kv_grid = G2;
        out->kv_smem = ko;
        static_assert(sizeof(q4s::KvParams) <= sizeof(out->kv_params), "StepPlan k / v params storage");
        memcpy(out->kv_params, &kp, sizeof(kp));
        out->S = S;
        out->C = C;
        out->smem = (size_t)off + (size_t)slots * slot;
        static_assert(sizeof(q4s::Params) <= sizeof(out->params), "StepPlan params storage");
        memcpy(out->params, &p, sizeof(p));
        *ok = true;
        return Q4_OK;
    }
    return Q4_OK;
}

// Fills the device tables (layer descriptors, tensor maps) for the plan
// (host copies in `host`, uploaded by the caller) and the pointers of the
// launch.
q4_status step_bind(StepPlan* sp, const StepArgs& a, void* host_layers, void* host_maps) {
    q4s::Params p;
    memcpy(&p, sp->params, sizeof(p));
    q4s::LayerDesc* Ld = static_cast<q4s::LayerDesc*>(host_layers);
    CUtensorMap* maps = static_cast<CUtensorMap*>(host_maps);
    for (int l = 0; l < a.L; ++l) {
        const q4_layer_weights& w = a.layers[l];
        auto lin = [](const q4_linear& m) { return q4s::Lin{m.Wq, m.scales, m.biases}; };
        Ld[l].q = lin(w.q);
        Ld[l].k = lin(w.k);
        Ld[l].v = lin(w.v);
        Ld[l].gate = lin(w.gate);
        Ld[l].up = lin(w.up);
        Ld[l].attn_norm = w.attn_norm;
        Ld[l].ffn_norm = w.ffn_norm;
        const q4_linear* cm[2] = {&w.o, &w.down};
        const int spans[2] = {p.qspan, p.fspan}, spans_s[2] = {p.qspan_s, p.fspan_s};
        for (int m = 0; m < 2; ++m) {
            const q4_linear& lw = *cm[m];
            const uint64_t K = (uint64_t)lw.K, N = (uint64_t)lw.N;
            q4_status st = make_map(&maps[6 * l + 3 * m], CU_TENSOR_MAP_DATA_TYPE_UINT32, lw.Wq, K / 8, N, K / 2,
                                    (uint32_t)spans[m] * 8u, (uint32_t)p.ro, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != Q4_OK) return st;
            st = make_map(&maps[6 * l + 3 * m + 1], CU_TENSOR_MAP_DATA_TYPE_UINT16, lw.scales, K / 64, N, K / 32,
                          (uint32_t)spans_s[m], (uint32_t)p.ro, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != Q4_OK) return st;
            st = make_map(&maps[6 * l + 3 * m + 2], CU_TENSOR_MAP_DATA_TYPE_UINT16, lw.biases, K / 64, N, K / 32,
                          (uint32_t)spans_s[m], (uint32_t)p.ro, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (st != Q4_OK) return st;
        }
    }
    p.layers = static_cast<const q4s::LayerDesc*>(a.dev_layers);
    p.maps = static_cast<const CUtensorMap*>(a.dev_maps);
    p.x = a.x;
    p.h = a.h;
    p.h_mid = a.h_mid;
    p.q = a.q;
    p.k = a.k;
    p.v = a.v;
    p.act = a.act;
    p.xch = a.xch;
    p.htag = a.htag;
    p.ctr = a.ctr;
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    p.err = dev->err_word;
    memcpy(sp->params, &p, sizeof(p));
    q4s::KvParams kp;
    memcpy(&kp, sp->kv_params, sizeof(kp));
    kp.layers = p.layers;
    kp.x = a.x;
    kp.k = a.k;
    kp.v = a.v;
    kp.htag = a.htag;
    kp.ctr = a.ctr;
    kp.err = dev->err_word;
    memcpy(sp->kv_params, &kp, sizeof(kp));
    return Q4_OK;
}

q4_status step_launch(const StepPlan& sp, cudaStream_t stream) {
    q4s::Params p;
    memcpy(&p, sp.params, sizeof(p));
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)sp.S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(sp.C * sp.S));
    cfg.blockDim = dim3(q4s::kThreads);
    cfg.dynamicSmemBytes = sp.smem;
    cfg.stream = stream;
    // The clusters wait on one another, so all of them must be resident at
    // once: the plan sizes the grid by the occupancy query, the launch follows
    // the previous step's kernels on the stream (the GPU is otherwise idle for
    // it), and every cross-cluster wait is bounded.
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, q4s::q4_step_kernel, p);
    if (e != cudaSuccess) return cuda_fail(e, "clustered decode step launch");
    // the k / v rows: launched once every clustered CTA runs (programmatic
    // dependent launch; that kernel triggers at its start), on the free SMs;
    // it reads only the exchange words, which it polls, and never waits on
    // the clustered kernel's completion before its own end
    q4s::KvParams kp;
    memcpy(&kp, sp.kv_params, sizeof(kp));
    cudaLaunchConfig_t kc = {};
    cudaLaunchAttribute ka[1];
    ka[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    ka[0].val.programmaticStreamSerializationAllowed = 1;
    kc.gridDim = dim3((unsigned)sp.kv_grid);
    kc.blockDim = dim3(q4s::kKvThreads);
    kc.dynamicSmemBytes = sp.kv_smem;
    kc.stream = stream;
    kc.attrs = ka;
    kc.numAttrs = 1;
    e = cudaLaunchKernelEx(&kc, q4s::q4_step_kv_kernel, kp);
    if (e != cudaSuccess) return cuda_fail(e, "clustered decode step k / v launch");
    return Q4_OK;
}

}  // namespace q4i

#ifdef Q4_STEP_TRACE
// Trace build only: copies the timestamps (2 x 4096 64-bit words) to `out`.
extern "C" int q4_step_trace_read(void* out) {
    return (int)cudaMemcpyFromSymbol(out, q4s::g_step_trace, sizeof(unsigned long long) * 2 * 4096);
}
#endif
