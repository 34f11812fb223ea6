// Decode attention for one token over a preallocated KV cache, with rotary
// position embedding (BaseRT: optimal LLM inference on Apple Silicon with
// native Metal, §3.3 lists RoPE, attention and normalisation among the decode
// kernels, and §3.2 keeps the KV cache preallocated so the decode loop
// allocates nothing).
//
// Shape: Hq query heads and Hkv key/value heads of head_dim d (query head h
// reads kv head h / (Hq / Hkv)); the cache of one layer is fp16
// [Hkv][max_seq][d]; the token's position is read from device memory, so a
// captured decode graph replays unchanged from step to step.
//
// GB300 design: attention of one token is a memory-bound pass over the cache
// (2 x Hkv x d x 2 bytes per position), so it is split over positions
// (flash-decoding): one CTA per (kv head, chunk of 64 positions) brings the
// chunk's keys and values into shared memory with two bulk copies (the
// positions of a head are contiguous, 16 KB each at d = 128) on one mbarrier,
// rotates the group's queries meanwhile, scores every query head of the group
// (a warp per position, lanes across d), turns the scores into exp(s - max),
// and accumulates the values (threads across d and positions, the partial
// sums added in shared memory); a second kernel merges
// the chunks' (max, sum, partial output) per head.  The rotation's sines and
// cosines are computed once per step in fp64 (the angle pos * theta^(-2i/d)
// reaches thousands of radians) by the first append kernel of the step into a
// table the other kernels read; the rotations themselves are fp32.  Inside a
// decode step only the first layer launches that append kernel: in the other
// layers the CTA whose chunk holds the new position appends the token itself.
//
// Prefill (second half of the file): for a chunk of prompt tokens, one table
// of rotations per chunk, an append kernel per layer writing the chunk's
// rotated keys and values into the caches, and a causal attention that is a
// dense contraction (every token against every earlier key), so it runs on
// the tensor cores, flash-attention style.
#include <cuda_fp16.h>
#include <math.h>

#include "q4_device.cuh"
#include "q4_internal.h"
#include "q4_tc.cuh"

namespace q4a {

constexpr int kChunk = 64;    // positions per CTA
constexpr int kThreads = 256;
constexpr int kMaxGroup = 8;  // query heads per kv head

__device__ __forceinline__ void rope_cs(int pos, int i, int d, double log2_theta, float& c, float& s) {
    const double ang = (double)pos * exp2(-2.0 * (double)i / (double)d * log2_theta);
    double sd, cd;
    sincos(ang, &sd, &cd);
    c = (float)cd;
    s = (float)sd;
}

__device__ __forceinline__ bool pos_ok(int pos, int max_seq, int* err) {
    if (pos < 0 || pos >= max_seq) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(err, q4d::kErrDeviceCheck);
        return false;
    }
    return true;
}

// The new key, rotated, and the new value into position *pos of the caches.
// Grid Hkv, block d/2: thread i turns the pair (i, i + d/2).  With kTable the
// sines and cosines are computed here (fp64) and block 0 stores them in `cs`
// for the other kernels of the step; otherwise they are read from `cs`.
template <bool kTable>
__global__ void rope_append_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                   uint16_t* __restrict__ kc, uint16_t* __restrict__ vc, const int32_t* pos_p, int d,
                                   int max_seq, double log2_theta, float2* cs, int* err) {
    const int h = blockIdx.x, i = threadIdx.x, half = d / 2;
    const int pos = *pos_p;
    if (!pos_ok(pos, max_seq, err)) return;
    float c, s;
    if constexpr (kTable) {
        rope_cs(pos, i, d, log2_theta, c, s);
        if (h == 0) cs[i] = make_float2(c, s);
    } else {
        const float2 t = cs[i];
        c = t.x;
        s = t.y;
    }
    const float lo = __half2float(__ushort_as_half(k[h * d + i]));
    const float hi = __half2float(__ushort_as_half(k[h * d + i + half]));
    const size_t base = ((size_t)h * max_seq + pos) * d;
    kc[base + i] = __half_as_ushort(__float2half_rn(lo * c - hi * s));
    kc[base + i + half] = __half_as_ushort(__float2half_rn(hi * c + lo * s));
    vc[base + i] = v[h * d + i];
    vc[base + i + half] = v[h * d + i + half];
}

// Dynamic shared memory of the split kernel: the chunk's keys and values,
// the rotated queries, the scores and the value pass's partial sums.
constexpr size_t split_smem(int D) {
    return (size_t)2 * kChunk * D * 2 + (size_t)kMaxGroup * D * 4 + (size_t)kMaxGroup * kChunk * 4 +
           (size_t)kThreads * kMaxGroup * 4;
}

// One (kv head, chunk) of the attention: for each query head g of the group,
// m = max score, l = sum exp(s - m), acc = sum exp(s - m) v over the chunk.
template <int D>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const uint16_t* __restrict__ q,
                                                              const uint16_t* kc,  // bulk-copy sources; the
                                                              const uint16_t* vc,  // append writes via kc_w / vc_w
                                                              const int32_t* pos_p,
                                                              int G, int max_seq, int n_splits,
                                                              const float2* __restrict__ cs,
                                                              float* __restrict__ part_ml,
                                                              float* __restrict__ part_acc,
                                                              const uint16_t* __restrict__ k_new,
                                                              const uint16_t* __restrict__ v_new,
                                                              uint16_t* kc_w, uint16_t* vc_w, int* err) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t* ks = reinterpret_cast<uint16_t*>(smem);  // [kChunk][D]
    uint16_t* vs = ks + kChunk * D;                    // [kChunk][D]
    float* qr = reinterpret_cast<float*>(vs + kChunk * D);  // [kMaxGroup][D]
    float* sc = qr + kMaxGroup * D;                         // [kMaxGroup][kChunk]
    float* red = sc + kMaxGroup * kChunk;                   // [kThreads / D][kMaxGroup][D]
    __shared__ __align__(8) uint64_t bar;
    const int kvh = blockIdx.x, split = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pos = *pos_p;
    if (!pos_ok(pos, max_seq, err)) return;
    const int n = pos + 1, j0 = split * kChunk, j1 = min(j0 + kChunk, n), cnt = j1 - j0;
    const int h0 = kvh * G;
    if (cnt <= 0) return;  // past the context: the merge reads only the live chunks
    const uint32_t b = q4d::smem_addr(&bar);
    if (tid == 0) {
        q4d::mbar_init(b, 1);
        q4d::fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)cnt * D * 2;
        q4d::mbar_arrive_expect_tx(b, 2 * bytes);
        q4d::bulk_g2s(q4d::smem_addr(ks), kc + ((size_t)kvh * max_seq + j0) * D, bytes, b);
        q4d::bulk_g2s(q4d::smem_addr(vs), vc + ((size_t)kvh * max_seq + j0) * D, bytes, b);
    }
    // rotated queries, scaled by 1/sqrt(d), while the copies are in flight
    const float scale = rsqrtf((float)D);
    for (int t = tid; t < G * (D / 2); t += kThreads) {
        const int g = t / (D / 2), i = t % (D / 2);
        const float2 r = cs[i];
        const float lo = __half2float(__ushort_as_half(q[(h0 + g) * D + i]));
        const float hi = __half2float(__ushort_as_half(q[(h0 + g) * D + i + D / 2]));
        qr[g * D + i] = (lo * r.x - hi * r.y) * scale;
        qr[g * D + i + D / 2] = (hi * r.x + lo * r.y) * scale;
    }
    // every thread waits (bounded) for the chunk; on expiry (latched in
    // `err`) the block waits once more for its copies, then leaves
    const bool late = !q4d::mbar_wait(b, 0, err);
    if (__syncthreads_or(late)) {
        q4d::mbar_wait(b, 0, nullptr);
        return;
    }
    // Without a separate append launch (k_new set), the CTA whose chunk holds
    // the new position rotates the token's key, stores key and value in the
    // cache and over the stale row of its shared copy.
    if (k_new && pos >= j0 && pos < j1) {
        const int rs = pos - j0;
        const size_t base = ((size_t)kvh * max_seq + pos) * D;
        for (int i = tid; i < D / 2; i += kThreads) {
            const float2 r = cs[i];
            const float lo = __half2float(__ushort_as_half(k_new[kvh * D + i]));
            const float hi = __half2float(__ushort_as_half(k_new[kvh * D + i + D / 2]));
            const uint16_t klo = __half_as_ushort(__float2half_rn(lo * r.x - hi * r.y));
            const uint16_t khi = __half_as_ushort(__float2half_rn(hi * r.x + lo * r.y));
            const uint16_t vlo = v_new[kvh * D + i], vhi = v_new[kvh * D + i + D / 2];
            ks[rs * D + i] = klo;
            ks[rs * D + i + D / 2] = khi;
            vs[rs * D + i] = vlo;
            vs[rs * D + i + D / 2] = vhi;
            kc_w[base + i] = klo;
            kc_w[base + i + D / 2] = khi;
            vc_w[base + i] = vlo;
            vc_w[base + i + D / 2] = vhi;
        }
        __syncthreads();
    }
    // scores: a warp per position, lanes across d
    constexpr int E = D / 32;  // elements per lane (2 or 4)
    for (int j = warp; j < cnt; j += kThreads / 32) {
        float kf[E];
        if constexpr (E == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(ks + j * D + lane * 4);
            const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            kf[0] = x.x; kf[1] = x.y; kf[2] = y.x; kf[3] = y.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(ks + j * D + lane * 2);
            const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&raw));
            kf[0] = x.x; kf[1] = x.y;
        }
        for (int g = 0; g < G; ++g) {
            float acc = 0.f;
            if constexpr (E == 4) {
                const float4 qq = reinterpret_cast<const float4*>(qr + g * D)[lane];
                acc = fmaf(qq.x, kf[0], fmaf(qq.y, kf[1], fmaf(qq.z, kf[2], qq.w * kf[3])));
            } else {
                const float2 qq = reinterpret_cast<const float2*>(qr + g * D)[lane];
                acc = fmaf(qq.x, kf[0], qq.y * kf[1]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) sc[g * kChunk + j] = acc;
        }
    }
    __syncthreads();
    // per head: max, exp, sum (a warp per head)
    for (int g = warp; g < G; g += kThreads / 32) {
        float m = -INFINITY;
        for (int j = lane; j < cnt; j += 32) m = fmaxf(m, sc[g * kChunk + j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int j = lane; j < cnt; j += 32) {
            const float p = expf(sc[g * kChunk + j] - m);
            sc[g * kChunk + j] = p;
            l += p;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            float* ml = part_ml + ((size_t)(h0 + g) * n_splits + split) * 2;
            ml[0] = m;
            ml[1] = l;
        }
    }
    __syncthreads();
    // values: thread t takes dimension t % D and every (kThreads / D)-th
    // position from t / D on; the parts are added in index order after
    {
        constexpr int VS = kThreads / D;  // 2 (d = 128) or 4 (d = 64)
        const int dim = tid % D, part = tid / D;
        for (int g = 0; g < G; ++g) {
            const float* pg = sc + g * kChunk;
            float a0 = 0.f, a1 = 0.f;
            int j = part;
            for (; j + VS < cnt; j += 2 * VS) {
                a0 = fmaf(pg[j], __half2float(__ushort_as_half(vs[j * D + dim])), a0);
                a1 = fmaf(pg[j + VS], __half2float(__ushort_as_half(vs[(j + VS) * D + dim])), a1);
            }
            if (j < cnt) a0 = fmaf(pg[j], __half2float(__ushort_as_half(vs[j * D + dim])), a0);
            red[(part * kMaxGroup + g) * D + dim] = a0 + a1;
        }
        __syncthreads();
        for (int t2 = tid; t2 < G * D; t2 += kThreads) {
            const int g = t2 / D, dd = t2 % D;
            float s = 0.f;
#pragma unroll
            for (int pp = 0; pp < VS; ++pp) s += red[(pp * kMaxGroup + g) * D + dd];
            part_acc[((size_t)(h0 + g) * n_splits + split) * D + dd] = s;
        }
    }
}

// a[h] = sum_s acc_s e^(m_s - M) / sum_s l_s e^(m_s - M) over the live chunks.
// The chunks' (max, sum) pairs are staged in shared memory with one load per
// thread; the partial outputs are read 4 chunks at a time.
constexpr int kMaxLive = 1024;  // chunks merged in one pass (max_seq <= 1024 * kChunk)

__global__ void attn_combine_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_acc,
                                    const int32_t* pos_p, int d, int max_seq, int n_splits,
                                    uint16_t* __restrict__ a) {
    __shared__ float2 mls[kMaxLive];
    __shared__ float wsh[kMaxLive];
    __shared__ float red[2];
    const int h = blockIdx.x, t = threadIdx.x;
    const int pos = *pos_p;
    if (pos < 0 || pos >= max_seq) return;  // latched by the split kernel
    const int live = min(pos / kChunk + 1, kMaxLive);
    const float2* ml = reinterpret_cast<const float2*>(part_ml) + (size_t)h * n_splits;
    for (int s = t; s < live; s += blockDim.x) mls[s] = ml[s];
    __syncthreads();
    if (t < 32) {
        float M = -INFINITY;
        for (int s = t; s < live; s += 32) M = fmaxf(M, mls[s].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        for (int s = t; s < live; s += 32) {
            const float w = expf(mls[s].x - M);
            wsh[s] = w;
            L = fmaf(mls[s].y, w, L);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (t == 0) red[0] = L;
    }
    __syncthreads();
    const float* pa = part_acc + (size_t)h * n_splits * d + t;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    int s = 0;
    for (; s + 3 < live; s += 4) {
        const float x0 = pa[(size_t)s * d], x1 = pa[(size_t)(s + 1) * d], x2 = pa[(size_t)(s + 2) * d],
                    x3 = pa[(size_t)(s + 3) * d];
        acc0 = fmaf(x0, wsh[s], acc0);
        acc1 = fmaf(x1, wsh[s + 1], acc1);
        acc2 = fmaf(x2, wsh[s + 2], acc2);
        acc3 = fmaf(x3, wsh[s + 3], acc3);
    }
    for (; s < live; ++s) acc0 = fmaf(pa[(size_t)s * d], wsh[s], acc0);
    a[h * d + t] = __half_as_ushort(__float2half_rn(((acc0 + acc1) + (acc2 + acc3)) / red[0]));
}

__global__ void pos_advance_kernel(int32_t* pos_p, int by) { *pos_p += by; }

// ------------------------------------------------------------ prefill ---
// Prompt tokens t = 0..C-1 of a chunk sit at positions *pos_p + t0 + t.

// (cos, sin) of every (token, pair) of the chunk, fp64 angles (one table per
// chunk, shared by every layer).  Grid C, block d/2.
__global__ void prefill_cs_kernel(const int32_t* pos_p, int t0, int d, double log2_theta, float2* cs) {
    const int t = blockIdx.x, i = threadIdx.x;
    float c, s;
    rope_cs(*pos_p + t0 + t, i, d, log2_theta, c, s);
    cs[(size_t)t * (d / 2) + i] = make_float2(c, s);
}

// Two floats as an fp16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// (x, y) as an fp16 pair plus the fp16 pair of what that rounding left out.
__device__ __forceinline__ void split_h2(float x, float y, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 f = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_h2(x - f.x, y - f.y);
}

// Rotated keys and values of the chunk into the caches.  Grid C (one block
// per token), block 256; a thread takes 8 consecutive rotation pairs of one
// head (16-byte loads and stores).  k, v: [C][Hkv*d].  With qrot (the
// tensor-core attention's input), also the token's queries q [C][Hq*d],
// rotated and scaled by log2(e) / sqrt(d), as fp16 hi + lo parts:
// qrot[part][head][t][d] (part 0 hi, 1 lo).
__device__ __forceinline__ void rot8(const uint4& a, const uint4& b, const float2* r, float* x1, float* x2) {
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float l0 = __half2float(__ushort_as_half((uint16_t)(wa[e >> 1] >> (16 * (e & 1)))));
        const float h0 = __half2float(__ushort_as_half((uint16_t)(wb[e >> 1] >> (16 * (e & 1)))));
        x1[e] = l0 * r[e].x - h0 * r[e].y;
        x2[e] = h0 * r[e].x + l0 * r[e].y;
    }
}

__global__ void prefill_append_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                      uint16_t* __restrict__ kc, uint16_t* __restrict__ vc, const int32_t* pos_p,
                                      int t0, int C, int Hkv, int d, int max_seq, const float2* __restrict__ cs,
                                      const uint16_t* __restrict__ q, int Hq, uint16_t* __restrict__ qrot, int* err) {
    const int t = blockIdx.x, half = d / 2, nc = half / 8;  // 16-byte chunks per half row
    const int p0 = *pos_p + t0;
    if (p0 < 0 || p0 + C > max_seq) {
        if (t == 0 && threadIdx.x == 0) atomicOr(err, q4d::kErrDeviceCheck);
        return;
    }
    const int nk = Hkv * nc, nq = qrot ? Hq * nc : 0;
    for (int x = threadIdx.x; x < nk + nq; x += blockDim.x) {
        const bool isk = x < nk;
        const int y = isk ? x : x - nk;
        const int h = y / nc, c = y - h * nc;
        float2 r[8];
        const float4* c4 = reinterpret_cast<const float4*>(cs + (size_t)t * half + 8 * c);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 w = c4[e];
            r[2 * e] = make_float2(w.x, w.y);
            r[2 * e + 1] = make_float2(w.z, w.w);
        }
        float x1[8], x2[8];
        if (isk) {
            const size_t src = (size_t)t * Hkv * d + (size_t)h * d + 8 * c;
            rot8(*reinterpret_cast<const uint4*>(k + src), *reinterpret_cast<const uint4*>(k + src + half), r, x1, x2);
            const size_t base = ((size_t)h * max_seq + p0 + t) * d + 8 * c;
            uint32_t o1[4], o2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                o1[e] = pack_h2(x1[2 * e], x1[2 * e + 1]);
                o2[e] = pack_h2(x2[2 * e], x2[2 * e + 1]);
            }
            *reinterpret_cast<uint4*>(kc + base) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
            *reinterpret_cast<uint4*>(kc + base + half) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
            *reinterpret_cast<uint4*>(vc + base) = *reinterpret_cast<const uint4*>(v + src);
            *reinterpret_cast<uint4*>(vc + base + half) = *reinterpret_cast<const uint4*>(v + src + half);
        } else {
            const float scale = rsqrtf((float)d) * 1.4426950408889634f;  // log2(e) / sqrt(d)
            const size_t src = (size_t)t * Hq * d + (size_t)h * d + 8 * c;
            rot8(*reinterpret_cast<const uint4*>(q + src), *reinterpret_cast<const uint4*>(q + src + half), r, x1, x2);
            uint32_t h1[4], l1[4], h2[4], l2[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                split_h2(x1[2 * e] * scale, x1[2 * e + 1] * scale, h1[e], l1[e]);
                split_h2(x2[2 * e] * scale, x2[2 * e + 1] * scale, h2[e], l2[e]);
            }
            const size_t o = ((size_t)h * C + t) * d + 8 * c, part = (size_t)Hq * C * d;
            *reinterpret_cast<uint4*>(qrot + o) = make_uint4(h1[0], h1[1], h1[2], h1[3]);
            *reinterpret_cast<uint4*>(qrot + o + half) = make_uint4(h2[0], h2[1], h2[2], h2[3]);
            *reinterpret_cast<uint4*>(qrot + part + o) = make_uint4(l1[0], l1[1], l1[2], l1[3]);
            *reinterpret_cast<uint4*>(qrot + part + o + half) = make_uint4(l2[0], l2[1], l2[2], l2[3]);
        }
    }
}

// Causal attention of a prompt chunk on the tensor cores (mma.sync
// m16n8k16, fp16 operands, fp32 accumulation), flash-attention style: a CTA
// takes 64 of the chunk's tokens for one query head (a warp per 16 tokens) and
// walks the keys 0..(position of its last token) in tiles of 64 positions,
// keeping a running (max, sum, output) per token.  Key and value tiles are
// staged by cp.async into shared memory (double-buffered), each 16-byte chunk
// of a row placed at chunk ^ (row & 7) so the ldmatrix reads of eight rows hit
// eight different bank groups.  The rotated query, scaled by log2(e)/sqrt(d),
// is held as two fp16 parts (hi + lo), so the scores carry the fp32 query;
// the probabilities enter the value product as fp16 (their sum stays fp32).
constexpr int kFQ = 64;        // query tokens per CTA
constexpr int kFK = 64;        // key positions per staged tile
constexpr int kFThreads = 128;

constexpr size_t prefill_smem(int D) { return (size_t)kFQ * D * 4 + (size_t)4 * kFK * D * 2; }

// Byte offset of 16-byte chunk `c` of row `r` in a swizzled [rows][D] fp16 tile.
template <int D>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)(r * D * 2 + ((c ^ (r & 7)) << 4));
}

// 16-byte global -> shared copy; src_bytes 0 fills the chunk with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// c += a * b for one 16x8x16 tile (a: 16x16 row-major fragment, b: 16x8).
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Grid (Hq, ceil(C / 64)), 128 threads; block y takes token block
// ceil(C / 64) - 1 - y.  Token t of the chunk (position
// p0 + t) attends over positions 0..p0 + t of its kv head's cache.
// Fragment layouts (PTX mma.m16n8k16): with g = lane / 4 and u = lane % 4, an
// A register pair covers (row g or g + 8, columns 2u, 2u + 1 or 2u + 8, 2u + 9),
// a B register (rows 2u, 2u + 1 or 2u + 8, 2u + 9, column g), an accumulator
// (row g or g + 8, columns 2u, 2u + 1); the score accumulators of two
// neighbouring 8-key tiles therefore are the A fragment of the probabilities
// for one 16-key step of the value product.
template <int D>
__global__ void __launch_bounds__(kFThreads) prefill_attn_kernel(const uint16_t* __restrict__ q,
                                                                const uint16_t* kc, const uint16_t* vc,
                                                                const int32_t* pos_p, int t0, int C, int Hq,
                                                                int G, int max_seq, const float2* __restrict__ cs,
                                                                uint16_t* __restrict__ a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NCH = D / 8;   // 16-byte chunks per row
    constexpr int KS = D / 16;   // 16-wide steps over the head dimension
    constexpr int DN = D / 8;    // 8-wide output tiles over the head dimension
    constexpr uint32_t TB = kFK * D * 2;
    float* qs = reinterpret_cast<float*>(smem);  // [kFQ][D] rotated, scaled queries
    const uint32_t kv0 = q4d::smem_addr(smem + (size_t)kFQ * D * 4);  // K0 V0 K1 V1
    const int h = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, u = lane & 3;
    const int kvh = h / G;
    const int p0 = *pos_p + t0;
    if (p0 < 0 || p0 + C > max_seq) return;  // latched by the append kernel
    // the last token blocks (the most keys under the causal mask) start first
    const int tq0 = (gridDim.y - 1 - blockIdx.y) * kFQ;
    const int n_keys = p0 + min(tq0 + kFQ, C);  // keys the CTA's last token sees
    const int n_tiles = (n_keys + kFK - 1) / kFK;
    const uint16_t* kh = kc + (size_t)kvh * max_seq * D;
    const uint16_t* vh = vc + (size_t)kvh * max_seq * D;

    // Tile j of keys and values into buffer j & 1; rows past n_keys are zero
    // (stale cache rows could hold anything, and 0 * NaN would reach the sums).
    auto issue = [&](int j) {
        const uint32_t kb = kv0 + (uint32_t)(j & 1) * 2u * TB, vb = kb + TB;
        for (int x = threadIdx.x; x < kFK * NCH; x += kFThreads) {
            const int r = x / NCH, c = x % NCH;
            const int key = j * kFK + r;
            const bool ok = key < n_keys;
            const size_t off = (size_t)(ok ? key : 0) * D + (size_t)c * 8;
            const uint32_t so = swz<D>(r, c);
            cp_async16(kb + so, kh + off, ok ? 16u : 0u);
            cp_async16(vb + so, vh + off, ok ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    issue(0);

    {
        const float scale = rsqrtf((float)D) * 1.4426950408889634f;  // log2(e) / sqrt(d)
        for (int x = threadIdx.x; x < kFQ * (D / 2); x += kFThreads) {
            const int i = x / (D / 2), pr = x % (D / 2);
            float lo = 0.f, hi = 0.f;
            if (tq0 + i < C) {
                const uint16_t* qrow = q + (size_t)(tq0 + i) * Hq * D + (size_t)h * D;
                const float2 r = cs[(size_t)(tq0 + i) * (D / 2) + pr];
                const float l0 = __half2float(__ushort_as_half(qrow[pr]));
                const float h0 = __half2float(__ushort_as_half(qrow[pr + D / 2]));
                lo = (l0 * r.x - h0 * r.y) * scale;
                hi = (h0 * r.x + l0 * r.y) * scale;
            }
            qs[i * D + pr] = lo;
            qs[i * D + pr + D / 2] = hi;
        }
    }
    __syncthreads();
    uint32_t qh[KS][4], ql[KS][4];
    {
        const float* r0 = qs + (warp * 16 + g) * D;
        const float* r1 = r0 + 8 * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int c0 = 16 * kk + 2 * u, c1 = c0 + 8;
            split_h2(r0[c0], r0[c0 + 1], qh[kk][0], ql[kk][0]);
            split_h2(r1[c0], r1[c0 + 1], qh[kk][1], ql[kk][1]);
            split_h2(r0[c1], r0[c1 + 1], qh[kk][2], ql[kk][2]);
            split_h2(r1[c1], r1[c1 + 1], qh[kk][3], ql[kk][3]);
        }
    }

    float o[DN][4];
#pragma unroll
    for (int dn = 0; dn < DN; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int wmin = p0 + tq0 + warp * 16;   // position of the warp's first token
    const int wmax = wmin + 15;
    const int pr0 = wmin + g, pr1 = pr0 + 8;  // positions of this thread's two rows
    const bool wlive = tq0 + warp * 16 < C;

    for (int j = 0; j < n_tiles; ++j) {
        if (j + 1 < n_tiles) {
            issue(j + 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        const uint32_t kb = kv0 + (uint32_t)(j & 1) * 2u * TB, vb = kb + TB;
#pragma unroll
        for (int sub = 0; sub < kFK / 32; ++sub) {
            const int key0 = j * kFK + sub * 32;
            if (!wlive || key0 > wmax) break;  // every key of the rest is masked for this warp
            float sc[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int kk = 0; kk < KS; kk += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(kb + swz<D>(sub * 32 + nt * 8 + (lane & 7), 2 * kk + (lane >> 3)), b0, b1, b2, b3);
                    mma16816(sc[nt], qh[kk], b0, b1);
                    mma16816(sc[nt], ql[kk], b0, b1);
                    mma16816(sc[nt], qh[kk + 1], b2, b3);
                    mma16816(sc[nt], ql[kk + 1], b2, b3);
                }
            }
            if (key0 + 31 > wmin) {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + nt * 8 + 2 * u + (e & 1);
                        if (key > (e < 2 ? pr0 : pr1)) sc[nt][e] = -INFINITY;
                    }
            }
            float x0 = m0, x1 = m1;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                x0 = fmaxf(x0, fmaxf(sc[nt][0], sc[nt][1]));
                x1 = fmaxf(x1, fmaxf(sc[nt][2], sc[nt][3]));
            }
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 1));
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, 2));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 1));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, 2));
            const float s0 = x0 == -INFINITY ? 0.f : x0, s1 = x1 == -INFINITY ? 0.f : x1;
            const float c0 = exp2f(m0 - s0), c1 = exp2f(m1 - s1);  // 0 while nothing was seen
            m0 = x0;
            m1 = x1;
            l0 *= c0;
            l1 *= c1;
#pragma unroll
            for (int dn = 0; dn < DN; ++dn) {
                o[dn][0] *= c0;
                o[dn][1] *= c0;
                o[dn][2] *= c1;
                o[dn][3] *= c1;
            }
            uint32_t pa[2][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const float e0 = exp2f(sc[nt][0] - s0), e1 = exp2f(sc[nt][1] - s0);
                const float e2 = exp2f(sc[nt][2] - s1), e3 = exp2f(sc[nt][3] - s1);
                l0 += e0 + e1;
                l1 += e2 + e3;
                pa[nt >> 1][(nt & 1) * 2 + 0] = pack_h2(e0, e1);
                pa[nt >> 1][(nt & 1) * 2 + 1] = pack_h2(e2, e3);
            }
#pragma unroll
            for (int kj = 0; kj < 2; ++kj) {
#pragma unroll
                for (int dn = 0; dn < DN; dn += 2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(vb + swz<D>(sub * 32 + kj * 16 + (lane & 15), dn + (lane >> 4)), b0, b1, b2, b3);
                    mma16816(o[dn], pa[kj], b0, b1);
                    mma16816(o[dn + 1], pa[kj], b2, b3);
                }
            }
        }
        __syncthreads();  // buffer j & 1 is refilled by the next iteration's issue
    }

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int t_r0 = tq0 + warp * 16 + g;
    if (t_r0 < C) {
        uint16_t* ar = a + (size_t)t_r0 * Hq * D + (size_t)h * D + 2 * u;
#pragma unroll
        for (int dn = 0; dn < DN; ++dn)
            *reinterpret_cast<uint32_t*>(ar + dn * 8) = pack_h2(o[dn][0] / l0, o[dn][1] / l0);
    }
    if (t_r0 + 8 < C) {
        uint16_t* ar = a + (size_t)(t_r0 + 8) * Hq * D + (size_t)h * D + 2 * u;
#pragma unroll
        for (int dn = 0; dn < DN; ++dn)
            *reinterpret_cast<uint32_t*>(ar + dn * 8) = pack_h2(o[dn][2] / l1, o[dn][3] / l1);
    }
}

// ------------------------------------------------ prefill, tcgen05 path ---
// Causal attention of a prompt chunk for head_dim 128 on the 5th-generation
// tensor cores.  A CTA takes one query head and 128 of the chunk's tokens
// (the MMA's M) and walks the keys in tiles of 128 positions (its N):
//   S = Q K^T   two MMA chains per tile (the rotated, scaled query as fp16 hi
//               and lo parts in shared memory, so the scores carry the fp32
//               query; the key tile by TMA, K-major), into one of two score
//               buffers in tensor memory;
//   P           the softmax warps (thread = query row = TMEM lane) read S,
//               mask, take exp2 against the row's reference maximum and write
//               P as fp16 into tensor memory;
//   O += P V    A = P from tensor memory, B = the value tile read MN-major
//               (head_dim contiguous in each position's row), O in tensor
//               memory.
// The MMA thread issues S of tile j before O += P V of tile j - 1, so the
// tensor core computes the next scores while the softmax warps work.  The
// reference maximum moves only when a row's maximum exceeds it by more than
// 8 (a factor 2^8 in exp2); then O and the row sum are rescaled.  P stays
// within 2^8 (fp16 keeps its relative precision at any magnitude) and O / sum
// is the same quotient.  The probabilities enter the value product as fp16;
// their sum stays fp32.
constexpr int kTQ = 128;              // query tokens per CTA (MMA M)
constexpr int kTK = 128;              // key positions per tile (MMA N of the scores)
constexpr int kTThreads = 384;        // warp 0: key tiles, 1: score MMAs, 2: value tiles, 3: value MMAs,
                                      // 4..11: softmax
constexpr uint32_t kTTile = 32768;    // one 128 x 128 fp16 tile: two 64-wide 128-byte-swizzled slabs
constexpr uint32_t kColS = 0;         // TMEM columns: scores 0..127, O 128..255, P 256..319 and
constexpr uint32_t kColO = 128;       //   320..383, the query's hi part 384..447 and lo part 448..511
constexpr uint32_t kColP = 256;       //   (fp16 pairs, the A operand of the score MMAs)
constexpr uint32_t kColQ = 384;

struct TcBars {
    uint64_t q_full, q_tmem, s_free, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2],
        drain;
    uint32_t tmem_base;
    volatile int abort;
    float xmax[2][2][kTQ];  // [tile parity][column half][row]: the halves' row maxima
    float xsum[2][kTQ];     // [column half][row]: the halves' row sums
};

constexpr size_t prefill_tc_smem() { return 1024 + 6 * (size_t)kTTile + sizeof(TcBars); }

// Byte offset of row r, 16-byte chunk c (c < 8) in a 128-byte-swizzled slab.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ bool tc_wait(TcBars& B, uint64_t& bar, uint32_t parity, int* err) {
    if (B.abort) return false;
    if (!q4d::mbar_wait(q4d::smem_addr(&bar), parity, err)) {
        B.abort = 1;
        return false;
    }
    return true;
}

// Grid (Hq, ceil(C / 128)), 384 threads, one CTA per SM (192 KB of shared
// memory, all 512 TMEM columns).  Block y takes token block
// gridDim.y - 1 - y (the blocks with the most keys start first).  tmK / tmV:
// the layer's caches as 2-D maps [Hkv * max_seq][128] fp16, boxes of 64 x 128.
__global__ void __launch_bounds__(kTThreads, 1)
    prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                           const __grid_constant__ CUtensorMap tmQ, const int32_t* pos_p, int t0, int C, int Hq,
                           int G, int max_seq, uint16_t* __restrict__ a, int* err) {
    constexpr int D = 128;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* qh_s = base;                  // query, fp16 hi part (two slabs: head_dim 0..63, 64..127)
    uint8_t* ql_s = base + kTTile;         // the lo part
    uint8_t* k_s = base + 2 * kTTile;      // key tiles, 2 stages
    uint8_t* v_s = base + 4 * kTTile;      // value tiles, 2 stages
    TcBars& B = *reinterpret_cast<TcBars*>(base + 6 * kTTile);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, kvh = h / G;
    const int p0 = *pos_p + t0;
    if (p0 < 0 || p0 + C > max_seq) return;  // latched by the append kernel
    const int tq0 = (gridDim.y - 1 - blockIdx.y) * kTQ;
    const int n_keys = p0 + min(tq0 + kTQ, C);  // keys the block's last token sees
    const int n_tiles = (n_keys + kTK - 1) / kTK;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            q4d::mbar_init(q4d::smem_addr(&B.k_full[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&B.k_empty[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&B.v_full[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&B.v_empty[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&B.s_full[i]), 1);
            q4d::mbar_init(q4d::smem_addr(&B.p_full[i]), 8);  // the softmax warps
            q4d::mbar_init(q4d::smem_addr(&B.pv_done[i]), 1);
        }
        q4d::mbar_init(q4d::smem_addr(&B.drain), 2);  // both issuers' last MMAs
        q4d::mbar_init(q4d::smem_addr(&B.q_full), 1);
        q4d::mbar_init(q4d::smem_addr(&B.q_tmem), 8);  // the softmax warps copied the query into TMEM
        q4d::mbar_init(q4d::smem_addr(&B.s_free), 8);  // the softmax warps have read the scores
        B.abort = 0;
        q4d::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         q4d::smem_addr(&B.tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Key (warp 0) or value (warp 2) tile j into stage j % 2, by lane 0.
    auto issue_tile = [&](int j) {
        const bool keys = warp == 0;
        const int st = j & 1;
        const uint32_t fb = q4d::smem_addr(keys ? &B.k_full[st] : &B.v_full[st]);
        uint8_t* dst = (keys ? k_s : v_s) + st * kTTile;
        q4d::mbar_arrive_expect_tx(fb, kTTile);
        const int y = kvh * max_seq + j * kTK;
        q4t::tma_load_2d(q4d::smem_addr(dst), keys ? &tmK : &tmV, 0, y, fb);
        q4t::tma_load_2d(q4d::smem_addr(dst + 16384), keys ? &tmK : &tmV, 64, y, fb);
    };
    __syncthreads();  // barriers initialised
    if (warp == 0 && lane == 0) {
        // the block's queries: hi and lo parts, two slabs each (rows past C
        // read the next head's rows or zeros; those rows are never stored)
        const uint32_t qb = q4d::smem_addr(&B.q_full);
        q4d::mbar_arrive_expect_tx(qb, 2 * kTTile);
        const int yh = h * C + tq0, yl = Hq * C + h * C + tq0;
        q4t::tma_load_2d(q4d::smem_addr(qh_s), &tmQ, 0, yh, qb);
        q4t::tma_load_2d(q4d::smem_addr(qh_s + 16384), &tmQ, 64, yh, qb);
        q4t::tma_load_2d(q4d::smem_addr(ql_s), &tmQ, 0, yl, qb);
        q4t::tma_load_2d(q4d::smem_addr(ql_s + 16384), &tmQ, 64, yl, qb);
    }
    if ((warp == 0 || warp == 2) && lane == 0)
        for (int j = 0; j < n_tiles && j < 2; ++j) issue_tile(j);
    q4t::fence_before();
    __syncthreads();
    q4t::fence_after();
    const uint32_t tmem = B.tmem_base;

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------ key / value tiles
        if (lane == 0) {
            uint64_t* full = warp == 0 ? B.k_full : B.v_full;
            uint64_t* empty = warp == 0 ? B.k_empty : B.v_empty;
            int j = 2;
            for (; j < n_tiles; ++j) {
                if (!tc_wait(B, empty[j & 1], ((j - 2) >> 1) & 1, err)) break;
                issue_tile(j);
            }
            if (B.abort) {
                // copies still in flight land before the CTA can exit
                if (warp == 0) q4d::mbar_wait(q4d::smem_addr(&B.q_full), 0, nullptr);
                const int issued = j < n_tiles ? j : n_tiles;
                for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
                    q4d::mbar_wait(q4d::smem_addr(&full[i & 1]), (i >> 1) & 1, nullptr);
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ------------------------------------------------ MMA issue
        // Two issuing threads (one tcgen05.mma takes ~40 ns to issue from a
        // thread): warp 1 the scores of every tile, warp 3 the value products.
        if (lane == 0) {
            const uint32_t id_s = q4t::idesc_f16_m128(kTK, 0), id_o = q4t::idesc_f16_m128(D, 1);
            // every descriptor is a base plus a constant start-address step
            // (16-byte units; the fields never carry: the tiles sit below
            // 256 KB), computed once
            bool ok = true;
            if (warp == 1) {
                const uint64_t dk0 = q4t::sw128_desc(q4d::smem_addr(k_s), 16, 1024);
                const uint64_t dk1 = q4t::sw128_desc(q4d::smem_addr(k_s + kTTile), 16, 1024);
                ok = tc_wait(B, B.q_tmem, 0, err);
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int st = j & 1;
                    if (!tc_wait(B, B.k_full[st], (j >> 1) & 1, err)) {
                        ok = false;
                        break;
                    }
                    // the score buffer is free once the softmax warps have read S_{j-1}
                    if (j >= 1 && !tc_wait(B, B.s_free, (j - 1) & 1, err)) {
                        ok = false;
                        break;
                    }
                    q4t::fence_after();
                    const uint64_t kd = st ? dk1 : dk0;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            // A: 16 head_dim = 8 TMEM columns of the query part; B: 32
                            // bytes within a 64-wide slab of the key tile, slabs 16 KB apart
                            const uint64_t off = (uint64_t)(((kk >> 2) * 16384 + (kk & 3) * 32) / 16);
                            q4t::mma_ts(tmem + kColS, tmem + kColQ + part * 64 + 8 * kk, kd + off, id_s,
                                        (part > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    q4t::commit(q4d::smem_addr(&B.k_empty[st]));
                    q4t::commit(q4d::smem_addr(&B.s_full[st]));
                }
            } else {
                const uint64_t dv0 = q4t::sw128_desc(q4d::smem_addr(v_s), 16384, 1024);
                const uint64_t dv1 = q4t::sw128_desc(q4d::smem_addr(v_s + kTTile), 16384, 1024);
                // O += P_i V_i (A = P from tensor memory, B = the value tile MN-major)
                for (int i = 0; i < n_tiles && ok; ++i) {
                    const int st = i & 1;
                    if (!tc_wait(B, B.p_full[st], (i >> 1) & 1, err) ||
                        !tc_wait(B, B.v_full[st], (i >> 1) & 1, err)) {
                        ok = false;
                        break;
                    }
                    q4t::fence_after();
                    const uint64_t vd = st ? dv1 : dv0;
                    const uint32_t pa = tmem + kColP + st * 64;
                    q4t::mma_ts(tmem + kColO, pa, vd, id_o, i > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 1; kk < kTK / 16; ++kk)  // 16 positions = 2048 bytes of the value tile
                        q4t::mma_ts(tmem + kColO, pa + 8 * kk, vd + (uint64_t)(kk * 2048 / 16), id_o, 1u);
                    q4t::commit(q4d::smem_addr(&B.v_empty[st]));
                    q4t::commit(q4d::smem_addr(&B.pv_done[st]));
                }
            }
            if (!ok) B.abort = 1;
            // every MMA this thread issued has finished before the CTA winds down
            q4t::commit(q4d::smem_addr(&B.drain));
            q4d::mbar_wait(q4d::smem_addr(&B.drain), 0, nullptr);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ softmax
        // Two warps per TMEM lane quarter: warp 4 + q takes score columns
        // 0..63 of rows 32 q .. 32 q + 31 (and O columns 0..63), warp 8 + q
        // columns 64..127; the pair meets on named barrier 1 + q to share
        // each tile's row maxima and, at the end, the row sums.
        const int sw = warp - 4;
        const int qw = sw & 3;                    // TMEM lane quarter (= warp % 4)
        const int hf = sw >> 2;                   // which half of the columns
        const int row = qw * 32 + lane;           // query row = TMEM lane
        const int pq = p0 + tq0 + row;            // its position
        const uint32_t lt = tmem + ((uint32_t)(qw * 32) << 16);
        const uint32_t pair_bar = 1 + qw;
        float m_ref = -INFINITY, l = 0.f;
        {
            // the query's part hf (0: hi, 1: lo) of this row into TMEM columns
            // kColQ + 64 hf ..: the slabs' 16-byte chunks hold 8 consecutive
            // head_dim values, i.e. 4 columns of fp16 pairs in order
            bool qbad = __any_sync(0xffffffffu, !tc_wait(B, B.q_full, 0, err));
            if (!qbad) {
                const uint8_t* qs = hf ? ql_s : qh_s;
                uint32_t qv[64];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4*>(qs + (c >> 3) * 16384 + sw_off(row, c & 7));
                    qv[4 * c] = w.x;
                    qv[4 * c + 1] = w.y;
                    qv[4 * c + 2] = w.z;
                    qv[4 * c + 3] = w.w;
                }
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) q4t::st16(lt + kColQ + hf * 64 + c0, qv + c0);
                q4t::st_wait();
                q4t::fence_before();
                __syncwarp();
                if (lane == 0) q4d::mbar_arrive(q4d::smem_addr(&B.q_tmem));
            }
        }
        // `bad` (a failed or skipped wait) is made warp-uniform after every
        // wait and pair-uniform at the pair's barrier, which both warps reach
        // once per tile: they leave the loop together, so neither waits on the
        // named barrier for a partner that has left
        bool bad = false;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            bad = __any_sync(0xffffffffu, bad || !tc_wait(B, B.s_full[st], (j >> 1) & 1, err));
            const int key0 = j * kTK + hf * (kTK / 2);  // key of this thread's first column
            const bool mask = j * kTK + kTK - 1 > p0 + tq0;  // some key of the tile above some row's position
            uint32_t r[kTK / 2];
            float mh = -INFINITY;
            if (!bad) {
                q4t::fence_after();
#pragma unroll
                for (int c0 = 0; c0 < kTK / 2; c0 += 16) q4t::ld16(lt + kColS + hf * (kTK / 2) + c0, r + c0);
                q4t::ld_wait();
                // the scores are in registers: the MMA may write the next tile's
                q4t::fence_before();
                __syncwarp();
                if (lane == 0) q4d::mbar_arrive(q4d::smem_addr(&B.s_free));
                if (mask) {
#pragma unroll
                    for (int e = 0; e < kTK / 2; ++e)
                        if (key0 + e > pq) r[e] = __float_as_uint(-INFINITY);
                }
#pragma unroll
                for (int e = 0; e < kTK / 2; ++e) mh = fmaxf(mh, __uint_as_float(r[e]));
            }
            B.xmax[st][hf][row] = mh;
            bad = q4d::named_bar_or(pair_bar, 64, bad);
            if (bad) break;
            const float mx = fmaxf(B.xmax[st][0][row], B.xmax[st][1][row]);
            float corr = 1.f;
            bool resc = false;
            if (mx > m_ref + 8.f) {
                if (m_ref != -INFINITY) {
                    corr = exp2f(m_ref - mx);
                    resc = true;
                }
                m_ref = mx;
            }
            const float msub = m_ref == -INFINITY ? 0.f : m_ref;
            // P = exp2(s - m_ref) as fp16 pairs, packed in place (pair i
            // into r[i], whose own score was read for pair i / 2)
            float sum = 0.f;
#pragma unroll
            for (int i2 = 0; i2 < kTK / 4; ++i2) {
                const float e0 = exp2f(__uint_as_float(r[2 * i2]) - msub);
                const float e1 = exp2f(__uint_as_float(r[2 * i2 + 1]) - msub);
                sum += e0 + e1;
                r[i2] = pack_h2(e0, e1);
            }
            l = l * corr + sum;
            // P buffer st was read by O += P V of tile j - 2, and O is written
            // by that of tile j - 1
            if (j >= 2) bad = __any_sync(0xffffffffu, !tc_wait(B, B.pv_done[st], ((j - 2) >> 1) & 1, err));
            if (j >= 1 && !bad) bad = __any_sync(0xffffffffu, !tc_wait(B, B.pv_done[st ^ 1], ((j - 1) >> 1) & 1, err));
            const bool zero_tail = j == n_tiles - 1 && (n_keys & (kTK - 1));
            if (zero_tail && !bad) bad = __any_sync(0xffffffffu, !tc_wait(B, B.v_full[st], (j >> 1) & 1, err));
            if (bad) continue;  // to the pair's barrier of the next tile (or past the loop)
            q4t::fence_after();
            if (__any_sync(0xffffffffu, resc)) {  // the TMEM load / store is warp-collective
                uint32_t o[D / 2];
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 16) q4t::ld16(lt + kColO + hf * (D / 2) + c0, o + c0);
                q4t::ld_wait();
#pragma unroll
                for (int e = 0; e < D / 2; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * corr);
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 16) q4t::st16(lt + kColO + hf * (D / 2) + c0, o + c0);
            }
#pragma unroll
            for (int c = 0; c < kTK / 4; c += 16) q4t::st16(lt + kColP + st * 64 + hf * (kTK / 4) + c, r + c);
            q4t::st_wait();
            if (zero_tail) {
                // the last tile's value rows past n_keys: stale cache rows may
                // hold anything, and 0 * NaN would reach O; zero them (this
                // thread: its row's slab hf)
                if (row >= n_keys - j * kTK) {
                    uint8_t* vt = v_s + st * kTTile + hf * 16384;
#pragma unroll
                    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vt + sw_off(row, c)) = make_uint4(0, 0, 0, 0);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            q4t::fence_before();
            __syncwarp();
            if (lane == 0) q4d::mbar_arrive(q4d::smem_addr(&B.p_full[st]));
        }
        // the row sum of both halves (both warps of the pair reach this barrier)
        B.xsum[hf][row] = l;
        bad = q4d::named_bar_or(pair_bar, 64, bad);
        if (!bad) {
            const int last = n_tiles - 1;
            if (tc_wait(B, B.pv_done[last & 1], (last >> 1) & 1, err)) {
                q4t::fence_after();
                const float inv = 1.0f / (B.xsum[0][row] + B.xsum[1][row]);
                uint16_t* ar = a + (size_t)(tq0 + row) * Hq * D + (size_t)h * D + hf * (D / 2);
                const bool live = tq0 + row < C;
                uint32_t ro[D / 2];
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 16) q4t::ld16(lt + kColO + hf * (D / 2) + c0, ro + c0);
                q4t::ld_wait();
#pragma unroll
                for (int c0 = 0; c0 < D / 2; c0 += 16) {
                    const uint32_t* rr = ro + c0;
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        o[e] = pack_h2(__uint_as_float(rr[2 * e]) * inv, __uint_as_float(rr[2 * e + 1]) * inv);
                    if (live) {
                        *reinterpret_cast<uint4*>(ar + c0) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(ar + c0 + 8) = make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
            }
        }
    }
    q4t::fence_before();
    __syncthreads();
    if (warp == 1) {
        q4t::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

}  // namespace q4a

namespace q4i {

// Workspace: the step's (cos, sin) table, then (max, sum) per head and chunk,
// then the chunks' partial outputs; each part 256-byte aligned.
size_t attn_workspace_bytes(int n_q_heads, int head_dim, int max_seq) {
    const size_t ns = (size_t)(max_seq + q4a::kChunk - 1) / q4a::kChunk;
    const size_t ml = (size_t)n_q_heads * ns * 2 * 4;
    return 256 * (((size_t)head_dim / 2 * 8 + 255) / 256) + ((ml + 255) & ~size_t(255)) +
           (size_t)n_q_heads * ns * head_dim * 4;
}

q4_status attn_validate(const q4_attention_desc& d) {
    if (!d.q || !d.k || !d.v || !d.k_cache || !d.v_cache || !d.pos || !d.a || !d.workspace)
        return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (d.head_dim != 64 && d.head_dim != 128) return fail(Q4_ERR_UNSUPPORTED, "head_dim=%d (64 or 128)", d.head_dim);
    if (d.n_kv_heads < 1 || d.n_q_heads < d.n_kv_heads || d.n_q_heads % d.n_kv_heads)
        return fail(Q4_ERR_INVALID_ARG, "n_q_heads=%d is not a multiple of n_kv_heads=%d", d.n_q_heads, d.n_kv_heads);
    if (d.n_q_heads / d.n_kv_heads > q4a::kMaxGroup)
        return fail(Q4_ERR_UNSUPPORTED, "more than %d query heads per kv head", q4a::kMaxGroup);
    if (d.max_seq < 1) return fail(Q4_ERR_INVALID_ARG, "max_seq=%d", d.max_seq);
    if (d.max_seq > q4a::kMaxLive * q4a::kChunk)
        return fail(Q4_ERR_UNSUPPORTED, "max_seq=%d above %d", d.max_seq, q4a::kMaxLive * q4a::kChunk);
    if (!(d.rope_theta > 1.0f)) return fail(Q4_ERR_INVALID_ARG, "rope_theta must be > 1");
    if ((reinterpret_cast<uintptr_t>(d.k_cache) & 15u) || (reinterpret_cast<uintptr_t>(d.v_cache) & 15u) ||
        (reinterpret_cast<uintptr_t>(d.workspace) & 255u))
        return fail(Q4_ERR_MISALIGNED, "caches must be 16-byte and the workspace 256-byte aligned");
    if (d.workspace_bytes < attn_workspace_bytes(d.n_q_heads, d.head_dim, d.max_seq))
        return fail(Q4_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", d.workspace_bytes,
                    attn_workspace_bytes(d.n_q_heads, d.head_dim, d.max_seq));
    return Q4_OK;
}

q4_status attn_enqueue(const q4_attention_desc& d, cudaStream_t s, bool compute_table) {
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    const int D = d.head_dim, G = d.n_q_heads / d.n_kv_heads;
    const int ns = (d.max_seq + q4a::kChunk - 1) / q4a::kChunk;
    const double l2t = log2((double)d.rope_theta);
    uint8_t* w = static_cast<uint8_t*>(d.workspace);
    float2* cs = reinterpret_cast<float2*>(w);
    float* ml = reinterpret_cast<float*>(w + 256 * (((size_t)D / 2 * 8 + 255) / 256));
    float* acc = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ml) +
                                          (((size_t)d.n_q_heads * ns * 2 * 4 + 255) & ~size_t(255)));
    // The first attention of a step computes the cos/sin table in its append
    // kernel; later ones append inside the split kernel (one launch fewer).
    if (compute_table)
        q4a::rope_append_kernel<true><<<d.n_kv_heads, D / 2, 0, s>>>(d.k, d.v, d.k_cache, d.v_cache, d.pos, D,
                                                                      d.max_seq, l2t, cs, dev->err_word);
    const uint16_t* k_new = compute_table ? nullptr : d.k;
    static std::atomic<int> marks128[64], marks64[64];
    const cudaError_t ea =
        D == 128 ? ensure_smem_attr(reinterpret_cast<const void*>(q4a::attn_split_kernel<128>), marks128,
                                    (int)q4a::split_smem(128))
                 : ensure_smem_attr(reinterpret_cast<const void*>(q4a::attn_split_kernel<64>), marks64,
                                    (int)q4a::split_smem(64));
    if (ea != cudaSuccess) return cuda_fail(ea, "cudaFuncSetAttribute(attn_split_kernel)");
    const dim3 grid(d.n_kv_heads, ns);
    if (D == 128)
        q4a::attn_split_kernel<128><<<grid, q4a::kThreads, q4a::split_smem(128), s>>>(
            d.q, d.k_cache, d.v_cache, d.pos, G, d.max_seq, ns, cs, ml, acc, k_new, d.v, d.k_cache, d.v_cache,
            dev->err_word);
    else
        q4a::attn_split_kernel<64><<<grid, q4a::kThreads, q4a::split_smem(64), s>>>(
            d.q, d.k_cache, d.v_cache, d.pos, G, d.max_seq, ns, cs, ml, acc, k_new, d.v, d.k_cache, d.v_cache,
            dev->err_word);
    q4a::attn_combine_kernel<<<d.n_q_heads, D, 0, s>>>(ml, acc, d.pos, D, d.max_seq, ns, d.a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return Q4_OK;
}

// The chunk's rotation table, then (head_dim 128) the rotated query's hi / lo
// parts for the tensor-core attention.
static size_t cs_table_bytes(int chunk, int head_dim) { return ((size_t)chunk * head_dim / 2 * 8 + 255) & ~size_t(255); }

size_t prefill_attn_cs_bytes(int chunk, int head_dim, int n_q_heads) {
    return cs_table_bytes(chunk, head_dim) + (head_dim == 128 ? 2 * (size_t)n_q_heads * chunk * head_dim * 2 : 0);
}

q4_status prefill_attn_table(const int32_t* pos, int t0, int C, int head_dim, float theta, void* cs, cudaStream_t s) {
    q4a::prefill_cs_kernel<<<C, head_dim / 2, 0, s>>>(pos, t0, head_dim, log2((double)theta),
                                                      static_cast<float2*>(cs));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill rotation table launch");
    return Q4_OK;
}

q4_status prefill_attn_enqueue(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* k_cache,
                               uint16_t* v_cache, const int32_t* pos, int t0, int C, int Hq, int Hkv, int D,
                               int max_seq, void* cs, uint16_t* a, cudaStream_t s) {
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    const float2* csp = static_cast<const float2*>(cs);
    // head_dim 128: the rotated query's hi / lo parts [2][Hq][C][128] after
    // the rotation table (prefill_attn_cs_bytes sized the region for both)
    uint16_t* qrot = D == 128 ? reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(cs) + cs_table_bytes(C, D)) : nullptr;
    q4a::prefill_append_kernel<<<C, 256, 0, s>>>(k, v, k_cache, v_cache, pos, t0, C, Hkv, D, max_seq, csp, q, Hq,
                                                 qrot, dev->err_word);
    cudaError_t e;
    if (D == 128) {
        // tcgen05 path: the caches as 2-D maps [Hkv * max_seq][128], boxes of
        // 64 head_dim x 128 positions with the 128-byte swizzle
        CUtensorMap tmK, tmV, tmQ;
        const uint64_t rows = (uint64_t)Hkv * (uint64_t)max_seq;
        if ((st = make_map(&tmQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qrot, 128, 2 * (uint64_t)Hq * (uint64_t)C, 256, 64,
                           q4a::kTQ, CU_TENSOR_MAP_SWIZZLE_128B)) != Q4_OK)
            return st;
        if ((st = make_map(&tmK, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, k_cache, 128, rows, 256, 64, q4a::kTK,
                           CU_TENSOR_MAP_SWIZZLE_128B)) != Q4_OK)
            return st;
        if ((st = make_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, v_cache, 128, rows, 256, 64, q4a::kTK,
                           CU_TENSOR_MAP_SWIZZLE_128B)) != Q4_OK)
            return st;
        static std::atomic<int> marks_tc[64];
        e = ensure_smem_attr(reinterpret_cast<const void*>(q4a::prefill_attn_tc_kernel), marks_tc,
                             (int)q4a::prefill_tc_smem());
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_attn_tc_kernel)");
        const dim3 grid(Hq, (C + q4a::kTQ - 1) / q4a::kTQ);
        q4a::prefill_attn_tc_kernel<<<grid, q4a::kTThreads, q4a::prefill_tc_smem(), s>>>(
            tmK, tmV, tmQ, pos, t0, C, Hq, Hq / Hkv, max_seq, a, dev->err_word);
    } else {
        static std::atomic<int> marks64[64];
        e = ensure_smem_attr(reinterpret_cast<const void*>(q4a::prefill_attn_kernel<64>), marks64,
                             (int)q4a::prefill_smem(64));
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill_attn_kernel)");
        const dim3 grid(Hq, (C + q4a::kFQ - 1) / q4a::kFQ);
        q4a::prefill_attn_kernel<64><<<grid, q4a::kFThreads, q4a::prefill_smem(64), s>>>(
            q, k_cache, v_cache, pos, t0, C, Hq, Hq / Hkv, max_seq, csp, a);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "prefill attention launch");
    return Q4_OK;
}

q4_status pos_advance(int32_t* pos, cudaStream_t s, int by) {
    q4a::pos_advance_kernel<<<1, 1, 0, s>>>(pos, by);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "position advance launch");
    return Q4_OK;
}

}  // namespace q4i

using namespace q4i;

extern "C" size_t q4_attention_workspace_bytes(int n_q_heads, int head_dim, int max_seq) {
    if (n_q_heads < 1 || head_dim < 1 || max_seq < 1) return 0;
    return attn_workspace_bytes(n_q_heads, head_dim, max_seq);
}

extern "C" q4_status q4_attention(const q4_attention_desc* desc, q4_stream_t stream) {
    clear_error();
    if (!desc) return fail(Q4_ERR_INVALID_ARG, "desc is NULL");
    q4_status st = attn_validate(*desc);
    if (st != Q4_OK) return st;
    return attn_enqueue(*desc, reinterpret_cast<cudaStream_t>(stream), true);
}
