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
// (flash-decoding): one CTA per (kv head, chunk of 256 positions) scores all
// query heads of the group against the chunk's keys (a warp per position,
// lanes across d, 8-byte loads), turns the scores into exp(s - max) in shared
// memory, and accumulates the values (a thread per dimension, coalesced 2-byte
// loads); a second kernel merges the chunks' (max, sum, partial output) per
// head.  The rotation angle pos * theta^(-2i/d) and its sine and cosine are
// computed in fp64 (a few operations per pair), the rotation itself in fp32.
#include <cuda_fp16.h>
#include <math.h>

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4a {

constexpr int kChunk = 256;   // positions per CTA
constexpr int kThreads = 128;
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
// Grid Hkv, block d/2: thread i turns the pair (i, i + d/2).
__global__ void rope_append_kernel(const uint16_t* __restrict__ k, const uint16_t* __restrict__ v,
                                   uint16_t* __restrict__ kc, uint16_t* __restrict__ vc, const int32_t* pos_p, int d,
                                   int max_seq, double log2_theta, int* err) {
    const int h = blockIdx.x, i = threadIdx.x, half = d / 2;
    const int pos = *pos_p;
    if (!pos_ok(pos, max_seq, err)) return;
    float c, s;
    rope_cs(pos, i, d, log2_theta, c, s);
    const float lo = __half2float(__ushort_as_half(k[h * d + i]));
    const float hi = __half2float(__ushort_as_half(k[h * d + i + half]));
    const size_t base = ((size_t)h * max_seq + pos) * d;
    kc[base + i] = __half_as_ushort(__float2half_rn(lo * c - hi * s));
    kc[base + i + half] = __half_as_ushort(__float2half_rn(hi * c + lo * s));
    vc[base + i] = v[h * d + i];
    vc[base + i + half] = v[h * d + i + half];
}

// One (kv head, chunk) of the attention: for each query head g of the group,
// m = max score, l = sum exp(s - m), acc = sum exp(s - m) v over the chunk.
template <int D>
__global__ void __launch_bounds__(kThreads) attn_split_kernel(const uint16_t* __restrict__ q,
                                                              const uint16_t* __restrict__ kc,
                                                              const uint16_t* __restrict__ vc, const int32_t* pos_p,
                                                              int G, int max_seq, int n_splits, double log2_theta,
                                                              float* __restrict__ part_ml,
                                                              float* __restrict__ part_acc, int* err) {
    __shared__ float qr[kMaxGroup][D];
    __shared__ float sc[kMaxGroup][kChunk];
    const int kvh = blockIdx.x, split = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pos = *pos_p;
    if (!pos_ok(pos, max_seq, err)) return;
    const int n = pos + 1, j0 = split * kChunk, j1 = min(j0 + kChunk, n), cnt = j1 - j0;
    const int h0 = kvh * G;
    if (cnt <= 0) return;  // past the context: the combine step reads only the live chunks
    // rotated queries, scaled by 1/sqrt(d)
    const float scale = rsqrtf((float)D);
    for (int t = tid; t < G * (D / 2); t += kThreads) {
        const int g = t / (D / 2), i = t % (D / 2);
        float c, s;
        rope_cs(pos, i, D, log2_theta, c, s);
        const float lo = __half2float(__ushort_as_half(q[(h0 + g) * D + i]));
        const float hi = __half2float(__ushort_as_half(q[(h0 + g) * D + i + D / 2]));
        qr[g][i] = (lo * c - hi * s) * scale;
        qr[g][i + D / 2] = (hi * c + lo * s) * scale;
    }
    __syncthreads();
    // scores: a warp per position, lanes across d
    constexpr int E = D / 32;  // elements per lane (2 or 4)
    const uint16_t* kbase = kc + (size_t)kvh * max_seq * D;
    for (int j = j0 + warp; j < j1; j += kThreads / 32) {
        float kf[E];
        if constexpr (E == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(kbase + (size_t)j * D + lane * 4);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            kf[0] = a.x; kf[1] = a.y; kf[2] = b.x; kf[3] = b.y;
        } else {
            const uint32_t raw = *reinterpret_cast<const uint32_t*>(kbase + (size_t)j * D + lane * 2);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw));
            kf[0] = a.x; kf[1] = a.y;
        }
        for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc = fmaf(qr[g][lane * E + e], kf[e], acc);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
            if (lane == 0) sc[g][j - j0] = acc;
        }
    }
    __syncthreads();
    // per head: max, exp, sum (a warp per head)
    for (int g = warp; g < G; g += kThreads / 32) {
        float m = -INFINITY;
        for (int j = lane; j < cnt; j += 32) m = fmaxf(m, sc[g][j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int j = lane; j < cnt; j += 32) {
            const float p = expf(sc[g][j] - m);
            sc[g][j] = p;
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
    // values: a thread per dimension
    if (tid < D) {
        float acc[kMaxGroup];
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) acc[g] = 0.f;
        const uint16_t* vb = vc + (size_t)kvh * max_seq * D + (size_t)j0 * D + tid;
        for (int j = 0; j < cnt; ++j) {
            const float vv = __half2float(__ushort_as_half(vb[(size_t)j * D]));
#pragma unroll
            for (int g = 0; g < kMaxGroup; ++g)
                if (g < G) acc[g] = fmaf(sc[g][j], vv, acc[g]);
        }
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g)
            if (g < G) part_acc[((size_t)(h0 + g) * n_splits + split) * D + tid] = acc[g];
    }
}

// a[h] = sum_s acc_s e^(m_s - M) / sum_s l_s e^(m_s - M) over the live chunks.
__global__ void attn_combine_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_acc,
                                    const int32_t* pos_p, int d, int max_seq, int n_splits,
                                    uint16_t* __restrict__ a) {
    const int h = blockIdx.x, t = threadIdx.x;
    const int pos = *pos_p;
    if (pos < 0 || pos >= max_seq) return;  // latched by the split kernel
    const int live = pos / kChunk + 1;
    const float* ml = part_ml + (size_t)h * n_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < live; ++s) M = fmaxf(M, ml[2 * s]);
    float L = 0.f, acc = 0.f;
    for (int s = 0; s < live; ++s) {
        const float w = expf(ml[2 * s] - M);
        L = fmaf(ml[2 * s + 1], w, L);
        acc = fmaf(part_acc[((size_t)h * n_splits + s) * d + t], w, acc);
    }
    a[h * d + t] = __half_as_ushort(__float2half_rn(acc / L));
}

__global__ void pos_advance_kernel(int32_t* pos_p) { *pos_p += 1; }

}  // namespace q4a

namespace q4i {

size_t attn_workspace_bytes(int n_q_heads, int head_dim, int max_seq) {
    const size_t ns = (size_t)(max_seq + q4a::kChunk - 1) / q4a::kChunk;
    const size_t ml = (size_t)n_q_heads * ns * 2 * 4;
    return ((ml + 255) & ~size_t(255)) + (size_t)n_q_heads * ns * head_dim * 4;
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
    if (!(d.rope_theta > 1.0f)) return fail(Q4_ERR_INVALID_ARG, "rope_theta must be > 1");
    if ((reinterpret_cast<uintptr_t>(d.k_cache) & 15u) || (reinterpret_cast<uintptr_t>(d.v_cache) & 15u) ||
        (reinterpret_cast<uintptr_t>(d.workspace) & 255u))
        return fail(Q4_ERR_MISALIGNED, "caches must be 16-byte and the workspace 256-byte aligned");
    if (d.workspace_bytes < attn_workspace_bytes(d.n_q_heads, d.head_dim, d.max_seq))
        return fail(Q4_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", d.workspace_bytes,
                    attn_workspace_bytes(d.n_q_heads, d.head_dim, d.max_seq));
    return Q4_OK;
}

q4_status attn_enqueue(const q4_attention_desc& d, cudaStream_t s) {
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    const int D = d.head_dim, G = d.n_q_heads / d.n_kv_heads;
    const int ns = (d.max_seq + q4a::kChunk - 1) / q4a::kChunk;
    const double l2t = log2((double)d.rope_theta);
    float* ml = static_cast<float*>(d.workspace);
    float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(d.workspace) +
                                          (((size_t)d.n_q_heads * ns * 2 * 4 + 255) & ~size_t(255)));
    q4a::rope_append_kernel<<<d.n_kv_heads, D / 2, 0, s>>>(d.k, d.v, d.k_cache, d.v_cache, d.pos, D, d.max_seq, l2t,
                                                            dev->err_word);
    const dim3 grid(d.n_kv_heads, ns);
    if (D == 128)
        q4a::attn_split_kernel<128><<<grid, q4a::kThreads, 0, s>>>(d.q, d.k_cache, d.v_cache, d.pos, G, d.max_seq, ns,
                                                                   l2t, ml, acc, dev->err_word);
    else
        q4a::attn_split_kernel<64><<<grid, q4a::kThreads, 0, s>>>(d.q, d.k_cache, d.v_cache, d.pos, G, d.max_seq, ns,
                                                                  l2t, ml, acc, dev->err_word);
    q4a::attn_combine_kernel<<<d.n_q_heads, D, 0, s>>>(ml, acc, d.pos, D, d.max_seq, ns, d.a);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    return Q4_OK;
}

q4_status pos_advance(int32_t* pos, cudaStream_t s) {
    q4a::pos_advance_kernel<<<1, 1, 0, s>>>(pos);
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
    return attn_enqueue(*desc, reinterpret_cast<cudaStream_t>(stream));
}
