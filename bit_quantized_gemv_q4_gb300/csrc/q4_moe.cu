// MoE prefill around the grouped GEMM: routing, gather of token rows into
// expert order, and the weighted combine.
//
// BaseRT: optimal LLM inference on Apple Silicon with native Metal, abstract
// and Fig. 1: MoE prefill on a Qwen3-30B-A3B-shaped model is where BaseRT's
// lead is largest.  The page does not describe routing; this library takes
//   * top-k of the fp16 router logits per token, ties to the lower expert;
//   * weights = softmax over the k chosen logits (fp32);
//   * rows sorted stably by (expert, token, rank); a token holds an expert at
//     most once, so (expert, token) already orders every row;
//   * out[t] = sum over ranks k of w[t][k] * Y[pos[t][k]], fp32, k in order.
// All integer outputs are deterministic (no atomics decide an order).
#include <cuda_fp16.h>

#include <mutex>

#include "q4_device.cuh"
#include "q4_internal.h"

namespace q4m {

constexpr int kMaxTopk = 8;
constexpr int kMaxExperts = 256;
constexpr int kBlockTokens = 32;  // tokens per counting block (one warp per token)
// Largest token count either routing entry point accepts: keeps every index
// the kernels form (token, block * experts, rows = tokens * topk) inside int.
constexpr int kMaxRouteTokens = 1 << 24;

// Order-preserving 16-bit key of an fp16 value (-0 folded onto +0).
__device__ __forceinline__ uint32_t half_key(uint16_t h) {
    if (h == 0x8000u) h = 0;
    return (h & 0x8000u) ? (uint32_t)(~h & 0xFFFFu) : (uint32_t)(h | 0x8000u);
}

// One warp per token: top-k by repeated warp arg-max over (key, -expert).
// Launched with kBlockTokens warps a block: the block also counts its
// tokens' experts into count[e * B + b] (the histogram route_scan_kernel
// turns into offsets), so no separate counting launch.
__global__ void __launch_bounds__(32 * kBlockTokens)
    route_topk_kernel(const uint16_t* __restrict__ logits, int T, int E, int topk, int32_t* __restrict__ ids,
                      float* __restrict__ wts, int B, int32_t* __restrict__ count) {
    __shared__ int32_t c[kMaxExperts];
    for (int e = threadIdx.x; e < E; e += blockDim.x) c[e] = 0;
    __syncthreads();
    const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (gw < T) {
    const int warp = (int)gw;
    const uint16_t* row = logits + (size_t)warp * E;
    constexpr int kPer = kMaxExperts / 32;
    uint32_t key[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        key[i] = e < E ? ((half_key(row[e]) << 16) | (uint32_t)(0xFFFF - e)) : 0u;
    }
    uint32_t chosen[kMaxTopk];
    for (int k = 0; k < topk; ++k) {
        uint32_t best = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) best = key[i] > best ? key[i] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint32_t other = __shfl_xor_sync(0xffffffffu, best, o);
            best = other > best ? other : best;
        }
        chosen[k] = best;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if (key[i] == best) key[i] = 0;
    }
    if (lane == 0) {
        float l[kMaxTopk];
        float mx = -INFINITY;
        for (int k = 0; k < topk; ++k) {
            const int e = 0xFFFF - (int)(chosen[k] & 0xFFFFu);
            ids[(size_t)warp * topk + k] = e;
            l[k] = __half2float(__ushort_as_half(row[e]));
            mx = fmaxf(mx, l[k]);
        }
        float sum = 0.f;
        for (int k = 0; k < topk; ++k) {
            l[k] = expf(l[k] - mx);
            sum += l[k];
        }
        for (int k = 0; k < topk; ++k) wts[(size_t)warp * topk + k] = l[k] / sum;
        for (int k = 0; k < topk; ++k) atomicAdd(&c[0xFFFF - (int)(chosen[k] & 0xFFFFu)], 1);
    }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) count[(size_t)e * B + blockIdx.x] = c[e];
}

// Exclusive scan of count[E*B] in (expert, block) order, in place; also
// offsets[e] = start of expert e, offsets[E] = total.  One CTA of 1024
// threads: each sums its contiguous range, the range sums are scanned with
// warp shuffles (within each warp, then across the 32 warp totals), and each
// thread rewrites its range with the running prefix.
__global__ void route_scan_kernel(int32_t* __restrict__ count, int E, int B, int32_t* __restrict__ offsets) {
    __shared__ int32_t wsum[32];
    const int n = E * B;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = threadIdx.x * per, hi = min(n, lo + per);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t s = 0;
    for (int i = lo; i < hi; ++i) s += count[i];
    int32_t v = s;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        wsum[lane] = w;  // inclusive totals of warps 0..lane
    }
    __syncthreads();
    const int32_t before = (warp ? wsum[warp - 1] : 0) + v - s;  // exclusive prefix of this thread's range
    int32_t run = before;
    for (int i = lo; i < hi; ++i) {
        const int32_t c = count[i];
        count[i] = run;
        if (i % B == 0) offsets[i / B] = run;
        run += c;
    }
    if (threadIdx.x == blockDim.x - 1) offsets[E] = before + s;
}

// Row of each (token, rank): base[e][b] + number of earlier tokens of the
// block that hold expert e.  One warp per block: the block's expert ids and
// each expert's base row are staged in shared memory, then the warp walks the
// tokens in order; lane k < topk takes the token's k-th expert and advances
// that expert's next row (a token holds an expert at most once, so the lanes'
// entries are distinct and the walk needs no atomics).
__global__ void route_scatter_kernel(const int32_t* __restrict__ ids, int T, int E, int topk, int B,
                                     const int32_t* __restrict__ base, int32_t* __restrict__ token_of,
                                     int32_t* __restrict__ expert_of, int32_t* __restrict__ pos) {
    __shared__ int32_t next_row[kMaxExperts];
    __shared__ int32_t ids_s[kBlockTokens * kMaxTopk];
    const int b = blockIdx.x, lane = threadIdx.x;
    const int t0 = b * kBlockTokens, nt = min(T - t0, kBlockTokens);
    for (int e = lane; e < E; e += 32) next_row[e] = base[(size_t)e * B + b];
    for (int i = lane; i < nt * topk; i += 32) ids_s[i] = ids[(size_t)t0 * topk + i];
    __syncwarp();
    for (int j = 0; j < nt; ++j) {
        if (lane < topk) {
            const int e = ids_s[j * topk + lane];
            const int r = next_row[e];
            next_row[e] = r + 1;
            token_of[r] = t0 + j;
            expert_of[r] = e;
            pos[(size_t)(t0 + j) * topk + lane] = r;
        }
        __syncwarp();
    }
}

__global__ void gather_kernel(const uint16_t* __restrict__ X, int K, const int32_t* __restrict__ token_of,
                              int R, uint16_t* __restrict__ Xs) {
    const int vec = K / 8;  // 16-byte vectors per row
    const size_t total = (size_t)R * vec;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / vec), c = (int)(i % vec);
        const uint4 v = reinterpret_cast<const uint4*>(X + (size_t)token_of[r] * K)[c];
        reinterpret_cast<uint4*>(Xs + (size_t)r * K)[c] = v;
    }
}

// 8 consecutive outputs per thread with 16-byte loads and stores (N % 8 == 0,
// Y and out 16-byte aligned); per element the same fp32 FMAs in the same
// rank order as combine_kernel, so the results are identical.
template <bool YF16, bool OF16>
__global__ void combine8_kernel(const void* __restrict__ Y, int N, const int32_t* __restrict__ pos,
                                const float* __restrict__ w, int T, int topk, void* __restrict__ out) {
    const int nv = N / 8;
    const size_t total = (size_t)T * nv;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / nv), c = (int)(i % nv);
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int k = 0; k < topk; ++k) {
            const size_t r = (size_t)pos[(size_t)t * topk + k];
            const float wk = w[(size_t)t * topk + k];
            float y[8];
            if (YF16) {
                const uint4 v = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(Y) + r * N)[c];
                const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&u[h]));
                    y[2 * h] = f.x;
                    y[2 * h + 1] = f.y;
                }
            } else {
                const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(Y) + r * N) + 2 * c;
                const float4 a = src[0], b = src[1];
                y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
                y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(wk, y[e], acc[e]);
        }
        if (OF16) {
            uint32_t u[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
                u[h] = (uint32_t)__half_as_ushort(__float2half_rn(acc[2 * h])) |
                       ((uint32_t)__half_as_ushort(__float2half_rn(acc[2 * h + 1])) << 16);
            reinterpret_cast<uint4*>(out)[i] = make_uint4(u[0], u[1], u[2], u[3]);
        } else {
            float4* dst = reinterpret_cast<float4*>(out) + 2 * i;
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
    }
}

template <bool YF16, bool OF16>
__global__ void combine_kernel(const void* __restrict__ Y, int N, const int32_t* __restrict__ pos,
                               const float* __restrict__ w, int T, int topk, void* __restrict__ out) {
    const size_t total = (size_t)T * N;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / N), n = (int)(i % N);
        float acc = 0.f;
        for (int k = 0; k < topk; ++k) {
            const size_t r = (size_t)pos[(size_t)t * topk + k];
            const float y = YF16 ? __half2float(__ushort_as_half(static_cast<const uint16_t*>(Y)[r * N + n]))
                                 : static_cast<const float*>(Y)[r * N + n];
            acc = fmaf(w[(size_t)t * topk + k], y, acc);
        }
        if (OF16)
            static_cast<uint16_t*>(out)[i] = __half_as_ushort(__float2half_rn(acc));
        else
            static_cast<float*>(out)[i] = acc;
    }
}

}  // namespace q4m

namespace q4i {
size_t moe_route_workspace_bytes(int T, int E, int topk) {
    (void)topk;
    if (T < 1 || E < 1) return 0;
    const size_t B = (size_t)(T + q4m::kBlockTokens - 1) / q4m::kBlockTokens;
    return (B * (size_t)E * sizeof(int32_t) + 255) & ~size_t(255);
}
}  // namespace q4i

using namespace q4i;

extern "C" {

size_t q4_moe_route_workspace_bytes(int T, int E, int topk) {
    clear_error();
    return moe_route_workspace_bytes(T, E, topk);
}

q4_status q4_moe_route(const uint16_t* logits, int T, int E, int topk, int32_t* topk_ids, float* topk_weights,
                       int32_t* offsets, int32_t* token_of, int32_t* expert_of, int32_t* pos, void* workspace,
                       size_t workspace_bytes, q4_stream_t stream) {
    clear_error();
    if (!logits || !topk_ids || !topk_weights || !offsets || !token_of || !expert_of || !pos || !workspace)
        return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (T < 1 || E < 1 || E > q4m::kMaxExperts || topk < 1 || topk > q4m::kMaxTopk || topk > E)
        return fail(Q4_ERR_INVALID_ARG, "T=%d E=%d topk=%d (need T>=1, 1<=E<=%d, 1<=topk<=min(E,%d))", T, E,
                    topk, q4m::kMaxExperts, q4m::kMaxTopk);
    if (T > q4m::kMaxRouteTokens) return fail(Q4_ERR_UNSUPPORTED, "T=%d above %d", T, q4m::kMaxRouteTokens);
    const size_t need = moe_route_workspace_bytes(T, E, topk);
    if (workspace_bytes < need) return fail(Q4_ERR_INVALID_ARG, "workspace %zu bytes, need %zu", workspace_bytes, need);
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int B = (T + q4m::kBlockTokens - 1) / q4m::kBlockTokens;
    int32_t* count = static_cast<int32_t*>(workspace);
    q4m::route_topk_kernel<<<B, 32 * q4m::kBlockTokens, 0, s>>>(logits, T, E, topk, topk_ids, topk_weights, B,
                                                                count);
    q4m::route_scan_kernel<<<1, 1024, 0, s>>>(count, E, B, offsets);
    q4m::route_scatter_kernel<<<B, 32, 0, s>>>(topk_ids, T, E, topk, B, count, token_of, expert_of, pos);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "q4_moe_route launch");
    return Q4_OK;
}

q4_status q4_moe_gather(const uint16_t* X, int T, int K, const int32_t* token_of, int R, uint16_t* X_sorted,
                        q4_stream_t stream) {
    clear_error();
    if (!X || !token_of || !X_sorted) return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (T < 1 || R < 1 || K < 8 || K % 8) return fail(Q4_ERR_INVALID_ARG, "T=%d R=%d K=%d (K %% 8 == 0)", T, R, K);
    if (!aligned16(X) || !aligned16(X_sorted)) return fail(Q4_ERR_MISALIGNED, "X and X_sorted must be 16-byte aligned");
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    const size_t total = (size_t)R * (K / 8);
    const int grid = (int)((total + 255) / 256 < (size_t)dev->sms * 8 ? (total + 255) / 256 : (size_t)dev->sms * 8);
    q4m::gather_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(X, K, token_of, R, X_sorted);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "q4_moe_gather launch");
    return Q4_OK;
}

q4_status q4_moe_combine(const void* Y, q4_dtype y_dtype, int N, const int32_t* pos, const float* topk_weights,
                         int T, int topk, void* out, q4_dtype out_dtype, q4_stream_t stream) {
    clear_error();
    if (!Y || !pos || !topk_weights || !out) return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (N < 1 || T < 1 || topk < 1 || topk > q4m::kMaxTopk) return fail(Q4_ERR_INVALID_ARG, "N=%d T=%d topk=%d", N, T, topk);
    if ((y_dtype != Q4_F32 && y_dtype != Q4_F16) || (out_dtype != Q4_F32 && out_dtype != Q4_F16))
        return fail(Q4_ERR_INVALID_ARG, "bad dtype");
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N % 8 == 0 && aligned16(Y) && aligned16(out)) {
        const size_t total8 = (size_t)T * (N / 8);
        const int g8 = (int)((total8 + 255) / 256 < (size_t)dev->sms * 8 ? (total8 + 255) / 256 : (size_t)dev->sms * 8);
        if (y_dtype == Q4_F16 && out_dtype == Q4_F16)
            q4m::combine8_kernel<true, true><<<g8, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
        else if (y_dtype == Q4_F16)
            q4m::combine8_kernel<true, false><<<g8, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
        else if (out_dtype == Q4_F16)
            q4m::combine8_kernel<false, true><<<g8, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
        else
            q4m::combine8_kernel<false, false><<<g8, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
        const cudaError_t e8 = cudaGetLastError();
        if (e8 != cudaSuccess) return cuda_fail(e8, "q4_moe_combine launch");
        return Q4_OK;
    }
    const size_t total = (size_t)T * N;
    const int grid = (int)((total + 255) / 256 < (size_t)dev->sms * 8 ? (total + 255) / 256 : (size_t)dev->sms * 8);
    if (y_dtype == Q4_F16 && out_dtype == Q4_F16)
        q4m::combine_kernel<true, true><<<grid, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
    else if (y_dtype == Q4_F16)
        q4m::combine_kernel<true, false><<<grid, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
    else if (out_dtype == Q4_F16)
        q4m::combine_kernel<false, true><<<grid, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
    else
        q4m::combine_kernel<false, false><<<grid, 256, 0, s>>>(Y, N, pos, topk_weights, T, topk, out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "q4_moe_combine launch");
    return Q4_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free routing.
//
// Some callers cannot allocate device memory: a plugin inside a host runtime
// that owns every device buffer and hands the plugin only the tensors it
// works on, or a serving loop whose allocator is fixed at load time.  For
// them q4_moe_route_noalloc runs the same four routing kernels as
// q4_moe_route, with the per-(expert, 32-token block) counters in the
// file-scope array below instead of a caller workspace.  The array lives on
// every device that loads the library until the process exits.
// ---------------------------------------------------------------------------
namespace q4m {
constexpr int kStaticRouteCounters = 1 << 16;  // 65536 int32 = 256 KB
static __device__ __align__(256) int32_t g_route_scratch[kStaticRouteCounters];
}  // namespace q4m

namespace {
constexpr int kScratchDevices = 64;  // current_device() refuses ordinals from 64 up
std::mutex g_route_scratch_mutex;
int32_t* g_route_scratch_ptr[kScratchDevices];  // device address of the array, per device ordinal
}  // namespace

extern "C" q4_status q4_moe_route_noalloc(const uint16_t* logits, int T, int E, int topk, int32_t* topk_ids,
                                          float* topk_weights, int32_t* offsets, int32_t* token_of,
                                          int32_t* expert_of, int32_t* pos, q4_stream_t stream) {
    clear_error();
    if (!logits || !topk_ids || !topk_weights || !offsets || !token_of || !expert_of || !pos)
        return fail(Q4_ERR_INVALID_ARG, "NULL pointer argument");
    if (T < 1 || E < 1 || E > q4m::kMaxExperts || topk < 1 || topk > q4m::kMaxTopk || topk > E)
        return fail(Q4_ERR_INVALID_ARG, "T=%d E=%d topk=%d (need T>=1, 1<=E<=%d, 1<=topk<=min(E,%d))", T, E,
                    topk, q4m::kMaxExperts, q4m::kMaxTopk);
    if (T > q4m::kMaxRouteTokens) return fail(Q4_ERR_UNSUPPORTED, "T=%d above %d", T, q4m::kMaxRouteTokens);
    const long long B = ((long long)T + q4m::kBlockTokens - 1) / q4m::kBlockTokens;
    if (B * E > q4m::kStaticRouteCounters)
        return fail(Q4_ERR_UNSUPPORTED,
                    "T=%d, E=%d need %lld counters; the static scratch holds %d (at most %lld tokens for E=%d); "
                    "use q4_moe_route with a workspace",
                    T, E, B * E, q4m::kStaticRouteCounters,
                    (long long)q4m::kBlockTokens * (q4m::kStaticRouteCounters / E), E);
    const DeviceInfo* dev = nullptr;
    q4_status st = current_device(&dev);
    if (st != Q4_OK) return st;
    if (dev->device < 0 || dev->device >= kScratchDevices)
        return fail(Q4_ERR_NO_DEVICE, "device ordinal %d outside 0..%d", dev->device, kScratchDevices - 1);
    int32_t* scratch = nullptr;
    {
        // Set-up, once per device, with that device current: the host-side
        // name of the array is not a device address; ask the runtime for it.
        std::lock_guard<std::mutex> lock(g_route_scratch_mutex);
        if (!g_route_scratch_ptr[dev->device]) {
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, q4m::g_route_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(routing scratch)");
            g_route_scratch_ptr[dev->device] = static_cast<int32_t*>(p);
        }
        scratch = g_route_scratch_ptr[dev->device];
    }
    // Every counter the kernels read is written first by route_topk_kernel,
    // so nothing in the array has to start at zero.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int Bi = (int)B;
    q4m::route_topk_kernel<<<Bi, 32 * q4m::kBlockTokens, 0, s>>>(logits, T, E, topk, topk_ids, topk_weights, Bi,
                                                                 scratch);
    q4m::route_scan_kernel<<<1, 1024, 0, s>>>(scratch, E, Bi, offsets);
    q4m::route_scatter_kernel<<<Bi, 32, 0, s>>>(topk_ids, T, E, topk, Bi, scratch, token_of, expert_of, pos);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "q4_moe_route_noalloc launch");
    return Q4_OK;
}
