// Host-side internals shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <stddef.h>
#include <stdint.h>

#include "../../include/q4.h"

namespace q4i {

// Records printf-style text as the calling thread's last error; returns s.
q4_status fail(q4_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
q4_status cuda_fail(cudaError_t e, const char* what);
void clear_error();

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int smem_optin = 0;       // max dynamic shared memory per block (opt-in)
    int smem_per_sm = 0;
    int cc_major = 0, cc_minor = 0;
    int* err_word = nullptr;  // device address of the error word (q4_api.cu)
};

// Info for the current device (cached per device).  Fails with
// Q4_ERR_NO_DEVICE if there is no device or it is not compute capability 10.3.
q4_status current_device(const DeviceInfo** out);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device when it is not already that high (the attribute persists).  `marks`
// is the call site's per-device high-water mark (64 devices), kept in atomics
// so concurrent host threads may launch; two threads may both set the
// attribute, which is harmless.
inline cudaError_t ensure_smem_attr(const void* kern, std::atomic<int>* marks, int bytes) {
    int dev = 0;
    cudaGetDevice(&dev);
    const bool tracked = dev >= 0 && dev < 64;
    if (tracked && bytes <= marks[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess || !tracked) return e;
    int cur = marks[dev].load(std::memory_order_relaxed);
    while (bytes > cur && !marks[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
    }
    return cudaSuccess;
}

// 2-D tensor map (q4_moe_gemm.cu): `inner` x `outer` elements of type dt,
// rows `row_bytes` apart, copied in boxes of box_inner x box_outer.
q4_status make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);

// ---- decode attention (q4_attn.cu) -----------------------------------------
size_t attn_workspace_bytes(int n_q_heads, int head_dim, int max_seq);
q4_status attn_validate(const q4_attention_desc& d);
// compute_table: this launch computes the step's RoPE (cos, sin) table (the
// first attention of a step); later ones read it from the same workspace.
q4_status attn_enqueue(const q4_attention_desc& d, cudaStream_t s, bool compute_table);
q4_status pos_advance(int32_t* pos, cudaStream_t s, int by = 1);
// Prefill with attention: the chunk's rotation table (fp64 angles) in `cs`
// (prefill_attn_cs_bytes; for head_dim 128 followed by the rotated query's
// fp16 hi / lo parts, which the append kernel writes), then per layer the
// cache append and the causal attention of the chunk's tokens (positions
// *pos + t0 + t).
size_t prefill_attn_cs_bytes(int chunk, int head_dim, int n_q_heads);
q4_status prefill_attn_table(const int32_t* pos, int t0, int C, int head_dim, float theta, void* cs, cudaStream_t s);
q4_status prefill_attn_enqueue(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* k_cache,
                               uint16_t* v_cache, const int32_t* pos, int t0, int C, int Hq, int Hkv, int D,
                               int max_seq, void* cs, uint16_t* a, cudaStream_t s);

// ---- dense GEMM on the grouped-GEMM kernel (q4_moe_gemm.cu) ---------------
q4_status gemm_launch(const q4_gemm_desc* d, q4_stream_t stream);
// The same, but when K splits (*kparts > 1) the fp32 partial sums are left
// in the workspace ([kparts][M][N]) for the caller to add: no reduce kernel,
// no epilogue (residual) applied.
q4_status gemm_launch_parts(const q4_gemm_desc* d, q4_stream_t stream, int* kparts);
// Y[i] = X W_i^T (fp16 [M][N_i]) for nseg <= 3 PLAIN matrices of one K, as
// one launch (the units of all matrices share the GPU); no residual, no split.
q4_status gemm_launch_multi(const q4_linear* w, void* const* Y, int nseg, const uint16_t* X, int M,
                            q4_stream_t stream);
// Bytes of fp32 partials a dense GEMM of this shape splits K into (0 = no split).
size_t gemm_split_bytes(int M, int N, int K, bool glu);

// ---- fused multi-segment GEMV (q4_gemv.cu) --------------------------------
q4_status validate_gemv(const q4_gemv_desc& d);

// Tagged activations, used inside a decode step: every activation element is
// a 32-bit word (fp16 value | 16-bit tag << 16), the tag naming the decode
// step and the stage that wrote it.  A kernel whose x is tagged does not wait
// for its predecessor grid to complete; it polls the words it needs.
struct GemvTagged {
    const uint32_t* x = nullptr;                       // tagged x, or nullptr (plain desc.x)
    int x_stage = 0;                                   // stage that writes x
    uint32_t* y[Q4_MAX_SEGMENTS] = {};                 // tagged copies of the outputs (optional)
    const uint32_t* res[Q4_MAX_SEGMENTS] = {};         // tagged residuals (instead of plain ones)
    int res_stage = 0;
    const uint32_t* step_ctr = nullptr;                // decode-step counter
    uint32_t* done_ctr = nullptr;                      // CTA completion counter (last stage only)
    int stage = 0, n_stages = 1;
    bool last = false;                                 // this launch advances step_ctr when done
};

// early_prefetch: weight copies may start before the programmatic-dependency
// wait (only when the weights are not written by a preceding kernel).
// bits: code width, 4 (Wq [N][K/8]) or 8 (Wq [N][K/4]).
q4_status launch_gemv(const q4_gemv_desc& d, cudaStream_t stream, bool pdl, bool early_prefetch,
                      const GemvTagged* tg = nullptr, int bits = 4);
// True when one launch of (M, K) fits in shared memory without splitting M.
bool gemv_fits_unsplit(int M, int K);

// ---- persistent decode step (q4_gemv.cu) -----------------------------------
// One cooperative launch runs every stage of a decode step (tagged hand-off
// between stages).  The per-stage kernel parameters are an opaque table of
// n * gemv_params_bytes() bytes that the caller copies to device memory.
size_t gemv_params_bytes();

struct PersistentGeom {
    int M = 0, n = 0, grid = 0, slots = 0;
    uint32_t slot_bytes = 0, meta_off = 0, ring_off = 0, x_bytes = 0;
    size_t smem = 0;
    const uint32_t* step_ctr = nullptr;
    uint32_t* done_ctr = nullptr;
};

// Fills host_params (n entries) and g from the stages and their tagged
// hand-off; *fits is false (and Q4_OK returned) when the step does not fit
// one persistent launch.
q4_status persistent_plan(const q4_gemv_desc* d, const GemvTagged* tg, int n, void* host_params,
                          PersistentGeom* g, bool* fits);
q4_status persistent_launch(const PersistentGeom& g, const void* dev_params, cudaStream_t stream);

// ---- clustered decode step (q4_step.cu) ------------------------------------
// The layer stack of an M = 1 decode step as one launch of thread-block
// clusters (two grid-wide hand-offs per layer), beside it a launch that
// computes the k and v rows on the SMs the clusters leave free; lm_head is
// launched after them.
constexpr int kStepMaxClusters = 20;  // the exchange buffer holds this many clusters' partials

struct StepArgs {
    int L = 0, H = 0, QN = 0, KVN = 0, F = 0;
    float eps = 1e-6f;
    const q4_layer_weights* layers = nullptr;  // host [L]
    const void* dev_layers = nullptr;          // workspace: L * step_layer_desc_bytes()
    const void* dev_maps = nullptr;            // workspace: 6 L tensor maps (64-byte aligned)
    const uint16_t* x = nullptr;
    uint16_t *h = nullptr, *h_mid = nullptr, *q = nullptr, *k = nullptr, *v = nullptr, *act = nullptr;
    unsigned long long* xch = nullptr;         // workspace: 2 L * kStepMaxClusters * H words
    uint32_t* htag = nullptr;                  // workspace: L * H tagged words (each layer's input h)
    uint32_t* ctr = nullptr;                   // workspace: step and finished-CTA counters (5 words)
};

struct StepPlan {
    int S = 0, C = 0;  // cluster size and cluster count
    size_t smem = 0;
    alignas(64) unsigned char params[512];
    int kv_grid = 0;   // the k / v launch
    size_t kv_smem = 0;
    alignas(64) unsigned char kv_params[256];
};

size_t step_layer_desc_bytes();
// *ok is false (and Q4_OK returned) when the shapes or the device do not allow the step.
q4_status step_plan(const StepArgs& a, StepPlan* out, bool* ok);
// Host copies of the layer descriptors (L entries) and tensor maps (6 L),
// which the caller uploads to dev_layers / dev_maps, and the launch pointers.
q4_status step_bind(StepPlan* sp, const StepArgs& a, void* host_layers, void* host_maps);
q4_status step_launch(const StepPlan& sp, cudaStream_t stream);

// ---- MoE (q4_moe.cu, q4_moe_gemm.cu) ---------------------------------------
size_t moe_route_workspace_bytes(int T, int E, int topk);

}  // namespace q4i
