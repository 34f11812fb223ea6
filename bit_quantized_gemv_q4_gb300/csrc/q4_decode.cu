// Decode-step scheduler: a whole layer stack of fused GEMV launches, captured
// once into a CUDA graph and replayed per token.
//
// BaseRT: optimal LLM inference on Apple Silicon with native Metal:
// * §3 "BaseRT runtime design": a low-overhead dispatch path that removes
//   per-operator dispatch, allocation and graph evaluation from the decode hot
//   path.  Here the first call plans and captures; every later call is one
//   cudaGraphLaunch.
// * §3.1 "Data-driven architecture descriptor": the model is data (the
//   q4_layer_table) and the engine never branches on the architecture.
// * §3.2 "Zero-allocation decode loop": activations live in a caller-owned
//   workspace laid out at plan time; replays allocate nothing.
// * §3.3 "Kernel fusion and specialisation": fused QKV and gate/up launches,
//   the pre-norm RMSNorms folded into the GEMV prologues, residual adds and
//   SiLU*up folded into the GEMV epilogues.
// Programmatic dependent launch links consecutive kernels so each kernel's
// weight stream (which never depends on its predecessor) starts while the
// predecessor is still running; only its activation reads wait.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <vector>

#include "q4_internal.h"

namespace q4i {
namespace {

struct Dims {
    int hidden = 0, qN = 0, kvN = 0, ffn = 0, vocab = 0, M = 0, L = 0;
    bool attn = false;  // Q4_DECODE_ATTENTION
    bool step = false;  // the clustered step may run the layers (the workspace holds its regions)
    int hd = 0, max_seq = 0;
};

struct Layout {
    size_t h = 0, h_mid = 0, q = 0, k = 0, v = 0, act = 0;
    size_t a = 0, attn_ws = 0, attn_ws_bytes = 0;  // attention output and its scratch (Q4_DECODE_ATTENTION)
    size_t params = 0;  // per-stage kernel parameters of the persistent launch
    // clustered step (M = 1 without attention): layer descriptors, tensor
    // maps, the partial-sum exchange and its counters
    size_t step_layers = 0, step_maps = 0, xch = 0, htag = 0, step_ctr = 0, step_end = 0;
    // tagged copies of the activations that later stages read, and counters
    size_t h_t = 0, hm_t = 0, q_t = 0, act_t = 0, ctr = 0, tagged_begin = 0, total = 0;
};

struct Plan {
    int device = -1;
    Dims dims;
    Layout lay;
    std::vector<q4_layer_weights> layers;
    q4_linear lm_head{};
    const uint16_t* final_norm = nullptr;
    float eps = 1e-6f;
    q4_dtype logits_dtype = Q4_F32;
    void* workspace = nullptr;
    size_t workspace_bytes = 0;
    int flags = 0;
    const void* x_key = nullptr;
    void* logits_key = nullptr;
    std::vector<q4_gemv_desc> stages;
    std::vector<q4_attention_desc> attn;  // per layer, with Q4_DECODE_ATTENTION
    int32_t* pos = nullptr;
    float rope_theta = 0.f;
    std::vector<GemvTagged> tagged;  // per stage, used when tagged_mode or persistent
    bool tagged_mode = false;
    bool persistent = false;         // one cooperative launch per step
    PersistentGeom geom;
    std::vector<uint8_t> params_host;  // kept alive for the asynchronous upload
    bool tagged_ready = false;       // tagged region zeroed
    bool fused = false;              // the clustered step runs the layers (then lm_head)
    StepPlan step;
    std::vector<uint8_t> step_layers_host, step_maps_host;  // kept alive for the upload
    bool step_ready = false;         // exchange region and counters zeroed
    cudaStream_t capture_stream = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

q4_status check_linear(const q4_linear& w, int N, int K, const char* what, int layer) {
    if (!w.Wq || !w.scales || !w.biases)
        return fail(Q4_ERR_INVALID_ARG, "layer %d %s: NULL weights", layer, what);
    if ((N > 0 && w.N != N) || (K > 0 && w.K != K) || w.N < 1 || w.K < 64 || w.K % 64)
        return fail(Q4_ERR_INVALID_ARG, "layer %d %s: shape %dx%d does not fit (want N=%d K=%d)", layer,
                    what, w.N, w.K, N, K);
    if (!aligned16(w.Wq) || !aligned16(w.scales) || !aligned16(w.biases))
        return fail(Q4_ERR_MISALIGNED, "layer %d %s: weights must be 16-byte aligned", layer, what);
    return Q4_OK;
}

q4_status table_dims(const q4_layer_table* t, Dims* d) {
    if (!t) return fail(Q4_ERR_INVALID_ARG, "table is NULL");
    if (t->n_layers < 0 || t->hidden < 64 || t->hidden % 64)
        return fail(Q4_ERR_INVALID_ARG, "n_layers=%d hidden=%d", t->n_layers, t->hidden);
    if (t->M < 1 || t->M > 8) return fail(Q4_ERR_UNSUPPORTED, "M=%d outside 1..8", t->M);
    if (t->n_layers > 0 && !t->layers) return fail(Q4_ERR_INVALID_ARG, "layers is NULL");
    if (t->logits_dtype != Q4_F32 && t->logits_dtype != Q4_F16) return fail(Q4_ERR_INVALID_ARG, "bad logits_dtype");
    d->hidden = t->hidden;
    d->M = t->M;
    d->L = t->n_layers;
    q4_status st;
    for (int l = 0; l < t->n_layers; ++l) {
        const q4_layer_weights& w = t->layers[l];
        const int H = t->hidden;
        if ((st = check_linear(w.q, 0, H, "q", l)) != Q4_OK) return st;
        if ((st = check_linear(w.k, 0, H, "k", l)) != Q4_OK) return st;
        if ((st = check_linear(w.v, 0, H, "v", l)) != Q4_OK) return st;
        if ((st = check_linear(w.o, H, w.q.N, "o", l)) != Q4_OK) return st;
        if ((st = check_linear(w.gate, 0, H, "gate", l)) != Q4_OK) return st;
        if ((st = check_linear(w.up, w.gate.N, H, "up", l)) != Q4_OK) return st;
        if ((st = check_linear(w.down, H, w.gate.N, "down", l)) != Q4_OK) return st;
        if (w.q.N % 8 || w.k.N % 8 || w.v.N % 8 || w.gate.N % 8)
            return fail(Q4_ERR_MISALIGNED, "layer %d: q/k/v/gate widths must be multiples of 8", l);
        if ((w.attn_norm && !aligned16(w.attn_norm)) || (w.ffn_norm && !aligned16(w.ffn_norm)))
            return fail(Q4_ERR_MISALIGNED, "layer %d: norm weights must be 16-byte aligned", l);
        if (d->qN < w.q.N) d->qN = w.q.N;
        if (d->kvN < w.k.N) d->kvN = w.k.N;
        if (d->kvN < w.v.N) d->kvN = w.v.N;
        if (d->ffn < w.gate.N) d->ffn = w.gate.N;
    }
    if ((st = check_linear(t->lm_head, 0, t->hidden, "lm_head", -1)) != Q4_OK) return st;
    if (t->flags & Q4_DECODE_ATTENTION) {
        if (t->M != 1) return fail(Q4_ERR_UNSUPPORTED, "Q4_DECODE_ATTENTION needs M = 1 (M=%d)", t->M);
        if (t->flags & (Q4_DECODE_TAGGED | Q4_DECODE_PERSISTENT))
            return fail(Q4_ERR_UNSUPPORTED, "Q4_DECODE_ATTENTION runs without TAGGED and PERSISTENT");
        if (!t->pos) return fail(Q4_ERR_INVALID_ARG, "pos is NULL");
        for (int l = 0; l < t->n_layers; ++l) {
            const q4_layer_weights& w = t->layers[l];
            q4_attention_desc a = {};
            a.q = a.k = a.v = a.a = reinterpret_cast<uint16_t*>(16);  // shapes only
            a.workspace = reinterpret_cast<void*>(256);
            a.k_cache = w.k_cache;
            a.v_cache = w.v_cache;
            a.pos = t->pos;
            a.head_dim = t->head_dim;
            a.max_seq = t->max_seq;
            a.rope_theta = t->rope_theta;
            if (t->head_dim < 1 || w.q.N % t->head_dim || w.k.N % t->head_dim || w.v.N != w.k.N)
                return fail(Q4_ERR_INVALID_ARG, "layer %d: q, k, v widths do not split into heads of %d", l,
                            t->head_dim);
            a.n_q_heads = w.q.N / t->head_dim;
            a.n_kv_heads = w.k.N / t->head_dim;
            a.workspace_bytes = attn_workspace_bytes(a.n_q_heads, a.head_dim, a.max_seq > 0 ? a.max_seq : 1);
            if ((st = attn_validate(a)) != Q4_OK) return st;
            if (w.o.K != w.q.N) return fail(Q4_ERR_INVALID_ARG, "layer %d: o.K != q.N", l);
        }
        d->attn = true;
        d->hd = t->head_dim;
        d->max_seq = t->max_seq;
    }
    d->step = t->M == 1 && !d->attn && t->n_layers > 0 && (t->flags & Q4_DECODE_CLUSTERED) &&
              !(t->flags & (Q4_DECODE_TAGGED | Q4_DECODE_PERSISTENT));
    if (t->final_norm && !aligned16(t->final_norm)) return fail(Q4_ERR_MISALIGNED, "final_norm must be 16-byte aligned");
    if (!(t->norm_eps >= 0.f)) return fail(Q4_ERR_INVALID_ARG, "norm_eps must be >= 0");
    d->vocab = t->lm_head.N;
    return Q4_OK;
}

Layout layout_of(const Dims& d) {
    Layout l;
    size_t off = 0;
    auto take = [&](size_t elems) {
        size_t o = off;
        off = align256(off + elems * 2);
        return o;
    };
    l.h = take((size_t)d.M * d.hidden);
    l.h_mid = take((size_t)d.M * d.hidden);
    l.q = take((size_t)d.M * (d.qN > 0 ? d.qN : 1));
    l.k = take((size_t)d.M * (d.kvN > 0 ? d.kvN : 1));
    l.v = take((size_t)d.M * (d.kvN > 0 ? d.kvN : 1));
    l.act = take((size_t)d.M * (d.ffn > 0 ? d.ffn : 1));
    if (d.attn) {
        l.a = take((size_t)d.M * (d.qN > 0 ? d.qN : 1));
        l.attn_ws_bytes = attn_workspace_bytes(d.qN / d.hd, d.hd, d.max_seq);
        l.attn_ws = take(l.attn_ws_bytes / 2 + 1);
    }
    l.params = take((size_t)(4 * d.L + 1) * gemv_params_bytes() / 2);
    if (d.step) {
        l.step_layers = take((size_t)d.L * step_layer_desc_bytes() / 2 + 1);
        l.step_maps = take((size_t)6 * d.L * sizeof(CUtensorMap) / 2);
        l.xch = take((size_t)2 * d.L * kStepMaxClusters * d.hidden * 4);
        l.htag = take((size_t)d.L * d.hidden * 2);
        l.step_ctr = take(64);
        l.step_end = off;
    }
    l.tagged_begin = off;
    l.h_t = take((size_t)d.M * d.hidden * 2);
    l.hm_t = take((size_t)d.M * d.hidden * 2);
    l.q_t = take((size_t)d.M * (d.qN > 0 ? d.qN : 1) * 2);
    l.act_t = take((size_t)d.M * (d.ffn > 0 ? d.ffn : 1) * 2);
    l.ctr = take(128);
    l.total = off;
    return l;
}

q4_segment seg_of(const q4_linear& w, void* y, const uint16_t* residual) {
    q4_segment s = {};
    s.Wq = w.Wq;
    s.scales = w.scales;
    s.biases = w.biases;
    s.N = w.N;
    s.ldy = w.N;
    s.y = y;
    s.residual = residual;
    return s;
}

void build_stages(Plan& p, const uint16_t* x, void* logits) {
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    uint16_t* h = reinterpret_cast<uint16_t*>(ws + p.lay.h);
    uint16_t* hm = reinterpret_cast<uint16_t*>(ws + p.lay.h_mid);
    uint16_t* q = reinterpret_cast<uint16_t*>(ws + p.lay.q);
    uint16_t* k = reinterpret_cast<uint16_t*>(ws + p.lay.k);
    uint16_t* v = reinterpret_cast<uint16_t*>(ws + p.lay.v);
    uint16_t* act = reinterpret_cast<uint16_t*>(ws + p.lay.act);
    uint16_t* a_buf = reinterpret_cast<uint16_t*>(ws + p.lay.a);
    const int M = p.dims.M, H = p.dims.hidden;
    uint32_t* h_t = reinterpret_cast<uint32_t*>(ws + p.lay.h_t);
    uint32_t* hm_t = reinterpret_cast<uint32_t*>(ws + p.lay.hm_t);
    uint32_t* q_t = reinterpret_cast<uint32_t*>(ws + p.lay.q_t);
    uint32_t* act_t = reinterpret_cast<uint32_t*>(ws + p.lay.act_t);
    uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + p.lay.ctr);
    const int NS = 4 * p.dims.L + 1;
    auto tagged = [&](int stage, const uint32_t* x, int x_stage) {
        GemvTagged t;
        t.x = x;
        t.x_stage = x_stage;
        t.step_ctr = ctr;
        t.done_ctr = ctr + 1;
        t.stage = stage;
        t.n_stages = NS;
        return t;
    };
    p.stages.clear();
    p.tagged.clear();
    p.attn.clear();
    for (int l = 0; l < p.dims.L; ++l) {
        // stages of layer l: 4l QKV, 4l+1 o, 4l+2 gate/up, 4l+3 down
        const uint32_t* h_in_t = l == 0 ? nullptr : h_t;  // layer 0 reads the caller's plain x
        GemvTagged t = tagged(4 * l, h_in_t, 4 * l - 1);
        t.y[0] = q_t;
        p.tagged.push_back(t);
        t = tagged(4 * l + 1, q_t, 4 * l);
        t.y[0] = hm_t;
        t.res[0] = h_in_t;
        t.res_stage = 4 * l - 1;
        p.tagged.push_back(t);
        t = tagged(4 * l + 2, hm_t, 4 * l + 1);
        t.y[0] = act_t;
        p.tagged.push_back(t);
        t = tagged(4 * l + 3, act_t, 4 * l + 2);
        t.y[0] = h_t;
        t.res[0] = hm_t;
        t.res_stage = 4 * l + 1;
        p.tagged.push_back(t);
    }
    {
        GemvTagged t = tagged(NS - 1, p.dims.L > 0 ? h_t : nullptr, NS - 2);
        t.last = true;
        p.tagged.push_back(t);
    }
    for (int l = 0; l < p.dims.L; ++l) {
        const q4_layer_weights& w = p.layers[l];
        const uint16_t* hin = l == 0 ? x : h;
        q4_gemv_desc d = {};
        // q, k, v in one launch
        d.M = M; d.K = H; d.x = hin; d.ldx = H; d.out_dtype = Q4_F16; d.mode = Q4_GEMV_PLAIN;
        d.x_rmsnorm = 1; d.norm_weight = w.attn_norm; d.norm_eps = p.eps;
        d.n_segments = 3;
        d.seg[0] = seg_of(w.q, q, nullptr);
        d.seg[1] = seg_of(w.k, k, nullptr);
        d.seg[2] = seg_of(w.v, v, nullptr);
        p.stages.push_back(d);
        if (p.dims.attn) {
            q4_attention_desc ad = {};
            ad.q = q;
            ad.k = k;
            ad.v = v;
            ad.k_cache = w.k_cache;
            ad.v_cache = w.v_cache;
            ad.pos = p.pos;
            ad.head_dim = p.dims.hd;
            ad.n_q_heads = w.q.N / p.dims.hd;
            ad.n_kv_heads = w.k.N / p.dims.hd;
            ad.max_seq = p.dims.max_seq;
            ad.rope_theta = p.rope_theta;
            ad.a = a_buf;
            ad.workspace = ws + p.lay.attn_ws;
            ad.workspace_bytes = p.lay.attn_ws_bytes;
            p.attn.push_back(ad);
        }
        // h' = h + Wo a (a = q without attention)
        d = {};
        d.M = M; d.K = w.o.K; d.x = p.dims.attn ? a_buf : q; d.ldx = w.o.K; d.out_dtype = Q4_F16; d.mode = Q4_GEMV_PLAIN;
        d.n_segments = 1;
        d.seg[0] = seg_of(w.o, hm, hin);
        p.stages.push_back(d);
        // act = SiLU(Wg h') * (Wu h')
        d = {};
        d.M = M; d.K = H; d.x = hm; d.ldx = H; d.out_dtype = Q4_F16; d.mode = Q4_GEMV_GLU;
        d.x_rmsnorm = 1; d.norm_weight = w.ffn_norm; d.norm_eps = p.eps;
        d.n_segments = 2;
        d.seg[0] = seg_of(w.gate, act, nullptr);
        d.seg[1] = seg_of(w.up, nullptr, nullptr);
        p.stages.push_back(d);
        // h = h' + Wd act
        d = {};
        d.M = M; d.K = w.down.K; d.x = act; d.ldx = w.down.K; d.out_dtype = Q4_F16; d.mode = Q4_GEMV_PLAIN;
        d.n_segments = 1;
        d.seg[0] = seg_of(w.down, h, hm);
        p.stages.push_back(d);
    }
    q4_gemv_desc d = {};
    d.M = M; d.K = H; d.x = p.dims.L > 0 ? h : x; d.ldx = H; d.out_dtype = p.logits_dtype;
    d.mode = Q4_GEMV_PLAIN; d.n_segments = 1;
    d.x_rmsnorm = 1; d.norm_weight = p.final_norm; d.norm_eps = p.eps;
    d.seg[0] = seg_of(p.lm_head, logits, nullptr);
    p.stages.push_back(d);
}

q4_status enqueue_stages(Plan& p, cudaStream_t s) {
    const bool pdl = !(p.flags & Q4_DECODE_NO_PDL);
    if (p.fused) {
        q4_status st = step_launch(p.step, s);
        if (st != Q4_OK) return st;
        return launch_gemv(p.stages.back(), s, pdl, true);
    }
    for (size_t i = 0; i < p.stages.size(); ++i) {
        q4_status st = launch_gemv(p.stages[i], s, pdl && i > 0, true, p.tagged_mode ? &p.tagged[i] : nullptr);
        if (st != Q4_OK) return st;
        // after layer l's QKV stage (stage 4l): append to the caches and attend
        if (p.dims.attn && i % 4 == 0 && i / 4 < p.attn.size()) {
            if ((st = attn_enqueue(p.attn[i / 4], s, i == 0)) != Q4_OK) return st;
        }
    }
    if (p.dims.attn) return pos_advance(p.pos, s);
    return Q4_OK;
}

// Plans the clustered step when every layer has the same shape and the
// device takes the clusters; uploads its tables into the workspace on `s`.
q4_status plan_fused(Plan& p, const uint16_t* x, cudaStream_t s) {
    const Dims& d = p.dims;
    const q4_layer_weights& w0 = p.layers[0];
    for (const q4_layer_weights& w : p.layers)
        if (w.q.N != w0.q.N || w.k.N != w0.k.N || w.v.N != w0.k.N || w.gate.N != w0.gate.N) return Q4_OK;
    uint8_t* ws = static_cast<uint8_t*>(p.workspace);
    StepArgs a;
    a.L = d.L;
    a.H = d.hidden;
    a.QN = w0.q.N;
    a.KVN = w0.k.N;
    a.F = w0.gate.N;
    a.eps = p.eps;
    a.layers = p.layers.data();
    a.dev_layers = ws + p.lay.step_layers;
    a.dev_maps = ws + p.lay.step_maps;
    a.x = x;
    a.h = reinterpret_cast<uint16_t*>(ws + p.lay.h);
    a.h_mid = reinterpret_cast<uint16_t*>(ws + p.lay.h_mid);
    a.q = reinterpret_cast<uint16_t*>(ws + p.lay.q);
    a.k = reinterpret_cast<uint16_t*>(ws + p.lay.k);
    a.v = reinterpret_cast<uint16_t*>(ws + p.lay.v);
    a.act = reinterpret_cast<uint16_t*>(ws + p.lay.act);
    a.xch = reinterpret_cast<unsigned long long*>(ws + p.lay.xch);
    a.htag = reinterpret_cast<uint32_t*>(ws + p.lay.htag);
    a.ctr = reinterpret_cast<uint32_t*>(ws + p.lay.step_ctr);
    bool ok = false;
    q4_status st = step_plan(a, &p.step, &ok);
    if (st != Q4_OK || !ok) return st;
    p.step_layers_host.assign((size_t)d.L * step_layer_desc_bytes(), 0);
    p.step_maps_host.assign((size_t)6 * d.L * sizeof(CUtensorMap) + 64, 0);
    // a 64-byte aligned host copy of the maps
    uint8_t* mh = p.step_maps_host.data();
    mh += (64 - (reinterpret_cast<uintptr_t>(mh) & 63)) & 63;
    if ((st = step_bind(&p.step, a, p.step_layers_host.data(), mh)) != Q4_OK) return st;
    cudaError_t e = cudaMemcpyAsync(ws + p.lay.step_layers, p.step_layers_host.data(), p.step_layers_host.size(),
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ws + p.lay.step_maps, mh, (size_t)6 * d.L * sizeof(CUtensorMap), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "uploading the clustered step's tables");
    p.fused = true;
    return Q4_OK;
}

void drop_graph(Plan& p) {
    if (p.exec) cudaGraphExecDestroy(p.exec);
    if (p.graph) cudaGraphDestroy(p.graph);
    p.exec = nullptr;
    p.graph = nullptr;
}

q4_status capture(Plan& p) {
    drop_graph(p);
    cudaError_t e;
    if (!p.capture_stream) {
        e = cudaStreamCreateWithFlags(&p.capture_stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) return cuda_fail(e, "creating the capture stream");
    }
    e = cudaStreamBeginCapture(p.capture_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamBeginCapture");
    q4_status st = enqueue_stages(p, p.capture_stream);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(p.capture_stream, &g);
    if (st != Q4_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture");
    p.graph = g;
    e = cudaGraphInstantiate(&p.exec, g, 0);
    if (e != cudaSuccess) {
        drop_graph(p);
        return cuda_fail(e, "cudaGraphInstantiate");
    }
    return Q4_OK;
}

// ---------------------------------------------------------------- prefill
// n[r] = fp16(h[r] / sqrt(mean(h[r]^2) + eps) * gamma), one warp per row,
// fp32 arithmetic; 16-byte accesses (hidden is a multiple of 64).
__global__ void rmsnorm_rows_kernel(const uint16_t* __restrict__ h, const uint16_t* __restrict__ gamma,
                                    uint16_t* __restrict__ n, int rows, int hidden, float eps) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const uint4* src = reinterpret_cast<const uint4*>(h + (size_t)warp * hidden);
    const int nv = hidden / 8;
    float ss = 0.f;
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = src[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = rsqrtf(ss / (float)hidden + eps);
    uint4* dst = reinterpret_cast<uint4*>(n + (size_t)warp * hidden);
    const uint4* gv = reinterpret_cast<const uint4*>(gamma);
    for (int i = lane; i < nv; i += 32) {
        const uint4 v = src[i];
        const uint4 g = gamma ? gv[i] : make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            const float2 gg = __half22float2(*reinterpret_cast<const __half2*>(&gw[j]));
            const __half2 hv = __floats2half2_rn(f.x * r * gg.x, f.y * r * gg.y);
            o[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// A split GEMM's fp32 partial sums added in part order to the residual,
// rounded to fp16 into h (in place over the residual), then the RMSNorm of
// that row into n -- the reduce kernel's and rmsnorm_rows_kernel's
// arithmetic in one launch.  One block of 4 warps per row: the warps share
// the partial sums (chunk i = lane + 32 t of the row goes to warp t % 4) and
// keep the rounded row in shared memory; warp 0 then forms the sum of
// squares in rmsnorm_rows_kernel's order (lane L over chunks L, L + 32, ...;
// a butterfly across lanes).  part: fp32 [kparts][rows][hidden]; dynamic
// shared memory: hidden fp16.
constexpr int kRnWarps = 4;

__global__ void __launch_bounds__(32 * kRnWarps) reduce_norm_rows_kernel(const float* __restrict__ part, int kparts,
                                                                        uint16_t* h, const uint16_t* __restrict__ gamma,
                                                                        uint16_t* __restrict__ n, int rows,
                                                                        int hidden, float eps) {
    extern __shared__ uint4 hs[];  // the row's rounded values
    __shared__ float r_row;
    const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (row >= rows) return;
    const size_t pr = (size_t)rows * hidden;
    uint4* hrow = reinterpret_cast<uint4*>(h + (size_t)row * hidden);
    const int nv = hidden / 8;
    for (int i = lane + 32 * warp; i < nv; i += 32 * kRnWarps) {
        const size_t o = (size_t)row * hidden + (size_t)i * 8;
        float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < kparts; ++k) {
            const float4 a = *reinterpret_cast<const float4*>(part + (size_t)k * pr + o);
            const float4 b = *reinterpret_cast<const float4*>(part + (size_t)k * pr + o + 4);
            y[0] += a.x; y[1] += a.y; y[2] += a.z; y[3] += a.w;
            y[4] += b.x; y[5] += b.y; y[6] += b.z; y[7] += b.w;
        }
        const uint4 rv = hrow[i];
        const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
        uint32_t out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&rw[j]));
            const __half2 hv = __floats2half2_rn(y[2 * j] + r.x, y[2 * j + 1] + r.y);
            out[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const uint4 hv4 = make_uint4(out[0], out[1], out[2], out[3]);
        hrow[i] = hv4;
        hs[i] = hv4;
    }
    __syncthreads();
    if (warp == 0) {
        float ss = 0.f;
        for (int i = lane; i < nv; i += 32) {
            const uint4 v = hs[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
                ss = fmaf(f.x, f.x, ss);
                ss = fmaf(f.y, f.y, ss);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) r_row = rsqrtf(ss / (float)hidden + eps);
    }
    __syncthreads();
    const float r = r_row;
    uint4* dst = reinterpret_cast<uint4*>(n + (size_t)row * hidden);
    const uint4* gv = reinterpret_cast<const uint4*>(gamma);
    for (int i = lane + 32 * warp; i < nv; i += 32 * kRnWarps) {
        const uint4 v = hs[i];
        const uint4 g = gamma ? gv[i] : make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
            const float2 gg = __half22float2(*reinterpret_cast<const __half2*>(&gw[j]));
            const __half2 hv = __floats2half2_rn(f.x * r * gg.x, f.y * r * gg.y);
            o[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

struct PrefillLayout {
    size_t n = 0, q = 0, k = 0, v = 0, act = 0, part = 0, part_bytes = 0, total = 0;
    size_t cs = 0, a = 0;  // with attention: the chunk's rotation table and attention output
};

PrefillLayout prefill_layout(const Dims& d, int chunk, const q4_layer_table* t) {
    PrefillLayout l;
    size_t off = 0;
    auto take = [&](size_t elems) {
        size_t o = off;
        off = align256(off + elems * 2);
        return o;
    };
    const size_t C = (size_t)chunk;
    l.n = take(C * d.hidden);
    l.q = take(C * (d.qN > 0 ? d.qN : 1));
    l.k = take(C * (d.kvN > 0 ? d.kvN : 1));
    l.v = take(C * (d.kvN > 0 ? d.kvN : 1));
    l.act = take(C * (d.ffn > 0 ? d.ffn : 1));
    // fp32 partial sums for the GEMMs that split K (small chunks leave output tiles for few SMs)
    size_t pb = 0;
    for (int i = 0; i < d.L; ++i) {
        const q4_layer_weights& w = t->layers[i];
        const size_t s[6] = {gemm_split_bytes(chunk, w.q.N, w.q.K, false),
                             gemm_split_bytes(chunk, w.k.N, w.k.K, false),
                             gemm_split_bytes(chunk, w.v.N, w.v.K, false),
                             gemm_split_bytes(chunk, w.o.N, w.o.K, false),
                             gemm_split_bytes(chunk, w.gate.N, w.gate.K, true),
                             gemm_split_bytes(chunk, w.down.N, w.down.K, false)};
        for (size_t b : s) pb = b > pb ? b : pb;
    }
    l.part_bytes = pb;
    l.part = take(pb / 2 + 1);
    if (d.attn) {
        l.cs = take(prefill_attn_cs_bytes(chunk, d.hd, d.qN / d.hd) / 2);
        l.a = take(C * (d.qN > 0 ? d.qN : 1));
    }
    l.total = off;
    return l;
}

q4_status prefill_dims(const q4_layer_table* t, int chunk, Dims* d) {
    if (!t) return fail(Q4_ERR_INVALID_ARG, "table is NULL");
    if (chunk < 1) return fail(Q4_ERR_INVALID_ARG, "chunk=%d", chunk);
    q4_layer_table c = *t;
    c.M = 1;  // the prefill ignores M
    return table_dims(&c, d);
}

q4_status gemm_of(const q4_linear& w, const q4_linear* up, const uint16_t* X, int M, void* Y,
                  const uint16_t* residual, void* part, size_t part_bytes, cudaStream_t s) {
    q4_gemm_desc g = {};
    g.M = M;
    g.X = X;
    g.w = w;
    if (up) g.up = *up;
    g.mode = up ? Q4_GEMV_GLU : Q4_GEMV_PLAIN;
    g.out_dtype = Q4_F16;
    g.Y = Y;
    g.residual = residual;
    g.workspace = part;
    g.workspace_bytes = part_bytes;
    return gemm_launch(&g, reinterpret_cast<q4_stream_t>(s));
}

// PLAIN GEMM with an fp16 residual (h = h + W x, in place) whose split-K
// partials, when it splits, are left for reduce_norm_rows_kernel (*kparts > 1).
q4_status gemm_res_parts(const q4_linear& w, const uint16_t* X, int M, uint16_t* h, void* part, size_t part_bytes,
                         cudaStream_t s, int* kparts) {
    q4_gemm_desc g = {};
    g.M = M;
    g.X = X;
    g.w = w;
    g.mode = Q4_GEMV_PLAIN;
    g.out_dtype = Q4_F16;
    g.Y = h;
    g.residual = h;
    g.workspace = part;
    g.workspace_bytes = part_bytes;
    return gemm_launch_parts(&g, reinterpret_cast<q4_stream_t>(s), kparts);
}

}  // namespace
}  // namespace q4i

using namespace q4i;

extern "C" {

size_t q4_prefill_workspace_bytes(const q4_layer_table* table, int chunk) {
    clear_error();
    Dims d;
    if (prefill_dims(table, chunk, &d) != Q4_OK) return 0;
    return prefill_layout(d, chunk, table).total;
}

q4_status q4_prefill_buffers(const q4_layer_table* table, int chunk, void* workspace, q4_prefill_buffers_t* out) {
    clear_error();
    if (!out || !workspace) return fail(Q4_ERR_INVALID_ARG, "out or workspace is NULL");
    Dims d;
    q4_status st = prefill_dims(table, chunk, &d);
    if (st != Q4_OK) return st;
    const PrefillLayout l = prefill_layout(d, chunk, table);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    out->n = reinterpret_cast<uint16_t*>(ws + l.n);
    out->q = reinterpret_cast<uint16_t*>(ws + l.q);
    out->k = reinterpret_cast<uint16_t*>(ws + l.k);
    out->v = reinterpret_cast<uint16_t*>(ws + l.v);
    out->act = reinterpret_cast<uint16_t*>(ws + l.act);
    out->a = d.attn ? reinterpret_cast<uint16_t*>(ws + l.a) : nullptr;
    return Q4_OK;
}

q4_status q4_prefill(const q4_layer_table* table, uint16_t* h, int T, int chunk, void* logits, void* workspace,
                     size_t workspace_bytes, q4_stream_t stream) {
    clear_error();
    Dims d;
    q4_status st = prefill_dims(table, chunk, &d);
    if (st != Q4_OK) return st;
    if (T < 0) return fail(Q4_ERR_INVALID_ARG, "T=%d", T);
    if (T > 0 && !h) return fail(Q4_ERR_INVALID_ARG, "h is NULL");
    if (!aligned16(h) || (logits && !aligned16(logits))) return fail(Q4_ERR_MISALIGNED, "h and logits must be 16-byte aligned");
    const PrefillLayout l = prefill_layout(d, chunk, table);
    if (!workspace) return fail(Q4_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return fail(Q4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (workspace_bytes < l.total) return fail(Q4_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, l.total);
    for (int i = 0; i < d.L; ++i) {
        const q4_layer_weights& w = table->layers[i];
        if (w.q.N % 128 || w.k.N % 128 || w.v.N % 128 || w.o.N % 128 || w.gate.N % 128 || w.down.N % 128)
            return fail(Q4_ERR_UNSUPPORTED, "layer %d: the prefill GEMM needs output widths that are multiples of 128", i);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float eps = table->norm_eps > 0.f ? table->norm_eps : 1e-6f;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint16_t* n = reinterpret_cast<uint16_t*>(ws + l.n);
    uint16_t* q = reinterpret_cast<uint16_t*>(ws + l.q);
    uint16_t* k = reinterpret_cast<uint16_t*>(ws + l.k);
    uint16_t* v = reinterpret_cast<uint16_t*>(ws + l.v);
    uint16_t* act = reinterpret_cast<uint16_t*>(ws + l.act);
    void* part = ws + l.part;
    const size_t pb = l.part_bytes;
    void* cs = ws + l.cs;
    uint16_t* a_buf = reinterpret_cast<uint16_t*>(ws + l.a);
    const int H = d.hidden;
    for (int t0 = 0; t0 < T; t0 += chunk) {
        const int C = T - t0 < chunk ? T - t0 : chunk;
        uint16_t* hc = h + (size_t)t0 * H;
        const int nb = (C + 7) / 8;
        if (d.attn && (st = prefill_attn_table(table->pos, t0, C, d.hd, table->rope_theta, cs, s)) != Q4_OK)
            return st;
        bool n_ready = false;  // the previous layer's down launch already wrote this layer's n
        // the fused reduce + RMSNorm keeps a row in (default-sized) shared memory
        const bool fuse_rn = (size_t)H * 2 <= 48 * 1024;
        for (int i = 0; i < d.L; ++i) {
            const q4_layer_weights& w = table->layers[i];
            cudaError_t e;
            if (!n_ready) {
                rmsnorm_rows_kernel<<<nb, 256, 0, s>>>(hc, w.attn_norm, n, C, H, eps);
                if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
            }
            n_ready = false;
            // q, k and v as one launch (their units share the GPU: at 512
            // tokens each alone fills a quarter to half of it) unless one
            // of them would split K
            if (gemm_split_bytes(C, w.q.N, w.q.K, false) == 0 && gemm_split_bytes(C, w.k.N, w.k.K, false) == 0 &&
                gemm_split_bytes(C, w.v.N, w.v.K, false) == 0) {
                const q4_linear qkv[3] = {w.q, w.k, w.v};
                void* const out[3] = {q, k, v};
                if ((st = gemm_launch_multi(qkv, out, 3, n, C, reinterpret_cast<q4_stream_t>(s))) != Q4_OK) return st;
            } else {
                if ((st = gemm_of(w.q, nullptr, n, C, q, nullptr, part, pb, s)) != Q4_OK) return st;
                if ((st = gemm_of(w.k, nullptr, n, C, k, nullptr, part, pb, s)) != Q4_OK) return st;
                if ((st = gemm_of(w.v, nullptr, n, C, v, nullptr, part, pb, s)) != Q4_OK) return st;
            }
            const uint16_t* o_in = q;
            if (d.attn) {
                if ((st = prefill_attn_enqueue(q, k, v, w.k_cache, w.v_cache, table->pos, t0, C, w.q.N / d.hd,
                                               w.k.N / d.hd, d.hd, d.max_seq, cs, a_buf, s)) != Q4_OK)
                    return st;
                o_in = a_buf;
            }
            // h' = h + Wo a and n' = rms(h') ffn_norm: when the GEMM splits K,
            // one kernel adds its partials to h and normalises (no separate
            // reduce and RMSNorm launches)
            int kp = 1;
            if (!fuse_rn) {
                if ((st = gemm_of(w.o, nullptr, o_in, C, hc, hc, part, pb, s)) != Q4_OK) return st;
            } else if ((st = gemm_res_parts(w.o, o_in, C, hc, part, pb, s, &kp)) != Q4_OK) {
                return st;
            }
            if (kp > 1)
                reduce_norm_rows_kernel<<<C, 32 * kRnWarps, (size_t)H * 2, s>>>(static_cast<const float*>(part), kp,
                                                                                hc, w.ffn_norm, n, C, H, eps);
            else
                rmsnorm_rows_kernel<<<nb, 256, 0, s>>>(hc, w.ffn_norm, n, C, H, eps);
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
            if ((st = gemm_of(w.gate, &w.up, n, C, act, nullptr, part, pb, s)) != Q4_OK) return st;
            // h = h' + Wdown act; when it splits K (and a layer follows), the
            // next layer's attention RMSNorm goes into the same kernel
            if (fuse_rn && i + 1 < d.L) {
                if ((st = gemm_res_parts(w.down, act, C, hc, part, pb, s, &kp)) != Q4_OK) return st;
                if (kp > 1) {
                    reduce_norm_rows_kernel<<<C, 32 * kRnWarps, (size_t)H * 2, s>>>(
                        static_cast<const float*>(part), kp, hc, table->layers[i + 1].attn_norm, n, C, H, eps);
                    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rmsnorm launch");
                    n_ready = true;
                }
            } else if ((st = gemm_of(w.down, nullptr, act, C, hc, hc, part, pb, s)) != Q4_OK) {
                return st;
            }
        }
    }
    if (d.attn && T > 0 && (st = pos_advance(table->pos, s, T)) != Q4_OK) return st;
    if (logits && T > 0) {
        q4_gemv_desc g = {};
        g.M = 1;
        g.K = H;
        g.x = h + (size_t)(T - 1) * H;
        g.n_segments = 1;
        g.seg[0].Wq = table->lm_head.Wq;
        g.seg[0].scales = table->lm_head.scales;
        g.seg[0].biases = table->lm_head.biases;
        g.seg[0].N = table->lm_head.N;
        g.seg[0].y = logits;
        g.out_dtype = table->logits_dtype;
        g.mode = Q4_GEMV_PLAIN;
        g.x_rmsnorm = 1;
        g.norm_weight = table->final_norm;
        g.norm_eps = eps;
        if ((st = validate_gemv(g)) != Q4_OK) return st;
        return launch_gemv(g, s, false, true);
    }
    return Q4_OK;
}

size_t q4_decode_workspace_bytes(const q4_layer_table* table) {
    clear_error();
    Dims d;
    if (table_dims(table, &d) != Q4_OK) return 0;
    return layout_of(d).total;
}

q4_status q4_decode_buffers(const q4_layer_table* table, q4_decode_buffers_t* out) {
    clear_error();
    if (!out) return fail(Q4_ERR_INVALID_ARG, "out is NULL");
    Dims d;
    q4_status st = table_dims(table, &d);
    if (st != Q4_OK) return st;
    if (!table->workspace) return fail(Q4_ERR_INVALID_ARG, "workspace is NULL");
    const Layout l = layout_of(d);
    uint8_t* ws = static_cast<uint8_t*>(table->workspace);
    out->h = reinterpret_cast<uint16_t*>(ws + l.h);
    out->h_mid = reinterpret_cast<uint16_t*>(ws + l.h_mid);
    out->q = reinterpret_cast<uint16_t*>(ws + l.q);
    out->k = reinterpret_cast<uint16_t*>(ws + l.k);
    out->v = reinterpret_cast<uint16_t*>(ws + l.v);
    out->act = reinterpret_cast<uint16_t*>(ws + l.act);
    out->a = d.attn ? reinterpret_cast<uint16_t*>(ws + l.a) : nullptr;
    return Q4_OK;
}

q4_status q4_decode_step(q4_layer_table* table, const uint16_t* x, void* logits, q4_stream_t stream) {
    clear_error();
    if (!table) return fail(Q4_ERR_INVALID_ARG, "table is NULL");
    if (!x || !logits) return fail(Q4_ERR_INVALID_ARG, "x or logits is NULL");
    if (!aligned16(x) || !aligned16(logits)) return fail(Q4_ERR_MISALIGNED, "x and logits must be 16-byte aligned");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    Plan* p = static_cast<Plan*>(table->plan);
    if (!p) {
        // First call: validate, lay out the workspace, build the stage list.
        Dims d;
        q4_status st = table_dims(table, &d);
        if (st != Q4_OK) return st;
        const Layout l = layout_of(d);
        if (!table->workspace) return fail(Q4_ERR_INVALID_ARG, "workspace is NULL");
        if ((reinterpret_cast<uintptr_t>(table->workspace) & 255u) != 0)
            return fail(Q4_ERR_MISALIGNED, "workspace must be 256-byte aligned");
        if (table->workspace_bytes < l.total)
            return fail(Q4_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", table->workspace_bytes, l.total);
        p = new Plan();
        cudaGetDevice(&p->device);
        p->dims = d;
        p->lay = l;
        p->layers.assign(table->layers, table->layers + table->n_layers);
        p->lm_head = table->lm_head;
        p->final_norm = table->final_norm;
        p->eps = table->norm_eps > 0.f ? table->norm_eps : 1e-6f;
        p->logits_dtype = table->logits_dtype;
        p->workspace = table->workspace;
        p->workspace_bytes = table->workspace_bytes;
        p->flags = table->flags;
        p->pos = table->pos;
        p->rope_theta = table->rope_theta;
        p->tagged_mode = (table->flags & Q4_DECODE_TAGGED) != 0;
        for (int l = 0; l < d.L && p->tagged_mode; ++l) {
            const q4_layer_weights& w = table->layers[l];
            p->tagged_mode = gemv_fits_unsplit(d.M, d.hidden) && gemv_fits_unsplit(d.M, w.o.K) &&
                             gemv_fits_unsplit(d.M, w.down.K);
        }
        table->plan = p;
    }
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev != p->device) return fail(Q4_ERR_INVALID_ARG, "table was planned on device %d, current is %d", p->device, dev);
    if (p->stages.empty() || x != p->x_key || logits != p->logits_key) {
        build_stages(*p, x, logits);
        p->x_key = x;
        p->logits_key = logits;
        drop_graph(*p);
        p->persistent = false;
        p->fused = false;
        if (p->dims.step) {
            q4_status st = plan_fused(*p, x, s);
            if (st != Q4_OK) return st;
        }
        if (p->flags & Q4_DECODE_PERSISTENT) {
            const int n = (int)p->stages.size();
            p->params_host.assign((size_t)n * gemv_params_bytes(), 0);
            bool fits = false;
            q4_status st = persistent_plan(p->stages.data(), p->tagged.data(), n, p->params_host.data(), &p->geom, &fits);
            if (st != Q4_OK) return st;
            if (fits) {
                cudaError_t e = cudaMemcpyAsync(static_cast<uint8_t*>(p->workspace) + p->lay.params,
                                                p->params_host.data(), p->params_host.size(), cudaMemcpyHostToDevice, s);
                if (e != cudaSuccess) return cuda_fail(e, "uploading the stage parameters");
                p->persistent = true;
            }
        }
    }
    if ((p->tagged_mode || p->persistent) && !p->tagged_ready) {
        // Once, on the caller's stream and outside any capture: tags start at
        // 1, so zeroed words never look ready; the step counter starts at 0.
        cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(p->workspace) + p->lay.tagged_begin, 0,
                                        p->lay.total - p->lay.tagged_begin, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the tagged activations");
        p->tagged_ready = true;
    }
    if (p->fused && !p->step_ready) {
        // Once, on the caller's stream and outside any capture: exchange tags
        // start at 1, so zeroed words never look current; the step counter starts at 0.
        cudaError_t e = cudaMemsetAsync(static_cast<uint8_t*>(p->workspace) + p->lay.xch, 0,
                                        p->lay.step_end - p->lay.xch, s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the exchange region");
        p->step_ready = true;
    }
    if (p->persistent)
        return persistent_launch(p->geom, static_cast<uint8_t*>(p->workspace) + p->lay.params, s);
    if (p->flags & Q4_DECODE_NO_GRAPH) return enqueue_stages(*p, s);
    if (!p->exec) {
        q4_status st = capture(*p);
        if (st != Q4_OK) return st;
    }
    cudaError_t e = cudaGraphLaunch(p->exec, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGraphLaunch");
    return Q4_OK;
}

int q4_decode_path(const q4_layer_table* table) {
    clear_error();
    if (!table || !table->plan) return 0;
    const Plan* p = static_cast<const Plan*>(table->plan);
    if (p->stages.empty()) return 0;
    if (p->fused) return 3;
    if (p->persistent) return 2;
    return 1;
}

q4_status q4_layer_table_release(q4_layer_table* table) {
    clear_error();
    if (!table) return fail(Q4_ERR_INVALID_ARG, "table is NULL");
    Plan* p = static_cast<Plan*>(table->plan);
    if (p) {
        drop_graph(*p);
        if (p->capture_stream) cudaStreamDestroy(p->capture_stream);
        delete p;
        table->plan = nullptr;
    }
    return Q4_OK;
}

}  // extern "C"
