/*
 * q4.h -- C ABI of the GB300 Q4 group-64 decode-matmul library.
 *
 * The library computes the decode-time matrix products of a 4-bit
 * group-quantised LLM with the dequantisation folded into the inner loop of
 * each kernel, never writing dequantised weights to memory (BaseRT: optimal
 * LLM inference on Apple Silicon with native Metal, §3.3 "Kernel fusion and
 * specialisation": dedicated GEMV (decode, M=1) and GEMM (prefill, M>1)
 * kernels per quantisation format, dequantisation integrated into the inner
 * loop, traffic reduced by the compression ratio).  It exposes a C API for
 * cross-language use (BaseRT §3, "BaseRT runtime design") and allocates
 * nothing on its hot calls: every buffer belongs to the caller (BaseRT §3.2,
 * "Zero-allocation decode loop"); error text lives in a static thread-local
 * buffer (same section).
 *
 * Conventions for every call
 * --------------------------
 * - Pointers are DEVICE pointers on the current CUDA device unless stated.
 *   The caller owns every buffer; the library never frees or keeps them
 *   beyond the call, except where a call's comment says so.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *   default stream).  They return after enqueueing.  A launch failure returns
 *   Q4_ERR_CUDA.  A condition detected on the device (a bounded wait that ran
 *   out, or bad routing offsets) is latched in a device error word and
 *   reported by q4_device_status().
 * - On any error the call enqueues nothing and q4_last_error() describes it.
 * - "fp16" means IEEE binary16 bit patterns passed as uint16_t.
 *
 * Q4 storage format (one matrix W of N output rows by K inputs, y = W x)
 * -----------------------------------------------------------------------
 * - Wq:     uint32 [N][K/8], row-major.  Weight k of row n is the 4-bit code
 *           q in bits 4*(k%8) .. 4*(k%8)+3 of word k/8 (lowest nibble first).
 * - scales: fp16 [N][K/64], row-major; biases: fp16 [N][K/64].
 * - w[n][k] = scales[n][k/64] * q + biases[n][k/64], q in 0..15.
 * - K must be a positive multiple of 64.  Wq, scales, biases and x must be
 *   16-byte aligned.
 * The pages name MLX/GGUF 4-bit files (MetalRT: AI inference performance
 * optimisation on Apple Silicon, §2.1) but print no bit layout; this is the
 * affine scale+bias group format with the layout fixed above.
 */
#ifndef Q4_H
#define Q4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *q4_stream_t;

typedef enum q4_status {
    Q4_OK = 0,
    Q4_ERR_INVALID_ARG = -1,  /* null pointer, bad size or shape */
    Q4_ERR_UNSUPPORTED = -2,  /* valid request the library does not serve (e.g. M > 8) */
    Q4_ERR_MISALIGNED = -3,   /* a pointer or leading dimension breaks the alignment rule */
    Q4_ERR_CUDA = -4,         /* a CUDA runtime call failed; see q4_last_error() */
    Q4_ERR_TIMEOUT = -5,      /* a device-side bounded wait ran out (reported by q4_device_status) */
    Q4_ERR_NO_DEVICE = -6,    /* no usable sm_103 device is current */
    Q4_ERR_DEVICE_CHECK = -7  /* device-side validation rejected data (e.g. routing offsets) */
} q4_status;

typedef enum q4_dtype { Q4_F32 = 0, Q4_F16 = 1 } q4_dtype;

/* Text of the last error raised on the calling thread ("" if none).  Static,
 * thread-local storage: valid until this thread's next library call. */
const char *q4_last_error(void);

/* Fixed text for a status code. */
const char *q4_status_string(q4_status status);

/* Library ABI version (major*100 + minor). */
int q4_version(void);

/* Synchronise `stream`, then read and clear the current device's error word.
 * Returns Q4_OK, Q4_ERR_TIMEOUT, Q4_ERR_DEVICE_CHECK or Q4_ERR_CUDA. */
q4_status q4_device_status(q4_stream_t stream);

/* Failure-detection self-test (no counterpart in the pages): enqueues one
 * small kernel on `stream` that runs the library's two bounded device waits
 * against conditions nothing will ever satisfy -- a tagged activation word
 * that no stage writes and an mbarrier no thread arrives on.  Each wait gives
 * up after its limit (2 s), latches Q4_ERR_TIMEOUT into the device error word
 * and returns, so the kernel ends normally (~4 s) and the context stays
 * usable; q4_device_status() then reports Q4_ERR_TIMEOUT.  No fault, trap or
 * endless loop is involved.  Returns launch errors only. */
q4_status q4_selftest_expired_wait(q4_stream_t stream);

/* ------------------------------------------------------------------------ *
 * 1. q4_gemv -- y[m][n] = sum_k w[n][k] * x[m][k], m < M, n < N.
 *
 * Decode matmul with the dequantisation inside the dot product (BaseRT §3.3).
 * x: fp16 [M][K] row-major.  y: fp32 [M][N] row-major (written, not read).
 * 1 <= M <= 8 (M = 1 is single-token decode; 2..8 is batched decode, each
 * weight is read once and used M times).  N >= 1.  Accumulation is fp32; the
 * per-element error is below 1e-3 * sum_k |w x| and the sum order is fixed,
 * so repeated calls give identical bits.
 * ------------------------------------------------------------------------ */
q4_status q4_gemv(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                  const uint16_t *x, float *y, int M, int N, int K, q4_stream_t stream);

/* 1b. q4_gemv8 -- the same product for 8-bit codes (BaseRT §3.3 and §4.1:
 * the runtime's kernels cover 2- to 16-bit formats; Q4 and Q8 are the ones
 * evaluated).  Wq: uint32 [N][K/4], 16-byte aligned; code k of row n is
 * bits 8*(k%4) .. 8*(k%4)+7 of word k/4 (lowest byte first), q in 0..255;
 * scales, biases: fp16 [N][K/64]; w = s*q + b.  Everything else (x, y, M, N,
 * K, alignment, errors, accuracy, determinism) as q4_gemv. */
q4_status q4_gemv8(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                   const uint16_t *x, float *y, int M, int N, int K, q4_stream_t stream);

/* ------------------------------------------------------------------------ *
 * 2. q4_gemv_ex -- several matrices that share one input x in ONE launch,
 *    with fused epilogues.
 *
 * BaseRT §3.3 fuses operator sequences of the attention path and the FFN
 * into single kernels (one launch and one global round trip saved each);
 * "Mac on-device AI performance breakthrough" §2.2 merges the Q, K, V
 * products into one operation.  Segments i < n_segments each compute
 * y_i = W_i x for the same x and K:
 *
 *   mode Q4_GEMV_PLAIN: y_i written in out_dtype.  If residual_i is set
 *     (out_dtype must be Q4_F16) the stored value is fp16(acc + residual)
 *     with the add in fp32; residual_i may alias y_i.
 *   mode Q4_GEMV_GLU: exactly two segments of equal N: seg[0] = gate,
 *     seg[1] = up.  Stores fp16( SiLU(gate x) * (up x) ) into seg[0].y
 *     (fp32 SiLU and product, one fp16 rounding); seg[1].y is ignored;
 *     out_dtype must be Q4_F16 and residuals must be NULL.
 *
 * Output rows of segment i are y_i[m*ldy_i + n]; ldy 0 means N_i.  x rows
 * are x[m*ldx + k]; ldx 0 means K; ldx must be a multiple of 8.
 *
 * x_rmsnorm = 1 applies an RMSNorm to each x row as it is loaded, the first
 * operation of a pre-norm transformer sublayer fused into the matmul (BaseRT
 * §3.3 fuses operator sequences of the attention path and the FFN; MetalRT
 * §5.1 keeps the norm in fp32):
 *     xn[m][k] = x[m][k] / sqrt(mean_k x[m][k]^2 + norm_eps) * norm_weight[k]
 * in fp32, used unrounded.  norm_weight: fp16 [K], NULL means all ones.
 * ------------------------------------------------------------------------ */
#define Q4_MAX_SEGMENTS 4

typedef enum q4_gemv_mode { Q4_GEMV_PLAIN = 0, Q4_GEMV_GLU = 1 } q4_gemv_mode;

typedef struct q4_segment {
    const uint32_t *Wq;
    const uint16_t *scales;
    const uint16_t *biases;
    int N;
    int ldy;
    void *y;
    const uint16_t *residual;
} q4_segment;

typedef struct q4_gemv_desc {
    int M;
    int K;
    const uint16_t *x;
    int ldx;
    int n_segments;
    q4_segment seg[Q4_MAX_SEGMENTS];
    q4_dtype out_dtype;
    q4_gemv_mode mode;
    int x_rmsnorm;
    const uint16_t *norm_weight;
    float norm_eps;
    int flags; /* Q4_GEMV_EARLY_WEIGHTS or 0 */
} q4_gemv_desc;

/* Launch with programmatic dependent launch and stream the weight tiles
 * before the previous kernel on the stream completes (x, residuals and y
 * still wait for it).  The caller promises that no kernel earlier on the
 * stream writes Wq, scales or biases -- true for a model's weights between
 * decode steps.  Back-to-back GEMVs then overlap one launch's weight stream
 * with the previous launch's tail (BaseRT §3: low-overhead dispatch). */
#define Q4_GEMV_EARLY_WEIGHTS 1

q4_status q4_gemv_ex(const q4_gemv_desc *desc, q4_stream_t stream);

/* q4_gemv for b-bit codes, b in {2, 3, 4, 5, 6, 8} (BaseRT §3.3 and §4.1:
 * a kernel per quantisation format, 2 to 16 bits).  Wq: uint32 [N][K*b/32];
 * code k of a row occupies bits b*k .. b*k+b-1 of the row's little-endian bit
 * stream (lowest bit first; a code crossing a word boundary continues in the
 * low bits of the next word) -- for b = 4 and 8 exactly the layouts of
 * q4_gemv and q4_gemv8.  scales, biases: fp16 [N][K/64]; w = s * q + b with
 * q in 0..2^b-1.  b = 2, 3, 5, 6 need M = 1 (else Q4_ERR_UNSUPPORTED);
 * b = 7 or outside 2..8 returns Q4_ERR_INVALID_ARG.  Other rules as
 * q4_gemv. */
q4_status q4_gemv_bits(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                       const uint16_t *x, float *y, int M, int N, int K, int bits,
                       q4_stream_t stream);

/* ------------------------------------------------------------------------ *
 * 3. q4_decode_step -- one decode step over a whole layer stack.
 *
 * Runs the matmul part of a transformer decode step as one stream of fused
 * GEMV launches: per layer a fused QKV launch, the o projection with the
 * residual add, a fused gate/up launch with the SiLU*up epilogue, the down
 * projection with the residual add; then lm_head.  BaseRT §3 removes
 * per-operator dispatch from the decode hot path and §3.1 describes the model
 * by a data descriptor the engine never branches on -- here that descriptor is
 * q4_layer_table.  The pages do not fix the dataflow between the GEMVs; this
 * library computes a pre-norm layer, for each layer, with h = x before the
 * first layer and rms(v) = v / sqrt(mean(v^2) + norm_eps):
 *
 *   n   = rms(h) * attn_norm                      (fused into the QKV launch)
 *   q, k, v = fp16(Wq n), fp16(Wk n), fp16(Wv n)  (k, v kept in the workspace)
 *   h'  = fp16(h + Wo q)          (q stands in for the attention output)
 *   n'  = rms(h') * ffn_norm                      (fused into the gate/up launch)
 *   act = fp16(SiLU(Wgate n') * (Wup n'))
 *   h   = fp16(h' + Wdown act)
 *
 * and finally logits = Wlm (rms(h) * final_norm) in logits_dtype.  By default
 * q stands in for the attention output (the matmul path alone).  With
 * Q4_DECODE_ATTENTION (M = 1), after the QKV stage the new key, rotated by
 * RoPE at position p = *table->pos, and the new value are written to position
 * p of the layer's caches, and a = fp16(attention of the RoPE-rotated q over
 * positions 0..p) replaces q as the input of o (section 6 describes the
 * attention); the step ends with *pos += 1.  A position outside
 * [0, max_seq) latches Q4_ERR_DEVICE_CHECK and leaves the caches alone.
 *
 * The first call on a table validates it and plans the step.  By default
 * each stage is its own kernel launch: the first call captures them into a
 * CUDA graph (programmatic dependent launch between the kernels, so each
 * kernel's weight stream starts before its predecessor ends); later calls
 * replay the graph.  With Q4_DECODE_PERSISTENT a step is ONE cooperative
 * kernel launch instead: one CTA per SM walks every stage in order, streaming
 * each stage's weights ahead through shared memory while it waits for that
 * stage's input; a stage starts once a completion counter in the workspace
 * shows every earlier stage done, and reads its input as tagged words
 * (below), instead of kernel boundaries; the per-stage kernel parameters are uploaded
 * into the workspace on `stream` on the first call and after a pointer
 * change, and calls on one table must then be ordered on one stream.  If the
 * step does not fit one persistent launch (x of the widest stage plus two
 * weight tiles exceeds shared memory) the flag is ignored.  A call with
 * different x or logits
 * pointers re-plans (and re-captures).  In the persistent launch, and with
 * Q4_DECODE_TAGGED for per-stage launches, activations pass from stage to
 * stage as 32-bit words holding the fp16 value and a 16-bit tag naming the
 * step and the writing stage; a stage polls the words it reads instead of
 * waiting for the whole previous kernel to finish.  The workspace therefore
 * also holds the stage parameters, these tagged copies and the step and
 * completion counters;
 * the tagged region is cleared on the first such call (on `stream`), and the
 * workspace must not be shared with another table while in use.  Host memory
 * for the plan is allocated on that first call
 * (load time); replays allocate nothing.  x: fp16 [M][hidden].  logits:
 * [M][vocab].  The workspace (device, >= q4_decode_workspace_bytes) holds the
 * activations; after a step it holds the LAST layer's q, k, v, h', act and the
 * final h (see q4_decode_buffers).  Weights must not change between calls
 * without q4_layer_table_release() (the plan caches their pointers).
 *
 * With Q4_DECODE_CLUSTERED (M = 1, no attention, every layer of the same
 * shape, hidden, q.N and gate.N multiples of 512, and a device that holds at
 * least two 16- or 8-CTA clusters of one CTA per SM at once; otherwise the
 * flag is ignored) the layer stack is ONE launch of thread-block clusters
 * (sized so that all of them are resident at once), the k and v rows a
 * second launch on the SMs the clusters leave free (it rebuilds each layer's
 * input from the clusters' exchange words, in their order, so k and v are the
 * bits the clusters would compute), and lm_head a third: cluster c owns a
 * block of whole 64-row groups of q (and of act), its CTAs share those
 * values through distributed shared memory, and each CTA multiplies its
 * rows of the matching column block of
 * Wo (Wdown); the clusters' partial sums meet in the workspace as 64-bit
 * words tagged with the step and the exchange, every cluster adds them in
 * the same fixed order and rounds h' (h) to fp16 as above -- two grid-wide
 * hand-offs per layer instead of four kernel boundaries.  The o / down
 * products are therefore summed in a different order than by the per-stage
 * launches (same bound against the oracle, different last bits), and the
 * step's results are the same bits run to run.  The workspace then also
 * holds the layer table, the o / down tensor maps and the exchange words
 * (zeroed on the first call, on `stream`; q4_decode_workspace_bytes counts
 * them when the table asks for the flag), and calls on one table must be
 * ordered on one stream.
 * ------------------------------------------------------------------------ */
typedef struct q4_linear {
    const uint32_t *Wq;
    const uint16_t *scales;
    const uint16_t *biases;
    int N; /* outputs */
    int K; /* inputs, multiple of 64 */
} q4_linear;

typedef struct q4_layer_weights {
    q4_linear q, k, v, o, gate, up, down;
    const uint16_t *attn_norm; /* fp16 [hidden] RMSNorm weight before QKV; NULL = ones */
    const uint16_t *ffn_norm;  /* fp16 [hidden] RMSNorm weight before gate/up; NULL = ones */
    uint16_t *k_cache;         /* Q4_DECODE_ATTENTION only: fp16 [k.N/head_dim][max_seq][head_dim] */
    uint16_t *v_cache;         /* likewise for the values; both 16-byte aligned */
} q4_layer_weights;

#define Q4_DECODE_NO_GRAPH 1 /* launch the kernels directly each call (no capture) */
#define Q4_DECODE_NO_PDL 2   /* no programmatic dependent launch between kernels */
#define Q4_DECODE_TAGGED 4    /* stages poll tagged activation words (see below) instead of
                                 waiting for their predecessor grid to complete */
#define Q4_DECODE_PERSISTENT 8 /* one persistent cooperative launch per step (see below);
                                  the three flags above then do not apply */
#define Q4_DECODE_ATTENTION 16 /* decode attention over each layer's KV cache replaces the
                                  a := q stand-in (see below); M must be 1, and
                                  Q4_DECODE_TAGGED / Q4_DECODE_PERSISTENT are refused */
#define Q4_DECODE_CLUSTERED 32 /* the layer stack as one launch of thread-block clusters
                                  (see below); M = 1 without attention, else ignored */

typedef struct q4_layer_table {
    int n_layers;
    int hidden;
    int M;                          /* tokens decoded together, 1..8 */
    const q4_layer_weights *layers; /* HOST array [n_layers]; read by the first call */
    q4_linear lm_head;
    const uint16_t *final_norm; /* fp16 [hidden] RMSNorm weight before lm_head; NULL = ones */
    float norm_eps;             /* 0 means 1e-6 */
    q4_dtype logits_dtype;
    void *workspace; /* device, 256-byte aligned */
    size_t workspace_bytes;
    int flags;  /* Q4_DECODE_* */
    void *plan; /* library-owned cache; zero-initialise, free with q4_layer_table_release */
    /* Q4_DECODE_ATTENTION only: */
    int head_dim;     /* 64 or 128; q.N and k.N = v.N are multiples, q heads a multiple of kv heads */
    int max_seq;      /* cache length in positions */
    float rope_theta; /* rotary base (> 1) */
    int32_t *pos;     /* device int32: the position this step writes and attends up to; the step
                         advances it by one after its last kernel */
} q4_layer_table;

/* Workspace bytes the table needs (0 if the table is malformed). */
size_t q4_decode_workspace_bytes(const q4_layer_table *table);

/* Device pointers into the workspace (all fp16, row-major [M][width]). */
typedef struct q4_decode_buffers_t {
    uint16_t *h;     /* [M][hidden] final h (input of lm_head) */
    uint16_t *h_mid; /* [M][hidden] last layer's h' */
    uint16_t *q;     /* [M][q.N] last layer's q */
    uint16_t *k;     /* [M][k.N] */
    uint16_t *v;     /* [M][v.N] */
    uint16_t *act;   /* [M][gate.N] last layer's SiLU(g)*u */
    uint16_t *a;     /* [M][q.N] last layer's attention output (Q4_DECODE_ATTENTION), else NULL */
} q4_decode_buffers_t;

q4_status q4_decode_buffers(const q4_layer_table *table, q4_decode_buffers_t *out);

q4_status q4_decode_step(q4_layer_table *table, const uint16_t *x, void *logits,
                         q4_stream_t stream);

/* How the planned step runs (no counterpart in the pages; for tests and
 * tuning): 0 = not planned yet, 1 = per-stage launches, 2 = one persistent
 * cooperative launch (Q4_DECODE_PERSISTENT), 3 = the clustered step plus
 * lm_head. */
int q4_decode_path(const q4_layer_table *table);

/* Frees the plan and its graph; the table can be used again afterwards. */
q4_status q4_layer_table_release(q4_layer_table *table);

/* ------------------------------------------------------------------------ *
 * 4. Mixture-of-experts prefill: route -> gather -> grouped GEMM (gate/up
 *    with SiLU*up, then down) -> combine.
 *
 * BaseRT's abstract and Fig. 1 report its largest lead on MoE prefill
 * (Qwen3-30B-A3B, 4-bit), and §3.4 "Prefill" runs prompts as GEMMs whose
 * arithmetic intensity grows with the sequence length.  The pages do not
 * describe routing; this library takes top-k of the fp16 router logits with
 * ties to the lower expert index, weights = softmax over the k chosen logits,
 * and sorts the T*topk routed rows stably by (expert, token, rank).
 * ------------------------------------------------------------------------ */

/* Workspace bytes q4_moe_route needs for T tokens and E experts. */
size_t q4_moe_route_workspace_bytes(int T, int E, int topk);

/* logits: fp16 [T][E].  Outputs (all written): topk_ids int32 [T][topk]
 * (descending logit), topk_weights fp32 [T][topk], offsets int32 [E+1]
 * (rows of expert e are offsets[e] .. offsets[e+1]-1), token_of / expert_of
 * int32 [T*topk] (source token and expert of each sorted row), pos int32
 * [T][topk] (sorted row of each (token, rank)).  1 <= topk <= min(E, 8),
 * E <= 256; T above 2^24 returns Q4_ERR_UNSUPPORTED before anything is
 * enqueued.  Integer outputs are bit-exact. */
q4_status q4_moe_route(const uint16_t *logits, int T, int E, int topk, int32_t *topk_ids,
                       float *topk_weights, int32_t *offsets, int32_t *token_of,
                       int32_t *expert_of, int32_t *pos, void *workspace,
                       size_t workspace_bytes, q4_stream_t stream);

/* q4_moe_route without a caller workspace: the pages have no counterpart to
 * this entry point.  It is for callers that cannot allocate device memory --
 * a plugin inside a host runtime that owns every device buffer and passes in
 * only the tensors to work on, or a serving loop whose allocations are fixed
 * at load time -- so it calls no cudaMalloc, cudaFree or allocating library
 * routine.  Same arguments, outputs and results as q4_moe_route.
 *
 * Its scratch (the per-(expert, 32-token block) counters) is a static
 * 256 KB array in the library, present on every device that loads the library
 * until the process exits: ceil(T/32) * E must not exceed 65536 (e.g. at most
 * 16384 tokens for 128 experts); larger requests (and T above 2^24) fail
 * with Q4_ERR_UNSUPPORTED before anything is enqueued.  The first call on a device looks up the
 * array's device address with that device current (a host-side set-up step;
 * make that first call before any stream capture).  Every call shares the
 * one array and the kernels write every counter they read, so nothing needs
 * clearing between calls; calls that can overlap on the GPU (other streams,
 * other host threads) race on it and must be ordered by the caller. */
q4_status q4_moe_route_noalloc(const uint16_t *logits, int T, int E, int topk, int32_t *topk_ids,
                               float *topk_weights, int32_t *offsets, int32_t *token_of,
                               int32_t *expert_of, int32_t *pos, q4_stream_t stream);

/* X_sorted[r][:] = X[token_of[r]][:] for r < R.  X: fp16 [T][K], K % 8 == 0. */
q4_status q4_moe_gather(const uint16_t *X, int T, int K, const int32_t *token_of, int R,
                        uint16_t *X_sorted, q4_stream_t stream);

typedef struct q4_moe_desc {
    int E; /* experts */
    int N; /* outputs per expert (GLU: width of gate = width of up) */
    int K; /* inputs, multiple of 64 */
    int R; /* routed rows in X */
    q4_gemv_mode mode; /* PLAIN: Y = X W_e^T; GLU: W_e holds 2N rows, gate then up,
                          Y = fp16(SiLU(X Wg^T) * (X Wu^T)) */
    q4_dtype out_dtype; /* GLU requires Q4_F16 */
} q4_moe_desc;

/* Grouped GEMM over routed experts: for every expert e and row r in
 * offsets[e] .. offsets[e+1]-1, Y[r][:] = (dequantised W_e) X[r][:].
 * Wq: uint32 [E][rows_e][K/8] with rows_e = N (PLAIN) or 2N (GLU); scales,
 * biases: fp16 [E][rows_e][K/64].  X: fp16 [R][K] sorted by expert.
 * expert_ids: int32 [R], the expert of each row (checked against offsets on
 * the device; a mismatch latches Q4_ERR_DEVICE_CHECK).  Y: [R][N].
 * Runs on the tensor cores (tcgen05, fp16 x fp16 -> fp32), weights
 * dequantised to fp16 in shared or tensor memory, never in global memory.
 * N must be a multiple of 128 (else Q4_ERR_UNSUPPORTED); Wq, scales, biases
 * and X must be 16-byte aligned (else Q4_ERR_MISALIGNED).  Launches with at
 * most 48 routed rows per expert on average take 32- or 64-token units,
 * which stage each unit's scales and biases in shared memory: a K whose
 * staging leaves no room for two pipeline stages (with 227 KB per block:
 * GLU above ~6300 (32-token units) or ~6000 (64), PLAIN above ~8800 or
 * ~8400) returns Q4_ERR_UNSUPPORTED.  Larger units take any K. */
q4_status q4_moe_gemm(const uint32_t *Wq, const uint16_t *scales, const uint16_t *biases,
                      const uint16_t *X, const int32_t *expert_ids, const int32_t *offsets,
                      void *Y, const q4_moe_desc *desc, q4_stream_t stream);

/* out[t][:] = sum_{k<topk} topk_weights[t][k] * Y[pos[t][k]][:], k in rank
 * order, fp32 accumulation.  Y: [T*topk][N] in y_dtype; out: [T][N] in
 * out_dtype. */
q4_status q4_moe_combine(const void *Y, q4_dtype y_dtype, int N, const int32_t *pos,
                         const float *topk_weights, int T, int topk, void *out,
                         q4_dtype out_dtype, q4_stream_t stream);

/* ------------------------------------------------------------------------ *
 * 5. Dense prefill: a GEMM over M tokens, and the chunked prefill of a whole
 *    layer stack.
 *
 * BaseRT §3.4 "Prefill": the prompt's tokens go through each matrix together,
 * as GEMMs whose arithmetic intensity grows with the token count, in chunks;
 * §3.3: the GEMM kernels dequantise in their inner loop like the GEMV.  The
 * GEMM here is the kernel of section 4 with one expert and no routing: codes
 * dequantised to fp16 in shared memory (w rounded once to fp16), tcgen05
 * fp16 x fp16 -> fp32 MMA, so X must be fp16.
 * ------------------------------------------------------------------------ */

typedef struct q4_gemm_desc {
    int M;                     /* tokens: rows of X and Y, >= 0 */
    const uint16_t *X;         /* fp16 [M][K], K = w.K; 16-byte aligned */
    q4_linear w;               /* the [N][K] matrix (PLAIN) or the gate matrix (GLU) */
    q4_linear up;              /* GLU: the up matrix, same N and K; ignored in PLAIN */
    q4_gemv_mode mode;         /* PLAIN: Y = X W^T; GLU: Y = fp16(SiLU(X Wg^T) * (X Wu^T)) */
    q4_dtype out_dtype;        /* GLU requires Q4_F16 */
    void *Y;                   /* [M][N] */
    const uint16_t *residual;  /* PLAIN with fp16 output only: Y = fp16(residual + X W^T),
                                  fp16 [M][N], may be the same buffer as Y; NULL = none */
    void *workspace;           /* optional, 16-byte aligned: when the output tiles do not
                                  fill the GPU and workspace_bytes >= q4_gemm_workspace_bytes,
                                  K is split over more units, fp32 partial sums go here and a
                                  second kernel adds them and applies the epilogue; NULL =
                                  never split */
    size_t workspace_bytes;
} q4_gemm_desc;

/* Workspace bytes that let q4_gemm split K for this shape (0: it would not
 * split).  Only K of 2048 or more is split, into the most parts whose units
 * still fit one wave of 152 (one per GB300 SM), at least 4 K steps of 64 per
 * unit. */
size_t q4_gemm_workspace_bytes(int M, int N, int K, q4_gemv_mode mode);

/* Y = X W^T on the tensor cores.  N must be a multiple of 128 (else
 * Q4_ERR_UNSUPPORTED); K any multiple of 64.  Wq, scales, biases and X must
 * be 16-byte aligned. */
q4_status q4_gemm(const q4_gemm_desc *desc, q4_stream_t stream);

/* Workspace bytes q4_prefill needs with chunks of `chunk` tokens (0 if the
 * table is malformed). */
size_t q4_prefill_workspace_bytes(const q4_layer_table *table, int chunk);

/* Prefill of T prompt tokens through the layer stack of `table`, `chunk`
 * tokens at a time, with the per-token dataflow of q4_decode_step (section 3):
 * per chunk and layer, an RMSNorm kernel writes n = fp16(rms(h) * attn_norm)
 * (the MMA takes fp16 operands, so n is stored in fp16 where the decode GEMV
 * keeps it in fp32), q, k, v = GEMMs of n, h' = fp16(h + Wo q), n' from h'
 * likewise, act = GLU GEMM of n', h = fp16(h' + Wdown act).
 * h: fp16 [T][hidden], 16-byte aligned; on entry the prompt's activations, on
 * return the final h (updated in place, chunk by chunk).  logits: [vocab] in
 * table->logits_dtype for the LAST token, = Wlm (rms(h[T-1]) * final_norm)
 * by the decode GEMV; NULL = none.  workspace: device, 256-byte aligned,
 * >= q4_prefill_workspace_bytes(table, chunk) bytes; after the call it holds
 * the last chunk's n', q, k, v and act (fp16 [chunk][width] each, in that
 * order, each slice 256-byte aligned), then room for the fp32 partial sums of
 * the GEMMs that split K (q4_gemm's workspace).  Every output width of the stack
 * except lm_head must be a multiple of 128 (else Q4_ERR_UNSUPPORTED).  Uses table->layers, hidden, norm_eps, lm_head,
 * final_norm and logits_dtype; ignores M, workspace and plan, and of the
 * flags reads only Q4_DECODE_ATTENTION: with it, token t of the prompt sits
 * at position p = *table->pos + t, its RoPE-rotated key and value are
 * written to position p of every layer's cache, it attends causally over
 * positions 0..p (a = fp16 attention output, replacing q as the input of o),
 * and *pos advances by T at the end, so decode steps continue the sequence;
 * positions beyond max_seq latch Q4_ERR_DEVICE_CHECK.  The prompt's attention
 * runs on the tensor cores: its scores carry the fp32 rotated query (as an
 * fp16 hi + lo pair) and its probabilities enter the value product in fp16
 * (sum kept in fp32), an error below 5e-4 * sum_j p_j |v_j| per output
 * element.  chunk >= 1, T >= 0; allocates nothing. */
q4_status q4_prefill(const q4_layer_table *table, uint16_t *h, int T, int chunk, void *logits,
                     void *workspace, size_t workspace_bytes, q4_stream_t stream);

/* Device pointers into a q4_prefill workspace (fp16, [chunk][width]): the
 * last chunk's n' (the ffn norm output), q, k, v, act and, with
 * Q4_DECODE_ATTENTION, the attention output a (else NULL). */
typedef struct q4_prefill_buffers_t {
    uint16_t *n, *q, *k, *v, *act, *a;
} q4_prefill_buffers_t;

q4_status q4_prefill_buffers(const q4_layer_table *table, int chunk, void *workspace, q4_prefill_buffers_t *out);

/* ------------------------------------------------------------------------ *
 * 6. Decode attention of one token over a preallocated KV cache.
 *
 * BaseRT §3.3 lists RoPE, attention and normalisation among the decode
 * kernels and §3.2 preallocates the KV cache; the pages print no formula.
 * RoPE (rotate-half form): for i < d/2 the pair (x_i, x_{i+d/2}) of every
 * head turns by p * theta^(-2i/d).  Query head h reads key/value head
 * h / (Hq / Hkv).  a_h = sum_j softmax_j(q_h . k_j / sqrt(d)) v_j over
 * positions j = 0..p, fp32 arithmetic, a stored in fp16.
 * ------------------------------------------------------------------------ */

typedef struct q4_attention_desc {
    const uint16_t *q;   /* fp16 [Hq * head_dim]: this token's queries, not rotated */
    const uint16_t *k;   /* fp16 [Hkv * head_dim]: its key, not rotated */
    const uint16_t *v;   /* fp16 [Hkv * head_dim]: its value */
    uint16_t *k_cache;   /* fp16 [Hkv][max_seq][head_dim]; position p receives the rotated key */
    uint16_t *v_cache;   /* fp16 [Hkv][max_seq][head_dim]; position p receives v */
    int32_t *pos;        /* device int32 p (read, not advanced); outside [0, max_seq) latches
                            Q4_ERR_DEVICE_CHECK and nothing is written */
    int n_q_heads, n_kv_heads;
    int head_dim;        /* 64 or 128 */
    int max_seq;
    float rope_theta;    /* > 1 */
    uint16_t *a;         /* fp16 [Hq * head_dim] out */
    void *workspace;     /* device, 256-byte aligned, >= q4_attention_workspace_bytes */
    size_t workspace_bytes;
} q4_attention_desc;

/* Scratch bytes for the per-chunk partial results (0 for bad sizes). */
size_t q4_attention_workspace_bytes(int n_q_heads, int head_dim, int max_seq);

/* Three kernels on `stream`: cache append, per-chunk attention, merge.  At
 * most 8 query heads per kv head (else Q4_ERR_UNSUPPORTED). */
q4_status q4_attention(const q4_attention_desc *desc, q4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4_H */
