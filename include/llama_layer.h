/*
 * llama_layer.h -- C ABI of the GB300 (sm_103a) LLaMA-style pre-norm decoder layer.
 *
 * What is computed (pages cited by title and section):
 *   h   = x + o_proj(GQA_causal(RoPE(q), RoPE(k), v)),  [q|k|v] = RMSNorm_1(x) W_qkv^T
 *   out = h + down(SiLU(RMSNorm_2(h) W_gate^T) * (RMSNorm_2(h) W_up^T))
 * "05 LLaMA3 Block — 从零件到发动机" §3.1 and §4.2 (pre-norm order, two separate norms);
 * "12 · 从 Transformer 到 LLaMA 系列" §八 (RMSNorm, SwiGLU, GQA attention, LlamaModel);
 * "第 10 章：现代 LLaMA 架构" §3 (even/odd RoPE pairs), §7 (KV-cache prefill/decode),
 * §9 (llama_block(x, position_ids, past_kv)).
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are caller-owned device memory; the library never
 *    allocates or frees device memory and never synchronises, except
 *    llama_get_device_status().  Scratch space is the caller's `workspace`, sized
 *    by the matching *_workspace_bytes() call.
 *  - Work is enqueued asynchronously on `cuda_stream` (a cudaStream_t; NULL = the
 *    legacy default stream) of the current device.
 *  - Layouts are row-major.  Linear weights use the nn.Linear layout [out, in]:
 *    wq [H*D, d], wk/wv [G*D, d], wo [d, H*D], w_gate/w_up [d_inter, d],
 *    w_down [d, d_inter].  Norm gammas are [d].  Activations are [B, S, d].
 *    The KV cache is K and V, each [B, G, max_T, D]; only G heads are stored.
 *  - Element type of activations, weights, gammas and the cache = dims.dtype
 *    (LLAMA_F32 or LLAMA_BF16); RoPE tables and logits are fp32.
 *  - Device pointers must be 16-byte aligned.
 *  - Return value: LLAMA_OK or a negative llama_status; errors never trap.
 *    Errors found on the device (a wait that timed out, a position or token out
 *    of range) are recorded in a per-device status word that
 *    llama_get_device_status() returns and clears.
 */
#ifndef LLAMA_LAYER_H
#define LLAMA_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  LLAMA_OK = 0,
  LLAMA_ERR_INVALID_ARG = -1,   /* null pointer, H % G != 0, odd D, S > max_pos or max_T, small workspace, misalignment */
  LLAMA_ERR_UNSUPPORTED = -2,   /* a shape the tiled bf16 path does not cover (e.g. D != 128, d % 128 != 0) */
  LLAMA_ERR_CUDA = -3,          /* a CUDA runtime error (launch failure, no device, ...) */
  LLAMA_ERR_TIMEOUT = -4,       /* a bounded device-side wait expired; the kernel gave up and returned */
  LLAMA_ERR_DEVICE_BOUNDS = -5, /* a device-side index check failed (position >= max_T or max_pos, token >= vocab) */
  LLAMA_ERR_SCRATCH_LIMIT = -6  /* the request needs more than llama_attention_decode_static's fixed scratch */
} llama_status;

typedef enum { LLAMA_F32 = 0, LLAMA_BF16 = 1 } llama_dtype;

/* Which head dimensions RoPE rotates together.  Both use the angle p * base^(-2i/D) for pair
 * i < D/2. */
typedef enum {
  LLAMA_ROPE_EVEN_ODD = 0, /* pairs (2i, 2i+1): "第 10 章：现代 LLaMA 架构" §2-§3 */
  LLAMA_ROPE_HALF = 1      /* pairs (i, i + D/2): "12 · 从 Transformer 到 LLaMA 系列" §八 apply_rope */
} llama_rope_style;

/* Layer hyper-parameters; mirrors the config fields of "第 10 章：现代 LLaMA 架构" §1
 * (hidden_size, intermediate_size, num_attention_heads, num_key_value_heads, rms_norm_eps). */
typedef struct {
  int32_t d_model;     /* d */
  int32_t n_heads;     /* H, query heads */
  int32_t n_kv_heads;  /* G, key/value heads; H % G == 0 ("12 · 从 Transformer 到 LLaMA 系列" §八 Attention) */
  int32_t head_dim;    /* D, even ("第 10 章：现代 LLaMA 架构" §3) */
  int32_t d_inter;     /* SwiGLU hidden size */
  float rms_eps;       /* inside the square root: rsqrt(mean(x^2) + eps) */
  int32_t dtype;       /* llama_dtype */
  int32_t rope_style;  /* llama_rope_style */
} llama_layer_dims;

/* Device pointers of one layer's parameters (no biases). */
typedef struct {
  const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} llama_layer_weights;

/* One layer's cache: K and V device buffers, each [B, G, max_T, D] of dims.dtype. */
typedef struct {
  void *k, *v;
  int32_t max_T;
} llama_kv_cache;

/* A stack of n_layers identical-shape layers plus embedding, final RMSNorm and an
 * untied LM head ("12 · 从 Transformer 到 LLaMA 系列" §八 LlamaModel). */
typedef struct {
  int32_t n_layers;
  int32_t vocab;
  llama_layer_dims dims;
  const llama_layer_weights *layers; /* HOST array of n_layers entries (device pointers inside) */
  const void *final_norm;            /* [d] */
  const void *embed;                 /* [vocab, d] */
  const void *lm_head;               /* [vocab, d] */
} llama_stack;

/* ---------------------------------------------------------------- layer entry points */

/* Workspace bytes that llama_layer_prefill needs for B sequences of S tokens. */
int llama_layer_prefill_workspace_bytes(const llama_layer_dims *dims, int32_t B, int32_t S, size_t *bytes);

/* Prefill: one decoder layer over B sequences of S tokens at positions 0..S-1
 * ("12 · 从 Transformer 到 LLaMA 系列" §八 LlamaBlock.forward; "第 10 章：现代 LLaMA 架构" §7
 * prefill).  x, out: device [B, S, d] (may not alias).  cos, sin: device fp32
 * [max_pos, D/2] tables (angle p * base^(-2i/D), see llama_rope_tables).  The
 * rotated K and the V of token s of sequence b are written to cache slot s
 * (slots [0, S) of every sequence).  Requires S <= max_pos and S <= cache.max_T. */
int llama_layer_prefill(const llama_layer_dims *dims, const llama_layer_weights *w, const void *x, void *out,
                        const float *cos, const float *sin, int32_t max_pos, llama_kv_cache cache, int32_t B,
                        int32_t S, void *workspace, size_t ws_bytes, void *cuda_stream);

/* Prefill of a chunk on top of what the cache already holds ("第 10 章：现代 LLaMA 架构" §7:
 * past_kv with position_ids = past_len + arange(T); §3 position_id = past_len): token s of
 * sequence b sits at position start[b] + s, its rotated K and its V go to cache slot
 * start[b] + s, and it attends to slots 0 .. start[b] + s (the cached ones as they are).
 * start: device int32 [B], required; lengths: device int32 [B] or NULL (all S): sequence b
 * brings lengths[b] <= S tokens and rows s >= lengths[b] of x are padding -- nothing of them
 * is stored in the cache and their rows of out are unspecified.  A sequence with start[b] < 0,
 * lengths[b] outside [0, S] or start[b] + lengths[b] beyond cache.max_T or max_pos is
 * recorded as LLAMA_ERR_DEVICE_BOUNDS and skipped.  Same workspace as llama_layer_prefill
 * (llama_layer_prefill_workspace_bytes(dims, B, S)). */
int llama_layer_prefill_chunk(const llama_layer_dims *dims, const llama_layer_weights *w, const void *x, void *out,
                              const float *cos, const float *sin, int32_t max_pos, const int32_t *start,
                              const int32_t *lengths, llama_kv_cache cache, int32_t B, int32_t S, void *workspace,
                              size_t ws_bytes, void *cuda_stream);

/* Workspace bytes that llama_layer_decode needs for B sequences and caches of max_T slots. */
int llama_layer_decode_workspace_bytes(const llama_layer_dims *dims, int32_t B, int32_t max_T, size_t *bytes);

/* Decode: one new token per sequence ("第 10 章：现代 LLaMA 架构" §7 decode and §3:
 * position_id = past_len).  x, out: device [B, d].  positions: device int32 [B];
 * token b sits at position p = positions[b], its rotated K and its V are written
 * to cache slot p, and it attends to slots 0..p (p + 1 keys; the slots below p
 * are the existing cache).  A p outside [0, min(max_T, max_pos)) is recorded as
 * LLAMA_ERR_DEVICE_BOUNDS and that sequence's cache is left untouched. */
int llama_layer_decode(const llama_layer_dims *dims, const llama_layer_weights *w, const void *x, void *out,
                       const float *cos, const float *sin, int32_t max_pos, const int32_t *positions,
                       llama_kv_cache cache, int32_t B, void *workspace, size_t ws_bytes, void *cuda_stream);

/* Workspace bytes that llama_stack_forward needs. */
int llama_stack_workspace_bytes(const llama_stack *stack, int32_t B, int32_t S, size_t *bytes);

/* Stack forward: logits = lm_head(RMSNorm_final(layers(embed[tokens]))) ("12 · 从
 * Transformer 到 LLaMA 系列" §八 LlamaModel.forward).  tokens: device int32 [B, S]
 * (a token outside [0, vocab) is recorded as LLAMA_ERR_DEVICE_BOUNDS and embeds as
 * zeros).  logits: device fp32 [B, S, vocab].  caches: NULL (K/V kept in the
 * workspace) or a HOST array of n_layers caches that receive slots [0, S). */
int llama_stack_forward(const llama_stack *stack, const int32_t *tokens, float *logits, const float *cos,
                        const float *sin, int32_t max_pos, const llama_kv_cache *caches, int32_t B, int32_t S,
                        void *workspace, size_t ws_bytes, void *cuda_stream);

/* Workspace bytes that llama_stack_decode needs for B sequences. */
int llama_stack_decode_workspace_bytes(const llama_stack *stack, int32_t B, size_t *bytes);

/* One autoregressive step of the whole model: the token tokens[b] of sequence b sits at
 * position positions[b]; its K and V go to slot positions[b] of every layer's cache and it
 * attends to slots 0..positions[b] ("第 10 章：现代 LLaMA 架构" §7 decode through every layer,
 * then the final RMSNorm and LM head of "12 · 从 Transformer 到 LLaMA 系列" §八
 * LlamaModel.forward).  tokens, positions: device int32 [B]; logits: device fp32 [B, vocab];
 * caches: HOST array of n_layers caches, each [B, G, max_T, D] on the device.  Prompt
 * lengths may differ per sequence.  A position outside a cache or max_pos, or a token
 * outside [0, vocab), is recorded as LLAMA_ERR_DEVICE_BOUNDS.  Allocation-free and
 * asynchronous, so it can be captured into a CUDA graph (see llama_stack_decode_graph). */
int llama_stack_decode(const llama_stack *stack, const int32_t *tokens, const int32_t *positions, float *logits,
                       const float *cos, const float *sin, int32_t max_pos, const llama_kv_cache *caches, int32_t B,
                       void *workspace, size_t ws_bytes, void *cuda_stream);

/* ---------------------------------------------------------------- CUDA graphs */

/* A captured decode step (opaque). */
typedef struct llama_graph llama_graph;

/* Captures one llama_stack_decode call with these arguments into a CUDA graph on the current
 * device and instantiates it.  Nothing runs: the capture records the kernels (on a private
 * stream) and validates the arguments exactly as llama_stack_decode does.  The graph keeps
 * the pointers, so each replay reads the tokens and positions then in those buffers and
 * writes the logits and cache slots they name; the stack, caches array contents and tables
 * must stay valid while the graph lives.  Creating a graph allocates the driver's graph
 * objects (no device buffers).  Not allowed while a trace (llama_trace_begin) is active.
 * *graph receives the handle, or NULL on error. */
int llama_stack_decode_graph(const llama_stack *stack, const int32_t *tokens, const int32_t *positions, float *logits,
                             const float *cos, const float *sin, int32_t max_pos, const llama_kv_cache *caches,
                             int32_t B, void *workspace, size_t ws_bytes, llama_graph **graph);

/* Replays the graph on cuda_stream (asynchronous); the current device must be the one the
 * graph was captured on. */
int llama_graph_launch(llama_graph *graph, void *cuda_stream);

/* Number of the library's kernels in one replay. */
int32_t llama_graph_kernel_count(const llama_graph *graph);

/* Releases the graph (NULL is a no-op). */
int llama_graph_destroy(llama_graph *graph);

/* ---------------------------------------------------------------- the steps, one by one
 * The layer entry points are compositions of these; they are exported so that each
 * step can be checked and timed on its own. */

/* y = gamma * x * rsqrt(mean(x^2) + eps) per row ("12 · 从 Transformer 到 LLaMA 系列" §八
 * RMSNorm; "3.2 核心组件逐一拆解" §3.2.1: fp32 arithmetic).  x, y: device [rows, d];
 * gamma: device [d]; all of dtype. */
int llama_rmsnorm(const void *x, const void *gamma, void *y, int32_t rows, int32_t d, float eps, int32_t dtype,
                  void *cuda_stream);

/* y = gamma * (x - mu) / sqrt(sigma^2 + eps) + beta per row, mu the row mean and sigma^2 the
 * biased row variance ("3.2 核心组件逐一拆解" §3.2.1, LayerNorm).  Not a step of the decoder
 * layer (which uses RMSNorm); exported so that the two normalisations can be compared on the
 * same rows.  x, y: device [rows, d]; gamma, beta: device [d]; all of dtype; 16-byte aligned.
 * fp32 arithmetic, one rounding to dtype.  rows == 0 is a no-op. */
int llama_layernorm(const void *x, const void *gamma, const void *beta, void *y, int32_t rows, int32_t d, float eps,
                    int32_t dtype, void *cuda_stream);

/* C = A B^T ("12 · 从 Transformer 到 LLaMA 系列" §八: nn.Linear, y = x W^T).  A: device
 * [M, K], B: device [N, K], both bf16; C: device [M, N], bf16 (c_f32 = 0) or fp32
 * (c_f32 = 1).  K % 8 == 0. */
int llama_linear_bf16(const void *A, const void *B, void *C, int32_t M, int32_t N, int32_t K, int32_t c_f32,
                      void *cuda_stream);

/* out = resid + A W^T (o_proj and down_proj with the residual add, "05 LLaMA3 Block — 从零件到
 * 发动机" §4.2 steps ④ and ⑧).  A: device [M, K]; W: device [N, K]; resid, out: device [M, N];
 * all bf16; resid and out may be the same buffer.  K % 8 == 0, N % 128 == 0. */
int llama_linear_residual(const void *A, const void *W, const void *resid, void *out, int32_t M, int32_t N,
                          int32_t K, void *cuda_stream);

/* out = SiLU(A W_gate^T) * (A W_up^T) ("3.2 核心组件逐一拆解" §3.2.2; "05 LLaMA3 Block — 从零件到
 * 发动机" §4.1).  A: device [M, K]; W_gate, W_up: device [I, K]; out: device [M, I]; bf16.
 * K % 8 == 0, I % 128 == 0. */
int llama_linear_swiglu(const void *A, const void *W_gate, const void *W_up, void *out, int32_t M, int32_t I,
                        int32_t K, void *cuda_stream);

/* [q|k|v] = xn [Wq;Wk;Wv]^T with RoPE on q and k ("第 10 章：现代 LLaMA 架构" §3 even/odd pairs,
 * §9 q_proj/k_proj/v_proj then apply_rope) for B sequences of S tokens at positions 0..S-1.
 * xn: device [B, S, d]; q_out: device [B, H, S, D]; k and v go to cache slots [0, S).  bf16
 * layers only (dims.dtype = LLAMA_BF16).  S <= max_pos and S <= cache.max_T. */
int llama_qkv_rope(const llama_layer_dims *dims, const void *xn, const void *wq, const void *wk, const void *wv,
                   const float *cos, const float *sin, int32_t max_pos, llama_kv_cache cache, void *q_out, int32_t B,
                   int32_t S, void *cuda_stream);

/* RMSNorm fused into the projection that consumes it: the bf16 layers' prefill runs these in
 * place of llama_rmsnorm followed by the plain projection.  The GEMM kernel itself normalises
 * row m of A as gamma * A[m] * rsqrt(mean(A[m]^2) + eps) ("12 · 从 Transformer 到 LLaMA 系列"
 * §八 RMSNorm; "3.2 核心组件逐一拆解" §3.2.1: the statistics in fp32) in its prologue -- each of
 * its CTAs takes a share of the rows, bit for bit what llama_rmsnorm stores -- writes the result
 * to xn and then multiplies xn: one launch, no separate normalisation kernel.
 * xn: device [M, K] bf16, caller-owned, 16-byte aligned, not aliasing A; it holds RMSNorm(A)
 * when the call completes.  sync: device int32, caller-owned scratch (any contents; the call
 * sets it to zero with a memset before the GEMM and the GEMM's CTAs count themselves in on it);
 * calls that may overlap on the GPU need separate ones.  The GEMM's CTAs wait for one another
 * (bounded: LLAMA_ERR_TIMEOUT after about a second), so they must all be resident at once: the
 * grid is at most one CTA per SM of the device.  bf16 data; K % 8 == 0. */

/* C = RMSNorm(A) B^T.  A: device [M, K]; gamma: device [K]; B: device [N, K]; C: device
 * [M, N], bf16 (c_f32 = 0) or fp32 (c_f32 = 1).  N % 8 == 0.  (The stack's final norm and LM
 * head.) */
int llama_norm_linear_bf16(const void *A, const void *gamma, float eps, const void *B, void *C, int32_t M, int32_t N,
                           int32_t K, int32_t c_f32, void *xn, int32_t *sync, void *cuda_stream);

/* out = SiLU(RMSNorm(A) W_gate^T) * (RMSNorm(A) W_up^T) (the post-attention norm and the gated
 * MLP's first half, "05 LLaMA3 Block — 从零件到发动机" §4.1-§4.2).  A: device [M, K]; gamma:
 * device [K]; W_gate, W_up: device [I, K]; out: device [M, I].  I % 128 == 0. */
int llama_norm_linear_swiglu(const void *A, const void *gamma, float eps, const void *W_gate, const void *W_up,
                             void *out, int32_t M, int32_t I, int32_t K, void *xn, int32_t *sync, void *cuda_stream);

/* llama_qkv_rope on RMSNorm(x) with gamma attn_norm and eps dims.rms_eps (the input norm of
 * the attention half, "05 LLaMA3 Block — 从零件到发动机" §4.2 step ②).  x, xn: device [B, S, d]. */
int llama_norm_qkv_rope(const llama_layer_dims *dims, const void *x, const void *attn_norm, const void *wq,
                        const void *wk, const void *wv, const float *cos, const float *sin, int32_t max_pos,
                        llama_kv_cache cache, void *q_out, int32_t B, int32_t S, void *xn, int32_t *sync,
                        void *cuda_stream);

/* Where llama_layer_prefill and llama_layer_prefill_chunk leave the layer's intermediate
 * activations in their workspace, for inspection once the call has completed on its stream
 * (each is overwritten by the next call that uses the workspace).  offsets receives 5 byte
 * offsets from the workspace start: [0] q after RoPE [B, H, S, D]; [1] attention output
 * [B, S, H*D]; [2] h = x + o_proj(attention) [B, S, d]; [3] the gated MLP activation
 * SiLU(gate) * up [B, S, d_inter]; [4] the normalised rows of the last RMSNorm, RMSNorm_2(h)
 * [B, S, d] (the gate/up GEMM's A operand); all of dims.dtype.  (K and V are in the cache.) */
int llama_layer_prefill_workspace_layout(const llama_layer_dims *dims, int32_t B, int32_t S, size_t *offsets);

/* Where llama_stack_forward leaves its last layer's data in its workspace (the same
 * inspection as above; a stack of n_layers = l + 1 layers computes exactly the first l + 1
 * layers of a longer one, so its last layer is layer l of that computation).  offsets
 * receives 3 byte offsets: [0] the last layer's input [B, S, d]; [1] its output; [2] the
 * last layer's prefill workspace, laid out as llama_layer_prefill_workspace_layout says. */
int llama_stack_workspace_layout(const llama_stack *stack, int32_t B, int32_t S, size_t *offsets);

/* Causal grouped-query attention over a cache ("12 · 从 Transformer 到 LLaMA 系列" §八
 * Attention; "深度学习进阶（三十）从 Transformer 到 LLaMA：现代 LLM 架构总览" §1.1
 * softmax(QK^T / sqrt(D)) V).  q: device [B, H, S, D] at positions 0..S-1; cache
 * slots [0, S) hold K, V; out: device [B, S, H*D].  Query head h reads KV head
 * h / (H/G); key j is visible to query i iff j <= i. */
int llama_attention_prefill(const llama_layer_dims *dims, const void *q, llama_kv_cache cache, void *out,
                            int32_t B, int32_t S, void *cuda_stream);

/* Workspace bytes of llama_attention_decode. */
int llama_attention_decode_workspace_bytes(const llama_layer_dims *dims, int32_t B, int32_t max_T, size_t *bytes);

/* One query per sequence at position positions[b] over cache slots 0..positions[b]
 * ("第 10 章：现代 LLaMA 架构" §7: score shape [B, H, 1, T_cache + 1]).  q: device
 * [B, H, D]; out: device [B, H*D].  A sequence whose position lies outside the cache (or
 * max_pos) gets a zero output row and LLAMA_ERR_DEVICE_BOUNDS in the status word.  bf16
 * layers need D = 128 and H / G in {1, 2, 4} or a multiple of 8. */
int llama_attention_decode(const llama_layer_dims *dims, const void *q, llama_kv_cache cache,
                           const int32_t *positions, void *out, int32_t B, void *workspace, size_t ws_bytes,
                           void *cuda_stream);

/* Decode attention without a workspace argument, for callers that cannot allocate device
 * memory: code whose device memory is owned entirely by another allocator (a framework's
 * caching pool, a fixed memory budget) and latency-critical loops where cudaMalloc or cudaFree
 * would synchronise the device.  The pages have no counterpart to this entry point; it computes
 * what llama_attention_decode computes, with the same arguments minus the workspace.
 * Its scratch is a fixed 16 MiB device array inside the library (every device that loads the
 * library holds one until the process exits); a request needs (min(B, 1024) * H + 256 * R)
 * * (D + 2) floats, R = min(H / G, 8), plus min(B, 1024) + 1 ints of it, and one that needs
 * more returns LLAMA_ERR_SCRATCH_LIMIT.  All calls on a device share that
 * array: calls that may overlap on the GPU (unordered streams) race on it.  Nothing in it needs
 * to start at zero.  The first call on each device looks up the array's device address (a host
 * query, no allocation); make that first call before any stream capture.  Never allocates or
 * frees device memory.  bf16 layers with D = 128 only. */
int llama_attention_decode_static(const llama_layer_dims *dims, const void *q, llama_kv_cache cache,
                                  const int32_t *positions, void *out, int32_t B, void *cuda_stream);

/* ---------------------------------------------------------------- host helpers and status */

/* RoPE tables on the HOST: cos/sin[p * (D/2) + i] = cos/sin(p * base^(-2i/D)), computed in
 * double precision and rounded to nearest fp32 ("12 · 从 Transformer 到 LLaMA 系列" §八
 * RotaryEmbedding; "深度学习进阶（三十）…" §4.2 theta_i = base^(-2i/d)).  cos_host, sin_host:
 * caller-owned host arrays of max_pos * D/2 floats. */
int llama_rope_tables(double base, int32_t head_dim, int32_t max_pos, float *cos_host, float *sin_host);

/* Synchronises `cuda_stream`, then returns and clears the current device's status word
 * (LLAMA_OK if no device-side error was recorded since the last call). */
int llama_get_device_status(void *cuda_stream);

/* Text of a status code (static storage). */
const char *llama_status_string(int status);

/* The record left by the first device-side wait that timed out since the library was
 * loaded: out[0] nanoseconds waited, out[1] polls, out[2] blockIdx.x | blockIdx.y << 32,
 * out[3] threadIdx.x, out[4] SM id, out[5] shared-memory address of the barrier | parity << 32,
 * out[6] gridDim.x | gridDim.y << 32 (zeros if none).  Copies min(n, 7) fields; synchronous. */
int llama_debug_timeout_record(int64_t *out, int32_t n);

/* Test of the bounded-wait path: launches one CTA that waits on an mbarrier that
 * nothing arrives at, for at most budget_ns nanoseconds (capped at 10 s), with the
 * same wait routine the tensor-core kernels use; the wait then records
 * LLAMA_ERR_TIMEOUT in the device status word and the kernel returns normally. */
int llama_debug_wait_probe(uint64_t budget_ns, void *cuda_stream);

/* Number of kernels the library enqueued on this process since load (for launch accounting). */
uint64_t llama_kernel_launch_count(void);

/* Per-thread kernel trace for measurement.  events: caller-owned cudaEvent_t handles
 * (n_events of them).  llama_trace_begin records events[0] on cuda_stream; afterwards,
 * until llama_trace_end, every kernel that this thread's calls enqueue is followed by
 * the next event, recorded on that call's stream (the i-th kernel runs between events
 * i and i+1).  llama_trace_end stops tracing and returns how many events were recorded. */
int llama_trace_begin(void *const *events, int32_t n_events, void *cuda_stream);
int32_t llama_trace_end(void);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_LAYER_H */
