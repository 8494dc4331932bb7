// Host-side interfaces between the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/llama_layer.h"

namespace llama {

// Devices a process may use with the library (per-device state is kept in arrays of this
// size; make_ctx refuses a device index beyond it).
constexpr int kMaxDevices = 64;

// Per-call launch context: the caller's stream and the current device's facts.
struct Ctx {
  cudaStream_t stream;
  int device;
  int num_sms;
  int* status;   // device address of this device's status word
  // Launch with programmatic stream serialisation (may overlap the previous kernel's tail).
  // A call's first kernel goes without it, so that everything queued before the call has
  // finished when any kernel of the call starts.
  bool pdl = true;
  // The GEMMs' weight operands are written by nothing that may still run: their producers
  // may load weight tiles before griddepcontrol.wait.  Set by the composite entry points,
  // whose weights are the caller's parameters.
  bool static_weights = false;
};

// Fills `c` for the current device; returns LLAMA_OK or LLAMA_ERR_CUDA.
int make_ctx(void* stream, Ctx* c);

// Launches `kern` on c.stream with programmatic stream serialisation (the kernel calls
// pdl_trigger / pdl_wait, see common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(const Ctx& c, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = c.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
// The same with thread-block clusters of cluster_x CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(const Ctx& c, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = cluster_x;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (c.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}
// Checks cudaGetLastError after a launch, counts it and records the next trace event.
int after_launch(const Ctx& c);
// True while llama_trace_begin's events are being recorded on this thread.
bool trace_active();

// ---------------------------------------------------------------- tensor maps (tmap.cu)
// 2-D bf16 row-major matrix [rows, cols] with row stride `ld` elements; box = 64 columns
// (128 bytes, 128-byte swizzle) by `box_rows` rows.  Out-of-range elements read as 0.
bool make_tmap_2d(CUtensorMap* tm, const void* base, uint64_t cols, uint64_t rows, uint64_t ld,
                  uint32_t box_rows);
// 3-D bf16 tensor [n2][n1][n0] with strides (elements) s1 (between n1 rows) and s2
// (between n2 planes); box = 64 x box1 x 1 with 128-byte swizzle.
bool make_tmap_3d(CUtensorMap* tm, const void* base, uint64_t n0, uint64_t n1, uint64_t n2, uint64_t s1,
                  uint64_t s2, uint32_t box1);

// ---------------------------------------------------------------- RMSNorm (rmsnorm.cu)
int rmsnorm(const Ctx& c, const void* x, const void* gamma, void* y, int rows, int d, float eps, int dtype);

// ---------------------------------------------------------------- LayerNorm (layernorm.cu)
// y = gamma * (x - mean) * rsqrt(biased variance + eps) + beta per row.
int layernorm(const Ctx& c, const void* x, const void* gamma, const void* beta, void* y, int rows, int d, float eps,
              int dtype);

// ---------------------------------------------------------------- tcgen05 GEMMs (gemm_tc.cu)
// RMSNorm of operand A in the GEMM's prologue (see gemm_tc.cu): the GEMM first writes
// RMSNorm(X) = gamma * X * rsqrt(mean(X^2) + eps) into xn, then multiplies xn.
struct NormPro {
  const void* gamma;   // device [K]
  float eps;
  void* xn;            // device [M, K] bf16, 16-byte aligned: receives RMSNorm(X), the A operand
  int* count;          // device int, zero before the launch (the prologue's grid-wide count)
};

// All compute C = X W^T with X [M, K] and W [N, K] bf16 row-major, fp32 accumulation.
// norm (may be null): X is normalised per row first, RMSNorm(X) W^T.
int gemm_plain(const Ctx& c, const void* X, const void* W, void* C, int M, int N, int K, bool c_f32,
               const NormPro* norm = nullptr);
// out = resid + X W^T  (bf16); resid and out may alias.
int gemm_residual(const Ctx& c, const void* X, const void* W, const void* resid, void* out, int M, int N, int K);
// out[:, n] = SiLU(X W_gate^T)[:, n] * (X W_up^T)[:, n]  (bf16, [M, I]).
int gemm_swiglu(const Ctx& c, const void* X, const void* Wg, const void* Wu, void* out, int M, int I, int K,
                const NormPro* norm = nullptr);
// [q|k|v] = X [Wq;Wk;Wv]^T for B sequences of S tokens at positions 0..S-1; RoPE on q, k;
// q -> q_out [B, H, S, D]; k, v -> cache slots [0, S) of [B, G, T_max, D].
// rope_half: pairs (i, i + D/2) instead of (2i, 2i+1).  start (device [B], may be null):
// token s of sequence b sits at position start[b] + s and goes to that cache slot; lens
// (device [B], may be null = S): tokens s >= lens[b] are padding and stored nowhere.
int gemm_qkv_rope(const Ctx& c, const void* X, const void* Wq, const void* Wk, const void* Wv, int B, int S,
                  int K, int H, int G, int D, const float* cos, const float* sin, void* q_out, void* k_cache,
                  void* v_cache, int T_max, int rope_half, const int32_t* start = nullptr,
                  const int32_t* lens = nullptr, int max_pos = 0, const NormPro* norm = nullptr);
// Weight-streaming form for few tokens: P[s][t][n] = sum over split s of W[n, k] X[t, k] in fp32,
// with W the row-concatenation of up to three matrices (rows multiples of 128).
int gemm_tokens_partial(const Ctx& c, const void* const* W, const int* w_rows, int n_w, const void* X,
                        int n_tok, int K, int splits, float* P);
// Split count for the weight-streaming form (exactly the count that gemm_tokens_partial uses).
int choose_splits(int num_sms, int w_rows_total, int K, int n_tok);

// ---------------------------------------------------------------- attention
// start / lens as for gemm_qkv_rope: query s of sequence b at position start[b] + s sees
// cache slots 0 .. start[b] + s; output rows s >= lens[b] are not written.
int attn_prefill_tc(const Ctx& c, const void* q, const void* k_cache, const void* v_cache, void* out, int B,
                    int S, int H, int G, int D, int T_max, const int32_t* start = nullptr,
                    const int32_t* lens = nullptr, int max_pos = 0);
size_t attn_decode_ws_bytes(int B, int H, int G, int D);
int attn_decode(const Ctx& c, int dtype, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* positions, void* out, int B, int H, int G, int D, int T_max, int max_pos,
                void* ws);

// ---------------------------------------------------------------- fp32 SIMT path (simt_f32.cu)
// mode 0: C = X W^T; 1: out = resid + X W^T; 2: out = SiLU(X Wg^T) * (X Wu^T);
// 3: QKV + RoPE scatter (positions: null -> token m of sequence b at m % S, else
// positions[b] + m % S; lens: null, or tokens m % S >= lens[b] are padding and stored nowhere).
int simt_linear(const Ctx& c, int mode, const float* X, const float* W0, const float* W1, const float* W2,
                const float* resid, float* out, int M, int N, int K);
int simt_qkv_rope(const Ctx& c, const float* X, const float* Wq, const float* Wk, const float* Wv, int B, int S,
                  int K, int H, int G, int D, const float* cos, const float* sin, const int32_t* positions,
                  int max_pos, float* q_out, float* k_cache, float* v_cache, int T_max, int rope_half,
                  const int32_t* lens = nullptr);
int simt_attention(const Ctx& c, const float* q, const float* k_cache, const float* v_cache,
                   const int32_t* positions, float* out, int B, int S, int H, int G, int D, int T_max,
                   int max_pos, const int32_t* lens = nullptr);

// ---------------------------------------------------------------- small kernels (misc.cu)
// rows of `row_bytes` bytes (a multiple of 16) of any element type
int embed_gather(const Ctx& c, const int32_t* tokens, const void* table, void* x, int n_tok, int row_bytes,
                 int vocab);
// Decode epilogues on the fp32 split partials P [splits][n_tok][N].
int fix_qkv_rope(const Ctx& c, const float* P, int splits, int n_tok, int H, int G, int D,
                 const int32_t* positions, int max_pos, const float* cos, const float* sin, void* q_out,
                 void* k_cache, void* v_cache, int T_max, int rope_half);
int fix_residual(const Ctx& c, const float* P, int splits, int n_tok, int N, const void* resid, void* out);
// h = resid + sum of the splits (bf16), then hn = RMSNorm(h) with gamma (bf16); one CTA per token.
int fix_residual_rmsnorm(const Ctx& c, const float* P, int splits, int n_tok, int N, const void* resid,
                         const void* gamma, float eps, void* h_out, void* hn_out);
int fix_swiglu(const Ctx& c, const float* P, int splits, int n_tok, int I, void* out);
// out = the sum of the splits (fp32 [n_tok, N]); N % 4 == 0.
int fix_sum_f32(const Ctx& c, const float* P, int splits, int n_tok, int N, float* out);

}  // namespace llama
