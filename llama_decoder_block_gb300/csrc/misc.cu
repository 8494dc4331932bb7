// Small HBM-bound kernels: the token-embedding gather and the epilogues of the
// weight-streaming (decode) GEMMs, which sum the fp32 split-K partials and apply the
// fused op of each projection.
#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

// x[t, :] = table[tokens[t], :] ("12 · 从 Transformer 到 LLaMA 系列" §八 nn.Embedding), one warp per token.
__global__ void embed_kernel(const int32_t* __restrict__ tokens, const uint4* __restrict__ table,
                             uint4* __restrict__ x, int n_tok, int vec_per_row, int vocab, int* status) {
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= n_tok) return;
  const int id = tokens[t];
  uint4* dst = x + static_cast<long long>(t) * vec_per_row;
  if (id < 0 || id >= vocab) {
    if (lane == 0) report(status, LLAMA_ERR_DEVICE_BOUNDS);
    for (int i = lane; i < vec_per_row; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = table + static_cast<long long>(id) * vec_per_row;
  for (int i = lane; i < vec_per_row; i += 32) dst[i] = __ldg(src + i);
}

__device__ __forceinline__ float split_sum(const float* P, int splits, long long stride, long long idx) {
  float a = 0.f;
  for (int s = 0; s < splits; ++s) a += P[s * stride + idx];
  return a;
}

// one thread per (token, column pair) of [q heads | k heads | v heads]
__global__ void fix_qkv_kernel(const float* __restrict__ P, int splits, int n_tok, int H, int G, int D,
                               const int32_t* __restrict__ positions, int max_pos, const float* __restrict__ cos,
                               const float* __restrict__ sin, __nv_bfloat16* __restrict__ q_out,
                               __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache, int T_max,
                               int* status) {
  const int N = (H + 2 * G) * D;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n_tok) * (N / 2)) return;
  const int t = static_cast<int>(idx / (N / 2));
  const int col = static_cast<int>(idx % (N / 2)) * 2;
  const int pos = positions[t];
  if (pos < 0 || pos >= max_pos || pos >= T_max) {
    if (col == 0) report(status, LLAMA_ERR_DEVICE_BOUNDS);
    return;
  }
  const long long stride = static_cast<long long>(n_tok) * N;
  float e = split_sum(P, splits, stride, static_cast<long long>(t) * N + col);
  float o = split_sum(P, splits, stride, static_cast<long long>(t) * N + col + 1);
  const int hh = col / D, j = col % D;
  if (hh < H + G) {   // RoPE at the token's own position
    const float c = cos[static_cast<long long>(pos) * (D / 2) + j / 2];
    const float sn = sin[static_cast<long long>(pos) * (D / 2) + j / 2];
    const float re = e * c - o * sn, ro = e * sn + o * c;
    e = re;
    o = ro;
  }
  __nv_bfloat16* dst;
  if (hh < H) dst = q_out + (static_cast<long long>(t) * H + hh) * D;
  else if (hh < H + G) dst = k_cache + ((static_cast<long long>(t) * G + (hh - H)) * T_max + pos) * D;
  else dst = v_cache + ((static_cast<long long>(t) * G + (hh - H - G)) * T_max + pos) * D;
  *reinterpret_cast<__nv_bfloat162*>(dst + j) = __floats2bfloat162_rn(e, o);
}

__global__ void fix_residual_kernel(const float* __restrict__ P, int splits, int n_tok, int N,
                                    const __nv_bfloat16* __restrict__ resid, __nv_bfloat16* __restrict__ out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(n_tok) * N;
  if (idx >= total) return;
  out[idx] = __float2bfloat16_rn(__bfloat162float(resid[idx]) + split_sum(P, splits, total, idx));
}

__global__ void fix_swiglu_kernel(const float* __restrict__ P, int splits, int n_tok, int I,
                                  __nv_bfloat16* __restrict__ out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n_tok) * I) return;
  const int t = static_cast<int>(idx / I), n = static_cast<int>(idx % I);
  const long long stride = static_cast<long long>(n_tok) * 2 * I;
  const float gsum = split_sum(P, splits, stride, static_cast<long long>(t) * 2 * I + n);
  const float usum = split_sum(P, splits, stride, static_cast<long long>(t) * 2 * I + I + n);
  out[idx] = __float2bfloat16_rn(silu_f(gsum) * usum);
}

}  // namespace

int embed_gather(const Ctx& c, const int32_t* tokens, const void* table, void* x, int n_tok, int row_bytes,
                 int vocab) {
  if (n_tok == 0) return LLAMA_OK;
  const int vec = row_bytes / 16;
  embed_kernel<<<(n_tok + 7) / 8, 256, 0, c.stream>>>(tokens, static_cast<const uint4*>(table),
                                                      static_cast<uint4*>(x), n_tok, vec, vocab, c.status);
  return after_launch(c);
}

int fix_qkv_rope(const Ctx& c, const float* P, int splits, int n_tok, int H, int G, int D, const int32_t* positions,
                 int max_pos, const float* cos, const float* sin, void* q_out, void* k_cache, void* v_cache,
                 int T_max) {
  const long long total = static_cast<long long>(n_tok) * ((H + 2 * G) * D / 2);
  if (total == 0) return LLAMA_OK;
  fix_qkv_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, c.stream>>>(
      P, splits, n_tok, H, G, D, positions, max_pos, cos, sin, static_cast<__nv_bfloat16*>(q_out),
      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), T_max, c.status);
  return after_launch(c);
}

int fix_residual(const Ctx& c, const float* P, int splits, int n_tok, int N, const void* resid, void* out) {
  const long long total = static_cast<long long>(n_tok) * N;
  if (total == 0) return LLAMA_OK;
  fix_residual_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, c.stream>>>(
      P, splits, n_tok, N, static_cast<const __nv_bfloat16*>(resid), static_cast<__nv_bfloat16*>(out));
  return after_launch(c);
}

int fix_swiglu(const Ctx& c, const float* P, int splits, int n_tok, int I, void* out) {
  const long long total = static_cast<long long>(n_tok) * I;
  if (total == 0) return LLAMA_OK;
  fix_swiglu_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, c.stream>>>(
      P, splits, n_tok, I, static_cast<__nv_bfloat16*>(out));
  return after_launch(c);
}

}  // namespace llama
