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
  pdl_trigger();
  pdl_wait();
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

// Sum over the splits of 4 consecutive fp32 partials (16-byte aligned), in split order.  The
// loads of the first MAXL splits are all issued before the first add (a fixed, predicated
// unroll), so a thread waits for one round trip to L2, not one per split.
template <int MAXL = 4>
__device__ __forceinline__ float4 split_sum4(const float* P, int splits, long long stride, long long idx) {
  float4 b[MAXL];
#pragma unroll
  for (int s = 0; s < MAXL; ++s)
    if (s < splits) b[s] = __ldcs(reinterpret_cast<const float4*>(P + s * stride + idx));
  float4 a = b[0];
#pragma unroll
  for (int s = 1; s < MAXL; ++s)
    if (s < splits) { a.x += b[s].x; a.y += b[s].y; a.z += b[s].z; a.w += b[s].w; }
  for (int s = MAXL; s < splits; ++s) {
    const float4 c = __ldcs(reinterpret_cast<const float4*>(P + s * stride + idx));
    a.x += c.x; a.y += c.y; a.z += c.z; a.w += c.w;
  }
  return a;
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float a, float b, float c, float d) {
  uint2 w;
  w.x = pack_bf16(a, b);
  w.y = pack_bf16(c, d);
  *reinterpret_cast<uint2*>(dst) = w;
}

// grid (ceil(N / 1024), n_tok): 4 consecutive columns of [q heads | k heads | v heads] per thread.
// With half-split pairs a thread of the first half of a q or k head also takes the partner
// columns j + D/2 ... j + D/2 + 3, and threads of the second half have nothing to do.
__global__ void fix_qkv_kernel(const float* __restrict__ P, int splits, int n_tok, int H, int G, int D,
                               const int32_t* __restrict__ positions, int max_pos, const float* __restrict__ cos,
                               const float* __restrict__ sin, __nv_bfloat16* __restrict__ q_out,
                               __nv_bfloat16* __restrict__ k_cache, __nv_bfloat16* __restrict__ v_cache, int T_max,
                               int rope_half, int* status) {
  pdl_trigger();
  pdl_wait();
  const int N = (H + 2 * G) * D;
  const int t = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (col >= N) return;
  const int pos = positions[t];
  if (pos < 0 || pos >= max_pos || pos >= T_max) {
    if (col == 0) report(status, LLAMA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int hh = col / D, j = col - hh * D;
  __nv_bfloat16* dst;
  if (hh < H) dst = q_out + (static_cast<long long>(t) * H + hh) * D;
  else if (hh < H + G) dst = k_cache + ((static_cast<long long>(t) * G + (hh - H)) * T_max + pos) * D;
  else dst = v_cache + ((static_cast<long long>(t) * G + (hh - H - G)) * T_max + pos) * D;
  const long long stride = static_cast<long long>(n_tok) * N, at = static_cast<long long>(t) * N + col;
  if (rope_half && hh < H + G) {   // pairs (j + i, j + i + D/2), angle index j + i
    if (j >= D / 2) return;
    const float4 x1 = split_sum4(P, splits, stride, at), x2 = split_sum4(P, splits, stride, at + D / 2);
    const float* cr = cos + static_cast<long long>(pos) * (D / 2) + j;
    const float* sr = sin + static_cast<long long>(pos) * (D / 2) + j;
    const float a[4] = {x1.x, x1.y, x1.z, x1.w}, b[4] = {x2.x, x2.y, x2.z, x2.w};
    float lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo[i] = a[i] * cr[i] - b[i] * sr[i];
      hi[i] = b[i] * cr[i] + a[i] * sr[i];
    }
    store_bf16x4(dst + j, lo[0], lo[1], lo[2], lo[3]);
    store_bf16x4(dst + j + D / 2, hi[0], hi[1], hi[2], hi[3]);
    return;
  }
  const float4 v = split_sum4(P, splits, stride, at);
  float e0 = v.x, o0 = v.y, e1 = v.z, o1 = v.w;
  if (hh < H + G) {   // RoPE at the token's own position, pairs (j, j+1) and (j+2, j+3)
    const float* cr = cos + static_cast<long long>(pos) * (D / 2) + j / 2;
    const float* sr = sin + static_cast<long long>(pos) * (D / 2) + j / 2;
    const float c0 = cr[0], s0 = sr[0], c1 = cr[1], s1 = sr[1];
    const float r0 = e0 * c0 - o0 * s0, r1 = e0 * s0 + o0 * c0;
    const float r2 = e1 * c1 - o1 * s1, r3 = e1 * s1 + o1 * c1;
    e0 = r0; o0 = r1; e1 = r2; o1 = r3;
  }
  store_bf16x4(dst + j, e0, o0, e1, o1);
}

// grid (ceil(N / 1024), n_tok): out = resid + sum of the splits, 4 columns per thread
__global__ void fix_residual_kernel(const float* __restrict__ P, int splits, int n_tok, int N,
                                    const __nv_bfloat16* __restrict__ resid, __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (col >= N) return;
  const long long idx = static_cast<long long>(t) * N + col;
  const float4 v = split_sum4(P, splits, static_cast<long long>(n_tok) * N, idx);
  const uint2 r = *reinterpret_cast<const uint2*>(resid + idx);
  store_bf16x4(out + idx, bf16_lo(r.x) + v.x, bf16_hi(r.x) + v.y, bf16_lo(r.y) + v.z, bf16_hi(r.y) + v.w);
}

// One CTA per token: h = resid + sum of the splits (stored in bf16), then hn = RMSNorm(h) from
// the stored h ("12 · 从 Transformer 到 LLaMA 系列" §八 RMSNorm; fp32 arithmetic).
constexpr int kNormFixThreads = 512;
__global__ void __launch_bounds__(kNormFixThreads) fix_residual_rmsnorm_kernel(const float* __restrict__ P, int splits,
                                                                   int n_tok, int N,
                                                                   const __nv_bfloat16* __restrict__ resid,
                                                                   const __nv_bfloat16* __restrict__ gamma, float eps,
                                                                   __nv_bfloat16* __restrict__ h_out,
                                                                   __nv_bfloat16* __restrict__ hn_out) {
  pdl_trigger();
  pdl_wait();
  constexpr int MAXV = 4;   // 4-column groups per thread: N <= 512 * 4 * 4 = 8192
  constexpr int WARPS = kNormFixThreads / 32;
  __shared__ float red[WARPS];
  const int t = blockIdx.x;
  const long long row = static_cast<long long>(t) * N;
  float hv[MAXV][4];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int col = (i * blockDim.x + threadIdx.x) * 4;
    if (col < N) {
      const float4 v = split_sum4<8>(P, splits, static_cast<long long>(n_tok) * N, row + col);
      const uint2 r = *reinterpret_cast<const uint2*>(resid + row + col);
      const uint32_t w0 = pack_bf16(bf16_lo(r.x) + v.x, bf16_hi(r.x) + v.y);
      const uint32_t w1 = pack_bf16(bf16_lo(r.y) + v.z, bf16_hi(r.y) + v.w);
      *reinterpret_cast<uint2*>(h_out + row + col) = make_uint2(w0, w1);
      hv[i][0] = bf16_lo(w0); hv[i][1] = bf16_hi(w0); hv[i][2] = bf16_lo(w1); hv[i][3] = bf16_hi(w1);
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(hv[i][e], hv[i][e], ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) tot += red[w];
  const float r = rsqrtf(tot / static_cast<float>(N) + eps);
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int col = (i * blockDim.x + threadIdx.x) * 4;
    if (col < N) {
      const uint2 g = *reinterpret_cast<const uint2*>(gamma + col);
      store_bf16x4(hn_out + row + col, bf16_lo(g.x) * (hv[i][0] * r), bf16_hi(g.x) * (hv[i][1] * r),
                   bf16_lo(g.y) * (hv[i][2] * r), bf16_hi(g.y) * (hv[i][3] * r));
    }
  }
}

// grid (ceil(I / 1024), n_tok): a = SiLU(gate) * up from the split sums, 4 columns per thread
__global__ void fix_swiglu_kernel(const float* __restrict__ P, int splits, int n_tok, int I,
                                  __nv_bfloat16* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= I) return;
  const long long stride = static_cast<long long>(n_tok) * 2 * I;
  const float4 gs = split_sum4(P, splits, stride, static_cast<long long>(t) * 2 * I + n);
  const float4 us = split_sum4(P, splits, stride, static_cast<long long>(t) * 2 * I + I + n);
  store_bf16x4(out + static_cast<long long>(t) * I + n, silu_f(gs.x) * us.x, silu_f(gs.y) * us.y,
               silu_f(gs.z) * us.z, silu_f(gs.w) * us.w);
}

}  // namespace

int embed_gather(const Ctx& c, const int32_t* tokens, const void* table, void* x, int n_tok, int row_bytes,
                 int vocab) {
  if (n_tok == 0) return LLAMA_OK;
  const int vec = row_bytes / 16;
  launch_pdl(c, embed_kernel, dim3((n_tok + 7) / 8), dim3(256), 0, tokens, static_cast<const uint4*>(table),
             static_cast<uint4*>(x), n_tok, vec, vocab, c.status);
  return after_launch(c);
}

int fix_qkv_rope(const Ctx& c, const float* P, int splits, int n_tok, int H, int G, int D, const int32_t* positions,
                 int max_pos, const float* cos, const float* sin, void* q_out, void* k_cache, void* v_cache,
                 int T_max, int rope_half) {
  const int N = (H + 2 * G) * D;
  if (n_tok == 0) return LLAMA_OK;
  launch_pdl(c, fix_qkv_kernel, dim3((N / 4 + 255) / 256, n_tok), dim3(256), 0,
      P, splits, n_tok, H, G, D, positions, max_pos, cos, sin, static_cast<__nv_bfloat16*>(q_out),
      static_cast<__nv_bfloat16*>(k_cache), static_cast<__nv_bfloat16*>(v_cache), T_max, rope_half, c.status);
  return after_launch(c);
}

namespace {

// grid (ceil(N / 1024), n_tok): out = sum of the splits in fp32, 4 columns per thread
__global__ void fix_sum_f32_kernel(const float* __restrict__ P, int splits, int n_tok, int N,
                                   float* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.y;
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (col >= N) return;
  const long long at = static_cast<long long>(t) * N + col;
  *reinterpret_cast<float4*>(out + at) = split_sum4(P, splits, static_cast<long long>(n_tok) * N, at);
}

}  // namespace

int fix_sum_f32(const Ctx& c, const float* P, int splits, int n_tok, int N, float* out) {
  if (n_tok == 0) return LLAMA_OK;
  launch_pdl(c, fix_sum_f32_kernel, dim3((N / 4 + 255) / 256, n_tok), dim3(256), 0, P, splits, n_tok, N, out);
  return after_launch(c);
}

int fix_residual(const Ctx& c, const float* P, int splits, int n_tok, int N, const void* resid, void* out) {
  if (n_tok == 0) return LLAMA_OK;
  launch_pdl(c, fix_residual_kernel, dim3((N / 4 + 255) / 256, n_tok), dim3(256), 0,
      P, splits, n_tok, N, static_cast<const __nv_bfloat16*>(resid), static_cast<__nv_bfloat16*>(out));
  return after_launch(c);
}

int fix_residual_rmsnorm(const Ctx& c, const float* P, int splits, int n_tok, int N, const void* resid,
                         const void* gamma, float eps, void* h_out, void* hn_out) {
  if (n_tok == 0) return LLAMA_OK;
  if (N % 4 != 0 || N > kNormFixThreads * 4 * 4) return LLAMA_ERR_UNSUPPORTED;
  launch_pdl(c, fix_residual_rmsnorm_kernel, dim3(n_tok), dim3(kNormFixThreads), 0,
      P, splits, n_tok, N, static_cast<const __nv_bfloat16*>(resid), static_cast<const __nv_bfloat16*>(gamma), eps,
      static_cast<__nv_bfloat16*>(h_out), static_cast<__nv_bfloat16*>(hn_out));
  return after_launch(c);
}

int fix_swiglu(const Ctx& c, const float* P, int splits, int n_tok, int I, void* out) {
  if (n_tok == 0) return LLAMA_OK;
  launch_pdl(c, fix_swiglu_kernel, dim3((I / 4 + 255) / 256, n_tok), dim3(256), 0, P, splits, n_tok, I,
             static_cast<__nv_bfloat16*>(out));
  return after_launch(c);
}

}  // namespace llama
