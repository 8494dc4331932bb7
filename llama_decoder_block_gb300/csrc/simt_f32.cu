// fp32 path of the layer: the same dataflow as the bf16 path with plain fp32 FMA
// (no TF32), for layers stored in fp32.  Small shapes only need correctness here, so
// each output (or RoPE pair) is one thread and each attention query row one warp.
#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

// mode 0: out = X W0^T; 1: out = resid + X W0^T; 2: out = SiLU(X W0^T) * (X W1^T)
__global__ void simt_linear_kernel(int mode, const float* __restrict__ X, const float* __restrict__ W0,
                                   const float* __restrict__ W1, const float* __restrict__ resid,
                                   float* __restrict__ out, int M, int N, int K) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(M) * N) return;
  const int m = static_cast<int>(idx / N), n = static_cast<int>(idx % N);
  const float* x = X + static_cast<long long>(m) * K;
  const float* w0 = W0 + static_cast<long long>(n) * K;
  float a = 0.f;
  for (int k = 0; k < K; ++k) a = fmaf(x[k], w0[k], a);
  if (mode == 1) {
    a += resid[idx];
  } else if (mode == 2) {
    const float* w1 = W1 + static_cast<long long>(n) * K;
    float u = 0.f;
    for (int k = 0; k < K; ++k) u = fmaf(x[k], w1[k], u);
    a = silu_f(a) * u;
  }
  out[idx] = a;
}

// One thread per (token row m, column pair of [q heads | k heads | v heads]): pair i of a head
// is the columns (2i, 2i+1), or (i, i + D/2) with rope_half.
__global__ void simt_qkv_kernel(const float* __restrict__ X, const float* __restrict__ Wq,
                                const float* __restrict__ Wk, const float* __restrict__ Wv, int B, int S, int K,
                                int H, int G, int D, const float* __restrict__ cos, const float* __restrict__ sin,
                                const int32_t* __restrict__ positions, int max_pos, float* __restrict__ q_out,
                                float* __restrict__ k_cache, float* __restrict__ v_cache, int T_max, int rope_half,
                                const int32_t* __restrict__ lens, int* status) {
  const int pairs = (H + 2 * G) * D / 2;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(B) * S * pairs) return;
  const int m = static_cast<int>(idx / pairs);
  const int col = static_cast<int>(idx % pairs) * 2;
  const int b = m / S, s = m % S;
  if (lens != nullptr && (lens[b] < 0 || lens[b] > S)) {
    report(status, LLAMA_ERR_DEVICE_BOUNDS);
    return;
  }
  if (lens != nullptr && s >= lens[b]) return;   // padding of a shorter sequence: stored nowhere
  const int pos = positions ? positions[b] + s : s;
  if (pos < 0 || pos >= max_pos || pos >= T_max) {
    report(status, LLAMA_ERR_DEVICE_BOUNDS);
    return;
  }
  const int hh = col / D, i = (col % D) / 2;
  const int j0 = rope_half ? i : 2 * i, j1 = rope_half ? i + D / 2 : 2 * i + 1;
  const float* w;
  if (hh < H) w = Wq + static_cast<long long>(hh * D) * K;
  else if (hh < H + G) w = Wk + static_cast<long long>((hh - H) * D) * K;
  else w = Wv + static_cast<long long>((hh - H - G) * D) * K;
  const float* w0 = w + static_cast<long long>(j0) * K;
  const float* w1 = w + static_cast<long long>(j1) * K;
  const float* x = X + static_cast<long long>(m) * K;
  float e = 0.f, o = 0.f;
  for (int k = 0; k < K; ++k) {
    e = fmaf(x[k], w0[k], e);
    o = fmaf(x[k], w1[k], o);
  }
  if (hh < H + G) {   // RoPE on q and k: the pair (j0, j1) turns by pos * base^(-2i/D)
    const float c = cos[static_cast<long long>(pos) * (D / 2) + i];
    const float sn = sin[static_cast<long long>(pos) * (D / 2) + i];
    const float re = e * c - o * sn, ro = e * sn + o * c;
    e = re;
    o = ro;
  }
  float* dst;
  if (hh < H) dst = q_out + ((static_cast<long long>(b) * H + hh) * S + s) * D;
  else if (hh < H + G) dst = k_cache + ((static_cast<long long>(b) * G + (hh - H)) * T_max + pos) * D;
  else dst = v_cache + ((static_cast<long long>(b) * G + (hh - H - G)) * T_max + pos) * D;
  dst[j0] = e;
  dst[j1] = o;
}

// One warp per (b, h, s): online softmax over keys 0..pos of KV head h / (H/G).  Rows
// s >= lens[b] (padding) are not computed and not written.
__global__ void simt_attention_kernel(const float* __restrict__ q, const float* __restrict__ kc,
                                      const float* __restrict__ vc, const int32_t* __restrict__ positions,
                                      const int32_t* __restrict__ lens, float* __restrict__ out, int B, int S, int H,
                                      int G, int D, int T_max, int max_pos, int* status) {
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(B) * H * S) return;
  const int s = static_cast<int>(wid % S);
  const int h = static_cast<int>((wid / S) % H);
  const int b = static_cast<int>(wid / (static_cast<long long>(S) * H));
  const int g = h / (H / G);
  if (lens != nullptr && (s >= lens[b] || lens[b] > S)) return;
  const int pos = positions ? positions[b] + s : s;
  float* o_row = out + (static_cast<long long>(b) * S + s) * H * D + h * D;
  if (pos < 0 || pos >= max_pos || pos >= T_max) {
    if (lane == 0) report(status, LLAMA_ERR_DEVICE_BOUNDS);
    for (int d = lane; d < D; d += 32) o_row[d] = 0.f;
    return;
  }
  const float* qr = q + ((static_cast<long long>(b) * H + h) * S + s) * D;
  const float scale = rsqrtf(static_cast<float>(D));
  constexpr int MAXV = 8;   // D <= 256
  float qv[MAXV], acc[MAXV];
#pragma unroll
  for (int t = 0; t < MAXV; ++t) {
    const int d = lane + 32 * t;
    qv[t] = d < D ? qr[d] * scale : 0.f;
    acc[t] = 0.f;
  }
  float m_run = -INFINITY, l_run = 0.f;
  const long long base = (static_cast<long long>(b) * G + g) * T_max;
  for (int key = 0; key <= pos; ++key) {
    const float* kr = kc + (base + key) * D;
    float dot = 0.f;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
      const int d = lane + 32 * t;
      if (d < D) dot = fmaf(qv[t], kr[d], dot);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    const float m_new = fmaxf(m_run, dot);
    const float alpha = expf(m_run - m_new);
    const float p = expf(dot - m_new);
    l_run = l_run * alpha + p;
    const float* vr = vc + (base + key) * D;
#pragma unroll
    for (int t = 0; t < MAXV; ++t) {
      const int d = lane + 32 * t;
      if (d < D) acc[t] = fmaf(p, vr[d], acc[t] * alpha);
    }
    m_run = m_new;
  }
#pragma unroll
  for (int t = 0; t < MAXV; ++t) {
    const int d = lane + 32 * t;
    if (d < D) o_row[d] = acc[t] / l_run;
  }
}

}  // namespace

int simt_linear(const Ctx& c, int mode, const float* X, const float* W0, const float* W1, const float* W2,
                const float* resid, float* out, int M, int N, int K) {
  (void)W2;
  const long long total = static_cast<long long>(M) * N;
  if (total == 0) return LLAMA_OK;
  simt_linear_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, c.stream>>>(mode, X, W0, W1, resid, out,
                                                                                      M, N, K);
  return after_launch(c);
}

int simt_qkv_rope(const Ctx& c, const float* X, const float* Wq, const float* Wk, const float* Wv, int B, int S,
                  int K, int H, int G, int D, const float* cos, const float* sin, const int32_t* positions,
                  int max_pos, float* q_out, float* k_cache, float* v_cache, int T_max, int rope_half,
                  const int32_t* lens) {
  const long long total = static_cast<long long>(B) * S * ((H + 2 * G) * D / 2);
  if (total == 0) return LLAMA_OK;
  simt_qkv_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, c.stream>>>(
      X, Wq, Wk, Wv, B, S, K, H, G, D, cos, sin, positions, max_pos, q_out, k_cache, v_cache, T_max, rope_half,
      lens, c.status);
  return after_launch(c);
}

int simt_attention(const Ctx& c, const float* q, const float* k_cache, const float* v_cache,
                   const int32_t* positions, float* out, int B, int S, int H, int G, int D, int T_max,
                   int max_pos, const int32_t* lens) {
  if (D > 256) return LLAMA_ERR_UNSUPPORTED;
  const long long threads = static_cast<long long>(B) * H * S * 32;
  if (threads == 0) return LLAMA_OK;
  simt_attention_kernel<<<static_cast<unsigned>((threads + 127) / 128), 128, 0, c.stream>>>(
      q, k_cache, v_cache, positions, lens, out, B, S, H, G, D, T_max, max_pos, c.status);
  return after_launch(c);
}

}  // namespace llama
