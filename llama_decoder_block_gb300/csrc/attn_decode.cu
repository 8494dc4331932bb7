// Decode attention: one new query per sequence over its cached keys, split along the keys.
//
// Query of sequence b sits at position p = positions[b] and sees cache slots 0..p
// ("第 10 章：现代 LLaMA 架构" §7: q_len = 1, k_len = past_len + 1, score shape
// [B, H, 1, T_cache + 1]; §6: the G cached K/V heads are shared by H/G query heads).
//
// Memory-bound: the cache is read once.  CTA = (key split, KV head g, sequence b);
// each 16-byte load of a K or V row serves all H/G query heads of the group.  A
// half-warp covers one 128-element key row (8 bf16 per lane), a warp two keys per
// step, four steps unrolled so that eight 16-byte loads per lane are in flight.
// Each CTA leaves (m, l, O) of its split; the combine kernel merges the splits.
#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int HD = 128;
constexpr int SPLIT = 512;        // keys per CTA
constexpr int WARPS = 4;
constexpr int UNROLL = 4;         // key pairs per warp in flight

__device__ __forceinline__ float half_warp_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

__device__ __forceinline__ void unpack8(const uint4 w, float* f) {
  f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
  f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
}

template <int REP>
__global__ void __launch_bounds__(WARPS * 32)
    attn_decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kc,
                             const __nv_bfloat16* __restrict__ vc, const int32_t* __restrict__ positions,
                             float* __restrict__ o_part, float* __restrict__ m_part, float* __restrict__ l_part,
                             int H, int G, int T_max, int max_pos, int n_split, float scale_log2, int* status) {
  const int sp = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, sub = lane & 15;
  const int pos = positions[b];
  const bool valid_pos = pos >= 0 && pos < T_max && pos < max_pos;
  if (!valid_pos && sp == 0 && g == 0 && threadIdx.x == 0) report(status, LLAMA_ERR_DEVICE_BOUNDS);
  const int n_keys = valid_pos ? pos + 1 : 0;
  const int k_begin = sp * SPLIT;
  const int k_end = min(k_begin + SPLIT, n_keys);
  const int h0 = g * REP;
  const long long part = (static_cast<long long>(b) * H + h0) * n_split + sp;   // index of (b, h0, sp)

  __shared__ float s_m[WARPS][REP], s_l[WARPS][REP];
  __shared__ float s_o[WARPS][REP][HD];

  if (k_begin >= k_end) {   // empty split: neutral element of the merge
    if (threadIdx.x < REP) {
      m_part[part + threadIdx.x * n_split] = -INFINITY;
      l_part[part + threadIdx.x * n_split] = 0.f;
    }
    return;
  }

  float qv[REP][8];
#pragma unroll
  for (int r = 0; r < REP; ++r) {
    const uint4 w = *reinterpret_cast<const uint4*>(q + (static_cast<long long>(b) * H + h0 + r) * HD + sub * 8);
    unpack8(w, qv[r]);
#pragma unroll
    for (int e = 0; e < 8; ++e) qv[r][e] *= scale_log2;
  }
  float m_run[REP], l_run[REP], acc[REP][8];
#pragma unroll
  for (int r = 0; r < REP; ++r) {
    m_run[r] = -INFINITY;
    l_run[r] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;
  }

  const long long head_base = (static_cast<long long>(b) * G + g) * T_max;
  // the loop bound is uniform over the warp (the shuffles need all 32 lanes)
  for (int kw0 = k_begin + warp * 2; kw0 < k_end; kw0 += WARPS * 2 * UNROLL) {
    uint4 kw[UNROLL], vw[UNROLL];
    bool kv_ok[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int key = kw0 + half + u * WARPS * 2;
      kv_ok[u] = key < k_end;
      const long long off = (head_base + (kv_ok[u] ? key : k_begin)) * HD + sub * 8;
      kw[u] = __ldcs(reinterpret_cast<const uint4*>(kc + off));
      vw[u] = __ldcs(reinterpret_cast<const uint4*>(vc + off));
    }
    float s[UNROLL][REP];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float kf[8];
      unpack8(kw[u], kf);
#pragma unroll
      for (int r = 0; r < REP; ++r) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) d = fmaf(qv[r][e], kf[e], d);
        s[u][r] = half_warp_sum(d);
      }
    }
#pragma unroll
    for (int r = 0; r < REP; ++r) {
      float mx = m_run[r];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) mx = kv_ok[u] ? fmaxf(mx, s[u][r]) : mx;
      const float alpha = (mx == -INFINITY) ? 1.f : exp2f(m_run[r] - mx);   // nothing seen yet
      l_run[r] *= alpha;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[r][e] *= alpha;
      m_run[r] = mx;
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float vf[8];
      unpack8(vw[u], vf);
#pragma unroll
      for (int r = 0; r < REP; ++r) {
        const float pr = kv_ok[u] ? exp2f(s[u][r] - m_run[r]) : 0.f;
        l_run[r] += pr;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr, vf[e], acc[r][e]);
      }
    }
  }

  // merge the two half-warps (same dims, different keys)
#pragma unroll
  for (int r = 0; r < REP; ++r) {
    const float mo = __shfl_xor_sync(0xffffffffu, m_run[r], 16);
    const float lo = __shfl_xor_sync(0xffffffffu, l_run[r], 16);
    const float mm = fmaxf(m_run[r], mo);
    const float a = (m_run[r] == -INFINITY) ? 0.f : exp2f(m_run[r] - mm);
    const float ao = (mo == -INFINITY) ? 0.f : exp2f(mo - mm);
    l_run[r] = l_run[r] * a + lo * ao;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float oo = __shfl_xor_sync(0xffffffffu, acc[r][e], 16);
      acc[r][e] = acc[r][e] * a + oo * ao;
    }
    m_run[r] = mm;
  }
  if (half == 0) {
#pragma unroll
    for (int r = 0; r < REP; ++r) {
#pragma unroll
      for (int e = 0; e < 8; ++e) s_o[warp][r][sub * 8 + e] = acc[r][e];
      if (sub == 0) {
        s_m[warp][r] = m_run[r];
        s_l[warp][r] = l_run[r];
      }
    }
  }
  __syncthreads();
  // merge the warps: thread t owns dim t of every head of the group
  const int d = threadIdx.x;
#pragma unroll
  for (int r = 0; r < REP; ++r) {
    float mm = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) mm = fmaxf(mm, s_m[w][r]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      const float a = (s_m[w][r] == -INFINITY) ? 0.f : exp2f(s_m[w][r] - mm);
      l += s_l[w][r] * a;
      o += s_o[w][r][d] * a;
    }
    o_part[(part + r * n_split) * HD + d] = o;
    if (d == 0) {
      m_part[part + r * n_split] = mm;
      l_part[part + r * n_split] = l;
    }
  }
}

// out[b, h*D + d] = sum_s e^(m_s - M) O_s[d] / sum_s e^(m_s - M) l_s
__global__ void __launch_bounds__(HD) attn_decode_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ m_part,
                                                                 const float* __restrict__ l_part,
                                                                 __nv_bfloat16* __restrict__ out, int n_split) {
  const long long bh = blockIdx.x;
  const int d = threadIdx.x;
  float mm = -INFINITY;
  for (int s = 0; s < n_split; ++s) mm = fmaxf(mm, m_part[bh * n_split + s]);
  float l = 0.f, o = 0.f;
  if (mm != -INFINITY) {
    for (int s = 0; s < n_split; ++s) {
      const float ms = m_part[bh * n_split + s];
      if (ms == -INFINITY) continue;
      const float a = exp2f(ms - mm);
      l += l_part[bh * n_split + s] * a;
      o += o_part[(bh * n_split + s) * HD + d] * a;
    }
  }
  out[bh * HD + d] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
}

}  // namespace

size_t attn_decode_ws_bytes(int B, int H, int D, int T_max) {
  const size_t n_split = (T_max + SPLIT - 1) / SPLIT;
  const size_t parts = static_cast<size_t>(B) * H * n_split;
  return parts * D * sizeof(float) + 2 * parts * sizeof(float) + 256;
}

int attn_decode(const Ctx& c, int dtype, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* positions, void* out, int B, int H, int G, int D, int T_max, int max_pos, void* ws) {
  if (dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (D != HD) return LLAMA_ERR_UNSUPPORTED;
  const int rep = H / G;
  const int n_split = (T_max + SPLIT - 1) / SPLIT;
  const size_t parts = static_cast<size_t>(B) * H * n_split;
  float* o_part = static_cast<float*>(ws);
  float* m_part = o_part + parts * D;
  float* l_part = m_part + parts;
  const dim3 grid(n_split, G, B);
  const float sl = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  const auto* qq = static_cast<const __nv_bfloat16*>(q);
  const auto* kk = static_cast<const __nv_bfloat16*>(k_cache);
  const auto* vv = static_cast<const __nv_bfloat16*>(v_cache);
  switch (rep) {
    case 1: attn_decode_split_kernel<1><<<grid, WARPS * 32, 0, c.stream>>>(qq, kk, vv, positions, o_part, m_part, l_part, H, G, T_max, max_pos, n_split, sl, c.status); break;
    case 2: attn_decode_split_kernel<2><<<grid, WARPS * 32, 0, c.stream>>>(qq, kk, vv, positions, o_part, m_part, l_part, H, G, T_max, max_pos, n_split, sl, c.status); break;
    case 4: attn_decode_split_kernel<4><<<grid, WARPS * 32, 0, c.stream>>>(qq, kk, vv, positions, o_part, m_part, l_part, H, G, T_max, max_pos, n_split, sl, c.status); break;
    case 8: attn_decode_split_kernel<8><<<grid, WARPS * 32, 0, c.stream>>>(qq, kk, vv, positions, o_part, m_part, l_part, H, G, T_max, max_pos, n_split, sl, c.status); break;
    default: return LLAMA_ERR_UNSUPPORTED;
  }
  int rc = after_launch(c);
  if (rc != LLAMA_OK) return rc;
  attn_decode_combine_kernel<<<B * H, HD, 0, c.stream>>>(o_part, m_part, l_part, static_cast<__nv_bfloat16*>(out),
                                                         n_split);
  return after_launch(c);
}

}  // namespace llama

// ---------------------------------------------------------------------------------------
// Decode attention with its scratch in a fixed device array, for callers that cannot
// allocate device memory: code whose device memory is owned entirely by another allocator
// (a framework's caching pool, a fixed memory budget) and latency-critical loops in which
// cudaMalloc / cudaFree would synchronise the device.  The caller passes inputs and outputs
// only; the split partials live in g_decode_scratch below.

#include <atomic>

namespace llama {
namespace {

// Largest scratch the fixed-array entry point serves: the split partials of
// B * H * ceil(max_T / 512) (query head, key split) pairs, (D + 2) floats each.  At B = 64,
// H = 32, max_T = 4096, D = 128 that is 8.5 MB.
constexpr size_t kDecodeScratchBytes = 16u << 20;

// File-scope device array: every device that loads the library holds its own copy until the
// process exits, and all calls on a device share it.  Each call writes every slot it later
// reads (empty key splits write their neutral (m, l) entry), so nothing needs clearing, but
// two calls that overlap on the GPU (different streams, no ordering) race on it.
static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

// Device address of g_decode_scratch, looked up once per device (host code must not use
// the symbol itself: on the host it only names a stand-in).
std::atomic<void*> g_decode_scratch_addr[64];

}  // namespace
}  // namespace llama

extern "C" int llama_attention_decode_static(const llama_layer_dims* dims, const void* q, llama_kv_cache cache,
                                             const int32_t* positions, void* out, int32_t B, void* cuda_stream) {
  using namespace llama;
  if (dims == nullptr || q == nullptr || out == nullptr || positions == nullptr || cache.k == nullptr ||
      cache.v == nullptr || B <= 0 || cache.max_T <= 0)
    return LLAMA_ERR_INVALID_ARG;
  if (dims->n_heads <= 0 || dims->n_kv_heads <= 0 || dims->n_heads % dims->n_kv_heads != 0)
    return LLAMA_ERR_INVALID_ARG;
  auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (misaligned(q) || misaligned(out) || misaligned(cache.k) || misaligned(cache.v)) return LLAMA_ERR_INVALID_ARG;
  if (dims->dtype != LLAMA_BF16 || dims->head_dim != HD) return LLAMA_ERR_UNSUPPORTED;
  if (attn_decode_ws_bytes(B, dims->n_heads, dims->head_dim, cache.max_T) > kDecodeScratchBytes)
    return LLAMA_ERR_SCRATCH_LIMIT;
  Ctx c;
  int rc = make_ctx(cuda_stream, &c);
  if (rc != LLAMA_OK) return rc;
  void* scratch = g_decode_scratch_addr[c.device].load(std::memory_order_acquire);
  if (scratch == nullptr) {
    // first call on this device (which is current): look the array's device address up
    if (cudaGetSymbolAddress(&scratch, g_decode_scratch) != cudaSuccess || scratch == nullptr)
      return LLAMA_ERR_CUDA;
    g_decode_scratch_addr[c.device].store(scratch, std::memory_order_release);
  }
  return attn_decode(c, dims->dtype, q, cache.k, cache.v, positions, out, B, dims->n_heads, dims->n_kv_heads,
                     dims->head_dim, cache.max_T, cache.max_T, scratch);
}
