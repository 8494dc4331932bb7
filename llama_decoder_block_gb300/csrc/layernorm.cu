// LayerNorm: y = gamma * (x - mu) * rsqrt(var + eps) + beta, one warp per row, with mu the
// row mean and var the biased row variance ("3.2 核心组件逐一拆解" §3.2.1, LayerNorm).
//
// Not a step of the decoder layer, which uses RMSNorm: it exists so that the two
// normalisations can be timed against each other on the same rows.  Same structure
// as rmsnorm.cu: every row is read once and written once, and the bf16 kernel keeps
// the whole row in registers, so the centred second moment costs no extra memory
// traffic (only a second warp reduction), and gamma and beta are two parameter reads.
#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int kWarpsPerCta = 2;   // small CTAs: the last wave of rows is short (measured best of 2, 4, 8, 16)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// bf16, d == VPL * 256: lane owns VPL 16-byte vectors (8 elements each) of its row.
template <int VPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    layernorm_bf16_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma,
                          const uint4* __restrict__ beta, uint4* __restrict__ y, int rows, float inv_d, float eps) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* xr = x + static_cast<long long>(row) * (VPL * 32);
  uint4 v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[i] = __ldcs(xr + i * 32 + lane);
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) s += bf16_lo(w[j]) + bf16_hi(w[j]);
  }
  const float mu = warp_sum(s) * inv_d;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]) - mu, b = bf16_hi(w[j]) - mu;
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  const float r = rsqrtf(warp_sum(ss) * inv_d + eps);
  uint4* yr = y + static_cast<long long>(row) * (VPL * 32);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint4 g = __ldg(gamma + i * 32 + lane);
    const uint4 bt = __ldg(beta + i * 32 + lane);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    const uint32_t bw[4] = {bt.x, bt.y, bt.z, bt.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16(fmaf(bf16_lo(gw[j]), (bf16_lo(w[j]) - mu) * r, bf16_lo(bw[j])),
                       fmaf(bf16_hi(gw[j]), (bf16_hi(w[j]) - mu) * r, bf16_hi(bw[j])));
    __stcs(yr + i * 32 + lane, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// Any d and either dtype: three passes over the row (the later ones hit L1).
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    layernorm_generic_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
                             T* __restrict__ y, int rows, int d, float eps) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* xr = x + static_cast<long long>(row) * d;
  float s = 0.f;
  for (int i = lane; i < d; i += 32) s += static_cast<float>(xr[i]);
  const float mu = warp_sum(s) / static_cast<float>(d);
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float a = static_cast<float>(xr[i]) - mu;
    ss = fmaf(a, a, ss);
  }
  const float r = rsqrtf(warp_sum(ss) / static_cast<float>(d) + eps);
  T* yr = y + static_cast<long long>(row) * d;
  for (int i = lane; i < d; i += 32)
    yr[i] = static_cast<T>(
        fmaf(static_cast<float>(gamma[i]), (static_cast<float>(xr[i]) - mu) * r, static_cast<float>(beta[i])));
}

}  // namespace

int layernorm(const Ctx& c, const void* x, const void* gamma, const void* beta, void* y, int rows, int d, float eps,
              int dtype) {
  if (rows == 0) return LLAMA_OK;
  const dim3 grid((rows + kWarpsPerCta - 1) / kWarpsPerCta), block(kWarpsPerCta * 32);
  if (dtype == LLAMA_BF16 && d % 256 == 0 && d <= 4096 && (d / 256 & (d / 256 - 1)) == 0) {
    const uint4* xv = static_cast<const uint4*>(x);
    const uint4* gv = static_cast<const uint4*>(gamma);
    const uint4* bv = static_cast<const uint4*>(beta);
    uint4* yv = static_cast<uint4*>(y);
    const float inv_d = 1.0f / static_cast<float>(d);
    switch (d / 256) {
      case 1: launch_pdl(c, layernorm_bf16_kernel<1>, grid, block, 0, xv, gv, bv, yv, rows, inv_d, eps); break;
      case 2: launch_pdl(c, layernorm_bf16_kernel<2>, grid, block, 0, xv, gv, bv, yv, rows, inv_d, eps); break;
      case 4: launch_pdl(c, layernorm_bf16_kernel<4>, grid, block, 0, xv, gv, bv, yv, rows, inv_d, eps); break;
      case 8: launch_pdl(c, layernorm_bf16_kernel<8>, grid, block, 0, xv, gv, bv, yv, rows, inv_d, eps); break;
      default: launch_pdl(c, layernorm_bf16_kernel<16>, grid, block, 0, xv, gv, bv, yv, rows, inv_d, eps); break;
    }
  } else if (dtype == LLAMA_BF16) {
    launch_pdl(c, layernorm_generic_kernel<__nv_bfloat16>, grid, block, 0, static_cast<const __nv_bfloat16*>(x),
               static_cast<const __nv_bfloat16*>(gamma), static_cast<const __nv_bfloat16*>(beta),
               static_cast<__nv_bfloat16*>(y), rows, d, eps);
  } else {
    launch_pdl(c, layernorm_generic_kernel<float>, grid, block, 0, static_cast<const float*>(x),
               static_cast<const float*>(gamma), static_cast<const float*>(beta), static_cast<float*>(y), rows, d,
               eps);
  }
  return after_launch(c);
}

}  // namespace llama
