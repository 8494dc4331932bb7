// RMSNorm: y = gamma * x * rsqrt(mean(x^2) + eps), one warp per row.
// "12 · 从 Transformer 到 LLaMA 系列" §八 RMSNorm; "3.2 核心组件逐一拆解" §3.2.1 (the sum of
// squares and the scaling in fp32, the result cast back to the storage type).
//
// HBM-bound: every row is read once and written once.  A lane issues all of its
// 16-byte loads of the row before the warp reduction, so each warp keeps a whole
// row (8 KB at d = 4096, bf16) in flight.
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
    rmsnorm_bf16_kernel(const uint4* __restrict__ x, const uint4* __restrict__ gamma, uint4* __restrict__ y, int rows,
                        float inv_d, float eps) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* xr = x + static_cast<long long>(row) * (VPL * 32);
  uint4 v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[i] = __ldcs(xr + i * 32 + lane);   // streamed once
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w[j]), b = bf16_hi(w[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss * inv_d + eps);
  uint4* yr = y + static_cast<long long>(row) * (VPL * 32);
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint4 g = __ldg(gamma + i * 32 + lane);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = pack_bf16(bf16_lo(gw[j]) * (bf16_lo(w[j]) * r), bf16_hi(gw[j]) * (bf16_hi(w[j]) * r));
    __stcs(yr + i * 32 + lane, make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// Any d and either dtype: two passes over the row (the second one hits L1).
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    rmsnorm_generic_kernel(const T* __restrict__ x, const T* __restrict__ gamma, T* __restrict__ y, int rows, int d,
                           float eps) {
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* xr = x + static_cast<long long>(row) * d;
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float a = static_cast<float>(xr[i]);
    ss = fmaf(a, a, ss);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / static_cast<float>(d) + eps);
  T* yr = y + static_cast<long long>(row) * d;
  for (int i = lane; i < d; i += 32)
    yr[i] = static_cast<T>(static_cast<float>(gamma[i]) * (static_cast<float>(xr[i]) * r));
}

}  // namespace

int rmsnorm(const Ctx& c, const void* x, const void* gamma, void* y, int rows, int d, float eps, int dtype) {
  if (rows == 0) return LLAMA_OK;
  const dim3 grid((rows + kWarpsPerCta - 1) / kWarpsPerCta), block(kWarpsPerCta * 32);
  if (dtype == LLAMA_BF16 && d % 256 == 0 && d <= 4096) {
    const uint4* xv = static_cast<const uint4*>(x);
    const uint4* gv = static_cast<const uint4*>(gamma);
    uint4* yv = static_cast<uint4*>(y);
    const float inv_d = 1.0f / static_cast<float>(d);
    switch (d / 256) {
      case 1: launch_pdl(c, rmsnorm_bf16_kernel<1>, grid, block, 0, xv, gv, yv, rows, inv_d, eps); break;
      case 2: launch_pdl(c, rmsnorm_bf16_kernel<2>, grid, block, 0, xv, gv, yv, rows, inv_d, eps); break;
      case 4: launch_pdl(c, rmsnorm_bf16_kernel<4>, grid, block, 0, xv, gv, yv, rows, inv_d, eps); break;
      case 8: launch_pdl(c, rmsnorm_bf16_kernel<8>, grid, block, 0, xv, gv, yv, rows, inv_d, eps); break;
      case 16: launch_pdl(c, rmsnorm_bf16_kernel<16>, grid, block, 0, xv, gv, yv, rows, inv_d, eps); break;
      default:
        launch_pdl(c, rmsnorm_generic_kernel<__nv_bfloat16>, grid, block, 0, static_cast<const __nv_bfloat16*>(x),
                   static_cast<const __nv_bfloat16*>(gamma), static_cast<__nv_bfloat16*>(y), rows, d, eps);
    }
  } else if (dtype == LLAMA_BF16) {
    launch_pdl(c, rmsnorm_generic_kernel<__nv_bfloat16>, grid, block, 0, static_cast<const __nv_bfloat16*>(x),
               static_cast<const __nv_bfloat16*>(gamma), static_cast<__nv_bfloat16*>(y), rows, d, eps);
  } else {
    launch_pdl(c, rmsnorm_generic_kernel<float>, grid, block, 0, static_cast<const float*>(x),
               static_cast<const float*>(gamma), static_cast<float*>(y), rows, d, eps);
  }
  return after_launch(c);
}

}  // namespace llama
