// Causal grouped-query flash attention for prefill on the 5th-generation tensor cores.
//
// O_h = softmax(Q_h K_g^T / sqrt(D), key j visible to query i iff j <= i) V_g, g = h / (H/G)
// ("12 · 从 Transformer 到 LLaMA 系列" §八 Attention with is_causal=True and the KV heads
// repeated along dim 1; "深度学习进阶（三十）…" §1.1; "第 10 章：现代 LLaMA 架构" §6: K/V stay
// G heads in the cache and are shared logically, never copied H/G times).
//
// One CTA per (128-query tile, head, sequence), tiles with the most keys first.
//   warp 0     TMA: the Q tile once, then K_j, V_j tiles (128 keys) into a 2-stage ring,
//              read straight from the [B, G, max_T, D] cache
//   warp 1     TMEM allocator and MMA issuer: S_j = Q K_j^T (into one of two TMEM S
//              buffers, so S_{j+1} is computed while the softmax of S_j runs), then
//              O += P_j V_j with V as an MN-major operand
//   warps 2-5  online softmax (one query row per thread, exp2 with the scale folded in),
//              P_j as bf16 into 128-byte-swizzled shared memory, rescale of O in TMEM
//              when the running max moves, and the final O / l epilogue
// fp32 statistics and accumulators; D = 128.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int BQ = 128;
constexpr int BKV = 128;
constexpr int HD = 128;
constexpr int CHUNK = 128 * 128;      // one 64-column half of a 128-row bf16 tile
constexpr int TILE = 2 * CHUNK;       // 128 rows x 128 columns bf16
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;   // S0 [0,128), S1 [128,256), O [256,384)

struct AttnParams {
  int B, S, H, G, n_qt;
  float scale_log2;                   // log2(e) / sqrt(D)
  __nv_bfloat16* out;                 // [B, S, H*D]
  int* status;
};

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + TILE;            // 2 stages
  uint8_t* sV = smem + 3 * TILE;        // 2 stages
  uint8_t* sP = smem + 5 * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * TILE);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;         // [2]
  uint64_t* kv_empty = bars + 3;        // [2]
  uint64_t* s_full = bars + 5;          // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* o_done = bars + 8;
  uint64_t* drain = bars + 9;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = p.n_qt - 1 - static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / (p.H / p.G);
  const int q0 = qt * BQ;
  const int nt = qt + 1;                // key tiles 0..qt

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(kv_full + i), 1);
      mbar_init(smem_u32(kv_empty + i), 1);
      mbar_init(smem_u32(s_full + i), 1);
    }
    mbar_init(smem_u32(p_full), 4);
    mbar_init(smem_u32(o_done), 1);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      bool ok = true;
      int issued = 0;
      const uint32_t qb = smem_u32(q_full);
      mbar_expect_tx(qb, TILE);
      tma_load_3d(smem_u32(sQ), &tmQ, qb, 0, q0, b * p.H + h);
      tma_load_3d(smem_u32(sQ + CHUNK), &tmQ, qb, 64, q0, b * p.H + h);
      for (int j = 0; j < nt; ++j) {
        const int st = j & 1;
        if (!mbar_wait(smem_u32(kv_empty + st), ((j >> 1) & 1) ^ 1u, p.status, abort_flag)) { ok = false; break; }
        const uint32_t fb = smem_u32(kv_full + st);
        mbar_expect_tx(fb, 2 * TILE);
        const int row = j * BKV, plane = b * p.G + g;
        tma_load_3d(smem_u32(sK + st * TILE), &tmK, fb, 0, row, plane);
        tma_load_3d(smem_u32(sK + st * TILE + CHUNK), &tmK, fb, 64, row, plane);
        tma_load_3d(smem_u32(sV + st * TILE), &tmV, fb, 0, row, plane);
        tma_load_3d(smem_u32(sV + st * TILE + CHUNK), &tmV, fb, 64, row, plane);
        ++issued;
      }
      if (!ok) {
        mbar_wait_slow(qb, 0, nullptr, nullptr, kWaitBudgetNs);
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
          mbar_wait_slow(smem_u32(kv_full + (j & 1)), (j >> 1) & 1, nullptr, nullptr, kWaitBudgetNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false);
      constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, true);
      const uint32_t aq = smem_u32(sQ), ap = smem_u32(sP);
      bool ok = mbar_wait(smem_u32(q_full), 0, p.status, abort_flag) &&
                mbar_wait(smem_u32(kv_full), 0, p.status, abort_flag);
      bool issued = false;
      auto issue_qk = [&](int sbuf, int st) {
        const uint32_t bk = smem_u32(sK + st * TILE);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
          tc_mma_bf16(tmem_base + sbuf * 128, sdesc_sw128(aq + off, 16, 1024), sdesc_sw128(bk + off, 16, 1024),
                      IDESC_QK, kk > 0 ? 1u : 0u);
        }
      };
      if (ok) {
        tc_fence_after();
        issue_qk(0, 0);
        issued = true;
        tc_commit(smem_u32(s_full));
      }
      for (int j = 0; j < nt && ok; ++j) {
        if (j + 1 < nt) {
          const int st1 = (j + 1) & 1;
          if (!mbar_wait(smem_u32(kv_full + st1), ((j + 1) >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
          tc_fence_after();
          issue_qk(st1, st1);
          tc_commit(smem_u32(s_full + st1));
        }
        if (!mbar_wait(smem_u32(p_full), j & 1, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t bv = smem_u32(sV + (j & 1) * TILE);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(ap + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024);
          // V tile: 128 key rows of 128 bytes per 64-wide d half; K step = 16 rows = 2048 bytes,
          // the second d half is CHUNK bytes further (leading byte offset), 8-row groups 1024 apart
          const uint64_t bd = sdesc_sw128(bv + kk * 2048, CHUNK, 1024);
          tc_mma_bf16(tmem_base + 256, ad, bd, IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(o_done));
        tc_commit(smem_u32(kv_empty + (j & 1)));
      }
      if (!ok && issued) {
        tc_commit(smem_u32(drain));
        mbar_wait_slow(smem_u32(drain), 0, nullptr, nullptr, kWaitBudgetNs);
      }
    }
  } else {
    // -------------------------------------------------------------- softmax warps 2..5
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = q0 + row;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t r[32];
    bool ok = true;
    uint8_t* prow = sP + row * 128;
    const uint32_t swz = static_cast<uint32_t>(row & 7);
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(smem_u32(s_full + sb), (j >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem_base + t_lane + sb * 128;
      const bool diag = (j == qt);
      const int kbase = j * BKV;
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tS + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float s = __uint_as_float(r[i]);
          const int key = kbase + c * 32 + i;
          if (diag && (key > qi || key >= p.S)) s = -INFINITY;
          mx = fmaxf(mx, s);
        }
      }
      const float m_new = fmaxf(m_run, mx * sl);
      const float alpha = exp2f(m_run - m_new);
      if (j > 0) {
        // P_{j-1} V_{j-1} must be complete before O is rescaled and P is overwritten
        if (!mbar_wait(smem_u32(o_done), (j - 1) & 1, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(tmem_base + t_lane + 256 + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tmem_base + t_lane + 256 + c * 32, r);
          }
        }
      }
      float rowsum = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tS + c * 32, r);
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = kbase + c * 32 + i;
          const bool masked = diag && (key > qi || key >= p.S);
          pv[i] = masked ? 0.f : exp2f(fmaf(__uint_as_float(r[i]), sl, -m_new));
          rowsum += pv[i];
        }
        // keys c*32 .. c*32+31 live in 64-key chunk (c >> 1), 16-byte units (c & 1)*4 + u
        uint8_t* base = prow + (c >> 1) * CHUNK;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t unit = static_cast<uint32_t>((c & 1) * 4 + u) ^ swz;
          uint4 w;
          w.x = pack_bf16(pv[8 * u + 0], pv[8 * u + 1]);
          w.y = pack_bf16(pv[8 * u + 2], pv[8 * u + 3]);
          w.z = pack_bf16(pv[8 * u + 4], pv[8 * u + 5]);
          w.w = pack_bf16(pv[8 * u + 6], pv[8 * u + 7]);
          *reinterpret_cast<uint4*>(base + unit * 16) = w;
        }
      }
      l_run = l_run * alpha + rowsum;
      m_run = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(p_full));
    }
    if (ok && mbar_wait(smem_u32(o_done), (nt - 1) & 1, p.status, abort_flag)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      __nv_bfloat16* dst = p.out + (static_cast<long long>(b) * p.S + qi) * (static_cast<long long>(p.H) * HD) + h * HD;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tmem_base + t_lane + 256 + c * 32, r);
        if (qi < p.S) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(r[8 * u + 0]) * inv_l, __uint_as_float(r[8 * u + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(r[8 * u + 2]) * inv_l, __uint_as_float(r[8 * u + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(r[8 * u + 4]) * inv_l, __uint_as_float(r[8 * u + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(r[8 * u + 6]) * inv_l, __uint_as_float(r[8 * u + 7]) * inv_l);
            d4[u] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

constexpr size_t kSmemBytes = 1024 + 6 * TILE + 11 * 8 + 16;

}  // namespace

int attn_prefill_tc(const Ctx& c, const void* q, const void* k_cache, const void* v_cache, void* out, int B, int S,
                    int H, int G, int D, int T_max) {
  if (D != HD) return LLAMA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv;
  // Q [B*H][S][D]; K, V: valid slots [0, S) of [B*G][T_max][D] (rows >= S read as 0)
  if (!make_tmap_3d(&tq, q, HD, S, static_cast<uint64_t>(B) * H, HD, static_cast<uint64_t>(S) * HD, BQ) ||
      !make_tmap_3d(&tk, k_cache, HD, S, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD, BKV) ||
      !make_tmap_3d(&tv, v_cache, HD, S, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD, BKV))
    return LLAMA_ERR_INVALID_ARG;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBytes));
  });
  if (attr_err != cudaSuccess) return LLAMA_ERR_CUDA;
  AttnParams p;
  p.B = B;
  p.S = S;
  p.H = H;
  p.G = G;
  p.n_qt = (S + BQ - 1) / BQ;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = c.status;
  attn_prefill_kernel<<<dim3(p.n_qt, H, B), NUM_THREADS, kSmemBytes, c.stream>>>(tq, tk, tv, p);
  return after_launch(c);
}

}  // namespace llama
