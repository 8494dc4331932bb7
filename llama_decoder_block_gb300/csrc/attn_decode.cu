// Decode attention: one new query per sequence over its cached keys, split along the keys.
//
// Query of sequence b sits at position p = positions[b] and sees cache slots 0..p
// ("第 10 章：现代 LLaMA 架构" §7: q_len = 1, k_len = past_len + 1, score shape
// [B, H, 1, T_cache + 1]; §6: the G cached K/V heads are shared by H/G query heads).
//
// HBM-bound: the cache is read once, by TMA, 128 keys (32 KB of K and 32 KB of V) per
// tile through a 3-stage ring.  A persistent CTA walks work items (sequence b, KV head g,
// 1024-key split) and keeps the ring full across items.  The products run on the tensor
// cores with the keys as the 128-row dimension: S^T = K Q^T (M = 128 keys, N = 16 query-head
// columns of which H/G are real) and O^T += V^T P^T (M = 128 head dims, V read as an
// MN-major operand straight from the cache layout), so the SIMT work per key is one row of
// the online softmax per thread.  P^T and the TMEM S^T are double-buffered, so the softmax
// of tile t overlaps the products of tile t-1.  Each item leaves (m, l, O) for its split;
// the combine kernel merges the splits.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int HD = 128;
constexpr int SPLIT = 1024;                 // keys per work item
constexpr int KT = 128;                     // keys per tile
constexpr int NQ = 16;                      // query-head columns of the MMAs (H/G <= 8 real)
constexpr int STAGES = 3;
constexpr int KV_CHUNK = KT * 128;          // 64 head dims of 128 keys, bf16: 16 KB
constexpr int KV_TILE = 2 * KV_CHUNK;       // 32 KB
constexpr int Q_CHUNK = NQ * 128;           // 64 head dims of 16 query rows: 2 KB
constexpr int Q_TILE = 2 * Q_CHUNK;
constexpr int P_CHUNK = NQ * 128;           // 64 keys of 16 query rows: 2 KB
constexpr int P_TILE = 2 * P_CHUNK;
constexpr int DEC_THREADS = 192;            // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr uint32_t DEC_TMEM_COLS = 64;      // S^T buffers at 0 and 16, O^T buffers at 32 and 48
constexpr int POS_CACHE = 1024;             // positions staged in shared memory (larger B reads global)
constexpr float kDecRescaleLog2 = 8.0f;

struct DecParams {
  const int32_t* positions;
  float* o_part;
  float* m_part;
  float* l_part;
  int B, H, G, T_max, max_pos, n_split, n_items;
  float scale_log2;
  int* status;
};

struct DecItem {
  int b, g, c, k_begin, k_end, ntile;
  bool bad_position;
};

__device__ __forceinline__ DecItem dec_item(const DecParams& p, const int* pos_s, int it) {
  DecItem d;
  d.c = it % p.n_split;
  d.g = (it / p.n_split) % p.G;
  d.b = it / (p.n_split * p.G);
  const int pos = d.b < POS_CACHE ? pos_s[d.b] : p.positions[d.b];
  const bool ok = pos >= 0 && pos < p.T_max && pos < p.max_pos;
  d.bad_position = !ok;
  const int n_keys = ok ? pos + 1 : 0;
  d.k_begin = d.c * SPLIT;
  d.k_end = min(d.k_begin + SPLIT, n_keys);
  d.ntile = d.k_end > d.k_begin ? (d.k_end - d.k_begin + KT - 1) / KT : 0;
  return d;
}

template <int REP>
__global__ void __launch_bounds__(DEC_THREADS, 1)
    attn_decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const DecParams p) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + STAGES * KV_TILE;
  uint8_t* sQ = smem + 2 * STAGES * KV_TILE;            // 2 slots
  uint8_t* sP = sQ + 2 * Q_TILE;                         // 2 buffers of P^T: 16 rows x 128 keys
  float* red = reinterpret_cast<float*>(sP + 2 * P_TILE);   // [2 buffers][4 warps][8 heads]
  int* pos_s = reinterpret_cast<int*>(red + 64);            // [POS_CACHE]
  uint64_t* bars = reinterpret_cast<uint64_t*>(pos_s + POS_CACHE);
  uint64_t* kv_full = bars;                  // [STAGES]
  uint64_t* kv_empty = bars + STAGES;        // [STAGES]
  uint64_t* q_full = bars + 2 * STAGES;      // [2]
  uint64_t* q_empty = q_full + 2;            // [2]
  uint64_t* s_full = q_empty + 2;            // [2]
  uint64_t* o_done = s_full + 2;             // [2] by the parity of the tile
  uint64_t* p_full = o_done + 2;
  uint64_t* o_free = p_full + 1;             // [2] by the parity of the item
  uint64_t* drain = o_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(kv_full + i), 1);
      mbar_init(smem_u32(kv_empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(q_full + i), 1);
      mbar_init(smem_u32(q_empty + i), 1);
      mbar_init(smem_u32(s_full + i), 1);
      mbar_init(smem_u32(o_done + i), 1);
    }
    mbar_init(smem_u32(p_full), 4);
    mbar_init(smem_u32(o_free), 4);
    mbar_init(smem_u32(o_free + 1), 4);
    mbar_init(smem_u32(drain), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  pdl_wait();   // positions may come from the previous kernel
  for (int i = threadIdx.x; i < min(p.B, POS_CACHE); i += DEC_THREADS) pos_s[i] = p.positions[i];
  // P^T rows beyond H/G stay zero (their O^T columns are never read)
  for (int i = threadIdx.x; i < 2 * P_TILE / 16; i += DEC_THREADS)
    reinterpret_cast<uint4*>(sP)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), DEC_TMEM_COLS);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();   // inputs written by the previous kernel are read from here on

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t tcount = 0, icount = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
        const DecItem d = dec_item(p, pos_s, it);
        if (d.ntile == 0) continue;
        const uint32_t qs = icount & 1;
        if (!mbar_wait(smem_u32(q_empty + qs), ((icount >> 1) & 1) ^ 1u, p.status, abort_flag)) { ok = false; break; }
        mbar_expect_tx(smem_u32(q_full + qs), Q_TILE);
        const int qrow = d.b * p.H + d.g * REP;
        tma_load_2d(smem_u32(sQ + qs * Q_TILE), &tmQ, smem_u32(q_full + qs), 0, qrow);
        tma_load_2d(smem_u32(sQ + qs * Q_TILE + Q_CHUNK), &tmQ, smem_u32(q_full + qs), 64, qrow);
        const int plane = d.b * p.G + d.g;
        for (int t = 0; t < d.ntile; ++t, ++tcount) {
          const uint32_t st = tcount % STAGES;
          if (!mbar_wait(smem_u32(kv_empty + st), ((tcount / STAGES) & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(kv_full + st);
          mbar_expect_tx(fb, 2 * KV_TILE);
          const int row = d.k_begin + t * KT;
          tma_load_3d(smem_u32(sK + st * KV_TILE), &tmK, fb, 0, row, plane);
          tma_load_3d(smem_u32(sK + st * KV_TILE + KV_CHUNK), &tmK, fb, 64, row, plane);
          tma_load_3d(smem_u32(sV + st * KV_TILE), &tmV, fb, 0, row, plane);
          tma_load_3d(smem_u32(sV + st * KV_TILE + KV_CHUNK), &tmV, fb, 64, row, plane);
        }
        ++icount;
      }
      if (!ok) {   // leave no copy in flight: wait for the last load issued into each stage
        for (uint32_t s = 0; s < STAGES; ++s) {
          if (tcount <= s) continue;
          const uint32_t last = tcount - 1 - ((tcount - 1 - s) % STAGES);
          mbar_wait_slow(smem_u32(kv_full + s), (last / STAGES) & 1, nullptr, nullptr, kWaitBudgetNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t IDESC_S = idesc_bf16(128, NQ, false);
      constexpr uint32_t IDESC_O = idesc_bf16(128, NQ, false, true);
      uint32_t tcount = 0, icount = 0;
      bool ok = true, issued = false;
      auto issue_pv = [&](uint32_t tc, bool first, uint32_t ob) -> bool {
        if (!mbar_wait(smem_u32(p_full), tc & 1, p.status, abort_flag)) return false;
        // O^T buffer ob was last read by the epilogue of the item two before this one
        if (first && icount >= 2 && !mbar_wait(smem_u32(o_free + ob), ((icount - 2) >> 1) & 1, p.status, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t av = smem_u32(sV + (tc % STAGES) * KV_TILE), bp = smem_u32(sP + (tc & 1) * P_TILE);
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          // A = V^T: 128 head dims (MN-major: a 64-dim half per 128-byte row, the other half
          // KV_CHUNK bytes further), K step = 16 keys = 2048 bytes; B = P^T: 16 rows of keys
          tc_mma_bf16(tmem_base + 32 + ob * 16, sdesc_sw128(av + kk * 2048, KV_CHUNK, 1024),
                      sdesc_sw128(bp + (kk >> 2) * P_CHUNK + (kk & 3) * 32, 16, 1024), IDESC_O,
                      (first && kk == 0) ? 0u : 1u);
        }
        tc_commit(smem_u32(o_done + (tc & 1)));
        tc_commit(smem_u32(kv_empty + (tc % STAGES)));
        return true;
      };
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
        const DecItem d = dec_item(p, pos_s, it);
        if (d.ntile == 0) continue;
        const uint32_t qs = icount & 1;
        if (!mbar_wait(smem_u32(q_full + qs), (icount >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
        const uint32_t aq = smem_u32(sQ + qs * Q_TILE);
        for (int t = 0; t < d.ntile && ok; ++t) {
          const uint32_t tc = tcount + t, st = tc % STAGES;
          if (!mbar_wait(smem_u32(kv_full + st), (tc / STAGES) & 1, p.status, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t ak = smem_u32(sK + st * KV_TILE);
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * KV_CHUNK + (kk & 3) * 32;
            tc_mma_bf16(tmem_base + (tc & 1) * 16, sdesc_sw128(ak + off, 16, 1024),
                        sdesc_sw128(aq + (kk >> 2) * Q_CHUNK + (kk & 3) * 32, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(smem_u32(s_full + (tc & 1)));
          if (t > 0 && !issue_pv(tc - 1, t == 1, icount & 1)) { ok = false; break; }
        }
        if (!ok) break;
        tc_commit(smem_u32(q_empty + qs));
        if (!issue_pv(tcount + d.ntile - 1, d.ntile == 1, icount & 1)) { ok = false; break; }
        tcount += d.ntile;
        ++icount;
      }
      if (!ok && issued) {
        tc_commit(smem_u32(drain));
        mbar_wait_slow(smem_u32(drain), 0, nullptr, nullptr, kWaitBudgetNs);
      }
    }
  } else {
    // -------------------------------------------------------------- softmax and epilogue
    const int sw = warp - 2;                          // 0..3
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;             // key of the tile (S^T) / head dim (O^T)
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl = p.scale_log2;
    uint32_t tcount = 0, icount = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const DecItem d = dec_item(p, pos_s, it);
      const long long part = (static_cast<long long>(d.b) * p.H + d.g * REP) * p.n_split + d.c;
      if (d.ntile == 0) {   // empty split: the neutral element of the merge
        if (d.bad_position && d.c == 0 && d.g == 0 && sw == 0 && lane == 0) report(p.status, LLAMA_ERR_DEVICE_BOUNDS);
        if (sw == 0 && lane < REP) {
          p.m_part[part + lane * p.n_split] = -INFINITY;
          p.l_part[part + lane * p.n_split] = 0.f;
        }
        continue;
      }
      float m_run[REP], lsum[REP];
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        m_run[h] = -INFINITY;
        lsum[h] = 0.f;
      }
      for (int t = 0; t < d.ntile; ++t, ++tcount) {
        const uint32_t pb = tcount & 1;
        if (!mbar_wait(smem_u32(s_full + pb), (tcount >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[8];
        {
          uint32_t a[4], b4[4];
          tmem_ld4(tmem_base + t_lane + pb * 16, a);
          if (REP > 4) tmem_ld4(tmem_base + t_lane + pb * 16 + 4, b4);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            sr[h] = a[h];
            sr[4 + h] = REP > 4 ? b4[h] : 0u;
          }
        }
        const int key = d.k_begin + t * KT + row;
        const bool valid = key < d.k_end;
        float* rb = red + pb * 32;
        float s[REP];
#pragma unroll
        for (int h = 0; h < REP; ++h) {
          s[h] = valid ? __uint_as_float(sr[h]) * sl : -INFINITY;
          float v = s[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) rb[sw * 8 + h] = v;
        }
        named_barrier(1, 128);   // red is double-buffered by tile parity: one barrier per tile
        bool need = false;
        float alpha[REP], pv[REP];
#pragma unroll
        for (int h = 0; h < REP; ++h) {
          const float tmax = fmaxf(fmaxf(rb[h], rb[8 + h]), fmaxf(rb[16 + h], rb[24 + h]));
          const bool nh = tmax > m_run[h] + kDecRescaleLog2;
          const float m_new = nh ? tmax : m_run[h];
          alpha[h] = nh ? ex2_approx(m_run[h] - m_new) : 1.0f;
          m_run[h] = m_new;
          need |= nh;
          pv[h] = valid ? ex2_approx(s[h] - m_new) : 0.f;
          lsum[h] = lsum[h] * alpha[h] + pv[h];
        }
        // O^T rescale: the previous tile's product must have landed (same decision in every
        // thread: the tile maxima and m_run are shared)
        if (need && t > 0) {
          const uint32_t prev = tcount - 1;
          if (!mbar_wait(smem_u32(o_done + (prev & 1)), (prev >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t to = tmem_base + t_lane + 32 + (icount & 1) * 16;
          uint32_t oa[4], ob[4];
          tmem_ld4(to, oa);
          if (REP > 4) tmem_ld4(to + 4, ob);
#pragma unroll
          for (int h = 0; h < REP; ++h) {
            if (h < 4) oa[h] = __float_as_uint(__uint_as_float(oa[h]) * alpha[h]);
            else ob[h - 4] = __float_as_uint(__uint_as_float(ob[h - 4]) * alpha[h]);
          }
          tmem_st4(to, oa);
          if (REP > 4) tmem_st4(to + 4, ob);
        }
        // P^T buffer pb was last read by the product of tile tcount - 2
        if (tcount >= 2) {
          const uint32_t prev2 = tcount - 2;
          if (!mbar_wait(smem_u32(o_done + pb), (prev2 >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
        }
        // P^T[h][key]: row h (128-byte rows, 16-byte units swizzled by h % 8), key `row`
        {
          uint8_t* pbuf = sP + pb * P_TILE + (row >> 6) * P_CHUNK;
          const int unit = (row & 63) >> 3, within = (row & 7) * 2;
#pragma unroll
          for (int h = 0; h < REP; ++h)
            *reinterpret_cast<__nv_bfloat16*>(pbuf + h * 128 + ((unit ^ (h & 7)) << 4) + within) =
                __float2bfloat16_rn(pv[h]);
        }
        // keys past the sequence end: zero their V rows so that 0 * (stale value) stays 0;
        // the warp clears one 256-byte row at a time, 16 bytes per lane (no bank conflicts)
        {
          uint32_t bad = __ballot_sync(0xffffffffu, !valid);
          uint8_t* vs = sV + (tcount % STAGES) * KV_TILE;
          while (bad != 0u) {
            const int r = quarter * 32 + __ffs(bad) - 1;
            bad &= bad - 1u;
            if (lane < 16)
              *reinterpret_cast<uint4*>(vs + (lane >> 3) * KV_CHUNK + r * 128 + (lane & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(p_full));
      }
      if (!ok) break;
      // item epilogue: wait for the last product, write this split's (m, l, O)
      const uint32_t last = tcount - 1;
      if (!mbar_wait(smem_u32(o_done + (last & 1)), (last >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t oa[4], ob[4];
      tmem_ld4(tmem_base + t_lane + 32 + (icount & 1) * 16, oa);
      if (REP > 4) tmem_ld4(tmem_base + t_lane + 36 + (icount & 1) * 16, ob);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(o_free + (icount & 1)));
      float* rb = red + (last & 1) * 32;   // free: every thread passed this tile's barrier
      named_barrier(1, 128);
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        float v = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) rb[sw * 8 + h] = v;
      }
      named_barrier(1, 128);
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        const float o = h < 4 ? __uint_as_float(oa[h]) : __uint_as_float(ob[h - 4]);
        p.o_part[(part + h * p.n_split) * HD + row] = o;
        if (row == 0) {
          p.m_part[part + h * p.n_split] = m_run[h];
          p.l_part[part + h * p.n_split] = rb[h] + rb[8 + h] + rb[16 + h] + rb[24 + h];
        }
      }
      named_barrier(1, 128);   // rb is reused by the next item's first tiles
      ++icount;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, DEC_TMEM_COLS);
  }
}

constexpr size_t kDecSmemBytes = 1024 + 2 * STAGES * KV_TILE + 2 * Q_TILE + 2 * P_TILE + 64 * 4 + POS_CACHE * 4 +
                                 (2 * STAGES + 13) * 8 + 16;

// out[b, h*D + d] = sum_s e^(m_s - M) O_s[d] / sum_s e^(m_s - M) l_s
__global__ void __launch_bounds__(HD) attn_decode_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ m_part,
                                                                 const float* __restrict__ l_part,
                                                                 __nv_bfloat16* __restrict__ out, int n_split) {
  pdl_trigger();
  pdl_wait();
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

template <int REP>
cudaError_t launch_decode(const Ctx& c, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecParams& p) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_decode_tc_kernel<REP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kDecSmemBytes));
  });
  if (attr_err != cudaSuccess) return attr_err;
  return launch_pdl(c, attn_decode_tc_kernel<REP>, dim3(std::min(p.n_items, c.num_sms)), dim3(DEC_THREADS),
                    kDecSmemBytes, tq, tk, tv, p);
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
  const int rep = H / G;
  if (D != HD) return LLAMA_ERR_UNSUPPORTED;
  const int n_split = (T_max + SPLIT - 1) / SPLIT;
  const size_t parts = static_cast<size_t>(B) * H * n_split;
  DecParams p;
  p.o_part = static_cast<float*>(ws);
  p.m_part = p.o_part + parts * D;
  p.l_part = p.m_part + parts;
  p.positions = positions;
  p.B = B;
  p.H = H;
  p.G = G;
  p.T_max = T_max;
  p.max_pos = max_pos;
  p.n_split = n_split;
  p.n_items = B * G * n_split;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  p.status = c.status;
  CUtensorMap tq, tk, tv;
  // Q [B*H][D] in 16-row boxes (the group's H/G heads, then padding rows that are ignored);
  // K, V [B*G][T_max][D] in 128-key boxes (keys past T_max read as 0)
  if (!make_tmap_2d(&tq, q, HD, static_cast<uint64_t>(B) * H, HD, NQ) ||
      !make_tmap_3d(&tk, k_cache, HD, T_max, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD, KT) ||
      !make_tmap_3d(&tv, v_cache, HD, T_max, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD, KT))
    return LLAMA_ERR_INVALID_ARG;
  cudaError_t err;
  switch (rep) {
    case 1: err = launch_decode<1>(c, tq, tk, tv, p); break;
    case 2: err = launch_decode<2>(c, tq, tk, tv, p); break;
    case 4: err = launch_decode<4>(c, tq, tk, tv, p); break;
    case 8: err = launch_decode<8>(c, tq, tk, tv, p); break;
    default: return LLAMA_ERR_UNSUPPORTED;
  }
  if (err != cudaSuccess) return LLAMA_ERR_CUDA;
  int rc = after_launch(c);
  if (rc != LLAMA_OK) return rc;
  launch_pdl(c, attn_decode_combine_kernel, dim3(B * H), dim3(HD), 0, p.o_part, p.m_part, p.l_part,
             static_cast<__nv_bfloat16*>(out), n_split);
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
// B * H * ceil(max_T / 1024) (query head, key split) pairs, (D + 2) floats each.  At B = 64,
// H = 32, max_T = 4096, D = 128 that is 4.3 MB.
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
