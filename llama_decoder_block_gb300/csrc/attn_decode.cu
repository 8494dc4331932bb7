// Decode attention: one new query per sequence over its cached keys, split along the keys.
//
// Query of sequence b sits at position p = positions[b] and sees cache slots 0..p
// ("第 10 章：现代 LLaMA 架构" §7: q_len = 1, k_len = past_len + 1, score shape
// [B, H, 1, T_cache + 1]; §6: the G cached K/V heads are shared by H/G query heads).
//
// HBM-bound: the cache is read once, by TMA, 128 keys (32 KB of K and 32 KB of V) per
// tile through a 3-stage ring.  The work is balanced over the persistent CTAs: all
// (sequence b, KV head g, key tile) triples are laid out on one axis, ordered by b, then g,
// then tile, and CTA c takes the c-th of gridDim.x equal ranges of it.  A CTA's range falls
// into segments, one per (b, g) it touches, and the ring stays full across segments.  The products run on the tensor
// cores with the keys as the 128-row dimension: S^T = K Q^T (M = 128 keys, N = 16 query-head
// columns of which H/G are real) and O^T += V^T P^T (M = 128 head dims, V read as an
// MN-major operand straight from the cache layout), so the SIMT work per key is one row of
// the online softmax per thread.  P^T and the TMEM S^T are double-buffered, so the softmax
// of tile t overlaps the products of tile t-1.  Each item leaves (m, l, O) for its split;
// each segment leaves (m, l, O) in its own slot and the combine kernel merges the segments
// of each (b, g).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int HD = 128;
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
constexpr int POS_CACHE = 1024;             // sequences per launch (positions and tile prefix sums in smem)
constexpr int kDecMaxCtas = 256;            // upper bound of the grid (one CTA per SM)
constexpr float kDecRescaleLog2 = 8.0f;

struct DecParams {
  const int32_t* positions;
  float* o_part;   // [slot][REP][HD]
  float* m_part;   // [slot][REP]
  float* l_part;   // [slot][REP]
  int* prefix;     // [B + 1] tile prefix sums over the sequences, for the combine
  int B, H;
  int G;           // kernel groups per sequence: KV heads x chunks
  int chunks;      // groups of REP query heads per KV head (H / G_kv / REP)
  int T_max, max_pos;
  float scale_log2;
  int* status;
};

// One segment: tiles [k_begin / KT, k_begin / KT + ntile) of (b, g), keys [k_begin, k_end).
// Its partials go to slot b * G + g + blockIdx.x: along the axis both b * G + g and the CTA
// index never decrease and one of them grows from one segment to the next, so slots are
// unique and fewer than B * G + gridDim.x.
struct DecItem {
  int b, g, k_begin, k_end, ntile, slot;
};

// Segment starting at axis position `pos` of a CTA whose range ends at `end`.  pre_s[b] is
// the number of tiles of sequences before b (one KV head), so (b, g, tile) sits at
// G * pre_s[b] + g * n_b + tile with n_b = pre_s[b + 1] - pre_s[b].
__device__ __forceinline__ DecItem dec_seg(const DecParams& p, const int* pre_s, const int* pos_s, long long pos,
                                           long long end) {
  int lo = 0, hi = p.B - 1;   // the last sequence whose first tile is at or before pos
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(p.G) * pre_s[mid] <= pos) lo = mid;
    else hi = mid - 1;
  }
  DecItem d;
  d.b = lo;
  const int n_b = pre_s[lo + 1] - pre_s[lo];   // >= 1: pos lies inside this sequence's tiles
  const long long local = pos - static_cast<long long>(p.G) * pre_s[lo];
  d.g = static_cast<int>(local / n_b);
  const int t = static_cast<int>(local - static_cast<long long>(d.g) * n_b);
  d.ntile = static_cast<int>(min(static_cast<long long>(n_b - t), end - pos));
  d.k_begin = t * KT;
  d.k_end = min((t + d.ntile) * KT, pos_s[lo] + 1);
  d.slot = lo * p.G + d.g + static_cast<int>(blockIdx.x);
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
  int* pre_s = pos_s + POS_CACHE;                           // [POS_CACHE + 1], padded to + 2
  uint64_t* bars = reinterpret_cast<uint64_t*>(pre_s + POS_CACHE + 2);
  uint64_t* kv_full = bars;                  // [STAGES]
  uint64_t* kv_empty = bars + STAGES;        // [STAGES]
  uint64_t* q_full = bars + 2 * STAGES;      // [2]
  uint64_t* q_empty = q_full + 2;            // [2]
  uint64_t* s_full = q_empty + 2;            // [2]
  uint64_t* o_done = s_full + 2;             // [2] by the parity of the tile
  // [2] by the parity of the tile: the MMA issuer issues S of tile t before it waits for P of
  // tile t - 1, so the softmax may finish both before that wait looks; with one barrier the
  // phase of t - 1 could then be overtaken and never seen
  uint64_t* p_full = o_done + 2;
  uint64_t* o_free = p_full + 2;             // [2] by the parity of the item
  uint64_t* drain = o_free + 2;
  // the softmax warps' own barrier (4 arrivals), waited on with the bounded wait: after a wait
  // that gave up, no warp is left in a hardware barrier that the others never reach
  uint64_t* grp = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
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
    mbar_init(smem_u32(p_full + 1), 4);
    mbar_init(smem_u32(o_free), 4);
    mbar_init(smem_u32(o_free + 1), 4);
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(grp), 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
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
  pdl_wait();   // inputs written by the previous kernel (positions, q, the cache) are read from here on
  for (int i = threadIdx.x; i < p.B; i += DEC_THREADS) pos_s[i] = p.positions[i];
  __syncthreads();
  if (warp == 0) {   // tiles per sequence (0 for a position outside the cache), prefix-summed
    int run = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      int n = 0;
      if (b < p.B) {
        const int pos = pos_s[b];
        const bool ok = pos >= 0 && pos < p.T_max && pos < p.max_pos;
        if (!ok && blockIdx.x == 0) report(p.status, LLAMA_ERR_DEVICE_BOUNDS);
        n = ok ? pos / KT + 1 : 0;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < p.B) pre_s[b + 1] = run + incl;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pre_s[0] = 0;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i <= p.B; i += DEC_THREADS) p.prefix[i] = pre_s[i];
  // this CTA's range of the (b, g, tile) axis
  const long long axis = static_cast<long long>(p.G) * pre_s[p.B];
  const long long r0 = axis * blockIdx.x / gridDim.x, r1 = axis * (blockIdx.x + 1) / gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      // the cache is read once per step: evict-first keeps the segment partials and the step's
      // activations in L2 while it streams through
      const uint64_t kv_policy = l2_evict_first_policy();
      uint32_t tcount = 0, icount = 0;
      bool ok = true;
      for (long long pos = r0; pos < r1 && ok;) {
        const DecItem d = dec_seg(p, pre_s, pos_s, pos, r1);
        pos += d.ntile;
        const uint32_t qs = icount & 1;
        if (!mbar_wait(smem_u32(q_empty + qs), ((icount >> 1) & 1) ^ 1u, p.status, abort_flag)) { ok = false; break; }
        mbar_expect_tx(smem_u32(q_full + qs), Q_TILE);
        const int qrow = d.b * p.H + d.g * REP;
        tma_load_2d(smem_u32(sQ + qs * Q_TILE), &tmQ, smem_u32(q_full + qs), 0, qrow);
        tma_load_2d(smem_u32(sQ + qs * Q_TILE + Q_CHUNK), &tmQ, smem_u32(q_full + qs), 64, qrow);
        const int plane = (d.b * p.G + d.g) / p.chunks;   // the cache plane of KV head g / chunks
        for (int t = 0; t < d.ntile; ++t, ++tcount) {
          const uint32_t st = tcount % STAGES;
          if (!mbar_wait(smem_u32(kv_empty + st), ((tcount / STAGES) & 1) ^ 1u, p.status, abort_flag)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(kv_full + st);
          mbar_expect_tx(fb, 2 * KV_TILE);
          const int row = d.k_begin + t * KT;
          tma_load_3d_hint(smem_u32(sK + st * KV_TILE), &tmK, fb, 0, row, plane, kv_policy);
          tma_load_3d_hint(smem_u32(sK + st * KV_TILE + KV_CHUNK), &tmK, fb, 64, row, plane, kv_policy);
          tma_load_3d_hint(smem_u32(sV + st * KV_TILE), &tmV, fb, 0, row, plane, kv_policy);
          tma_load_3d_hint(smem_u32(sV + st * KV_TILE + KV_CHUNK), &tmV, fb, 64, row, plane, kv_policy);
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
        if (!mbar_wait(smem_u32(p_full + (tc & 1)), (tc >> 1) & 1, p.status, abort_flag)) return false;
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
      for (long long pos = r0; pos < r1 && ok;) {
        const DecItem d = dec_seg(p, pre_s, pos_s, pos, r1);
        pos += d.ntile;
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
    uint32_t gph = 0;   // phases of grp passed
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(grp));
      const bool r = mbar_wait(smem_u32(grp), gph & 1u, p.status, abort_flag);
      ++gph;
      return r;
    };
    for (long long pos = r0; pos < r1 && ok;) {
      const DecItem d = dec_seg(p, pre_s, pos_s, pos, r1);
      pos += d.ntile;
      const long long part = static_cast<long long>(d.slot) * REP;
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
        // red is double-buffered by tile parity: one barrier per tile
        if (!group_sync()) { ok = false; break; }
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
        if (lane == 0) mbar_arrive(smem_u32(p_full + pb));
      }
      if (!ok) break;
      // segment epilogue: wait for the last product, write this segment's (m, l, O)
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
      if (!group_sync()) { ok = false; break; }
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        float v = lsum[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) rb[sw * 8 + h] = v;
      }
      if (!group_sync()) { ok = false; break; }
#pragma unroll
      for (int h = 0; h < REP; ++h) {
        const float o = h < 4 ? __uint_as_float(oa[h]) : __uint_as_float(ob[h - 4]);
        p.o_part[(part + h) * HD + row] = o;
        if (row == 0) {
          p.m_part[part + h] = m_run[h];
          p.l_part[part + h] = rb[h] + rb[8 + h] + rb[16 + h] + rb[24 + h];
        }
      }
      if (!group_sync()) { ok = false; break; }   // rb is reused by the next segment's first tiles
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

constexpr size_t kDecSmemBytes = 1024 + 2 * STAGES * KV_TILE + 2 * Q_TILE + 2 * P_TILE + 64 * 4 +
                                 (2 * POS_CACHE + 2) * 4 + (2 * STAGES + 15) * 8 + 16;
static_assert(kDecSmemBytes <= 232448, "decode attention exceeds the shared memory of one CTA");
static_assert(kDecSmemBytes >= kTmemKernelMinSmem, "a TMEM-holding kernel must not share an SM with another");

// out[b, h*D + d] = sum_s e^(m_s - M) O_s[d] / sum_s e^(m_s - M) l_s over the segments s of
// (b, g = h / rep): the CTAs whose ranges meet the tiles [G pre[b] + g n_b, ... + n_b) of the
// axis.  CTA c's range starts at floor(c T / n_ctas), so the CTA holding tile t is
// floor(((t + 1) n_ctas - 1) / T).  A sequence with no tiles (position outside the cache)
// gets zeros.
__global__ void __launch_bounds__(HD) attn_decode_combine_kernel(const float* __restrict__ o_part,
                                                                 const float* __restrict__ m_part,
                                                                 const float* __restrict__ l_part,
                                                                 const int* __restrict__ prefix,
                                                                 __nv_bfloat16* __restrict__ out, int B, int H, int G,
                                                                 int n_ctas) {
  pdl_trigger();
  pdl_wait();
  const int bh = blockIdx.x, b = bh / H, h = bh - b * H, rep = H / G, g = h / rep, hr = h - g * rep;
  const int d = threadIdx.x;
  const int n_b = prefix[b + 1] - prefix[b];
  float res = 0.f;
  if (n_b > 0) {
    const long long T = static_cast<long long>(G) * prefix[B];
    const long long first = static_cast<long long>(G) * prefix[b] + static_cast<long long>(g) * n_b;
    const long long last = first + n_b - 1;
    const int c0 = static_cast<int>(((first + 1) * n_ctas - 1) / T);
    const int c1 = static_cast<int>(((last + 1) * n_ctas - 1) / T);
    const long long slot0 = static_cast<long long>(b) * G + g;
    // a CTA with an empty range (fewer tiles than CTAs) wrote no slot
    auto empty = [&](int c) { return T * c / n_ctas == T * (c + 1) / n_ctas; };
    float mm = -INFINITY;
    for (int c = c0; c <= c1; ++c)
      if (!empty(c)) mm = fmaxf(mm, m_part[(slot0 + c) * rep + hr]);
    float l = 0.f, o = 0.f;
    for (int c = c0; c <= c1; ++c) {
      if (empty(c)) continue;
      const long long i = (slot0 + c) * rep + hr;
      const float a = exp2f(m_part[i] - mm);
      l += l_part[i] * a;
      o += o_part[i * HD + d] * a;
    }
    res = l > 0.f ? o / l : 0.f;
  }
  out[static_cast<long long>(bh) * HD + d] = __float2bfloat16_rn(res);
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
  return launch_pdl(c, attn_decode_tc_kernel<REP>, dim3(std::min(c.num_sms, kDecMaxCtas)), dim3(DEC_THREADS),
                    kDecSmemBytes, tq, tk, tv, p);
}

}  // namespace

// Query heads per kernel group (at most 8) and kernel groups per KV head.
void dec_groups(int H, int G, int* rep_k, int* chunks) {
  const int rep = (G > 0 && H >= G) ? H / G : 1;
  *chunks = rep > 8 ? rep / 8 : 1;
  *rep_k = rep / *chunks;
}

size_t attn_decode_ws_bytes(int B, int H, int G, int D) {
  // one launch per POS_CACHE sequences, all reusing the same workspace
  int rep_k, chunks;
  dec_groups(H, G, &rep_k, &chunks);
  const size_t bc = static_cast<size_t>(std::max(0, std::min(B, POS_CACHE)));
  const size_t slots = bc * static_cast<size_t>(std::max(G, 1)) * chunks + kDecMaxCtas;
  return slots * rep_k * (D + 2) * sizeof(float) + (bc + 1) * sizeof(int) + 256;
}

int attn_decode(const Ctx& c, int dtype, const void* q, const void* k_cache, const void* v_cache,
                const int32_t* positions, void* out, int B, int H, int G, int D, int T_max, int max_pos, void* ws) {
  if (dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (D != HD) return LLAMA_ERR_UNSUPPORTED;
  const int rep_full = H / G;
  if (rep_full != 1 && rep_full != 2 && rep_full != 4 && rep_full % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  // more than 8 query heads per KV head: the kernel takes them 8 at a time, as `chunks`
  // groups that read the same cache plane
  int rep, chunks;
  dec_groups(H, G, &rep, &chunks);
  const int Gk = G * chunks;
  const int n_ctas = std::min(c.num_sms, kDecMaxCtas);
  const size_t bmax = static_cast<size_t>(std::min(B, POS_CACHE));
  const size_t slots = bmax * Gk + kDecMaxCtas;
  DecParams p;
  p.o_part = static_cast<float*>(ws);
  p.m_part = p.o_part + slots * rep * D;
  p.l_part = p.m_part + slots * rep;
  p.prefix = reinterpret_cast<int*>(p.l_part + slots * rep);
  p.H = H;
  p.G = Gk;
  p.chunks = chunks;
  p.T_max = T_max;
  p.max_pos = max_pos;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  p.status = c.status;
  for (int b0 = 0; b0 < B; b0 += POS_CACHE) {
    const int bc = std::min(POS_CACHE, B - b0);
    const size_t q_off = static_cast<size_t>(b0) * H * D * 2, kv_off = static_cast<size_t>(b0) * G * T_max * D * 2;
    const uint8_t* qc = static_cast<const uint8_t*>(q) + q_off;
    const uint8_t* kc = static_cast<const uint8_t*>(k_cache) + kv_off;
    const uint8_t* vc = static_cast<const uint8_t*>(v_cache) + kv_off;
    p.positions = positions + b0;
    p.B = bc;
    CUtensorMap tq, tk, tv;
    // Q [B*H][D] in 16-row boxes (the group's H/G heads, then padding rows that are ignored);
    // K, V [B*G][T_max][D] in 128-key boxes (keys past T_max read as 0)
    if (!make_tmap_2d(&tq, qc, HD, static_cast<uint64_t>(bc) * H, HD, NQ) ||
        !make_tmap_3d(&tk, kc, HD, T_max, static_cast<uint64_t>(bc) * G, HD, static_cast<uint64_t>(T_max) * HD, KT) ||
        !make_tmap_3d(&tv, vc, HD, T_max, static_cast<uint64_t>(bc) * G, HD, static_cast<uint64_t>(T_max) * HD, KT))
      return LLAMA_ERR_INVALID_ARG;
    cudaError_t err;
    switch (rep) {
      case 1: err = launch_decode<1>(c, tq, tk, tv, p); break;
      case 2: err = launch_decode<2>(c, tq, tk, tv, p); break;
      case 4: err = launch_decode<4>(c, tq, tk, tv, p); break;
      default: err = launch_decode<8>(c, tq, tk, tv, p); break;
    }
    if (err != cudaSuccess) return LLAMA_ERR_CUDA;
    int rc = after_launch(c);
    if (rc != LLAMA_OK) return rc;
    launch_pdl(c, attn_decode_combine_kernel, dim3(bc * H), dim3(HD), 0, p.o_part, p.m_part, p.l_part, p.prefix,
               reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(out) + q_off), bc, H, Gk, n_ctas);
    if ((rc = after_launch(c)) != LLAMA_OK) return rc;
  }
  return LLAMA_OK;
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

// Largest scratch the fixed-array entry point serves: the segment partials of
// min(B, 1024) * H + 256 * min(H / G, 8) (query head, segment) pairs, (D + 2) floats each,
// and min(B, 1024) + 1 ints.  At B = 64, H = 32, G = 8, D = 128 that is 2.1 MB.
constexpr size_t kDecodeScratchBytes = 16u << 20;

// File-scope device array: every device that loads the library holds its own copy until the
// process exits, and all calls on a device share it.  Each call writes every slot it later
// reads (the combine reads only the segments that the same call's CTAs wrote), so nothing
// needs clearing, but two calls that overlap on the GPU (different streams, no ordering)
// race on it.
static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

// Device address of g_decode_scratch, looked up once per device (host code must not use
// the symbol itself: on the host it only names a stand-in).
std::atomic<void*> g_decode_scratch_addr[kMaxDevices];

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
  if (attn_decode_ws_bytes(B, dims->n_heads, dims->n_kv_heads, dims->head_dim) > kDecodeScratchBytes)
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
