// Causal grouped-query flash attention for prefill on the 5th-generation tensor cores.
//
// O_h = softmax(Q_h K_g^T / sqrt(D), key j visible to query i iff j <= i) V_g, g = h / (H/G)
// ("12 · 从 Transformer 到 LLaMA 系列" §八 Attention with is_causal=True and the KV heads
// repeated along dim 1; "深度学习进阶（三十）…" §1.1; "第 10 章：现代 LLaMA 架构" §6: K/V stay
// G heads in the cache and are shared logically, never copied H/G times).
//
// Persistent: one CTA per SM walks a list of work items, each a pair of 128-query blocks 2i
// and 2i+1 of one head of one sequence.  The items are ordered longest first (the last query
// pairs read the most keys) and dealt out in a snake over rounds of one item per CTA, so each
// CTA's total is close to the mean; the next item's Q and K/V loads overlap the current item's
// last products.  Both query tiles read every K/V tile once from shared memory.
//   warp 0      TMA: an item's two Q tiles (once the previous item's last S product has read
//               its own), then K_j, V_j (128 keys each) into 2-stage rings straight from the
//               [B, G, max_T, D] cache: K and V into 2-stage rings of their own, each stage
//               released as soon as its last reader is done (K_j after the S products of key
//               tile j, V_j after its P V products), so each K tile goes out well ahead of its
//               S products (the wait for the next S was half of a softmax warp's time with one
//               2-stage ring for both)
//   warp 1      TMEM allocator and MMA issuer, ping-pong between the two tiles:
//               S_t = Q_t K_j^T into TMEM; once the softmax of tile t has written P_t,
//               O_t += P_t V_j with P_t read from TMEM and V as an MN-major smem operand,
//               then at once S_t for the next K tile, so one tile's softmax overlaps the
//               other tile's MMAs
//   warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: one query row per thread,
//               read from TMEM in one 128-column load per key tile; the row max, exp2 with
//               the scale folded in, P as bf16 written over S in TMEM (one 64-column
//               store); O is rescaled only when the running max grows by more than 2^8
//               (the final O / l uses the same reference max, so the result is exact)
// fp32 statistics and accumulators; D = 128.
//
// A chunk on top of a cache ("第 10 章：现代 LLaMA 架构" §7, past_kv with position_ids =
// past_len + arange(T)): query s of sequence b sits at position start[b] + s and sees cache
// slots 0 .. start[b] + s, so a query tile reads the key tiles up to its last query's
// position and masks the ones its first query does not fully see.  Queries s >= lens[b]
// pad the chunk: they are computed but not stored, and the V rows of keys at or past
// start[b] + lens[b] are zeroed in shared memory before P V (stale cache slots may hold
// anything; 0 * NaN would leak into valid rows).
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
constexpr int NUM_THREADS = 384;
constexpr int K_STAGES = 2;           // K ring (3 stages measured no faster); V ring: 2 stages
constexpr uint32_t TMEM_COLS = 512;   // S/P of tile t at [128t, 128t+128), O of tile t at 256 + 128t
constexpr float kRescaleLog2 = 8.0f;  // rescale O when the max grows by more than 2^8

struct AttnParams {
  int B, S, H, G, n_qt, n_pairs;
  int n_items;                        // n_pairs * H * B work items (one query pair of one head)
  const int32_t* start;               // [B] or null (0)
  const int32_t* lens;                // [B] or null (S)
  int T_max, max_pos;
  float scale_log2;                   // log2(e) / sqrt(D)
  __nv_bfloat16* out;                 // [B, S, H*D]
  int* status;
};

// Work item i: the (z+1)-th longest query pair (z = i / (H B)) of head h, sequence b (h varies
// fastest, so the heads that share a KV head sit next to each other).  CTA c takes items
// c, 2G-1-c, 2G+c, 4G-1-c, ... (G CTAs): a snake over rounds of G items, so a CTA that drew
// one of the longest pairs in a round draws one of the shortest in the next.
struct AttnItem {
  int b, h, g, pair, pos0, len;
  bool hasA, hasB;
  int nkt[2], nt, n_valid;
};

__device__ __forceinline__ int item_of(int c, int r) {
  const int G = static_cast<int>(gridDim.x);
  return r * G + ((r & 1) ? G - 1 - c : c);
}

__device__ __forceinline__ AttnItem make_item(const AttnParams& p, int i, bool report_bounds) {
  AttnItem it;
  const int hb = p.H * p.B;
  const int z = i / hb, rem = i - z * hb;
  it.b = rem / p.H;
  it.h = rem - it.b * p.H;
  it.g = it.h / (p.H / p.G);
  it.pair = p.n_pairs - 1 - z;
  // this sequence's chunk: queries [0, len) at positions pos0 + s; keys [0, pos0 + len)
  it.pos0 = 0;
  it.len = p.S;
  if (p.start != nullptr) {
    it.pos0 = p.start[it.b];
    it.len = p.lens != nullptr ? p.lens[it.b] : p.S;
    if (it.pos0 < 0 || it.len < 0 || it.len > p.S || it.pos0 + it.len > p.T_max || it.pos0 + it.len > p.max_pos) {
      if (report_bounds && z == 0 && it.h == 0) report(p.status, LLAMA_ERR_DEVICE_BOUNDS);
      it.len = 0;
    }
  }
  const int qa = 2 * it.pair, qb = 2 * it.pair + 1;
  it.hasA = qa * BQ < it.len;
  it.hasB = qb * BQ < it.len;
  // key tiles that tile t reads: up to the position of its last query
  it.nkt[0] = it.hasA ? (it.pos0 + min(qa * BQ + BQ, it.len) - 1) / BKV + 1 : 0;
  it.nkt[1] = it.hasB ? (it.pos0 + min(qb * BQ + BQ, it.len) - 1) / BKV + 1 : 0;
  it.nt = it.hasB ? it.nkt[1] : it.nkt[0];
  it.n_valid = it.pos0 + it.len;
  return it;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                               // 2 tiles
  uint8_t* sK = smem + 2 * TILE;                    // K_STAGES stages
  uint8_t* sV = smem + (2 + K_STAGES) * TILE;       // 2 stages
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (4 + K_STAGES) * TILE);
  uint64_t* q_full = bars;
  uint64_t* s_full = bars + 1;          // [2] per tile
  uint64_t* p_full = bars + 3;          // [2] per tile
  uint64_t* o_done = bars + 5;          // [2] per tile
  uint64_t* drain = bars + 7;
  uint64_t* q_empty = bars + 8;         // the Q tiles of an item may be overwritten
  uint64_t* v_full = bars + 9;          // [2] per V stage
  uint64_t* v_empty = bars + 11;        // [2] per V stage
  uint64_t* k_full = bars + 13;         // [K_STAGES] per K stage
  uint64_t* k_empty = bars + 13 + K_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 13 + 2 * K_STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(q_full), 1);
    mbar_init(smem_u32(q_empty), 1);
    for (int i = 0; i < K_STAGES; ++i) {
      mbar_init(smem_u32(k_full + i), 1);
      mbar_init(smem_u32(k_empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(v_full + i), 1);
      mbar_init(smem_u32(v_empty + i), 1);
      mbar_init(smem_u32(s_full + i), 1);
      mbar_init(smem_u32(p_full + i), 4);
      mbar_init(smem_u32(o_done + i), 1);
    }
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
  pdl_wait();   // inputs written by the previous kernel are read from here on

  // Every role walks the same items in the same order; the barrier phases run on across items:
  // K/V tile g of the CTA (counted over its items) sits in stage g & 1, and S/P of tile t and
  // the O products of tile t are counted per tile.
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      bool ok = true;
      uint32_t kvc = 0, qc = 0, kc_issued = 0, vc_issued = 0;
      for (int r = 0; ok; ++r) {
        const int i = item_of(c, r);
        if (i >= p.n_items) break;
        const AttnItem it = make_item(p, i, true);
        if (!it.hasA) continue;
        // the previous item's S products have read its Q tiles
        if (qc > 0 && !mbar_wait(smem_u32(q_empty), (qc - 1) & 1, p.status, abort_flag)) { ok = false; break; }
        const uint32_t qbar = smem_u32(q_full);
        const int qplane = it.b * p.H + it.h;
        mbar_expect_tx(qbar, it.hasB ? 2 * TILE : TILE);
        for (int t = 0; t < (it.hasB ? 2 : 1); ++t) {
          const int qrow = (2 * it.pair + t) * BQ;
          tma_load_3d(smem_u32(sQ + t * TILE), &tmQ, qbar, 0, qrow, qplane);
          tma_load_3d(smem_u32(sQ + t * TILE + CHUNK), &tmQ, qbar, 64, qrow, qplane);
        }
        ++qc;
        const int plane = it.b * p.G + it.g;
        for (int j = 0; j < it.nt; ++j, ++kvc) {
          const uint32_t st = kvc & 1, ph = ((kvc >> 1) & 1) ^ 1u;
          const uint32_t kst = kvc % K_STAGES, kph = ((kvc / K_STAGES) & 1) ^ 1u;
          const int row = j * BKV;
          if (!mbar_wait(smem_u32(k_empty + kst), kph, p.status, abort_flag)) { ok = false; break; }
          const uint32_t kb = smem_u32(k_full + kst);
          mbar_expect_tx(kb, TILE);
          tma_load_3d(smem_u32(sK + kst * TILE), &tmK, kb, 0, row, plane);
          tma_load_3d(smem_u32(sK + kst * TILE + CHUNK), &tmK, kb, 64, row, plane);
          ++kc_issued;
          if (!mbar_wait(smem_u32(v_empty + st), ph, p.status, abort_flag)) { ok = false; break; }
          const uint32_t vb = smem_u32(v_full + st);
          mbar_expect_tx(vb, TILE);
          tma_load_3d(smem_u32(sV + st * TILE), &tmV, vb, 0, row, plane);
          tma_load_3d(smem_u32(sV + st * TILE + CHUNK), &tmV, vb, 64, row, plane);
          ++vc_issued;
        }
      }
      if (!ok) {
        // leave no copy in flight: the last Q load and the last two K and V loads
        if (qc > 0) mbar_wait_slow(smem_u32(q_full), (qc - 1) & 1, nullptr, nullptr, kWaitBudgetNs);
        for (uint32_t g = (kc_issued > K_STAGES ? kc_issued - K_STAGES : 0); g < kc_issued; ++g)
          mbar_wait_slow(smem_u32(k_full + g % K_STAGES), (g / K_STAGES) & 1, nullptr, nullptr, kWaitBudgetNs);
        for (uint32_t g = (vc_issued > 2 ? vc_issued - 2 : 0); g < vc_issued; ++g)
          mbar_wait_slow(smem_u32(v_full + (g & 1)), (g >> 1) & 1, nullptr, nullptr, kWaitBudgetNs);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // The whole warp walks the loop (its operands stay warp-uniform) and one elected lane
    // issues each product and commit: from a single diverged lane an issue costs about as
    // long as a 128 x 128 x 16 product runs, and the bookkeeping between products would
    // leave the tensor core idle.
    constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false);
    constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, true);
    const uint64_t dQ = sdesc_sw128(smem_u32(sQ), 16, 1024);
    const uint64_t dK = sdesc_sw128(smem_u32(sK), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(sV), CHUNK, 1024);
    // every lane waits (they stay in step); a timeout or abort seen by any lane ends the loop
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      const bool r = mbar_wait(smem_u32(bar), parity, p.status, abort_flag);
      return __all_sync(0xffffffffu, r) != 0;
    };
    auto issue_s = [&](int t, uint32_t kst) {
      const uint64_t aq = dQ + static_cast<uint64_t>((t * TILE) >> 4);
      const uint64_t bk = dK + static_cast<uint64_t>((kst * TILE) >> 4);
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * CHUNK + (kk & 3) * 32) >> 4;
        tc_mma_bf16_warp(tmem_base + t * 128, aq + off, bk + off, IDESC_QK, kk > 0 ? 1u : 0u);
      }
      tc_commit_warp(smem_u32(s_full + t));
    };
    // O_t += P_t V_j; o_done[t] only after the item's last one (the softmax's rescale of O
    // before P_t V_j needs P_t V_{j-1} complete, which s_full[t] for S_t(j) already implies:
    // S_t(j) is issued after it, and a commit tracks all earlier products of its thread)
    auto issue_pv = [&](int t, uint32_t st, bool first, bool last) {
      const uint64_t bv = dV + static_cast<uint64_t>((st * TILE) >> 4);
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk) {
        // V: 128 key rows of 128 bytes per 64-wide d half; K step = 16 rows = 2048 bytes,
        // the second d half is CHUNK bytes further (leading byte offset), 8-row groups 1024 apart
        tc_mma_bf16_ts_warp(tmem_base + 256 + t * 128, tmem_base + t * 128 + kk * 8,
                            bv + static_cast<uint64_t>((kk * 2048) >> 4), IDESC_PV, (!first || kk > 0) ? 1u : 0u);
      }
      if (last) tc_commit_warp(smem_u32(o_done + t));
    };
    bool ok = true, issued = false;
    uint32_t kvc = 0, qc = 0, k_seen = ~0u;
    uint32_t pc[2] = {0u, 0u};   // P arrivals consumed, per tile
    for (int r = 0; ok; ++r) {
      const int i = item_of(c, r);
      if (i >= p.n_items) break;
      const AttnItem it = make_item(p, i, false);
      if (!it.hasA) continue;
      auto active = [&](int t, int j) { return j < it.nkt[t]; };
      if (!wait_all(q_full, qc & 1) || !wait_all(k_full + kvc % K_STAGES, (kvc / K_STAGES) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the Q tiles are free for the next item once this item's last S product is done:
      // commit q_empty right after issuing it; K_j is free once the S products of key tile j
      // are (the last one is tile B's when B reads key tile j, else tile A's)
      int s_left = it.nkt[0] + it.nkt[1];
      auto issue_s_counted = [&](int t, int j, uint32_t kst) {
        issue_s(t, kst);
        if (--s_left == 0) tc_commit_warp(smem_u32(q_empty));
        if (t == 1 || !active(1, j)) tc_commit_warp(smem_u32(k_empty + kst));
      };
      issue_s_counted(0, 0, kvc % K_STAGES);
      if (it.hasB) issue_s_counted(1, 0, kvc % K_STAGES);
      issued = true;
      for (int j = 0; j < it.nt && ok; ++j) {
        const uint32_t g = kvc + j;
        if (!wait_all(v_full + (g & 1), (g >> 1) & 1)) { ok = false; break; }
        for (int t = 0; t < 2 && ok; ++t) {
          if (!active(t, j)) continue;
          if (!wait_all(p_full + t, pc[t] & 1)) { ok = false; break; }
          ++pc[t];
          tc_fence_after();
          issue_pv(t, g & 1, j == 0, !active(t, j + 1));
          if (active(t, j + 1)) {
            const uint32_t gn = g + 1;
            // K_{j+1} once per key tile (tile B's S follows tile A's)
            if (gn != k_seen) {
              if (!wait_all(k_full + gn % K_STAGES, (gn / K_STAGES) & 1)) { ok = false; break; }
              k_seen = gn;
              tc_fence_after();
            }
            issue_s_counted(t, j + 1, gn % K_STAGES);
          }
        }
        if (ok) tc_commit_warp(smem_u32(v_empty + (g & 1)));
      }
      if (!ok) break;
      kvc += it.nt;
      ++qc;
    }
    if (!ok && issued) {
      // all products of the issuing lane must finish before the TMEM is released
      tc_commit_warp(smem_u32(drain));
      if (lane == 0) mbar_wait_slow(smem_u32(drain), 0, nullptr, nullptr, kWaitBudgetNs);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // -------------------------------------------------------------- softmax of tile t
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem_base + t_lane + t * 128;        // S, and P written over it
    const uint32_t tO = tmem_base + t_lane + 256 + t * 128;
    const float sl = p.scale_log2;
    uint32_t r[128];   // the row's 128 scores, then (first 64) its P as packed bf16 pairs
    bool ok = true;
    // K/V tiles of the CTA's items so far; S tiles of tile t so far; items of tile t so far
    uint32_t kvc = 0, tc_run = 0, oc = 0;
    for (int rr = 0; ok; ++rr) {
      const int i = item_of(c, rr);
      if (i >= p.n_items) break;
      const AttnItem it = make_item(p, i, false);
      if (!it.hasA) continue;
      const uint32_t kvbase = kvc;
      kvc += it.nt;
      if (t == 1 && !it.hasB) continue;   // this item has no second query tile
      const int qi = (2 * it.pair + t) * BQ + row;
      float m_run = -INFINITY, l_run = 0.f;
      const int n_t = it.nkt[t];
      const int qpos = it.pos0 + qi;                 // this row's position: keys 0 .. qpos
      for (int j = 0; j < n_t; ++j) {
        const uint32_t sj = tc_run + j;
        if (!mbar_wait(smem_u32(s_full + t), sj & 1, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const int kbase = j * BKV;
        // the whole row of S in one TMEM round trip
        tmem_ld128(tS, r);
        // the tile reaches past the first query's position: mask key > position
        const bool diag = kbase + BKV - 1 > it.pos0 + (2 * it.pair + t) * BQ;
        if (diag) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (kbase + k > qpos) r[k] = __float_as_uint(-INFINITY);
        }
        // two scores per max instruction, in four independent chains (only the two softmax
        // warps of a sub-partition share its issue slots: a single chain would wait on latency)
        float m4[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) m4[u] = fmaxf(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1]));
#pragma unroll
        for (int k = 8; k < 128; k += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u) m4[u] = fmax3(m4[u], __uint_as_float(r[k + 2 * u]), __uint_as_float(r[k + 2 * u + 1]));
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float mxs = mx * sl;
        const bool need = mxs > m_run + kRescaleLog2;    // also true on the first tile
        const bool any_need = __any_sync(0xffffffffu, need);
        const float m_new = need ? mxs : m_run;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
        m_run = m_new;
        // P = 2^(S * scale - m) (masked scores are -inf: P = 0), packed in place: pair k goes
        // to r[k] once r[2k], r[2k + 1] are read; keys 2c, 2c+1 land in S column c
        // S * scale - m two scores per instruction; the row sum in two packed accumulators
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          float x0, x1;
          fma2(x0, x1, __uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]), sl, sl, -m_run, -m_run);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const int a = 2 * (k & 1);
          add2(sum4[a], sum4[a + 1], sum4[a], sum4[a + 1], p0, p1);
          r[k] = pack_bf16(p0, p1);
        }
        add2(sum4[0], sum4[1], sum4[0], sum4[1], sum4[2], sum4[3]);
        const float rowsum = sum4[0] + sum4[1];
        tmem_st64(tS, r);
        if (any_need) {
          if (j > 0) {
            // O is rescaled before this tile's P V (which waits for p_full below); P_{j-1} V_{j-1}
            // has landed: it was issued before S_j, whose completion s_full signalled
            uint32_t o32[32];
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
              tmem_ld32(tO + cc * 32, o32);
#pragma unroll
              for (int k = 0; k < 32; ++k) o32[k] = __float_as_uint(__uint_as_float(o32[k]) * alpha);
              tmem_st32(tO + cc * 32, o32);
            }
          }
          l_run *= alpha;
        }
        l_run += rowsum;
        // keys at or past the last valid one: zero their V rows before any P V of this tile
        // (done by tile 0 if it reads this tile, else by tile 1; the MMA issuer orders tile
        // 1's product after tile 0's P), once the tile's V has landed
        const bool zero_v = kbase + BKV > it.n_valid && (t == 0 || j >= it.nkt[0]);
        if (zero_v) {
          const uint32_t g = kvbase + j;
          if (!mbar_wait(smem_u32(v_full + (g & 1)), (g >> 1) & 1, p.status, abort_flag)) { ok = false; break; }
        }
        if (zero_v && kbase + row >= it.n_valid) {
          uint8_t* vrow = sV + ((kvbase + j) & 1) * TILE + row * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            reinterpret_cast<uint4*>(vrow)[u] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(vrow + CHUNK)[u] = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(p_full + t));
      }
      if (!ok) break;
      tc_run += n_t;
      // the item's last product (this thread's reads of O come before the next item's first
      // P V, which waits for this warp's next arrival on p_full)
      if (!mbar_wait(smem_u32(o_done + t), oc & 1, p.status, abort_flag)) { ok = false; break; }
      ++oc;
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      __nv_bfloat16* dst =
          p.out + (static_cast<long long>(it.b) * p.S + qi) * (static_cast<long long>(p.H) * HD) + it.h * HD;
      uint32_t o32[32];
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tO + cc * 32, o32);
        if (qi < it.len) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + cc * 32);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(o32[8 * u + 0]) * inv_l, __uint_as_float(o32[8 * u + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(o32[8 * u + 2]) * inv_l, __uint_as_float(o32[8 * u + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(o32[8 * u + 4]) * inv_l, __uint_as_float(o32[8 * u + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(o32[8 * u + 6]) * inv_l, __uint_as_float(o32[8 * u + 7]) * inv_l);
            d4[u] = w;
          }
        }
      }
      tc_fence_before();
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

constexpr size_t kSmemBytes = 1024 + (4 + K_STAGES) * TILE + (13 + 2 * K_STAGES) * 8 + 16;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kSmemBytes >= kTmemKernelMinSmem, "a TMEM-holding kernel must not share an SM with another");

}  // namespace

int attn_prefill_tc(const Ctx& c, const void* q, const void* k_cache, const void* v_cache, void* out, int B, int S,
                    int H, int G, int D, int T_max, const int32_t* start, const int32_t* lens, int max_pos) {
  if (D != HD) return LLAMA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv;
  // Q [B*H][S][D]; K, V: [B*G][T_max][D] with the slots a chunk can reach as the extent:
  // [0, S) from position 0 (rows >= S read as 0), the whole cache on top of one
  const uint64_t kv_rows = start != nullptr ? static_cast<uint64_t>(T_max) : static_cast<uint64_t>(S);
  if (!make_tmap_3d(&tq, q, HD, S, static_cast<uint64_t>(B) * H, HD, static_cast<uint64_t>(S) * HD, BQ) ||
      !make_tmap_3d(&tk, k_cache, HD, kv_rows, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD,
                    BKV) ||
      !make_tmap_3d(&tv, v_cache, HD, kv_rows, static_cast<uint64_t>(B) * G, HD, static_cast<uint64_t>(T_max) * HD,
                    BKV))
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
  p.n_pairs = (p.n_qt + 1) / 2;
  const long long items = static_cast<long long>(p.n_pairs) * H * B;
  if (items > (1ll << 30)) return LLAMA_ERR_UNSUPPORTED;
  p.n_items = static_cast<int>(items);
  p.start = start;
  p.lens = lens;
  p.T_max = T_max;
  p.max_pos = max_pos;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = c.status;
  if (p.n_items == 0) return LLAMA_OK;
  // persistent: one CTA per SM walks its share of the items
  launch_pdl(c, attn_prefill_kernel, dim3(std::min(p.n_items, c.num_sms)), dim3(NUM_THREADS), kSmemBytes, tq, tk,
             tv, p);
  return after_launch(c);
}

}  // namespace llama
