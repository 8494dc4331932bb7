// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
// C = X W^T ("12 · 从 Transformer 到 LLaMA 系列" §八: every projection of the layer is an
// nn.Linear without bias).  One CTA per SM walks a list of output tiles:
//   warp 0     TMA producer: 128x64 A tile + BNx64 B tile per stage (128-byte swizzle)
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma 128xBNx16 into a TMEM accumulator
//   warps 2-5  epilogue: tcgen05.ld of the accumulator rows, fused op, stores to HBM
//   warps 6-9  (RMSNorm-fused form only) operand A: see below
// Two TMEM accumulators let the epilogue of tile i overlap the main loop of tile i+1.
//
// RMSNorm fused into the A operand ("12 · 从 Transformer 到 LLaMA 系列" §八 RMSNorm: y = gamma *
// x * rsqrt(mean(x^2) + eps); "3.2 核心组件逐一拆解" §3.2.1: the statistics in fp32).  TMA brings
// the raw x tile of each k-block (and that k-block's 64 gammas) into a shared-memory ring of its
// own; four norm warps read it once, each thread one row, form bf16(gamma_k * (x_mk * r_m)) --
// the normalised row rounded where a standalone RMSNorm would store it -- and store it into one
// of two A slots in tensor memory, from which the MMAs read their A operand.  Shared memory
// carries the same bytes as in the plain form (the tensor cores' own A reads move to TMEM), which
// matters because these GEMMs are bound by shared-memory bandwidth: a transform written back to
// shared memory cost a third more time.  The row scales r_m = rsqrt(mean_k x_mk^2 + eps) come
// with the input: from a row-statistics pass over the layer input, or from the residual
// epilogue that produced x (below).  The normalised activation never goes through HBM.
// Tensor memory: the two accumulators (2 x 224 columns) and the two A slots (32 columns each).
//
// Row statistics in the residual epilogue: a tile adds the squares of its rounded outputs of
// row m into part[nb][m]; the last of the row's column tiles to finish (a per-row ticket)
// sums part[0..num_nb)[m] in column order and writes r_m, so the result does not depend on
// which tile finishes last.
// Epilogues: plain store (bf16 / fp32), residual add (o_proj, down_proj;
// "05 LLaMA3 Block — 从零件到发动机" §4.2 steps ④ ⑧), SiLU(gate) * up
// ("3.2 核心组件逐一拆解" §3.2.2; gate and up tiles share one accumulator), QKV with
// even/odd RoPE and the scatter of k, v into the cache layout ("第 10 章：现代 LLaMA 架构"
// §3, §6), and fp32 split-K partials for the weight-streaming (few-token) form.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace llama {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_TILE_BYTES = BM * BK * 2;
constexpr int NUM_THREADS = 192;
constexpr int NORM_THREADS = 128;   // the norm warps of the RMSNorm-fused form

template <bool NORM>
constexpr int threads_of() {
  return NORM ? NUM_THREADS + NORM_THREADS : NUM_THREADS;
}

enum Epi : int { EPI_BF16 = 0, EPI_F32 = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_QKV = 4, EPI_PARTIAL = 5 };

// How a 128-row block of an operand maps to one of the kernel's tensor maps.
struct RowMap {
  int nseg;          // 1..3 row-concatenated matrices
  int seg_end[3];    // cumulative row ends (multiples of 128)
};

struct TMaps {
  CUtensorMap m[7];
};

struct Params {
  int M, N, K;                  // kernel frame: C[M, N] = A[M, K] B[N, K]^T
  int num_mb, num_nb, num_splits, kb_per_split, num_kb;
  int group_m;
  int weight_first;             // 0, or 1 / 2: operand A / B is a weight that may be loaded before
                                // griddepcontrol.wait (the first STAGES k-blocks of it are)
  RowMap amap, bmap;
  int a_map0, b_map0;
  int b32_map0;                 // QKV on tiles that are not head-aligned: the weight maps again
                                // with 32-row boxes, for tiles that cross a q|k or k|v boundary
  int n_maps;                   // tensor maps in use
  void* out;
  long long ldo;
  const __nv_bfloat16* resid;
  long long ldr;
  // QKV + RoPE
  const float* cos;
  const float* sin;
  int S, H, G, D, T_max;
  int rope_half;                // pairs (i, i + D/2) instead of (2i, 2i+1)
  const int32_t* start;         // [B] cached length before this chunk (null: 0)
  const int32_t* lens;          // [B] valid tokens of the chunk (null: S)
  int max_pos;
  __nv_bfloat16* q_out;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  // RMSNorm-fused form: operand A = bf16(norm_gamma_k * (x_mk * norm_r_m)), x the A operand
  const __nv_bfloat16* norm_gamma;   // [K]
  const float* norm_r;               // [M] rsqrt(mean_k x_mk^2 + eps)
  // residual epilogue: the row statistics of the output for the next RMSNorm (null: none)
  float* stat_part;                  // [num_nb][M] sums of squares of each tile's outputs
  float* stat_r;                     // [M] rsqrt(sum / N + stat_eps), by the row's last tile
  int* stat_ticket;                  // [M] column tiles done; zero before, reset by the last
  float stat_inv_n, stat_eps;
  int* status;
};

__device__ __forceinline__ void resolve_rows(const RowMap& rm, int vrow, int& map, int& row) {
  map = 0;
  int start = 0;
  if (rm.nseg > 1 && vrow >= rm.seg_end[0]) { map = 1; start = rm.seg_end[0]; }
  if (rm.nseg > 2 && vrow >= rm.seg_end[1]) { map = 2; start = rm.seg_end[1]; }
  row = vrow - start;
}

__device__ __forceinline__ void tile_coords(const Params& p, int t, int& mb, int& nb, int& split) {
  split = t % p.num_splits;
  t /= p.num_splits;
  const int per_group = p.group_m * p.num_nb;
  const int g = t / per_group, r = t % per_group;
  const int first_m = g * p.group_m;
  const int gm = min(p.group_m, p.num_mb - first_m);
  mb = first_m + r % gm;
  nb = r / gm;
}

// ------------------------------------------------------------------ epilogue helpers

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v, int valid) {
  if (valid < 32 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
    // whole groups of 8 as 16-byte stores, the rest one by one (static register indices)
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (8 * g + 8 <= valid) {
        uint4 w;
        w.x = pack_bf16(v[8 * g + 0], v[8 * g + 1]);
        w.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
        w.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
        w.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
        reinterpret_cast<uint4*>(dst)[g] = w;
      }
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i >= (valid & ~7) && i < valid) dst[i] = __float2bfloat16_rn(v[i]);
    return;
  }
  if (valid >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint4 w;
      w.x = pack_bf16(v[8 * g + 0], v[8 * g + 1]);
      w.y = pack_bf16(v[8 * g + 2], v[8 * g + 3]);
      w.z = pack_bf16(v[8 * g + 4], v[8 * g + 5]);
      w.w = pack_bf16(v[8 * g + 6], v[8 * g + 7]);
      d4[g] = w;
    }
  } else {
    for (int i = 0; i < valid; ++i) dst[i] = __float2bfloat16_rn(v[i]);
  }
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v, int valid) {
  if (valid >= 32) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4 w = s4[g];
      v[8 * g + 0] = bf16_lo(w.x); v[8 * g + 1] = bf16_hi(w.x);
      v[8 * g + 2] = bf16_lo(w.y); v[8 * g + 3] = bf16_hi(w.y);
      v[8 * g + 4] = bf16_lo(w.z); v[8 * g + 5] = bf16_hi(w.z);
      v[8 * g + 6] = bf16_lo(w.w); v[8 * g + 7] = bf16_hi(w.w);
    }
  } else {
    for (int i = 0; i < 32; ++i) v[i] = i < valid ? __bfloat162float(src[i]) : 0.f;
  }
}

// Stages of the shared-memory A ring (the raw x tiles of the RMSNorm-fused form), and TMEM A slots.
template <bool NORM, int STAGES>
constexpr int a_stages_of() {
  return NORM ? 4 : STAGES;
}
constexpr int kNormASlots = 2;

template <int BN, int EPI, int STAGES, bool NORM>
__global__ void __launch_bounds__(threads_of<NORM>())
    gemm_tc_kernel(const __grid_constant__ TMaps tm, const Params p) {
  constexpr int B_TILE_BYTES = BN * BK * 2;
  constexpr int SA = a_stages_of<NORM, STAGES>();
  // B arrives in 128-row boxes, or as one box when BN is not a multiple of 128 (BN <= 256);
  // gate/up tiles as two boxes of BN/2 rows, one from each matrix
  constexpr int B_BOX_ROWS = EPI == EPI_SWIGLU ? BN / 2 : BN % 128 == 0 ? 128 : BN;
  constexpr int B_BOXES = BN / B_BOX_ROWS;
  // bytes that TMA brings per stage towards the MMA barrier (in the RMSNorm-fused form the raw A
  // tile and its gammas arrive on a barrier of their own, for the norm warps)
  constexpr uint32_t STAGE_TX = NORM ? B_TILE_BYTES : A_TILE_BYTES + B_TILE_BYTES;
  constexpr uint32_t A_TX = A_TILE_BYTES + BK * 2;
  constexpr uint32_t ACC_COLS = 2 * BN + (NORM ? kNormASlots * BK / 2 : 0);
  constexpr uint32_t TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN, false);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(ACC_COLS <= 512, "two accumulators (and the A slots) in tensor memory");

  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + SA * A_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_TILE_BYTES);
  uint64_t* full_bar = bars;                      // [STAGES] A and B landed (fused form: B)
  uint64_t* empty_bar = bars + STAGES;            // [STAGES] the stage's MMAs are done
  uint64_t* tfull_bar = bars + 2 * STAGES;
  uint64_t* tempty_bar = bars + 2 * STAGES + 2;
  uint64_t* drain_bar = bars + 2 * STAGES + 4;
  // fused form: per raw A stage, landed / read by the norm warps; per TMEM A slot, written by the
  // norm warps / read by the MMAs
  uint64_t* araw_bar = bars + 2 * STAGES + 5;
  uint64_t* afree_bar = araw_bar + SA;
  uint64_t* tready_bar = afree_bar + SA;
  uint64_t* tfree_bar = tready_bar + kNormASlots;
  constexpr int BAR_WORDS = 2 * STAGES + 5 + (NORM ? 2 * SA + 2 * kNormASlots : 0);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + BAR_WORDS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // [SA][BK] gammas of each A stage (fused form), 16-byte aligned for the bulk copy
  uint8_t* sG = reinterpret_cast<uint8_t*>(bars + ((BAR_WORDS + 2) & ~1));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = p.num_mb * p.num_nb * p.num_splits;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(full_bar + i), 1);
      mbar_init(smem_u32(empty_bar + i), 1);
    }
    if constexpr (NORM) {
      for (int i = 0; i < SA; ++i) {
        mbar_init(smem_u32(araw_bar + i), 1);
        mbar_init(smem_u32(afree_bar + i), 4);
      }
      for (int i = 0; i < kNormASlots; ++i) {
        mbar_init(smem_u32(tready_bar + i), 4);
        mbar_init(smem_u32(tfree_bar + i), 1);
      }
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(tfull_bar + i), 1);
      mbar_init(smem_u32(tempty_bar + i), 4);
    }
    mbar_init(smem_u32(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_maps; ++i) tma_prefetch_desc(&tm.m[i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_a = tmem_base + 2 * BN;      // the A slots of the fused form
  // inputs written by the previous kernel are read from here on (the producer waits below,
  // after issuing the weight tiles that depend on nothing in flight)
  if (!(warp == 0 && lane == 0)) pdl_wait();

  // The (tile, k-block) steps of this CTA in order, walked by cursors (no divisions per step).
  struct Cursor {
    int t, kb, kb1, mb, nb, split;
  };
  auto cursor_at_tile = [&](Cursor& c, int t) {
    c.t = t;
    if (t < num_tiles) {
      tile_coords(p, t, c.mb, c.nb, c.split);
      c.kb = c.split * p.kb_per_split;
      c.kb1 = min(c.kb + p.kb_per_split, p.num_kb);
    }
  };
  auto cursor_next = [&](Cursor& c) {
    if (++c.kb == c.kb1) cursor_at_tile(c, c.t + static_cast<int>(gridDim.x));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      auto load_a = [&](int stage, int kb, int mb) {
        int a_map, a_row;
        resolve_rows(p.amap, mb * BM, a_map, a_row);
        if constexpr (NORM) {
          // the raw x tile and its gammas, for the norm warps
          const uint32_t ab = smem_u32(araw_bar + stage);
          mbar_expect_tx(ab, A_TX);
          tma_load_2d(smem_u32(sA + stage * A_TILE_BYTES), &tm.m[p.a_map0 + a_map], ab, kb * BK, a_row);
          bulk_load(smem_u32(sG + stage * BK * 2), p.norm_gamma + kb * BK, BK * 2, ab);
        } else {
          tma_load_2d(smem_u32(sA + stage * A_TILE_BYTES), &tm.m[p.a_map0 + a_map], smem_u32(full_bar + stage),
                      kb * BK, a_row);
        }
      };
      auto load_b = [&](int stage, int kb, int nb) {
        if constexpr (EPI == EPI_QKV && BN % 128 != 0) {
          int m0, r0, m1, r1;
          resolve_rows(p.bmap, nb * BN, m0, r0);
          resolve_rows(p.bmap, nb * BN + BN - 1, m1, r1);
          if (m0 != m1) {   // the tile crosses a boundary between two of the matrices
            for (int bx = 0; bx < BN / 32; ++bx) {
              int b_map, b_row;
              resolve_rows(p.bmap, nb * BN + bx * 32, b_map, b_row);
              tma_load_2d(smem_u32(sB + stage * B_TILE_BYTES + bx * 32 * 128), &tm.m[p.b32_map0 + b_map],
                          smem_u32(full_bar + stage), kb * BK, b_row);
            }
            return;
          }
        }
#pragma unroll
        for (int bx = 0; bx < B_BOXES; ++bx) {
          // (this thread's issue latency bounds the ring's lead over TMA latency: no divisions)
          int b_map, b_row;
          if constexpr (EPI == EPI_SWIGLU) {   // tile nb = [gate rows BN/2*nb.. | the same up rows]
            b_map = bx;
            b_row = nb * B_BOX_ROWS;
          } else {
            resolve_rows(p.bmap, nb * BN + bx * B_BOX_ROWS, b_map, b_row);
          }
          tma_load_2d(smem_u32(sB + stage * B_TILE_BYTES + bx * B_BOX_ROWS * 128), &tm.m[p.b_map0 + b_map],
                      smem_u32(full_bar + stage), kb * BK, b_row);
        }
      };
      // the first STAGES k-blocks' weight tiles go out before the dependency wait: the ring
      // starts empty, so these stages need no empty-barrier wait
      int pre = 0;
      if (p.weight_first != 0) {
        for (int t = blockIdx.x; t < num_tiles && pre < STAGES; t += gridDim.x) {
          int mb, nb, split;
          tile_coords(p, t, mb, nb, split);
          const int kb0 = split * p.kb_per_split;
          const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
          for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
            mbar_expect_tx(smem_u32(full_bar + pre), STAGE_TX);
            if (p.weight_first == 1) load_a(pre, kb, mb);   // (never with NORM: A is the activation)
            else load_b(pre, kb, nb);
          }
        }
      }
      pdl_wait();
      bool ok = true;
      if constexpr (NORM) {
        // Before the weight tile of step s goes out, the raw x tiles of steps up to s + SA - 1 do,
        // each into a stage that the norm warps have read (they run ahead of the MMAs by the
        // TMEM A slots).
        constexpr int LEAD = SA - 1;
        Cursor ca, cb;
        cursor_at_tile(ca, blockIdx.x);
        cursor_at_tile(cb, blockIdx.x);
        int sa = 0, sb = 0, stage_a = 0, stage_b = 0;
        uint32_t phase_a = 0, phase_b = 0;
        uint32_t used_a = 0, par_a = 0, used_b = 0, par_b = 0;
        for (; cb.t < num_tiles && ok; cursor_next(cb), ++sb) {
          for (; ca.t < num_tiles && sa <= sb + LEAD; cursor_next(ca), ++sa) {
            if (!mbar_wait(smem_u32(afree_bar + stage_a), phase_a ^ 1u, p.status, abort_flag)) { ok = false; break; }
            load_a(stage_a, ca.kb, ca.mb);
            used_a |= 1u << stage_a;
            par_a = (par_a & ~(1u << stage_a)) | (phase_a << stage_a);
            if (++stage_a == SA) { stage_a = 0; phase_a ^= 1u; }
          }
          if (!ok) break;
          if (sb >= pre) {
            if (!mbar_wait(smem_u32(empty_bar + stage_b), phase_b ^ 1u, p.status, abort_flag)) { ok = false; break; }
            mbar_expect_tx(smem_u32(full_bar + stage_b), STAGE_TX);
            load_b(stage_b, cb.kb, cb.nb);
          }
          used_b |= 1u << stage_b;
          par_b = (par_b & ~(1u << stage_b)) | (phase_b << stage_b);
          if (++stage_b == STAGES) { stage_b = 0; phase_b ^= 1u; }
        }
        if (!ok) {
          // leave no copy in flight: wait (bounded) for the last load into every stage used
          for (int s = 0; s < SA; ++s)
            if (used_a & (1u << s))
              mbar_wait_slow(smem_u32(araw_bar + s), (par_a >> s) & 1u, nullptr, nullptr, kWaitBudgetNs);
          for (int s = 0; s < STAGES; ++s)
            if (used_b & (1u << s))
              mbar_wait_slow(smem_u32(full_bar + s), (par_b >> s) & 1u, nullptr, nullptr, kWaitBudgetNs);
        }
      } else {
        int stage = 0, step = 0;
        uint32_t phase = 0;
        uint32_t used_mask = 0, last_parity = 0;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
          int mb, nb, split;
          tile_coords(p, t, mb, nb, split);
          const int kb0 = split * p.kb_per_split;
          const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
          for (int kb = kb0; kb < kb1; ++kb, ++step) {
            if (step < pre) {   // the weight half of this stage is already on its way
              if (p.weight_first == 1) load_b(stage, kb, nb);
              else load_a(stage, kb, mb);
            } else {
              if (!mbar_wait(smem_u32(empty_bar + stage), phase ^ 1u, p.status, abort_flag)) { ok = false; break; }
              mbar_expect_tx(smem_u32(full_bar + stage), STAGE_TX);
              load_a(stage, kb, mb);
              load_b(stage, kb, nb);
            }
            used_mask |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok) {
          // leave no copy in flight: wait (bounded) for the last load into every stage used
          for (int s = 0; s < STAGES; ++s)
            if (used_mask & (1u << s))
              mbar_wait_slow(smem_u32(full_bar + s), (last_parity >> s) & 1u, nullptr, nullptr, kWaitBudgetNs);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int stage = 0, slot = 0;
      uint32_t phase = 0, slot_phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb, split;
        tile_coords(p, t, mb, nb, split);
        const int kb0 = split * p.kb_per_split;
        const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
        if (!mbar_wait(smem_u32(tempty_bar + acc), acc_phase ^ 1u, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_u32(full_bar + stage), phase, p.status, abort_flag)) { ok = false; break; }
          if constexpr (NORM) {
            if (!mbar_wait(smem_u32(tready_bar + slot), slot_phase, p.status, abort_flag)) { ok = false; break; }
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sB + stage * B_TILE_BYTES);
          if constexpr (NORM) {
            // A from its TMEM slot: row m in lane m, k-block columns packed two per 32-bit column
            const uint32_t a_tmem = tmem_a + static_cast<uint32_t>(slot * (BK / 2));
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              tc_mma_bf16_ts(d_tmem, a_tmem + k * 8, sdesc_sw128(b_addr + k * 32, 16, 1024), IDESC,
                             (kb > kb0 || k > 0) ? 1u : 0u);
          } else {
            const uint32_t a_addr = smem_u32(sA + stage * A_TILE_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
              const uint64_t ad = sdesc_sw128(a_addr + k * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(b_addr + k * 32, 16, 1024);
              tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
            }
          }
          issued = true;
          tc_commit(smem_u32(empty_bar + stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if constexpr (NORM) {
            tc_commit(smem_u32(tfree_bar + slot));
            if (++slot == kNormASlots) { slot = 0; slot_phase ^= 1u; }
          }
        }
        if (!ok) break;
        tc_commit(smem_u32(tfull_bar + acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && issued) {
        // all MMAs of this thread must finish before the TMEM is released
        tc_commit(smem_u32(drain_bar));
        mbar_wait_slow(smem_u32(drain_bar), 0, nullptr, nullptr, kWaitBudgetNs);
      }
    }
  } else if (NORM && warp >= 6) {
    // -------------------------------------------------------------- norm warps 6..9: operand A
    // A warp may only reach the TMEM lanes of its quarter (warp % 4): thread `lane` of warp w
    // owns row 32 (w % 4) + lane of the tile and writes its 64 k-values of each k-block, packed
    // two per 32-bit column, into the 32 columns of the step's A slot.  In the raw tile the row's
    // 16-byte chunk j lies at j ^ (row & 7) (the 128-byte swizzle of the TMA box).
    const int row = (warp & 3) * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float rc = 0.f, rn = 0.f;   // this row's scale in the current tile and in the next one
    Cursor c;
    cursor_at_tile(c, blockIdx.x);
    if (c.t < num_tiles) rc = c.mb * BM + row < p.M ? __ldcg(p.norm_r + c.mb * BM + row) : 0.f;
    int stage = 0, slot = 0;
    uint32_t phase = 0, slot_phase = 0;
    bool ok = true;
    while (c.t < num_tiles && ok) {
      const int t_next = c.t + static_cast<int>(gridDim.x);
      if (t_next < num_tiles) {   // the next tile's scale: its latency hides behind this tile
        int mb, nb, split;
        tile_coords(p, t_next, mb, nb, split);
        rn = mb * BM + row < p.M ? __ldcg(p.norm_r + mb * BM + row) : 0.f;
      }
      for (; c.kb < c.kb1; ++c.kb) {
        if (!mbar_wait(smem_u32(araw_bar + stage), phase, p.status, abort_flag)) { ok = false; break; }
        const uint8_t* xrow = sA + stage * A_TILE_BYTES + row * 128;
        const uint8_t* grow = sG + stage * BK * 2;
        uint32_t o[32];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xrow + ((jj ^ (row & 7)) << 4));
          const uint4 gv = *reinterpret_cast<const uint4*>(grow + jj * 16);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
          // gamma * (x * r) in fp32, rounded once: the value a standalone RMSNorm stores
#pragma unroll
          for (int q = 0; q < 4; ++q)
            o[4 * jj + q] = pack_bf16(bf16_lo(gw[q]) * (bf16_lo(xw[q]) * rc), bf16_hi(gw[q]) * (bf16_hi(xw[q]) * rc));
        }
        // the raw stage is no longer needed: order these generic-proxy reads before the TMA
        // (async-proxy) writes that refill it once the producer sees the arrival
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(afree_bar + stage));
        if (++stage == SA) { stage = 0; phase ^= 1u; }
        // the slot's previous MMAs are done: overwrite it
        if (!mbar_wait(smem_u32(tfree_bar + slot), slot_phase ^ 1u, p.status, abort_flag)) { ok = false; break; }
        tc_fence_after();
        tmem_st32(tmem_a + t_lane + static_cast<uint32_t>(slot * (BK / 2)), o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tready_bar + slot));
        if (++slot == kNormASlots) { slot = 0; slot_phase ^= 1u; }
      }
      if (!ok) break;
      rc = rn;
      cursor_at_tile(c, t_next);
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..5
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb, split;
      tile_coords(p, t, mb, nb, split);
      if (!mbar_wait(smem_u32(tfull_bar + acc), acc_phase, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + t_lane + static_cast<uint32_t>(acc * BN);
      const int m = mb * BM + row;
      uint32_t r[32];
      float v[32];

      if constexpr (EPI == EPI_BF16 || EPI == EPI_F32 || EPI == EPI_RESID) {
        // residual rows of the next chunk are loaded one chunk ahead (their latency then
        // overlaps this chunk's TMEM load, add and store)
        uint4 res_n[4];
        auto load_resid = [&](int c) {
          if constexpr (EPI == EPI_RESID) {
            const int n0 = nb * BN + c * 32;
            if (c < BN / 32 && m < p.M && n0 + 32 <= p.N) {
              const uint4* src = reinterpret_cast<const uint4*>(p.resid + m * p.ldr + n0);
#pragma unroll
              for (int g = 0; g < 4; ++g) res_n[g] = src[g];
            }
          }
        };
        load_resid(0);
        float ss = 0.f;   // row statistics: the sum of squares of this row's rounded outputs
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint4 res_c[4];
#pragma unroll
          for (int g = 0; g < 4; ++g) res_c[g] = res_n[g];
          load_resid(c + 1);
          tmem_ld32(t_acc + c * 32, r);
          const int n0 = nb * BN + c * 32;
          const int valid = min(32, p.N - n0);
          if (m < p.M && valid > 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            if constexpr (EPI == EPI_F32) {
              float* dst = static_cast<float*>(p.out) + m * p.ldo + n0;
              if (valid >= 32) {
                float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
                for (int g = 0; g < 8; ++g) d4[g] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
              } else {
                for (int i = 0; i < valid; ++i) dst[i] = v[i];
              }
            } else {
              if constexpr (EPI == EPI_RESID) {
                float rr[32];
                if (valid >= 32) {
#pragma unroll
                  for (int g = 0; g < 4; ++g) {
                    const uint4 w = res_c[g];
                    rr[8 * g + 0] = bf16_lo(w.x); rr[8 * g + 1] = bf16_hi(w.x);
                    rr[8 * g + 2] = bf16_lo(w.y); rr[8 * g + 3] = bf16_hi(w.y);
                    rr[8 * g + 4] = bf16_lo(w.z); rr[8 * g + 5] = bf16_hi(w.z);
                    rr[8 * g + 6] = bf16_lo(w.w); rr[8 * g + 7] = bf16_hi(w.w);
                  }
                } else {
                  load_bf16x32(p.resid + m * p.ldr + n0, rr, valid);
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] += rr[i];
                if (p.stat_part != nullptr) {
#pragma unroll
                  for (int i = 0; i < 32; ++i) {
                    const float hb = __bfloat162float(__float2bfloat16_rn(v[i]));   // the stored value
                    ss = i < valid ? fmaf(hb, hb, ss) : ss;
                  }
                }
              }
              store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + m * p.ldo + n0, v, valid);
            }
          }
        }
        if constexpr (EPI == EPI_RESID) {
          if (p.stat_part != nullptr && m < p.M) {
            // this tile's share of row m; the row's last column tile to finish completes r_m
            p.stat_part[static_cast<long long>(nb) * p.M + m] = ss;
            __threadfence();
            if (atomicAdd(p.stat_ticket + m, 1) == p.num_nb - 1) {
              __threadfence();
              float tot = 0.f;
#pragma unroll 4
              for (int q = 0; q < p.num_nb; ++q) tot += __ldcg(p.stat_part + static_cast<long long>(q) * p.M + m);
              p.stat_r[m] = rsqrtf(tot * p.stat_inv_n + p.stat_eps);
              p.stat_ticket[m] = 0;
            }
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // columns [0, BN/2) of the tile are gate rows BN/2*nb.., [BN/2, BN) the matching up rows.
        // Every TMEM load covers 32 columns starting at a multiple of 32; when the halves are not
        // (BN/2 = 112) the up values of an output chunk come from two such loads, 16 apart.
        constexpr int HALF = BN / 2;
        constexpr int SHIFT = HALF % 32;
        static_assert(SHIFT == 0 || SHIFT == 16, "gate/up halves of 16-column multiples");
#pragma unroll 1
        for (int c0 = 0; c0 < HALF; c0 += 32) {
          uint32_t u[32];
          tmem_ld32(t_acc + c0, r);
          if constexpr (SHIFT == 0) {
            tmem_ld32(t_acc + HALF + c0, u);
          } else {
            uint32_t u0[32];
            const int ua = HALF + c0 - SHIFT;   // aligned start of the load holding the first up value
            tmem_ld32(t_acc + ua, u0);
#pragma unroll
            for (int i = 0; i < 16; ++i) u[i] = u0[16 + i];
            if (c0 + 16 < HALF) {
              tmem_ld32(t_acc + ua + 32, u0);
#pragma unroll
              for (int i = 0; i < 16; ++i) u[16 + i] = u0[i];
            }
          }
          const int n0 = nb * HALF + c0;
          const int valid = min(min(32, HALF - c0), p.N - n0);
          if (m < p.M && valid > 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = silu_f(__uint_as_float(r[i])) * __uint_as_float(u[i]);
            store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + m * p.ldo + n0, v, valid);
          }
        }
      } else if constexpr (EPI == EPI_QKV) {
        // the tile's columns are part of [q heads | k heads | v heads]; token s of sequence b sits at position start[b] + s, and only tokens s < lens[b]
        // are stored (the others pad the chunk)
        const int b = m / p.S, s_in = m - (m / p.S) * p.S;
        int s = s_in;
        bool keep = m < p.M;
        if (keep && p.start != nullptr) {
          const int st = p.start[b], len = p.lens != nullptr ? p.lens[b] : p.S;
          if (st < 0 || len < 0 || len > p.S || st + len > p.T_max || st + len > p.max_pos) {
            if (s_in == 0) report(p.status, LLAMA_ERR_DEVICE_BOUNDS);
            keep = false;
          }
          keep = keep && s_in < len;
          s = st + s_in;
        }
        const int half_d = p.D >> 1;
        // RoPE angles of chunk c for this row's position, when chunk c is part of a q or k head
        // of this tile: 16 pairs (even/odd: angle index j0/2 ..) or, for a chunk of the first
        // half of a head, 32 pairs (half-split: angle index j0 ..)
        float cs_n[32], sn_n[32];
        auto load_angles = [&](int c) {
          const int col0 = nb * BN + c * 32;
          const int hh = col0 / p.D, j0 = col0 - hh * p.D;
          if (!keep || c >= BN / 32 || hh >= p.H + p.G || (p.rope_half && j0 >= half_d)) return;
          const int first = p.rope_half ? j0 : j0 / 2;
          const float4* cr = reinterpret_cast<const float4*>(p.cos + static_cast<long long>(s) * half_d + first);
          const float4* sr = reinterpret_cast<const float4*>(p.sin + static_cast<long long>(s) * half_d + first);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i >= 4 && !p.rope_half) break;
            const float4 cv = cr[i], sv = sr[i];
            cs_n[4 * i] = cv.x; cs_n[4 * i + 1] = cv.y; cs_n[4 * i + 2] = cv.z; cs_n[4 * i + 3] = cv.w;
            sn_n[4 * i] = sv.x; sn_n[4 * i + 1] = sv.y; sn_n[4 * i + 2] = sv.z; sn_n[4 * i + 3] = sv.w;
          }
        };
        load_angles(0);
        // 32-column chunks of the tile, each inside one head (D = 128): column col0 of
        // [q heads | k heads | v heads] is element j0 of head hh
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col0 = nb * BN + c * 32;
          const int hh = col0 / p.D, j0 = col0 - hh * p.D;
          if (hh >= p.H + 2 * p.G) break;
          if (p.rope_half && hh < p.H + p.G) {
            // half-split pairs (j, j + D/2), angle index j: the head's two halves are both in
            // this tile (the host gives this form head-aligned 256-column tiles); the chunks
            // of the first half take the pairs
            if (j0 >= half_d) continue;
            __nv_bfloat16* dst = hh < p.H
                ? p.q_out + ((static_cast<long long>(b) * p.H + hh) * p.S + s_in) * p.D
                : p.k_cache + ((static_cast<long long>(b) * p.G + (hh - p.H)) * p.T_max + s) * p.D;
            // this chunk's 32 angles, loaded here (32 pairs per chunk: a look-ahead copy would
            // not fit the registers of the RMSNorm-fused form)
            load_angles(c);
            uint32_t r2[32];
            tmem_ld32(t_acc + c * 32, r);
            tmem_ld32(t_acc + c * 32 + half_d, r2);
            if (!keep) continue;
            float w2[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float x1 = __uint_as_float(r[i]), x2 = __uint_as_float(r2[i]);
              v[i] = x1 * cs_n[i] - x2 * sn_n[i];
              w2[i] = x2 * cs_n[i] + x1 * sn_n[i];
            }
            store_bf16x32(dst + j0, v, 32);
            store_bf16x32(dst + j0 + half_d, w2, 32);
            continue;
          }
          // this chunk's angles were loaded during the previous chunk; load the next chunk's
          // now, so that their L2 latency overlaps this chunk's TMEM load and arithmetic
          float cs_c[16], sn_c[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            cs_c[i] = cs_n[i];
            sn_c[i] = sn_n[i];
          }
          load_angles(c + 1);
          tmem_ld32(t_acc + c * 32, r);
          if (!keep) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          __nv_bfloat16* dst;
          if (hh < p.H + p.G) {
            // RoPE on q and k: pair (2i, 2i+1) rotated by angle s * base^(-2i/D)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float e = v[2 * i], o = v[2 * i + 1];
              v[2 * i] = e * cs_c[i] - o * sn_c[i];
              v[2 * i + 1] = e * sn_c[i] + o * cs_c[i];
            }
          }
          if (hh < p.H)
            dst = p.q_out + ((static_cast<long long>(b) * p.H + hh) * p.S + s_in) * p.D;
          else if (hh < p.H + p.G)
            dst = p.k_cache + ((static_cast<long long>(b) * p.G + (hh - p.H)) * p.T_max + s) * p.D;
          else
            dst = p.v_cache + ((static_cast<long long>(b) * p.G + (hh - p.H - p.G)) * p.T_max + s) * p.D;
          store_bf16x32(dst + j0, v, 32);
        }
      } else if constexpr (EPI == EPI_PARTIAL) {
        // kernel M = weight rows, N = tokens: P[split][token][row] in fp32
        float* P = static_cast<float*>(p.out);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          tmem_ld32(t_acc + c * 32, r);
          if (m < p.M) {
            const int n0 = nb * BN + c * 32;
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
              const int n = n0 + i;
              if (n < p.N) P[(static_cast<long long>(split) * p.N + n) * p.ldo + m] = __uint_as_float(r[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty_bar + acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
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

template <int BN, int EPI, int STAGES, bool NORM>
constexpr size_t smem_bytes() {
  // alignment slack, the rings, the barriers, the TMEM slot and the abort flag (padded to 16
  // bytes), the gammas of each A stage
  constexpr int SA = a_stages_of<NORM, STAGES>();
  constexpr int bar_words = 2 * STAGES + 5 + (NORM ? 2 * SA + 2 * kNormASlots : 0);
  return 1024 + SA * A_TILE_BYTES + STAGES * BN * BK * 2 + ((bar_words + 2) & ~1) * 8 + (NORM ? SA * BK * 2 : 0);
}

template <int BN, int EPI, int STAGES, bool NORM = false>
int launch(const Ctx& c, const TMaps& tm, Params p) {
  auto kern = gemm_tc_kernel<BN, EPI, STAGES, NORM>;
  constexpr size_t smem = smem_bytes<BN, EPI, STAGES, NORM>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  static_assert(smem >= kTmemKernelMinSmem, "a TMEM-holding kernel must not share an SM with another");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  });
  if (attr_err != cudaSuccess) return LLAMA_ERR_CUDA;
  p.status = c.status;
  if (!c.static_weights) p.weight_first = 0;
  const int tiles = p.num_mb * p.num_nb * p.num_splits;
  if (tiles == 0) return LLAMA_OK;
  if (NORM && (p.norm_gamma == nullptr || p.norm_r == nullptr || p.num_splits != 1 || p.K % BK != 0 ||
               p.amap.nseg != 1 || p.weight_first == 1 || (reinterpret_cast<uintptr_t>(p.norm_gamma) & 15) != 0))
    return LLAMA_ERR_INVALID_ARG;
  const int grid = std::min(tiles, c.num_sms);
  launch_pdl(c, kern, dim3(grid), dim3(threads_of<NORM>()), smem, tm, p);
  return after_launch(c);
}

// RMSNorm-fused form: operand A (its tensor map) is x [M, K]; gamma [K] and the row scales r [M].
void set_norm(Params& p, const NormIn& n) {
  p.norm_gamma = static_cast<const __nv_bfloat16*>(n.gamma);
  p.norm_r = n.r;
}

// Rounds of num_sms tiles times the tile width: the time of a GEMM with M rows and n_blocks
// column blocks of width bn, a round's time taken as proportional to its width.
long long round_cost(int M, int n_blocks, int bn, int num_sms) {
  const long long tiles = static_cast<long long>((M + BM - 1) / BM) * n_blocks;
  return (tiles + num_sms - 1) / num_sms * bn;
}

// Tile width (256 or 224 columns) with the least round cost for N output columns; ties keep 256.
int tile_width_for(int M, int N, int num_sms) {
  return round_cost(M, (N + 223) / 224, 224, num_sms) < round_cost(M, (N + 255) / 256, 256, num_sms) ? 224 : 256;
}

Params base_params(int M, int N, int K, int BN) {
  Params p{};
  p.M = M;
  p.N = N;
  p.K = K;
  p.num_mb = (M + BM - 1) / BM;
  p.num_nb = (N + BN - 1) / BN;
  p.num_kb = (K + BK - 1) / BK;
  p.num_splits = 1;
  p.kb_per_split = p.num_kb;
  p.weight_first = 2;   // B holds the weights (kept only when the context says they are static)
  // tile order: a group of group_m row blocks walks all column blocks, so that group's rows
  // of A stay in L2 while the weights stream; take every row block when all of A fits in
  // 48 MB (the weights then stream from DRAM once), else about 32 MB of A per group
  const size_t a_block_bytes = static_cast<size_t>(BM) * K * 2;
  const size_t a_bytes = a_block_bytes * p.num_mb;
  p.group_m = a_bytes <= (48u << 20) ? std::max(1, p.num_mb)
                                     : std::max(8, static_cast<int>((32u << 20) / std::max<size_t>(a_block_bytes, 1)));
  p.amap.nseg = 1;
  p.amap.seg_end[0] = 1 << 30;
  p.bmap.nseg = 1;
  p.bmap.seg_end[0] = 1 << 30;
  p.b32_map0 = 0;
  p.n_maps = 2;
  return p;
}

}  // namespace

int gemm_plain(const Ctx& c, const void* X, const void* W, void* C, int M, int N, int K, bool c_f32,
               const NormIn* norm) {
  const int bn = tile_width_for(M, N, c.num_sms);
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], W, K, N, K, bn == 256 ? 128 : bn))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, N, K, bn);
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.out = C;
  p.ldo = N;
  if (norm != nullptr) {
    // 224-column tiles: the two accumulators leave tensor memory room for the A slots
    if (bn != 224) {
      if (!make_tmap_2d(&tm.m[1], W, K, N, K, 224)) return LLAMA_ERR_INVALID_ARG;
      p = base_params(M, N, K, 224);
      p.a_map0 = 0;
      p.b_map0 = 1;
      p.out = C;
      p.ldo = N;
    }
    set_norm(p, *norm);
    return c_f32 ? launch<224, EPI_F32, 5, true>(c, tm, p) : launch<224, EPI_BF16, 5, true>(c, tm, p);
  }
  if (bn == 256) return c_f32 ? launch<256, EPI_F32, 4>(c, tm, p) : launch<256, EPI_BF16, 4>(c, tm, p);
  return c_f32 ? launch<224, EPI_F32, 5>(c, tm, p) : launch<224, EPI_BF16, 5>(c, tm, p);
}

int residual_col_tiles(const Ctx& c, int M, int N) {
  const int bn = tile_width_for(M, N, c.num_sms);
  return (N + bn - 1) / bn;
}

int gemm_residual(const Ctx& c, const void* X, const void* W, const void* resid, void* out, int M, int N, int K,
                  const RowStatsOut* stats) {
  // 224-column tiles when they finish in fewer tile-column rounds (e.g. N = 4096 at M = 2048:
  // 304 tiles fill 2 rounds of 152 SMs, where 256 tiles of 256 columns leave the second
  // round two-thirds full)
  const int bn = tile_width_for(M, N, c.num_sms);
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], W, K, N, K, bn == 256 ? 128 : bn))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, N, K, bn);
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.out = out;
  p.ldo = N;
  p.resid = static_cast<const __nv_bfloat16*>(resid);
  p.ldr = N;
  if (stats != nullptr) {
    if (stats->part == nullptr || stats->r == nullptr || stats->ticket == nullptr) return LLAMA_ERR_INVALID_ARG;
    p.stat_part = stats->part;
    p.stat_r = stats->r;
    p.stat_ticket = stats->ticket;
    p.stat_inv_n = 1.0f / static_cast<float>(N);
    p.stat_eps = stats->eps;
  }
  return bn == 256 ? launch<256, EPI_RESID, 4>(c, tm, p) : launch<224, EPI_RESID, 5>(c, tm, p);
}

int gemm_swiglu(const Ctx& c, const void* X, const void* Wg, const void* Wu, void* out, int M, int I, int K,
                const NormIn* norm) {
  if (norm != nullptr) {
    // 224-column tiles (112 gate + 112 up rows): the two accumulators leave tensor memory room
    // for the A slots of the RMSNorm-fused form
    TMaps tm{};
    if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], Wg, K, I, K, 112) ||
        !make_tmap_2d(&tm.m[2], Wu, K, I, K, 112))
      return LLAMA_ERR_INVALID_ARG;
    Params p = base_params(M, 2 * ((I + 111) / 112) * 112, K, 224);
    p.N = I;
    p.a_map0 = 0;
    p.b_map0 = 1;
    p.n_maps = 3;
    p.out = out;
    p.ldo = I;
    set_norm(p, *norm);
    return launch<224, EPI_SWIGLU, 5, true>(c, tm, p);
  }
  // kernel N runs over 256-column tiles, each = 128 gate rows + the same 128 up rows (measured:
  // 240-column tiles, which fill the SM-count rounds better at I = 11008, M = 2048, run slower)
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], Wg, K, I, K, 128) ||
      !make_tmap_2d(&tm.m[2], Wu, K, I, K, 128))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, 2 * ((I + 127) / 128) * 128, K, 256);
  p.N = I;   // output width (used by the epilogue's bounds)
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.n_maps = 3;
  p.out = out;
  p.ldo = I;
  return launch<256, EPI_SWIGLU, 4>(c, tm, p);
}

int gemm_qkv_rope(const Ctx& c, const void* X, const void* Wq, const void* Wk, const void* Wv, int B, int S, int K,
                  int H, int G, int D, const float* cos, const float* sin, void* q_out, void* k_cache,
                  void* v_cache, int T_max, int rope_half, const int32_t* start, const int32_t* lens,
                  int max_pos, const NormIn* norm) {
  const int M = B * S;
  // 224-column tiles when they fill the SM-count rounds better (the half-split pairs (j, j+64)
  // need whole heads in a tile: 256 columns = two heads); a 224-column tile that crosses the
  // q|k or k|v boundary takes its weights in 32-row boxes from the maps at b32_map0.  The
  // RMSNorm-fused form always takes 224 columns (tensor memory holds its A slots) and so not the
  // half-split pairs.
  if (norm != nullptr && rope_half) return LLAMA_ERR_UNSUPPORTED;
  const int bn = rope_half ? 256 : norm != nullptr ? 224 : tile_width_for(M, (H + 2 * G) * D, c.num_sms);
  const int box = bn == 256 ? 128 : bn;
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], Wq, K, H * D, K, box) ||
      !make_tmap_2d(&tm.m[2], Wk, K, G * D, K, box) || !make_tmap_2d(&tm.m[3], Wv, K, G * D, K, box))
    return LLAMA_ERR_INVALID_ARG;
  if (bn != 256 && (!make_tmap_2d(&tm.m[4], Wq, K, H * D, K, 32) || !make_tmap_2d(&tm.m[5], Wk, K, G * D, K, 32) ||
                    !make_tmap_2d(&tm.m[6], Wv, K, G * D, K, 32)))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, (H + 2 * G) * D, K, bn);
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.b32_map0 = 4;
  p.n_maps = bn == 256 ? 4 : 7;
  p.bmap.nseg = 3;
  p.bmap.seg_end[0] = H * D;
  p.bmap.seg_end[1] = (H + G) * D;
  p.bmap.seg_end[2] = (H + 2 * G) * D;
  p.cos = cos;
  p.sin = sin;
  p.S = S;
  p.H = H;
  p.G = G;
  p.D = D;
  p.T_max = T_max;
  p.rope_half = rope_half;
  p.start = start;
  p.lens = lens;
  p.max_pos = max_pos;
  p.q_out = static_cast<__nv_bfloat16*>(q_out);
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  if (norm != nullptr) {
    set_norm(p, *norm);
    return launch<224, EPI_QKV, 5, true>(c, tm, p);
  }
  return bn == 256 ? launch<256, EPI_QKV, 4>(c, tm, p) : launch<224, EPI_QKV, 5>(c, tm, p);
}

int choose_splits(int num_sms, int w_rows_total, int K, int n_tok) {
  // Cost of streaming the weights once with s splits, relative to a perfectly balanced
  // stream: the slowest SM handles ceil(tiles / SMs) tiles of ceil(kb / s) k-blocks; the fp32
  // partials add 2 * s * n_tok * rows * 4 bytes (written, then read by the fixup kernel)
  // against rows * K * 2 bytes of weights.
  const int mb = (w_rows_total + BM - 1) / BM;
  const int kb = (K + BK - 1) / BK;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= std::max(1, kb / 4); ++s) {
    const int per = (kb + s - 1) / s;
    const int se = (kb + per - 1) / per;   // the count actually used: no empty split
    const int rounds = (mb * se + num_sms - 1) / num_sms;
    const double cost = static_cast<double>(rounds) * per * num_sms / (static_cast<double>(mb) * kb) +
                        4.0 * se * n_tok / static_cast<double>(K);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = se;
    }
  }
  return best;
}

int gemm_tokens_partial(const Ctx& c, const void* const* W, const int* w_rows, int n_w, const void* X, int n_tok,
                        int K, int splits, float* P) {
  if (n_w < 1 || n_w > 3) return LLAMA_ERR_INVALID_ARG;
  TMaps tm{};
  int total = 0;
  Params p = base_params(0, n_tok, K, 64);
  for (int i = 0; i < n_w; ++i) {
    if (!make_tmap_2d(&tm.m[i], W[i], K, w_rows[i], K, 128)) return LLAMA_ERR_INVALID_ARG;
    total += w_rows[i];
    p.amap.seg_end[i] = total;
  }
  if (!make_tmap_2d(&tm.m[n_w], X, K, n_tok, K, 64)) return LLAMA_ERR_INVALID_ARG;
  p.M = total;
  p.num_mb = (total + BM - 1) / BM;
  p.amap.nseg = n_w;
  p.a_map0 = 0;
  p.b_map0 = n_w;
  p.n_maps = n_w + 1;
  splits = std::max(1, std::min(splits, p.num_kb));
  p.kb_per_split = (p.num_kb + splits - 1) / splits;
  p.num_splits = (p.num_kb + p.kb_per_split - 1) / p.kb_per_split;   // every split non-empty
  if (p.num_splits != splits) return LLAMA_ERR_INVALID_ARG;          // callers pass choose_splits()
  p.out = P;
  p.ldo = total;
  // No weight loads before griddepcontrol.wait here: measured on the decode step, streaming
  // weights under the preceding fixup kernel slows that kernel more than it saves.
  p.weight_first = 0;
  return launch<64, EPI_PARTIAL, 8>(c, tm, p);
}

}  // namespace llama
