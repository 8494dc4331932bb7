// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
// C = X W^T ("12 · 从 Transformer 到 LLaMA 系列" §八: every projection of the layer is an
// nn.Linear without bias).  One CTA per SM walks a list of output tiles:
//   warp 0     TMA producer: 128x64 A tile + BNx64 B tile per stage (128-byte swizzle)
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma 128xBNx16 into a TMEM accumulator
//   warps 2-5  epilogue: tcgen05.ld of the accumulator rows, fused op, stores to HBM
// Two TMEM accumulators let the epilogue of tile i overlap the main loop of tile i+1.
//
// RMSNorm in the prologue ("12 · 从 Transformer 到 LLaMA 系列" §八 RMSNorm: y = gamma * x *
// rsqrt(mean(x^2) + eps); "3.2 核心组件逐一拆解" §3.2.1: the statistics in fp32).  When the A
// operand is the normalised activation, the GEMM normalises it itself before its main loop: the
// epilogue warps, idle until the first accumulator is ready, take the rows of x in turn (one warp
// per row, the row's sum of squares reduced across the warp in fp32), write gamma * (x * r) as
// bf16 -- exactly what a standalone RMSNorm stores -- into the A buffer, and count themselves in
// on a grid-wide counter.  The TMA producer issues the weight tiles of its first stages, waits
// (bounded) for the count to reach every prologue warp of the grid, and then streams the
// normalised rows as A as usual.  The main loop is the plain GEMM's: the normalisation touches
// no shared memory (the GEMMs are bound by shared-memory bandwidth, and every form that
// rewrote or re-staged the operand between TMA and the tensor cores measured 50-90 % slower).
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

enum Epi : int { EPI_BF16 = 0, EPI_F32 = 1, EPI_RESID = 2, EPI_SWIGLU = 3, EPI_QKV = 4, EPI_PARTIAL = 5 };
// How the CTAs of a launch share weight tiles: one CTA per tile; clusters of two CTAs on
// consecutive row blocks whose B tile reaches both through TMA multicast; or pairs of CTAs
// whose even CTA issues two-SM products over both CTAs' halves of B.
enum TileMode : int { kSingle = 0, kShareB = 1, kPair = 2 };

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
  // RMSNorm in the prologue (null pro_out: none): rows [0, M) of pro_x [M, K] normalised with
  // pro_gamma [K] into pro_out [M, K], the buffer operand A is read from
  const __nv_bfloat16* pro_x;
  const __nv_bfloat16* pro_gamma;
  __nv_bfloat16* pro_out;
  float pro_inv_k, pro_eps;
  int* pro_count;               // prologue warps done (zero before the launch)
  int* status;
};

__device__ __forceinline__ float warp_sum32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Rows gw, gw + nw, ... of the prologue's RMSNorm, K = VPL * 256: lane owns 16-byte vectors
// i * 32 + lane of its row (the order of the standalone RMSNorm kernel, so both give the same
// bits); the next row's loads are issued before this row's reduction.
template <int VPL>
__device__ __noinline__ void prologue_rows(const Params& p, int gw, int nw, int lane) {
  const uint4* x = reinterpret_cast<const uint4*>(p.pro_x);
  const uint4* g = reinterpret_cast<const uint4*>(p.pro_gamma);
  uint4* y = reinterpret_cast<uint4*>(p.pro_out);
  uint4 v[VPL], vn[VPL];
  int row = gw;
  if (row < p.M) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = __ldcs(x + static_cast<long long>(row) * (VPL * 32) + i * 32 + lane);
  }
  for (; row < p.M; row += nw) {
    const int nrow = row + nw;
    if (nrow < p.M) {
#pragma unroll
      for (int i = 0; i < VPL; ++i) vn[i] = __ldcs(x + static_cast<long long>(nrow) * (VPL * 32) + i * 32 + lane);
    }
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
    ss = warp_sum32(ss);
    const float r = rsqrtf(ss * p.pro_inv_k + p.pro_eps);
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const uint4 gv = __ldg(g + i * 32 + lane);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      const uint32_t gw4[4] = {gv.x, gv.y, gv.z, gv.w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o[j] = pack_bf16(bf16_lo(gw4[j]) * (bf16_lo(w[j]) * r), bf16_hi(gw4[j]) * (bf16_hi(w[j]) * r));
      y[static_cast<long long>(row) * (VPL * 32) + i * 32 + lane] = make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = vn[i];
  }
}

// Any K: lane-strided elements, two passes over the row (the second from L1).
__device__ __noinline__ void prologue_rows_generic(const Params& p, int gw, int nw, int lane) {
  for (int row = gw; row < p.M; row += nw) {
    const __nv_bfloat16* xr = p.pro_x + static_cast<long long>(row) * p.K;
    float ss = 0.f;
    for (int i = lane; i < p.K; i += 32) {
      const float a = __bfloat162float(xr[i]);
      ss = fmaf(a, a, ss);
    }
    ss = warp_sum32(ss);
    const float r = rsqrtf(ss * p.pro_inv_k + p.pro_eps);
    __nv_bfloat16* yr = p.pro_out + static_cast<long long>(row) * p.K;
    for (int i = lane; i < p.K; i += 32)
      yr[i] = __float2bfloat16_rn(__bfloat162float(p.pro_gamma[i]) * (__bfloat162float(xr[i]) * r));
  }
}

// Wait (bounded) until *count reaches target; false (and LLAMA_ERR_TIMEOUT recorded) if it
// does not within the wait budget or another wait of the CTA gave up.
__device__ __noinline__ bool wait_count(const int* count, int target, int* status, volatile int* abort_flag) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
    if (v >= target) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer_ns();
      if (now - t0 > kWaitBudgetNs) {
        report_timeout(status, now - t0, it, 0xFFFFFFFFu, static_cast<uint32_t>(target));
        *abort_flag = 1;
        return false;
      }
    }
    __nanosleep(64);
  }
}

__device__ __forceinline__ void resolve_rows(const RowMap& rm, int vrow, int& map, int& row) {
  map = 0;
  int start = 0;
  if (rm.nseg > 1 && vrow >= rm.seg_end[0]) { map = 1; start = rm.seg_end[0]; }
  if (rm.nseg > 2 && vrow >= rm.seg_end[1]) { map = 2; start = rm.seg_end[1]; }
  row = vrow - start;
}

// Work unit u of a launch with clusters of CM CTAs along M: the CM CTAs of a cluster take the
// row blocks CM * i + rank of the same column block (and split), so they share its weight
// tile.  The order is tile_coords' over CM-row-block units (CM = 1: the same tiles).
template <int CM>
__device__ __forceinline__ void unit_coords(const Params& p, int u, int rank, int& mb, int& nb, int& split) {
  split = u % p.num_splits;
  u /= p.num_splits;
  const int units_m = p.num_mb / CM, gmm = max(1, p.group_m / CM);
  const int per_group = gmm * p.num_nb;
  const int g = u / per_group, r = u % per_group;
  const int first_m = g * gmm;
  const int gm = min(gmm, units_m - first_m);
  mb = (first_m + r % gm) * CM + rank;
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

// MODE kShareB: clusters of two CTAs on consecutive row blocks of one column block.  Each CTA
// loads its own A tile and half of the B (weight) tile's boxes, which TMA multicast writes into
// both CTAs' stage: half the weight reads from L2.  A stage is refilled once both CTAs'
// products have read it (each empty barrier counts one commit from each).
// MODE kPair: two-SM products.  The pair takes the two row blocks as one 256 x BN tile: each
// CTA loads its own A tile and half of B's rows, and the even CTA issues M = 256 products
// (.cta_group::2) that read both CTAs' shared memory and write each CTA's 128 rows of D into
// its own TMEM: a third less operand traffic into each SM per k-block than either form above
// (the 128 x 256 tiles are bound by that traffic, not by the tensor cores), and deeper rings in
// the same shared memory.  The odd CTA's copies complete on the even CTA's full barriers; the
// even CTA's commits reach both CTAs' empty and accumulator-full barriers; both CTAs'
// epilogues release the even CTA's accumulators.  (Measured faster than kShareB at 256-column
// tiles, slower at 224: those take kShareB.)
template <int BN, int EPI, int STAGES, int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ TMaps tm, const Params p) {
  constexpr int CM = MODE == kSingle ? 1 : 2;   // CTAs per cluster
  constexpr bool kPairMma = MODE == kPair;
  // B rows this CTA holds per stage: the whole tile, or its half in a pair
  constexpr int B_ROWS = kPairMma ? BN / 2 : BN;
  constexpr int B_TILE_BYTES = B_ROWS * BK * 2;
  // B arrives in 128-row boxes, or as one box of all its rows when that is not a multiple of
  // 128 (<= 256), as two halves in kShareB clusters (each CTA loads one for both); gate/up
  // tiles: BN/2 gate rows (128, or 120 in 240-column pairs), then the same up rows (in a pair,
  // the even CTA holds the gate rows, the odd one the up rows)
  constexpr int B_BOX_ROWS =
      EPI == EPI_SWIGLU ? BN / 2 : B_ROWS % 128 == 0 ? 128 : (MODE == kShareB ? BN / 2 : B_ROWS);
  constexpr int B_BOXES = B_ROWS / B_BOX_ROWS;
  static_assert(MODE == kSingle || (EPI != EPI_PARTIAL && (MODE == kShareB ? B_BOXES % 2 == 0
                                                                           : (BN % 128 == 0 || EPI == EPI_SWIGLU))),
                "clusters split B into whole boxes, one half per CTA");
  constexpr uint16_t kBoth = 3;                 // cluster ranks 0 and 1
  constexpr uint32_t STAGE_TX = A_TILE_BYTES + B_TILE_BYTES;
  // columns per accumulator: the tile width rounded up to 32, so that the second accumulator
  // starts on a 32-column boundary (256 for 240-column tiles)
  constexpr int ACC_COLS = (BN + 31) / 32 * 32;
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS <= 32    ? 32
                                 : 2 * ACC_COLS <= 64  ? 64
                                 : 2 * ACC_COLS <= 128 ? 128
                                 : 2 * ACC_COLS <= 256 ? 256
                                                       : 512;
  constexpr uint32_t IDESC = idesc_bf16(kPairMma ? 2 * BM : BM, BN, false);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128 and 256");

  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_TILE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_TILE_BYTES);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + STAGES;
  uint64_t* tfull_bar = bars + 2 * STAGES;
  uint64_t* tempty_bar = bars + 2 * STAGES + 2;
  uint64_t* drain_bar = bars + 2 * STAGES + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // work units (tiles, or tile pairs in clusters) walked by this CTA's cluster
  const int num_units = p.num_mb / CM * p.num_nb * p.num_splits;
  const int unit0 = static_cast<int>(blockIdx.x) / CM, unit_step = static_cast<int>(gridDim.x) / CM;
  const int rank = CM == 1 ? 0 : static_cast<int>(cluster_ctarank());

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(full_bar + i), 1);
      mbar_init(smem_u32(empty_bar + i), MODE == kShareB ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(tfull_bar + i), 1);
      mbar_init(smem_u32(tempty_bar + i), kPairMma ? 8 : 4);   // the epilogue warps of every CTA of a pair
    }
    mbar_init(smem_u32(drain_bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < p.n_maps; ++i) tma_prefetch_desc(&tm.m[i]);
  }
  if (warp == 1) {
    if constexpr (kPairMma) {
      tmem_alloc2(smem_u32(tmem_slot), TMEM_COLS);   // the same columns in both CTAs
      tmem_relinquish2();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (CM > 1)
    cluster_sync();   // the peer's barriers are initialised before any signal reaches them
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // inputs written by the previous kernel are read from here on (the producer waits below,
  // after issuing the weight tiles that depend on nothing in flight)
  if (!(warp == 0 && lane == 0)) pdl_wait();
  // Prologue RMSNorm (the forms whose A can be a normalised activation): every warp of the CTA
  // normalises its share of the rows of A before taking up its role (the producer after issuing
  // its first weight tiles), then counts itself in.
  constexpr bool kPrologue = EPI == EPI_BF16 || EPI == EPI_F32 || EPI == EPI_SWIGLU || EPI == EPI_QKV;
  const bool prologue = kPrologue && p.pro_out != nullptr;
  auto run_prologue = [&]() {
    const int gw = static_cast<int>(blockIdx.x) * (NUM_THREADS / 32) + warp;
    const int nw = static_cast<int>(gridDim.x) * (NUM_THREADS / 32);
    switch (p.K % 256 == 0 && p.K <= 4096 ? p.K / 256 : 0) {
      case 1: prologue_rows<1>(p, gw, nw, lane); break;
      case 2: prologue_rows<2>(p, gw, nw, lane); break;
      case 4: prologue_rows<4>(p, gw, nw, lane); break;
      case 8: prologue_rows<8>(p, gw, nw, lane); break;
      case 16: prologue_rows<16>(p, gw, nw, lane); break;
      default: prologue_rows_generic(p, gw, nw, lane);
    }
    // the rows go to other CTAs' TMA loads: order the generic stores before them
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(p.pro_count, 1);
  };
  if (prologue && warp >= 1) run_prologue();

  if (warp == 0) {
    {
      // ------------------------------------------------------------ TMA producer (lane 0)
      // one box into this CTA's stage; in a pair the odd CTA's copies complete on the even
      // CTA's full barrier (the even CTA's products read both CTAs' stages)
      // (kShareB: B boxes go to the same stage of both CTAs of the cluster)
      const uint32_t full_pair0 = kPairMma ? cluster_map(smem_u32(full_bar), 0) : 0u;
      const uint64_t evict_first = EPI == EPI_PARTIAL ? l2_evict_first_policy() : 0;
      auto load_box = [&](uint32_t dst, const CUtensorMap* map, int stage, int c0, int c1, bool b_box) {
        if (EPI == EPI_PARTIAL && !b_box) {
          // the weight-streaming form reads each weight once per call: evict-first, so that the
          // stream does not push the split partials out of L2 before the fixup kernel reads them
          // (as dirty lines they would also be written back to HBM: ~8 µs of a decode step)
          tma_load_2d_hint(dst, map, smem_u32(full_bar + stage), c0, c1, evict_first);
          return;
        }
        if (kPairMma && rank == 1)
          tma_load_2d_pair(dst, map, full_pair0 + static_cast<uint32_t>(stage) * 8u, c0, c1);
        else if (MODE == kShareB && b_box)
          tma_load_2d_mc(dst, map, smem_u32(full_bar + stage), c0, c1, kBoth);
        else
          tma_load_2d(dst, map, smem_u32(full_bar + stage), c0, c1);
      };
      // the bytes a stage's full barrier waits for (kShareB: this CTA's A and all of B; pairs:
      // the even CTA's counts both CTAs' copies, the odd CTA's is not used)
      auto expect_stage = [&](int stage) {
        if (!kPairMma || rank == 0) mbar_expect_tx(smem_u32(full_bar + stage), kPairMma ? 2 * STAGE_TX : STAGE_TX);
      };
      auto load_a = [&](int stage, int kb, int mb) {
        int a_map, a_row;
        resolve_rows(p.amap, mb * BM, a_map, a_row);
        load_box(smem_u32(sA + stage * A_TILE_BYTES), &tm.m[p.a_map0 + a_map], stage, kb * BK, a_row, false);
      };
      // this CTA's B rows of tile nb: all of them, or its half in a pair
      auto load_b = [&](int stage, int kb, int nb) {
        const int row0 = nb * BN + (kPairMma ? rank * B_ROWS : 0);
        if constexpr (EPI == EPI_QKV && BN % 128 != 0) {
          int m0, r0, m1, r1;
          resolve_rows(p.bmap, row0, m0, r0);
          resolve_rows(p.bmap, row0 + B_ROWS - 1, m1, r1);
          if (m0 != m1) {   // the rows cross a boundary between two of the matrices: 32-row boxes
            for (int bx = MODE == kShareB ? rank : 0; bx < B_ROWS / 32; bx += CM) {
              int b_map, b_row;
              resolve_rows(p.bmap, row0 + bx * 32, b_map, b_row);
              load_box(smem_u32(sB + stage * B_TILE_BYTES + bx * 32 * 128), &tm.m[p.b32_map0 + b_map], stage,
                       kb * BK, b_row, true);
            }
            return;
          }
        }
#pragma unroll
        for (int bx = 0; bx < B_BOXES; ++bx) {
          if (MODE == kShareB && bx % 2 != rank) continue;   // the other CTA loads this box for both
          // (this thread's issue latency bounds the ring's lead over TMA latency: no divisions)
          int b_map, b_row;
          if constexpr (EPI == EPI_SWIGLU) {   // tile nb = [gate rows BN/2*nb.. | the same up rows]
            b_map = kPairMma ? rank : bx;
            b_row = nb * B_BOX_ROWS;
          } else {
            resolve_rows(p.bmap, row0 + bx * B_BOX_ROWS, b_map, b_row);
          }
          load_box(smem_u32(sB + stage * B_TILE_BYTES + bx * B_BOX_ROWS * 128), &tm.m[p.b_map0 + b_map], stage,
                   kb * BK, b_row, true);
        }
      };
      // the first STAGES k-blocks' weight tiles go out before the dependency wait: the ring
      // starts empty, so these stages need no empty-barrier wait
      int pre = 0;
      if (lane == 0 && p.weight_first != 0) {
        for (int u = unit0; u < num_units && pre < STAGES; u += unit_step) {
          int mb, nb, split;
          unit_coords<CM>(p, u, rank, mb, nb, split);
          const int kb0 = split * p.kb_per_split;
          const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
          for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
            expect_stage(pre);
            if (p.weight_first == 1) load_a(pre, kb, mb);
            else load_b(pre, kb, nb);
          }
        }
      }
      if (lane == 0) pdl_wait();
      __syncwarp();
      if (prologue) run_prologue();
      if (lane == 0) {
        bool ok = true;
        if (prologue) {
          // every warp of the grid has written its rows of A
          ok = wait_count(p.pro_count, (NUM_THREADS / 32) * static_cast<int>(gridDim.x), p.status, abort_flag);
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        int stage = 0, step = 0;
        uint32_t phase = 0;
        uint32_t used_mask = 0, last_parity = 0;
        for (int u = unit0; u < num_units && ok; u += unit_step) {
          int mb, nb, split;
          unit_coords<CM>(p, u, rank, mb, nb, split);
          const int kb0 = split * p.kb_per_split;
          const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
          for (int kb = kb0; kb < kb1; ++kb, ++step) {
            if (step < pre) {   // the weight half of this stage is already on its way
              if (p.weight_first == 1) load_b(stage, kb, nb);
              else load_a(stage, kb, mb);
            } else {
              if (!mbar_wait(smem_u32(empty_bar + stage), phase ^ 1u, p.status, abort_flag)) { ok = false; break; }
              expect_stage(stage);
              load_a(stage, kb, mb);
              load_b(stage, kb, nb);
            }
            used_mask |= 1u << stage;
            last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if constexpr (CM > 1) {
          // every stage's last fill released by both CTAs' products: no commit of the other
          // CTA is still on its way to this CTA's barriers when it leaves
          for (int i = 0; i < STAGES && ok; ++i) {
            if (!mbar_wait(smem_u32(empty_bar + stage), phase ^ 1u, p.status, abort_flag)) ok = false;
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
        if (!ok && !(kPairMma && rank == 1)) {
          // leave no copy in flight: wait (bounded) for the last load into every stage used (in
          // a pair the even CTA's full barriers count the odd CTA's copies too, and the cluster
          // barrier at the end keeps the odd CTA until then)
          for (int s = 0; s < STAGES; ++s)
            if (used_mask & (1u << s))
              mbar_wait_slow(smem_u32(full_bar + s), (last_parity >> s) & 1u, nullptr, nullptr, kWaitBudgetNs);
        }
      }
    }
  } else if (warp == 1 && kPairMma && rank == 1) {
    // the odd CTA of a pair: its products are issued by the even CTA
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issuer
    // The whole warp walks the loop (operands stay warp-uniform) and one elected lane issues
    // each product and commit: issued from a single diverged lane a product costs about half
    // of what a 128 x 256 x 16 product runs, leaving little time for the waits between stages.
    const uint64_t dA = sdesc_sw128(smem_u32(sA), 16, 1024);
    const uint64_t dB = sdesc_sw128(smem_u32(sB), 16, 1024);
    // remote = the barrier also receives arrivals from the other CTA of the pair (the wait
    // acquires at cluster scope)
    auto wait_all = [&](uint64_t* bar, uint32_t parity, bool remote = false) {
      const bool r = kPairMma && remote ? mbar_wait<true>(smem_u32(bar), parity, p.status, abort_flag)
                                      : mbar_wait(smem_u32(bar), parity, p.status, abort_flag);
      return __all_sync(0xffffffffu, r) != 0;
    };
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    bool issued = false;
    for (int u = unit0; u < num_units && ok; u += unit_step) {
      int mb, nb, split;
      unit_coords<CM>(p, u, rank, mb, nb, split);
      const int kb0 = split * p.kb_per_split;
      const int kb1 = min(kb0 + p.kb_per_split, p.num_kb);
      if (!wait_all(tempty_bar + acc, acc_phase ^ 1u, true)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_all(full_bar + stage, phase, true)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = dA + static_cast<uint64_t>((stage * A_TILE_BYTES) >> 4);
        const uint64_t bd = dB + static_cast<uint64_t>((stage * B_TILE_BYTES) >> 4);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {   // 16 K elements = 32 bytes further along the row
          if constexpr (kPairMma)
            tc_mma2_bf16_warp(d_tmem, ad + 2 * k, bd + 2 * k, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
          else
            tc_mma_bf16_warp(d_tmem, ad + 2 * k, bd + 2 * k, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
        }
        issued = true;
        if constexpr (kPairMma)
          tc_commit2_mc_warp(smem_u32(empty_bar + stage), kBoth);   // both CTAs' stage is free
        else if constexpr (MODE == kShareB)
          tc_commit_mc_warp(smem_u32(empty_bar + stage), kBoth);    // both CTAs' copy of B read
        else
          tc_commit_warp(smem_u32(empty_bar + stage));
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if constexpr (kPairMma)
        tc_commit2_mc_warp(smem_u32(tfull_bar + acc), kBoth);   // both CTAs' rows are done
      else
        tc_commit_warp(smem_u32(tfull_bar + acc));
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (!ok && issued) {
      // all products of the issuing lane must finish before the TMEM is released
      if constexpr (kPairMma)
        tc_commit2_mc_warp(smem_u32(drain_bar), 1);
      else
        tc_commit_warp(smem_u32(drain_bar));
      if (lane == 0) mbar_wait_slow(smem_u32(drain_bar), 0, nullptr, nullptr, kWaitBudgetNs);
      __syncwarp();
    }
  } else {
    // -------------------------------------------------------------- epilogue warps 2..5
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = unit0; u < num_units; u += unit_step) {
      int mb, nb, split;
      unit_coords<CM>(p, u, rank, mb, nb, split);
      if (!mbar_wait(smem_u32(tfull_bar + acc), acc_phase, p.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t t_acc = tmem_base + t_lane + static_cast<uint32_t>(acc * ACC_COLS);
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
              }
              store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + m * p.ldo + n0, v, valid);
            }
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        // columns [0, BN/2) of the tile are gate rows BN/2*nb.., [BN/2, BN) the matching up rows
        constexpr int HALF = BN / 2;
        static_assert(HALF % 8 == 0, "gate/up halves of whole 8-column chunks");
        if constexpr (HALF % 32 != 0) {
          // 120-column halves (240-column tiles): 8 columns at a time, the up half starting at
          // column 120 of the accumulator
#pragma unroll 1
          for (int c = 0; c < HALF / 8; ++c) {
            uint32_t g8[8], u8[8];
            tmem_ld8(t_acc + c * 8, g8);
            tmem_ld8(t_acc + HALF + c * 8, u8);
            const int n0 = nb * HALF + c * 8;
            const int valid = min(8, p.N - n0);
            if (m < p.M && valid > 0) {
              float w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = silu_f(__uint_as_float(g8[i])) * __uint_as_float(u8[i]);
              __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + m * p.ldo + n0;
              if (valid == 8 && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                uint4 w;
                w.x = pack_bf16(w8[0], w8[1]);
                w.y = pack_bf16(w8[2], w8[3]);
                w.z = pack_bf16(w8[4], w8[5]);
                w.w = pack_bf16(w8[6], w8[7]);
                *reinterpret_cast<uint4*>(dst) = w;
              } else {
                for (int i = 0; i < valid; ++i) dst[i] = __float2bfloat16_rn(w8[i]);
              }
            }
          }
        }
#pragma unroll 1
        for (int c = 0; c < (HALF % 32 == 0 ? HALF / 32 : 0); ++c) {
          uint32_t u[32];
          tmem_ld32(t_acc + c * 32, r);
          tmem_ld32(t_acc + HALF + c * 32, u);
          const int n0 = nb * HALF + c * 32;
          const int valid = min(32, p.N - n0);
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
            // this chunk's angles came one rope chunk ahead; the next rope chunk is the second
            // quarter of this head or the first of the next head (the tile is head-aligned)
            float cs_c[32], sn_c[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              cs_c[i] = cs_n[i];
              sn_c[i] = sn_n[i];
            }
            load_angles(j0 + 32 < half_d ? c + 1 : c + 3);
            uint32_t r2[32];
            tmem_ld32(t_acc + c * 32, r);
            tmem_ld32(t_acc + c * 32 + half_d, r2);
            if (!keep) continue;
            float w2[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float x1 = __uint_as_float(r[i]), x2 = __uint_as_float(r2[i]);
              v[i] = x1 * cs_c[i] - x2 * sn_c[i];
              w2[i] = x2 * cs_c[i] + x1 * sn_c[i];
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
      if (lane == 0) {
        if constexpr (kPairMma)
          mbar_arrive_cluster(cluster_map(smem_u32(tempty_bar + acc), 0));   // the even CTA's
        else
          mbar_arrive(smem_u32(tempty_bar + acc));
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
  }

  tc_fence_before();
  if constexpr (CM > 1)
    cluster_sync();   // no CTA leaves while the other may still write its shared memory
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if constexpr (kPairMma)
      tmem_dealloc2(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int BN, int EPI, int STAGES, int MODE>
constexpr size_t smem_bytes() {
  return 1024 + STAGES * (A_TILE_BYTES + (MODE == kPair ? BN / 2 : BN) * BK * 2) + (2 * STAGES + 5) * 8 + 16;
}

template <int BN, int EPI, int STAGES, int MODE = kSingle>
int launch(const Ctx& c, const TMaps& tm, Params p) {
  constexpr int CM = MODE == kSingle ? 1 : 2;
  auto kern = gemm_tc_kernel<BN, EPI, STAGES, MODE>;
  constexpr size_t smem = smem_bytes<BN, EPI, STAGES, MODE>();
  static_assert(smem <= 227 * 1024, "shared memory per CTA");
  static_assert(smem >= kTmemKernelMinSmem, "a TMEM-holding kernel must not share an SM with another");
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;   // clusters of CM CTAs that can be resident at once
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (attr_err == cudaSuccess && CM > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(c.num_sms / CM * CM);
      cfg.blockDim = dim3(NUM_THREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CM;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
      if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
    }
  });
  if (attr_err != cudaSuccess) return LLAMA_ERR_CUDA;
  p.status = c.status;
  if (!c.static_weights) p.weight_first = 0;
  if (p.num_mb % CM != 0 || (CM > 1 && p.num_splits != 1)) return LLAMA_ERR_INVALID_ARG;
  const int units = p.num_mb / CM * p.num_nb * p.num_splits;
  if (units == 0) return LLAMA_OK;
  if (p.pro_out != nullptr && (EPI == EPI_RESID || EPI == EPI_PARTIAL || p.pro_x == nullptr ||
                              p.pro_gamma == nullptr || p.pro_count == nullptr))
    return LLAMA_ERR_INVALID_ARG;
  if constexpr (CM == 1) {
    launch_pdl(c, kern, dim3(std::min(units, c.num_sms)), dim3(NUM_THREADS), smem, tm, p);
  } else {
    const int clusters = std::min(units, std::min(max_clusters, c.num_sms / CM));
    launch_pdl_cluster(c, kern, dim3(clusters * CM), dim3(NUM_THREADS), smem, CM, tm, p);
  }
  return after_launch(c);
}

// Clusters of two CTAs on consecutive row blocks, where the row blocks pair up.
bool use_clusters(int M) { return (M + BM - 1) / BM % 2 == 0; }

// Clusters where the row blocks pair up: two-SM products at 256 columns (their rings hold
// half of each B tile per stage, so 6 stages), multicast clusters at 224.
template <int BN, int EPI, int STAGES>
int launch_cl(const Ctx& c, const TMaps& tm, const Params& p, bool clusters) {
  if (!clusters) return launch<BN, EPI, STAGES, kSingle>(c, tm, p);
  if constexpr (BN == 256)
    return launch<BN, EPI, 6, kPair>(c, tm, p);
  else
    return launch<BN, EPI, STAGES, kShareB>(c, tm, p);
}

// Rows of the weight boxes: 128, or the whole tile width (BN < 256), halved in clusters.
uint32_t weight_box_rows(int bn, bool clusters) { return bn == 256 ? 128u : clusters ? bn / 2 : bn; }

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

// Gate/up tile width in two-SM pairs: 240 (120 gate + 120 up columns) when its rounds of pair
// units are at least 3 % narrower in total than those of 256-column tiles, else 256.
int swiglu_pair_width(int M, int I, int num_sms) {
  const long long pairs_m = (M + BM - 1) / BM / 2, clusters = std::max(1, num_sms / 2);
  auto cost = [&](int half) {
    const long long units = pairs_m * ((I + half - 1) / half);
    return (units + clusters - 1) / clusters * (2 * half);
  };
  return cost(120) * 100 <= cost(128) * 97 ? 240 : 256;
}

// RMSNorm in the prologue: A (the tensor map at a_map0) is built on n.xn, which the prologue
// fills with RMSNorm(X).
void set_prologue(Params& p, const void* X, const NormPro& n) {
  p.pro_x = static_cast<const __nv_bfloat16*>(X);
  p.pro_gamma = static_cast<const __nv_bfloat16*>(n.gamma);
  p.pro_out = static_cast<__nv_bfloat16*>(n.xn);
  p.pro_inv_k = 1.0f / static_cast<float>(p.K);
  p.pro_eps = n.eps;
  p.pro_count = n.count;
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
               const NormPro* norm) {
  const int bn = tile_width_for(M, N, c.num_sms);
  const bool cl = use_clusters(M);
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], norm ? norm->xn : X, K, M, K, 128) ||
      !make_tmap_2d(&tm.m[1], W, K, N, K, weight_box_rows(bn, cl)))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, N, K, bn);
  if (norm != nullptr) set_prologue(p, X, *norm);
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.out = C;
  p.ldo = N;
  if (bn == 256) return c_f32 ? launch_cl<256, EPI_F32, 4>(c, tm, p, cl) : launch_cl<256, EPI_BF16, 4>(c, tm, p, cl);
  return c_f32 ? launch_cl<224, EPI_F32, 5>(c, tm, p, cl) : launch_cl<224, EPI_BF16, 5>(c, tm, p, cl);
}

int gemm_residual(const Ctx& c, const void* X, const void* W, const void* resid, void* out, int M, int N, int K) {
  // 224-column tiles when they finish in fewer tile-column rounds (e.g. N = 4096 at M = 2048:
  // 304 tiles fill 2 rounds of 152 SMs, where 256 tiles of 256 columns leave the second
  // round two-thirds full)
  const int bn = tile_width_for(M, N, c.num_sms);
  const bool cl = use_clusters(M);
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], W, K, N, K, weight_box_rows(bn, cl)))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, N, K, bn);
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.out = out;
  p.ldo = N;
  p.resid = static_cast<const __nv_bfloat16*>(resid);
  p.ldr = N;
  return bn == 256 ? launch_cl<256, EPI_RESID, 4>(c, tm, p, cl) : launch_cl<224, EPI_RESID, 5>(c, tm, p, cl);
}

int gemm_swiglu(const Ctx& c, const void* X, const void* Wg, const void* Wu, void* out, int M, int I, int K,
                const NormPro* norm) {
  // kernel N runs over tiles of `half` gate rows + the same `half` up rows: 256 columns, or in
  // two-SM pairs 240 when that saves at least 3 % of the rounds' width (I = 11008, M = 2048: 10
  // rounds of 736 pair units at 240 against 10 of 688 at 256, the last one nearly empty;
  // measured 217.9-218.1 against 218.6-220.4 us).  Without pairs 240-column tiles ran slower
  // (each CTA then takes all 240 weight rows per k-block).
  const bool cl = use_clusters(M);
  const int bn = cl && swiglu_pair_width(M, I, c.num_sms) == 240 ? 240 : 256;
  const int half = bn / 2;
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], norm ? norm->xn : X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], Wg, K, I, K, half) ||
      !make_tmap_2d(&tm.m[2], Wu, K, I, K, half))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, 2 * ((I + half - 1) / half) * half, K, bn);
  if (norm != nullptr) set_prologue(p, X, *norm);
  p.N = I;   // output width (used by the epilogue's bounds)
  p.a_map0 = 0;
  p.b_map0 = 1;
  p.n_maps = 3;
  p.out = out;
  p.ldo = I;
  if (bn == 240) return launch<240, EPI_SWIGLU, 7, kPair>(c, tm, p);
  return launch_cl<256, EPI_SWIGLU, 4>(c, tm, p, cl);
}

int gemm_qkv_rope(const Ctx& c, const void* X, const void* Wq, const void* Wk, const void* Wv, int B, int S, int K,
                  int H, int G, int D, const float* cos, const float* sin, void* q_out, void* k_cache,
                  void* v_cache, int T_max, int rope_half, const int32_t* start, const int32_t* lens,
                  int max_pos, const NormPro* norm) {
  const int M = B * S;
  // 224-column tiles when they fill the SM-count rounds better (the half-split pairs (j, j+64)
  // need whole heads in a tile: 256 columns = two heads); a 224-column tile that crosses the
  // q|k or k|v boundary takes its weights in 32-row boxes from the maps at b32_map0
  const int bn = rope_half ? 256 : tile_width_for(M, (H + 2 * G) * D, c.num_sms);
  const bool cl = use_clusters(M);
  const uint32_t box = weight_box_rows(bn, cl);
  TMaps tm{};
  if (!make_tmap_2d(&tm.m[0], norm ? norm->xn : X, K, M, K, 128) || !make_tmap_2d(&tm.m[1], Wq, K, H * D, K, box) ||
      !make_tmap_2d(&tm.m[2], Wk, K, G * D, K, box) || !make_tmap_2d(&tm.m[3], Wv, K, G * D, K, box))
    return LLAMA_ERR_INVALID_ARG;
  if (bn != 256 && (!make_tmap_2d(&tm.m[4], Wq, K, H * D, K, 32) || !make_tmap_2d(&tm.m[5], Wk, K, G * D, K, 32) ||
                    !make_tmap_2d(&tm.m[6], Wv, K, G * D, K, 32)))
    return LLAMA_ERR_INVALID_ARG;
  Params p = base_params(M, (H + 2 * G) * D, K, bn);
  if (norm != nullptr) set_prologue(p, X, *norm);
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
  return bn == 256 ? launch_cl<256, EPI_QKV, 4>(c, tm, p, cl) : launch_cl<224, EPI_QKV, 5>(c, tm, p, cl);
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
