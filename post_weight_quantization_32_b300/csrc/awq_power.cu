// The layer's output power mean((X W^T)^2) on the tensor cores ("AWQ
// (activation-aware weight quantization)", "What the simulations show": the
// relative output error divides ||X W^T - X Wq^T||^2 by ||X W^T||^2; the
// notebook's "Output MSE vs bit width" reports the same ratio).
//
// The product is never stored: each tile of 128 W rows against a tile of
// tokens of X is accumulated in tensor memory and the epilogue squares the
// accumulator and sums it.  The plain GEMM route (product written as
// float32, then squared) moved 4 MB out and back and left most SMs idle on
// short layers; here the only traffic is W and X.  Two forms:
//   power_split_kernel    layers with few 128 x 128 tiles: the two (or four)
//                         CTAs of a cluster share a tile, each over a share
//                         of K, and add their partial products over
//                         distributed shared memory before squaring; a
//                         one-CTA launch adds the CTAs' float64 partials in
//                         order.
//   power_mma_kernel      the others: persistent CTAs over (128-row, 32- to
//                         256-token) units, two alternating accumulators, the
//                         units' partials added in unit order by the last CTA.
//
// Roles (192 threads) in both:
//   warp 0       tensor memory owner and TMA loader: W blocks (128 rows x 64
//                columns) and X blocks (tokens x 64 columns), 128-byte
//                swizzled, into a ring of stages
//   warp 1       tcgen05.mma issuer (kind::f16, M = 128, N = the token tile,
//                K = 16), both operands from shared memory
//   warps 2..5   epilogue: thread = row; each warp reads the tensor-memory
//                lane quarter it may access and squares and sums its row
//                (float32 over 16 columns, float64 across them); the four
//                warps add their sums in a fixed order.
// The loader and MMA warps run their loops as whole warps, the elected lane
// issuing, and count their ring positions (no division in a loop).  Every
// summation order is fixed, so repeated calls give identical results.
// Rows past `out`, tokens past N and columns past `in` are read by TMA as
// zeros and add nothing.  Every wait is bounded; a timeout sets the status
// word to AWQ_ERR_TIMEOUT.
#include <algorithm>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kPThreads = 192;
constexpr int kPRows = 128;
constexpr int kPKB = 64;                        // K columns per block
constexpr uint32_t kPWTile = kPRows * kPKB * 2;  // 16 KB
constexpr int kPMaxStages = 8;
constexpr uint32_t kPCtrl = 1024;
constexpr uint32_t kPRingBudget = 200u * 1024u;

// Per token tile NT: K blocks a ring stage holds (two, so one wait, fence
// and commit serve eight MMAs; one for the widest tile), the stage's bytes
// and the number of stages.
template <int NT> struct PowTile {
  static constexpr int kKps = NT == 256 ? 1 : 2;
  static constexpr uint32_t kXTile = (uint32_t)NT * 128u;
  static constexpr uint32_t kStage = (uint32_t)kKps * (kPWTile + kXTile);
  static constexpr int kStages =
      (int)(kPRingBudget / kStage) < kPMaxStages ? (int)(kPRingBudget / kStage) : kPMaxStages;
  static constexpr uint32_t kTmemCols = 2u * NT < 32u ? 32u : 2u * NT;  // two accumulators
  static constexpr size_t kSmem = kPCtrl + 1024 + (size_t)kStages * kStage;
};

struct PowCtrl {
  uint64_t full[kPMaxStages], empty[kPMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int last;
  double red[4];
};
static_assert(sizeof(PowCtrl) <= kPCtrl, "control block too large");

struct PowArgs {
  int n_tt;         // token tiles
  int n_units;      // row tiles x token tiles
  int n_st;         // ring stages a unit (K blocks / K blocks a stage, rounded up)
  double denom;     // N * out
  double* partials; // [n_units]
  uint32_t* ticket; // zeroed before the launch
  uint32_t* diag;   // four words of wait diagnostics
  double* power;
  int32_t* status;
  uint64_t wait_limit_ns;
};

// One stage's copies: expect the bytes on bar, then W and X blocks at K
// column x (and, for two blocks a stage, x + 64).
__device__ __forceinline__ void tma_stage_elect(uint32_t bar, uint32_t bytes, uint32_t w_dst,
                                                uint32_t x_dst, const CUtensorMap* mw,
                                                const CUtensorMap* mx, int32_t x, int32_t wrow,
                                                int32_t xrow) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%2], [%4, {%6, %7}], [%0];\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%3], [%5, {%6, %8}], [%0];\n\t}" ::"r"(bar),
      "r"(bytes), "r"(w_dst), "r"(x_dst), "l"(reinterpret_cast<uint64_t>(mw)),
      "l"(reinterpret_cast<uint64_t>(mx)), "r"(x), "r"(wrow), "r"(xrow)
      : "memory");
}
__device__ __forceinline__ void tma_pair_elect(uint32_t w_dst, uint32_t x_dst, uint32_t bar,
                                               const CUtensorMap* mw, const CUtensorMap* mx,
                                               int32_t x, int32_t wrow, int32_t xrow) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%3, {%5, %6}], [%2];\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%1], [%4, {%5, %7}], [%2];\n\t}" ::"r"(w_dst),
      "r"(x_dst), "r"(bar), "l"(reinterpret_cast<uint64_t>(mw)),
      "l"(reinterpret_cast<uint64_t>(mx)), "r"(x), "r"(wrow), "r"(xrow)
      : "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: arrive with release semantics,
// then wait with acquire semantics (shared-memory writes before it are
// visible to the whole cluster after it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}
// The address in CTA `rank`'s shared memory that corresponds to this CTA's
// shared-memory address `a`.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_shared_cluster_f32x4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// Barrier 1 over the four epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Barrier 1 over the four epilogue warps that also ANDs v over them, so all
// four take the same branch.
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// kind::f16 instruction descriptor: float32 accumulator, A and B both fp16
// (format 0) or both bf16 (format 1), K-major, N >> 3 at [17,23), M >> 4 at
// [24,29).
__host__ __device__ constexpr uint32_t idesc_16bit(uint32_t M, uint32_t N, bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

template <bool BF16, int NT>
__global__ void __launch_bounds__(kPThreads, 1)
    power_mma_kernel(const __grid_constant__ CUtensorMap tmW,
                     const __grid_constant__ CUtensorMap tmX, const PowArgs p) {
  using Tile = PowTile<NT>;
  constexpr int KPS = Tile::kKps;
  constexpr uint32_t S = (uint32_t)Tile::kStages;
  extern __shared__ uint8_t psmem_raw[];
  const uint32_t raw = smem_addr(psmem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  PowCtrl& c = *reinterpret_cast<PowCtrl*>(psmem_raw + (base - raw));
  // stage layout: KPS W blocks (16 KB each), then KPS X blocks (NT x 128 B
  // each); every block starts on a 1024-byte boundary
  const uint32_t ring = base + kPCtrl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(smem_addr(&c.full[i]), 1);
      mbar_init(smem_addr(&c.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&c.acc_full[i]), 1);
      mbar_init(smem_addr(&c.acc_empty[i]), 4);
    }
    mbar_init(smem_addr(&c.drain), 1);
    c.abort = 0;
    c.last = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&c.tmem_base), Tile::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // W and X may come from earlier kernels; the ticket from the memset
  const uint32_t tmem = c.tmem_base;
  volatile int* abort = &c.abort;
  const uint64_t lim = p.wait_limit_ns;
  const int n_units = p.n_units, n_tt = p.n_tt, n_st = p.n_st;

  if (warp == 0) {
    // -------------------------------------------------------------- loader
    uint32_t q = 0, st = 0, ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const int rt = u / n_tt, tt = u - (u / n_tt) * n_tt;
      for (int ks = 0; ks < n_st; ++ks) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.empty[st]), ph ^ 1, abort, lim,
                                               p.diag, 41, q));
        if (!ok) break;
        const uint32_t dst = ring + st * Tile::kStage;
        const uint32_t bar = smem_addr(&c.full[st]);
        tma_stage_elect(bar, Tile::kStage, dst, dst + KPS * kPWTile, &tmW, &tmX, ks * KPS * kPKB,
                        rt * kPRows, tt * NT);
        if (KPS == 2)
          tma_pair_elect(dst + kPWTile, dst + 2 * kPWTile + Tile::kXTile, bar, &tmW, &tmX,
                         (ks * KPS + 1) * kPKB, rt * kPRows, tt * NT);
        ++q;
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
      }
    }
    int never_set = 0;  // drain the copies still in flight
    for (uint32_t m = q > S ? q - S : 0; m < q; ++m)
      mbar_wait(smem_addr(&c.full[m % S]), (m / S) & 1, &never_set, lim);
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_16bit(kPRows, (uint32_t)NT, BF16);
    uint32_t q = 0, j = 0, st = 0, ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const uint32_t acc = j & 1;
      if (j >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.acc_empty[acc]), ((j - 2) / 2) & 1,
                                               abort, lim, p.diag, 42, j));
      if (!ok) break;
      tc_fence_after();
      const uint32_t d_t = tmem + acc * (Tile::kTmemCols / 2);
      for (int ks = 0; ks < n_st; ++ks) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(smem_addr(&c.full[st]), ph, abort, lim, p.diag, 43, q));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sb = ring + st * Tile::kStage;
#pragma unroll
        for (int b = 0; b < KPS; ++b) {
          const uint64_t adesc = smem_desc_sw128(sb + b * kPWTile);
          const uint64_t bdesc = smem_desc_sw128(sb + KPS * kPWTile + b * Tile::kXTile);
#pragma unroll
          for (int k = 0; k < kPKB / 16; ++k)  // 16 columns = 32 bytes = 2 in the address field
            umma_ss_elect(d_t, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                          (ks | b | k) != 0 ? 1u : 0u);
        }
        umma_commit_elect(smem_addr(&c.empty[st]));
        ++q;
        if (++st == S) {
          st = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      umma_commit_elect(smem_addr(&c.acc_full[acc]));
      ++j;
    }
    umma_commit_elect(smem_addr(&c.drain));
    int never_set = 0;
    mbar_wait(smem_addr(&c.drain), 0, &never_set, lim);
  } else {
    // ------------------------------------------------------------ epilogue
    const int qd = warp & 3;  // the tensor-memory lane quarter this warp may access
    const int e = warp - 2;   // position in the fixed order of the warps' sums
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    uint32_t j = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      const uint32_t acc = j & 1;
      const bool ok = mbar_wait(smem_addr(&c.acc_full[acc]), (j / 2) & 1, abort, lim, p.diag, 44,
                                j);
      if (!epi_all(ok)) break;
      tc_fence_after();
      double rs = 0.0;
      const uint32_t cb = tmem + lane_addr + acc * (Tile::kTmemCols / 2);
#pragma unroll
      for (int cc = 0; cc < NT; cc += 16) {
        uint32_t v[16];
        tmem_ld16(cb + (uint32_t)cc, v);
        tmem_wait_ld();
        float s16 = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x = __uint_as_float(v[i]);
          s16 = fmaf(x, x, s16);
        }
        rs += (double)s16;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&c.acc_empty[acc]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
      if (lane == 0) c.red[e] = rs;
      epi_sync();
      if (e == 0 && lane == 0) p.partials[u] = ((c.red[0] + c.red[1]) + c.red[2]) + c.red[3];
      epi_sync();
      ++j;
    }
    // the last CTA to finish adds the units' partials in unit order
    if (e == 0 && lane == 0) {
      __threadfence();
      c.last = atomicAdd(p.ticket, 1u) == gridDim.x - 1 ? 1 : 0;
    }
    epi_sync();
    if (c.last) {
      __threadfence();
      const int t = e * 32 + lane;
      double sum = 0.0;
      for (int i = t; i < n_units; i += 128) sum += __ldcg(p.partials + i);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane == 0) c.red[e] = sum;
      epi_sync();
      if (t == 0) *p.power = (((c.red[0] + c.red[1]) + c.red[2]) + c.red[3]) / p.denom;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Tile::kTmemCols);
  }
  if (threadIdx.x == 0 && c.abort) set_status(p.status, ST_TIMEOUT);
}

// ---- split-K form, for layers with few 128 x NT tiles ---------------------
// The KS CTAs of a cluster share one tile (128 W rows x NT tokens, NT = 128):
// CTA r accumulates K blocks [r n_kb / KS, (r + 1) n_kb / KS) in tensor
// memory and stages its float32 accumulator in its own shared memory (over
// the drained ring) as [NT / 4][128 rows][4 tokens], so that a row's four
// consecutive tokens are one 16-byte vector and a warp's vectors are
// contiguous.  After a cluster barrier CTA r forms, for tokens
// [r NT / KS, (r + 1) NT / KS), the sum of the KS partial products in rank
// order, squares it and sums its rows; every output entry is formed in one
// fixed order.  Each CTA writes one float64 partial and a one-CTA launch adds
// them in order.  A 128-token tile reads W from shared memory once per 128
// tokens, where 64-token tiles were bound by shared-memory bandwidth (each
// 64-column block written by TMA and read by the MMA).
struct SplitArgs {
  int n_kb;          // K blocks of the layer
  int n_tt;          // token tiles
  double* partials;  // [grid]
  uint32_t* diag;
  int32_t* status;
  uint64_t wait_limit_ns;
};

template <int NT> struct SplitTile {
  static constexpr uint32_t kX = (uint32_t)NT * 128u;
  static constexpr uint32_t kStage = kPWTile + kX;
  static constexpr int kStages =
      (int)(kPRingBudget / kStage) < kPMaxStages ? (int)(kPRingBudget / kStage) : kPMaxStages;
  static constexpr size_t kSmem = kPCtrl + 1024 + (size_t)kStages * kStage;
  static_assert((size_t)NT * 128 * 4 <= (size_t)kStages * kStage, "staging must fit the ring");
};

template <bool BF16, int NT, int KS>
__global__ void __launch_bounds__(kPThreads, 1)
    power_split_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX, const SplitArgs p) {
  using Tile = SplitTile<NT>;
  constexpr uint32_t S = (uint32_t)Tile::kStages;
  extern __shared__ uint8_t psmem_raw[];
  const uint32_t raw = smem_addr(psmem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  PowCtrl& c = *reinterpret_cast<PowCtrl*>(psmem_raw + (base - raw));
  const uint32_t ring = base + kPCtrl;
  float* staged = reinterpret_cast<float*>(psmem_raw + (base - raw) + kPCtrl);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int tile = blockIdx.x / KS;
  const int rt = tile / p.n_tt, tt = tile - (tile / p.n_tt) * p.n_tt;
  const int kb0 = (int)((int64_t)rank * p.n_kb / KS);
  const int kb1 = (int)((int64_t)(rank + 1) * p.n_kb / KS);
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(smem_addr(&c.full[i]), 1);
      mbar_init(smem_addr(&c.empty[i]), 1);
    }
    mbar_init(smem_addr(&c.acc_full[0]), 1);
    mbar_init(smem_addr(&c.drain), 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(&c.tmem_base), NT);
    tmem_relinquish();
  }
  if (warp == 1 && lane == 0) {
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // W and X may come from earlier kernels
  const uint32_t tmem = c.tmem_base;
  volatile int* abort = &c.abort;
  const uint64_t lim = p.wait_limit_ns;

  if (warp == 0) {
    // -------------------------------------------------------------- loader
    uint32_t q = 0, st = 0, ph = 0;
    for (int kb = kb0; kb < kb1; ++kb) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_addr(&c.empty[st]), ph ^ 1, abort, lim, p.diag,
                                             45, q)))
        break;
      const uint32_t dst = ring + st * Tile::kStage;
      tma_stage_elect(smem_addr(&c.full[st]), Tile::kStage, dst, dst + kPWTile, &tmW, &tmX,
                      kb * kPKB, rt * kPRows, tt * NT);
      ++q;
      if (++st == S) {
        st = 0;
        ph ^= 1;
      }
    }
    int never_set = 0;  // drain the copies still in flight
    for (uint32_t m = q > S ? q - S : 0; m < q; ++m)
      mbar_wait(smem_addr(&c.full[m % S]), (m / S) & 1, &never_set, lim);
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_16bit(kPRows, (uint32_t)NT, BF16);
    uint32_t q = 0, st = 0, ph = 0;
    bool ok = true;
    for (int kb = kb0; kb < kb1; ++kb) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(smem_addr(&c.full[st]), ph, abort, lim, p.diag, 46, q));
      if (!ok) break;
      tc_fence_after();
      const uint64_t adesc = smem_desc_sw128(ring + st * Tile::kStage);
      const uint64_t bdesc = smem_desc_sw128(ring + st * Tile::kStage + kPWTile);
#pragma unroll
      for (int k = 0; k < kPKB / 16; ++k)
        umma_ss_elect(tmem, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                      (kb > kb0 || k > 0) ? 1u : 0u);
      umma_commit_elect(smem_addr(&c.empty[st]));
      ++q;
      if (++st == S) {
        st = 0;
        ph ^= 1;
      }
    }
    if (ok) umma_commit_elect(smem_addr(&c.acc_full[0]));
    umma_commit_elect(smem_addr(&c.drain));
    int never_set = 0;
    mbar_wait(smem_addr(&c.drain), 0, &never_set, lim);
  } else {
    // ------------------------------------------- epilogue: stage the product
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(qd * 32) << 16;
    const bool ok = mbar_wait(smem_addr(&c.acc_full[0]), 0, abort, lim, p.diag, 47, 0);
    if (epi_all(ok)) {
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < NT; cc += 16) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_addr + (uint32_t)cc, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(staged + ((cc + i) / 4 * 128 + row) * 4) =
              make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]),
                          __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
      }
      tc_fence_before();
    }
  }
  cluster_sync_all();  // every CTA's partial product is staged
  if (warp >= 2) {
    // ------------------------ this CTA's token slice, summed over the cluster
    constexpr int SL = NT / KS;
    const int e = warp - 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t loc = smem_addr(staged) + (uint32_t)(((int)rank * SL / 4 * 128 + row) * 16);
    uint32_t src[KS];
#pragma unroll
    for (int r = 0; r < KS; ++r) src[r] = map_shared_rank(loc, (uint32_t)r);
    double rs = 0.0;
#pragma unroll 1
    for (int c0 = 0; c0 < SL; c0 += 16) {
      float4 v[4][KS];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int r = 0; r < KS; ++r)
          v[i][r] = ld_shared_cluster_f32x4(src[r] + (uint32_t)(((c0 / 4 + i) * 128) * 16));
      float s16 = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);  // the partial products in rank order
#pragma unroll
        for (int r = 0; r < KS; ++r) {
          t.x += v[i][r].x;
          t.y += v[i][r].y;
          t.z += v[i][r].z;
          t.w += v[i][r].w;
        }
        s16 = fmaf(t.x, t.x, s16);
        s16 = fmaf(t.y, t.y, s16);
        s16 = fmaf(t.z, t.z, s16);
        s16 = fmaf(t.w, t.w, s16);
      }
      rs += (double)s16;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, o);
    if (lane == 0) c.red[e] = rs;
    epi_sync();
    if (e == 0 && lane == 0)
      p.partials[blockIdx.x] = ((c.red[0] + c.red[1]) + c.red[2]) + c.red[3];
  }
  cluster_sync_all();  // the other CTAs are done reading this one's staging
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, NT);
  }
  if (threadIdx.x == 0 && c.abort) set_status(p.status, ST_TIMEOUT);
}

// power = (sum of the n partials in a fixed order) / denom; one CTA.
__global__ void __launch_bounds__(256) power_finish_kernel(const double* __restrict__ partials,
                                                           int n, double denom,
                                                           double* __restrict__ power) {
  pdl_wait();
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < n; i += 256) s += partials[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) *power = red[0] / denom;
}

// Tokens a tile: the largest of 256, 128 and 64 that still gives every SM a
// unit (fewer tokens a tile re-read W from L2 more often), halved while the
// tile would still hold all N tokens, down to 32.
int power_token_tile(int64_t out, int64_t N, int sms) {
  const int64_t n_rt = (out + kPRows - 1) / kPRows;
  int nt = 64;
  for (int cand : {256, 128}) {
    if (n_rt * ((N + cand - 1) / cand) >= sms) {
      nt = cand;
      break;
    }
  }
  while (nt > 32 && nt / 2 >= N) nt /= 2;
  return nt;
}

int64_t power_units(int64_t out, int64_t N, int nt) {
  return ((out + kPRows - 1) / kPRows) * ((N + nt - 1) / nt);
}

template <bool BF16, int NT>
cudaError_t launch_power_tile(const CUtensorMap& mw, const CUtensorMap& mx, const PowArgs& a,
                              int grid, cudaStream_t stream) {
  auto k = power_mma_kernel<BF16, NT>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)PowTile<NT>::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)grid), dim3(kPThreads), PowTile<NT>::kSmem, stream, mw, mx,
                    a);
}

template <bool BF16>
cudaError_t launch_power_dt(int nt, const CUtensorMap& mw, const CUtensorMap& mx,
                            const PowArgs& a, int grid, cudaStream_t stream) {
  switch (nt) {
    case 32: return launch_power_tile<BF16, 32>(mw, mx, a, grid, stream);
    case 64: return launch_power_tile<BF16, 64>(mw, mx, a, grid, stream);
    case 128: return launch_power_tile<BF16, 128>(mw, mx, a, grid, stream);
    case 256: return launch_power_tile<BF16, 256>(mw, mx, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Split-K plan: 128-token tiles (N > 64), four CTAs a tile where the layer
// would otherwise leave most SMs idle, else two, as long as that many CTAs
// still fit one a SM and each keeps at least four K blocks; ks = 0 leaves
// the layer to the persistent kernel.  Measured on the notebook-shaped layer
// (4096 x 4096, 256 tokens): 128-token tiles split two ways 23.6 us, 256-token
// tiles split four ways 25.6 us (the cluster reduction reads three remote
// slices instead of one), two ways 29.7 us.
constexpr int kSplitNT = 128;
void split_plan(int64_t out, int64_t in, int64_t N, int sms, int& nt, int& ks) {
  nt = 0;
  ks = 0;
  if (N <= 64) return;
  nt = kSplitNT;
  const int64_t tiles = ((out + kPRows - 1) / kPRows) * ((N + nt - 1) / nt);
  const int64_t n_kb = (in + kPKB - 1) / kPKB;
  if (tiles * 4 <= sms / 2 && n_kb >= 16)
    ks = 4;
  else if (tiles * 2 <= sms && n_kb >= 8)
    ks = 2;
}

template <bool BF16, int NT, int KS>
cudaError_t launch_split_tile(const CUtensorMap& mw, const CUtensorMap& mx, const SplitArgs& a,
                              int grid, cudaStream_t stream) {
  auto k = power_split_kernel<BF16, NT, KS>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SplitTile<NT>::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl_cluster(k, dim3((unsigned)grid), (unsigned)KS, dim3(kPThreads),
                            SplitTile<NT>::kSmem, stream, mw, mx, a);
}

template <bool BF16>
cudaError_t launch_split_dt(int ks, const CUtensorMap& mw, const CUtensorMap& mx,
                            const SplitArgs& a, int grid, cudaStream_t stream) {
  return ks == 4 ? launch_split_tile<BF16, kSplitNT, 4>(mw, mx, a, grid, stream)
                 : launch_split_tile<BF16, kSplitNT, 2>(mw, mx, a, grid, stream);
}

}  // namespace

bool power_mma_eligible(int dt, int64_t out, int64_t in, int64_t N, const void* W, const void* X) {
  return (dt == kDtF16 || dt == kDtBF16) && in % 8 == 0 && out < (1ll << 31) &&
         N < (1ll << 31) && in < (1ll << 31) && (reinterpret_cast<uintptr_t>(W) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(X) & 15) == 0;
}

size_t power_mma_workspace_bytes(int64_t out, int64_t N) {
  // the partials: one per unit of the persistent kernel (the smallest tile
  // gives the most), or one per CTA of the split form (at most four per
  // 128-token tile)
  return 256 + (size_t)(power_units(out, N, 32) + 4 * power_units(out, N, 128)) * 8;
}

cudaError_t launch_power_mma(const void* W, const void* X, int dt, int64_t out, int64_t in,
                             int64_t N, void* workspace, double* power, int32_t* dev_status,
                             cudaStream_t stream) {
  if (!power_mma_eligible(dt, out, in, N, W, X)) return cudaErrorInvalidValue;
  const int sms = device_sm_count();
  const CUtensorMapDataType t =
      dt == kDtF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  {
    int snt, ks;
    split_plan(out, in, N, sms, snt, ks);
    if (ks > 0) {
      CUtensorMap mw, mx;
      if (!tensor_map_sw128(&mw, t, W, (uint64_t)in, (uint64_t)out, (uint64_t)in * 2, kPKB,
                            kPRows) ||
          !tensor_map_sw128(&mx, t, X, (uint64_t)in, (uint64_t)N, (uint64_t)in * 2, kPKB,
                            (uint32_t)snt))
        return cudaErrorInvalidValue;
      SplitArgs a{};
      a.n_kb = (int)((in + kPKB - 1) / kPKB);
      a.n_tt = (int)((N + snt - 1) / snt);
      const int grid = (int)(((out + kPRows - 1) / kPRows) * a.n_tt * ks);
      // words 16..19 of the control area: wait diagnostics; partials from byte 256
      a.partials = reinterpret_cast<double*>(wsb + 256);
      a.diag = reinterpret_cast<uint32_t*>(wsb) + 16;
      a.status = dev_status;
      a.wait_limit_ns = 2000000000ull;
      cudaError_t e = dt == kDtF16 ? launch_split_dt<false>(ks, mw, mx, a, grid, stream)
                                   : launch_split_dt<true>(ks, mw, mx, a, grid, stream);
      if (e != cudaSuccess) return e;
      return launch_pdl(power_finish_kernel, 1, 256, 0, stream, a.partials, grid,
                        (double)N * (double)out, power);
    }
  }
  const int nt = power_token_tile(out, N, sms);
  const int64_t n_units = power_units(out, N, nt);
  if (n_units >= (1ll << 31)) return cudaErrorInvalidValue;
  // control area (256 bytes): the ticket at word 0, wait diagnostics at
  // words 16..19; the partials from byte 256
  cudaError_t e = cudaMemsetAsync(wsb, 0, 256, stream);
  if (e != cudaSuccess) return e;
  CUtensorMap mw, mx;
  if (!tensor_map_sw128(&mw, t, W, (uint64_t)in, (uint64_t)out, (uint64_t)in * 2, kPKB, kPRows) ||
      !tensor_map_sw128(&mx, t, X, (uint64_t)in, (uint64_t)N, (uint64_t)in * 2, kPKB,
                        (uint32_t)nt))
    return cudaErrorInvalidValue;
  PowArgs a{};
  a.n_tt = (int)((N + nt - 1) / nt);
  a.n_units = (int)n_units;
  const int64_t n_kb = (in + kPKB - 1) / kPKB;
  const int kps = nt == 256 ? 1 : 2;
  a.n_st = (int)((n_kb + kps - 1) / kps);  // an odd last block pairs with an all-zero one
  a.denom = (double)N * (double)out;
  a.partials = reinterpret_cast<double*>(wsb + 256);
  a.ticket = reinterpret_cast<uint32_t*>(wsb);
  a.diag = reinterpret_cast<uint32_t*>(wsb) + 16;
  a.power = power;
  a.status = dev_status;
  a.wait_limit_ns = 2000000000ull;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(n_units, sms));
  return dt == kDtF16 ? launch_power_dt<false>(nt, mw, mx, a, grid, stream)
                      : launch_power_dt<true>(nt, mw, mx, a, grid, stream);
}

}  // namespace awq
