// The fused alpha-grid search: for every alpha of the grid it forms
//     dW_alpha = Q(W * s_alpha) / s_alpha - W
// tile by tile and scores sum((X dW_alpha^T)^2) on the tensor cores, never
// materialising X W^T or the dequantized weights.  By linearity this is the
// pages' ((X @ Wq.T - X @ W.T) ** 2).sum() ("AWQ (activation-aware weight
// quantization)", "Source code"; "AWQ vs GPTQ ...", awq_scales).
//
// Work unit = (128-row tile of W, a group of up to 8 alphas, a token tile of
// T <= 256 tokens).  One persistent CTA per SM walks a static list of units.
// Warp roles inside a CTA (512 threads, four warpgroups):
//   warpgroup 0 (56 registers a thread after setmaxnreg):
//     warp 0    TMA loads of W blocks (128 rows x 64 columns) together with
//               the matching 64 columns of the s and 2^e/s tables of the
//               unit's alphas, into one ring stage
//     warp 1    TMA loads of X blocks (T tokens x 64 columns, fp16)
//     warp 2    tensor memory owner and the tcgen05.mma issuer
//     warp 3    idle
//   Warps 0-2 run their loops as whole warps, the lane elect.sync picks
//   issuing each copy, MMA and commit, and every role counts its ring
//   positions: a loop on one lane, or a division by a ring depth per
//   iteration, cost hundreds of cycles an iteration here.
//   warpgroups 1 and 2 (200 registers a thread): producers, thread = one W
//     row.  Per 128-column job (one quantization group for group 128) and
//     alpha, pass 1 forms t = w * s in registers and the group's range;
//     pass 2 rounds t to the group's grid and writes -dW (fp16; the sign
//     does not change the squared error) straight into tensor memory,
//     where the MMA reads it as operand A.  Warpgroup 1 takes the even jobs
//     of a unit, warpgroup 2 the odd ones, each with its own ring bank and
//     dW slots; they run on into the next unit while the last MMAs of a
//     unit drain.
//   warpgroup 3 (56 registers a thread): epilogue.  After a unit's last MMA
//     it reads the fp32 accumulators (128 rows x T tokens per alpha) back,
//     squares and sums them, and frees the accumulator for the next unit.
// Tensor memory (512 columns): columns [0, 256) hold a_per accumulators of
// T columns; columns [256, 512) are eight 32-column slots of dW (64 fp16
// values per row each), four per producer warpgroup.  X is the MMA's B
// operand from shared memory in the 128-byte-swizzle K-major layout that
// TMA writes.  With one bank per consumer, every barrier's phases are
// consumed in order by a single party, so a parity wait can never be a
// full phase ahead.
//
// The GEMM runs on fp16 operands (11-bit significands) with fp32
// accumulation.  X arrives as fp16 scaled by a power of two, and dW is
// scaled by a per-alpha power of two folded into the 1/s table, both chosen
// from max|X| and max|W| so every value lies in fp16's normal range; the
// float64 reduction divides the exact powers of two out again.
//
// Rounding.  The producer rounds t * (1/scale) with one fused multiply-add
// against 1.5 * 2^23 (round to nearest even).  Next to an exact
// half-integer this can differ from rounding the correctly rounded quotient;
// either neighbour is half a step away, so only the sign of that entry's
// error changes, far less than the fp16 rounding of dW moves the score.
// Where every scale of an alpha is a power of two (alpha = 0, flat salience)
// t / scale falls on exact half-integers of the 16-bit weight lattice often,
// so those alphas use the correctly rounded quotient.  The group step is
// the exact float32 max(m / L, 1e-8) (asymmetric: (hi - lo) / maxq) as in
// the final quantizer.  The code clamps of the quantizers never act in
// exact arithmetic (|t| / scale <= L, and for the asymmetric grid
// round(t / scale) + zero stays in [0, maxq] because the zero point is the
// rounded -lo / scale), so the dequantized value is scale * round(t / scale)
// for both quantizers and the zero point cancels.  The one exception is an
// exact tie: when -lo / scale is k + 1/2 with k odd, round-half-even gives
// zero = k + 1 and the top entry rounds to code maxq + 1, which the clamp
// pulls back.  Exact ties are common only where every scale is a power of
// two (the weights then stay on their 16-bit lattice), so the correctly
// rounded path, which those alphas take, keeps the asymmetric upper clamp;
// elsewhere a tie needs an exact coincidence of products, and a near-tie
// only flips the sign of one half-step error.
//
// Every wait on an mbarrier is bounded (wall clock).  A wait that runs out
// raises a shared abort flag; all roles then stop issuing work, drain what
// they have in flight, free tensor memory and return, and the host sees
// AWQ_ERR_TIMEOUT in the status word.
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kThreads = 512;
constexpr int kRows = 128;       // MMA M: weight rows per tile
constexpr int kKB = 64;          // K columns per block: one 128-byte fp16 swizzle row
constexpr int kBankSlots = 4;    // dW slots in tensor memory per producer warpgroup
constexpr int kSlots = 2 * kBankSlots;
constexpr int kMaxSW = 8, kMaxSX = 8, kMaxAPer = 8;
constexpr uint32_t kSlotCol0 = 256;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: fma(x, r, M) - M = rint(x * r)
constexpr uint32_t kCtrlBytes = 1024;
constexpr int kMaxJobGroups = 4;  // groups a 64-column job can touch when they are >= 24 wide
// Register split after setmaxnreg: 128 * 48 + 256 * 200 + 128 * 56 = 64512
// must not exceed the 512 * 128 = 65536 registers the block is launched
// with (the build checks that every search kernel is compiled to 128
// registers).
constexpr uint32_t kRegsCtl = 56, kRegsProd = 200, kRegsEpi = 56;
constexpr uint32_t kLaunchRegs = 128;
static_assert(128 * kRegsCtl + 256 * kRegsProd + 128 * kRegsEpi <= kThreads * kLaunchRegs,
              "register split");

struct SearchArgs {
  const int32_t* pow2_s;  // [n_alpha]: nonzero when every scale of that alpha is a power of two
  double* partials;       // [n_alpha][n_tiles]
  int32_t* status;
  uint32_t* diag;         // 4 words: where a wait gave up
  int out, in, N;
  int n_alpha, a_per, n_ag, n_rt, n_tt, T, n_kb, n_units, n_tiles;
  int sw, sx;
  uint32_t w_stage;       // bytes of one W ring stage: W tile, then the scale block
  float Lf, maxqf;
  uint64_t wait_limit_ns;
  int test_timeout;
};

// Arguments read only by some instantiations (kept out of SearchArgs, which
// every kernel reads on every job): the precomputed group ranges of the
// wide-group kernels, and the per-alpha weight scaling of the kernels that
// read X already divided by s.
struct WideArgs {
  const float* gext;    // group extremes [n_alpha][out][ngroups] (x2 asym)
  const float* escale;  // [n_alpha]: 2^e_k, the power of two folded into the s table
  int group, ngroups;
};

struct Ctrl {
  uint64_t w_full[kMaxSW], w_empty[kMaxSW];
  uint64_t x_full[kMaxSX], x_empty[kMaxSX];
  uint64_t d_full[kSlots], d_empty[kSlots];
  uint64_t acc_full, acc_empty, epi_full, never, drain;
  uint32_t tmem_base;
  int abort;
  float epi[2][kMaxAPer][4];
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

template <typename WT>
__host__ __device__ constexpr uint32_t w_tile_bytes() {
  return (uint32_t)(kRows * kKB * sizeof(WT));
}

// Eight weights (columns 8*cc .. 8*cc+7 of the 64-column block) of `row`
// from a TMA stage in the 128-byte swizzle layout: the 16-byte chunk j of a
// 128-byte row r sits at chunk j ^ (r & 7).
template <typename WT>
__device__ __forceinline__ void load_w8(const uint8_t* stage, int row, int cc, float (&v)[8]);

template <>
__device__ __forceinline__ void load_w8<__nv_bfloat16>(const uint8_t* stage, int row, int cc,
                                                       float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(stage + row * 128 + ((cc ^ (row & 7)) << 4));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void load_w8<__half>(const uint8_t* stage, int row, int cc,
                                                float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(stage + row * 128 + ((cc ^ (row & 7)) << 4));
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
template <>
__device__ __forceinline__ void load_w8<float>(const uint8_t* stage, int row, int cc,
                                               float (&v)[8]) {
  // fp32 stages hold two 32-column boxes of 128 rows x 128 bytes
  const uint8_t* box = stage + (cc >> 2) * (kRows * 128);
  const int j0 = (cc & 3) * 2;
  const float4 a = *reinterpret_cast<const float4*>(box + row * 128 + ((j0 ^ (row & 7)) << 4));
  const float4 b =
      *reinterpret_cast<const float4*>(box + row * 128 + (((j0 + 1) ^ (row & 7)) << 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Eight consecutive floats of a scale-table row in shared memory (every
// lane reads the same address: a broadcast).
__device__ __forceinline__ void lds_f8(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ uint32_t pack_f16x2(float2 v) {
  __half2 h = __float22half2_rn(v);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Pass 2 for one 64-column K block of a job: -dW * 2^e = (t - q * scale) *
// (2^e / s) as 32 fp16 pairs.  q = round(t / scale): the fast form rounds
// t * (1/scale) with one fused multiply-add against 1.5 * 2^23; the EXACT
// form first forms the correctly rounded quotient q1 = q0 + (t - q0 *
// scale) * (1/scale), q0 = t * (1/scale), then rounds it.
// With CLAMP the rounded value is also capped at the group's top code
// (chi = 1.5 * 2^23 + maxq - zero, in the shifted domain).
//
// With DIV false (X arrives already divided by s) the fp16 pairs are the
// scaled rounding errors t - q * scale themselves and inv_row is unused.
template <bool EXACT, bool CLAMP, bool DIV, int G, int JC>
__device__ __forceinline__ void make_dw(const float (&t)[JC], int kbi, const float* inv_row,
                                        const float (&scl)[JC / G], const float (&rcp)[JC / G],
                                        const float (&chi)[JC / G], uint32_t (&pk)[32]) {
  const float2 mg2 = make_float2(kRoundMagic, kRoundMagic);
  const float2 nm2 = make_float2(-kRoundMagic, -kRoundMagic);
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const int cgi = kbi * 8 + cc;
    const int g = (cgi * 8) / G;
    float i8[8];
    if (DIV) lds_f8(inv_row + cc * 8, i8);
    const float2 rc2 = make_float2(rcp[g], rcp[g]);
    const float2 ns2 = make_float2(-scl[g], -scl[g]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 tv = make_float2(t[cgi * 8 + 2 * e], t[cgi * 8 + 2 * e + 1]);
      float2 av;
      if (EXACT) {
        const float2 q0 = __fmul2_rn(tv, rc2);
        const float2 r = __ffma2_rn(q0, ns2, tv);
        av = __fadd2_rn(__ffma2_rn(r, rc2, q0), mg2);
      } else {
        av = __ffma2_rn(tv, rc2, mg2);
      }
      if (CLAMP) {
        av.x = fminf(av.x, chi[g]);
        av.y = fminf(av.y, chi[g]);
      }
      const float2 qv = __fadd2_rn(av, nm2);
      const float2 ev = __ffma2_rn(qv, ns2, tv);  // t - q * scale
      if (DIV)
        pk[cc * 4 + e] = pack_f16x2(__fmul2_rn(ev, make_float2(i8[2 * e], i8[2 * e + 1])));
      else
        pk[cc * 4 + e] = pack_f16x2(ev);
    }
  }
}

// XS: X arrives as n_alpha fp16 copies X * 2^m_k / s_k (a 3-D tensor map
// [n_alpha][N][in]); the s table rows in the W stages hold s_k * 2^e_k and
// the producer writes (t - q * scale) * 2^e_k with no division by s (needs
// one alpha per unit).
template <typename WT, int G, bool SYM, bool XS = false>
__global__ void __launch_bounds__(kThreads, 1)
    awq_search_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmX,
                      const __grid_constant__ CUtensorMap tmS, const SearchArgs p,
                      const WideArgs wa) {
  // G == 0: groups wider than a job (a multiple of 256 columns or the whole
  // row) whose extremes come precomputed in p.gext
  // G < 0: any other group width that is a multiple of 8 (24, 48, 96, ...):
  // the extremes come precomputed as for G == 0, a 64-column job touches at
  // most kMaxJobGroups groups, and every 8-column chunk takes its group's
  // step
  constexpr bool GP = (G == 0);
  constexpr bool GV = (G < 0);
  constexpr int KBJ = (G == 128 || GP) ? 2 : 1;  // K blocks per producer job
  constexpr int JC = KBJ * kKB;                  // columns per producer job
  constexpr int NG = GP ? 1 : (GV ? JC / 8 : JC / G);  // groups (GV: chunks) per job
  constexpr int CPG = GP ? JC / 8 : (GV ? 1 : G / 8);  // 8-column chunks per group
  constexpr int GE = GP ? JC : (GV ? 8 : G);           // group width as one job sees it
  constexpr uint32_t W_TILE = w_tile_bytes<WT>();
  constexpr uint32_t FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  Ctrl& c = *reinterpret_cast<Ctrl*>(gbase);
  const uint32_t w_ring = base + kCtrlBytes;
  const uint8_t* w_ring_ptr = gbase + kCtrlBytes;
  const uint32_t W_STAGE = p.w_stage;
  const uint32_t S_BYTES = (XS ? 1u : 2u) * (uint32_t)p.a_per * kKB * 4u;  // s (and 2^e/s) rows
  const uint32_t X_STAGE = (uint32_t)p.T * 128u;
  const uint32_t x_ring = w_ring + (uint32_t)p.sw * W_STAGE;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.sw; ++i) {
      mbar_init(smem_addr(&c.w_full[i]), 1);
      mbar_init(smem_addr(&c.w_empty[i]), 4);
    }
    for (int i = 0; i < p.sx; ++i) {
      mbar_init(smem_addr(&c.x_full[i]), 1);
      mbar_init(smem_addr(&c.x_empty[i]), 1);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(smem_addr(&c.d_full[i]), 4);
      mbar_init(smem_addr(&c.d_empty[i]), 1);
    }
    mbar_init(smem_addr(&c.acc_full), 1);
    mbar_init(smem_addr(&c.acc_empty), 4);
    mbar_init(smem_addr(&c.epi_full), 4);
    mbar_init(smem_addr(&c.never), 1);
    mbar_init(smem_addr(&c.drain), 1);
    c.abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(&c.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
    tma_prefetch_map(&tmS);
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // the scale tables, X and the status words come from earlier kernels
  const uint32_t tmem = c.tmem_base;
  volatile int* abort = &c.abort;
  const uint64_t lim = p.wait_limit_ns;
  const int units_per_rt = p.n_ag * p.n_tt;
  const int n_kg = p.n_kb / KBJ;
  const uint32_t hw = (uint32_t)p.sw / 2;  // W stages per warpgroup bank

  if (warp < 4) {
    setmaxnreg_dec<kRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- W loader
      // (the whole warp runs the loop, the elected lane issues the copies)
      uint32_t m0 = 0, ph0 = 0, m1 = 0, ph1 = 0;  // next stage of each bank and its phase
      uint32_t wc0 = 0, wc1 = 0;                  // W blocks loaded into each bank
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const int rt = u / units_per_rt;
        const int ag = (u % units_per_rt) / p.n_tt;
        for (int kb = 0; kb < p.n_kb; ++kb) {
          const int b = (kb / KBJ) & 1;
          const uint32_t st = b ? hw + m1 : m0, ph = b ? ph1 : ph0;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.w_empty[st]), ph ^ 1, abort, lim,
                                                 p.diag, 1, (b ? wc1 : wc0) | (b << 30)));
          if (!ok) break;
          if (elect_one()) {
            const uint32_t bar = smem_addr(&c.w_full[st]);
            mbar_arrive_expect_tx(bar, W_TILE + S_BYTES);
            const uint32_t dst = w_ring + st * W_STAGE;
            if (sizeof(WT) == 4) {
              tma_load_2d(dst, &tmW, bar, kb * kKB, rt * kRows);
              tma_load_2d(dst + W_TILE / 2, &tmW, bar, kb * kKB + 32, rt * kRows);
            } else {
              tma_load_2d(dst, &tmW, bar, kb * kKB, rt * kRows);
            }
            if (XS)
              tma_load_2d(dst + W_TILE, &tmS, bar, kb * kKB, ag);
            else
              tma_load_3d(dst + W_TILE, &tmS, bar, kb * kKB, ag * p.a_per, 0);
          }
          __syncwarp();
          if (b) {
            ++wc1;
            if (++m1 == hw) {
              m1 = 0;
              ph1 ^= 1;
            }
          } else {
            ++wc0;
            if (++m0 == hw) {
              m0 = 0;
              ph0 ^= 1;
            }
          }
        }
      }
      int never_set = 0;  // drain: wait for the loads still in flight
      for (int b = 0; b < 2; ++b) {
        const uint32_t wc = b ? wc1 : wc0;
        for (uint32_t m = wc > hw ? wc - hw : 0; m < wc; ++m)
          mbar_wait(smem_addr(&c.w_full[b * hw + m % hw]), (m / hw) & 1, &never_set, lim);
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- X loader
      const uint32_t SX = (uint32_t)p.sx;
      uint32_t seq = 0, st = 0, ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const int tt = (u % units_per_rt) % p.n_tt;
        const int ag = (u % units_per_rt) / p.n_tt;
        for (int kb = 0; kb < p.n_kb; ++kb) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.x_empty[st]), ph ^ 1, abort, lim,
                                                 p.diag, 3, seq));
          if (!ok) break;
          if (elect_one()) {
            const uint32_t bar = smem_addr(&c.x_full[st]);
            mbar_arrive_expect_tx(bar, X_STAGE);
            if (XS)
              tma_load_3d(x_ring + st * X_STAGE, &tmX, bar, kb * kKB, tt * p.T, ag);
            else
              tma_load_2d(x_ring + st * X_STAGE, &tmX, bar, kb * kKB, tt * p.T);
          }
          __syncwarp();
          ++seq;
          if (++st == SX) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      int never_set = 0;
      for (uint32_t i = seq > SX ? seq - SX : 0; i < seq; ++i)
        mbar_wait(smem_addr(&c.x_full[i % SX]), (i / SX) & 1, &never_set, lim);
    } else if (warp == 2) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs the loop (the elected lane issues) and the ring
      // positions advance by counting, with no division in the loop.
      const uint32_t idesc = idesc_f16_f32(kRows, (uint32_t)p.T);
      const uint32_t SX = (uint32_t)p.sx;
      uint32_t x_st = 0, x_ph = 0;       // X stage and phase of the next unit's first block
      uint32_t d0 = 0, dp0 = 0, d1 = 0, dp1 = 0;  // next dW slot and phase of each bank
      uint32_t useq = 0;
      bool ok = true;
      if (p.test_timeout)
        ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.never), 0, abort, lim, p.diag, 5, 0));
      for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
        const int ag = (u % units_per_rt) / p.n_tt;
        const int na = min(p.a_per, p.n_alpha - ag * p.a_per);
        if (useq > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.acc_empty), (useq - 1) & 1, abort,
                                                 lim, p.diag, 6, useq));
          if (!ok) break;
          tc_fence_after();
        }
        for (int kg = 0; ok && kg < n_kg; ++kg) {
          const int b = kg & 1;
          for (int a = 0; ok && a < na; ++a) {
            uint32_t xs = x_st, xph = x_ph;
            for (int kbi = 0; kbi < KBJ; ++kbi) {
              if (a == 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.x_full[xs]), xph, abort, lim,
                                                       p.diag, 7, xs));
                if (!ok) break;
              }
              const uint32_t slot = b ? d1 : d0, sph = b ? dp1 : dp0;
              const uint32_t ds = b * kBankSlots + slot;
              ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.d_full[ds]), sph, abort, lim,
                                                     p.diag, 8, slot | (b << 30)));
              if (!ok) break;
              tc_fence_after();
              const uint32_t d_t = tmem + (uint32_t)(a * p.T);
              const uint32_t a_t = tmem + kSlotCol0 + ds * 32u;
              const uint64_t bdesc = smem_desc_sw128(x_ring + xs * X_STAGE);
#pragma unroll
              for (int k = 0; k < kKB / 16; ++k)
                umma_ts_elect(d_t, a_t + 8u * k, bdesc + (uint64_t)(2 * k), idesc,
                              (kg | kbi | k) != 0 ? 1u : 0u);
              umma_commit_elect(smem_addr(&c.d_empty[ds]));
              if (a == na - 1) umma_commit_elect(smem_addr(&c.x_empty[xs]));
              if (b) {
                if (++d1 == (uint32_t)kBankSlots) {
                  d1 = 0;
                  dp1 ^= 1;
                }
              } else {
                if (++d0 == (uint32_t)kBankSlots) {
                  d0 = 0;
                  dp0 ^= 1;
                }
              }
              if (++xs == SX) {
                xs = 0;
                xph ^= 1;
              }
            }
          }
          // the next job's X blocks follow this job's KBJ blocks in the ring
#pragma unroll
          for (int kbi = 0; kbi < KBJ; ++kbi) {
            if (++x_st == SX) {
              x_st = 0;
              x_ph ^= 1;
            }
          }
        }
        if (!ok) break;
        umma_commit_elect(smem_addr(&c.acc_full));
        ++useq;
      }
      umma_commit_elect(smem_addr(&c.drain));
      int never_set = 0;
      mbar_wait(smem_addr(&c.drain), 0, &never_set, lim);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ producers
    setmaxnreg_inc<kRegsProd>();
    const int wg = (warp - 4) >> 2;
    const int q = warp & 3;  // tensor memory lanes 32q .. 32q+31
    const int row = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    // the next W stage of this warpgroup's bank and its phase (counted: the
    // bank's stages are used in order), and the dW-slot counter
    uint32_t wsl = 0, wph = 0, dn = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      const int rem = u % units_per_rt;
      const int ag = rem / p.n_tt;
      const int na = min(p.a_per, p.n_alpha - ag * p.a_per);
      uint32_t exact_mask = 0;
      for (int a = 0; a < na; ++a)
        if (p.pow2_s[ag * p.a_per + a] != 0) exact_mask |= 1u << a;
      // XS: t is scaled by 2^e (one alpha per unit), and so are the step's
      // lower clamp 1e-8 and the group ranges read from memory
      const float esc = XS ? __ldg(wa.escale + ag) : 1.0f;
      const float clampk = 1e-8f * esc;
      // this thread's W row, for the group ranges read from memory (GP, GV)
      const int64_t grow = (GP || GV) ? min((int64_t)(u / units_per_rt) * kRows + row,
                                            (int64_t)p.out - 1)
                                      : 0;
      for (int kg = wg; ok && kg < n_kg; kg += 2) {
        const uint8_t* stg[KBJ];
        uint32_t wst[KBJ];
#pragma unroll
        for (int kbi = 0; kbi < KBJ; ++kbi) {
          uint32_t sl = wsl + kbi, ph = wph;  // KBJ <= hw: at most one wrap
          if (sl >= hw) {
            sl -= hw;
            ph ^= 1;
          }
          const uint32_t st = wg * hw + sl;
          wst[kbi] = st;
          stg[kbi] = w_ring_ptr + st * W_STAGE;
          if (ok)
            ok = mbar_wait(smem_addr(&c.w_full[st]), ph, abort, lim, p.diag, 10, sl | (wg << 30));
        }
        ok = __all_sync(FULL, ok);
        if (!ok) break;
        for (int a = 0; ok && a < na; ++a) {
          // pass 1: t = fl32(w * s) and each group's range
          float t[JC];
          float r0[NG][4], r1[NG][4];  // sym: running max|t|; asym: running min / max
#pragma unroll
          for (int g = 0; g < NG; ++g)
#pragma unroll
            for (int j = 0; j < 4; ++j) r0[g][j] = r1[g][j] = 0.0f;
          if constexpr (GP) {  // the group's extremes over all its jobs (loaded before pass 1
                               // so that the load overlaps it)
            const int64_t gi = ((int64_t)(ag * p.a_per + a) * p.out + grow) * wa.ngroups +
                               (kg * JC) / wa.group;  // kg * JC < in <= 2^24
            if (SYM) {
              r0[0][0] = __ldg(wa.gext + gi) * esc;
            } else {
              r0[0][0] = -__ldg(wa.gext + 2 * gi) * esc;
              r1[0][0] = __ldg(wa.gext + 2 * gi + 1) * esc;
            }
          }
          // GV: the extremes of the (at most kMaxJobGroups) groups the job touches
          float vlo[kMaxJobGroups], vhi[kMaxJobGroups];
          int vg0 = 0, vgn = 1;
          if constexpr (GV) {
            const int col0 = kg * JC;
            vg0 = col0 / wa.group;
            vgn = min((col0 + JC - 1) / wa.group, wa.ngroups - 1) - vg0 + 1;
            const int64_t gi0 = ((int64_t)(ag * p.a_per + a) * p.out + grow) * wa.ngroups + vg0;
#pragma unroll
            for (int i = 0; i < kMaxJobGroups; ++i) {
              vlo[i] = vhi[i] = 0.0f;
              if (i < vgn) {
                if (SYM) {
                  vhi[i] = __ldg(wa.gext + gi0 + i) * esc;
                } else {
                  vlo[i] = -__ldg(wa.gext + 2 * (gi0 + i)) * esc;
                  vhi[i] = __ldg(wa.gext + 2 * (gi0 + i) + 1) * esc;
                }
              }
            }
          }
#pragma unroll
          for (int cgi = 0; cgi < JC / 8; ++cgi) {
            const int kbi = cgi >> 3, cc = cgi & 7, g = cgi / CPG;
            float w8[8], s8[8];
            load_w8<WT>(stg[kbi], row, cc, w8);
            lds_f8(reinterpret_cast<const float*>(stg[kbi] + W_TILE) + a * kKB + cc * 8, s8);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 tv =
                  __fmul2_rn(make_float2(w8[2 * e], w8[2 * e + 1]), make_float2(s8[2 * e], s8[2 * e + 1]));
              t[cgi * 8 + 2 * e] = tv.x;
              t[cgi * 8 + 2 * e + 1] = tv.y;
              if constexpr (!GP && !GV) {
                if (SYM) {
                  r0[g][e] = fmax3f(r0[g][e], fabsf(tv.x), fabsf(tv.y));
                } else {
                  r0[g][e] = fmin3f(r0[g][e], tv.x, tv.y);
                  r1[g][e] = fmax3f(r1[g][e], tv.x, tv.y);
                }
              }
            }
          }
          if constexpr (XS) {
            // pass 2 reads no table: with one alpha per unit the stages are
            // free once pass 1 has read the weights and s
            __syncwarp();
            if (lane == 0)
              for (int kbi = 0; kbi < KBJ; ++kbi)
                mbar_arrive(smem_addr(&c.w_empty[wst[kbi]]));
          }
          // group steps
          float scl[NG], rcp[NG], chi[NG];
          if constexpr (GV) {
            // each group's step once, then every chunk takes its group's
            float vs[kMaxJobGroups], vr[kMaxJobGroups], vc[kMaxJobGroups];
#pragma unroll
            for (int i = 0; i < kMaxJobGroups; ++i) {
              if (SYM) {
                vs[i] = fmaxf(__fdiv_rn(vhi[i], p.Lf), clampk);
                vc[i] = 0.0f;
              } else {
                vs[i] = fmaxf(__fdiv_rn(__fsub_rn(vhi[i], vlo[i]), p.maxqf), clampk);
                vc[i] = kRoundMagic + p.maxqf - rintf(__fdiv_rn(-vlo[i], vs[i]));
              }
              vr[i] = __frcp_rn(vs[i]);
            }
            const int b1 = (vg0 + 1) * wa.group, b2 = b1 + wa.group, b3 = b2 + wa.group;
#pragma unroll
            for (int cgi = 0; cgi < NG; ++cgi) {
              const int col = kg * JC + cgi * 8;
              const int i = (col >= b1) + (col >= b2) + (col >= b3);
              scl[cgi] = i == 0 ? vs[0] : i == 1 ? vs[1] : i == 2 ? vs[2] : vs[3];
              rcp[cgi] = i == 0 ? vr[0] : i == 1 ? vr[1] : i == 2 ? vr[2] : vr[3];
              chi[cgi] = i == 0 ? vc[0] : i == 1 ? vc[1] : i == 2 ? vc[2] : vc[3];
            }
          }
#pragma unroll
          for (int g = 0; g < (GV ? 0 : NG); ++g) {
            if (SYM) {
              const float m = fmaxf(fmaxf(r0[g][0], r0[g][1]), fmaxf(r0[g][2], r0[g][3]));
              scl[g] = fmaxf(__fdiv_rn(m, p.Lf), clampk);
              chi[g] = 0.0f;
            } else {
              const float lo = fminf(fminf(r0[g][0], r0[g][1]), fminf(r0[g][2], r0[g][3]));
              const float hi = fmaxf(fmaxf(r1[g][0], r1[g][1]), fmaxf(r1[g][2], r1[g][3]));
              scl[g] = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), p.maxqf), clampk);
              chi[g] = kRoundMagic + p.maxqf - rintf(__fdiv_rn(-lo, scl[g]));
            }
            rcp[g] = __frcp_rn(scl[g]);
          }
          // pass 2: -dW * 2^e as fp16 pairs into a tensor memory slot
          const bool exact = (exact_mask >> a) & 1u;
#pragma unroll
          for (int kbi = 0; kbi < KBJ; ++kbi) {
            const uint32_t ds = wg * kBankSlots + dn % kBankSlots;
            ok = mbar_wait(smem_addr(&c.d_empty[ds]), ((dn / kBankSlots) & 1) ^ 1, abort, lim,
                           p.diag, 11, dn | (wg << 30));
            ok = __all_sync(FULL, ok);
            if (!ok) break;
            tc_fence_after();
            const float* inv_row =
                reinterpret_cast<const float*>(stg[kbi] + W_TILE) + (p.a_per + a) * kKB;
            uint32_t pk[32];
            if (exact)
              make_dw<true, !SYM, !XS, GE, JC>(t, kbi, inv_row, scl, rcp, chi, pk);
            else
              make_dw<false, false, !XS, GE, JC>(t, kbi, inv_row, scl, rcp, chi, pk);
            tmem_st32(tmem + lane_addr + kSlotCol0 + ds * 32u, pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&c.d_full[ds]));
            ++dn;
          }
        }
        if (!ok) break;
        // every alpha of the job is done with these stages (weights and tables)
        if constexpr (!XS) {
          __syncwarp();
          if (lane == 0)
            for (int kbi = 0; kbi < KBJ; ++kbi)
              mbar_arrive(smem_addr(&c.w_empty[wst[kbi]]));
        }
        wsl += KBJ;
        if (wsl >= hw) {
          wsl -= hw;
          wph ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp 12 + q reads tensor memory lanes 32q .. 32q+31 (rows of the tile)
    // once the unit's MMAs are done, squares and sums the accumulators, and
    // hands the accumulator back; the producers meanwhile run on into the
    // next unit.
    setmaxnreg_dec<kRegsEpi>();
    const int q = warp & 3;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    uint32_t useq = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.n_units; u += gridDim.x) {
      const int rem = u % units_per_rt;
      const int rt = u / units_per_rt, ag = rem / p.n_tt, tt = rem % p.n_tt;
      const int na = min(p.a_per, p.n_alpha - ag * p.a_per);
      ok = mbar_wait(smem_addr(&c.acc_full), useq & 1, abort, lim, p.diag, 12, useq);
      ok = __all_sync(FULL, ok);
      if (!ok) break;
      tc_fence_after();
      for (int a = 0; a < na; ++a) {
        float acc = 0.0f;
        const uint32_t cb = tmem + lane_addr + (uint32_t)(a * p.T);
        for (int cc = 0; cc < p.T; cc += 32) {  // T is a multiple of 32: two loads, one wait
          uint32_t v[16], w[16];
          tmem_ld16(cb + (uint32_t)cc, v);
          tmem_ld16(cb + (uint32_t)cc + 16u, w);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float f = __uint_as_float(v[i]);
            acc = fmaf(f, f, acc);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float f = __uint_as_float(w[i]);
            acc = fmaf(f, f, acc);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(FULL, acc, o);
        if (lane == 0) c.epi[useq & 1][a][q] = acc;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&c.acc_empty));
        mbar_arrive(smem_addr(&c.epi_full));
      }
      if (warp == 12) {
        bool ok2 = true;
        if (lane == 0) ok2 = mbar_wait(smem_addr(&c.epi_full), useq & 1, abort, lim, p.diag, 13, useq);
        __syncwarp();
        ok2 = __shfl_sync(FULL, ok2, 0);
        if (!ok2) {
          ok = false;
          break;
        }
        if (lane < na) {
          double s = 0.0;
          for (int w = 0; w < 4; ++w) s += (double)c.epi[useq & 1][lane][w];
          p.partials[(size_t)(ag * p.a_per + lane) * p.n_tiles + rt * p.n_tt + tt] = s;
        }
      }
      ++useq;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && c.abort) set_status(p.status, ST_TIMEOUT);
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D map of a row-major matrix, 128-byte swizzled boxes (the MMA operand layout).
bool make_map(CUtensorMap* m, CUtensorMapDataType t, const void* ptr, uint64_t cols, uint64_t rows,
              uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, t, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the two float32 scale tables s32 and inv_s32 ([n_alpha][in]
// each, table_bytes apart): box = 64 columns x a_per alphas x both tables,
// unswizzled; out-of-range columns and alphas read as zero.
bool make_scale_map(CUtensorMap* m, const float* s32, uint64_t in, uint64_t n_alpha,
                    uint64_t table_bytes, uint32_t a_per) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {in, n_alpha, 2};
  cuuint64_t strides[2] = {in * 4, table_bytes};
  cuuint32_t box[3] = {(cuuint32_t)kKB, a_per, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(s32), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over the n_alpha fp16 copies of X / s ([n_alpha][N][in]): boxes of
// 64 columns x T tokens of one alpha, 128-byte swizzle (the MMA's B layout).
bool make_xs_map(CUtensorMap* m, const void* xs, uint64_t in, uint64_t N, uint64_t n_alpha,
                 uint32_t T) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {in, N, n_alpha};
  cuuint64_t strides[2] = {in * 2, N * in * 2};
  cuuint32_t box[3] = {(cuuint32_t)kKB, T, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(xs), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over the scaled s table ([n_alpha][in] float32): boxes of 64
// columns of one alpha, unswizzled; out-of-range columns read as zero.
bool make_s_map(CUtensorMap* m, const float* ss32, uint64_t in, uint64_t n_alpha) {
  auto enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {in, n_alpha};
  cuuint64_t strides[1] = {in * 4};
  cuuint32_t box[2] = {(cuuint32_t)kKB, 1};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ss32), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const SearchArgs, const WideArgs);

template <typename WT>
KernelFn pick_xs(int group, int sym, int64_t in) {
  if (search_wide_group(group, in))
    return sym ? &awq_search_kernel<WT, 0, true, true> : &awq_search_kernel<WT, 0, false, true>;
  if (search_needs_ranges(group, in))
    return sym ? &awq_search_kernel<WT, -1, true, true> : &awq_search_kernel<WT, -1, false, true>;
  switch (group) {
    case 8: return sym ? &awq_search_kernel<WT, 8, true, true> : &awq_search_kernel<WT, 8, false, true>;
    case 16: return sym ? &awq_search_kernel<WT, 16, true, true> : &awq_search_kernel<WT, 16, false, true>;
    case 32: return sym ? &awq_search_kernel<WT, 32, true, true> : &awq_search_kernel<WT, 32, false, true>;
    case 64: return sym ? &awq_search_kernel<WT, 64, true, true> : &awq_search_kernel<WT, 64, false, true>;
    case 128:
      return sym ? &awq_search_kernel<WT, 128, true, true> : &awq_search_kernel<WT, 128, false, true>;
    default: return nullptr;
  }
}

template <typename WT>
KernelFn pick_g(int group, int sym, int64_t in, bool gp) {
  if (gp && search_wide_group(group, in))
    return sym ? &awq_search_kernel<WT, 0, true> : &awq_search_kernel<WT, 0, false>;
  if (gp) return sym ? &awq_search_kernel<WT, -1, true> : &awq_search_kernel<WT, -1, false>;
  switch (group) {
    case 8: return sym ? &awq_search_kernel<WT, 8, true> : &awq_search_kernel<WT, 8, false>;
    case 16: return sym ? &awq_search_kernel<WT, 16, true> : &awq_search_kernel<WT, 16, false>;
    case 32: return sym ? &awq_search_kernel<WT, 32, true> : &awq_search_kernel<WT, 32, false>;
    case 64: return sym ? &awq_search_kernel<WT, 64, true> : &awq_search_kernel<WT, 64, false>;
    case 128: return sym ? &awq_search_kernel<WT, 128, true> : &awq_search_kernel<WT, 128, false>;
    default: return nullptr;
  }
}

int max_dyn_smem() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return v;
}

}  // namespace

bool tensor_map_sw128(CUtensorMap* m, CUtensorMapDataType t, const void* ptr, uint64_t cols,
                      uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
  return make_map(m, t, ptr, cols, rows, row_bytes, box_cols, box_rows);
}

bool search_wide_group(int64_t group, int64_t in) {
  return in % 8 == 0 && group > 0 && in % group == 0 && (group % 256 == 0 || group == in);
}

namespace {
bool in_job_group(int64_t group) {
  return group == 8 || group == 16 || group == 32 || group == 64 || group == 128;
}
}  // namespace

bool search_needs_ranges(int64_t group, int64_t in) {
  if (search_wide_group(group, in)) return true;  // (one group per row included)
  return !in_job_group(group) && group > 0 && in % group == 0 && group % 8 == 0 && in % 8 == 0;
}

bool search_xs_eligible(int dt, int64_t in, int64_t N, int group, int grid) {
  // one alpha per unit (more than 128 tokens), a group inside one producer
  // job (8, 16, 32, 64 or 128 columns) or one read from precomputed ranges
  // (wider groups, or groups that straddle the jobs), 16-bit W, and
  // all n_alpha copies of X / s small enough to stay in L2 during the search
  const int64_t n_alpha = (int64_t)grid + 1;
  return dt != kDtF32 && N > 128 && in % 8 == 0 &&
         (in_job_group(group) || search_needs_ranges(group, in)) &&
         n_alpha * N * in * 2 <= ((int64_t)64 << 20);
}

bool search_supported(int dt, int64_t out, int64_t in, int64_t N, int bits, int group, int grid) {
  (void)dt; (void)bits; (void)grid;
  if (!in_job_group(group) && !search_needs_ranges(group, in)) return false;
  if (in % group != 0) return false;
  if (out > (1 << 24) || N > (1 << 24) || in > (1 << 24)) return false;
  return true;
}

SearchPlan plan_search(int dt, int64_t out, int64_t in, int64_t N, int n_alpha, int group,
                       bool gp, int sms, bool xs) {
  SearchPlan pl{};
  pl.n_tt = (int)((N + 255) / 256);
  const int64_t per = (N + pl.n_tt - 1) / pl.n_tt;
  pl.T = (int)((per + 31) / 32 * 32);
  pl.a_per = std::max(1, std::min({n_alpha, 256 / pl.T, kMaxAPer}));
  pl.n_ag = (n_alpha + pl.a_per - 1) / pl.a_per;
  pl.n_rt = (int)((out + kRows - 1) / kRows);
  pl.n_kb = (int)((in + kKB - 1) / kKB);
  // with precomputed group ranges a job always spans two K blocks; an odd
  // count gets one more block, which lies wholly past the last column (the
  // tensor-map loads fill it with zeros, so it adds nothing)
  if (gp) pl.n_kb += pl.n_kb & 1;
  pl.n_units = pl.n_rt * pl.n_ag * pl.n_tt;
  pl.n_tiles = pl.n_rt * pl.n_tt;
  const int kbj = (group == 128 || gp) ? 2 : 1;
  const size_t w_tile = (size_t)kRows * kKB * dtype_size(dt);
  pl.w_stage = align_up(w_tile + (xs ? 1 : 2) * (size_t)pl.a_per * kKB * 4, 1024);
  const size_t x_stage = (size_t)pl.T * 128;
  const size_t budget = (size_t)max_dyn_smem() - kCtrlBytes - 1024;
  // deepest W ring (two equal banks, each holding at least one job) that
  // leaves at least three X stages; then as many X stages as still fit
  pl.sw = 0;
  pl.sx = 0;
  for (int sw = kMaxSW; sw >= 2 * kbj && pl.sw == 0; sw -= 2) {
    if (sw * pl.w_stage + 3 * x_stage <= budget) {
      pl.sw = sw;
      pl.sx = (int)std::min<size_t>(kMaxSX, (budget - sw * pl.w_stage) / x_stage);
    }
  }
  pl.smem = kCtrlBytes + 1024 + pl.sw * pl.w_stage + pl.sx * x_stage;
  pl.grid = std::max(1, std::min(pl.n_units, sms));
  return pl;
}

cudaError_t launch_search(const void* W, const void* Xf16, int dt, int64_t out, int64_t in,
                          int64_t N, int bits, int group, int sym, int n_alpha,
                          const float* s32, const float* inv_s32, const int32_t* pow2_s,
                          const float* gext, const float* ss32, const float* escale,
                          double* partials, const SearchPlan& pl, int64_t wait_limit_ns,
                          int test_timeout, int32_t* dev_status, uint32_t* diag, cudaStream_t s,
                          cudaEvent_t ev0, cudaEvent_t ev1) {
  KernelFn fn = nullptr;
  CUtensorMapDataType wt;
  uint32_t wbox;
  const bool xs = ss32 != nullptr;
  if (xs && (pl.a_per != 1 || dt == kDtF32)) return cudaErrorInvalidValue;
  switch (dt) {
    case kDtF32:
      fn = pick_g<float>(group, sym, in, gext != nullptr);
      wt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
      wbox = 32;
      break;
    case kDtF16:
      fn = xs ? pick_xs<__half>(group, sym, in) : pick_g<__half>(group, sym, in, gext != nullptr);
      wt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
      wbox = 64;
      break;
    default:
      fn = xs ? pick_xs<__nv_bfloat16>(group, sym, in)
              : pick_g<__nv_bfloat16>(group, sym, in, gext != nullptr);
      wt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
      wbox = 64;
      break;
  }
  if (!fn || pl.sw < 2 || pl.sx < 3) return cudaErrorInvalidValue;
  if (search_needs_ranges(group, in) != (gext != nullptr)) return cudaErrorInvalidValue;
  CUtensorMap mw, mx, ms;
  if (!make_map(&mw, wt, W, (uint64_t)in, (uint64_t)out, (uint64_t)in * dtype_size(dt), wbox, kRows))
    return cudaErrorInvalidValue;
  if (xs) {
    if ((reinterpret_cast<uintptr_t>(ss32) & 15) != 0 || escale == nullptr) return cudaErrorInvalidValue;
    if (!make_xs_map(&mx, Xf16, (uint64_t)in, (uint64_t)N, (uint64_t)n_alpha, (uint32_t)pl.T))
      return cudaErrorInvalidValue;
    if (!make_s_map(&ms, ss32, (uint64_t)in, (uint64_t)n_alpha)) return cudaErrorInvalidValue;
  } else {
    const uintptr_t tbl = reinterpret_cast<uintptr_t>(inv_s32) - reinterpret_cast<uintptr_t>(s32);
    if (inv_s32 <= s32 || (tbl & 15) != 0 || (reinterpret_cast<uintptr_t>(s32) & 15) != 0)
      return cudaErrorInvalidValue;
    if (!make_map(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Xf16, (uint64_t)in, (uint64_t)N,
                  (uint64_t)in * 2, kKB, (uint32_t)pl.T))
      return cudaErrorInvalidValue;
    if (!make_scale_map(&ms, s32, (uint64_t)in, (uint64_t)n_alpha, (uint64_t)tbl,
                        (uint32_t)pl.a_per))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
  if (e != cudaSuccess) return e;
  SearchArgs a;
  a.pow2_s = pow2_s;
  a.partials = partials;
  a.status = dev_status;
  a.diag = diag;
  a.out = (int)out;
  a.in = (int)in;
  a.N = (int)N;
  a.n_alpha = n_alpha;
  a.a_per = pl.a_per;
  a.n_ag = pl.n_ag;
  a.n_rt = pl.n_rt;
  a.n_tt = pl.n_tt;
  a.T = pl.T;
  a.n_kb = pl.n_kb;
  a.n_units = pl.n_units;
  a.n_tiles = pl.n_tiles;
  a.sw = pl.sw;
  a.sx = pl.sx;
  a.w_stage = (uint32_t)pl.w_stage;
  a.Lf = (float)((1 << (bits - 1)) - 1);
  a.maxqf = (float)((1 << bits) - 1);
  a.wait_limit_ns = (uint64_t)(wait_limit_ns > 0 ? wait_limit_ns : 2000000000LL);
  a.test_timeout = test_timeout;
  if (ev0 && (e = cudaEventRecord(ev0, s)) != cudaSuccess) return e;
  WideArgs wa;
  wa.gext = gext;
  wa.escale = escale;
  wa.group = group;
  wa.ngroups = (int)(in / group);
  e = launch_pdl(fn, dim3((unsigned)pl.grid), dim3(kThreads), (size_t)pl.smem, s, mw, mx, ms, a,
                 wa);
  if (e == cudaSuccess && ev1) e = cudaEventRecord(ev1, s);
  return e;
}

}  // namespace awq
