// Conversion of awq_quantize_pack's outputs into the tensors a quantized
// checkpoint stores per linear layer ("AWQ vs GPTQ Quantization
// Architectures Compared", "What lands on disk"): qweight as 32-bit words of
// b-bit codes packed along the input axis, [in*b/32][out]; scales in FP16,
// [in/g][out]; qzeros as b-bit zero points packed along the output axis,
// [in/g][ceil(out*b/32)].
//
// With b dividing 32 and in a multiple of 32/b, word k of row o of the
// row-major codes already holds inputs (32/b)k .. (32/b)k + 32/b - 1 of
// output o, lowest input in the lowest bits, which is exactly the
// checkpoint's word (k, o): qweight is a transpose of whole words.  The
// scales are a transpose with rounding to FP16; the zero points are
// gathered down a column and packed.  All three are HBM-bound copies.
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kTile = 32;  // transpose tile (32 x 32 elements, 32 x 8 threads)

// dst[c][r] = f(src[r][c]) for an R x C matrix through a padded shared tile.
template <typename S, typename D, typename F>
__device__ __forceinline__ void transpose_tile(const S* __restrict__ src, D* __restrict__ dst,
                                               int64_t R, int64_t C, int64_t tile, F f) {
  __shared__ S buf[kTile][kTile + 1];
  const int64_t tiles_c = (C + kTile - 1) / kTile;
  const int64_t r0 = (tile / tiles_c) * kTile, c0 = (tile % tiles_c) * kTile;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < kTile; j += 8) {
    const int64_t r = r0 + ty + j, c = c0 + tx;
    if (r < R && c < C) buf[ty + j][tx] = src[r * C + c];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kTile; j += 8) {
    const int64_t c = c0 + ty + j, r = r0 + tx;
    if (r < R && c < C) dst[c * R + r] = f(buf[tx][ty + j]);
  }
}

// Blocks [0, t_q): qweight tiles; [t_q, t_q + t_s): scale tiles; the rest:
// zero-point words, one per thread.
__global__ void __launch_bounds__(256) export_kernel(
    const uint32_t* __restrict__ qweight, const float* __restrict__ scales,
    const uint8_t* __restrict__ zeros, int64_t out, int64_t nw, int64_t ng, int bits,
    int64_t t_q, int64_t t_s, uint32_t* __restrict__ qweight_t, __half* __restrict__ scales_h,
    uint32_t* __restrict__ qzeros, int64_t nzw, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  const int64_t b = blockIdx.x;
  if (b < t_q) {
    transpose_tile(qweight, qweight_t, out, nw, b, [](uint32_t v) { return v; });
  } else if (b < t_q + t_s) {
    bool bad = false;
    transpose_tile(scales, scales_h, out, ng, b - t_q, [&bad](float v) {
      const __half h = __float2half_rn(v);
      bad |= !(fabsf(__half2float(h)) <= 65504.0f);  // overflow to infinity, or NaN
      return h;
    });
    if (bad) set_status(dev_status, ST_NONFINITE);
  } else {
    // word (gi, w): zero points of outputs w*per .. w*per + per - 1 in group gi
    const int per = 32 / bits;
    const int64_t i = (b - t_q - t_s) * blockDim.x + threadIdx.x;
    if (i >= ng * nzw) return;
    const int64_t gi = i / nzw, w = i % nzw;
    uint32_t word = 0u;
    for (int k = 0; k < per; ++k) {
      const int64_t o = w * per + k;
      if (o < out) word |= (uint32_t)zeros[o * ng + gi] << (k * bits);
    }
    qzeros[i] = word;
  }
}

}  // namespace

cudaError_t launch_export_checkpoint(const uint32_t* qweight, const float* scales,
                                     const uint8_t* zeros, int64_t out, int64_t in, int bits,
                                     int group, uint32_t* qweight_t, void* scales_h,
                                     uint32_t* qzeros, int32_t* dev_status, cudaStream_t s) {
  const int64_t nw = in * bits / 32, ng = in / group, nzw = (out * bits + 31) / 32;
  const int64_t t_q = ((out + kTile - 1) / kTile) * ((nw + kTile - 1) / kTile);
  const int64_t t_s = ((out + kTile - 1) / kTile) * ((ng + kTile - 1) / kTile);
  const int64_t t_z = (ng * nzw + 255) / 256;
  const int64_t blocks = t_q + t_s + t_z;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  return launch_pdl(export_kernel, (unsigned)blocks, 256, 0, s, qweight, scales, zeros, out, nw,
                    ng, bits, t_q, t_s, qweight_t, static_cast<__half*>(scales_h), qzeros, nzw,
                    dev_status);
}

}  // namespace awq
