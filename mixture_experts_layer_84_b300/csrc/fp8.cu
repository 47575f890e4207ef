// FP8 (E4M3) rows with one power-of-two scale each, and the FP8 dispatch.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 低精度通信: the
// activations that enter the MoE up-projection are turned into FP8 before the
// dispatch, so the dispatch moves one byte per element and the up-projection
// runs its FP8 forward on them as they are; the scaling factors are integral
// powers of two.  The combine stays bf16.
//
// Row rule: s = the smallest integer >= -127 with amax <= 448 * 2^s, taken from
// the float32 bits of amax; codes = E4M3(x * 2^-s) rounded to nearest even
// (cvt.rn.satfinite through cuda_fp8.h).  x * 2^-s is exact in float32 (a
// power-of-two scaling of a bf16 value that stays within +-448), so the codes
// are a function of the input bits alone.
//
// quantize_rows_fp8     one warp per row: amax, then the codes (the row is read
//                       twice; the second read comes from L1/L2).
// dispatch_scatter_fp8  one warp per token: the same per-row rule on U, the
//                       codes written to each kept slot row of X8 and the scale
//                       2^s to x_scale; each token is quantised once for its k
//                       copies.
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  // amax = 1.M 2^(E-127) = (1.M / 2) 2^(E-126); 448 = 0.875 2^9, and 1.M / 2 > 0.875 iff M > 0.75 * 2^23
  const uint32_t b = __float_as_uint(amax);
  const int E = static_cast<int>((b >> 23) & 0xffu);
  if (E == 0) return -127;  // zero or subnormal
  const int s = E - 135 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
  return s < -127 ? -127 : s;
}

// 2^s exactly, s in [-127, 127] (2^-127 is a float32 subnormal)
__device__ __forceinline__ float pow2_exact(int s) {
  return s >= -126 ? __uint_as_float(static_cast<uint32_t>(s + 127) << 23) : __uint_as_float(1u << 22);
}

__device__ __forceinline__ float amax8(const uint4& v, float m) {
  float f[8];
  Vec16<bf16>::unpack(v, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// 8 bf16 values times `mul` (a power of two) as 8 E4M3 bytes, in order
__device__ __forceinline__ uint2 quant8(const uint4& v, float mul) {
  float f[8];
  Vec16<bf16>::unpack(v, f);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t q = __nv_cvt_float_to_fp8(f[i] * mul, __NV_SATFINITE, __NV_E4M3);
    w[i / 4] |= q << (8 * (i % 4));
  }
  return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

__global__ void __launch_bounds__(256) quantize_rows_fp8(const uint4* __restrict__ src, int64_t rows, int vpr,
                                                         uint2* __restrict__ dst, float* __restrict__ scale) {
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
    const uint4* row = src + r * vpr;
    float m = 0.f;
    for (int v = lane; v < vpr; v += 32) m = amax8(row[v], m);
    const int s = fp8_scale_exponent(warp_max(m));
    const float mul = pow2_exact(-s);
    for (int v = lane; v < vpr; v += 32) dst[r * vpr + v] = quant8(row[v], mul);
    if (lane == 0) scale[r] = pow2_exact(s);
  }
}

__global__ void __launch_bounds__(256) dispatch_scatter_fp8(const uint4* __restrict__ U,
                                                            const int32_t* __restrict__ slot_row,
                                                            uint2* __restrict__ X8, float* __restrict__ x_scale,
                                                            int64_t T, int k, int vpr) {
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < T; t += warps) {
    const int32_t my_row = lane < k ? slot_row[t * k + lane] : -1;
    const uint4* row = U + t * vpr;
    float m = 0.f;
    for (int v = lane; v < vpr; v += 32) m = amax8(row[v], m);
    const int s = fp8_scale_exponent(warp_max(m));
    const float mul = pow2_exact(-s);
    if (my_row >= 0) x_scale[my_row] = pow2_exact(s);
    // warp-uniform trip count: every lane reaches the shuffles below
    for (int base = 0; base < vpr; base += 32) {
      const int v = base + lane;
      uint2 q = make_uint2(0u, 0u);
      if (v < vpr) q = quant8(row[v], mul);
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
        if (r >= 0 && v < vpr) X8[static_cast<int64_t>(r) * vpr + v] = q;
      }
    }
  }
}

int row_blocks(int64_t rows) {
  const int64_t want = (rows + 7) / 8;
  return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8)));
}

}  // namespace

cudaError_t launch_quantize_fp8(int64_t rows, int cols, const void* src, uint8_t* dst, float* scale, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  quantize_rows_fp8<<<row_blocks(rows), 256, 0, s>>>(static_cast<const uint4*>(src), rows, cols / 8,
                                                     reinterpret_cast<uint2*>(dst), scale);
  return cudaGetLastError();
}

cudaError_t launch_scatter_fp8(const Plan& p, const void* U, const int32_t* slot_row, uint8_t* X8, float* x_scale,
                               cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  dispatch_scatter_fp8<<<row_blocks(p.T), 256, 0, s>>>(static_cast<const uint4*>(U), slot_row,
                                                       reinterpret_cast<uint2*>(X8), x_scale, p.T, p.k, p.h / 8);
  return cudaGetLastError();
}

}  // namespace moe
