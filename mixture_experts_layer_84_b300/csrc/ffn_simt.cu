// Grouped SwiGLU expert FFN in float32 on the CUDA cores (the float32 configs;
// tf32 tensor cores would not hold the float32 tolerance).
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 从稠密 FFN 到 MoE:
// FFN(u) = W_down (SiLU(W_gate u) ⊙ W_up u); section 专家计算：padding、
// block-sparse 与 grouped GEMM: one launch per half over the variable-length
// expert segments, located from the device-resident offsets (no host read).
//
// Block tile: 32 rows x 32 output columns, K in chunks of 32 staged in shared
// memory; each thread owns 2 x 2 outputs (times two for gate and up).
// blockIdx.x enumerates (expert, 32-row tile) pairs up to a bound that covers
// any segmentation; blocks past the last tile exit.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int SB = 32;  // rows, columns and K chunk of a tile

template <bool SWIGLU>
__global__ void __launch_bounds__(256) ffn_simt_f32(const float* __restrict__ A, const float* __restrict__ B0,
                                                    const float* __restrict__ B1, const int32_t* __restrict__ offsets,
                                                    int E, int K, int N, int64_t rows_cap, float* __restrict__ out,
                                                    int32_t* status) {
  __shared__ float As[SB][SB + 1];
  __shared__ float Bs0[SB][SB + 1];
  __shared__ float Bs1[SWIGLU ? SB : 1][SB + 1];
  __shared__ int s_e, s_mt;
  if (threadIdx.x == 0) {
    int slot = blockIdx.x, found = -1, mt = 0;
    bool bad = false;
    for (int e = 0; e < E; ++e) {  // every segment is checked before any block writes
      const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
      if (lo < 0 || hi < lo || static_cast<int64_t>(hi) > rows_cap) {
        bad = true;
        continue;
      }
      const int m = (hi - lo + SB - 1) / SB;
      if (found < 0 && slot < m) {
        found = e;
        mt = slot;
      }
      if (found < 0) slot -= m;
    }
    if (bad) {  // inconsistent segments: no writes
      set_status(status, MOE_DEV_BAD_OFFSETS);
      found = -1;
    }
    s_e = found;
    s_mt = mt;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int64_t row0 = static_cast<int64_t>(seg_lo(offsets, e)) + static_cast<int64_t>(s_mt) * SB;
  const int nrows = min(SB, seg_hi(offsets, e, rows_cap) - static_cast<int>(row0));
  const int n0 = blockIdx.y * SB;
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float g[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, up[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  const float* Be0 = B0 + static_cast<int64_t>(e) * N * K;
  const float* Be1 = SWIGLU ? B1 + static_cast<int64_t>(e) * N * K : nullptr;

  for (int k0 = 0; k0 < K; k0 += SB) {
    for (int i = threadIdx.x; i < SB * SB; i += blockDim.x) {
      const int r = i / SB, kk = i % SB;
      const bool kin = k0 + kk < K;
      As[kk][r] = (r < nrows && kin) ? A[(row0 + r) * K + k0 + kk] : 0.f;
      const bool nin = n0 + r < N;
      Bs0[kk][r] = (nin && kin) ? Be0[static_cast<int64_t>(n0 + r) * K + k0 + kk] : 0.f;
      if (SWIGLU) Bs1[kk][r] = (nin && kin) ? Be1[static_cast<int64_t>(n0 + r) * K + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < SB; ++kk) {
      const float a0 = As[kk][ty * 2], a1 = As[kk][ty * 2 + 1];
      const float b0 = Bs0[kk][tx * 2], b1 = Bs0[kk][tx * 2 + 1];
      g[0][0] = fmaf(a0, b0, g[0][0]);
      g[0][1] = fmaf(a0, b1, g[0][1]);
      g[1][0] = fmaf(a1, b0, g[1][0]);
      g[1][1] = fmaf(a1, b1, g[1][1]);
      if (SWIGLU) {
        const float c0 = Bs1[kk][tx * 2], c1 = Bs1[kk][tx * 2 + 1];
        up[0][0] = fmaf(a0, c0, up[0][0]);
        up[0][1] = fmaf(a0, c1, up[0][1]);
        up[1][0] = fmaf(a1, c0, up[1][0]);
        up[1][1] = fmaf(a1, c1, up[1][1]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = ty * 2 + i;
    if (r >= nrows) continue;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int n = n0 + tx * 2 + j;
      if (n >= N) continue;
      float v = g[i][j];
      if (SWIGLU) v = v / (1.f + expf(-v)) * up[i][j];  // SiLU(gate) * up
      out[(row0 + r) * N + n] = v;
    }
  }
}

cudaError_t launch_ffn_simt_f32(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                                const void* W_up, const void* W_down, void* act, void* Y, int32_t* status,
                                cudaStream_t s) {
  if (p.Tk == 0) return cudaSuccess;
  const int64_t mslots = (p.Tk + SB - 1) / SB + p.E;  // >= sum_e ceil(n_e / SB) for any split of Tk rows
  if (mslots > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 g1(static_cast<unsigned>(mslots), (p.d_e + SB - 1) / SB);
  ffn_simt_f32<true><<<g1, 256, 0, s>>>(static_cast<const float*>(X), static_cast<const float*>(W_gate),
                                        static_cast<const float*>(W_up), offsets, p.E, p.h, p.d_e, p.Tk,
                                        static_cast<float*>(act), status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 g2(static_cast<unsigned>(mslots), (p.h + SB - 1) / SB);
  ffn_simt_f32<false><<<g2, 256, 0, s>>>(static_cast<const float*>(act), static_cast<const float*>(W_down), nullptr,
                                         offsets, p.E, p.d_e, p.h, p.Tk, static_cast<float*>(Y), status);
  return cudaGetLastError();
}

}  // namespace moe
