// Combine back into token order with the residual, and the load statistics.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 从稠密 FFN 到 MoE:
// h'_t = u_t + sum_i g_{i,t} FFN_i(u_t); section 路由器：打分、top-k、加权求和,
// shapes listing: the index_add of the gate-weighted expert rows into token
// order; section 专家容量与丢 token: a dropped pair adds nothing (residual only);
// section 负载均衡辅助损失：推导与梯度: f_i, P_i = (1/T) sum_t s_{i,t} and
// E * sum_i f_i P_i.
//
// combine_rows: one warp per token, 16-byte vectors; float32 accumulation of
// u_t + g_0 y_0 + g_1 y_1 + ... in choice order, rounded once.
// load_stats: one block; P_i sums the router's per-block partials in a fixed
// order (lane-strided then a butterfly), so it is identical from run to run.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int COMBINE_UNROLL = 2;

template <typename T>
__global__ void __launch_bounds__(256) combine_rows(const uint4* __restrict__ U, const uint4* __restrict__ Y,
                                                    const int32_t* __restrict__ slot_row,
                                                    const float* __restrict__ gate, uint4* __restrict__ out, int64_t n_tok,
                                                    int k, int vpr, int64_t rows_cap, int32_t* status) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < n_tok; t += warps) {
    int32_t my_row = -1;
    float my_g = 0.f;
    if (lane < k) {
      my_row = slot_row[t * k + lane];
      my_g = gate[t * k + lane];
      if (my_row < -1 || my_row >= rows_cap) {
        set_status(status, MOE_DEV_BAD_ROW);
        my_row = -1;
      }
    }
    // warp-uniform trip count: every lane reaches the shuffles below
    for (int base = 0; base < vpr; base += 32 * COMBINE_UNROLL) {
      float acc[COMBINE_UNROLL][N];
#pragma unroll
      for (int u = 0; u < COMBINE_UNROLL; ++u) {
        const int v = base + lane + 32 * u;
        if (v < vpr) Vec16<T>::unpack(ldg_stream(U + t * vpr + v), acc[u]);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (r < 0) continue;
#pragma unroll
        for (int u = 0; u < COMBINE_UNROLL; ++u) {
          const int v = base + lane + 32 * u;
          if (v < vpr) {
            float y[N];
            Vec16<T>::unpack(ldg_stream(Y + static_cast<int64_t>(r) * vpr + v), y);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[u][i] = fmaf(g, y[i], acc[u][i]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < COMBINE_UNROLL; ++u) {
        const int v = base + lane + 32 * u;
        if (v < vpr) out[t * vpr + v] = Vec16<T>::pack(acc[u]);
      }
    }
  }
}

constexpr int STATS_THREADS = 1024;

__global__ void __launch_bounds__(STATS_THREADS) load_stats(const float* __restrict__ ppart, int n_parts,
                                                            const int32_t* __restrict__ counts_routed, int64_t n_tok,
                                                            int k, int E, float* __restrict__ f,
                                                            float* __restrict__ P, float* __restrict__ aux) {
  __shared__ float fp[1024];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nwarps = blockDim.x / 32;
  for (int e = warp; e < E; e += nwarps) {
    float s = 0.f;
    for (int b = lane; b < n_parts; b += 32) s += ppart[static_cast<int64_t>(b) * E + e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const float Pi = n_tok > 0 ? s / static_cast<float>(n_tok) : 0.f;
      const float fi = n_tok > 0 ? static_cast<float>(counts_routed[e]) / static_cast<float>(n_tok * k) : 0.f;
      P[e] = Pi;
      f[e] = fi;
      fp[e] = fi * Pi;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int e = 0; e < E; ++e) a += fp[e];
    *aux = static_cast<float>(E) * a;
  }
}

cudaError_t launch_combine(const Plan& p, const void* U, const void* Y, const int32_t* slot_row, const float* gate,
                           const int32_t* counts_routed, void* out, float* f, float* P, float* aux, uint8_t* ws,
                           cudaStream_t s) {
  int32_t* status = ws_status(p, ws);
  if (p.T > 0) {
    const int vpr = p.h * (p.bf16 ? 2 : 4) / 16;
    const int64_t want = (p.T + 7) / 8;
    const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
    if (p.bf16)
      combine_rows<bf16><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(U), static_cast<const uint4*>(Y), slot_row,
                                                gate, static_cast<uint4*>(out), p.T, p.k, vpr, p.Tk, status);
    else
      combine_rows<float><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(U), static_cast<const uint4*>(Y), slot_row,
                                                 gate, static_cast<uint4*>(out), p.T, p.k, vpr, p.Tk, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const float* ppart = reinterpret_cast<const float*>(ws + p.ws_ppart);
  load_stats<<<1, STATS_THREADS, 0, s>>>(ppart, p.T > 0 ? p.sel_blocks : 0, counts_routed, p.T, p.k, p.E, f, P, aux);
  return cudaGetLastError();
}

}  // namespace moe
