// Combine back into token order with the residual, and the load statistics.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 从稠密 FFN 到 MoE:
// h'_t = u_t + sum_i g_{i,t} FFN_i(u_t); section 路由器：打分、top-k、加权求和,
// shapes listing: the index_add of the gate-weighted expert rows into token
// order; section 专家容量与丢 token: a dropped pair adds nothing (residual only);
// section 负载均衡辅助损失：推导与梯度: f_i, P_i = (1/T) sum_t s_{i,t} and
// E * sum_i f_i P_i.
//
// combine_stats: one launch.  One warp per token, 16-byte vectors; float32 accumulation of
// u_t + (shared experts' rows) + g_0 y_0 + g_1 y_1 + ... in choice order, rounded once (section
// 细粒度专家与共享专家: h'_t = u_t + sum_s FFN_s(u_t) + sum_i g_{i,t} FFN_i(u_t)).  The block that
// finishes last forms f_i, P_i, aux and the z-loss from the router's per-block sums in a fixed
// order, so they are identical from run to run.
// balance_bias_update: the loss-free balancing step of section 无辅助损失的负载均衡.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_UNROLL = 2;   // 4 measured slower with k = 6..8
constexpr int STAT_GROUPS = 32;     // first-level slices of the statistics reduction

// Row combine and statistics in one launch.
//   Rows: one warp per token (grid-stride), 16-byte vectors; float32 accumulation of u_t, then the
//   shared experts' rows in order, then g_j y_j for j ascending, rounded once.  Few registers keep
//   many warps resident, which is what keeps enough loads in flight.
//   Statistics in two levels: the first `groups` blocks each add a slice of the rows of the router's
//   per-block score sums, every column, in row order; the block that finishes last (an atomic
//   count; nobody waits) adds those partial rows in group order (P_i, and the z-loss in column E),
//   forms f_i from the routed counts and aux = E sum_i f_i P_i in expert order, and resets the
//   count for the next call.  Every result is the same from run to run.
template <typename T>
__global__ void __launch_bounds__(COMBINE_THREADS, 4) combine_stats(
    const uint4* __restrict__ U, const uint4* __restrict__ Y, const uint4* __restrict__ Y_shared, int n_shared,
    const int32_t* __restrict__ slot_row, const float* __restrict__ gate, uint4* __restrict__ out, int64_t n_tok,
    int k, int vpr, int64_t rows_cap, int32_t* status, const float* __restrict__ ppart,
    const int32_t* __restrict__ ppart_rows, const int32_t* __restrict__ counts_routed, int E, float* __restrict__ f,
    float* __restrict__ P, float* __restrict__ aux, float* __restrict__ z_loss, int32_t* __restrict__ done_count,
    float* __restrict__ part2, int groups, int spu) {
  constexpr int N = Vec16<T>::N;
  // statistics, first level: block g < groups adds rows [g R, (g+1) R) of the router's per-block
  // sums, every column, in row order (loads issued eight at a time)
  if (static_cast<int>(blockIdx.x) < groups && n_tok > 0) {
    const int n_parts = *ppart_rows;
    const int R = (n_parts + groups - 1) / groups;
    const int b0 = min(n_parts, static_cast<int>(blockIdx.x) * R), b1 = min(n_parts, b0 + R);
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      float s = 0.f;
      for (int b = b0; b < b1; b += 8) {
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = b + q < b1 ? ppart[static_cast<int64_t>(b + q) * (E + 1) + e] : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (b + q < b1) s += v[q];
      }
      part2[static_cast<int64_t>(blockIdx.x) * (E + 1) + e] = s;
    }
  }

  // rows: warp tasks of `spu` consecutive 32 x COMBINE_UNROLL-vector pieces of one token row (the
  // whole row when there are tokens enough for every warp; fewer pieces when there are not, so that
  // short batches still spread over all warps)
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  const int pieces = (vpr + 32 * COMBINE_UNROLL - 1) / (32 * COMBINE_UNROLL);
  const int tasks_per_tok = (pieces + spu - 1) / spu;
  // task = t * tasks_per_tok + q advances by `warps` a step: (t, q) is carried along without division
  const int64_t first = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
  const int64_t dt = warps / tasks_per_tok;
  const int dq = static_cast<int>(warps - dt * tasks_per_tok);
  int64_t t = first / tasks_per_tok;
  int q = static_cast<int>(first - t * tasks_per_tok);
  for (; t < n_tok; t += dt, q += dq) {
    if (q >= tasks_per_tok) {
      q -= tasks_per_tok;
      ++t;
      if (t >= n_tok) break;
    }
    const int v_lo = q * spu * 32 * COMBINE_UNROLL;
    const int v_hi = min(vpr, (q + 1) * spu * 32 * COMBINE_UNROLL);
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
    for (int base = v_lo; base < v_hi; base += 32 * COMBINE_UNROLL) {
      float acc[COMBINE_UNROLL][N];
#pragma unroll
      for (int u = 0; u < COMBINE_UNROLL; ++u) {
        const int v = base + lane + 32 * u;
        if (v < v_hi) Vec16<T>::unpack(ldg_stream(U + t * vpr + v), acc[u]);
      }
      for (int sh = 0; sh < n_shared; ++sh) {
#pragma unroll
        for (int u = 0; u < COMBINE_UNROLL; ++u) {
          const int v = base + lane + 32 * u;
          if (v < v_hi) {
            float y[N];
            Vec16<T>::unpack(ldg_stream(Y_shared + (static_cast<int64_t>(sh) * n_tok + t) * vpr + v), y);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[u][i] += y[i];
          }
        }
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
        const float g = __shfl_sync(0xffffffffu, my_g, j);
        if (r < 0) continue;
#pragma unroll
        for (int u = 0; u < COMBINE_UNROLL; ++u) {
          const int v = base + lane + 32 * u;
          if (v < v_hi) {
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
        if (v < v_hi) out[t * vpr + v] = Vec16<T>::pack(acc[u]);
      }
    }
  }

  // statistics, by the last block to finish
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(done_count, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  // second level: the groups' partial sums in group order
  const int G = n_tok > 0 ? groups : 0;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    float s = 0.f;
    for (int b = 0; b < G; b += 8) {
      float v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = b + q < G ? __ldcg(part2 + static_cast<int64_t>(b + q) * (E + 1) + e) : 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (b + q < G) s += v[q];
    }
    const float mean = n_tok > 0 ? s / static_cast<float>(n_tok) : 0.f;
    if (e < E) {
      P[e] = mean;
      f[e] = n_tok > 0 ? static_cast<float>(counts_routed[e]) / static_cast<float>(n_tok * k) : 0.f;
    } else if (z_loss) {
      *z_loss = mean;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int i = 0; i < E; ++i) a += f[i] * P[i];
    *aux = static_cast<float>(E) * a;
    *done_count = 0;  // ready for the next call
  }
}

// b_i += u * sign(mean(c) - c_i), the sign taken exactly on integers: sign(sum_j c_j - E c_i).
__global__ void __launch_bounds__(1024) balance_bias_update(int E, const int32_t* __restrict__ counts, float u,
                                                            float* __restrict__ bias) {
  __shared__ long long part[32];
  long long s = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s += counts[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += part[w];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const long long d = total - static_cast<long long>(E) * counts[e];
    bias[e] += d > 0 ? u : d < 0 ? -u : 0.f;
  }
}

cudaError_t launch_balance_bias_update(int E, const int32_t* counts_routed, float u, float* bias, cudaStream_t s) {
  balance_bias_update<<<1, 1024, 0, s>>>(E, counts_routed, u, bias);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Plan& p, const void* U, const void* Y, const void* Y_shared, const int32_t* slot_row,
                           const float* gate, const int32_t* counts_routed, void* out, float* f, float* P, float* aux,
                           float* z_loss, uint8_t* ws, cudaStream_t s) {
  int32_t* status = ws_status(p, ws);
  const float* ppart = reinterpret_cast<const float*>(ws + p.ws_ppart);
  int32_t* done = reinterpret_cast<int32_t*>(ws + p.ws_status + 128);
  float* part2 = reinterpret_cast<float*>(ws + p.ws_stats2);
  const int vpr = p.h * (p.bf16 ? 2 : 4) / 16;
  // one warp per token, or per piece of a token row when the tokens are few (at most 8 blocks an SM)
  const int pieces_per_row = (vpr + 32 * COMBINE_UNROLL - 1) / (32 * COMBINE_UNROLL);
  const int64_t want = (p.T * pieces_per_row + 7) / 8;
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8)));
  const int n_sh = Y_shared ? p.n_shared : 0;
  const uint4* ysh = static_cast<const uint4*>(Y_shared);
  const int groups = std::min(STAT_GROUPS, blocks);
  // pieces of a row per warp task: the whole row unless that leaves warps idle
  const int pieces = (vpr + 32 * COMBINE_UNROLL - 1) / (32 * COMBINE_UNROLL);
  const int64_t total_warps = static_cast<int64_t>(blocks) * (COMBINE_THREADS / 32);
  const int64_t want_tasks = total_warps * 2;
  int spu = pieces;
  while (spu > 1 && p.T * ((pieces + spu - 1) / spu) < want_tasks) spu = (spu + 1) / 2;
  if (p.bf16)
    combine_stats<bf16><<<blocks, COMBINE_THREADS, 0, s>>>(
        static_cast<const uint4*>(U), static_cast<const uint4*>(Y), ysh, n_sh, slot_row, gate,
        static_cast<uint4*>(out), p.T, p.k, vpr, p.Tk, status, ppart, ws_ppart_rows(p, ws), counts_routed, p.E, f, P,
        aux, z_loss, done, part2, groups, spu);
  else
    combine_stats<float><<<blocks, COMBINE_THREADS, 0, s>>>(
        static_cast<const uint4*>(U), static_cast<const uint4*>(Y), ysh, n_sh, slot_row, gate,
        static_cast<uint4*>(out), p.T, p.k, vpr, p.Tk, status, ppart, ws_ppart_rows(p, ws), counts_routed, p.E, f, P,
        aux, z_loss, done, part2, groups, spu);
  return cudaGetLastError();
}

}  // namespace moe
