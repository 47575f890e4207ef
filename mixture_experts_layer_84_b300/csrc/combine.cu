// Combine back into token order with the residual, and the load statistics.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 从稠密 FFN 到 MoE:
// h'_t = u_t + sum_i g_{i,t} FFN_i(u_t); section 路由器：打分、top-k、加权求和,
// shapes listing: the index_add of the gate-weighted expert rows into token
// order; section 专家容量与丢 token: a dropped pair adds nothing (residual only);
// section 负载均衡辅助损失：推导与梯度: f_i, P_i = (1/T) sum_t s_{i,t} and
// E * sum_i f_i P_i.
//
// combine_stats: one launch.  Each block streams its (token, row segment) units through a
// shared-memory ring with bulk copies -- the segment of u_t, of the shared experts' rows and of the
// token's kept expert rows -- and adds u_t + (shared experts' rows) + g_0 y_0 + g_1 y_1 + ... in
// float32, in choice order, rounded once (section 细粒度专家与共享专家: h'_t = u_t + sum_s FFN_s(u_t)
// + sum_i g_{i,t} FFN_i(u_t)).  The block that finishes last forms f_i, P_i, aux and the z-loss
// from the router's per-block sums in a fixed order, so they are identical from run to run.
// balance_bias_update: the loss-free balancing step of section 无辅助损失的负载均衡.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

constexpr int COMBINE_THREADS = 256;
constexpr int STAT_GROUPS = 32;                      // first-level slices of the statistics reduction
constexpr uint32_t COMBINE_UNIT_BYTES = 24 * 1024;   // source bytes of one work unit, at most
constexpr uint32_t COMBINE_RING_BYTES = 192 * 1024;  // the ring of unit slots
constexpr int COMBINE_MAX_SLOTS = 32;
constexpr uint64_t COMBINE_WAIT_LIMIT_NS = 2000000000ull;

// Row combine and statistics in one launch.
//   Rows: a work unit is one column segment of one token's row (segs segments per row, each
//   seg_bytes long).  Its sources -- the segment of u_t, of each shared expert's row and of each
//   kept expert row of the token -- are copied into a slot of a shared-memory ring with bulk
//   copies (cp.async.bulk, completion on the slot's mbarrier), issued by one thread up to nslots - 1
//   units ahead.  Every thread then adds its 16-byte vectors of the unit in float32 in a fixed order
//   -- u_t, the shared rows in order, then g_j y_j for j ascending -- rounds once and stores them
//   (consecutive threads, consecutive vectors).  A block takes a contiguous range of units; the
//   routing of its tokens (slot_row, gate) is staged in shared memory first.
//   Statistics in two levels: the first `groups` blocks each add a slice of the rows of the router's
//   per-block score sums, every column, in row order; the block that finishes last (an atomic
//   count; nobody waits) adds those partial rows in group order (P_i, and the z-loss in column E),
//   forms f_i from the routed counts and aux = E sum_i f_i P_i in expert order, and resets the
//   count for the next call.  Every result is the same from run to run.
struct CombineGeo {
  int segs;            // column segments per row
  uint32_t seg_bytes;  // bytes of one segment of one row
  int nsrc;            // source rows of a unit, at most: 1 + n_shared + k
  uint32_t slot_bytes; // nsrc * seg_bytes
  int nslots;
};

inline CombineGeo combine_geo(int h, int elem, int n_shared, int k) {
  CombineGeo g;
  const uint32_t row_bytes = static_cast<uint32_t>(h) * elem;
  g.nsrc = 1 + n_shared + k;
  g.segs = 1;
  while (static_cast<uint64_t>(g.nsrc) * row_bytes / g.segs > COMBINE_UNIT_BYTES && row_bytes % (g.segs * 2 * 16) == 0)
    g.segs *= 2;
  g.seg_bytes = row_bytes / g.segs;
  g.slot_bytes = g.nsrc * g.seg_bytes;
  g.nslots = static_cast<int>(std::max<uint32_t>(2, std::min<uint32_t>(COMBINE_MAX_SLOTS, COMBINE_RING_BYTES / g.slot_bytes)));
  return g;
}

template <typename T>
__global__ void __launch_bounds__(COMBINE_THREADS, 1) combine_stats(
    const uint8_t* __restrict__ U, const uint8_t* __restrict__ Y, const uint8_t* __restrict__ Y_shared, int n_shared,
    const int32_t* __restrict__ slot_row, const float* __restrict__ gate, uint8_t* __restrict__ out, int64_t n_tok,
    int k, int segs, uint32_t seg_bytes, int nslots, int64_t units_per_block, int64_t rows_cap, int32_t* status,
    const float* __restrict__ ppart, const int32_t* __restrict__ ppart_rows, const int32_t* __restrict__ counts_routed,
    int E, float* __restrict__ f, float* __restrict__ P, float* __restrict__ aux, float* __restrict__ z_loss,
    int32_t* __restrict__ done_count, float* __restrict__ part2, int groups) {
  constexpr int N = Vec16<T>::N;
  const uint32_t row_bytes = seg_bytes * segs;
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

  // rows
  const int64_t units = n_tok * segs;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * units_per_block;
  const int64_t u1 = min(units, u0 + units_per_block);
  if (u0 < u1) {
    extern __shared__ __align__(128) uint8_t csm[];
    const int64_t t_lo = u0 / segs, t_hi = (u1 - 1) / segs;
    const int nt = static_cast<int>(t_hi - t_lo + 1);
    int32_t* rows_s = reinterpret_cast<int32_t*>(csm);               // [nt][k]
    float* gate_s = reinterpret_cast<float*>(rows_s + nt * k);       // [nt][k]
    uint8_t* ring = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(gate_s + nt * k) + 127) & ~static_cast<uintptr_t>(127));
    const uint32_t slot_bytes = seg_bytes * (1 + n_shared + k);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + static_cast<size_t>(nslots) * slot_bytes);
    __shared__ int abort_s;
    for (int i = threadIdx.x; i < nt * k; i += blockDim.x) {
      int32_t r = slot_row[t_lo * k + i];
      if (r < -1 || r >= rows_cap) {
        set_status(status, MOE_DEV_BAD_ROW);
        r = -1;
      }
      rows_s[i] = r;
      gate_s[i] = gate[t_lo * k + i];
    }
    if (threadIdx.x == 0) {
      abort_s = 0;
      for (int i = 0; i < nslots; ++i) ptx::mbar_init(&full[i], 1);
      ptx::fence_mbarrier_init();
      ptx::fence_proxy_async_smem();
    }
    __syncthreads();
    const int64_t n_units = u1 - u0;
    // slot layout of unit i: u_t, the shared rows, then one segment per choice j (kept or not)
    auto issue = [&](int64_t i) {
      const int64_t u = u0 + i;
      const int64_t t = u / segs;
      const uint32_t off = static_cast<uint32_t>(u - t * segs) * seg_bytes;
      uint8_t* slot = ring + static_cast<size_t>(i % nslots) * slot_bytes;
      uint64_t* bar = &full[i % nslots];
      const int32_t* rr = rows_s + (t - t_lo) * k;
      uint32_t bytes = seg_bytes * (1 + n_shared);
      for (int j = 0; j < k; ++j) bytes += rr[j] >= 0 ? seg_bytes : 0;
      ptx::mbar_arrive_expect_tx(bar, bytes);
      ptx::bulk_load(slot, U + t * row_bytes + off, seg_bytes, bar);
      for (int sh = 0; sh < n_shared; ++sh)
        ptx::bulk_load(slot + (1 + sh) * seg_bytes, Y_shared + (static_cast<int64_t>(sh) * n_tok + t) * row_bytes + off,
                       seg_bytes, bar);
      for (int j = 0; j < k; ++j)
        if (rr[j] >= 0)
          ptx::bulk_load(slot + (1 + n_shared + j) * seg_bytes, Y + static_cast<int64_t>(rr[j]) * row_bytes + off,
                         seg_bytes, bar);
    };
    int64_t issued = 0;
    if (threadIdx.x == 0)
      for (; issued < static_cast<int64_t>(nslots - 1) && issued < n_units; ++issued) issue(issued);
    const int vps = static_cast<int>(seg_bytes / 16);
    int64_t i = 0;
    for (; i < n_units; ++i) {
      if (threadIdx.x == 0) {
        const uint64_t tw = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(&full[i % nslots], static_cast<uint32_t>((i / nslots) & 1))) {
          if (ptx::globaltimer_ns() - tw > COMBINE_WAIT_LIMIT_NS) {
            abort_s = 1;
            break;
          }
        }
      }
      __syncthreads();  // the unit has landed (or the wait gave up); the previous slot is free
      if (abort_s) break;
      if (threadIdx.x == 0 && issued < n_units) issue(issued++);  // into the slot of unit i - 1
      const int64_t u = u0 + i;
      const int64_t t = u / segs;
      const uint32_t off = static_cast<uint32_t>(u - t * segs) * seg_bytes;
      const uint4* slot = reinterpret_cast<const uint4*>(ring + static_cast<size_t>(i % nslots) * slot_bytes);
      const int32_t* rr = rows_s + (t - t_lo) * k;
      const float* gg = gate_s + (t - t_lo) * k;
      uint4* dst = reinterpret_cast<uint4*>(out + t * row_bytes + off);
      for (int v = threadIdx.x; v < vps; v += blockDim.x) {
        float acc[N];
        Vec16<T>::unpack(slot[v], acc);
        for (int sh = 0; sh < n_shared; ++sh) {
          float y[N];
          Vec16<T>::unpack(slot[(1 + sh) * vps + v], y);
#pragma unroll
          for (int q = 0; q < N; ++q) acc[q] += y[q];
        }
        for (int j = 0; j < k; ++j) {
          if (rr[j] < 0) continue;
          float y[N];
          Vec16<T>::unpack(slot[(1 + n_shared + j) * vps + v], y);
          const float g = gg[j];
#pragma unroll
          for (int q = 0; q < N; ++q) acc[q] = fmaf(g, y[q], acc[q]);
        }
        dst[v] = Vec16<T>::pack(acc);
      }
    }
    if (abort_s && threadIdx.x == 0) {
      set_status(status, MOE_DEV_TIMEOUT);
      // copies still in flight (units i .. issued - 1) land in this block's shared memory: wait for
      // them (bounded)
      for (int64_t q = i; q < issued; ++q) {
        const uint64_t tw = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(&full[q % nslots], static_cast<uint32_t>((q / nslots) & 1)) &&
               ptx::globaltimer_ns() - tw < COMBINE_WAIT_LIMIT_NS) {
        }
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
  const int n_sh = Y_shared ? p.n_shared : 0;
  CombineGeo g = combine_geo(p.h, p.bf16 ? 2 : 4, n_sh, p.k);
  const int sms = current_sm_count();
  const int64_t units = p.T * g.segs;
  // one block per SM, more when a block's routing metadata would pass 24 KB of shared memory
  const int64_t tok_cap = std::max<int64_t>(1, 24 * 1024 / (8 * p.k));
  const int64_t want = std::max<int64_t>(sms, (p.T + tok_cap - 1) / tok_cap);
  const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(units, want)));
  const int64_t per = (units + blocks - 1) / blocks;
  g.nslots = static_cast<int>(std::max<int64_t>(2, std::min<int64_t>(g.nslots, per + 1)));  // no idle slots
  const int64_t tok_span = per / g.segs + 2;  // tokens a block's unit range touches, at most
  const size_t smem = sizeof(int32_t) * 2 * static_cast<size_t>(tok_span) * p.k + 128 +
                      static_cast<size_t>(g.nslots) * g.slot_bytes + 8 * static_cast<size_t>(g.nslots);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const int groups = std::min(STAT_GROUPS, blocks);
  auto kern = p.bf16 ? combine_stats<bf16> : combine_stats<float>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<blocks, COMBINE_THREADS, smem, s>>>(
      static_cast<const uint8_t*>(U), static_cast<const uint8_t*>(Y), static_cast<const uint8_t*>(Y_shared), n_sh,
      slot_row, gate, static_cast<uint8_t*>(out), p.T, p.k, g.segs, g.seg_bytes, g.nslots, per, p.Tk, status, ppart,
      ws_ppart_rows(p, ws), counts_routed, p.E, f, P, aux, z_loss, done, part2, groups);
  return cudaGetLastError();
}

}  // namespace moe
