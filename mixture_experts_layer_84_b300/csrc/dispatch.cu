// Capacity-limited dispatch: slots, drop mask, expert offsets and the row
// copy X[row] = U[token].
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 专家容量与丢 token:
// C = ceil(CF * T * k / E); slots of an expert are filled in token order and
// the overflow is dropped; with top-k every token's first choice is placed
// before any second choice.  Section 路由器：打分、top-k、加权求和, shapes
// listing: the (token, expert) pairs are grouped by expert and X = U[token of
// each row], with per-expert counts and offsets for the grouped FFN.
//
// The pairs are walked in priority order p = 0 .. T*k-1 (choice-major:
// p = j*T + t; token-major: p = t*k + j).  The slot of a pair is the number
// of earlier pairs with the same expert -- an exclusive prefix count, so it is
// computed with scans, never with an atomic whose order could leak into the
// result.  Choice-major priority (the default) takes three launches, dispatch_hist,
// dispatch_colscan and dispatch_place (two when the histograms are small, one when the batch is),
// described where they are defined.  Token-major
// priority and the workspace-free entry point take these four:
//   dispatch_count   per chunk of positions, a histogram over experts;
//   dispatch_scan    one block: per expert, the exclusive prefix over chunks,
//                    the routed/kept counts, and offsets = exclusive scan of
//                    the kept counts;
//   dispatch_assign  per chunk, per warp: ranks among equal experts inside the
//                    warp (match_any) on top of the chunk and warp bases;
//                    writes slot_row and row_token;
//   dispatch_scatter one warp per token, 16-byte copies: each U row is read
//                    once and written to the (up to k) rows it was kept in.
//                    Skipped when X is NULL: the FP8 dispatch (fp8.cu) copies
//                    quantised rows instead, and the gathered first GEMM reads
//                    the rows of U itself.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

constexpr int DISPATCH_THREADS = 256;
constexpr int SCATTER_UNROLL = 4;
constexpr int DISPATCH_WARPS = DISPATCH_THREADS / 32;
constexpr int SCAN_THREADS = 1024;

__device__ __forceinline__ void position_to_pair(int64_t p, int64_t T, int k, int priority, int64_t* t, int* j) {
  if (priority == MOE_PRIORITY_CHOICE_MAJOR) {
    *j = static_cast<int>(p / T);
    *t = p - static_cast<int64_t>(*j) * T;
  } else {
    *t = p / k;
    *j = static_cast<int>(p - *t * k);
  }
}

__global__ void __launch_bounds__(DISPATCH_THREADS) dispatch_count(const int32_t* __restrict__ idx, int64_t T, int k,
                                                                   int E, int priority, int chunk,
                                                                   int32_t* __restrict__ hist, int32_t* status) {
  extern __shared__ int32_t h_cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h_cnt[e] = 0;
  __syncthreads();
  const int64_t Tk = T * k;
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t p1 = min(p0 + chunk, Tk);
  bool bad = false;
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    int64_t t;
    int j;
    position_to_pair(p, T, k, priority, &t, &j);
    const int e = idx[t * k + j];
    if (e >= 0 && e < E)
      atomicAdd(&h_cnt[e], 1);  // integer counts: the order of the adds does not matter
    else
      bad = true;
  }
  if (bad) set_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[static_cast<int64_t>(blockIdx.x) * E + e] = h_cnt[e];
}

// One block.  Thread (g, e), tid = g*E + e, owns chunks [g*nc/G, (g+1)*nc/G) of expert e.
// On return hist[c][e] holds the exclusive prefix of expert e over chunks < c.
__global__ void __launch_bounds__(SCAN_THREADS) dispatch_scan(int32_t* __restrict__ hist, int n_chunks, int E, int G,
                                                              int64_t C, int64_t Tk,
                                                              int32_t* __restrict__ counts_routed,
                                                              int32_t* __restrict__ counts_kept,
                                                              int32_t* __restrict__ offsets,
                                                              int64_t* __restrict__ n_dropped) {
  __shared__ int32_t gsum[SCAN_THREADS];
  __shared__ int32_t kept_s[SCAN_THREADS];
  const int tid = threadIdx.x;
  const int g = tid / E, e = tid % E;
  const bool active = g < G;
  int cb = 0, ce = 0;
  if (active) {
    cb = static_cast<int>((static_cast<int64_t>(n_chunks) * g) / G);
    ce = static_cast<int>((static_cast<int64_t>(n_chunks) * (g + 1)) / G);
    int32_t s = 0;
    for (int c = cb; c < ce; ++c) s += hist[static_cast<int64_t>(c) * E + e];
    gsum[tid] = s;
  }
  __syncthreads();
  if (tid < E) {
    int32_t run = 0;
    for (int gg = 0; gg < G; ++gg) {
      const int32_t v = gsum[gg * E + tid];
      gsum[gg * E + tid] = run;
      run += v;
    }
    counts_routed[tid] = run;
    const int32_t kept = static_cast<int32_t>(min(static_cast<int64_t>(run), C));
    counts_kept[tid] = kept;
    kept_s[tid] = kept;
  }
  __syncthreads();
  if (active) {
    int32_t run = gsum[tid];
    for (int c = cb; c < ce; ++c) {
      const int64_t o = static_cast<int64_t>(c) * E + e;
      const int32_t v = hist[o];
      hist[o] = run;
      run += v;
    }
  }
  if (tid < 32) {  // offsets = exclusive scan of the kept counts (warp 0)
    const int per = (E + 31) / 32;
    const int lo = min(E, tid * per), hi = min(E, lo + per);
    int32_t s = 0;
    for (int i = lo; i < hi; ++i) s += kept_s[i];
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (tid >= o) incl += y;
    }
    int32_t run = incl - s;
    for (int i = lo; i < hi; ++i) {
      offsets[i] = run;
      run += kept_s[i];
    }
    const int32_t A = __shfl_sync(0xffffffffu, incl, 31);
    if (tid == 0) {
      offsets[E] = A;
      *n_dropped = Tk - A;
    }
  }
}

__global__ void __launch_bounds__(DISPATCH_THREADS) dispatch_assign(
    const int32_t* __restrict__ idx, int64_t T, int k, int E, int priority, int chunk,
    const int32_t* __restrict__ base, const int32_t* __restrict__ offsets, int64_t C,
    int32_t* __restrict__ slot_row, int32_t* __restrict__ row_token) {
  extern __shared__ int32_t wc[];  // [DISPATCH_WARPS][E]
  for (int i = threadIdx.x; i < DISPATCH_WARPS * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t Tk = T * k;
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t p1 = min(p0 + chunk, Tk);
  const int seg = chunk / DISPATCH_WARPS;
  const int64_t q0 = p0 + static_cast<int64_t>(warp) * seg;
  const int64_t q1 = min(q0 + seg, p1);
  int32_t* my = wc + warp * E;
  const uint32_t lt_mask = (1u << lane) - 1u;

  // pass 1: per-warp counts (q0, q1 are warp-uniform)
  for (int64_t q = q0; q < q1; q += 32) {
    const int64_t p = q + lane;
    int e = -1;
    if (p < q1) {
      int64_t t;
      int j;
      position_to_pair(p, T, k, priority, &t, &j);
      e = idx[t * k + j];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // warp bases on top of the chunk base, warps in order
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t run = base[static_cast<int64_t>(blockIdx.x) * E + e];
    for (int w = 0; w < DISPATCH_WARPS; ++w) {
      const int32_t v = wc[w * E + e];
      wc[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // pass 2: slot = warp base + rank among the equal experts of earlier lanes
  for (int64_t q = q0; q < q1; q += 32) {
    const int64_t p = q + lane;
    int e = -1;
    int64_t t = 0;
    int j = 0;
    if (p < q1) {
      position_to_pair(p, T, k, priority, &t, &j);
      e = idx[t * k + j];
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int32_t slot = e >= 0 ? my[e] + __popc(peers & lt_mask) : -1;
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
    if (p < q1) {
      const int64_t pair = t * k + j;
      if (e >= 0 && slot < C) {
        const int32_t row = offsets[e] + slot;
        slot_row[pair] = row;
        row_token[row] = static_cast<int32_t>(t);
      } else {
        slot_row[pair] = -1;
      }
    }
  }
}

// One warp per token (grid-stride): lane l copies 16-byte vectors l, l+32, ...
__global__ void __launch_bounds__(256) dispatch_scatter(const uint4* __restrict__ U, const int32_t* __restrict__ slot_row,
                                                        uint4* __restrict__ X, int64_t T, int k, int vpr) {
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < T; t += warps) {
    const int32_t my_row = lane < k ? slot_row[t * k + lane] : -1;
    const uint4* src = U + t * vpr;
    // warp-uniform trip count: every lane reaches the shuffles below
    for (int base = 0; base < vpr; base += 32 * SCATTER_UNROLL) {
      uint4 val[SCATTER_UNROLL];
#pragma unroll
      for (int u = 0; u < SCATTER_UNROLL; ++u) {
        const int v = base + lane + 32 * u;
        if (v < vpr) val[u] = ldg_stream(src + v);
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0) continue;
        uint4* dst = X + static_cast<int64_t>(r) * vpr;
#pragma unroll
        for (int u = 0; u < SCATTER_UNROLL; ++u) {
          const int v = base + lane + 32 * u;
          if (v < vpr) dst[v] = val[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Choice-major dispatch in three launches (two or one for small histograms or batches).  Pairs are
// grouped into token chunks of TC tokens; with every token's first choice before any second
// choice, the slot of pair (t, j) choosing expert e is
//   sum_{j' < j} cnt[j'][e]  +  sum_{chunks c' < c(t)} h[c'][j][e]  +  #{t' < t in t's chunk : idx[t'][j] = e},
// cnt[j][e] being the pairs of choice j that chose e over all tokens and h[c][j][e] those of chunk c.
//   dispatch_hist    per chunk, h[c][j][e];
//   dispatch_colscan one warp per (j, e) column: exclusive prefixes over the chunks and the column
//                    total; the block that finishes last (an atomic ticket, nobody waits) forms the
//                    choice bases, the routed and kept counts, the offsets and n_dropped;
//   dispatch_place  per chunk and choice: ranks among equal experts inside each warp (match_any)
//                   on top of the chunk's base and the earlier warps' counts; writes slot_row and
//                   row_token; meanwhile the chunk's U rows (contiguous) arrive in shared memory
//                   in large bulk loads, two buffers deep; then each warp writes 512-byte pieces
//                   of the staged rows to all of their kept rows with coalesced 16-byte stores
//                   (skipped when X is NULL).
// When the histograms are small (chunks x k x E <= 8192 counts), there is no column-scan launch:
// every placement block adds the raw chunk counts itself -- the chunks before its own, and all of
// them -- forms the choice bases and the offsets in shared memory, and block 0 writes the routed
// and kept counts, the offsets and n_dropped.  Integer sums: the same values as the scan's.  When
// the batch itself is small (T k <= 8192 expert ids) there is no histogram launch either: every
// placement block counts all the ids (those before its chunk, and all of them), so the dispatch is
// one launch.
constexpr int PLACE_THREADS = 256;
constexpr size_t COPY_SMEM_BYTES = 100 * 1024;       // shared memory of one dispatch_place block: two fit an SM
constexpr uint64_t COPY_WAIT_LIMIT_NS = 2000000000ull;
constexpr int PLACE_WARPS = PLACE_THREADS / 32;
constexpr int HIST_THREADS = 1024;
// chunks x k x E counts each placement block adds itself (measured: the 8-expert shape's 4096 take
// its dispatch from 28.7 to 20.5 us; the 128-expert shape's 32768 gained nothing over the scan)
constexpr int64_t SELF_SCAN_MAX = 8192;
constexpr int64_t SELF_COUNT_MAX = 8192;  // T k expert ids each placement block counts itself

__global__ void __launch_bounds__(HIST_THREADS) dispatch_hist(const int32_t* __restrict__ idx, int64_t T, int k,
                                                              int E, int tc, int32_t* __restrict__ hist,
                                                              int32_t* status) {
  extern __shared__ int32_t h_s[];  // [k][E]
  const int kE = k * E;
  for (int i = threadIdx.x; i < kE; i += blockDim.x) h_s[i] = 0;
  __syncthreads();
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tc;
  const int64_t t1 = min(t0 + tc, T);
  bool bad = false;
  for (int64_t i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int j = static_cast<int>(i % k);
    const int e = idx[i];
    if (e >= 0 && e < E)
      atomicAdd(&h_s[j * E + e], 1);  // integer counts: the order of the adds does not matter
    else
      bad = true;
  }
  if (bad) set_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  int32_t* mine = hist + static_cast<int64_t>(blockIdx.x) * kE;
  for (int i = threadIdx.x; i < kE; i += blockDim.x) mine[i] = h_s[i];
}

// One warp per (choice j, expert e) column of the chunk histograms: lane l adds the chunks
// [l m, (l+1) m), the warp scans the lane sums, and every chunk's entry becomes the exclusive prefix
// over the earlier chunks; the column total goes to cnt[j][e].  The block that finishes last (an
// atomic ticket, nobody waits) forms the choice bases (the pairs of earlier choices per expert),
// the routed and kept counts, the offsets and n_dropped, and resets the ticket.
__global__ void __launch_bounds__(256) dispatch_colscan(int32_t* __restrict__ hist, int n_chunks, int k, int E,
                                                        int64_t C, int64_t Tk, int32_t* __restrict__ ticket,
                                                        int32_t* __restrict__ counts_routed,
                                                        int32_t* __restrict__ counts_kept,
                                                        int32_t* __restrict__ offsets,
                                                        int64_t* __restrict__ n_dropped) {
  const int kE = k * E;
  const int lane = threadIdx.x % 32;
  const int col = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  int32_t* cnt = hist + static_cast<int64_t>(n_chunks + 1) * kE;  // [k][E] column totals
  if (col < kE) {
    const int m = (n_chunks + 31) / 32;
    const int c0 = min(n_chunks, lane * m), c1 = min(n_chunks, c0 + m);
    // up to 8 chunks a lane are loaded at once and kept in registers (one round trip)
    int32_t vals[8];
    int32_t s = 0;
    if (m <= 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) vals[q] = c0 + q < c1 ? hist[static_cast<int64_t>(c0 + q) * kE + col] : 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) s += vals[q];
    } else {
      for (int c = c0; c < c1; ++c) s += hist[static_cast<int64_t>(c) * kE + col];
    }
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int32_t run = incl - s;
    if (m <= 8) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (c0 + q < c1) hist[static_cast<int64_t>(c0 + q) * kE + col] = run;
        run += vals[q];
      }
    } else {
      for (int c = c0; c < c1; ++c) {
        const int64_t o = static_cast<int64_t>(c) * kE + col;
        const int32_t v = hist[o];
        hist[o] = run;
        run += v;
      }
    }
    if (lane == 31) cnt[col] = incl;
  }
  __shared__ int last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (!last) return;
  __threadfence();
  __shared__ int32_t kept_s[1024];
  int32_t* cbase = hist + static_cast<int64_t>(n_chunks) * kE;  // [k][E] choice bases
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t c[16];  // k <= 16: every choice's total loaded at once
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = j < k ? __ldcg(cnt + j * E + e) : 0;
    int32_t run = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < k) cbase[j * E + e] = run;
      run += c[j];
    }
    counts_routed[e] = run;
    const int32_t kept = static_cast<int32_t>(min(static_cast<int64_t>(run), C));
    counts_kept[e] = kept;
    kept_s[e] = kept;
  }
  __syncthreads();
  if (threadIdx.x < 32) {  // offsets = exclusive scan of the kept counts (warp 0)
    const int per = (E + 31) / 32;
    const int lo = min(E, lane * per), hi = min(E, lo + per);
    int32_t s = 0;
    for (int i = lo; i < hi; ++i) s += kept_s[i];
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int32_t run = incl - s;
    for (int i = lo; i < hi; ++i) {
      offsets[i] = run;
      run += kept_s[i];
    }
    const int32_t A = __shfl_sync(0xffffffffu, incl, 31);
    if (lane == 0) {
      offsets[E] = A;
      *n_dropped = Tk - A;
      *ticket = 0;  // ready for the next call
    }
  }
}

// stage_bases: 0 reads the chunk's bases from the scanned histogram, 1 stages them in shared memory,
// 2 computes them from the raw chunk counts (no column scan), 3 from the expert ids themselves (no
// histogram either; see above).
__global__ void __launch_bounds__(PLACE_THREADS) dispatch_place(
    const int32_t* __restrict__ idx, int64_t T, int k, int E, int tc, int n_chunks, int64_t C,
    const int32_t* __restrict__ hist, int32_t* __restrict__ offsets, int32_t* __restrict__ slot_row,
    int32_t* __restrict__ row_token, const void* __restrict__ U, void* __restrict__ X, uint32_t row_bytes, int nb,
    int32_t* status, int stage_bases, int32_t* __restrict__ counts_routed, int32_t* __restrict__ counts_kept,
    int64_t* __restrict__ n_dropped) {
  extern __shared__ int32_t sm[];
  int32_t* wc = sm;                          // [PLACE_WARPS][E]
  int32_t* rows_s = sm + PLACE_WARPS * E;    // [tc][k]
  int32_t* idx_s = rows_s + tc * k;          // [tc][k]: the chunk's expert ids
  int32_t* base_s = idx_s + tc * k;          // [k][E]: chunk prefix + choice base (when staged)
  int32_t* tot_s = base_s + k * E;           // self scan: [k][E] column totals
  int32_t* off_s = tot_s + k * E;            // self scan: [E + 1] offsets
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int kE = k * E;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tc;
  const int n = static_cast<int>(min(static_cast<int64_t>(tc), T - t0));
  const int seg = (tc + PLACE_WARPS - 1) / PLACE_WARPS;  // tokens per warp
  const int w0 = min(n, warp * seg), w1 = min(n, w0 + seg);
  int32_t* my = wc + warp * E;
  const uint32_t lt_mask = (1u << lane) - 1u;
  const int32_t* base = hist + static_cast<int64_t>(blockIdx.x) * kE;
  const int32_t* cbase = hist + static_cast<int64_t>(n_chunks) * kE;
  // the row copy's staging: two buffers of `nb` rows after the ranking's arrays, and their barriers;
  // the first two parts of the chunk's rows start loading now, under the ranking
  const bool copy = X != nullptr && n > 0 && nb > 0;
  const int parts = copy ? (n + nb - 1) / nb : 0;
  // (128-byte aligned by an offset from the shared array, not an integer round trip, so that the
  // compiler keeps the reads of the staged rows in the shared state space)
  uint8_t* after = reinterpret_cast<uint8_t*>(base_s + (stage_bases >= 2 ? 2 * kE + E + 1 : stage_bases ? kE : 0));
  uint8_t* buf0 = after + ((128u - (ptx::smem_u32(after) & 127u)) & 127u);
  uint64_t* bar = reinterpret_cast<uint64_t*>(buf0 + 2 * static_cast<size_t>(nb) * row_bytes);
  const uint8_t* usrc = reinterpret_cast<const uint8_t*>(U) + t0 * row_bytes;
  auto load_part = [&](int q) {  // part q into buffer q & 1 (one thread)
    const uint32_t bytes = static_cast<uint32_t>(min(nb, n - q * nb)) * row_bytes;
    uint64_t* bb = &bar[q & 1];
    ptx::mbar_arrive_expect_tx(bb, bytes);
    ptx::bulk_load(buf0 + static_cast<size_t>(q & 1) * nb * row_bytes,
                   usrc + static_cast<int64_t>(q) * nb * row_bytes, bytes, bb);
  };
  if (copy && threadIdx.x == 0) {
    ptx::mbar_init(&bar[0], 1);
    ptx::mbar_init(&bar[1], 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
    for (int q = 0; q < min(2, parts); ++q) load_part(q);
  }
  // everything the ranking reads, staged with loads that are all in flight together
  for (int i = threadIdx.x; i < n * k; i += blockDim.x) idx_s[i] = idx[t0 * k + i];
  if (stage_bases == 1)
    for (int i = threadIdx.x; i < kE; i += blockDim.x) base_s[i] = base[i] + cbase[i];
  // (stage_bases 2 and 3 below)
  if (stage_bases >= 2) {
    for (int i = threadIdx.x; i < kE; i += blockDim.x) {
      base_s[i] = 0;
      tot_s[i] = 0;
    }
    __syncthreads();
    // columns (j, e): `parts` threads each add every parts-th chunk, before this one and all; four
    // columns a thread with 16-byte loads when k E allows (the chunk rows are 16-byte aligned then)
    const int b = static_cast<int>(blockIdx.x);
    if (stage_bases == 3) {
      // every expert id of the batch: position p = t k + j lies before the chunk when p < t0 k
      const int Tk = static_cast<int>(T) * k, p0 = static_cast<int>(t0) * k;
      bool bad = false;
      for (int i = threadIdx.x; i < Tk; i += blockDim.x) {
        const int e = idx[i];
        if (e < 0 || e >= E) {
          bad = true;
          continue;
        }
        const int col = (i % k) * E + e;
        atomicAdd(&tot_s[col], 1);  // integer counts: the order of the adds does not matter
        if (i < p0) atomicAdd(&base_s[col], 1);
      }
      if (bad && b == 0) set_status(status, MOE_DEV_BAD_EXPERT_ID);
    } else if ((kE & 3) == 0) {
      const int q4 = kE / 4;
      const int parts = q4 < PLACE_THREADS ? PLACE_THREADS / q4 : 1;
      for (int t = threadIdx.x; t < parts * q4; t += blockDim.x) {
        const int col = (t % q4) * 4, part = t / q4;
        int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
#pragma unroll 8
        for (int c = part; c < n_chunks; c += parts) {
          const int4 v = *reinterpret_cast<const int4*>(hist + static_cast<int64_t>(c) * kE + col);
          tot.x += v.x;
          tot.y += v.y;
          tot.z += v.z;
          tot.w += v.w;
          if (c < b) {
            pre.x += v.x;
            pre.y += v.y;
            pre.z += v.z;
            pre.w += v.w;
          }
        }
        atomicAdd(&base_s[col], pre.x);  // integer counts: the order of the adds does not matter
        atomicAdd(&base_s[col + 1], pre.y);
        atomicAdd(&base_s[col + 2], pre.z);
        atomicAdd(&base_s[col + 3], pre.w);
        atomicAdd(&tot_s[col], tot.x);
        atomicAdd(&tot_s[col + 1], tot.y);
        atomicAdd(&tot_s[col + 2], tot.z);
        atomicAdd(&tot_s[col + 3], tot.w);
      }
    } else {
      const int parts = kE < PLACE_THREADS ? PLACE_THREADS / kE : 1;
      for (int t = threadIdx.x; t < parts * kE; t += blockDim.x) {
        const int col = t % kE, part = t / kE;
        int32_t pre = 0, tot = 0;
#pragma unroll 4
        for (int c = part; c < n_chunks; c += parts) {
          const int32_t v = hist[static_cast<int64_t>(c) * kE + col];
          tot += v;
          pre += c < b ? v : 0;
        }
        atomicAdd(&base_s[col], pre);
        atomicAdd(&tot_s[col], tot);
      }
    }
    __syncthreads();
    // choice bases (the pairs of earlier choices per expert), routed and kept counts
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int32_t run = 0;
      for (int j = 0; j < k; ++j) {
        base_s[j * E + e] += run;
        run += tot_s[j * E + e];
      }
      const int32_t kept = static_cast<int32_t>(min(static_cast<int64_t>(run), C));
      off_s[e] = kept;
      if (blockIdx.x == 0) {
        counts_routed[e] = run;
        counts_kept[e] = kept;
      }
    }
    __syncthreads();
    if (warp == 0) {  // offsets = exclusive scan of the kept counts
      const int per = (E + 31) / 32;
      const int lo = min(E, lane * per), hi = min(E, lo + per);
      int32_t s = 0;
      for (int i = lo; i < hi; ++i) s += off_s[i];
      int32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int32_t run = incl - s;
      for (int i = lo; i < hi; ++i) {
        const int32_t v = off_s[i];
        off_s[i] = run;
        if (blockIdx.x == 0) offsets[i] = run;
        run += v;
      }
      const int32_t A = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) {
        off_s[E] = A;
        if (blockIdx.x == 0) {
          offsets[E] = A;
          *n_dropped = T * k - A;
        }
      }
    }
  }
  __syncthreads();
  for (int j = 0; j < k; ++j) {
    for (int i = threadIdx.x; i < PLACE_WARPS * E; i += blockDim.x) wc[i] = 0;
    __syncthreads();
    // pass 1: per-warp counts of choice j (w0, w1 are warp-uniform)
    for (int q = w0; q < w1; q += 32) {
      const int r = q + lane;
      int e = -1;
      if (r < w1) {
        e = idx_s[r * k + j];
        if (e < 0 || e >= E) e = -1;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    // warp bases: choice base + chunk prefix + earlier warps, warps in order
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      int32_t run = stage_bases ? base_s[j * E + e] : cbase[j * E + e] + base[j * E + e];
      for (int w = 0; w < PLACE_WARPS; ++w) {
        const int32_t v = wc[w * E + e];
        wc[w * E + e] = run;
        run += v;
      }
    }
    __syncthreads();
    // pass 2: slot = warp base + rank among the equal experts of earlier lanes
    for (int q = w0; q < w1; q += 32) {
      const int r = q + lane;
      int e = -1;
      if (r < w1) {
        e = idx_s[r * k + j];
        if (e < 0 || e >= E) e = -1;
      }
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      const int32_t slot = e >= 0 ? my[e] + __popc(peers & lt_mask) : -1;
      __syncwarp();
      if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
      __syncwarp();
      if (r < w1) {
        const int64_t t = t0 + r;
        int32_t row = -1;
        if (e >= 0 && slot < C) {
          row = (stage_bases >= 2 ? off_s[e] : offsets[e]) + slot;
          row_token[row] = static_cast<int32_t>(t);
        }
        slot_row[t * k + j] = row;
        rows_s[r * k + j] = row;
      }
    }
    __syncthreads();
  }
  if (!copy) return;
  // the row copy: part pi (rows pi nb .. of the chunk) is written out while part pi + 1 loads; each
  // warp takes 512-byte pieces (row r, 32 16-byte vectors) and stores each to every kept row of r
  __shared__ int abort_s;
  if (threadIdx.x == 0) abort_s = 0;
  const int vpr = static_cast<int>(row_bytes / 16);
  const int upr = (vpr + 31) / 32;  // 512-byte pieces per row
  int pi = 0;
  for (; pi < parts; ++pi) {
    if (threadIdx.x == 0) {
      const uint64_t tw = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&bar[pi & 1], static_cast<uint32_t>((pi >> 1) & 1))) {
        if (ptx::globaltimer_ns() - tw > COPY_WAIT_LIMIT_NS) {
          abort_s = 1;
          break;
        }
      }
    }
    __syncthreads();
    if (abort_s) break;
    const int r0 = pi * nb, nr = min(nb, n - r0);
    const uint4* src = reinterpret_cast<const uint4*>(buf0 + static_cast<size_t>(pi & 1) * nb * row_bytes);
    for (int u = warp; u < nr * upr; u += PLACE_WARPS) {
      const int r = u / upr;
      const int v = (u - r * upr) * 32 + lane;
      const int32_t my_row = lane < k ? rows_s[(r0 + r) * k + lane] : -1;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (v < vpr) val = src[r * vpr + v];
      for (int j = 0; j < k; ++j) {
        const int32_t row = __shfl_sync(0xffffffffu, my_row, j);
        if (row >= 0 && v < vpr) reinterpret_cast<uint4*>(X)[static_cast<int64_t>(row) * vpr + v] = val;
      }
    }
    __syncthreads();  // buffer pi & 1 has been read by every warp
    if (threadIdx.x == 0 && pi + 2 < parts) {
      ptx::fence_proxy_async_smem();
      load_part(pi + 2);
    }
  }
  if (abort_s && threadIdx.x == 0) {
    set_status(status, MOE_DEV_TIMEOUT);
    // parts pi and pi + 1 may still be loading into this block's shared memory: wait for them (bounded)
    for (int q = pi; q < min(pi + 2, parts); ++q) {
      const uint64_t tw = ptx::globaltimer_ns();
      while (!ptx::mbar_try_wait(&bar[q & 1], static_cast<uint32_t>((q >> 1) & 1)) &&
             ptx::globaltimer_ns() - tw < COPY_WAIT_LIMIT_NS) {
      }
    }
  }
}

cudaError_t launch_dispatch(const Plan& p, const void* U, const int32_t* idx, int32_t* counts_routed,
                            int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token, void* X,
                            int64_t* n_dropped, uint8_t* ws, cudaStream_t s) {
  int32_t* hist = reinterpret_cast<int32_t*>(ws + p.ws_hist);
  int32_t* status = ws_status(p, ws);
  if (p.priority == MOE_PRIORITY_CHOICE_MAJOR && p.dp_chunks > 0) {
    int32_t* ticket = reinterpret_cast<int32_t*>(ws + p.ws_status + 192);
    const size_t hsm = sizeof(int32_t) * static_cast<size_t>(p.k) * p.E;
    if (hsm > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(dispatch_hist, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(hsm));
      if (e != cudaSuccess) return e;
    }
    // small batches: the placement blocks count the expert ids themselves (one launch)
    const bool self_count = p.Tk <= SELF_COUNT_MAX;
    cudaError_t e = cudaSuccess;
    if (!self_count) {
      dispatch_hist<<<p.dp_chunks, HIST_THREADS, hsm, s>>>(idx, p.T, p.k, p.E, p.dp_tc, hist, status);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    const int cols = p.k * p.E;
    // small histograms: the placement blocks scan them themselves (no column-scan launch)
    const bool self_scan = self_count || static_cast<int64_t>(p.dp_chunks) * cols <= SELF_SCAN_MAX;
    if (!self_scan) {
      dispatch_colscan<<<(cols + 7) / 8, 256, 0, s>>>(hist, p.dp_chunks, p.k, p.E, p.C, p.Tk, ticket, counts_routed,
                                                       counts_kept, offsets, n_dropped);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    const uint32_t row_bytes = static_cast<uint32_t>(p.h) * (p.bf16 ? 2 : 4);
    // the chunk's bases in shared memory when they fit 16 KB (self scan: with the totals and offsets)
    const int stage_bases = self_count ? 3 : self_scan ? 2 : p.k * p.E <= 4096 ? 1 : 0;
    const size_t staged = stage_bases >= 2 ? 2 * static_cast<size_t>(cols) + p.E + 1 : stage_bases ? cols : 0;
    const size_t meta = sizeof(int32_t) * (static_cast<size_t>(PLACE_WARPS) * p.E + 2 * static_cast<size_t>(p.dp_tc) * p.k +
                                           staged);
    // two row buffers in what is left of COPY_SMEM_BYTES (at most the chunk each); rows too wide for
    // two buffers in any block are copied by dispatch_scatter after the placement instead
    const size_t room = meta + 128 + 16 < COPY_SMEM_BYTES ? COPY_SMEM_BYTES - meta - 128 - 16 : 0;
    int nb = X ? static_cast<int>(std::min<size_t>(p.dp_tc, room / 2 / row_bytes)) : 0;
    if (X && nb == 0 && meta + 128 + 2 * static_cast<size_t>(row_bytes) + 16 <= 200 * 1024) nb = 1;
    const bool scatter_after = X && nb == 0;
    const size_t psm = meta + (nb > 0 ? 128 + 2 * static_cast<size_t>(nb) * row_bytes + 16 : 0);
    if (psm > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(dispatch_place, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(psm));
      if (e != cudaSuccess) return e;
    }
    dispatch_place<<<p.dp_chunks, PLACE_THREADS, psm, s>>>(idx, p.T, p.k, p.E, p.dp_tc, p.dp_chunks, p.C, hist,
                                                            offsets, slot_row, row_token, U, nb > 0 ? X : nullptr,
                                                            row_bytes, nb, status, stage_bases, counts_routed,
                                                            counts_kept, n_dropped);
    e = cudaGetLastError();
    if (e != cudaSuccess || !scatter_after) return e;
    const int vpr = static_cast<int>(row_bytes / 16);
    const int64_t want = (p.T + 7) / 8;
    const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
    dispatch_scatter<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(U), slot_row, static_cast<uint4*>(X), p.T, p.k,
                                            vpr);
    return cudaGetLastError();
  }
  const size_t hist_smem = sizeof(int32_t) * p.E;
  if (p.n_chunks > 0) {
    dispatch_count<<<p.n_chunks, DISPATCH_THREADS, hist_smem, s>>>(idx, p.T, p.k, p.E, p.priority, p.chunk, hist,
                                                                   status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int epow = 1;
  while (epow < p.E) epow <<= 1;
  int G = SCAN_THREADS / epow;
  if (G > p.n_chunks) G = p.n_chunks > 0 ? p.n_chunks : 1;
  if (G < 1) G = 1;
  dispatch_scan<<<1, SCAN_THREADS, 0, s>>>(hist, p.n_chunks, p.E, G, p.C, p.Tk, counts_routed, counts_kept, offsets,
                                           n_dropped);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_chunks == 0) return e;
  const size_t wc_smem = sizeof(int32_t) * DISPATCH_WARPS * p.E;
  dispatch_assign<<<p.n_chunks, DISPATCH_THREADS, wc_smem, s>>>(idx, p.T, p.k, p.E, p.priority, p.chunk, hist,
                                                                offsets, p.C, slot_row, row_token);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (!X) return cudaSuccess;  // routing metadata only (the FP8 dispatch copies the rows itself)
  const int elem = p.bf16 ? 2 : 4;
  const int vpr = p.h * elem / 16;
  const int64_t want = (p.T + 7) / 8;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
  dispatch_scatter<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(U), slot_row, static_cast<uint4*>(X), p.T, p.k,
                                          vpr);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Dispatch without a caller-provided workspace (moe_dispatch_noalloc).
//
// The only scratch dispatch needs is the per-chunk histogram, [n_chunks, E]
// int32.  Here it lives in one file-scope device array instead of the
// workspace, so the caller allocates nothing beyond its inputs and outputs.
// The array exists once per device for as long as the library is loaded, and
// every call on a device shares it.  dispatch_count rewrites every entry a call
// reads before the scan reads it, so nothing in it has to start at zero.  Calls
// that overlap on the GPU (different streams, no ordering between them) race on
// it.
static __device__ __align__(256) int32_t g_noalloc_hist[MOE_NOALLOC_HIST_MAX];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
int32_t* g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};  // unique id of the context the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (ids are never reused within a process, so
// a device reset or a switch to another context shows up as a new id); 0 if there is none.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_noalloc_hist in the current context.  In host code the array's name is only
// a host-side stand-in, so the kernels get this address, never the name.  It is looked up once per
// device and kept with the id of the context it was found in; a call from another context (after
// a device reset, or with a context the caller made current) looks it up again.
cudaError_t noalloc_hist_ptr(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  const unsigned long long ctx = current_context_id();
  if (!g_noalloc_ptr[dev] || ctx == 0 || ctx != g_noalloc_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_hist);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    g_noalloc_ctx[dev] = current_context_id();  // the lookup made the device's context current
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_dispatch_noalloc(const Plan& p, const void* U, const int32_t* idx, int32_t* counts_routed,
                                    int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                    void* X, int64_t* n_dropped, int32_t* status, cudaStream_t s) {
  if (static_cast<int64_t>(p.n_chunks) * p.E > MOE_NOALLOC_HIST_MAX) return cudaErrorInvalidValue;
  int32_t* hist = nullptr;
  cudaError_t e = noalloc_hist_ptr(&hist);
  if (e != cudaSuccess) return e;
  if (status) {
    e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
  }
  if (p.n_chunks > 0) {
    dispatch_count<<<p.n_chunks, DISPATCH_THREADS, sizeof(int32_t) * p.E, s>>>(idx, p.T, p.k, p.E, p.priority,
                                                                               p.chunk, hist, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int epow = 1;
  while (epow < p.E) epow <<= 1;
  int G = SCAN_THREADS / epow;
  if (G > p.n_chunks) G = p.n_chunks > 0 ? p.n_chunks : 1;
  if (G < 1) G = 1;
  dispatch_scan<<<1, SCAN_THREADS, 0, s>>>(hist, p.n_chunks, p.E, G, p.C, p.Tk, counts_routed, counts_kept, offsets,
                                           n_dropped);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_chunks == 0) return e;
  dispatch_assign<<<p.n_chunks, DISPATCH_THREADS, sizeof(int32_t) * DISPATCH_WARPS * p.E, s>>>(
      idx, p.T, p.k, p.E, p.priority, p.chunk, hist, offsets, p.C, slot_row, row_token);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int vpr = p.h * (p.bf16 ? 2 : 4) / 16;
  const int64_t want = (p.T + 7) / 8;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
  dispatch_scatter<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(U), slot_row, static_cast<uint4*>(X), p.T, p.k,
                                          vpr);
  return cudaGetLastError();
}

}  // namespace moe
