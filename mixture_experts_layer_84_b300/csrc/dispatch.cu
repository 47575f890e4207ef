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
// result:
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

namespace moe {

constexpr int DISPATCH_THREADS = 256;
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

constexpr int SCATTER_UNROLL = 4;

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

cudaError_t launch_dispatch(const Plan& p, const void* U, const int32_t* idx, int32_t* counts_routed,
                            int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token, void* X,
                            int64_t* n_dropped, uint8_t* ws, cudaStream_t s) {
  int32_t* hist = reinterpret_cast<int32_t*>(ws + p.ws_hist);
  int32_t* status = ws_status(p, ws);
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
