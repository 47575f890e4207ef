// Router logits on the tensor cores: H = U W_r (and U W_noise for the noisy
// router) as bf16 x bf16 products accumulated in float32.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section
// 路由器：打分、top-k、加权求和: the router linear H = U W_r (W_r in R^{h x E},
// column i = expert i's centroid) and the noisy top-k logits
// (x W_g)_i + N(0,1) * Softplus((x W_noise)_i).
//
// Two launches replace the CUDA-core partial-logits kernel for bf16:
//   route_pack_wt   transposes W_r (and W_noise below it) into a K-major
//                   [N, h] bf16 matrix in the workspace, rows >= E (or 2E)
//                   zero, N = the MMA width (a multiple of 16, <= 256);
//   route_logits_tc one CTA per (128-token tile, slice of h): TMA stages
//                   U 128x64 and Wt Nx64 tiles (128-byte swizzle) into a
//                   4-stage ring, one thread issues tcgen05.mma 128xNx16
//                   into a tensor-memory accumulator, and four warps write the
//                   float32 slice sums [split][T][E] (noise slice sums after
//                   the first E columns) that route_select adds up in a fixed
//                   order before scoring and top-k.
// Every mbarrier wait is bounded; a wait that gives up records
// MOE_DEV_TIMEOUT after draining what is in flight.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "select.cuh"

namespace moe {
namespace rtc {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UK = 16;
constexpr int STAGES = 4;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr size_t BAR_BYTES = 128;

__host__ __device__ constexpr uint32_t b_bytes(int N) { return static_cast<uint32_t>(N) * BK * 2; }
__host__ __device__ constexpr uint32_t stage_bytes(int N) { return A_BYTES + b_bytes(N); }
inline size_t smem_bytes(int N) { return 1024 + STAGES * static_cast<size_t>(stage_bytes(N)) + BAR_BYTES; }

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
  return true;
}

// Wt[n][c] = W_r[c][n] (n < E), W_noise[c][n - E] (noisy, E <= n < 2E), else 0.
__global__ void __launch_bounds__(256) route_pack_wt(const bf16* __restrict__ W_r, const bf16* __restrict__ W_noise,
                                                     int h, int E, int N, bf16* __restrict__ Wt) {
  __shared__ bf16 tile[32][33];
  const int n0 = blockIdx.x * 32, c0 = blockIdx.y * 32;
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int c = c0 + y, n = n0 + threadIdx.x;
    bf16 v = __float2bfloat16_rn(0.f);
    if (c < h) {
      if (n < E)
        v = W_r[static_cast<int64_t>(c) * E + n];
      else if (W_noise && n < 2 * E)
        v = W_noise[static_cast<int64_t>(c) * E + (n - E)];
    }
    tile[y][threadIdx.x] = v;
  }
  __syncthreads();
  for (int y = threadIdx.y; y < 32; y += blockDim.y) {
    const int n = n0 + y, c = c0 + threadIdx.x;
    if (n < N && c < h) Wt[static_cast<int64_t>(n) * h + c] = tile[threadIdx.x][y];
  }
}

template <int N>
__global__ void __launch_bounds__(THREADS, 1)
    route_logits_tc(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW, int64_t T,
                    int h, int E, int splits, float* __restrict__ part, float* __restrict__ npart, int32_t* status) {
  constexpr uint32_t STAGE = stage_bytes(N);
  constexpr uint32_t TMEM_COLS = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);  // (shared state space kept)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t mt = blockIdx.x / splits;
  const int split = static_cast<int>(blockIdx.x % splits);
  const int nkb = (h + BK - 1) / BK;
  const int kb_beg = static_cast<int>((static_cast<int64_t>(nkb) * split) / splits);
  const int kb_end = static_cast<int>((static_cast<int64_t>(nkb) * (split + 1)) / splits);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmU);
      ptx::prefetch_tmap(&tmW);
      const uint64_t pol_u = ptx::policy_evict_first();
      const uint64_t pol_w = ptx::policy_evict_last();
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      for (int kb = kb_beg; kb < kb_end; ++kb) {
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) break;
        uint8_t* sa = smem + stage * STAGE;
        ptx::mbar_arrive_expect_tx(&full[stage], STAGE);
        ptx::tma_load_2d(sa, &tmU, kb * BK, static_cast<int32_t>(mt * BM), &full[stage], pol_u);
        ptx::tma_load_2d(sa + A_BYTES, &tmW, kb * BK, 0, &full[stage], pol_w);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) wait_drain(&full[s], (armed_phase >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, N);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int kb = kb_beg; kb < kb_end; ++kb) {
        if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + stage * STAGE);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UK; ++kk)
          ptx::mma_bf16_ss(tmem_base, ptx::sdesc_kmajor_sw128(sa + kk * UK * 2),
                           ptx::sdesc_kmajor_sw128(sb + kk * UK * 2), IDESC, (kb > kb_beg || kk) ? 1u : 0u);
        ptx::mma_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // complete (or, after a timeout, drained): the epilogue may read the accumulator
      ptx::mma_commit(tfull);
      (void)ok;
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int64_t t = mt * BM + q * 32 + lane;
    const bool ready = wait_drain(tfull, 0);
    if (__all_sync(0xffffffffu, ready) && !*abort_flag) {
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      const bool vec = (E & 3) == 0;
#pragma unroll 1
      for (int c = 0; c < N; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tb + c, v);
        ptx::tmem_wait_ld();
        if (t < T) {
          // columns [0, E): router logits; [E, 2E): noise logits (npart != nullptr)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float* dst = half == 0 ? part : npart;
            if (!dst) continue;
            const int lo = half * E;
            const int64_t row = (static_cast<int64_t>(split) * T + t) * E;
            if (vec && c >= lo && c + 32 <= lo + E) {
              float4* d4 = reinterpret_cast<float4*>(dst + row + (c - lo));
#pragma unroll
              for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int col = c + i;
                if (col >= lo && col < lo + E) dst[row + (col - lo)] = __uint_as_float(v[i]);
              }
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) set_status(status, MOE_DEV_TIMEOUT);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static bool make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N>
static cudaError_t launch_n(const Plan& p, const CUtensorMap& tmU, const CUtensorMap& tmW, float* part, float* npart,
                            int32_t* status, cudaStream_t s) {
  const size_t smem = smem_bytes(N);
  cudaError_t e = cudaFuncSetAttribute(route_logits_tc<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t mtiles = (p.T + BM - 1) / BM;
  route_logits_tc<N><<<static_cast<unsigned>(mtiles * p.route_splits), THREADS, smem, s>>>(
      tmU, tmW, p.T, p.h, p.E, p.route_splits, part, npart, status);
  return cudaGetLastError();
}

}  // namespace rtc

cudaError_t launch_route_logits_tc(const Plan& p, const void* U, const void* W_r, const void* W_noise, float* part,
                                   float* npart, uint8_t* ws, cudaStream_t s) {
  using namespace rtc;
  bf16* Wt = reinterpret_cast<bf16*>(ws + p.ws_wt);
  const int N = p.route_tc_n;
  route_pack_wt<<<dim3((N + 31) / 32, (p.h + 31) / 32), dim3(32, 8), 0, s>>>(
      static_cast<const bf16*>(W_r), p.noisy ? static_cast<const bf16*>(W_noise) : nullptr, p.h, p.E, N, Wt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CUtensorMap tmU, tmW;
  if (!make_tmap(&tmU, U, static_cast<uint64_t>(p.T), p.h, BM) || !make_tmap(&tmW, Wt, N, p.h, N))
    return cudaErrorNotSupported;
  int32_t* status = ws_status(p, ws);
  switch (N) {
#define MOE_RTC_CASE(n) \
  case n: return launch_n<n>(p, tmU, tmW, part, npart, status, s);
    MOE_RTC_CASE(16) MOE_RTC_CASE(32) MOE_RTC_CASE(48) MOE_RTC_CASE(64) MOE_RTC_CASE(80) MOE_RTC_CASE(96)
    MOE_RTC_CASE(112) MOE_RTC_CASE(128) MOE_RTC_CASE(144) MOE_RTC_CASE(160) MOE_RTC_CASE(176) MOE_RTC_CASE(192)
    MOE_RTC_CASE(208) MOE_RTC_CASE(224) MOE_RTC_CASE(240) MOE_RTC_CASE(256)
#undef MOE_RTC_CASE
  }
  return cudaErrorInvalidValue;
}


// ---------------------------------------------------------------------------------------------
// The fused router: logits on the tensor cores, then scores, top-k, gates and the P / z partials
// in the epilogue, with no float32 logit round trip through global memory.
//
// A cluster of CS CTAs owns one 128-token tile; CTA c of the cluster runs the K-blocks
// [c nkb / CS, (c+1) nkb / CS) of h through a TMA ring and tcgen05.mma 128 x N x 16 into its
// tensor memory (N = E, or 2E with the noise columns, rounded up to 16).  After a cluster barrier
// (every CTA is past its main loop), its four epilogue warps push each float32 accumulator row to
// the cluster CTA that owns the row -- CTA c owns rows [c R, (c+1) R), R = 128 / CS -- with 16-byte
// remote stores into distributed shared memory.  After a second barrier each CTA adds the CS slices
// of its logits in rank order (run-to-run identical) from its own shared memory, then the bias
// and the noise eps * softplus(noise logit), stages them for select_tokens (select.cuh) in passes
// of NTH / G tokens, and adds its per-expert score sums and LSE^2 sum into one ppart row.
namespace rfu {

using namespace rtc;

// NTH = 256 or 512 threads: warp 0 TMA, warp 1 MMA, warps 2-3 stage the biases, warps 4-7 read the
// accumulator out; every warp reduces and selects
constexpr int MAX_STAGES = 8;
constexpr size_t RF_BAR_BYTES = 256;  // full[8], empty[8], tfull, tensor-memory address, abort flag

struct Geometry {
  int N, stages, PN, TB, LD, sel_floats;
  uint32_t stage_bytes;
  size_t p_bytes, work, smem;
};

// Shared memory of the fused router: the TMA stages, reused after the main loop for the partial
// tile P [128][N + 1] and the select staging (sx [TB][LD], zsq [TB], gsc [TB][n_group],
// colsum [E + 1]), then the barriers, then the logit bias, the selection bias and each expert's
// position in a staged row [E] each.
// G = lanes per token of the selection.
__host__ __device__ inline Geometry geometry(int N, int E, int n_group, int stages, int G, int threads) {
  Geometry g;
  g.N = N;
  g.stages = stages;
  g.stage_bytes = A_BYTES + b_bytes(N);
  g.PN = N + 4;  // 16-byte rows for the remote vector stores
  g.TB = threads / G;
  const int C = (E + G - 1) / G;
  g.LD = G * ((C & 1) ? C + 2 : C + 1);
  g.p_bytes = sizeof(float) * 128 * static_cast<size_t>(g.PN);
  g.sel_floats = g.TB * g.LD + g.TB + g.TB * (n_group > 1 ? n_group : 0) + (E + 1) + threads;
  const size_t ring = static_cast<size_t>(stages) * g.stage_bytes;
  const size_t tail = g.p_bytes + sizeof(float) * static_cast<size_t>(g.sel_floats);
  g.work = ((ring > tail ? ring : tail) + 15) / 16 * 16;
  g.smem = 1024 + g.work + RF_BAR_BYTES + 3 * sizeof(float) * static_cast<size_t>(E);  // + bias_s, selb_s, pos_s
  return g;
}

// 16-byte store to a cluster CTA's shared memory (address from mapa).
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

template <int KP, int G, int NTH>
__global__ void __launch_bounds__(NTH, NTH == 512 ? 1 : 2)
    route_fused(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmW, int64_t T, int h,
                int E, int N, int stages, int cs, const float* __restrict__ b_r, const float* __restrict__ sel_bias,
                const float* __restrict__ eps, int noisy, float* __restrict__ logits_out, int32_t* __restrict__ idx,
                float* __restrict__ gate, float* __restrict__ ppart, int32_t* __restrict__ ppart_rows, int k,
                int score_fn, int renorm, int n_group, int topk_group, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  // the 1024-byte aligned base as an offset from the shared array itself (not an integer round
  // trip), so that the compiler keeps every access through it in the shared state space
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const Geometry geo = geometry(N, E, n_group, stages, G, NTH);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + geo.work);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* Q = reinterpret_cast<float*>(smem);                       // [cs][R][PN], after the main loop
  float* sx = reinterpret_cast<float*>(smem + geo.p_bytes);       // select staging
  float* zsq = sx + geo.TB * geo.LD;
  float* gsc = zsq + geo.TB;
  float* colsum = gsc + geo.TB * (n_group > 1 ? n_group : 0);
  float* colpart = colsum + (E + 1);                               // [NTH] column-sum partials
  float* bias_s = reinterpret_cast<float*>(smem + geo.work + RF_BAR_BYTES);  // b_r (or zeros) [E]
  float* selb_s = bias_s + E;                                                  // sel_bias [E]
  int* pos_s = reinterpret_cast<int*>(selb_s + E);                             // SelLayout::at(0, e) [E]

  const uint32_t tmem_cols = N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
  const uint32_t STAGE = geo.stage_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(blockIdx.x % cs);
  const int64_t mt = blockIdx.x / cs;
  const int nkb = (h + BK - 1) / BK;
  const int kb_beg = (nkb * rank) / cs, kb_end = (nkb * (rank + 1)) / cs;
  // the tile rows this CTA selects for: [rank R, (rank+1) R) of the tile
  const int R = BM / cs;
  const int64_t row0 = mt * BM + static_cast<int64_t>(rank) * R;
  const int64_t left = T - row0;
  const int rows_here = left <= 0 ? 0 : left < R ? static_cast<int>(left) : R;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(tfull, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmU);
      ptx::prefetch_tmap(&tmW);
      const uint64_t pol_u = ptx::policy_evict_first();
      const uint64_t pol_w = ptx::policy_evict_last();
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      for (int kb = kb_beg; kb < kb_end; ++kb) {
        if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) break;
        uint8_t* sa = smem + stage * STAGE;
        ptx::mbar_arrive_expect_tx(&full[stage], STAGE);
        ptx::tma_load_2d(sa, &tmU, kb * BK, static_cast<int32_t>(mt * BM), &full[stage], pol_u);
        ptx::tma_load_2d(sa + A_BYTES, &tmW, kb * BK, 0, &full[stage], pol_w);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < stages; ++s)
        if ((armed >> s) & 1u) wait_drain(&full[s], (armed_phase >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t IDESC = ptx::idesc_bf16_f32(BM, N);
      uint32_t stage = 0, phase = 0;
      for (int kb = kb_beg; kb < kb_end; ++kb) {
        if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_LIMIT_NS)) break;
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + stage * STAGE);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / UK; ++kk)
          ptx::mma_bf16_ss(tmem_base, ptx::sdesc_kmajor_sw128(sa + kk * UK * 2),
                           ptx::sdesc_kmajor_sw128(sb + kk * UK * 2), IDESC, (kb > kb_beg || kk) ? 1u : 0u);
        ptx::mma_commit(&empty[stage]);
        if (++stage == static_cast<uint32_t>(stages)) {
          stage = 0;
          phase ^= 1u;
        }
      }
      ptx::mma_commit(tfull);  // complete (or drained after a timeout): the accumulator may be read
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    // under the main loop: the biases into shared memory, and this CTA's rows of the noise into L2
    // (the epilogue reads them with all its loads in flight, but one CTA per SM has few warps)
    const int i0 = threadIdx.x - 64;
    const SelLayout L(E, G);
    for (int e = i0; e < E; e += 64) {
      bias_s[e] = b_r ? b_r[e] : 0.f;
      selb_s[e] = sel_bias ? sel_bias[e] : 0.f;
      pos_s[e] = L.at(0, e);
    }
    if (noisy && rows_here > 0) {
      const char* nb = reinterpret_cast<const char*>(eps + row0 * E);
      const int64_t bytes = static_cast<int64_t>(rows_here) * E * static_cast<int64_t>(sizeof(float));
      for (int64_t off = static_cast<int64_t>(i0) * 128; off < bytes; off += 64 * 128) ptx::prefetch_l2(nb + off);
    }
  }
  // the accumulator is complete (or the pipeline gave up); every CTA of the cluster must be past its
  // main loop before any partial row lands in a peer's shared memory (which held its TMA stages)
  const bool readout = warp >= 4 && warp < 8;
  bool ready = true;
  if (readout) ready = __all_sync(0xffffffffu, wait_drain(tfull, 0));
  if (readout && !ready) *abort_flag = 1;
  __syncthreads();
  ptx::cluster_sync_all();
  // partial rows to their owners: tile row i belongs to cluster CTA i / R, which keeps slot
  // [rank][i % R] of Q [cs][R][PN] for it (16-byte remote stores)
  if (readout && !*abort_flag) {
    const int q = warp & 3;
    const int i = q * 32 + lane;
    const int owner = i / R, li = i - owner * R;
    const uint32_t dst = ptx::mapa_shared(ptx::smem_u32(Q + (rank * R + li) * geo.PN), static_cast<uint32_t>(owner));
    ptx::tc_fence_after();
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
    for (int c = 0; c < N; c += 32) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(tb + c, v);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i4 = 0; i4 < 8; ++i4)
        if (c + 4 * i4 < N)  // N is a multiple of 16, not of 32
          st_cluster_v4(dst + static_cast<uint32_t>(c + 4 * i4) * 4u, v[4 * i4], v[4 * i4 + 1], v[4 * i4 + 2],
                        v[4 * i4 + 3]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, tmem_cols);
  ptx::cluster_sync_all();  // every partial row has arrived
  const bool ok = !*abort_flag;

  // rows [rank R, (rank+1) R) of the tile: the CS slices summed in rank order from local shared
  // memory, then bias and noise; the pass's rows x E entries in order, RB a thread at a time with
  // their noise loads issued together.  The loop is kept compact (it runs once per CTA, from a cold
  // instruction cache): (row, expert) advance by additions, the staged position comes from pos_s.
  if (ok) {
    constexpr int RB = 4;
    const int dr = NTH / E, de = NTH - (NTH / E) * E;
    for (int p0 = 0; p0 < rows_here; p0 += geo.TB) {
      const int rows = min(geo.TB, rows_here - p0);
      const int n_el = rows * E;
      const float* eps_p = noisy ? eps + (row0 + p0) * E : nullptr;
      float* lo_p = logits_out ? logits_out + (row0 + p0) * E : nullptr;
      const SelLayout L(E, G);
      int r = static_cast<int>(threadIdx.x) / E;
      int e = static_cast<int>(threadIdx.x) - r * E;
#pragma unroll 1
      for (int i = threadIdx.x; i < n_el; i += RB * NTH) {
        float ev[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) ev[u] = (noisy && i + u * NTH < n_el) ? eps_p[i + u * NTH] : 0.f;
#pragma unroll
        for (int u = 0; u < RB; ++u) {
          if (i + u * NTH < n_el) {
            const float* qr = Q + (p0 + r) * geo.PN + e;
            float x = 0.f, z = 0.f;
#pragma unroll 1
            for (int c = 0; c < cs; ++c) {
              x += qr[c * R * geo.PN];
              if (noisy) z += qr[c * R * geo.PN + E];
            }
            if (b_r) x += bias_s[e];
            if (noisy) x = fmaf(ev[u], softplus_f32(z), x);
            if (lo_p) lo_p[i + u * NTH] = x;
            sx[r * L.LD + pos_s[e]] = x;
          }
          r += dr;
          e += de;
          if (e >= E) {
            e -= E;
            ++r;
          }
        }
      }
      __syncthreads();
      select_tokens<KP, G>(sx, zsq, gsc, rows, row0 + p0, E, k, score_fn, renorm, n_group, topk_group,
                           sel_bias ? selb_s : nullptr, idx, gate, pos_s);
      __syncthreads();
      score_column_sums_split(sx, zsq, rows, E, G, colsum, colpart, p0 > 0);
      __syncthreads();
    }
    if (rows_here == 0)
      for (int e = threadIdx.x; e <= E; e += NTH) colsum[e] = 0.f;
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += NTH) ppart[static_cast<int64_t>(blockIdx.x) * (E + 1) + e] = colsum[e];
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *ppart_rows = static_cast<int32_t>(gridDim.x);
  if (threadIdx.x == 0 && !ok) set_status(status, MOE_DEV_TIMEOUT);
}

template <int KP, int G, int NTH>
cudaError_t launch_fused_g(const Plan& p, const CUtensorMap& tmU, const CUtensorMap& tmW, const float* b_r,
                           const float* sel_bias, const float* eps, float* logits_out, int32_t* idx, float* gate,
                           float* ppart, int32_t* rows, int32_t* status, cudaStream_t s) {
  const Geometry geo = geometry(p.route_tc_n, p.E, p.n_group, p.rf_stages, G, NTH);
  auto kern = route_fused<KP, G, NTH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(geo.smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(p.rf_tiles * p.rf_cs));
  lc.blockDim = dim3(NTH);
  lc.dynamicSmemBytes = geo.smem;
  lc.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(p.rf_cs);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, tmU, tmW, p.T, p.h, p.E, p.route_tc_n, p.rf_stages, p.rf_cs, b_r, sel_bias,
                            eps, p.noisy ? 1 : 0, logits_out, idx, gate, ppart, rows, p.k, p.score_fn, p.renorm,
                            p.n_group, p.topk_group, status);
}

template <int KP>
cudaError_t launch_fused_kp(const Plan& p, const CUtensorMap& tmU, const CUtensorMap& tmW, const float* b_r,
                            const float* sel_bias, const float* eps, float* logits_out, int32_t* idx, float* gate,
                            float* ppart, int32_t* rows, int32_t* status, cudaStream_t s) {
  // 512 threads: twice the lanes per token (half the experts per lane) when the CTA's rows still
  // fit one selection pass that way; otherwise the usual lanes, so that the rows take one pass of
  // 512 / G tokens instead of two (the 128 rows of a one-CTA tile of the 128-expert router),
  // while that fits shared memory
  if (p.rf_threads == 512) {
    const int G = select_lanes_for(p.E);
    const int R = 128 / p.rf_cs;
    const bool wide = R <= 512 / (2 * G) ||
                      geometry(p.route_tc_n, p.E, p.n_group, p.rf_stages, G, 512).smem > 232448;
    if (wide) {
      switch (G) {
#define MOE_RFU_G2(gg, g2) \
  case gg: return launch_fused_g<KP, g2, 512>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
        MOE_RFU_G2(1, 2) MOE_RFU_G2(2, 4) MOE_RFU_G2(4, 8) MOE_RFU_G2(8, 16)
#undef MOE_RFU_G2
      }
    } else {
      switch (G) {
#define MOE_RFU_G1(gg) \
  case gg: return launch_fused_g<KP, gg, 512>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
        MOE_RFU_G1(1) MOE_RFU_G1(2) MOE_RFU_G1(4) MOE_RFU_G1(8)
#undef MOE_RFU_G1
      }
    }
    return cudaErrorInvalidValue;
  }
  switch (select_lanes_for(p.E)) {
#define MOE_RFU_G(gg) \
  case gg: return launch_fused_g<KP, gg, 256>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
    MOE_RFU_G(1) MOE_RFU_G(2) MOE_RFU_G(4) MOE_RFU_G(8)
#undef MOE_RFU_G
  }
  return cudaErrorInvalidValue;
}

}  // namespace rfu

cudaError_t launch_pack_router(const Plan& p, const void* W_r, const void* W_noise, void* Wt, cudaStream_t s) {
  const int N = p.route_tc_n;
  rtc::route_pack_wt<<<dim3((N + 31) / 32, (p.h + 31) / 32), dim3(32, 8), 0, s>>>(
      static_cast<const bf16*>(W_r), p.noisy ? static_cast<const bf16*>(W_noise) : nullptr, p.h, p.E, N,
      static_cast<bf16*>(Wt));
  return cudaGetLastError();
}

cudaError_t launch_route_fused(const Plan& p, const void* U, const void* Wt, const float* b_r, const float* sel_bias,
                               const float* eps, float* logits_out, int32_t* idx, float* gate, uint8_t* ws,
                               cudaStream_t s) {
  using namespace rtc;
  if (p.T == 0) return cudaSuccess;
  CUtensorMap tmU, tmW;
  if (!make_tmap(&tmU, U, static_cast<uint64_t>(p.T), p.h, BM) || !make_tmap(&tmW, Wt, p.route_tc_n, p.h, p.route_tc_n))
    return cudaErrorNotSupported;
  float* ppart = reinterpret_cast<float*>(ws + p.ws_ppart);
  int32_t* rows = ws_ppart_rows(p, ws);
  int32_t* status = ws_status(p, ws);
  if (p.k <= 2) return rfu::launch_fused_kp<2>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
  if (p.k <= 4) return rfu::launch_fused_kp<4>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
  if (p.k <= 8) return rfu::launch_fused_kp<8>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
  return rfu::launch_fused_kp<16>(p, tmU, tmW, b_r, sel_bias, eps, logits_out, idx, gate, ppart, rows, status, s);
}

}  // namespace moe
