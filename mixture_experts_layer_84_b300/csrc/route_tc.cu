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
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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

}  // namespace moe
