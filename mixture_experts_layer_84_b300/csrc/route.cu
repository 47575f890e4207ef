// Router: H = U W_r (+ b_r) (+ eps * softplus(U W_noise)), softmax / sigmoid
// scores, top-k with ties to the lower expert id, gates, and per-block sums
// of the scores for P_i.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section
// 路由器：打分、top-k、加权求和 (router linear, scoring, top-k, gates; the noisy
// top-k logits of Shazeer et al.), section softmax 门控还是 sigmoid 门控 (the
// scoring/renormalisation table), section 负载均衡辅助损失：推导与梯度 (P_i, and
// the sigmoid form s' = s / sum_j s_j).
//
// Two launches.  route_partial_logits streams U once: each block owns BT
// tokens and one slice of h, stages U and W_r chunks in shared memory with
// cp.async double buffering and accumulates in float32 registers; small T is
// split along h so the grid still covers the GPU.  route_select then sums the
// slices in a fixed order (run-to-run identical), adds bias and noise, and
// handles one token per warp: scores, k rounds of a warp arg-max, gates and
// the score sums.
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {

template <int EP>
struct RouteTile {
  static constexpr int THREADS = 256;
  static constexpr int TX = EP < 32 ? EP : 32;       // threads across experts
  static constexpr int TY = THREADS / TX;            // threads across tokens
  static constexpr int BT = route_bt_for(EP);
  static constexpr int TPT = BT / TY;                // tokens per thread
  static constexpr int EPT = EP / TX;                // experts per thread
  static constexpr int KC = route_kc_for(EP);
  static constexpr int UPAD = 8;                     // keeps 16-byte rows, breaks bank aliasing
  static_assert(TPT >= 1 && EPT >= 1, "tile");
};

template <typename T, int EP, bool NOISY>
__global__ void __launch_bounds__(256) route_partial_logits(const T* __restrict__ U, const T* __restrict__ W_r,
                                                            const T* __restrict__ W_noise, int64_t n_tok, int h,
                                                            int E, int splits, float* __restrict__ part,
                                                            float* __restrict__ npart) {
  using Tile = RouteTile<EP>;
  constexpr int BT = Tile::BT, KC = Tile::KC, TX = Tile::TX, TY = Tile::TY;
  constexpr int TPT = Tile::TPT, EPT = Tile::EPT, UP = KC + Tile::UPAD;
  constexpr int VE = 16 / sizeof(T);  // elements per 16-byte copy
  extern __shared__ __align__(16) uint8_t smem_raw[];
  T* Us = reinterpret_cast<T*>(smem_raw);                 // [2][BT][UP]
  T* Ws = Us + 2 * BT * UP;                               // [2][KC][EP]
  T* Wn = Ws + 2 * KC * EP;                               // [2][KC][EP] (noisy only)

  const int tid = threadIdx.x;
  const int tx = tid % TX, ty = tid / TX;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x / splits) * BT;
  const int split = blockIdx.x % splits;
  const int nkc = (h + KC - 1) / KC;
  const int kc_beg = static_cast<int>((static_cast<int64_t>(nkc) * split) / splits);
  const int kc_end = static_cast<int>((static_cast<int64_t>(nkc) * (split + 1)) / splits);
  const bool w_vec = ((E * static_cast<int>(sizeof(T))) % 16) == 0;

  // expert columns E..EP-1 of the weight tiles stay zero
  for (int i = tid; i < 2 * KC * EP * (NOISY ? 2 : 1); i += blockDim.x) Ws[i] = from_f32<T>(0.f);
  __syncthreads();

  auto load_chunk = [&](int kc, int buf) {
    const int c0 = kc * KC;
    T* us = Us + buf * BT * UP;
    for (int i = tid; i < BT * (KC / VE); i += blockDim.x) {
      const int r = i / (KC / VE), v = i % (KC / VE);
      const int64_t t = t0 + r;
      const int c = c0 + v * VE;
      const bool ok = (t < n_tok) && (c < h);
      const T* src = ok ? U + t * h + c : U;
      ptx::cp_async_16(us + r * UP + v * VE, src, ok ? 16u : 0u);
    }
    T* ws = Ws + buf * KC * EP;
    T* wn = Wn + buf * KC * EP;
    if (w_vec) {
      const int vpr = E / VE;  // 16-byte copies per weight row
      for (int i = tid; i < KC * vpr; i += blockDim.x) {
        const int r = i / vpr, v = i % vpr;
        const int c = c0 + r;
        const bool ok = c < h;
        ptx::cp_async_16(ws + r * EP + v * VE, ok ? W_r + static_cast<int64_t>(c) * E + v * VE : W_r, ok ? 16u : 0u);
        if (NOISY)
          ptx::cp_async_16(wn + r * EP + v * VE, ok ? W_noise + static_cast<int64_t>(c) * E + v * VE : W_noise,
                           ok ? 16u : 0u);
      }
    } else {
      for (int i = tid; i < KC * E; i += blockDim.x) {
        const int r = i / E, e = i % E;
        const int c = c0 + r;
        ws[r * EP + e] = c < h ? W_r[static_cast<int64_t>(c) * E + e] : from_f32<T>(0.f);
        if (NOISY) wn[r * EP + e] = c < h ? W_noise[static_cast<int64_t>(c) * E + e] : from_f32<T>(0.f);
      }
    }
    ptx::cp_async_commit();
  };

  float acc[TPT][EPT], accn[NOISY ? TPT : 1][NOISY ? EPT : 1];
#pragma unroll
  for (int i = 0; i < TPT; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) acc[i][j] = 0.f;
  if (NOISY) {
#pragma unroll
    for (int i = 0; i < (NOISY ? TPT : 1); ++i)
#pragma unroll
      for (int j = 0; j < (NOISY ? EPT : 1); ++j) accn[i][j] = 0.f;
  }

  if (kc_beg < kc_end) load_chunk(kc_beg, 0);
  for (int kc = kc_beg; kc < kc_end; ++kc) {
    const int buf = (kc - kc_beg) & 1;
    if (kc + 1 < kc_end) {
      load_chunk(kc + 1, buf ^ 1);
      ptx::cp_async_wait<1>();
    } else {
      ptx::cp_async_wait<0>();
    }
    __syncthreads();
    const T* us = Us + buf * BT * UP;
    const T* ws = Ws + buf * KC * EP;
    const T* wn = Wn + buf * KC * EP;
#pragma unroll 4
    for (int c = 0; c < KC; ++c) {
      float u[TPT], w[EPT];
#pragma unroll
      for (int i = 0; i < TPT; ++i) u[i] = to_f32(us[(ty + i * TY) * UP + c]);
#pragma unroll
      for (int j = 0; j < EPT; ++j) w[j] = to_f32(ws[c * EP + tx + j * TX]);
#pragma unroll
      for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = fmaf(u[i], w[j], acc[i][j]);
      if (NOISY) {
#pragma unroll
        for (int j = 0; j < EPT; ++j) w[j] = to_f32(wn[c * EP + tx + j * TX]);
#pragma unroll
        for (int i = 0; i < (NOISY ? TPT : 1); ++i)
#pragma unroll
          for (int j = 0; j < (NOISY ? EPT : 1); ++j) accn[i][j] = fmaf(u[i], w[j], accn[i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    const int64_t t = t0 + ty + i * TY;
    if (t >= n_tok) continue;
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tx + j * TX;
      if (e >= E) continue;
      const int64_t o = (static_cast<int64_t>(split) * n_tok + t) * E + e;
      part[o] = acc[i][j];
      if (NOISY) npart[o] = accn[NOISY ? i : 0][NOISY ? j : 0];
    }
  }
}

__device__ __forceinline__ float softplus_f32(float x) { return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

constexpr int KMAX = 16;
constexpr int SEL_WARPS = 8;
constexpr int SEL_TPW = kSelTokens / SEL_WARPS;  // tokens per warp

// One token per warp.  EV = logits held per lane (expert e = lane + 32 m).
template <int EV>
__global__ void __launch_bounds__(SEL_WARPS * 32) route_select(
    const float* __restrict__ part, const float* __restrict__ npart, int splits, const float* __restrict__ b_r,
    const float* __restrict__ eps, const float* __restrict__ logits_in, float* __restrict__ logits_out,
    int32_t* __restrict__ idx, float* __restrict__ gate, float* __restrict__ ppart, int64_t n_tok, int E, int k,
    int score_fn, int renorm) {
  __shared__ float red[SEL_WARPS][EV * 32];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float pacc[EV];
#pragma unroll
  for (int m = 0; m < EV; ++m) pacc[m] = 0.f;

  for (int tt = 0; tt < SEL_TPW; ++tt) {
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * SEL_WARPS + warp) * SEL_TPW + tt;
    if (t >= n_tok) break;  // warp-uniform
    float v[EV];
#pragma unroll
    for (int m = 0; m < EV; ++m) {
      const int e = lane + 32 * m;
      float x = -FLT_MAX;
      if (e < E) {
        if (logits_in) {
          x = logits_in[t * E + e];
        } else {
          x = 0.f;
          for (int s = 0; s < splits; ++s) x += part[(static_cast<int64_t>(s) * n_tok + t) * E + e];
          if (b_r) x += b_r[e];
          if (npart) {
            float n = 0.f;
            for (int s = 0; s < splits; ++s) n += npart[(static_cast<int64_t>(s) * n_tok + t) * E + e];
            x = fmaf(eps[t * E + e], softplus_f32(n), x);
          }
        }
        if (logits_out) logits_out[t * E + e] = x;
      }
      v[m] = x;
    }

    // scores of every expert (for P) -- softmax over E or independent sigmoids
    float s[EV];
    float mx = 0.f, denom_all = 0.f;
    if (score_fn == MOE_SCORE_SOFTMAX) {
      float lm = -FLT_MAX;
#pragma unroll
      for (int m = 0; m < EV; ++m)
        if (lane + 32 * m < E) lm = fmaxf(lm, v[m]);
      mx = warp_max(lm);
      float ls = 0.f;
#pragma unroll
      for (int m = 0; m < EV; ++m) {
        s[m] = (lane + 32 * m < E) ? expf(v[m] - mx) : 0.f;
        ls += s[m];
      }
      denom_all = warp_sum(ls);
#pragma unroll
      for (int m = 0; m < EV; ++m) pacc[m] += s[m] / denom_all;
    } else {
      float ls = 0.f;
#pragma unroll
      for (int m = 0; m < EV; ++m) {
        s[m] = (lane + 32 * m < E) ? 1.f / (1.f + expf(-v[m])) : 0.f;
        ls += s[m];
      }
      const float tot = warp_sum(ls);
#pragma unroll
      for (int m = 0; m < EV; ++m) pacc[m] += s[m] / tot;
    }

    // k rounds of arg-max: highest logit, ties to the lower expert id
    uint32_t taken = 0;
    float sel_sum = 0.f, my_s = 0.f;
    int my_e = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k) break;
      float bv = -FLT_MAX;
      int be = 0x7fffffff;
#pragma unroll
      for (int m = 0; m < EV; ++m) {
        const int e = lane + 32 * m;
        if (e < E && !((taken >> m) & 1u) && (v[m] > bv || be == 0x7fffffff)) {
          bv = v[m];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      const float sj = (score_fn == MOE_SCORE_SOFTMAX) ? expf(bv - mx) / denom_all : 1.f / (1.f + expf(-bv));
      sel_sum += sj;
      if (lane == j) {
        my_e = be;
        my_s = sj;
      }
    }
    if (lane < k) {
      idx[t * k + lane] = my_e;
      gate[t * k + lane] = renorm ? my_s / sel_sum : my_s;
    }
  }

  // per-block score sums in a fixed order: warps 0..7
#pragma unroll
  for (int m = 0; m < EV; ++m) red[warp][lane + 32 * m] = pacc[m];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < SEL_WARPS; ++w) acc += red[w][e];
    ppart[static_cast<int64_t>(blockIdx.x) * E + e] = acc;
  }
}

namespace {

template <typename T, int EP, bool NOISY>
cudaError_t launch_partial(const Plan& p, const void* U, const void* W_r, const void* W_noise, float* part,
                           float* npart, cudaStream_t s) {
  using Tile = RouteTile<EP>;
  const size_t smem = sizeof(T) * (2 * Tile::BT * (Tile::KC + Tile::UPAD) + 2 * Tile::KC * EP * (NOISY ? 2 : 1));
  auto kern = route_partial_logits<T, EP, NOISY>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(static_cast<unsigned>(p.route_rowblocks * p.route_splits));
  kern<<<grid, Tile::THREADS, smem, s>>>(static_cast<const T*>(U), static_cast<const T*>(W_r),
                                         static_cast<const T*>(W_noise), p.T, p.h, p.E, p.route_splits, part, npart);
  return cudaGetLastError();
}

template <typename T, int EP>
cudaError_t launch_partial_n(const Plan& p, const void* U, const void* W_r, const void* W_noise, float* part,
                             float* npart, cudaStream_t s) {
  return p.noisy ? launch_partial<T, EP, true>(p, U, W_r, W_noise, part, npart, s)
                 : launch_partial<T, EP, false>(p, U, W_r, W_noise, part, npart, s);
}

template <typename T>
cudaError_t launch_partial_t(const Plan& p, const void* U, const void* W_r, const void* W_noise, float* part,
                             float* npart, cudaStream_t s) {
  switch (p.route_ep) {
    case 8: return launch_partial_n<T, 8>(p, U, W_r, W_noise, part, npart, s);
    case 16: return launch_partial_n<T, 16>(p, U, W_r, W_noise, part, npart, s);
    case 32: return launch_partial_n<T, 32>(p, U, W_r, W_noise, part, npart, s);
    case 64: return launch_partial_n<T, 64>(p, U, W_r, W_noise, part, npart, s);
    case 128: return launch_partial_n<T, 128>(p, U, W_r, W_noise, part, npart, s);
    case 256: return launch_partial_n<T, 256>(p, U, W_r, W_noise, part, npart, s);
    case 512: return launch_partial_n<T, 512>(p, U, W_r, W_noise, part, npart, s);
    case 1024: return launch_partial_n<T, 1024>(p, U, W_r, W_noise, part, npart, s);
  }
  return cudaErrorInvalidValue;
}

template <int EV>
cudaError_t launch_select_ev(const Plan& p, const float* part, const float* npart, int splits, const float* b_r,
                             const float* eps, const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                             float* ppart, cudaStream_t s) {
  route_select<EV><<<p.sel_blocks, SEL_WARPS * 32, 0, s>>>(part, npart, splits, b_r, eps, logits_in, logits_out,
                                                           idx, gate, ppart, p.T, p.E, p.k, p.score_fn, p.renorm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const Plan& p, const void* U, const void* W_r, const float* b_r, const void* W_noise,
                         const float* eps, const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                         uint8_t* ws, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  float* part = reinterpret_cast<float*>(ws + p.ws_part);
  float* npart = p.noisy ? reinterpret_cast<float*>(ws + p.ws_npart) : nullptr;
  float* ppart = reinterpret_cast<float*>(ws + p.ws_ppart);
  int splits = p.route_splits;
  if (!logits_in) {
    cudaError_t e = p.route_tc_n > 0 ? launch_route_logits_tc(p, U, W_r, W_noise, part, npart, ws, s)
                    : p.bf16         ? launch_partial_t<bf16>(p, U, W_r, W_noise, part, npart, s)
                                     : launch_partial_t<float>(p, U, W_r, W_noise, part, npart, s);
    if (e != cudaSuccess) return e;
  } else {
    npart = nullptr;
    splits = 0;
  }
  const int ev = (p.E + 31) / 32;
  if (ev <= 1) return launch_select_ev<1>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
  if (ev <= 2) return launch_select_ev<2>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
  if (ev <= 4) return launch_select_ev<4>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
  if (ev <= 8) return launch_select_ev<8>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
  if (ev <= 16)
    return launch_select_ev<16>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
  return launch_select_ev<32>(p, part, npart, splits, b_r, eps, logits_in, logits_out, idx, gate, ppart, s);
}

}  // namespace moe
