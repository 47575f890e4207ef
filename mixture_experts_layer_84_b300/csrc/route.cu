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
// Two launches.  The logits come in h-slices: from route_logits_tc (bf16, tensor cores, in
// route_tc.cu) or from route_partial_logits here (CUDA cores), which streams U once: each block
// owns BT tokens and one slice of h, stages U and W_r chunks in shared memory with cp.async
// double buffering and accumulates in float32 registers; small T is split along h so the grid
// still covers the GPU.  route_select then
//   1. stages a tile of tokens: the whole block sums each logit's slices in a fixed order
//      (run-to-run identical) and adds bias and noise;
//   2. gives each token G lanes (G = E / 32 rounded up to a power of two), each with a chunk of
//      the experts: maximum and exp-sum by butterflies, then (section 设备受限与节点受限路由,
//      with groups) the group scores and the kept-group mask, then a running top-k list per
//      lane on the selection key (the logit, or score + bias with a loss-free selection bias,
//      section 无辅助损失的负载均衡), merged across the lanes bitonically; gates from the scores;
//   3. writes the tile's per-expert score sums and LSE^2 sums (section Router z-loss) for
//      moe_combine's statistics.
#include <float.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "select.cuh"

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

// Selection over G lanes per token, TB = blockDim.x / G tokens per block.
//   1. the block stages the tile's final logits in shared memory with coalesced loads: slice sums
//      added in slice order, + bias, + eps * softplus(noise slice sums) (or the given logits in
//      stage mode); the logits also go to logits_out here;
//   2. select_tokens (select.cuh): scores, the top-k (logits, or score + bias with a selection
//      bias; limited to the best groups with n_group > 1), gates, normalised scores, LSE^2;
//   3. score_column_sums: the block's per-expert score sums and LSE^2 sum in a ppart row (E + 1
//      floats) for moe_combine's statistics.
// KP = k rounded up to a power of two (the lists live in registers).
template <int KP, int G>
__global__ void __launch_bounds__(SELECT_THREADS) route_select(
    const float* __restrict__ part, const float* __restrict__ npart, int splits, const float* __restrict__ b_r,
    const float* __restrict__ sel_bias, const float* __restrict__ eps, const float* __restrict__ logits_in,
    float* __restrict__ logits_out, int32_t* __restrict__ idx, float* __restrict__ gate, float* __restrict__ ppart,
    int32_t* __restrict__ ppart_rows, int64_t n_tok, int E, int k, int score_fn, int renorm, int n_group,
    int topk_group) {
  const int TB = static_cast<int>(blockDim.x) / G;
  extern __shared__ float sx[];  // [TB][LD], then zsq[TB], then (groups) gsc[TB][n_group]
  const SelLayout L(E, G);
  float* zsq = sx + TB * L.LD;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TB;
  const int rows = static_cast<int>(n_tok - t0 < TB ? n_tok - t0 : TB);
  if (blockIdx.x == 0 && threadIdx.x == 0) *ppart_rows = static_cast<int32_t>(gridDim.x);

  // 1. final logits of the tile; rows t0 .. t0 + rows - 1 are contiguous in every input, so the
  // whole block sweeps the tile's rows x E entries in order (coalesced, and every lane busy
  // even when E is small)
  const int n_el = rows * E;
  const bool e_pow2 = (E & (E - 1)) == 0;
  const int e_shift = __ffs(E) - 1;
#pragma unroll 2
  for (int i = threadIdx.x; i < n_el; i += blockDim.x) {
    const int r = e_pow2 ? i >> e_shift : i / E, e = i - r * E;
    const int64_t g = t0 * E + i;
    float x;
    if (logits_in) {
      x = logits_in[g];
    } else {
      // every slice's value is loaded before any is added (one memory latency, not `splits`),
      // then added in slice order
      const int64_t stride = n_tok * E;
      float v[16];
#pragma unroll
      for (int sp = 0; sp < 16; ++sp) v[sp] = sp < splits ? part[sp * stride + g] : 0.f;
      x = v[0];
#pragma unroll
      for (int sp = 1; sp < 16; ++sp)
        if (sp < splits) x += v[sp];
      if (b_r) x += b_r[e];
      if (npart) {
#pragma unroll
        for (int sp = 0; sp < 16; ++sp) v[sp] = sp < splits ? npart[sp * stride + g] : 0.f;
        float nz = v[0];
#pragma unroll
        for (int sp = 1; sp < 16; ++sp)
          if (sp < splits) nz += v[sp];
        x = fmaf(eps[g], softplus_f32(nz), x);
      }
    }
    if (logits_out) logits_out[g] = x;
    sx[L.at(r, e)] = x;
  }
  __syncthreads();

  // 2. G lanes per token: scores, top-k, gates
  select_tokens<KP, G>(sx, zsq, zsq + TB, rows, t0, E, k, score_fn, renorm, n_group, topk_group, sel_bias, idx, gate);
  __syncthreads();

  // 3. the tile's score sums and z-loss sum, tokens in order
  score_column_sums(sx, zsq, rows, E, G, ppart + static_cast<int64_t>(blockIdx.x) * (E + 1), false);
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

template <int KP, int G>
cudaError_t launch_select_g(const Plan& p, const float* part, const float* npart, int splits, const float* b_r,
                            const float* sel_bias, const float* eps, const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                            float* ppart, int32_t* rows, cudaStream_t s) {
  const size_t smem = select_smem_bytes(p.E, p.sel_tokens, p.n_group);
  auto kern = route_select<KP, G>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kern<<<p.sel_blocks, p.sel_threads, smem, s>>>(part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx,
                                                  gate, ppart, rows, p.T, p.E, p.k, p.score_fn, p.renorm,
                                                  p.n_group, p.topk_group);
  return cudaGetLastError();
}

template <int KP>
cudaError_t launch_select_kp(const Plan& p, const float* part, const float* npart, int splits, const float* b_r,
                             const float* sel_bias, const float* eps, const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                             float* ppart, int32_t* rows, cudaStream_t s) {
  switch (select_lanes_for(p.E)) {
#define MOE_SEL_G(gg) \
  case gg: return launch_select_g<KP, gg>(p, part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx, gate, ppart, rows, s);
    MOE_SEL_G(1) MOE_SEL_G(2) MOE_SEL_G(4) MOE_SEL_G(8) MOE_SEL_G(16) MOE_SEL_G(32)
#undef MOE_SEL_G
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_route(const Plan& p, const void* U, const void* W_r, const float* b_r, const float* sel_bias,
                         const void* W_noise, const float* eps, const float* logits_in, float* logits_out, int32_t* idx, float* gate,
                         uint8_t* ws, cudaStream_t s, const void* W_r_packed) {
  if (p.T == 0) return cudaSuccess;
  if (!logits_in && p.route_fused) {
    const void* Wt = W_r_packed;
    if (!Wt) {
      void* w = ws + p.ws_wt;
      const cudaError_t e = launch_pack_router(p, W_r, W_noise, w, s);
      if (e != cudaSuccess) return e;
      Wt = w;
    }
    return launch_route_fused(p, U, Wt, b_r, sel_bias, eps, logits_out, idx, gate, ws, s);
  }
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
  int32_t* rows = ws_ppart_rows(p, ws);
  if (p.k <= 2) return launch_select_kp<2>(p, part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx, gate, ppart, rows, s);
  if (p.k <= 4) return launch_select_kp<4>(p, part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx, gate, ppart, rows, s);
  if (p.k <= 8) return launch_select_kp<8>(p, part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx, gate, ppart, rows, s);
  return launch_select_kp<16>(p, part, npart, splits, b_r, sel_bias, eps, logits_in, logits_out, idx, gate, ppart, rows, s);
}

}  // namespace moe
