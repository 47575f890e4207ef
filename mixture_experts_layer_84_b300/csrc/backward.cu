// Backward of the router side of the MoE layer: the combine and the gates.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe):
//   section 路由器：打分、top-k、加权求和 (how the router learns): with the
//   upstream gradient delta_t = dL/dh'_t, dL/dg_{i,t} = delta_t^T FFN_i(u_t) for
//   the selected experts, passed on through dg/dH to the logits;
//   section 负载均衡辅助损失：推导与梯度 (梯度往哪推): f is a constant and
//   d(sum_i f_i P_i)/dH_{t,k} = (1/T) s_k (f_k - sum_i f_i s_i) (softmax),
//   (1/T) s'_k (1 - s_k) (f_k - sum_i f_i s'_i) (sigmoid, s' = s / sum_j s_j);
//   section Router z-loss: dL_z/dH_{t,k} = (2/T) LSE(H_t) softmax(H_t)_k.
//
// combine_backward: one warp per token.  For each kept pair (choice order)
//   d_gate = dO_t . Y[row] (float32, each lane's partial sum then a fixed
//   butterfly) and dY[row] = g dO_t (rounded once); a dropped pair gets
//   d_gate = 0 and no dY row.
// dispatch_backward: dU_t = dO_t + sum of the dX rows of its kept pairs (the
//   residual and the permute's backward), one warp per token.
// route_backward: G lanes per token (as in the selection), each with a chunk
//   of <= 32 experts read straight from the float32 logits:
//   dH = dg/dH^T d_gate + w_aux * d(E sum f P)/dH + w_z * dL_z/dH.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

template <typename T>
__global__ void __launch_bounds__(256) combine_backward(const uint4* __restrict__ dO, const uint4* __restrict__ Y,
                                                        const int32_t* __restrict__ slot_row,
                                                        const float* __restrict__ gate, float* __restrict__ d_gate,
                                                        uint4* __restrict__ dY, int64_t n_tok, int k, int vpr,
                                                        int64_t rows_cap, int32_t* status) {
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
    for (int j = 0; j < k; ++j) {
      const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
      const float g = __shfl_sync(0xffffffffu, my_g, j);
      float dot = 0.f;
      if (r >= 0) {
        for (int v = lane; v < vpr; v += 32) {
          float o[N], y[N];
          Vec16<T>::unpack(ldg_stream(dO + t * vpr + v), o);
          Vec16<T>::unpack(ldg_stream(Y + static_cast<int64_t>(r) * vpr + v), y);
#pragma unroll
          for (int i = 0; i < N; ++i) {
            dot = fmaf(o[i], y[i], dot);
            o[i] *= g;
          }
          dY[static_cast<int64_t>(r) * vpr + v] = Vec16<T>::pack(o);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      if (lane == 0) d_gate[t * k + j] = dot;
    }
  }
}

constexpr int RB_THREADS = 256;

template <int G>
__global__ void __launch_bounds__(RB_THREADS) route_backward(const float* __restrict__ H,
                                                             const int32_t* __restrict__ idx,
                                                             const float* __restrict__ d_gate,
                                                             const int32_t* __restrict__ counts_routed, int64_t n_tok,
                                                             int E, int k, int score_fn, int renorm, float w_aux,
                                                             float w_z, float* __restrict__ dH) {
  constexpr int TB = RB_THREADS / G;
  const int r = threadIdx.x / G, g = threadIdx.x % G;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * TB + r;
  const bool tok = t < n_tok;
  const int C = (E + G - 1) / G;
  const int e0 = g * C, e1 = min(E, e0 + C);
  const float* Ht = H + (tok ? t : 0) * E;
  const bool softmax = score_fn == MOE_SCORE_SOFTMAX;
  const float inv_tk = 1.f / static_cast<float>(n_tok * k);

  // per-token reductions over all E: max, exp-sum, sigmoid sum
  float mx = -INFINITY;
  if (tok)
    for (int e = e0; e < e1; ++e) mx = fmaxf(mx, Ht[e]);
#pragma unroll
  for (int o = 1; o < G; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum_exp = 0.f, sum_sig = 0.f;
  if (tok) {
    for (int e = e0; e < e1; ++e) {
      sum_exp += expf(Ht[e] - mx);
      sum_sig += 1.f / (1.f + expf(-Ht[e]));
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    sum_exp += __shfl_xor_sync(0xffffffffu, sum_exp, o);
    sum_sig += __shfl_xor_sync(0xffffffffu, sum_sig, o);
  }
  // the score-weighted mean load sum_i f_i s_i (sigmoid: with s' = s / sum s)
  float fs = 0.f;
  if (tok && w_aux != 0.f) {
    for (int e = e0; e < e1; ++e) {
      const float se = softmax ? expf(Ht[e] - mx) / sum_exp : (1.f / (1.f + expf(-Ht[e]))) / sum_sig;
      fs = fmaf(static_cast<float>(counts_routed[e]) * inv_tk, se, fs);
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) fs += __shfl_xor_sync(0xffffffffu, fs, o);

  // dL/ds of the selected experts (every lane of the token computes the same k values)
  float dsel[16];
  int sel[16];
  float sum_ds_s = 0.f;  // sum_j ds_j s_j, the softmax Jacobian's shared term
  if (tok) {
    float sv[16], S = 0.f, dg_g = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      sel[j] = -1;
      dsel[j] = 0.f;
      sv[j] = 0.f;
      if (j < k) {
        const int e = idx[t * k + j];
        if (e >= 0 && e < E) {  // an id outside [0, E) contributes nothing
          sel[j] = e;
          const float x = Ht[e];
          sv[j] = softmax ? expf(x - mx) / sum_exp : 1.f / (1.f + expf(-x));
          S += sv[j];
        }
      }
    }
    if (renorm) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < k) dg_g = fmaf(d_gate[t * k + j], sv[j] / S, dg_g);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < k && sel[j] >= 0) {
        const float dgj = d_gate[t * k + j];
        dsel[j] = renorm ? (dgj - dg_g) / S : dgj;
        sum_ds_s = fmaf(dsel[j], sv[j], sum_ds_s);
      }
    }
  }
  if (!tok) return;
  const float lse = mx + logf(sum_exp);
  const float aux_scale = static_cast<float>(E) / static_cast<float>(n_tok);
  const float z_scale = 2.f / static_cast<float>(n_tok) * lse;
  for (int e = e0; e < e1; ++e) {
    const float x = Ht[e];
    const float sm = expf(x - mx) / sum_exp;
    const float sg = 1.f / (1.f + expf(-x));
    float ds = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < k && sel[j] == e) ds += dsel[j];
    float d = softmax ? sm * (ds - sum_ds_s) : ds * sg * (1.f - sg);
    if (w_aux != 0.f) {
      const float fe = static_cast<float>(counts_routed[e]) * inv_tk;
      d += w_aux * aux_scale * (softmax ? sm * (fe - fs) : (sg / sum_sig) * (1.f - sg) * (fe - fs));
    }
    if (w_z != 0.f) d += w_z * z_scale * sm;
    dH[t * E + e] = d;
  }
}

// dU_t = dO_t + sum over kept j (choice order) of dX[row(t, j)]: the residual plus the backward of
// the permute X = U[token of each row]; one warp per token, float32 accumulation, one rounding.
template <typename T>
__global__ void __launch_bounds__(256) dispatch_backward(const uint4* __restrict__ dO, const uint4* __restrict__ dX,
                                                         const int32_t* __restrict__ slot_row,
                                                         const uint4* __restrict__ extra,
                                                         const uint4* __restrict__ more, int n_more,
                                                         uint4* __restrict__ dU, int64_t n_tok, int k, int vpr,
                                                         int64_t rows_cap, int32_t* status) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x % 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x / 32);
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; t < n_tok; t += warps) {
    int32_t my_row = -1;
    if (lane < k) {
      my_row = slot_row[t * k + lane];
      if (my_row < -1 || my_row >= rows_cap) {
        set_status(status, MOE_DEV_BAD_ROW);
        my_row = -1;
      }
    }
    for (int v0 = 0; v0 < vpr; v0 += 32) {
      const int v = v0 + lane;
      float acc[N];
      if (v < vpr) {
        Vec16<T>::unpack(ldg_stream(dO + t * vpr + v), acc);
        // the router's and the shared experts' input gradients (each rounded once already)
        for (int a = 0; a < 1 + n_more; ++a) {
          const uint4* src = a == 0 ? extra : more + static_cast<int64_t>(a - 1) * n_tok * vpr;
          if (!src) continue;
          float x[N];
          Vec16<T>::unpack(ldg_stream(src + t * vpr + v), x);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] += x[i];
        }
      }
      for (int j = 0; j < k; ++j) {
        const int32_t r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0 || v >= vpr) continue;
        float x[N];
        Vec16<T>::unpack(ldg_stream(dX + static_cast<int64_t>(r) * vpr + v), x);
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] += x[i];
      }
      if (v < vpr) dU[t * vpr + v] = Vec16<T>::pack(acc);
    }
  }
}

cudaError_t launch_dispatch_backward(const Plan& p, const void* dO, const void* dX, const int32_t* slot_row, void* dU,
                                     uint8_t* ws, cudaStream_t s, const void* extra, const void* more, int n_more) {
  if (p.T == 0) return cudaSuccess;
  const int vpr = p.h * (p.bf16 ? 2 : 4) / 16;
  const int64_t want = (p.T + 7) / 8;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
  int32_t* status = ws_status(p, ws);
  if (p.bf16)
    dispatch_backward<bf16><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(dO), static_cast<const uint4*>(dX),
                                                   slot_row, static_cast<const uint4*>(extra),
                                                   static_cast<const uint4*>(more), more ? n_more : 0,
                                                   static_cast<uint4*>(dU), p.T, p.k, vpr, p.Tk, status);
  else
    dispatch_backward<float><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(dO), static_cast<const uint4*>(dX),
                                                    slot_row, static_cast<const uint4*>(extra),
                                                    static_cast<const uint4*>(more), more ? n_more : 0,
                                                    static_cast<uint4*>(dU), p.T, p.k, vpr, p.Tk, status);
  return cudaGetLastError();
}

// [dH | dN] in bf16, rows of rb_np columns (zero past the used ones): dN = dH * eps * sigmoid(U W_noise),
// the noise logits summed from the router's h-slices in slice order.
__global__ void router_grad_pack(const float* __restrict__ dH, const float* __restrict__ eps,
                                 const float* __restrict__ npart, int splits, int64_t n_tok, int E, int np,
                                 bf16* __restrict__ out) {
  const int64_t n = n_tok * np;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = i / np;
    const int c = static_cast<int>(i - t * np);
    float v = 0.f;
    if (c < E) {
      v = dH[t * E + c];
    } else if (npart && c < 2 * E) {
      const int e = c - E;
      float z = npart[t * E + e];
      for (int sp = 1; sp < splits; ++sp) z += npart[(static_cast<int64_t>(sp) * n_tok + t) * E + e];
      v = dH[t * E + e] * eps[t * E + e] / (1.f + __expf(-z));
    }
    out[i] = __float2bfloat16_rn(v);
  }
}

// [W_r | W_noise] as a bf16 [h, np] matrix (zero past the used columns).
template <typename T>
__global__ void router_weight_pack(const T* __restrict__ W_r, const T* __restrict__ W_noise, int h, int E, int np,
                                   bf16* __restrict__ out) {
  const int64_t n = static_cast<int64_t>(h) * np;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / np;
    const int c = static_cast<int>(i - r * np);
    float v = 0.f;
    if (c < E)
      v = to_f32(W_r[r * E + c]);
    else if (W_noise && c < 2 * E)
      v = to_f32(W_noise[r * E + (c - E)]);
    out[i] = __float2bfloat16_rn(v);
  }
}

// dW [h, np] float32 -> dW_r [h, E] and dW_noise [h, E].
__global__ void router_wgrad_split(const float* __restrict__ dW, int h, int E, int np, float* __restrict__ dW_r,
                                   float* __restrict__ dW_noise) {
  const int64_t n = static_cast<int64_t>(h) * E;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / E;
    const int e = static_cast<int>(i - r * E);
    dW_r[i] = dW[r * np + e];
    if (dW_noise) dW_noise[i] = dW[r * np + E + e];
  }
}

// db_r[e] = sum over tokens of dH[t, e]: block b owns 32 experts (lane = expert), warp w adds
// rows w, w + 32, ..., then warp 0 adds the 32 warp sums in order.
__global__ void __launch_bounds__(1024) column_sums(const float* __restrict__ dH, int64_t n_tok, int E,
                                                    float* __restrict__ out) {
  __shared__ float part[32][33];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < E)
    for (int64_t t = warp; t < n_tok; t += 32) s += dH[t * E + e];
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < E) {
    float tot = 0.f;
    for (int w = 0; w < 32; ++w) tot += part[w][lane];
    out[e] = tot;
  }
}

cudaError_t launch_router_input_backward(const Plan& p, const void* U, const void* W_r, const void* W_noise,
                                         const float* eps, const float* dH, void* dU_r, float* dW_r, float* dW_noise,
                                         float* db_r, uint8_t* ws, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  int32_t* status = ws_status(p, ws);
  bf16* dHb = reinterpret_cast<bf16*>(ws + p.ws_rb_dh);
  bf16* Wb = reinterpret_cast<bf16*>(ws + p.ws_rb_w);
  float* dW = reinterpret_cast<float*>(ws + p.ws_rb_dw);
  const float* npart = nullptr;
  int splits = 1;
  if (p.noisy) {
    // the noise logits U W_noise again, as h-slice sums in the router's workspace
    float* part = reinterpret_cast<float*>(ws + p.ws_part);
    float* np_ = reinterpret_cast<float*>(ws + p.ws_npart);
    const cudaError_t e = launch_route_logits_tc(p, U, W_r, W_noise, part, np_, ws, s);
    if (e != cudaSuccess) return e;
    npart = np_;
    splits = p.route_splits;
  }
  const int blocks = current_sm_count() * 4;
  router_grad_pack<<<blocks, 256, 0, s>>>(dH, p.noisy ? eps : nullptr, npart, splits, p.T, p.E, p.rb_np, dHb);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  router_weight_pack<bf16><<<blocks, 256, 0, s>>>(static_cast<const bf16*>(W_r),
                                                  p.noisy ? static_cast<const bf16*>(W_noise) : nullptr, p.h, p.E,
                                                  p.rb_np, Wb);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // dU_r = [dH | dN] [W_r | W_noise]^T: M = T, N = h, K = rb_np
  e = launch_dense_gemm_tc(dHb, p.T, p.rb_np, Wb, p.h, dU_r, status, s);
  if (e != cudaSuccess) return e;
  // [dW_r | dW_noise] = U^T [dH | dN]: M = h, N = rb_np, K = T
  e = launch_dense_wgrad_tc(U, dHb, p.T, p.h, p.rb_np, dW, status, s);
  if (e != cudaSuccess) return e;
  router_wgrad_split<<<blocks, 256, 0, s>>>(dW, p.h, p.E, p.rb_np, dW_r, p.noisy ? dW_noise : nullptr);
  e = cudaGetLastError();
  if (e != cudaSuccess || !db_r) return e;
  column_sums<<<(p.E + 31) / 32, 1024, 0, s>>>(dH, p.T, p.E, db_r);
  return cudaGetLastError();
}

cudaError_t launch_combine_backward(const Plan& p, const void* dO, const void* Y, const int32_t* slot_row,
                                    const float* gate, float* d_gate, void* dY, uint8_t* ws, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  const int vpr = p.h * (p.bf16 ? 2 : 4) / 16;
  const int64_t want = (p.T + 7) / 8;
  const int blocks = static_cast<int>(std::min<int64_t>(want, static_cast<int64_t>(current_sm_count()) * 8));
  int32_t* status = ws_status(p, ws);
  if (p.bf16)
    combine_backward<bf16><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(dO), static_cast<const uint4*>(Y),
                                                  slot_row, gate, d_gate, static_cast<uint4*>(dY), p.T, p.k, vpr, p.Tk,
                                                  status);
  else
    combine_backward<float><<<blocks, 256, 0, s>>>(static_cast<const uint4*>(dO), static_cast<const uint4*>(Y),
                                                   slot_row, gate, d_gate, static_cast<uint4*>(dY), p.T, p.k, vpr,
                                                   p.Tk, status);
  return cudaGetLastError();
}

cudaError_t launch_route_backward(const Plan& p, const float* logits, const int32_t* idx, const float* d_gate,
                                  const int32_t* counts_routed, float w_aux, float w_z, float* dH, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  switch (select_lanes_for(p.E)) {
#define MOE_RB_G(gg)                                                                                          \
  case gg: {                                                                                                  \
    const int64_t blocks = (p.T + RB_THREADS / gg - 1) / (RB_THREADS / gg);                                   \
    route_backward<gg><<<static_cast<unsigned>(blocks), RB_THREADS, 0, s>>>(                                  \
        logits, idx, d_gate, counts_routed, p.T, p.E, p.k, p.score_fn, p.renorm, w_aux, w_z, dH);             \
    return cudaGetLastError();                                                                                \
  }
    MOE_RB_G(1) MOE_RB_G(2) MOE_RB_G(4) MOE_RB_G(8) MOE_RB_G(16) MOE_RB_G(32)
#undef MOE_RB_G
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
