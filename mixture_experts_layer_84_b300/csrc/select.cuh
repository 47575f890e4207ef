// Scoring, top-k selection and gates of a tile of tokens whose final router logits are staged in
// shared memory, and the tile's per-expert score sums for P_i and LSE^2 sum for the z-loss.  Used
// by the selection kernel (route.cu) and by the fused router (route_tc.cu).
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 路由器：打分、top-k、加权求和
// (scores, top-k, gates), section softmax 门控还是 sigmoid 门控 (softmax or sigmoid scores, gates
// with or without renormalisation), section 负载均衡辅助损失：推导与梯度 (P_i, the sigmoid form
// s' = s / sum_j s_j), section Router z-loss 与数值稳定 (L_z = (1/T) sum_t LSE(H_t)^2), section
// 无辅助损失的负载均衡 (selection on score + bias) and section 设备受限与节点受限路由 (top-k limited
// to the best groups).
//
// Layout of the staged tile: each token has G lanes (G = E / 32 rounded up to a power of two);
// lane g owns the expert chunk [g C, (g+1) C), C = ceil(E / G), stored with an odd stride CS so
// that the 32 lanes of a warp hit 32 different banks.  Token r, expert e sits at
// sx[r LD + (e / C) CS + e % C], LD = G CS.
#pragma once

#include <float.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int KMAX = 16;

// softplus(x) = max(x, 0) + log(1 + e^-|x|) with the fast exponential and logarithm: an absolute
// error of a few 1e-7, against noise logits of order one.
__device__ __forceinline__ float softplus_f32(float x) { return fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x))); }

// (value, expert id) order of the selection: larger value first, equal values by the lower id.
__device__ __forceinline__ bool before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// 1 / (1 + e^-x) with a correctly rounded reciprocal (the same value as the IEEE division).
__device__ __forceinline__ float sigmoid_f32(float x) { return __frcp_rn(1.f + __expf(-x)); }

// (v, i) into the list (tv, ti), kept in `before` order, the last entry dropping out.  All KP
// comparisons are made first and every entry then takes its new value independently (the entries
// from the insertion point on shift down by one), so the dependency chain is a few instructions
// long instead of KP compare-and-swaps.
template <int KP>
__device__ __forceinline__ void insert_sorted(float (&tv)[KP], int (&ti)[KP], float v, int i) {
  bool gt[KP];
#pragma unroll
  for (int j = 0; j < KP; ++j) gt[j] = before(v, i, tv[j], ti[j]);
#pragma unroll
  for (int j = KP - 1; j > 0; --j) {
    tv[j] = gt[j - 1] ? tv[j - 1] : (gt[j] ? v : tv[j]);
    ti[j] = gt[j - 1] ? ti[j - 1] : (gt[j] ? i : ti[j]);
  }
  tv[0] = gt[0] ? v : tv[0];
  ti[0] = gt[0] ? i : ti[0];
}

struct SelLayout {
  int C, CS, LD;
  __device__ __forceinline__ SelLayout(int E, int G) {
    C = (E + G - 1) / G;
    CS = (C & 1) ? C + 2 : C + 1;  // odd
    LD = G * CS;
  }
  __device__ __forceinline__ int at(int r, int e) const {
    const int cg = e / C;
    return r * LD + cg * CS + (e - cg * C);
  }
};

// Step 2 for the staged tokens r = threadIdx.x / G < rows (global ids t0 + r): the G lanes of a
// token combine their chunks' maxima and exp-sums with xor shuffles; with groups (n_group > 1)
// each lane scores groups g, g + G, ... (the sum of a group's k / topk_group best affinities,
// score + bias with a selection bias) into gsc[r][n_group] and every lane of the token ranks them
// into a keep mask; each lane keeps a running top-KP list of its chunk keyed by the logit (or
// score + bias), the lanes merge their lists bitonically (the elementwise better of one list and
// the other reversed is bitonic and holds the top KP of both); the gates come from the selected
// experts' scores.  Then the normalised scores (for P) are written back in place and LSE^2 into
// zsq[r].  Every thread of the block must call this (the shuffles span whole warps).  Scores use
// the fast exponential (a few ulps; the selection compares logits, or score + bias with a margin
// far above that), and the normalised scores one reciprocal of the denominator per token.
// pos (nullable): each expert's position in a staged row, SelLayout::at(0, e), in shared memory.
template <int KP, int G>
__device__ void select_tokens(float* sx, float* zsq, float* gsc, int rows, int64_t t0, int E, int k, int score_fn,
                              int renorm, int n_group, int topk_group, const float* __restrict__ sel_bias,
                              int32_t* __restrict__ idx, float* __restrict__ gate, const int* pos = nullptr) {
  const SelLayout L(E, G);
  const int r = threadIdx.x / G, g = threadIdx.x % G;
  const bool tok = r < rows;
  const int e0 = g * L.C;
  const int e1 = min(E, e0 + L.C);
  float* rowp = sx + r * L.LD;
  float* chunk = rowp + g * L.CS;
  const bool softmax = score_fn == MOE_SCORE_SOFTMAX;
  float mx = -INFINITY;
  if (tok)
    for (int e = e0; e < e1; ++e) mx = fmaxf(mx, chunk[e - e0]);
#pragma unroll
  for (int o = 1; o < G; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum_exp = 0.f, denom = 0.f;
  if (tok) {
    for (int e = e0; e < e1; ++e) {
      const float x = chunk[e - e0];
      const float ex = __expf(x - mx);
      sum_exp += ex;
      denom += softmax ? ex : sigmoid_f32(x);
    }
  }
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    sum_exp += __shfl_xor_sync(0xffffffffu, sum_exp, o);
    denom += __shfl_xor_sync(0xffffffffu, denom, o);
  }
  uint32_t keep = 0xffffffffu;
  int gsz = E;  // experts per group
  if (n_group > 1) {
    gsz = E / n_group;
    const int r_top = k / topk_group;
    float* gs = gsc + r * n_group;
    if (tok) {
      for (int q = g; q < n_group; q += G) {
        float best[KP];
#pragma unroll
        for (int j = 0; j < KP; ++j) best[j] = -INFINITY;
        for (int e = q * gsz; e < (q + 1) * gsz; ++e) {
          const float x = sx[pos ? r * L.LD + pos[e] : L.at(r, e)];
          float a = softmax ? __expf(x - mx) / denom : sigmoid_f32(x);
          if (sel_bias) a += sel_bias[e];
#pragma unroll
          for (int j = 0; j < KP; ++j) {
            if (j < r_top && a > best[j]) {
              const float t = best[j];
              best[j] = a;
              a = t;
            }
          }
        }
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < KP; ++j)
          if (j < r_top) sum += best[j];
        gs[q] = sum;
      }
    }
    __syncwarp();
    keep = 0;
    if (tok) {
      for (int q = 0; q < n_group; ++q) {
        const float v = gs[q];
        int rank = 0;
        for (int q2 = 0; q2 < n_group; ++q2) rank += (gs[q2] > v || (gs[q2] == v && q2 < q)) ? 1 : 0;
        if (rank < topk_group) keep |= 1u << q;
      }
    }
  }
  float tv[KP];
  int ti[KP];
#pragma unroll
  for (int j = 0; j < KP; ++j) {
    tv[j] = -INFINITY;
    ti[j] = 0x7fffffff;
  }
  if (tok) {
    int grp = e0 / gsz, grp_end = (grp + 1) * gsz;  // the group of expert e, tracked as e advances
    for (int e = e0; e < e1; ++e) {
      if (e == grp_end) {
        ++grp;
        grp_end += gsz;
      }
      if (!((keep >> grp) & 1u)) continue;  // outside the kept groups (never without groups: grp = 0)
      const float x = chunk[e - e0];
      const float key = sel_bias ? (softmax ? __expf(x - mx) / denom : sigmoid_f32(x)) + sel_bias[e] : x;
      if (before(key, e, tv[KP - 1], ti[KP - 1])) insert_sorted<KP>(tv, ti, key, e);
    }
  }
  // combine the G lanes' lists (consecutive lanes of one warp)
#pragma unroll
  for (int o = 1; o < G; o <<= 1) {
    float bv[KP];
    int bi[KP];
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      bv[j] = __shfl_xor_sync(0xffffffffu, tv[KP - 1 - j], o);  // the partner's list, reversed
      bi[j] = __shfl_xor_sync(0xffffffffu, ti[KP - 1 - j], o);
    }
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      if (before(bv[j], bi[j], tv[j], ti[j])) {
        tv[j] = bv[j];
        ti[j] = bi[j];
      }
    }
#pragma unroll
    for (int st = KP / 2; st > 0; st >>= 1) {
#pragma unroll
      for (int j = 0; j < KP; ++j) {
        if ((j & st) == 0 && before(tv[j + st], ti[j + st], tv[j], ti[j])) {
          const float tvj = tv[j];
          const int tij = ti[j];
          tv[j] = tv[j + st];
          ti[j] = ti[j + st];
          tv[j + st] = tvj;
          ti[j + st] = tij;
        }
      }
    }
  }
  if (tok) {
    // gates from the scores of the selected experts (their logits are in the staged row)
    float sel_s[KP], sel_sum = 0.f;
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      sel_s[j] = 0.f;
      if (j < k) {
        const float x = sx[pos ? r * L.LD + pos[ti[j]] : L.at(r, ti[j])];
        sel_s[j] = softmax ? __expf(x - mx) / denom : sigmoid_f32(x);
        sel_sum += sel_s[j];
      }
    }
    const int64_t t = t0 + r;
#pragma unroll
    for (int j = 0; j < KP; ++j) {
      if (j < k && j % G == g) {
        idx[t * k + j] = ti[j];
        gate[t * k + j] = renorm ? sel_s[j] / sel_sum : sel_s[j];
      }
    }
  }
  // every lane has read what it needs from the row before any lane overwrites its chunk
  __syncwarp();
  if (tok) {
    const float inv = 1.f / denom;
    for (int e = e0; e < e1; ++e) {
      const float x = chunk[e - e0];
      chunk[e - e0] = (softmax ? __expf(x - mx) : sigmoid_f32(x)) * inv;
    }
    if (g == 0) {
      const float lse = mx + logf(sum_exp);
      zsq[r] = lse * lse;
    }
  }
}

// Step 3: out[e] = the sum over the tile's rows, in order, of the normalised scores of expert e
// (e < E), and out[E] = the sum of the rows' LSE^2; added to out when `accumulate`.  The caller
// synchronises the block between select_tokens and this.
__device__ __forceinline__ void score_column_sums(const float* sx, const float* zsq, int rows, int E, int G,
                                                  float* out, bool accumulate) {
  const SelLayout L(E, G);
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    float acc = 0.f;
    if (e < E) {
      const float* col = sx + L.at(0, e);
      for (int i = 0; i < rows; ++i) acc += col[i * L.LD];
    } else {
      for (int i = 0; i < rows; ++i) acc += zsq[i];
    }
    out[e] = accumulate ? out[e] + acc : acc;
  }
}

// score_column_sums with the rows split among all threads: row group q of NG = blockDim.x / (E + 1)
// groups (at least one) adds rows [q rows / NG, (q+1) rows / NG) of column e into part[q (E + 1) + e];
// then thread e adds the NG group sums in order.  The block synchronises inside; `part` holds
// blockDim.x floats.
__device__ __forceinline__ void score_column_sums_split(const float* sx, const float* zsq, int rows, int E, int G,
                                                        float* out, float* part, bool accumulate) {
  const SelLayout L(E, G);
  const int W = E + 1;
  const int NG = max(1, static_cast<int>(blockDim.x) / W);
  for (int t = threadIdx.x; t < NG * W; t += blockDim.x) {
    const int q = t / W, e = t - q * W;
    const int i0 = (rows * q) / NG, i1 = (rows * (q + 1)) / NG;
    float acc = 0.f;
    if (e < E) {
      const float* col = sx + L.at(0, e);
      for (int i = i0; i < i1; ++i) acc += col[i * L.LD];
    } else {
      for (int i = i0; i < i1; ++i) acc += zsq[i];
    }
    part[t] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < W; e += blockDim.x) {
    float acc = 0.f;
    for (int q = 0; q < NG; ++q) acc += part[q * W + e];
    out[e] = accumulate ? out[e] + acc : acc;
  }
}

}  // namespace moe
