// Plain CPU oracle of the single-GPU MoE layer: forward, statistics and backward.
//
// TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU legs load this
// library (through oracle/moe_oracle.py); the MoE library never does, and the two share no code.
// Every function is the method's definition written out with plain loops, in the order and
// notation of the pages, accumulating in double.  Loops over independent rows (tokens, weight
// rows, expert rows) run in parallel with OpenMP; every output element is computed by one thread
// in a fixed order, so results do not depend on the thread count.  Sorting is done with the
// standard library.
//
// Sources (page title, section):
//   [FFN] "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), 从稠密 FFN 到 MoE:
//         FFN(u) = W_down (SiLU(W_gate u) * W_up u); h'_t = u_t + sum_i g_{i,t} FFN_i(u_t).
//   [RTR] same page, 路由器：打分、top-k、加权求和: H = U W_r; scores; top-k; gates; the noisy
//         top-k logits (x W_g)_i + N(0,1) Softplus((x W_noise)_i); the shapes listing (permute
//         by expert, grouped FFN, index_add back); how the router learns (the gate gradient).
//   [SCR] same page, softmax 门控还是 sigmoid 门控: softmax or sigmoid scores, gates with or
//         without renormalisation over the selected experts.
//   [CAP] same page, 专家容量与丢 token: C = ceil(CF * T * k / E); slots filled in token order,
//         every token's first choice before any second choice; overflow dropped (residual only).
//   [AUX] same page, 负载均衡辅助损失：推导与梯度: f_i, P_i = (1/T) sum_t s_{i,t}, E sum f_i P_i;
//         sigmoid scores enter P through s' = s / sum_j s_j; the gradient with f held constant.
//   [ZL]  same page, Router z-loss 与数值稳定: L_z = (1/T) sum_t LSE(H_t)^2 and its gradient.
//   [SHR] same page, 细粒度专家与共享专家: shared experts take every token with weight 1.
//   [LFB] same page, 无辅助损失的负载均衡: select on s + b, gate from s; b += u sign(mean c - c);
//         MaxVio = (max load - mean load) / mean load.
//   [GRP] same page, 设备受限与节点受限路由: groups ranked by the sum of their best affinities.
//   [FP8] same page, 低精度通信: FP8 activations into the up-projection, power-of-two scales.
//   [BWD] same page, 专家计算：padding、block-sparse 与 grouped GEMM: the experts' backward.
//
// Readings where the pages are silent (the same readings the library follows): selection on the
// float32 logits, ties to the lower expert id; no capacity limit means C = T; f counts the
// router's assignments before drops, over T*k; a dropped pair adds nothing and the kept gates
// are not renormalised; rows of an expert segment in slot order; groups are contiguous blocks of
// E/n_group experts scored on their k/topk_group best affinities (s, or s + b with a selection
// bias), ties to the lower group id; FP8 is E4M3 (largest 448, round to nearest even) with one
// power-of-two scale per token row and per gate/up weight row.
//
// Arrays are row-major.  Inputs that may come in the layer's own precision are passed as a
// pointer plus a type code (0 float64, 1 float32, 2 bfloat16) and widened exactly to double on
// read.  Index arrays are int64.  Nothing here allocates memory that outlives a call.
#include <omp.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <limits>
#include <vector>

#define ORC_API extern "C" __attribute__((visibility("default")))

namespace {

enum { DT_F64 = 0, DT_F32 = 1, DT_BF16 = 2 };
enum { SOFTMAX = 0, SIGMOID = 1 };
enum { CHOICE_MAJOR = 0, TOKEN_MAJOR = 1 };

const double INF = std::numeric_limits<double>::infinity();

// Element i of an array in float64, float32 or bfloat16 (a bfloat16 is the high half of a
// float32), as a double: exact.
inline double elem(const void* p, int dt, int64_t i) {
  if (dt == DT_F64) return static_cast<const double*>(p)[i];
  if (dt == DT_F32) return static_cast<const float*>(p)[i];
  const uint32_t bits = static_cast<uint32_t>(static_cast<const uint16_t*>(p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return f;
}

void widen(const void* p, int dt, int64_t first, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = elem(p, dt, first + i);
}

double dot(const double* a, const double* b, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }

// SiLU(x) = x sigmoid(x), written x / (1 + e^-x).
double silu(double x) { return x / (1.0 + std::exp(-x)); }

// Softplus(x) = ln(1 + e^x) in the form that cannot overflow: max(x, 0) + ln(1 + e^-|x|).
double softplus(double x) { return std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x))); }

// ---------------------------------------------------------------- router [RTR], [SCR]

// Scores of one token's logits: softmax over the E experts (max-shifted), or a sigmoid each.
void score_row(const double* H, int E, int fn, double* s) {
  if (fn == SOFTMAX) {
    double m = -INF;
    for (int e = 0; e < E; ++e) m = std::max(m, H[e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += std::exp(H[e] - m);
    for (int e = 0; e < E; ++e) s[e] = std::exp(H[e] - m) / z;
  } else {
    for (int e = 0; e < E; ++e) s[e] = sigmoid(H[e]);
  }
}

// Is expert a ranked before expert b?  Allowed experts first (group-limited routing), then the
// larger key, then the lower expert id.
bool ranks_before(const double* key, const uint8_t* allowed, int a, int b) {
  if (allowed && allowed[a] != allowed[b]) return allowed[a] > allowed[b];
  if (key[a] != key[b]) return key[a] > key[b];
  return a < b;
}

// The k best experts of one token, best first: k rounds, each taking the best expert not yet taken.
void topk_row(const double* key, const uint8_t* allowed, int E, int k, int64_t* idx) {
  std::vector<uint8_t> taken(E, 0);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e)
      if (!taken[e] && (best < 0 || ranks_before(key, allowed, e, best))) best = e;
    taken[best] = 1;
    idx[j] = best;
  }
}

// Sum of the r largest of n values.
double sum_of_largest(const double* v, int n, int r) {
  std::vector<double> c(v, v + n);
  std::sort(c.begin(), c.end(), [](double a, double b) { return a > b; });
  double s = 0.0;
  for (int i = 0; i < r && i < n; ++i) s += c[i];
  return s;
}

// [GRP]: group q holds experts [q S, (q+1) S), S = E / n_group; its score is the sum of its r best
// affinities; the topk_group best groups are kept (ties to the lower group id).
void group_mask_row(const double* aff, int E, int n_group, int topk_group, int k, uint8_t* allowed) {
  const int S = E / n_group, r = k / topk_group;
  std::vector<double> gs(n_group);
  for (int q = 0; q < n_group; ++q) gs[q] = sum_of_largest(aff + q * S, S, r);
  std::vector<uint8_t> keep(n_group, 0);
  for (int round = 0; round < topk_group; ++round) {
    int best = -1;
    for (int q = 0; q < n_group; ++q)
      if (!keep[q] && (best < 0 || gs[q] > gs[best])) best = q;
    keep[best] = 1;
  }
  for (int e = 0; e < E; ++e) allowed[e] = keep[e / S];
}

// ---------------------------------------------------------------- experts [FFN], [FP8]

// E4M3 nearest value, ties to even, saturating at +-448.  E4M3 has 3 mantissa bits: in the binade
// [2^e, 2^(e+1)), e >= -6, neighbours are 2^(e-3) apart; below 2^-6 (subnormals) 2^-9 apart.
double e4m3_round(double x) {
  const double a = std::fabs(x);
  double quantum = std::ldexp(1.0, -9);
  if (a >= std::ldexp(1.0, -6)) {
    int E2;
    std::frexp(a, &E2);                       // a = m 2^E2, m in [0.5, 1): binade e = E2 - 1
    quantum = std::ldexp(1.0, (E2 - 1) - 3);
  }
  const double r = std::min(std::nearbyint(a / quantum) * quantum, 448.0);  // nearbyint: to even
  return std::copysign(r, x);
}

// The smallest integer s >= -127 with amax <= 448 * 2^s (-127 when amax = 0).
int64_t pow2_scale_exponent(double amax) {
  if (!(amax > 0.0)) return -127;
  int64_t s = static_cast<int64_t>(std::floor(std::log2(amax / 448.0)));  // a guess, then exact
  while (amax > 448.0 * std::ldexp(1.0, static_cast<int>(s))) ++s;
  while (s > -127 && amax <= 448.0 * std::ldexp(1.0, static_cast<int>(s - 1))) --s;
  return std::max<int64_t>(s, -127);
}

// One row quantised to E4M3 with one power-of-two scale and dequantised again, in place.
void fp8_roundtrip_row(double* row, int64_t n) {
  double amax = 0.0;
  for (int64_t i = 0; i < n; ++i) amax = std::max(amax, std::fabs(row[i]));
  const int s = static_cast<int>(pow2_scale_exponent(amax));
  for (int64_t i = 0; i < n; ++i) row[i] = std::ldexp(e4m3_round(std::ldexp(row[i], -s)), s);
}

// One expert on n rows x [n, h]: a = SiLU(x W_gate^T) * (x W_up^T) [n, d], y = a W_down^T [n, h].
// W_gate, W_up are [d, h] and W_down [h, d] at element offsets wg_off, wu_off, wd_off of their
// arrays.  fp8_w: each W_gate and W_up row is quantised to E4M3 (its own power-of-two scale) and
// dequantised before use ([FP8]).
void expert_rows(int64_t n, int h, int d, const double* x, const void* Wg, int wg_dt, int64_t wg_off, const void* Wu,
                 int wu_dt, int64_t wu_off, const void* Wd, int wd_dt, int64_t wd_off, int fp8_w, double* y,
                 double* a) {
  if (n <= 0) return;
#pragma omp parallel
  {
    std::vector<double> wg(h), wu(h);
#pragma omp for schedule(static)
    for (int j = 0; j < d; ++j) {
      widen(Wg, wg_dt, wg_off + static_cast<int64_t>(j) * h, h, wg.data());
      widen(Wu, wu_dt, wu_off + static_cast<int64_t>(j) * h, h, wu.data());
      if (fp8_w) {
        fp8_roundtrip_row(wg.data(), h);
        fp8_roundtrip_row(wu.data(), h);
      }
      for (int64_t r = 0; r < n; ++r) {
        const double G = dot(x + r * h, wg.data(), h);
        const double Up = dot(x + r * h, wu.data(), h);
        a[r * d + j] = silu(G) * Up;
      }
    }
    std::vector<double> wd(d);
#pragma omp for schedule(static)
    for (int m = 0; m < h; ++m) {
      widen(Wd, wd_dt, wd_off + static_cast<int64_t>(m) * d, d, wd.data());
      for (int64_t r = 0; r < n; ++r) y[r * h + m] = dot(a + r * d, wd.data(), d);
    }
  }
}

double now_s() {
  return std::chrono::duration<double>(std::chrono::steady_clock::now().time_since_epoch()).count();
}

}  // namespace

// ================================================================ exported stages

ORC_API int orc_threads(void) { return omp_get_max_threads(); }
ORC_API void orc_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }

ORC_API void orc_softplus(int64_t n, const double* x, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = softplus(x[i]);
}

ORC_API void orc_round_f32(int64_t n, const double* x, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = static_cast<double>(static_cast<float>(x[i]));
}

// [RTR] H = U W_r (+ b_r) (+ eps * Softplus(U W_noise)); U [T, h], W_r and W_noise [h, E] (column i
// = expert i), b_r [E], eps [T, E] standard-normal draws.  W_noise == NULL: no noise.
ORC_API void orc_router_logits(int64_t T, int h, int E, const void* U, int u_dt, const void* W_r, int wr_dt,
                               const void* b_r, int b_dt, const void* W_noise, int wn_dt, const void* eps,
                               int eps_dt, double* H) {
  std::vector<double> wr(static_cast<size_t>(h) * E), wn;
  widen(W_r, wr_dt, 0, static_cast<int64_t>(h) * E, wr.data());
  if (W_noise) {
    wn.resize(static_cast<size_t>(h) * E);
    widen(W_noise, wn_dt, 0, static_cast<int64_t>(h) * E, wn.data());
  }
#pragma omp parallel
  {
    std::vector<double> u(h);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      widen(U, u_dt, t * h, h, u.data());
      for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int c = 0; c < h; ++c) acc += u[c] * wr[static_cast<size_t>(c) * E + e];
        if (b_r) acc += elem(b_r, b_dt, e);
        if (W_noise) {
          double z = 0.0;
          for (int c = 0; c < h; ++c) z += u[c] * wn[static_cast<size_t>(c) * E + e];
          acc += elem(eps, eps_dt, t * E + e) * softplus(z);
        }
        H[t * E + e] = acc;
      }
    }
  }
}

// [RTR], [SCR] scores s [T, E] of logits H [T, E].
ORC_API void orc_scores(int64_t T, int E, const double* H, int fn, double* s) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) score_row(H + t * E, E, fn, s + t * E);
}

// [RTR] top-k ids [T, k] by key [T, E], best first, ties to the lower id; allowed [T, E] (NULL: all)
// ranks every allowed expert ahead of every other one.
ORC_API void orc_topk(int64_t T, int E, const double* key, int k, const uint8_t* allowed, int64_t* idx) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) topk_row(key + t * E, allowed ? allowed + t * E : nullptr, E, k, idx + t * k);
}

// [GRP] group scores [T, n_group]: each group's sum of its r largest affinities.
ORC_API void orc_group_scores(int64_t T, int E, const double* aff, int n_group, int r, double* out) {
  const int S = E / n_group;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int q = 0; q < n_group; ++q) out[t * n_group + q] = sum_of_largest(aff + t * E + q * S, S, r);
}

// [GRP] allowed [T, E]: the experts of each token's topk_group best groups.
ORC_API void orc_group_limited_mask(int64_t T, int E, const double* aff, int n_group, int topk_group, int k,
                                    uint8_t* allowed) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) group_mask_row(aff + t * E, E, n_group, topk_group, k, allowed + t * E);
}

// [SCR] gates [T, k]: g_j = s_{i_j} / sum_{j'} s_{i_j'} (renorm) or s_{i_j}.
ORC_API void orc_gates(int64_t T, int E, int k, const double* s, const int64_t* idx, int renorm, double* gate) {
  for (int64_t t = 0; t < T; ++t) {
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += s[t * E + idx[t * k + j]];
    for (int j = 0; j < k; ++j) {
      const double v = s[t * E + idx[t * k + j]];
      gate[t * k + j] = renorm ? v / sum : v;
    }
  }
}

// [RTR], [SCR], [LFB], [GRP] routing from logits H [T, E]: the logits are rounded to float32
// (logits32), scored (s); the selection key is the logit, or s + sel_bias with a loss-free
// selection bias (sel_key); with n_group > 1 the top-k is limited to the experts of the
// topk_group best groups, scored on s (s + b with a bias) (allowed, may be NULL otherwise); idx and
// the gates from s.
ORC_API void orc_route(int64_t T, int E, const double* H, int k, int fn, int renorm, const double* sel_bias,
                       int n_group, int topk_group, double* logits32, double* s, double* sel_key, uint8_t* allowed,
                       int64_t* idx, double* gate) {
  orc_round_f32(T * E, H, logits32);
  orc_scores(T, E, logits32, fn, s);
  for (int64_t t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) sel_key[t * E + e] = sel_bias ? s[t * E + e] + sel_bias[e] : logits32[t * E + e];
  const uint8_t* mask = nullptr;
  if (n_group > 1) {
    orc_group_limited_mask(T, E, sel_bias ? sel_key : s, n_group, topk_group, k, allowed);
    mask = allowed;
  }
  orc_topk(T, E, sel_key, k, mask, idx);
  orc_gates(T, E, k, s, idx, renorm, gate);
}

// [CAP] C = ceil(CF * T * k / E), exact on the float32 value of CF; CF <= 0: C = T; override > 0
// wins.  CF * T * k is exact in long double (24 + 31 bits); the quotient's ceiling is corrected
// with exact products.
ORC_API int64_t orc_capacity(int64_t T, int E, int k, float cf, int64_t override_c) {
  if (override_c > 0) return override_c;
  if (!(cf > 0.0f)) return T;
  const long double num = static_cast<long double>(cf) * static_cast<long double>(T * k);
  long double q = std::ceil(num / E);
  while (q > 0 && (q - 1) * E >= num) q -= 1;
  while (q * E < num) q += 1;
  return static_cast<int64_t>(q);
}

// [CAP] + the permute of [RTR]'s shapes listing.  The (token, choice) pairs are walked in priority
// order (choice-major: every token's first choice, in token order, before any second choice;
// token-major: a token's choices together); the n-th pair that chose expert e gets slot n of e and
// is kept iff n < C.  Kept rows are packed expert by expert in slot order: offsets = exclusive
// prefix sum of the kept counts, row = offsets[e] + slot, row_token[row] = its token.
// Returns the number of dropped pairs.
ORC_API int64_t orc_dispatch(int64_t T, int k, int E, const int64_t* idx, int64_t C, int priority,
                             int64_t* counts_routed, int64_t* counts_kept, int64_t* offsets, int64_t* slot,
                             int64_t* slot_row, int64_t* row_token) {
  for (int e = 0; e < E; ++e) counts_routed[e] = 0;
  for (int64_t p = 0; p < T * k; ++p) {
    int64_t t;
    int j;
    if (priority == CHOICE_MAJOR) {
      j = static_cast<int>(p / T);
      t = p - static_cast<int64_t>(j) * T;
    } else {
      t = p / k;
      j = static_cast<int>(p - t * k);
    }
    const int64_t e = idx[t * k + j];
    slot[t * k + j] = counts_routed[e]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    counts_kept[e] = std::min(counts_routed[e], C);
    offsets[e + 1] = offsets[e] + counts_kept[e];
  }
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int64_t pair = t * k + j, e = idx[pair];
      if (slot[pair] < C) {
        slot_row[pair] = offsets[e] + slot[pair];
        row_token[slot_row[pair]] = t;
      } else {
        slot_row[pair] = -1;
      }
    }
  return T * k - offsets[E];
}

// [RTR] shapes listing: X[r] = U[row_token[r]].
ORC_API void orc_permute(int64_t A, int h, const void* U, int u_dt, const int64_t* row_token, double* X) {
  for (int64_t r = 0; r < A; ++r) widen(U, u_dt, row_token[r] * h, h, X + r * h);
}

// [FFN] one expert on rows x [n, h] (see expert_rows); fp8_x quantises each x row to E4M3 with its
// own power-of-two scale first, fp8_w each W_gate / W_up row ([FP8]).
ORC_API void orc_expert_rows(int64_t n, int h, int d, const double* x, const void* Wg, int wg_dt, int64_t wg_off,
                             const void* Wu, int wu_dt, int64_t wu_off, const void* Wd, int wd_dt, int64_t wd_off,
                             int fp8_x, int fp8_w, double* y, double* a) {
  if (!fp8_x) {
    expert_rows(n, h, d, x, Wg, wg_dt, wg_off, Wu, wu_dt, wu_off, Wd, wd_dt, wd_off, fp8_w, y, a);
    return;
  }
  std::vector<double> xq(x, x + n * h);
  for (int64_t r = 0; r < n; ++r) fp8_roundtrip_row(xq.data() + r * h, h);
  expert_rows(n, h, d, xq.data(), Wg, wg_dt, wg_off, Wu, wu_dt, wu_off, Wd, wd_dt, wd_off, fp8_w, y, a);
}

// [RTR] shapes listing (grouped FFN) with [FFN]'s expert: Y, act over the expert segments
// rows offsets[e] .. offsets[e+1] of X [A, h]; W_gate, W_up [E, d, h], W_down [E, h, d].
ORC_API void orc_expert_ffn(int64_t A, int h, int d, int E, const double* X, const int64_t* offsets, const void* Wg,
                            int wg_dt, const void* Wu, int wu_dt, const void* Wd, int wd_dt, int fp8_w, double* Y,
                            double* act) {
  for (int64_t i = 0; i < A * h; ++i) Y[i] = 0.0;
  for (int64_t i = 0; i < A * d; ++i) act[i] = 0.0;
  const int64_t hd = static_cast<int64_t>(h) * d;
  for (int e = 0; e < E; ++e) {
    const int64_t lo = offsets[e], hi = offsets[e + 1];
    if (hi > lo)
      expert_rows(hi - lo, h, d, X + lo * h, Wg, wg_dt, e * hd, Wu, wu_dt, e * hd, Wd, wd_dt, e * hd, fp8_w, Y + lo * h,
                  act + lo * d);
  }
}

// [FP8] E4M3 rounding of n values.
ORC_API void orc_e4m3_round(int64_t n, const double* x, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round(x[i]);
}

// [FP8] the 8-bit codes (sign << 7 | exponent field << 3 | mantissa) of E4M3 values.
ORC_API void orc_e4m3_bits(int64_t n, const double* v, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    const double a = std::fabs(v[i]);
    int field = 0, mant;
    if (a >= std::ldexp(1.0, -6)) {
      int E2;
      std::frexp(a, &E2);
      const int e = E2 - 1;
      field = e + 7;
      mant = static_cast<int>((std::ldexp(a, -e) - 1.0) * 8.0);
    } else {
      mant = static_cast<int>(a * 512.0);
    }
    out[i] = static_cast<uint8_t>((std::signbit(v[i]) ? 0x80 : 0) | (field << 3) | mant);
  }
}

// [FP8] per amax, the smallest s >= -127 with amax <= 448 2^s.
ORC_API void orc_pow2_scale_exponents(int64_t n, const double* amax, int64_t* s) {
  for (int64_t i = 0; i < n; ++i) s[i] = pow2_scale_exponent(amax[i]);
}

// [FP8] rows [n, c] -> E4M3 codes (as values) and one power-of-two exponent per row.
ORC_API void orc_quantize_rows_fp8(int64_t n, int64_t c, const void* A, int a_dt, double* codes, int64_t* s) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    double amax = 0.0;
    for (int64_t i = 0; i < c; ++i) amax = std::max(amax, std::fabs(elem(A, a_dt, r * c + i)));
    s[r] = pow2_scale_exponent(amax);
    for (int64_t i = 0; i < c; ++i)
      codes[r * c + i] = e4m3_round(std::ldexp(elem(A, a_dt, r * c + i), static_cast<int>(-s[r])));
  }
}

ORC_API void orc_dequantize_rows_fp8(int64_t n, int64_t c, const double* codes, const int64_t* s, double* out) {
  for (int64_t r = 0; r < n; ++r)
    for (int64_t i = 0; i < c; ++i) out[r * c + i] = std::ldexp(codes[r * c + i], static_cast<int>(s[r]));
}

// [SHR] Y_sh [n_s, T, h]: each shared expert's FFN on every token row of U [T, h].
ORC_API void orc_shared_ffn(int n_s, int64_t T, int h, int d, const void* U, int u_dt, const void* Wg, int wg_dt,
                            const void* Wu, int wu_dt, const void* Wd, int wd_dt, double* Y_sh) {
  std::vector<double> u(static_cast<size_t>(T) * h), a(static_cast<size_t>(T) * d);
  widen(U, u_dt, 0, T * h, u.data());
  const int64_t hd = static_cast<int64_t>(h) * d;
  for (int i = 0; i < n_s; ++i)
    expert_rows(T, h, d, u.data(), Wg, wg_dt, i * hd, Wu, wu_dt, i * hd, Wd, wd_dt, i * hd, 0, Y_sh + i * T * h,
                a.data());
}

// [FFN] layer output with [RTR]'s index_add: out_t = u_t + sum_s Y_sh[s, t] + sum_j g_{t,j} Y[row(t, j)]
// over the kept pairs, j ascending; a dropped pair adds nothing ([CAP]).  Y_sh may be NULL.
ORC_API void orc_combine(int64_t T, int h, int k, const void* U, int u_dt, const double* Y, const int64_t* slot_row,
                         const double* gate, int n_s, const double* Y_sh, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double* o = out + t * h;
    widen(U, u_dt, t * h, h, o);
    for (int s = 0; s < n_s; ++s)
      for (int c = 0; c < h; ++c) o[c] += Y_sh[(s * T + t) * h + c];
    for (int j = 0; j < k; ++j) {
      const int64_t row = slot_row[t * k + j];
      if (row < 0) continue;
      for (int c = 0; c < h; ++c) o[c] += gate[t * k + j] * Y[row * h + c];
    }
  }
}

// [AUX], [LFB] f_i = counts_i / (T k); P_i = (1/T) sum_t s'_{i,t} (s' = s / sum_j s_j for sigmoid
// scores, s for softmax); aux = E sum_i f_i P_i; MaxVio = (max c - mean c) / mean c.
// out: [aux, maxvio].
ORC_API void orc_load_stats(int E, int64_t T, double k, const double* counts, const double* s, int fn, double* f,
                            double* P, double* out) {
  for (int e = 0; e < E; ++e) {
    f[e] = counts[e] / (static_cast<double>(T) * k);
    P[e] = 0.0;
  }
  for (int64_t t = 0; t < T; ++t) {
    double S = 1.0;
    if (fn == SIGMOID) {
      S = 0.0;
      for (int e = 0; e < E; ++e) S += s[t * E + e];
    }
    for (int e = 0; e < E; ++e) P[e] += s[t * E + e] / S;
  }
  double aux = 0.0, cmax = -INF, csum = 0.0;
  for (int e = 0; e < E; ++e) {
    P[e] /= static_cast<double>(T);
    aux += f[e] * P[e];
    cmax = std::max(cmax, counts[e]);
    csum += counts[e];
  }
  const double mean = csum / E;
  out[0] = E * aux;
  out[1] = mean > 0 ? (cmax - mean) / mean : 0.0;
}

// [ZL] L_z = (1/T) sum_t (m_t + ln sum_j e^{H_tj - m_t})^2, m_t = max_j H_tj; 0 when T = 0.
ORC_API double orc_z_loss(int64_t T, int E, const double* H) {
  if (T == 0) return 0.0;
  double sum = 0.0;
  for (int64_t t = 0; t < T; ++t) {
    double m = -INF;
    for (int e = 0; e < E; ++e) m = std::max(m, H[t * E + e]);
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += std::exp(H[t * E + e] - m);
    const double lse = m + std::log(z);
    sum += lse * lse;
  }
  return sum / T;
}

// [LFB] e_i = mean(c) - c_i; b_i <- b_i + u sign(e_i).
ORC_API void orc_balance_bias_update(int E, const double* b, const double* counts, double u, double* out) {
  double mean = 0.0;
  for (int e = 0; e < E; ++e) mean += counts[e];
  mean /= E;
  for (int e = 0; e < E; ++e) {
    const double err = mean - counts[e];
    out[e] = b[e] + u * ((err > 0) - (err < 0));
  }
}

// Per token, the smallest gap between adjacent values among its k+1 largest keys (inf with fewer
// than two): used by the tests to keep routing decisions away from ties.
ORC_API void orc_topk_margins(int64_t T, int E, const double* key, int k, double* out) {
  for (int64_t t = 0; t < T; ++t) {
    std::vector<double> v(key + t * E, key + (t + 1) * E);
    std::sort(v.begin(), v.end(), [](double a, double b) { return a > b; });
    const int n = std::min(E, k + 1);
    double m = INF;
    for (int i = 0; i + 1 < n; ++i) m = std::min(m, v[i] - v[i + 1]);
    out[t] = m;
  }
}

// Per token, the gap between the topk_group-th and the next group score (inf when every group is kept).
ORC_API void orc_group_margins(int64_t T, int E, const double* aff, int n_group, int topk_group, int k, double* out) {
  const int S = E / n_group, r = k / topk_group;
  for (int64_t t = 0; t < T; ++t) {
    if (topk_group >= n_group) {
      out[t] = INF;
      continue;
    }
    std::vector<double> gs(n_group);
    for (int q = 0; q < n_group; ++q) gs[q] = sum_of_largest(aff + t * E + q * S, S, r);
    std::sort(gs.begin(), gs.end(), [](double a, double b) { return a > b; });
    out[t] = gs[topk_group - 1] - gs[topk_group];
  }
}

// ================================================================ the whole forward

// The layer forward, stage by stage ([RTR] .. [AUX]), timing each stage with a steady clock.
//   H_in [T, E] (NULL: the logits come from U W_r (+ b_r) (+ noise)); sel_bias [E] or NULL;
//   n_s shared experts of size d_s (0: none); fp8: E4M3 token rows and gate/up weight rows.
// Outputs (caller-sized): logits32, s, sel_key [T, E]; allowed [T, E] (n_group > 1);
//   idx [T, k]; gate [T, k]; counts_routed, counts_kept [E]; offsets [E+1]; slot, slot_row [T k];
//   row_token, X [T k, h], act [T k, d], Y [T k, h] (rows 0 .. A-1 valid); Y_sh [n_s, T, h];
//   out [T, h]; f, P [E]; U_codes [T, h], U_s [T] (fp8); scal = [C, n_dropped, aux, maxvio, z_loss];
//   seconds = [router logits, selection, dispatch, experts, shared experts, combine, statistics].
ORC_API void orc_layer_forward(
    int64_t T, int h, int E, int k, int d, int fn, int renorm, float cf, int64_t cap_override, int priority,
    const void* U, int u_dt, const void* W_r, int wr_dt, const void* b_r, int b_dt, const void* W_noise, int wn_dt,
    const void* eps, int eps_dt, const double* H_in, const void* Wg, int wg_dt, const void* Wu, int wu_dt,
    const void* Wd, int wd_dt, const double* sel_bias, int n_group, int topk_group, int n_s, int d_s,
    const void* Wg_sh, int wgs_dt, const void* Wu_sh, int wus_dt, const void* Wd_sh, int wds_dt, int fp8,
    double* logits32, double* s, double* sel_key, uint8_t* allowed, int64_t* idx, double* gate,
    int64_t* counts_routed, int64_t* counts_kept, int64_t* offsets, int64_t* slot, int64_t* slot_row,
    int64_t* row_token, double* X, double* act, double* Y, double* Y_sh, double* out, double* f, double* P,
    double* U_codes, int64_t* U_s, double* scal, double* seconds) {
  double t0 = now_s();
  std::vector<double> H;
  if (!H_in) {
    H.resize(static_cast<size_t>(T) * E);
    orc_router_logits(T, h, E, U, u_dt, W_r, wr_dt, b_r, b_dt, W_noise, wn_dt, eps, eps_dt, H.data());
    H_in = H.data();
  }
  double t1 = now_s();
  seconds[0] = t1 - t0;
  orc_route(T, E, H_in, k, fn, renorm, sel_bias, n_group, topk_group, logits32, s, sel_key, allowed, idx, gate);
  t0 = now_s();
  seconds[1] = t0 - t1;
  const int64_t C = orc_capacity(T, E, k, cf, cap_override);
  const int64_t dropped =
      orc_dispatch(T, k, E, idx, C, priority, counts_routed, counts_kept, offsets, slot, slot_row, row_token);
  const int64_t A = offsets[E];
  if (fp8) {
    std::vector<double> deq(static_cast<size_t>(T) * h);
    orc_quantize_rows_fp8(T, h, U, u_dt, U_codes, U_s);
    orc_dequantize_rows_fp8(T, h, U_codes, U_s, deq.data());
    orc_permute(A, h, deq.data(), DT_F64, row_token, X);
  } else {
    orc_permute(A, h, U, u_dt, row_token, X);
  }
  t1 = now_s();
  seconds[2] = t1 - t0;
  orc_expert_ffn(A, h, d, E, X, offsets, Wg, wg_dt, Wu, wu_dt, Wd, wd_dt, fp8, Y, act);
  t0 = now_s();
  seconds[3] = t0 - t1;
  if (n_s > 0) orc_shared_ffn(n_s, T, h, d_s, U, u_dt, Wg_sh, wgs_dt, Wu_sh, wus_dt, Wd_sh, wds_dt, Y_sh);
  t1 = now_s();
  seconds[4] = t1 - t0;
  orc_combine(T, h, k, U, u_dt, Y, slot_row, gate, n_s, Y_sh, out);
  t0 = now_s();
  seconds[5] = t0 - t1;
  std::vector<double> counts(E);
  for (int e = 0; e < E; ++e) counts[e] = static_cast<double>(counts_routed[e]);
  double st[2];
  orc_load_stats(E, T, k, counts.data(), s, fn, f, P, st);
  scal[0] = static_cast<double>(C);
  scal[1] = static_cast<double>(dropped);
  scal[2] = st[0];
  scal[3] = st[1];
  scal[4] = orc_z_loss(T, E, logits32);
  seconds[6] = now_s() - t0;
}

// Out rows (and the expert rows they use) for a sample of n tokens of a full-size layer: each kept
// pair's expert row is one expert applied to one token row ([FFN]), given here as y [n, k, h]
// (rows of dropped pairs unused); out = u + sum_s Y_sh[s] + sum_j g_j y_j over the kept pairs.
ORC_API void orc_sampled_combine(int64_t n, int h, int k, const double* u, const double* y, const int64_t* slot_row,
                                 const double* gate, int n_s, const double* Y_sh, double* out) {
  for (int64_t t = 0; t < n; ++t) {
    double* o = out + t * h;
    for (int c = 0; c < h; ++c) o[c] = u[t * h + c];
    for (int s = 0; s < n_s; ++s)
      for (int c = 0; c < h; ++c) o[c] += Y_sh[(s * n + t) * h + c];
    for (int j = 0; j < k; ++j) {
      if (slot_row[t * k + j] < 0) continue;
      for (int c = 0; c < h; ++c) o[c] += gate[t * k + j] * y[(t * k + j) * h + c];
    }
  }
}

// ================================================================ backward [RTR], [AUX], [ZL], [BWD]

// Backward of the combine for dO [T, h]: per kept pair d_gate = dO_t . Y[row] and dY[row] = g dO_t;
// dropped pairs get d_gate = 0.  dY [A, h] is written in full (zero rows for no pair).
ORC_API void orc_combine_backward(int64_t T, int h, int k, int64_t A, const double* dO, const double* Y,
                                  const int64_t* slot_row, const double* gate, double* d_gate, double* dY) {
  for (int64_t i = 0; i < A * h; ++i) dY[i] = 0.0;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      const int64_t row = slot_row[t * k + j];
      if (row < 0) {
        d_gate[t * k + j] = 0.0;
        continue;
      }
      d_gate[t * k + j] = dot(dO + t * h, Y + row * h, h);
      for (int c = 0; c < h; ++c) dY[row * h + c] = gate[t * k + j] * dO[t * h + c];
    }
}

// dL/dH [T, E] from dL/dg [T, k] through the gates (the top-k set held fixed):
// renorm: g_j = s_j / S, dg_j/ds_m = (delta_jm - g_j) / S; then softmax ds_i/dH_m = s_i (delta_im - s_m),
// sigmoid ds_i/dH_i = s_i (1 - s_i).
ORC_API void orc_gate_backward(int64_t T, int E, int k, const double* H, const int64_t* idx, const double* d_gate,
                               int fn, int renorm, double* dH) {
#pragma omp parallel
  {
    std::vector<double> s(E), ds(E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      score_row(H + t * E, E, fn, s.data());
      for (int e = 0; e < E; ++e) ds[e] = 0.0;
      double S = 0.0, wg = 0.0;
      for (int j = 0; j < k; ++j) S += s[idx[t * k + j]];
      for (int j = 0; j < k; ++j) wg += d_gate[t * k + j] * (s[idx[t * k + j]] / S);
      for (int j = 0; j < k; ++j) {
        const int64_t e = idx[t * k + j];
        ds[e] += renorm ? (d_gate[t * k + j] - wg) / S : d_gate[t * k + j];
      }
      if (fn == SOFTMAX) {
        double sd = 0.0;
        for (int e = 0; e < E; ++e) sd += ds[e] * s[e];
        for (int e = 0; e < E; ++e) dH[t * E + e] = s[e] * (ds[e] - sd);
      } else {
        for (int e = 0; e < E; ++e) dH[t * E + e] = ds[e] * s[e] * (1.0 - s[e]);
      }
    }
  }
}

// [AUX] d(E sum_i f_i P_i)/dH with f constant: softmax (E/T) s_k (f_k - sum_i f_i s_i); sigmoid
// (E/T) s'_k (1 - s_k) (f_k - sum_i f_i s'_i), s' = s / sum_j s_j.
ORC_API void orc_aux_loss_grad(int64_t T, int E, const double* H, const double* f, int fn, double* out) {
#pragma omp parallel
  {
    std::vector<double> s(E), sp(E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      score_row(H + t * E, E, fn, s.data());
      double S = 1.0;
      if (fn == SIGMOID) {
        S = 0.0;
        for (int e = 0; e < E; ++e) S += s[e];
      }
      double mean = 0.0;
      for (int e = 0; e < E; ++e) {
        sp[e] = s[e] / S;
        mean += f[e] * sp[e];
      }
      for (int e = 0; e < E; ++e) {
        const double sat = fn == SIGMOID ? 1.0 - s[e] : 1.0;
        out[t * E + e] = static_cast<double>(E) / T * sp[e] * sat * (f[e] - mean);
      }
    }
  }
}

// [ZL] dL_z/dH_{t,k} = (2/T) LSE(H_t) softmax(H_t)_k.
ORC_API void orc_z_loss_grad(int64_t T, int E, const double* H, double* out) {
#pragma omp parallel
  {
    std::vector<double> s(E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      double m = -INF;
      for (int e = 0; e < E; ++e) m = std::max(m, H[t * E + e]);
      double z = 0.0;
      for (int e = 0; e < E; ++e) z += std::exp(H[t * E + e] - m);
      const double lse = m + std::log(z);
      score_row(H + t * E, E, SOFTMAX, s.data());
      for (int e = 0; e < E; ++e) out[t * E + e] = 2.0 / T * lse * s[e];
    }
  }
}

// dL/dH for L = (loss through the gates) + w_aux E sum f P + w_z L_z.
ORC_API void orc_router_backward(int64_t T, int E, int k, const double* H, const int64_t* idx, const double* d_gate,
                                 const double* f, int fn, int renorm, double w_aux, double w_z, double* dH) {
  orc_gate_backward(T, E, k, H, idx, d_gate, fn, renorm, dH);
  std::vector<double> g(static_cast<size_t>(T) * E);
  if (w_aux != 0.0) {
    orc_aux_loss_grad(T, E, H, f, fn, g.data());
    for (int64_t i = 0; i < T * E; ++i) dH[i] += w_aux * g[i];
  }
  if (w_z != 0.0) {
    orc_z_loss_grad(T, E, H, g.data());
    for (int64_t i = 0; i < T * E; ++i) dH[i] += w_z * g[i];
  }
}

// [BWD] gradients of y = W_down (SiLU(W_gate x) * W_up x) for rows x [n, h] and dL/dy [n, h]:
// G = x W_gate^T, Up = x W_up^T, s = sigmoid(G): d_act = dy W_down, dUp = d_act G s,
// dG = d_act Up s (1 + G (1 - s)), dx = dG W_gate + dUp W_up, dW_gate = dG^T x, dW_up = dUp^T x,
// dW_down = dy^T act.  Weights at element offsets of their arrays; dW_* are written (not added).
ORC_API void orc_swiglu_backward(int64_t n, int h, int d, const double* x, const void* Wg, int wg_dt, int64_t wg_off,
                                 const void* Wu, int wu_dt, int64_t wu_off, const void* Wd, int wd_dt, int64_t wd_off,
                                 const double* dy, double* d_act, double* dG, double* dUp, double* dx, double* dW_gate,
                                 double* dW_up, double* dW_down) {
  std::vector<double> wg(static_cast<size_t>(d) * h), wu(static_cast<size_t>(d) * h), wd(static_cast<size_t>(h) * d);
  widen(Wg, wg_dt, wg_off, static_cast<int64_t>(d) * h, wg.data());
  widen(Wu, wu_dt, wu_off, static_cast<int64_t>(d) * h, wu.data());
  widen(Wd, wd_dt, wd_off, static_cast<int64_t>(h) * d, wd.data());
  std::vector<double> act(static_cast<size_t>(n) * d);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int j = 0; j < d; ++j) {
      const double G = dot(x + r * h, &wg[static_cast<size_t>(j) * h], h);
      const double Up = dot(x + r * h, &wu[static_cast<size_t>(j) * h], h);
      const double sg = 1.0 / (1.0 + std::exp(-G));
      double da = 0.0;
      for (int m = 0; m < h; ++m) da += dy[r * h + m] * wd[static_cast<size_t>(m) * d + j];
      act[r * d + j] = G * sg * Up;
      d_act[r * d + j] = da;
      dUp[r * d + j] = da * G * sg;
      dG[r * d + j] = da * Up * sg * (1.0 + G * (1.0 - sg));
    }
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r)
    for (int c = 0; c < h; ++c) {
      double acc = 0.0;
      for (int j = 0; j < d; ++j)
        acc += dG[r * d + j] * wg[static_cast<size_t>(j) * h + c] + dUp[r * d + j] * wu[static_cast<size_t>(j) * h + c];
      dx[r * h + c] = acc;
    }
#pragma omp parallel for schedule(static)
  for (int j = 0; j < d; ++j)
    for (int c = 0; c < h; ++c) {
      double ag = 0.0, au = 0.0;
      for (int64_t r = 0; r < n; ++r) {
        ag += dG[r * d + j] * x[r * h + c];
        au += dUp[r * d + j] * x[r * h + c];
      }
      dW_gate[static_cast<size_t>(j) * h + c] = ag;
      dW_up[static_cast<size_t>(j) * h + c] = au;
    }
#pragma omp parallel for schedule(static)
  for (int m = 0; m < h; ++m)
    for (int j = 0; j < d; ++j) {
      double acc = 0.0;
      for (int64_t r = 0; r < n; ++r) acc += dy[r * h + m] * act[r * d + j];
      dW_down[static_cast<size_t>(m) * d + j] = acc;
    }
}

// [BWD] the grouped backward over the expert segments of X [A, h] with dY [A, h]: per row d_act,
// dG, dUp [A, d] and dX [A, h]; per expert dW_gate, dW_up [E, d, h] and dW_down [E, h, d] (zero
// for an expert with no rows).
ORC_API void orc_expert_ffn_backward(int64_t A, int h, int d, int E, const double* X, const int64_t* offsets,
                                     const void* Wg, int wg_dt, const void* Wu, int wu_dt, const void* Wd, int wd_dt,
                                     const double* dY, double* d_act, double* dG, double* dUp, double* dX,
                                     double* dW_gate, double* dW_up, double* dW_down) {
  const int64_t hd = static_cast<int64_t>(h) * d;
  for (int64_t i = 0; i < A * d; ++i) d_act[i] = dG[i] = dUp[i] = 0.0;
  for (int64_t i = 0; i < A * h; ++i) dX[i] = 0.0;
  for (int64_t i = 0; i < E * hd; ++i) dW_gate[i] = dW_up[i] = dW_down[i] = 0.0;
  for (int e = 0; e < E; ++e) {
    const int64_t lo = offsets[e], hi = offsets[e + 1];
    if (hi > lo)
      orc_swiglu_backward(hi - lo, h, d, X + lo * h, Wg, wg_dt, e * hd, Wu, wu_dt, e * hd, Wd, wd_dt, e * hd, dY + lo * h,
                          d_act + lo * d, dG + lo * d, dUp + lo * d, dX + lo * h, dW_gate + e * hd, dW_up + e * hd,
                          dW_down + e * hd);
  }
}

// dL/dU from the residual and the permute X = U[perm]: dU_t = dO_t + sum_{kept j} dX[row(t, j)].
ORC_API void orc_dispatch_backward(int64_t T, int h, int k, const double* dO, const double* dX,
                                   const int64_t* slot_row, double* dU) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int c = 0; c < h; ++c) {
      double acc = dO[t * h + c];
      for (int j = 0; j < k; ++j) {
        const int64_t row = slot_row[t * k + j];
        if (row >= 0) acc += dX[row * h + c];
      }
      dU[t * h + c] = acc;
    }
}

// [RTR] backward of H = U W_r + b_r (+ eps Softplus(U W_noise)): dU = dH W_r^T (+ dN W_noise^T),
// dW_r = U^T dH, db_r = sum_t dH, and with noise dN = dH eps sigmoid(U W_noise) (Softplus' =
// sigmoid), dW_noise = U^T dN.
ORC_API void orc_router_input_backward(int64_t T, int h, int E, const void* U, int u_dt, const void* W_r, int wr_dt,
                                       const double* dH, const void* W_noise, int wn_dt, const void* eps, int eps_dt,
                                       double* dU, double* dW_r, double* db_r, double* dW_noise) {
  std::vector<double> u(static_cast<size_t>(T) * h), wr(static_cast<size_t>(h) * E), wn, dN;
  widen(U, u_dt, 0, T * h, u.data());
  widen(W_r, wr_dt, 0, static_cast<int64_t>(h) * E, wr.data());
  if (W_noise) {
    wn.resize(static_cast<size_t>(h) * E);
    widen(W_noise, wn_dt, 0, static_cast<int64_t>(h) * E, wn.data());
    dN.resize(static_cast<size_t>(T) * E);
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
      for (int e = 0; e < E; ++e) {
        double z = 0.0;
        for (int c = 0; c < h; ++c) z += u[t * h + c] * wn[static_cast<size_t>(c) * E + e];
        dN[t * E + e] = dH[t * E + e] * elem(eps, eps_dt, t * E + e) * sigmoid(z);
      }
  }
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int c = 0; c < h; ++c) {
      double acc = 0.0;
      for (int e = 0; e < E; ++e) acc += dH[t * E + e] * wr[static_cast<size_t>(c) * E + e];
      if (W_noise)
        for (int e = 0; e < E; ++e) acc += dN[t * E + e] * wn[static_cast<size_t>(c) * E + e];
      dU[t * h + c] = acc;
    }
#pragma omp parallel for schedule(static)
  for (int c = 0; c < h; ++c)
    for (int e = 0; e < E; ++e) {
      double a = 0.0, an = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        a += u[t * h + c] * dH[t * E + e];
        if (W_noise) an += u[t * h + c] * dN[t * E + e];
      }
      dW_r[static_cast<size_t>(c) * E + e] = a;
      if (W_noise) dW_noise[static_cast<size_t>(c) * E + e] = an;
    }
  for (int e = 0; e < E; ++e) {
    double a = 0.0;
    for (int64_t t = 0; t < T; ++t) a += dH[t * E + e];
    db_r[e] = a;
  }
}

// Gradients of L = <dO, out> + w_aux E sum_i f_i P_i + w_z L_z through the whole layer, with the
// routing decisions (top-k set, slots, drops) of the forward held fixed and f constant
// ([RTR], [AUX], [ZL], [BWD], [SHR]).  Forward results in: logits32 [T, E], idx [T, k],
// slot_row [T k], gate [T, k], X, Y [A, h], offsets [E+1], f [E].  Outputs: dU [T, h],
// d_gate [T, k], dY [A, h], dH [T, E], dW_r [h, E], db_r [E], dW_noise [h, E] (noisy), d_act, dG,
// dUp [A, d], dX [A, h], dW_gate, dW_up [E, d, h], dW_down [E, h, d], and per shared expert
// dW_gate_sh, dW_up_sh [n_s, d_s, h], dW_down_sh [n_s, h, d_s].
ORC_API void orc_layer_backward(
    int64_t T, int h, int E, int k, int d, int fn, int renorm, double w_aux, double w_z, const void* U, int u_dt,
    const void* W_r, int wr_dt, const void* W_noise, int wn_dt, const void* eps, int eps_dt, const void* Wg, int wg_dt,
    const void* Wu, int wu_dt, const void* Wd, int wd_dt, int n_s, int d_s, const void* Wg_sh, int wgs_dt,
    const void* Wu_sh, int wus_dt, const void* Wd_sh, int wds_dt, const double* logits32, const int64_t* idx,
    const int64_t* slot_row, const double* gate, int64_t A, const double* X, const double* Y, const int64_t* offsets,
    const double* f, const double* dO, double* dU, double* d_gate, double* dY, double* dH, double* dW_r, double* db_r,
    double* dW_noise, double* d_act, double* dG, double* dUp, double* dX, double* dW_gate, double* dW_up,
    double* dW_down, double* dW_gate_sh, double* dW_up_sh, double* dW_down_sh) {
  orc_combine_backward(T, h, k, A, dO, Y, slot_row, gate, d_gate, dY);
  orc_router_backward(T, E, k, logits32, idx, d_gate, f, fn, renorm, w_aux, w_z, dH);
  orc_expert_ffn_backward(A, h, d, E, X, offsets, Wg, wg_dt, Wu, wu_dt, Wd, wd_dt, dY, d_act, dG, dUp, dX, dW_gate,
                          dW_up, dW_down);
  std::vector<double> dU_r(static_cast<size_t>(T) * h);
  orc_router_input_backward(T, h, E, U, u_dt, W_r, wr_dt, dH, W_noise, wn_dt, eps, eps_dt, dU_r.data(), dW_r, db_r,
                            dW_noise);
  orc_dispatch_backward(T, h, k, dO, dX, slot_row, dU);
  for (int64_t i = 0; i < T * h; ++i) dU[i] += dU_r[i];
  if (n_s > 0) {
    std::vector<double> u(static_cast<size_t>(T) * h), a(static_cast<size_t>(T) * d_s), g(a.size()), up(a.size()),
        dx(static_cast<size_t>(T) * h);
    widen(U, u_dt, 0, T * h, u.data());
    const int64_t hd = static_cast<int64_t>(h) * d_s;
    for (int i = 0; i < n_s; ++i) {
      orc_swiglu_backward(T, h, d_s, u.data(), Wg_sh, wgs_dt, i * hd, Wu_sh, wus_dt, i * hd, Wd_sh, wds_dt, i * hd, dO,
                          a.data(), g.data(), up.data(), dx.data(), dW_gate_sh + i * hd, dW_up_sh + i * hd,
                          dW_down_sh + i * hd);
      for (int64_t j = 0; j < T * h; ++j) dU[j] += dx[j];
    }
  }
}
