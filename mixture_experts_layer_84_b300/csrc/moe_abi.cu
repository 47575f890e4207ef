// C ABI of libmoe: argument validation, the launch plan and workspace
// carve-up, and the launch sequence of each entry point (include/moe.h).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <stdlib.h>

#include <algorithm>

#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

thread_local char g_last_error[512] = "";

moe_status fail(moe_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

moe_status cuda_fail(const char* where, cudaError_t e) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorString(e), cudaGetErrorName(e));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ceil(cf * Tk / E), exact on the float32 value of cf (cf = m * 2^ex with an integer m).
int64_t capacity_exact(int64_t Tk, int E, float cf) {
  if (Tk == 0) return 0;
  int ex = 0;
  const float fr = frexpf(cf, &ex);  // cf = fr * 2^ex, fr in [0.5, 1)
  const uint64_t m = static_cast<uint64_t>(ldexpf(fr, 24));
  ex -= 24;  // cf = m * 2^ex exactly
  typedef unsigned __int128 u128;
  u128 num = static_cast<u128>(m) * static_cast<u128>(Tk);
  u128 den = static_cast<u128>(E);
  if (ex >= 0) {
    if (ex > 60) return INT64_MAX;
    num <<= ex;
  } else {
    if (-ex > 100) return 1;  // 0 < cf*Tk/E < 1
    den <<= -ex;
  }
  const u128 q = (num + den - 1) / den;
  return q > static_cast<u128>(INT64_MAX) ? INT64_MAX : static_cast<int64_t>(q);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A device array argument: required unless it holds no bytes; aligned as given.
moe_status check_ptr(const char* fn, const char* name, const void* p, size_t bytes, size_t align) {
  if (bytes > 0 && p == nullptr) return fail(MOE_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
  if (p != nullptr && !aligned(p, align))
    return fail(MOE_ERR_INVALID_ARG, "%s: %s is not %zu-byte aligned", fn, name, align);
  return MOE_OK;
}

#define CHECK(expr)                   \
  do {                                \
    moe_status st_ = (expr);          \
    if (st_ != MOE_OK) return st_;    \
  } while (0)

}  // namespace

moe_status make_plan(const moe_config* cfg, Plan* p, const char** msg) {
  static thread_local char buf[256];
  auto bad = [&](moe_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    *msg = buf;
    return st;
  };
  if (!cfg) return bad(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->T < 0) return bad(MOE_ERR_INVALID_ARG, "T = %lld < 0", static_cast<long long>(cfg->T));
  if (cfg->h < 1 || cfg->E < 1 || cfg->k < 1 || cfg->d_e < 1)
    return bad(MOE_ERR_INVALID_ARG, "h, E, k, d_e must be >= 1 (got %d, %d, %d, %d)", cfg->h, cfg->E, cfg->k,
               cfg->d_e);
  if (cfg->k > cfg->E) return bad(MOE_ERR_INVALID_ARG, "k = %d > E = %d", cfg->k, cfg->E);
  if (cfg->dtype != MOE_F32 && cfg->dtype != MOE_BF16) return bad(MOE_ERR_INVALID_ARG, "dtype %d", cfg->dtype);
  if (cfg->score_fn != MOE_SCORE_SOFTMAX && cfg->score_fn != MOE_SCORE_SIGMOID)
    return bad(MOE_ERR_INVALID_ARG, "score_fn %d", cfg->score_fn);
  if (cfg->priority != MOE_PRIORITY_CHOICE_MAJOR && cfg->priority != MOE_PRIORITY_TOKEN_MAJOR)
    return bad(MOE_ERR_INVALID_ARG, "priority %d", cfg->priority);
  if (cfg->capacity < 0) return bad(MOE_ERR_INVALID_ARG, "capacity = %d < 0", cfg->capacity);
  if (!isfinite(cfg->capacity_factor)) return bad(MOE_ERR_INVALID_ARG, "capacity_factor is not finite");
  if (cfg->n_shared < 0 || cfg->n_shared > 16)
    return bad(MOE_ERR_INVALID_ARG, "n_shared = %d outside 0..16", cfg->n_shared);
  if (cfg->n_shared > 0 && (cfg->d_shared < 8 || cfg->d_shared % 8 != 0))
    return bad(MOE_ERR_UNSUPPORTED, "d_shared = %d must be a positive multiple of 8", cfg->d_shared);
  if (cfg->n_shared > 0 && cfg->dtype == MOE_BF16 &&
      static_cast<int64_t>(cfg->n_shared) * std::max(cfg->h, cfg->d_shared) >= (int64_t(1) << 31))
    return bad(MOE_ERR_UNSUPPORTED, "n_shared * max(h, d_shared) >= 2^31");
  if (cfg->n_group > 1) {
    if (cfg->n_group > MAX_GROUPS) return bad(MOE_ERR_UNSUPPORTED, "n_group = %d > %d", cfg->n_group, MAX_GROUPS);
    if (cfg->E % cfg->n_group != 0)
      return bad(MOE_ERR_INVALID_ARG, "E = %d is not a multiple of n_group = %d", cfg->E, cfg->n_group);
    if (cfg->topk_group < 1 || cfg->topk_group > cfg->n_group)
      return bad(MOE_ERR_INVALID_ARG, "topk_group = %d outside 1..n_group = %d", cfg->topk_group, cfg->n_group);
    if (cfg->k % cfg->topk_group != 0)
      return bad(MOE_ERR_INVALID_ARG, "k = %d is not a multiple of topk_group = %d", cfg->k, cfg->topk_group);
    if (static_cast<int64_t>(cfg->topk_group) * (cfg->E / cfg->n_group) < cfg->k)
      return bad(MOE_ERR_INVALID_ARG, "k = %d > topk_group * E / n_group = %d", cfg->k,
                 cfg->topk_group * (cfg->E / cfg->n_group));
  } else if (cfg->n_group < 0) {
    return bad(MOE_ERR_INVALID_ARG, "n_group = %d < 0", cfg->n_group);
  }
  if (cfg->E > 1024) return bad(MOE_ERR_UNSUPPORTED, "E = %d > 1024", cfg->E);
  if (cfg->k > 16) return bad(MOE_ERR_UNSUPPORTED, "k = %d > 16", cfg->k);
  if (cfg->h % 8 != 0 || cfg->d_e % 8 != 0)
    return bad(MOE_ERR_UNSUPPORTED, "h = %d and d_e = %d must be multiples of 8", cfg->h, cfg->d_e);
  const int64_t Tk = cfg->T * cfg->k;
  if (Tk >= (int64_t(1) << 31)) return bad(MOE_ERR_UNSUPPORTED, "T * k = %lld >= 2^31", static_cast<long long>(Tk));
  if (cfg->dtype == MOE_BF16 && static_cast<int64_t>(cfg->E) * std::max(cfg->h, cfg->d_e) >= (int64_t(1) << 31))
    return bad(MOE_ERR_UNSUPPORTED, "E * max(h, d_e) >= 2^31");

  Plan q;
  q.T = cfg->T;
  q.h = cfg->h;
  q.E = cfg->E;
  q.k = cfg->k;
  q.d_e = cfg->d_e;
  q.Tk = Tk;
  q.bf16 = cfg->dtype == MOE_BF16;
  q.noisy = cfg->noisy != 0;
  q.score_fn = cfg->score_fn;
  q.renorm = cfg->renorm != 0;
  q.priority = cfg->priority;
  q.n_shared = cfg->n_shared;
  q.d_shared = cfg->d_shared;
  if (cfg->n_group > 1) {
    q.n_group = cfg->n_group;
    q.topk_group = cfg->topk_group;
  }
  if (cfg->capacity > 0)
    q.C = cfg->capacity;
  else if (cfg->capacity_factor <= 0.f)
    q.C = cfg->T;
  else
    q.C = capacity_exact(Tk, cfg->E, cfg->capacity_factor);

  int ep = 8;
  while (ep < q.E) ep <<= 1;
  q.route_ep = ep;
  q.route_bt = route_bt_for(ep);
  q.route_kc = route_kc_for(ep);
  q.route_rowblocks = static_cast<int>((q.T + q.route_bt - 1) / q.route_bt);
  const int nkc = (q.h + q.route_kc - 1) / q.route_kc;
  int splits = q.route_rowblocks > 0 ? (512 + q.route_rowblocks - 1) / q.route_rowblocks : 1;
  splits = std::max(1, std::min(splits, std::min(16, nkc)));
  // bf16 with at most 256 logit columns per token (E, or 2E for the noisy router): tensor cores,
  // 128-token tiles, h split so that the tiles x slices cover the GPU with >= 4 k-blocks a slice
  const int n_cols = q.noisy ? 2 * q.E : q.E;
  if (q.bf16 && n_cols <= 256) {
    q.route_tc_n = (n_cols + 15) / 16 * 16;
    const int64_t mtiles = (q.T + 127) / 128;
    const int nkb = (q.h + 63) / 64;
    int64_t want = mtiles > 0 ? (148 + mtiles - 1) / mtiles : 1;
    want = std::min<int64_t>(want, std::max(1, nkb / 4));
    splits = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, 16)));
  }
  q.route_splits = splits;
  // the fused router: one 128-token tile per cluster of rf_cs CTAs, each CTA a slice of h (at least
  // two 64-wide K-blocks), clusters of up to 8 while the grid stays within about one wave
  if (q.route_tc_n > 0) {
    q.route_fused = true;
    q.rf_tiles = static_cast<int>((q.T + 127) / 128);
    const int nkb = (q.h + 63) / 64;
    int cs = 1;
    while (cs < 8 && static_cast<int64_t>(q.rf_tiles) * cs * 2 <= 160 && nkb >= cs * 4) cs *= 2;
    // (MOE_ROUTE_CS=1|2|4|8 overrides the cluster size, for measurement)
    if (const char* env = getenv("MOE_ROUTE_CS")) {
      const int v = atoi(env);
      if (v == 1 || v == 2 || v == 4 || v == 8) cs = v;
    }
    q.rf_cs = cs;
    // ring depth: four stages when the grid takes several waves (two CTAs share an SM, one's
    // epilogue overlapping the other's loads); when it fits one wave, as deep as ~100 KB allows
    // (up to eight), so that two CTAs still fit an SM: clusters of 8 CTAs that need 8 SMs of one
    // GPC each do not all fit at once (measured: 28 vs 16 us on the Mixtral router)
    const int stage_kb = 16 + q.route_tc_n * 128 / 1024;
    q.rf_stages = static_cast<int64_t>(q.rf_tiles) * cs > 148 ? 4 : std::max(4, std::min(8, 100 / stage_kb));
    // one wave whose four-stage ring already fills an SM (N > 96: the 256-expert and the noisy
    // 128-expert routers): 512 threads, so that the epilogue has 16 warps to hide its latencies
    q.rf_threads = static_cast<int64_t>(q.rf_tiles) * cs <= 148 && 4 * stage_kb > 113 ? 512 : 256;
  }
  // selection blocks: 256 threads, fewer (down to a warp) when T is small, so that the
  // blocks still spread over about twice the SMs
  {
    const int G = select_lanes_for(q.E);
    int64_t threads = q.T > 0 ? G * ((q.T + 2 * 148 - 1) / (2 * 148)) : SELECT_THREADS;
    threads = (threads + 31) / 32 * 32;
    q.sel_threads = static_cast<int>(std::max<int64_t>(std::max(32, G), std::min<int64_t>(SELECT_THREADS, threads)));
    q.sel_tokens = q.sel_threads / G;
  }
  q.sel_blocks = static_cast<int>((q.T + q.sel_tokens - 1) / q.sel_tokens);
  // dispatch chunks: about two per SM (multiples of 256 positions, 256 .. 4096), so small
  // batches still spread over the GPU and large ones keep the histogram short
  {
    int64_t c = (Tk + 2 * 148 - 1) / (2 * 148);
    c = (c + 255) / 256 * 256;
    q.chunk = static_cast<int>(std::max<int64_t>(256, std::min<int64_t>(kDispatchChunk, c)));
  }
  q.n_chunks = static_cast<int>((Tk + q.chunk - 1) / q.chunk);
  // choice-major dispatch: token chunks of 8 .. 256 tokens, about two per SM
  {
    int tc = 8;
    while (tc < 256 && static_cast<int64_t>(tc) * 2 * 148 < q.T) tc *= 2;
    q.dp_tc = tc;
    q.dp_chunks = static_cast<int>((q.T + tc - 1) / tc);
  }

  size_t off = 0;
  q.ws_status = off;
  off += 256;
  const size_t logits_bytes = sizeof(float) * static_cast<size_t>(splits) * q.T * q.E;
  q.ws_part = off;
  off += align256(logits_bytes);
  q.ws_npart = off;
  if (q.noisy) off += align256(logits_bytes);
  q.ws_ppart = off;
  const int64_t ppart_rows = std::max<int64_t>(q.sel_blocks, static_cast<int64_t>(q.rf_tiles) * q.rf_cs);
  off += align256(sizeof(float) * static_cast<size_t>(ppart_rows) * (q.E + 1));
  q.ws_stats2 = off;
  off += align256(sizeof(float) * 32 * static_cast<size_t>(q.E + 1));
  q.ws_hist = off;
  off += align256(sizeof(int32_t) * std::max(static_cast<size_t>(q.n_chunks) * q.E,
                                             (static_cast<size_t>(q.dp_chunks) + 2) * q.k * q.E));
  q.ws_wt = off;
  if (q.route_tc_n > 0) off += align256(sizeof(uint16_t) * static_cast<size_t>(q.route_tc_n) * q.h);
  q.rb_np = ((q.noisy ? 2 * q.E : q.E) + 7) / 8 * 8;
  q.ws_rb_dh = off;
  off += align256(sizeof(uint16_t) * static_cast<size_t>(q.T) * q.rb_np);
  q.ws_rb_w = off;
  off += align256(sizeof(uint16_t) * static_cast<size_t>(q.h) * q.rb_np);
  q.ws_rb_dw = off;
  off += align256(sizeof(float) * static_cast<size_t>(q.h) * q.rb_np);
  q.ws_total = off;
  *p = q;
  return MOE_OK;
}

namespace {

moe_status plan_or_fail(const char* fn, const moe_config* cfg, Plan* p) {
  const char* msg = "";
  const moe_status st = make_plan(cfg, p, &msg);
  if (st != MOE_OK) return fail(st, "%s: %s", fn, msg);
  return MOE_OK;
}

moe_status check_route_args(const char* fn, const Plan& p, const void* U, const void* W_r, const void* W_noise,
                            const float* eps, const float* logits_in, const float* logits_out, const int32_t* idx,
                            const float* gate, const void* ws) {
  const size_t es = p.bf16 ? 2 : 4;
  const size_t TE = static_cast<size_t>(p.T) * p.E;
  if (!logits_in) {
    CHECK(check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * es, 16));
    CHECK(check_ptr(fn, "W_r", W_r, p.T > 0 ? static_cast<size_t>(p.h) * p.E * es : 0, es));
    if (p.noisy) {
      CHECK(check_ptr(fn, "W_noise", W_noise, p.T > 0 ? static_cast<size_t>(p.h) * p.E * es : 0, es));
      CHECK(check_ptr(fn, "eps", eps, TE * 4, 4));
    }
  } else {
    CHECK(check_ptr(fn, "logits_in", logits_in, TE * 4, 4));
  }
  CHECK(check_ptr(fn, "logits_out", logits_out, 0, 4));
  CHECK(check_ptr(fn, "idx", idx, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "gate", gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "ws", ws, p.ws_total, 256));
  return MOE_OK;
}

moe_status check_dispatch_args(const char* fn, const Plan& p, const void* U, const int32_t* idx,
                               const int32_t* counts_routed, const int32_t* counts_kept, const int32_t* offsets,
                               const int32_t* slot_row, const int32_t* row_token, const void* X,
                               const int64_t* n_dropped, const void* ws) {
  const size_t es = p.bf16 ? 2 : 4;
  CHECK(check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(check_ptr(fn, "idx", idx, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "counts_routed", counts_routed, static_cast<size_t>(p.E) * 4, 4));
  CHECK(check_ptr(fn, "counts_kept", counts_kept, static_cast<size_t>(p.E) * 4, 4));
  CHECK(check_ptr(fn, "offsets", offsets, static_cast<size_t>(p.E + 1) * 4, 4));
  CHECK(check_ptr(fn, "slot_row", slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "row_token", row_token, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "X", X, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(check_ptr(fn, "n_dropped", n_dropped, 8, 8));
  CHECK(check_ptr(fn, "ws", ws, p.ws_total, 256));
  return MOE_OK;
}

moe_status check_ffn_args(const char* fn, const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                          const void* W_up, const void* W_down, const void* act, const void* Y, const void* ws) {
  const size_t es = p.bf16 ? 2 : 4;
  const size_t wbytes = p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * p.h * es : 0;
  CHECK(check_ptr(fn, "X", X, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(check_ptr(fn, "offsets", offsets, static_cast<size_t>(p.E + 1) * 4, 4));
  CHECK(check_ptr(fn, "W_gate", W_gate, wbytes, 16));
  CHECK(check_ptr(fn, "W_up", W_up, wbytes, 16));
  CHECK(check_ptr(fn, "W_down", W_down, wbytes, 16));
  CHECK(check_ptr(fn, "act", act, static_cast<size_t>(p.Tk) * p.d_e * es, 16));
  CHECK(check_ptr(fn, "Y", Y, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(check_ptr(fn, "ws", ws, p.ws_total, 256));
  return MOE_OK;
}

moe_status check_combine_args(const char* fn, const Plan& p, const void* U, const void* Y, const int32_t* slot_row,
                              const float* gate, const int32_t* counts_routed, const void* out, const float* f,
                              const float* P, const float* aux, const void* ws) {
  const size_t es = p.bf16 ? 2 : 4;
  CHECK(check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(check_ptr(fn, "Y", Y, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(check_ptr(fn, "slot_row", slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "gate", gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(check_ptr(fn, "counts_routed", counts_routed, static_cast<size_t>(p.E) * 4, 4));
  CHECK(check_ptr(fn, "out", out, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(check_ptr(fn, "f", f, static_cast<size_t>(p.E) * 4, 4));
  CHECK(check_ptr(fn, "P", P, static_cast<size_t>(p.E) * 4, 4));
  CHECK(check_ptr(fn, "aux", aux, 4, 4));
  CHECK(check_ptr(fn, "ws", ws, p.ws_total, 256));
  return MOE_OK;
}

}  // namespace

cudaError_t launch_expert_ffn(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                              const void* W_up, const void* W_down, void* act, void* Y, uint8_t* ws, cudaStream_t s) {
  if (p.bf16) return launch_ffn_tc(p, X, offsets, W_gate, W_up, W_down, act, Y, ws_status(p, ws), s);
  return launch_ffn_simt_f32(p, X, offsets, W_gate, W_up, W_down, act, Y, ws_status(p, ws), s);
}

// Shared expert i is a grouped FFN with one segment of all T rows (no offsets): the same
// kernels, planned with E = 1, T rows and d_shared.
cudaError_t launch_shared_ffn(const Plan& p, const void* U, const void* W_gate_sh, const void* W_up_sh,
                              const void* W_down_sh, void* act_sh, void* Y_sh, uint8_t* ws, cudaStream_t s) {
  if (p.T == 0 || p.n_shared == 0) return cudaSuccess;
  Plan q = p;
  q.E = 1;
  q.k = 1;
  q.Tk = p.T;
  q.d_e = p.d_shared;
  const size_t es = p.bf16 ? 2 : 4;
  const size_t w_in = static_cast<size_t>(p.d_shared) * p.h * es;  // one shared expert's W_gate / W_up / W_down
  for (int i = 0; i < p.n_shared; ++i) {
    const uint8_t* wg = static_cast<const uint8_t*>(W_gate_sh) + i * w_in;
    const uint8_t* wu = static_cast<const uint8_t*>(W_up_sh) + i * w_in;
    const uint8_t* wd = static_cast<const uint8_t*>(W_down_sh) + i * w_in;
    uint8_t* y = static_cast<uint8_t*>(Y_sh) + static_cast<size_t>(i) * p.T * p.h * es;
    uint8_t* a = static_cast<uint8_t*>(act_sh) + static_cast<size_t>(i) * p.T * p.d_shared * es;
    const cudaError_t e = launch_expert_ffn(q, U, nullptr, wg, wu, wd, a, y, ws, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

moe_status check_shared_args(const char* fn, const Plan& p, const void* U, const void* W_gate_sh, const void* W_up_sh,
                             const void* W_down_sh, const void* act_sh, const void* Y_sh) {
  if (p.n_shared == 0) return MOE_OK;
  const size_t es = p.bf16 ? 2 : 4;
  const size_t w = p.T > 0 ? static_cast<size_t>(p.n_shared) * p.d_shared * p.h * es : 0;
  CHECK(check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(check_ptr(fn, "W_gate_shared", W_gate_sh, w, 16));
  CHECK(check_ptr(fn, "W_up_shared", W_up_sh, w, 16));
  CHECK(check_ptr(fn, "W_down_shared", W_down_sh, w, 16));
  CHECK(check_ptr(fn, "act_shared", act_sh, static_cast<size_t>(p.n_shared) * p.T * p.d_shared * es, 16));
  CHECK(check_ptr(fn, "Y_shared", Y_sh, static_cast<size_t>(p.n_shared) * p.T * p.h * es, 16));
  return MOE_OK;
}

}  // namespace moe

using moe::Plan;

MOE_API const char* moe_version(void) { return "moe-b300 0.1 sm_103a"; }

MOE_API const char* moe_status_string(moe_status status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

MOE_API const char* moe_last_error(void) { return moe::g_last_error; }

MOE_API moe_status moe_capacity(const moe_config* cfg, int64_t* C) {
  Plan p;
  CHECK(moe::plan_or_fail("moe_capacity", cfg, &p));
  if (!C) return moe::fail(MOE_ERR_INVALID_ARG, "moe_capacity: C is NULL");
  *C = p.C;
  return MOE_OK;
}

MOE_API moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
  Plan p;
  CHECK(moe::plan_or_fail("moe_workspace_size", cfg, &p));
  if (!bytes) return moe::fail(MOE_ERR_INVALID_ARG, "moe_workspace_size: bytes is NULL");
  *bytes = p.ws_total;
  return MOE_OK;
}

MOE_API moe_status moe_router_pack_size(const moe_config* cfg, size_t* bytes) {
  Plan p;
  CHECK(moe::plan_or_fail("moe_router_pack_size", cfg, &p));
  if (!bytes) return moe::fail(MOE_ERR_INVALID_ARG, "moe_router_pack_size: bytes is NULL");
  *bytes = p.route_tc_n > 0 ? sizeof(uint16_t) * static_cast<size_t>(p.route_tc_n) * p.h : 0;
  return MOE_OK;
}

MOE_API moe_status moe_pack_router(const moe_config* cfg, const void* W_r, const void* W_noise, void* W_r_packed,
                                   moe_stream_t stream) {
  static const char* fn = "moe_pack_router";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (p.route_tc_n == 0)
    return moe::fail(MOE_ERR_UNSUPPORTED, "%s: this config's router reads W_r as it is (float32, or > 256 columns)",
                     fn);
  const size_t wbytes = sizeof(uint16_t) * static_cast<size_t>(p.h) * p.E;
  CHECK(moe::check_ptr(fn, "W_r", W_r, wbytes, 2));
  if (p.noisy) CHECK(moe::check_ptr(fn, "W_noise", W_noise, wbytes, 2));
  CHECK(moe::check_ptr(fn, "W_r_packed", W_r_packed, sizeof(uint16_t) * static_cast<size_t>(p.route_tc_n) * p.h, 16));
  const cudaError_t e = moe::launch_pack_router(p, W_r, W_noise, W_r_packed, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_route_packed(const moe_config* cfg, const void* U, const void* W_r_packed, const float* b_r,
                                    const float* sel_bias, const float* eps, float* logits_out, int32_t* idx,
                                    float* gate, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_route_packed";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!p.route_fused)
    return moe::fail(MOE_ERR_UNSUPPORTED, "%s: this config's router does not use packed weights", fn);
  // W_r and W_noise are replaced by the packed matrix: pass it for both pointer checks
  CHECK(moe::check_route_args(fn, p, U, W_r_packed, W_r_packed, eps, nullptr, logits_out, idx, gate, ws));
  CHECK(moe::check_ptr(fn, "W_r_packed", W_r_packed, sizeof(uint16_t) * static_cast<size_t>(p.route_tc_n) * p.h, 16));
  CHECK(moe::check_ptr(fn, "b_r", b_r, 0, 4));
  CHECK(moe::check_ptr(fn, "sel_bias", sel_bias, 0, 4));
  const cudaError_t e = moe::launch_route(p, U, nullptr, b_r, sel_bias, nullptr, eps, nullptr, logits_out, idx, gate,
                                          static_cast<uint8_t*>(ws), stream, W_r_packed);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_route(const moe_config* cfg, const void* U, const void* W_r, const float* b_r,
                             const float* sel_bias, const void* W_noise, const float* eps, const float* logits_in,
                             float* logits_out, int32_t* idx, float* gate, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_route";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_route_args(fn, p, U, W_r, W_noise, eps, logits_in, logits_out, idx, gate, ws));
  CHECK(moe::check_ptr(fn, "b_r", b_r, 0, 4));
  CHECK(moe::check_ptr(fn, "sel_bias", sel_bias, 0, 4));
  const cudaError_t e = moe::launch_route(p, U, W_r, b_r, sel_bias, W_noise, eps, logits_in, logits_out, idx, gate,
                                          static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_dispatch(const moe_config* cfg, const void* U, const int32_t* idx, int32_t* counts_routed,
                                int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                void* X, int64_t* n_dropped, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_dispatch";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  // X may be NULL (routing metadata only): U stands in for it in the pointer checks
  CHECK(moe::check_dispatch_args(fn, p, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, X ? X : U,
                                 n_dropped, ws));
  CHECK(moe::check_ptr(fn, "X", X, 0, 16));
  const cudaError_t e = moe::launch_dispatch(p, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, X,
                                             n_dropped, static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_dispatch_noalloc(const moe_config* cfg, const void* U, const int32_t* idx,
                                        int32_t* counts_routed, int32_t* counts_kept, int32_t* offsets,
                                        int32_t* slot_row, int32_t* row_token, void* X, int64_t* n_dropped,
                                        int32_t* status, moe_stream_t stream) {
  static const char* fn = "moe_dispatch_noalloc";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  const int64_t hist = static_cast<int64_t>(p.n_chunks) * p.E;
  if (hist > MOE_NOALLOC_HIST_MAX)
    return moe::fail(MOE_ERR_UNSUPPORTED,
                     "%s: ceil(T*k/%d) * E = %lld exceeds the static histogram of %d entries; use moe_dispatch", fn,
                     p.chunk, static_cast<long long>(hist), MOE_NOALLOC_HIST_MAX);
  const size_t es = p.bf16 ? 2 : 4;
  CHECK(moe::check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "idx", idx, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "counts_routed", counts_routed, static_cast<size_t>(p.E) * 4, 4));
  CHECK(moe::check_ptr(fn, "counts_kept", counts_kept, static_cast<size_t>(p.E) * 4, 4));
  CHECK(moe::check_ptr(fn, "offsets", offsets, static_cast<size_t>(p.E + 1) * 4, 4));
  CHECK(moe::check_ptr(fn, "slot_row", slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "row_token", row_token, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "X", X, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "n_dropped", n_dropped, 8, 8));
  CHECK(moe::check_ptr(fn, "status", status, 0, 4));
  const cudaError_t e = moe::launch_dispatch_noalloc(p, U, idx, counts_routed, counts_kept, offsets, slot_row,
                                                     row_token, X, n_dropped, status, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const void* X, const int32_t* offsets, const void* W_gate,
                                  const void* W_up, const void* W_down, void* act, void* Y, void* ws,
                                  moe_stream_t stream) {
  static const char* fn = "moe_expert_ffn";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_ffn_args(fn, p, X, offsets, W_gate, W_up, W_down, act, Y, ws));
  const cudaError_t e = moe::launch_expert_ffn(p, X, offsets, W_gate, W_up, W_down, act, Y,
                                               static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_expert_ffn_gather(const moe_config* cfg, const void* U, const int32_t* row_token,
                                         const int32_t* offsets, const void* W_gate, const void* W_up,
                                         const void* W_down, void* act, void* Y, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_expert_ffn_gather";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!p.bf16) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the gathered up-projection needs a bf16 config", fn);
  // U stands in for X in the shared checks; row_token is read for the first A = offsets[E] rows
  CHECK(moe::check_ffn_args(fn, p, U, offsets, W_gate, W_up, W_down, act, Y, ws));
  CHECK(moe::check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * 2, 16));
  CHECK(moe::check_ptr(fn, "row_token", row_token, static_cast<size_t>(p.Tk) * 4, 4));
  const cudaError_t e = moe::launch_ffn_tc(p, nullptr, offsets, W_gate, W_up, W_down, act, Y,
                                           moe::ws_status(p, static_cast<uint8_t*>(ws)), stream, U, row_token);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_combine(const moe_config* cfg, const void* U, const void* Y, const void* Y_shared,
                               const int32_t* slot_row, const float* gate, const int32_t* counts_routed, void* out,
                               float* f, float* P, float* aux, float* z_loss, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_combine";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_combine_args(fn, p, U, Y, slot_row, gate, counts_routed, out, f, P, aux, ws));
  CHECK(moe::check_ptr(fn, "z_loss", z_loss, 0, 4));
  if (p.n_shared > 0)
    CHECK(moe::check_ptr(fn, "Y_shared", Y_shared, static_cast<size_t>(p.n_shared) * p.T * p.h * (p.bf16 ? 2 : 4),
                         16));
  const cudaError_t e = moe::launch_combine(p, U, Y, p.n_shared > 0 ? Y_shared : nullptr, slot_row, gate,
                                            counts_routed, out, f, P, aux, z_loss,
                                            static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_shared_ffn(const moe_config* cfg, const void* U, const void* W_gate_shared,
                                  const void* W_up_shared, const void* W_down_shared, void* act_shared,
                                  void* Y_shared, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_shared_ffn";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (p.n_shared == 0) return moe::fail(MOE_ERR_INVALID_ARG, "%s: cfg->n_shared is 0", fn);
  CHECK(moe::check_shared_args(fn, p, U, W_gate_shared, W_up_shared, W_down_shared, act_shared, Y_shared));
  CHECK(moe::check_ptr(fn, "ws", ws, p.ws_total, 256));
  const cudaError_t e = moe::launch_shared_ffn(p, U, W_gate_shared, W_up_shared, W_down_shared, act_shared, Y_shared,
                                               static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_balance_bias_update(const moe_config* cfg, const int32_t* counts_routed, float u, float* bias,
                                           moe_stream_t stream) {
  static const char* fn = "moe_balance_bias_update";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!isfinite(u)) return moe::fail(MOE_ERR_INVALID_ARG, "%s: u is not finite", fn);
  CHECK(moe::check_ptr(fn, "counts_routed", counts_routed, static_cast<size_t>(p.E) * 4, 4));
  CHECK(moe::check_ptr(fn, "bias", bias, static_cast<size_t>(p.E) * 4, 4));
  const cudaError_t e = moe::launch_balance_bias_update(p.E, counts_routed, u, bias, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_combine_backward(const moe_config* cfg, const void* dO, const void* Y, const int32_t* slot_row,
                                        const float* gate, float* d_gate, void* dY, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_combine_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  const size_t es = p.bf16 ? 2 : 4;
  CHECK(moe::check_ptr(fn, "dO", dO, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "Y", Y, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "slot_row", slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "gate", gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "d_gate", d_gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "dY", dY, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "ws", ws, p.ws_total, 256));
  const cudaError_t e = moe::launch_combine_backward(p, dO, Y, slot_row, gate, d_gate, dY, static_cast<uint8_t*>(ws),
                                                     stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_route_backward(const moe_config* cfg, const float* logits, const int32_t* idx,
                                      const float* d_gate, const int32_t* counts_routed, float w_aux, float w_z,
                                      float* dH, moe_stream_t stream) {
  static const char* fn = "moe_route_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!isfinite(w_aux) || !isfinite(w_z)) return moe::fail(MOE_ERR_INVALID_ARG, "%s: w_aux / w_z not finite", fn);
  CHECK(moe::check_ptr(fn, "logits", logits, static_cast<size_t>(p.T) * p.E * 4, 4));
  CHECK(moe::check_ptr(fn, "idx", idx, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "d_gate", d_gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "counts_routed", counts_routed, w_aux != 0.f ? static_cast<size_t>(p.E) * 4 : 0, 4));
  CHECK(moe::check_ptr(fn, "dH", dH, static_cast<size_t>(p.T) * p.E * 4, 4));
  const cudaError_t e = moe::launch_route_backward(p, logits, idx, d_gate, counts_routed, w_aux, w_z, dH, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_expert_ffn_backward(const moe_config* cfg, const void* X, const int32_t* offsets,
                                           const void* W_gate, const void* W_up, const void* W_down, const void* act,
                                           const void* dY, void* d_act, void* dG, void* dUp, void* dX,
                                           float* dW_gate, float* dW_up, float* dW_down, void* ws,
                                           moe_stream_t stream) {
  static const char* fn = "moe_expert_ffn_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!p.bf16) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the expert backward runs on bf16 (tcgen05) only", fn);
  CHECK(moe::check_ffn_args(fn, p, X, offsets, W_gate, W_up, W_down, act, dY, ws));
  const size_t rows_d = static_cast<size_t>(p.Tk) * p.d_e * 2, rows_h = static_cast<size_t>(p.Tk) * p.h * 2;
  const size_t wgrad = p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * p.h * 4 : 0;
  CHECK(moe::check_ptr(fn, "d_act", d_act, rows_d, 16));
  CHECK(moe::check_ptr(fn, "dG", dG, rows_d, 16));
  CHECK(moe::check_ptr(fn, "dUp", dUp, rows_d, 16));
  CHECK(moe::check_ptr(fn, "dX", dX, rows_h, 16));
  CHECK(moe::check_ptr(fn, "dW_gate", dW_gate, wgrad, 16));
  CHECK(moe::check_ptr(fn, "dW_up", dW_up, wgrad, 16));
  CHECK(moe::check_ptr(fn, "dW_down", dW_down, wgrad, 16));
  const cudaError_t e = moe::launch_ffn_backward_tc(p, X, offsets, W_gate, W_up, W_down, act, dY, d_act, dG, dUp, dX,
                                                    dW_gate, dW_up, dW_down,
                                                    moe::ws_status(p, static_cast<uint8_t*>(ws)), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_dispatch_backward(const moe_config* cfg, const void* dO, const void* dX,
                                         const int32_t* slot_row, void* dU, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_dispatch_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  const size_t es = p.bf16 ? 2 : 4;
  CHECK(moe::check_ptr(fn, "dO", dO, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "dX", dX, static_cast<size_t>(p.Tk) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "slot_row", slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "dU", dU, static_cast<size_t>(p.T) * p.h * es, 16));
  CHECK(moe::check_ptr(fn, "ws", ws, p.ws_total, 256));
  const cudaError_t e = moe::launch_dispatch_backward(p, dO, dX, slot_row, dU, static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_router_input_backward(const moe_config* cfg, const void* U, const void* W_r,
                                             const void* W_noise, const float* eps, const float* dH, void* dU_router,
                                             float* dW_r, float* dW_noise, float* db_r, void* ws,
                                             moe_stream_t stream) {
  static const char* fn = "moe_router_input_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!p.bf16) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the router backward runs on bf16 (tcgen05) only", fn);
  if (p.noisy && p.route_tc_n == 0)
    return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the noisy router backward needs 2E <= 256", fn);
  const size_t TE = static_cast<size_t>(p.T) * p.E, hE = static_cast<size_t>(p.h) * p.E;
  CHECK(moe::check_ptr(fn, "U", U, static_cast<size_t>(p.T) * p.h * 2, 16));
  CHECK(moe::check_ptr(fn, "W_r", W_r, p.T > 0 ? hE * 2 : 0, 16));
  if (p.noisy) {
    CHECK(moe::check_ptr(fn, "W_noise", W_noise, p.T > 0 ? hE * 2 : 0, 16));
    CHECK(moe::check_ptr(fn, "eps", eps, TE * 4, 4));
    CHECK(moe::check_ptr(fn, "dW_noise", dW_noise, p.T > 0 ? hE * 4 : 0, 16));
  }
  CHECK(moe::check_ptr(fn, "dH", dH, TE * 4, 4));
  CHECK(moe::check_ptr(fn, "dU_router", dU_router, static_cast<size_t>(p.T) * p.h * 2, 16));
  CHECK(moe::check_ptr(fn, "dW_r", dW_r, p.T > 0 ? hE * 4 : 0, 16));
  CHECK(moe::check_ptr(fn, "db_r", db_r, 0, 4));
  CHECK(moe::check_ptr(fn, "ws", ws, p.ws_total, 256));
  const cudaError_t e = moe::launch_router_input_backward(p, U, W_r, W_noise, eps, dH, dU_router, dW_r, dW_noise,
                                                          db_r, static_cast<uint8_t*>(ws), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_layer_backward(const moe_config* cfg, const moe_layer_args* a, const moe_layer_grads* g,
                                      void* ws, moe_stream_t stream) {
  static const char* fn = "moe_layer_backward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!a || !g) return moe::fail(MOE_ERR_INVALID_ARG, "%s: args or grads is NULL", fn);
  if (!p.bf16) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the backward runs on bf16 (tcgen05) only", fn);
  if (p.noisy && p.route_tc_n == 0)
    return moe::fail(MOE_ERR_UNSUPPORTED, "%s: the noisy router backward needs 2E <= 256", fn);
  if (!isfinite(g->w_aux) || !isfinite(g->w_z)) return moe::fail(MOE_ERR_INVALID_ARG, "%s: w_aux / w_z", fn);
  const size_t es = 2, Th = static_cast<size_t>(p.T) * p.h * es, Tkh = static_cast<size_t>(p.Tk) * p.h * es;
  const size_t Tkd = static_cast<size_t>(p.Tk) * p.d_e * es, TE = static_cast<size_t>(p.T) * p.E * 4;
  const size_t wg = p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * p.h * 4 : 0;
  const size_t hE = p.T > 0 ? static_cast<size_t>(p.h) * p.E * 4 : 0;
  // what the forward saved
  CHECK(moe::check_ffn_args(fn, p, a->X, a->offsets, a->W_gate, a->W_up, a->W_down, a->act, a->Y, ws));
  CHECK(moe::check_ptr(fn, "U", a->U, Th, 16));
  CHECK(moe::check_ptr(fn, "W_r", a->W_r, p.T > 0 ? static_cast<size_t>(p.h) * p.E * 2 : 0, 16));
  CHECK(moe::check_ptr(fn, "logits_out", a->logits_out, TE, 4));
  CHECK(moe::check_ptr(fn, "idx", a->idx, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "gate", a->gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "slot_row", a->slot_row, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "counts_routed", a->counts_routed, g->w_aux != 0.f ? static_cast<size_t>(p.E) * 4 : 0, 4));
  if (p.noisy) {
    CHECK(moe::check_ptr(fn, "W_noise", a->W_noise, p.T > 0 ? static_cast<size_t>(p.h) * p.E * 2 : 0, 16));
    CHECK(moe::check_ptr(fn, "eps", a->eps, TE, 4));
    CHECK(moe::check_ptr(fn, "dW_noise", g->dW_noise, hE, 16));
  }
  CHECK(moe::check_shared_args(fn, p, a->U, a->W_gate_shared, a->W_up_shared, a->W_down_shared, a->act_shared,
                               a->Y_shared));
  // gradients and scratch
  CHECK(moe::check_ptr(fn, "dO", g->dO, Th, 16));
  CHECK(moe::check_ptr(fn, "d_gate", g->d_gate, static_cast<size_t>(p.Tk) * 4, 4));
  CHECK(moe::check_ptr(fn, "dY", g->dY, Tkh, 16));
  CHECK(moe::check_ptr(fn, "dH", g->dH, TE, 4));
  CHECK(moe::check_ptr(fn, "d_act", g->d_act, Tkd, 16));
  CHECK(moe::check_ptr(fn, "dG", g->dG, Tkd, 16));
  CHECK(moe::check_ptr(fn, "dUp", g->dUp, Tkd, 16));
  CHECK(moe::check_ptr(fn, "dX", g->dX, Tkh, 16));
  CHECK(moe::check_ptr(fn, "dU_router", g->dU_router, Th, 16));
  CHECK(moe::check_ptr(fn, "dU", g->dU, Th, 16));
  CHECK(moe::check_ptr(fn, "dW_gate", g->dW_gate, wg, 16));
  CHECK(moe::check_ptr(fn, "dW_up", g->dW_up, wg, 16));
  CHECK(moe::check_ptr(fn, "dW_down", g->dW_down, wg, 16));
  CHECK(moe::check_ptr(fn, "dW_r", g->dW_r, hE, 16));
  CHECK(moe::check_ptr(fn, "db_r", g->db_r, 0, 4));
  if (p.n_shared > 0) {
    const size_t Td = static_cast<size_t>(p.T) * p.d_shared * es;
    const size_t wsh = p.T > 0 ? static_cast<size_t>(p.n_shared) * p.d_shared * p.h * 4 : 0;
    CHECK(moe::check_ptr(fn, "d_act_shared", g->d_act_shared, Td, 16));
    CHECK(moe::check_ptr(fn, "dG_shared", g->dG_shared, Td, 16));
    CHECK(moe::check_ptr(fn, "dUp_shared", g->dUp_shared, Td, 16));
    CHECK(moe::check_ptr(fn, "dX_shared", g->dX_shared, static_cast<size_t>(p.n_shared) * Th, 16));
    CHECK(moe::check_ptr(fn, "dW_gate_shared", g->dW_gate_shared, wsh, 16));
    CHECK(moe::check_ptr(fn, "dW_up_shared", g->dW_up_shared, wsh, 16));
    CHECK(moe::check_ptr(fn, "dW_down_shared", g->dW_down_shared, wsh, 16));
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* status = moe::ws_status(p, w);
  cudaError_t e = moe::launch_combine_backward(p, g->dO, a->Y, a->slot_row, a->gate, g->d_gate, g->dY, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/combine", e);
  e = moe::launch_route_backward(p, a->logits_out, a->idx, g->d_gate, a->counts_routed, g->w_aux, g->w_z, g->dH,
                                 stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/route", e);
  e = moe::launch_ffn_backward_tc(p, a->X, a->offsets, a->W_gate, a->W_up, a->W_down, a->act, g->dY, g->d_act, g->dG,
                                  g->dUp, g->dX, g->dW_gate, g->dW_up, g->dW_down, status, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/experts", e);
  if (p.n_shared > 0 && p.T > 0) {
    moe::Plan q = p;
    q.E = 1;
    q.k = 1;
    q.Tk = p.T;
    q.d_e = p.d_shared;
    const size_t w_in = static_cast<size_t>(p.d_shared) * p.h;
    for (int i = 0; i < p.n_shared; ++i) {
      e = moe::launch_ffn_backward_tc(
          q, a->U, nullptr, static_cast<const uint16_t*>(a->W_gate_shared) + i * w_in,
          static_cast<const uint16_t*>(a->W_up_shared) + i * w_in,
          static_cast<const uint16_t*>(a->W_down_shared) + i * w_in,
          static_cast<const uint16_t*>(a->act_shared) + static_cast<size_t>(i) * p.T * p.d_shared, g->dO,
          g->d_act_shared, g->dG_shared, g->dUp_shared,
          static_cast<uint16_t*>(g->dX_shared) + static_cast<size_t>(i) * p.T * p.h, g->dW_gate_shared + i * w_in,
          g->dW_up_shared + i * w_in, g->dW_down_shared + i * w_in, status, stream);
      if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/shared", e);
    }
  }
  e = moe::launch_router_input_backward(p, a->U, a->W_r, a->W_noise, a->eps, g->dH, g->dU_router, g->dW_r,
                                        g->dW_noise, g->db_r, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/router", e);
  e = moe::launch_dispatch_backward(p, g->dO, g->dX, a->slot_row, g->dU, w, stream, g->dU_router,
                                    p.n_shared > 0 ? g->dX_shared : nullptr, p.n_shared);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_backward/dispatch", e);
  return MOE_OK;
}

MOE_API moe_status moe_layer_forward(const moe_config* cfg, const moe_layer_args* a, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_layer_forward";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  if (!a) return moe::fail(MOE_ERR_INVALID_ARG, "%s: args is NULL", fn);
  CHECK(moe::check_route_args(fn, p, a->U, a->W_r, a->W_noise, a->eps, nullptr, a->logits_out, a->idx, a->gate, ws));
  CHECK(moe::check_ptr(fn, "b_r", a->b_r, 0, 4));
  // X == NULL: the dispatch writes no rows and the first GEMM gathers them from U (bf16)
  const bool gather = a->X == nullptr;
  if (gather && !p.bf16)
    return moe::fail(MOE_ERR_UNSUPPORTED, "%s: X == NULL (gathered up-projection) needs a bf16 config", fn);
  const void* X = gather ? a->U : a->X;  // U stands in for a missing X in the pointer checks
  CHECK(moe::check_dispatch_args(fn, p, a->U, a->idx, a->counts_routed, a->counts_kept, a->offsets, a->slot_row,
                                 a->row_token, X, a->n_dropped, ws));
  CHECK(moe::check_ffn_args(fn, p, X, a->offsets, a->W_gate, a->W_up, a->W_down, a->act, a->Y, ws));
  CHECK(moe::check_combine_args(fn, p, a->U, a->Y, a->slot_row, a->gate, a->counts_routed, a->out, a->f, a->P,
                                a->aux, ws));
  CHECK(moe::check_ptr(fn, "z_loss", a->z_loss, 0, 4));
  CHECK(moe::check_ptr(fn, "sel_bias", a->sel_bias, 0, 4));
  CHECK(moe::check_shared_args(fn, p, a->U, a->W_gate_shared, a->W_up_shared, a->W_down_shared, a->act_shared,
                               a->Y_shared));
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaError_t e = moe::launch_route(p, a->U, a->W_r, a->b_r, a->sel_bias, a->W_noise, a->eps, nullptr, a->logits_out,
                                    a->idx, a->gate, w, stream, a->W_r_packed);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward/route", e);
  e = moe::launch_dispatch(p, a->U, a->idx, a->counts_routed, a->counts_kept, a->offsets, a->slot_row, a->row_token,
                           a->X, a->n_dropped, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward/dispatch", e);
  e = gather ? moe::launch_ffn_tc(p, nullptr, a->offsets, a->W_gate, a->W_up, a->W_down, a->act, a->Y,
                                  moe::ws_status(p, w), stream, a->U, a->row_token)
             : moe::launch_expert_ffn(p, a->X, a->offsets, a->W_gate, a->W_up, a->W_down, a->act, a->Y, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward/expert_ffn", e);
  if (p.n_shared > 0) {
    e = moe::launch_shared_ffn(p, a->U, a->W_gate_shared, a->W_up_shared, a->W_down_shared, a->act_shared,
                               a->Y_shared, w, stream);
    if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward/shared_ffn", e);
  }
  e = moe::launch_combine(p, a->U, a->Y, p.n_shared > 0 ? a->Y_shared : nullptr, a->slot_row, a->gate,
                          a->counts_routed, a->out, a->f, a->P, a->aux, a->z_loss, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward/combine", e);
  return MOE_OK;
}

// ---- FP8 dispatch and up-projection ---------------------------------------------------------

namespace moe {

moe_status check_fp8(const char* fn, const Plan& p) {
  if (!p.bf16) return fail(MOE_ERR_UNSUPPORTED, "%s: the FP8 path needs a bf16 config", fn);
  if (p.h % 16 != 0) return fail(MOE_ERR_UNSUPPORTED, "%s: h = %d must be a multiple of 16", fn, p.h);
  return MOE_OK;
}

moe_status check_fp8_rows(const char* fn, const Plan& p, const uint8_t* X8, const float* x_scale) {
  CHECK(check_ptr(fn, "X8", X8, static_cast<size_t>(p.Tk) * p.h, 16));
  CHECK(check_ptr(fn, "x_scale", x_scale, static_cast<size_t>(p.Tk) * 4, 4));
  return MOE_OK;
}

moe_status check_fp8_weights(const char* fn, const Plan& p, const uint8_t* W_gate8, const uint8_t* W_up8,
                             const float* s_gate, const float* s_up, const void* W_down) {
  const size_t w = p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * p.h : 0;
  CHECK(check_ptr(fn, "W_gate8", W_gate8, w, 16));
  CHECK(check_ptr(fn, "W_up8", W_up8, w, 16));
  CHECK(check_ptr(fn, "s_gate", s_gate, p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * 4 : 0, 4));
  CHECK(check_ptr(fn, "s_up", s_up, p.Tk > 0 ? static_cast<size_t>(p.E) * p.d_e * 4 : 0, 4));
  CHECK(check_ptr(fn, "W_down", W_down, w * 2, 16));
  return MOE_OK;
}

}  // namespace moe

MOE_API moe_status moe_quantize_fp8(int64_t rows, int32_t cols, const void* src, uint8_t* dst, float* scale,
                                    moe_stream_t stream) {
  static const char* fn = "moe_quantize_fp8";
  if (rows < 0 || cols < 1) return moe::fail(MOE_ERR_INVALID_ARG, "%s: rows = %lld, cols = %d", fn,
                                             static_cast<long long>(rows), cols);
  if (cols % 8 != 0) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: cols = %d must be a multiple of 8", fn, cols);
  if (rows >= (int64_t(1) << 40) / cols) return moe::fail(MOE_ERR_UNSUPPORTED, "%s: rows * cols too large", fn);
  const size_t n = static_cast<size_t>(rows) * cols;
  CHECK(moe::check_ptr(fn, "src", src, n * 2, 16));
  CHECK(moe::check_ptr(fn, "dst", dst, n, 8));
  CHECK(moe::check_ptr(fn, "scale", scale, static_cast<size_t>(rows) * 4, 4));
  const cudaError_t e = moe::launch_quantize_fp8(rows, cols, src, dst, scale, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_dispatch_fp8(const moe_config* cfg, const void* U, const int32_t* idx,
                                    int32_t* counts_routed, int32_t* counts_kept, int32_t* offsets,
                                    int32_t* slot_row, int32_t* row_token, uint8_t* X8, float* x_scale,
                                    int64_t* n_dropped, void* ws, moe_stream_t stream) {
  static const char* fn = "moe_dispatch_fp8";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_fp8(fn, p));
  // X is replaced by X8: check the rest with U standing in for it
  CHECK(moe::check_dispatch_args(fn, p, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, U,
                                 n_dropped, ws));
  CHECK(moe::check_fp8_rows(fn, p, X8, x_scale));
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaError_t e = moe::launch_dispatch(p, U, idx, counts_routed, counts_kept, offsets, slot_row, row_token, nullptr,
                                       n_dropped, w, stream);
  if (e == cudaSuccess) e = moe::launch_scatter_fp8(p, U, slot_row, X8, x_scale, stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_expert_ffn_fp8(const moe_config* cfg, const uint8_t* X8, const float* x_scale,
                                      const int32_t* offsets, const uint8_t* W_gate8, const uint8_t* W_up8,
                                      const float* s_gate, const float* s_up, const void* W_down, void* act, void* Y,
                                      void* ws, moe_stream_t stream) {
  static const char* fn = "moe_expert_ffn_fp8";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_fp8(fn, p));
  CHECK(moe::check_fp8_rows(fn, p, X8, x_scale));
  CHECK(moe::check_fp8_weights(fn, p, W_gate8, W_up8, s_gate, s_up, W_down));
  CHECK(moe::check_ptr(fn, "offsets", offsets, static_cast<size_t>(p.E + 1) * 4, 4));
  CHECK(moe::check_ptr(fn, "act", act, static_cast<size_t>(p.Tk) * p.d_e * 2, 16));
  CHECK(moe::check_ptr(fn, "Y", Y, static_cast<size_t>(p.Tk) * p.h * 2, 16));
  CHECK(moe::check_ptr(fn, "ws", ws, p.ws_total, 256));
  uint8_t* w = static_cast<uint8_t*>(ws);
  const cudaError_t e = moe::launch_ffn_fp8_tc(p, X8, x_scale, offsets, W_gate8, W_up8, s_gate, s_up, W_down, act,
                                               Y, moe::ws_status(p, w), stream);
  return e == cudaSuccess ? MOE_OK : moe::cuda_fail(fn, e);
}

MOE_API moe_status moe_layer_forward_fp8(const moe_config* cfg, const moe_layer_args* a, const moe_fp8_args* f8,
                                         void* ws, moe_stream_t stream) {
  static const char* fn = "moe_layer_forward_fp8";
  Plan p;
  CHECK(moe::plan_or_fail(fn, cfg, &p));
  CHECK(moe::check_fp8(fn, p));
  if (!a || !f8) return moe::fail(MOE_ERR_INVALID_ARG, "%s: args or fp8 args is NULL", fn);
  CHECK(moe::check_route_args(fn, p, a->U, a->W_r, a->W_noise, a->eps, nullptr, a->logits_out, a->idx, a->gate, ws));
  CHECK(moe::check_ptr(fn, "b_r", a->b_r, 0, 4));
  CHECK(moe::check_dispatch_args(fn, p, a->U, a->idx, a->counts_routed, a->counts_kept, a->offsets, a->slot_row,
                                 a->row_token, a->U, a->n_dropped, ws));
  CHECK(moe::check_fp8_rows(fn, p, f8->X8, f8->x_scale));
  CHECK(moe::check_fp8_weights(fn, p, f8->W_gate8, f8->W_up8, f8->s_gate, f8->s_up, a->W_down));
  CHECK(moe::check_ptr(fn, "act", a->act, static_cast<size_t>(p.Tk) * p.d_e * 2, 16));
  CHECK(moe::check_combine_args(fn, p, a->U, a->Y, a->slot_row, a->gate, a->counts_routed, a->out, a->f, a->P,
                                a->aux, ws));
  CHECK(moe::check_ptr(fn, "z_loss", a->z_loss, 0, 4));
  CHECK(moe::check_ptr(fn, "sel_bias", a->sel_bias, 0, 4));
  CHECK(moe::check_shared_args(fn, p, a->U, a->W_gate_shared, a->W_up_shared, a->W_down_shared, a->act_shared,
                               a->Y_shared));
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaError_t e = moe::launch_route(p, a->U, a->W_r, a->b_r, a->sel_bias, a->W_noise, a->eps, nullptr, a->logits_out,
                                    a->idx, a->gate, w, stream, a->W_r_packed);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward_fp8/route", e);
  e = moe::launch_dispatch(p, a->U, a->idx, a->counts_routed, a->counts_kept, a->offsets, a->slot_row, a->row_token,
                           nullptr, a->n_dropped, w, stream);
  if (e == cudaSuccess) e = moe::launch_scatter_fp8(p, a->U, a->slot_row, f8->X8, f8->x_scale, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward_fp8/dispatch", e);
  e = moe::launch_ffn_fp8_tc(p, f8->X8, f8->x_scale, a->offsets, f8->W_gate8, f8->W_up8, f8->s_gate, f8->s_up,
                             a->W_down, a->act, a->Y, moe::ws_status(p, w), stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward_fp8/expert_ffn", e);
  if (p.n_shared > 0) {
    e = moe::launch_shared_ffn(p, a->U, a->W_gate_shared, a->W_up_shared, a->W_down_shared, a->act_shared,
                               a->Y_shared, w, stream);
    if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward_fp8/shared_ffn", e);
  }
  e = moe::launch_combine(p, a->U, a->Y, p.n_shared > 0 ? a->Y_shared : nullptr, a->slot_row, a->gate,
                          a->counts_routed, a->out, a->f, a->P, a->aux, a->z_loss, w, stream);
  if (e != cudaSuccess) return moe::cuda_fail("moe_layer_forward_fp8/combine", e);
  return MOE_OK;
}

MOE_API moe_status moe_get_device_status(void* ws, moe_stream_t stream, int32_t* code) {
  static const char* fn = "moe_get_device_status";
  if (!ws || !moe::aligned(ws, 256)) return moe::fail(MOE_ERR_INVALID_ARG, "%s: ws is NULL or misaligned", fn);
  if (!code) return moe::fail(MOE_ERR_INVALID_ARG, "%s: code is NULL", fn);
  int32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess && h != 0) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return moe::cuda_fail(fn, e);
  *code = h;
  if (h != 0) return moe::fail(MOE_ERR_DEVICE, "%s: device status %d", fn, h);
  return MOE_OK;
}
