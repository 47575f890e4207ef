// Internal launch interface of libmoe (not exported).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Tile constants shared by the launch plan and the kernels.
constexpr int route_bt_for(int ep) { return ep <= 256 ? 32 : 8192 / ep; }  // tokens per partial-logits block
constexpr int route_kc_for(int ep) { return ep <= 128 ? 64 : 8192 / ep; }  // h chunk per pipeline stage
// The router's selection kernel: G lanes per token, each with a chunk of <= 32 experts
// (G = E / 32 rounded up to a power of two); blocks of up to SELECT_THREADS threads.
constexpr int SELECT_THREADS = 256;
constexpr int select_lanes_for(int E) {
  return E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : E <= 256 ? 8 : E <= 512 ? 16 : 32;
}
// Odd stride of one lane's chunk of C = ceil(E / G) logits in the select block's shared memory.
constexpr int select_chunk_stride(int E) {
  return (((E + select_lanes_for(E) - 1) / select_lanes_for(E)) & 1)
             ? (E + select_lanes_for(E) - 1) / select_lanes_for(E) + 2
             : (E + select_lanes_for(E) - 1) / select_lanes_for(E) + 1;
}
// Shared memory of a select block of `tokens` tokens: [tokens][G * CS] logits, one z value each,
// then (group-limited routing) [tokens][n_group] group scores.
constexpr size_t select_smem_bytes(int E, int tokens, int n_group = 0) {
  return sizeof(float) * static_cast<size_t>(tokens) *
         (select_lanes_for(E) * select_chunk_stride(E) + 1 + (n_group > 1 ? n_group : 0));
}
constexpr int MAX_GROUPS = 32;  // group-limited routing: kept groups fit one 32-bit mask

constexpr int kDispatchChunk = 4096;  // largest number of priority positions per dispatch chunk

// Sizes derived from one moe_config, and the carve-up of the workspace.
struct Plan {
  int64_t T = 0;
  int h = 0, E = 0, k = 0, d_e = 0;
  int64_t C = 0;           // expert capacity
  int64_t Tk = 0;          // T * k = rows of the capacity buffers X, act, Y
  bool bf16 = false;
  bool noisy = false;
  int score_fn = 0, renorm = 0, priority = 0;
  int n_shared = 0, d_shared = 0;  // shared experts and their intermediate size
  int n_group = 0, topk_group = 0; // group-limited routing (n_group > 1), else 0

  // router
  int route_ep = 0;        // E rounded up to the router's compile-time width
  int route_bt = 0;        // tokens per partial-logits block
  int route_kc = 0;        // K chunk of the partial-logits block
  int route_rowblocks = 0; // ceil(T / route_bt)
  int route_splits = 0;    // split of h across blocks (summed in fixed order by the select kernel)
  int route_tc_n = 0;      // > 0: bf16 logits on the tensor cores with this MMA width (E or 2E rounded up to 16)
  bool route_fused = false;// the fused router (route_tc.cu): logits, scores, top-k and gates in one kernel
  int rf_tiles = 0;        // its 128-token tiles
  int rf_cs = 0;           // CTAs per tile (a cluster), each with a slice of h
  int rf_stages = 0;       // its TMA ring depth
  int rf_threads = 256;    // threads a CTA: 512 when one CTA fills an SM anyway (more warps to select)
  int sel_threads = 0;     // threads per select block (G lanes per token)
  int sel_tokens = 0;      // tokens per select block
  int sel_blocks = 0;      // ceil(T / sel_tokens): number of P partial rows

  // dispatch
  int chunk = 0;           // priority positions per histogram chunk (token-major priority)
  int n_chunks = 0;
  int dp_tc = 0;           // tokens per chunk of the choice-major dispatch (8 .. 256)
  int dp_chunks = 0;

  // workspace byte offsets
  size_t ws_status = 0, ws_part = 0, ws_npart = 0, ws_ppart = 0, ws_hist = 0, ws_wt = 0, ws_total = 0;
  size_t ws_stats2 = 0;    // first-level partial sums of the statistics [32][E + 1] f32
  // router backward: [dH | dN] bf16 [T, rb_np], [W_r | W_noise] bf16 [h, rb_np], dW float32 [h, rb_np]
  int rb_np = 0;
  size_t ws_rb_dh = 0, ws_rb_w = 0, ws_rb_dw = 0;
};

// Validates the config and fills `plan`; on failure returns the status and a message.
moe_status make_plan(const moe_config* cfg, Plan* plan, const char** msg);

// W_r_packed: the router weights from launch_pack_router (NULL: packed into the workspace on each
// call when the fused router runs).
cudaError_t launch_route(const Plan& p, const void* U, const void* W_r, const float* b_r, const float* sel_bias,
                         const void* W_noise, const float* eps, const float* logits_in, float* logits_out,
                         int32_t* idx, float* gate, uint8_t* ws, cudaStream_t s, const void* W_r_packed = nullptr);

// Router weights for the tensor cores: Wt [route_tc_n, h] bf16, K-major (W_r transposed, W_noise
// transposed below it, zero rows up to route_tc_n).
cudaError_t launch_pack_router(const Plan& p, const void* W_r, const void* W_noise, void* Wt, cudaStream_t s);
// The fused router (bf16, route_tc_n > 0) from packed weights Wt.
cudaError_t launch_route_fused(const Plan& p, const void* U, const void* Wt, const float* b_r, const float* sel_bias,
                               const float* eps, float* logits_out, int32_t* idx, float* gate, uint8_t* ws,
                               cudaStream_t s);

// Router slice sums U W_r (and U W_noise) on the tensor cores (bf16, p.route_tc_n > 0).
cudaError_t launch_route_logits_tc(const Plan& p, const void* U, const void* W_r, const void* W_noise, float* part,
                                   float* npart, uint8_t* ws, cudaStream_t s);

cudaError_t launch_dispatch(const Plan& p, const void* U, const int32_t* idx, int32_t* counts_routed,
                            int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token, void* X,
                            int64_t* n_dropped, uint8_t* ws, cudaStream_t s);

// moe_dispatch with the histogram in the library's static device array (no workspace);
// status (nullable) is zeroed, then receives MOE_DEV_* codes.
cudaError_t launch_dispatch_noalloc(const Plan& p, const void* U, const int32_t* idx, int32_t* counts_routed,
                                    int32_t* counts_kept, int32_t* offsets, int32_t* slot_row, int32_t* row_token,
                                    void* X, int64_t* n_dropped, int32_t* status, cudaStream_t s);

cudaError_t launch_expert_ffn(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                              const void* W_up, const void* W_down, void* act, void* Y, uint8_t* ws, cudaStream_t s);

cudaError_t launch_combine(const Plan& p, const void* U, const void* Y, const void* Y_shared, const int32_t* slot_row,
                           const float* gate, const int32_t* counts_routed, void* out, float* f, float* P, float* aux,
                           float* z_loss, uint8_t* ws, cudaStream_t s);

// Every shared expert's SwiGLU FFN on all T tokens: Y_sh[s] = FFN_s(U) (act_sh is scratch).
cudaError_t launch_shared_ffn(const Plan& p, const void* U, const void* W_gate_sh, const void* W_up_sh,
                              const void* W_down_sh, void* act_sh, void* Y_sh, uint8_t* ws, cudaStream_t s);

// Backward of the combine: d_gate [T, k] = dO_t . Y[row], dY[row] = g dO_t.
cudaError_t launch_combine_backward(const Plan& p, const void* dO, const void* Y, const int32_t* slot_row,
                                    const float* gate, float* d_gate, void* dY, uint8_t* ws, cudaStream_t s);
// Backward of the gates, the aux loss and the z-loss to the router logits: dH [T, E].
cudaError_t launch_route_backward(const Plan& p, const float* logits, const int32_t* idx, const float* d_gate,
                                  const int32_t* counts_routed, float w_aux, float w_z, float* dH, cudaStream_t s);

// Backward of the grouped bf16 SwiGLU experts (tcgen05): d_act, dG, dUp, dX and float32 weight gradients.
cudaError_t launch_ffn_backward_tc(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                                   const void* W_up, const void* W_down, const void* act, const void* dY,
                                   void* d_act, void* dG, void* dUp, void* dX, float* dW_gate, float* dW_up,
                                   float* dW_down, int32_t* status, cudaStream_t s);
// out[rows, N] = A[rows, K] B[N, K]^T in bf16 on tcgen05 (one all-row segment).
cudaError_t launch_dense_gemm_tc(const void* A, int64_t rows, int K, const void* B, int N, void* out, int32_t* status,
                                 cudaStream_t s);
// out[M, N] (float32) = A^T B over `rows` rows (A [rows, M], B [rows, N] bf16) on tcgen05.
cudaError_t launch_dense_wgrad_tc(const void* A, const void* B, int64_t rows, int M, int N, float* out,
                                  int32_t* status, cudaStream_t s);
// Backward of the router linear (bf16): dU_r = [dH | dN] [W_r | W_noise]^T, dW_r, dW_noise, db_r.
cudaError_t launch_router_input_backward(const Plan& p, const void* U, const void* W_r, const void* W_noise,
                                         const float* eps, const float* dH, void* dU_r, float* dW_r, float* dW_noise,
                                         float* db_r, uint8_t* ws, cudaStream_t s);

// dU = dO + the dX rows of each token's kept pairs.
// (+ extra [T, h] and n_more further [T, h] blocks at `more`, each nullable)
cudaError_t launch_dispatch_backward(const Plan& p, const void* dO, const void* dX, const int32_t* slot_row, void* dU,
                                     uint8_t* ws, cudaStream_t s, const void* extra = nullptr,
                                     const void* more = nullptr, int n_more = 0);

// b_i += u * sign(mean(counts) - counts_i) for the loss-free balancing bias.
cudaError_t launch_balance_bias_update(int E, const int32_t* counts_routed, float u, float* bias, cudaStream_t s);

// Grouped bf16 GEMMs on tcgen05 (both FFN halves); returns cudaErrorNotSupported when the
// tensor maps cannot be built.
// gather_rows != NULL: X is not read; the first GEMM gathers row r of its A operand from
// gather_src[gather_rows[r]] ([T, h], the dispatch's row copy fused in).
cudaError_t launch_ffn_tc(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                          const void* W_up, const void* W_down, void* act, void* Y, int32_t* status,
                          cudaStream_t s, const void* gather_src = nullptr, const int32_t* gather_rows = nullptr);
cudaError_t launch_ffn_fp8_tc(const Plan& p, const uint8_t* X8, const float* x_scale, const int32_t* offsets,
                              const uint8_t* W_gate8, const uint8_t* W_up8, const float* s_gate, const float* s_up,
                              const void* W_down, void* act, void* Y, int32_t* status, cudaStream_t s);
cudaError_t launch_quantize_fp8(int64_t rows, int cols, const void* src, uint8_t* dst, float* scale, cudaStream_t s);
cudaError_t launch_scatter_fp8(const Plan& p, const void* U, const int32_t* slot_row, uint8_t* X8, float* x_scale,
                               cudaStream_t s);
cudaError_t launch_ffn_simt_f32(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                                const void* W_up, const void* W_down, void* act, void* Y, int32_t* status,
                                cudaStream_t s);

inline int32_t* ws_status(const Plan& p, uint8_t* ws) { return reinterpret_cast<int32_t*>(ws + p.ws_status); }
// Rows of per-block score sums the last router call left in the workspace (read by the statistics).
inline int32_t* ws_ppart_rows(const Plan& p, uint8_t* ws) {
  return reinterpret_cast<int32_t*>(ws + p.ws_status + 64);
}

// Streaming multiprocessors of the current device (148 on B300 if the query fails).
inline int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    return 148;
  return n;
}

}  // namespace moe
