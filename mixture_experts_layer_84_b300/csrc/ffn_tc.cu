// Grouped bf16 SwiGLU expert FFN on the 5th-generation tensor cores.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 从稠密 FFN 到 MoE:
// FFN(u) = W_down (SiLU(W_gate u) ⊙ W_up u); section 专家计算：padding、
// block-sparse 与 grouped GEMM: one launch runs the GEMMs of every expert over
// its own variable-length segment, scheduled tile by tile inside the kernel
// from the per-expert offsets; gate and up form one [h, 2 d_e] product,
// followed by the elementwise SiLU * up, then the down GEMM.
//
// Kernel (one persistent CTA per SM, 192 threads):
//   warp 0    TMA producer: 4-stage ring of {X tile 128x64, W tile 256x64}
//             (bf16, 128-byte swizzle; or X rows by four-row TMA gathers),
//             completion counted on mbarriers;
//   warp 1    allocates 512 tensor-memory columns (two 128x256 f32
//             accumulators) and one lane issues tcgen05.mma 128x256x16,
//             releasing smem stages and finished accumulators with
//             tcgen05.commit;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator (TMEM lane = tile row),
//             SiLU(gate) * up (first GEMM) or plain (second), bf16 rounding,
//             masked stores of the rows inside the expert segment.
// Gate|up fusion: a B stage holds 128 rows of W_gate[e] followed by the same
// 128 rows of W_up[e], so accumulator columns c and 128+c are the gate and up
// values of output column c; no repacking of the weights is needed.
// Tile order: expert by expert; inside an expert either row tiles vary fastest
// (the CTAs that run together share a weight tile, and the expert's rows are
// re-read once per column tile) or column tiles do (they share a row tile, and
// the expert's weights are re-read once per row tile), whichever re-reads the
// smaller operand; that operand gets the evict_last L2 hint.
// Every mbarrier wait is bounded (2 s); a wait that gives up makes every role
// leave its loop, in-flight copies and MMAs are drained (again bounded), the
// tensor memory is freed and MOE_DEV_TIMEOUT is recorded in the status word.
#include <cuda.h>

#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                       // tile rows = TMEM lanes
constexpr int BN = 256;                       // MMA N = B rows per stage
constexpr int BK = 64;                        // K per stage (one 128-byte swizzle row of bf16)
constexpr int UK = 16;                        // K per tcgen05.mma kind::f16
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;     // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;     // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t ACC_COLS = 256;            // f32 columns of one 128 x 256 accumulator
constexpr uint32_t TMEM_COLS = 512;           // two accumulators
constexpr int THREADS = 192;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_E = 1024;
constexpr size_t BAR_BYTES = 128;             // 13 mbarriers + tmem address + flags
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + sizeof(int) * (MAX_E + 1);
static_assert(SMEM_BYTES <= 232448, "shared memory");

// Bytes from the start of the dynamic shared array to its first 1024-byte aligned address (what
// the 128-byte swizzle and the TMA boxes need).  The aligned base is taken as an offset from the
// array rather than by rounding the pointer as an integer, so that the compiler can keep every
// access through it in the shared state space (measured: 0.6-5% faster grouped GEMMs).
__device__ __forceinline__ uint32_t aligned_1024(const uint8_t* smem_raw) {
  return (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
}

// Tile `tile` of the list ordered expert by expert; inside an expert, row tiles vary fastest (the
// CTAs running together share a B tile, and the A segment is re-read once per column tile), or with
// cols_fastest the column tiles do (they share an A row tile, and the expert's B is re-read once per
// row tile): the host picks whichever re-reads the smaller operand.
__device__ __forceinline__ void decode_tile(const int* tab, int E, int NT, int tile, int* e, int* nt, int* mt,
                                            int cols_fastest = 0) {
  int lo = 0, hi = E;  // tab[lo]*NT <= tile < tab[hi]*NT
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid] * NT <= tile)
      lo = mid;
    else
      hi = mid;
  }
  const int m_e = tab[lo + 1] - tab[lo];
  const int local = tile - tab[lo] * NT;
  *e = lo;
  if (cols_fastest) {
    *mt = local / NT;
    *nt = local - (*mt) * NT;
  } else {
    *nt = local / m_e;
    *mt = local - (*nt) * m_e;
  }
}

// L2 hints of the two operands for tile schedule `sched` (bit 0: column tiles fastest; bits 1-2: 0 keeps
// the operand that later tiles read again (evict_last), 1 gives no hint, 2 also marks the operand
// read once evict_first)
__device__ __forceinline__ void l2_policies(int sched, uint64_t* pol_a, uint64_t* pol_b) {
  const bool cols = sched & 1;
  const int mode = (sched >> 1) & 3;
  const uint64_t keep = mode == 0 ? ptx::policy_evict_last() : ptx::policy_evict_normal();
  const uint64_t once = mode == 2 ? ptx::policy_evict_first() : ptx::policy_evict_normal();
  *pol_a = cols ? once : keep;
  *pol_b = cols ? keep : once;
}

// Wait without regard to the abort flag (drains in-flight work before exit).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
  return true;
}

// SiLU(g) * u = g u / (1 + e^-g) with the fast exponential and division intrinsics: their
// relative error (a few float32 ulps) is far below the bf16 rounding of the result, and the
// epilogue must keep up with short (16 k-block) tiles; e^-g = inf gives 0, SiLU's limit.
__device__ __forceinline__ float silu_mul(float g, float u) { return __fdividef(g * u, 1.f + __expf(-g)); }

__device__ __forceinline__ void store_32(bf16* orow, int col0, int n_out, const uint32_t* packed) {
  if (col0 + 32 <= n_out) {
    uint4* d = reinterpret_cast<uint4*>(orow + col0);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
  } else {
    // the ragged end of a row: element by element, register indices only (no local copy)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = col0 + 2 * i;
      if (c < n_out) orow[c] = __ushort_as_bfloat16(static_cast<unsigned short>(packed[i] & 0xffffu));
      if (c + 1 < n_out) orow[c + 1] = __ushort_as_bfloat16(static_cast<unsigned short>(packed[i] >> 16));
    }
  }
}

// ---- gathered A operand (the dispatch's row copy fused into the first GEMM) -------------------
// Row r of the A operand is row tok[r] of the source ([rows, K] bf16, read through a tensor map
// whose box is one row of 64 columns).  The producer warp loads a 128-row stage with 32 four-row
// TMA gathers: lane L brings tile rows 4L..4L+3 into bytes [512 L, 512 L + 512) of the stage.  The
// 128-byte swizzle follows the shared-memory address, so the stage ends up exactly as one tiled
// load of 128 consecutive rows would leave it, and the MMA descriptors are unchanged.
struct Gather {
  const int32_t* tok;  // source row of every A row
  int64_t rows;        // rows of the source
};

// the source rows of A rows first_row .. first_row + 3 (rows past the kept rows, or ids out of
// range, read row 0; their results are never stored)
__device__ __forceinline__ int4 gather_rows4(const Gather& g, int64_t first_row, int64_t a_total, int32_t* status) {
  int32_t t[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t[i] = 0;
    if (first_row + i < a_total) {
      const int32_t v = g.tok[first_row + i];
      if (v < 0 || v >= g.rows)
        set_status(status, MOE_DEV_BAD_ROW);
      else
        t[i] = v;
    }
  }
  return make_int4(t[0], t[1], t[2], t[3]);
}

// SWIGLU: out[row, c] = SiLU(A W0^T)[row, c] * (A W1^T)[row, c], c < n_out (= d_e), W0/W1 rows per expert = d_e.
// plain:  out[row, c] = (A W0^T)[row, c],                         c < n_out (= h),   W0 rows per expert = h.
// FP8 (SwiGLU only): A, W0, W1 are E4M3 codes (kind::f8f6f4, 128 K-elements per 128-byte stage row), and
// each product is scaled back by a_scale[row] * b_scale[weight row] (powers of two) before SiLU * up.
// GATHER (SwiGLU, bf16): the A operand is gathered from g (the dispatch's row copy fused in).
template <bool SWIGLU, bool FP8 = false, bool GATHER = false>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const int32_t* __restrict__ offsets, int E, int K,
                    int b_rows_per_expert, int n_out, int64_t rows_cap, bf16* __restrict__ out, int32_t* status,
                    const float* __restrict__ a_scale = nullptr, const float* __restrict__ b0_scale = nullptr,
                    const float* __restrict__ b1_scale = nullptr, Gather g = Gather{}, int sched = 0) {
  static_assert(SWIGLU || !FP8, "the FP8 path is the up-projection");
  static_assert(!(GATHER && (FP8 || !SWIGLU)), "the gathered A operand is the bf16 up-projection's");
  constexpr int TILE_N = SWIGLU ? BN / 2 : BN;  // output columns per tile
  constexpr int BKE = FP8 ? 2 * BK : BK;        // K elements per stage (128 bytes of every row)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + aligned_1024(smem_raw);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_holder + 2);
  int* tab = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = (n_out + TILE_N - 1) / TILE_N;
  const int KB = (K + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
  }
  __syncthreads();
  // every CTA checks every segment before anything is written
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
    int m = 0;
    if (lo < 0 || hi < lo || static_cast<int64_t>(hi) > rows_cap)
      *bad_flag = 1;
    else
      m = (hi - lo + BM - 1) / BM;
    tab[e + 1] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    tab[0] = 0;
    for (int e = 0; e < E; ++e) tab[e + 1] += tab[e];
    if (*bad_flag && blockIdx.x == 0) set_status(status, MOE_DEV_BAD_OFFSETS);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 4);
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();
  if (*bad_flag) return;
  const int total = tab[E] * NT;
  if (static_cast<int>(blockIdx.x) >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (GATHER && warp == 0) {
    // the whole warp loads A (four rows a lane), lane 0 also the B tiles
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB0);
      ptx::prefetch_tmap(&tmB1);
    }
    uint64_t pol_a, pol_b;  // the operand that later tiles read again is kept in L2
    l2_policies(sched, &pol_a, &pol_b);
    const int64_t a_total = seg_hi(offsets, E - 1, rows_cap);
    uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int e, nt, mt;
      decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
      const int4 rows = gather_rows4(g, static_cast<int64_t>(seg_lo(offsets, e)) + mt * BM + 4 * lane, a_total, status);
      const int b_row = e * b_rows_per_expert + nt * TILE_N;
      for (int kb = 0; kb < KB; ++kb) {
        const bool got = ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint8_t* sa = stages + stage * STAGE_BYTES;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          ptx::tma_load_2d(sa + A_BYTES, &tmB0, kb * BK, b_row, &full[stage], pol_b);
          ptx::tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tmB1, kb * BK, b_row, &full[stage], pol_b);
        }
        __syncwarp();
        ptx::tma_gather4(sa + lane * 512, &tmA, kb * BK, rows.x, rows.y, rows.z, rows.w, &full[stage], pol_a);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // every copy this warp started has landed before the block may exit
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&full[s], (armed_phase >> s) & 1u);
    __syncwarp();
  } else if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB0);
      if (SWIGLU) ptx::prefetch_tmap(&tmB1);
      uint64_t pol_a, pol_b;  // the operand that later tiles read again is kept in L2
      l2_policies(sched, &pol_a, &pol_b);
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, nt, mt;
        decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
        const int a_row = seg_lo(offsets, e) + mt * BM;
        const int b_row = e * b_rows_per_expert + nt * TILE_N;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + stage * STAGE_BYTES;
          ptx::mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          ptx::tma_load_2d(sa, &tmA, kb * BKE, a_row, &full[stage], pol_a);
          if (SWIGLU) {
            ptx::tma_load_2d(sa + A_BYTES, &tmB0, kb * BKE, b_row, &full[stage], pol_b);
            ptx::tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tmB1, kb * BKE, b_row, &full[stage], pol_b);
          } else {
            ptx::tma_load_2d(sa + A_BYTES, &tmB0, kb * BKE, b_row, &full[stage], pol_b);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every copy this thread started has landed before the block may exit
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) mbar_wait_drain(&full[s], (armed_phase >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = FP8 ? ptx::idesc_e4m3_f32(BM, BN) : ptx::idesc_bf16_f32(BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!ptx::mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&full[stage], phase, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stages + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          // 32 bytes of K per MMA: 16 bf16 (kind::f16) or 32 E4M3 (kind::f8f6f4)
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            if (FP8)
              ptx::mma_f8_ss(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * 32), ptx::sdesc_kmajor_sw128(sb + kk * 32), IDESC,
                             (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::mma_bf16_ss(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * 32), ptx::sdesc_kmajor_sw128(sb + kk * 32),
                               IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&empty[stage]);  // stage is free once these MMAs have read it
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);  // accumulator complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit(drain);  // every MMA issued above has completed once this arrives
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const int r_local = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, nt, mt;
      decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
      const int seg = seg_lo(offsets, e);
      const int n_e = seg_hi(offsets, e, rows_cap) - seg;
      const bool row_ok = mt * BM + r_local < n_e;
      const int64_t row = static_cast<int64_t>(seg) + mt * BM + r_local;
      // the tcgen05.ld below is warp-collective: the warp leaves together or not at all
      const bool ready = ptx::mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, WAIT_LIMIT_NS);
      if (!__all_sync(0xffffffffu, ready)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      bf16* orow = out + row * n_out;
      if (SWIGLU) {
        const float xs = (FP8 && row_ok) ? a_scale[row] : 1.f;
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gv[32], uv[32], packed[16];
          ptx::tmem_ld_32x32b_x32(tb + c, gv);
          ptx::tmem_ld_32x32b_x32(tb + BN / 2 + c, uv);
          // FP8: lane i holds the scales of output column c + i (shared by every row)
          float my_sg = 1.f, my_su = 1.f;
          if (FP8) {
            const int col = nt * TILE_N + c + lane;
            const int64_t wrow = static_cast<int64_t>(e) * b_rows_per_expert + col;
            my_sg = col < n_out ? b0_scale[wrow] : 0.f;
            my_su = col < n_out ? b1_scale[wrow] : 0.f;
          }
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float g0 = __uint_as_float(gv[2 * i]), u0 = __uint_as_float(uv[2 * i]);
            float g1 = __uint_as_float(gv[2 * i + 1]), u1 = __uint_as_float(uv[2 * i + 1]);
            if (FP8) {
              g0 *= xs * __shfl_sync(0xffffffffu, my_sg, 2 * i);
              u0 *= xs * __shfl_sync(0xffffffffu, my_su, 2 * i);
              g1 *= xs * __shfl_sync(0xffffffffu, my_sg, 2 * i + 1);
              u1 *= xs * __shfl_sync(0xffffffffu, my_su, 2 * i + 1);
            }
            packed[i] = Vec16<bf16>::pack2(silu_mul(g0, u0), silu_mul(g1, u1));
          }
          if (row_ok) store_32(orow, nt * TILE_N + c, n_out, packed);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32], packed[16];
          ptx::tmem_ld_32x32b_x32(tb + c, v);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = Vec16<bf16>::pack2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          if (row_ok) store_32(orow, nt * TILE_N + c, n_out, packed);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) set_status(status, MOE_DEV_TIMEOUT);
}

// ---------------------------------------------------------------------------
// The same grouped GEMM on CTA pairs (cta_group::2): a cluster of two CTAs
// computes a 256-row tile; each CTA stages its own 128 rows of A and one half
// of the 256 B rows, so every stage is 32 KB per CTA instead of 48 KB, and the
// shared-memory traffic per tensor-core cycle drops by a third.  The even CTA
// issues the 256 x 256 x 16 MMAs for both; each CTA's tensor memory holds the
// fp32 accumulator of its own 128 rows.  For the SwiGLU half the even CTA
// stages the W_gate rows and the odd CTA the matching W_up rows, so
// accumulator columns c and 128 + c are again gate and up of column c.
//   full[s]   (even CTA) both CTAs' TMA bytes of stage s have landed
//   empty[s]  (both)     the MMAs that read stage s are done (multicast commit)
//   tfull[a]  (both)     accumulator a is complete (multicast commit)
//   tempty[a] (even CTA) the 8 epilogue warps of the pair have read accumulator a
constexpr int P_BM = 256;                        // rows per pair tile
constexpr int P_STAGES = 6;
constexpr uint32_t P_A_BYTES = 128 * BK * 2;     // 16 KB: this CTA's 128 rows
constexpr uint32_t P_B_BYTES = 128 * BK * 2;     // 16 KB: this CTA's half of the 256 B rows
constexpr uint32_t P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr size_t P_BAR_BYTES = 256;           // 17 mbarriers + tmem address + flags
// output staging: one 32-row x 64-column bf16 block (4 KB, 128-byte swizzle) per epilogue warp
constexpr size_t P_OUT_OFF = (P_STAGES * P_STAGE_BYTES + P_BAR_BYTES + sizeof(int) * (MAX_E + 1) + 1023) / 1024 * 1024;
constexpr uint32_t P_OUT_BYTES = 32 * 64 * 2;
constexpr size_t P_SMEM_BYTES = 1024 + P_OUT_OFF + 4 * P_OUT_BYTES;
static_assert(P_SMEM_BYTES <= 232448, "shared memory");
static_assert((2 * P_STAGES + 2 + 2 + 1) * 8 + 12 <= P_BAR_BYTES, "barriers fit P_BAR_BYTES");

__device__ __forceinline__ bool wait_cluster_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// GATHER (SwiGLU): each CTA gathers its 128 A rows (row ids from g) through tmA, whose box is one row.
template <bool SWIGLU, bool GATHER = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    grouped_gemm_tc_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmOut,
                         const int32_t* __restrict__ offsets, int E, int K,
                         int b_rows_per_expert, int n_out, int64_t rows_cap, bf16* __restrict__ out,
                         int32_t* status, Gather g = Gather{}, int sched = 0) {
  static_assert(SWIGLU || !GATHER, "the gathered A operand is the up-projection's");
  constexpr int TILE_N = SWIGLU ? BN / 2 : BN;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + aligned_1024(smem_raw);
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P_STAGES * P_STAGE_BYTES);
  uint64_t* empty = full + P_STAGES;
  uint64_t* tfull = empty + P_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_holder + 2);
  int* tab = reinterpret_cast<int*>(smem + P_STAGES * P_STAGE_BYTES + P_BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool even = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  const int NT = (n_out + TILE_N - 1) / TILE_N;
  const int KB = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
  }
  __syncthreads();
  // both CTAs of a pair read the same offsets and reach the same decisions below
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
    int m = 0;
    if (lo < 0 || hi < lo || static_cast<int64_t>(hi) > rows_cap)
      *bad_flag = 1;
    else
      m = (hi - lo + P_BM - 1) / P_BM;
    tab[e + 1] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    tab[0] = 0;
    for (int e = 0; e < E; ++e) tab[e + 1] += tab[e];
    if (*bad_flag && blockIdx.x == 0) set_status(status, MOE_DEV_BAD_OFFSETS);
    for (int s = 0; s < P_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 8);
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbarrier_init();
  }
  __syncthreads();
  if (*bad_flag) return;
  const int total = tab[E] * NT;
  if (cid >= total) return;
  // the peer's barriers must be initialised before anything can arrive on them
  ptx::cluster_sync_all();

  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (GATHER && warp == 0) {
    // the whole warp loads this CTA's A rows (four a lane), lane 0 also its half of the B rows
    const CUtensorMap* tmB = even ? &tmB0 : &tmB1;
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(tmB);
    }
    uint64_t pol_a, pol_b;  // the operand that later tiles read again is kept in L2
    l2_policies(sched, &pol_a, &pol_b);
    const int64_t a_total = seg_hi(offsets, E - 1, rows_cap);
    uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
    bool ok = true;
    for (int tile = cid; ok && tile < total; tile += ncl) {
      int e, nt, mt;
      decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
      const int4 rows = gather_rows4(
          g, static_cast<int64_t>(seg_lo(offsets, e)) + mt * P_BM + static_cast<int>(rank) * 128 + 4 * lane, a_total,
          status);
      const int b_row = e * b_rows_per_expert + nt * TILE_N;
      for (int kb = 0; kb < KB; ++kb) {
        const bool got = ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint8_t* sa = stages + stage * P_STAGE_BYTES;
        const uint32_t full_pair = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
        if (lane == 0) {
          if (even) ptx::mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
          ptx::tma_load_2d_pair(sa + P_A_BYTES, tmB, kb * BK, b_row, full_pair, pol_b);
        }
        __syncwarp();
        ptx::tma_gather4_pair(sa + lane * 512, &tmA, kb * BK, rows.x, rows.y, rows.z, rows.w, full_pair, pol_a);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == P_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      if (even) {
        // both CTAs' copies into every stage this CTA armed have landed before the pair may exit
        for (int s = 0; s < P_STAGES; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&full[s], (armed_phase >> s) & 1u);
      }
      if (*abort_flag) {
        // copies whose completion is counted in the other CTA cannot be awaited here: give them time
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB0);
      if (SWIGLU) ptx::prefetch_tmap(&tmB1);
      const CUtensorMap* tmB = (SWIGLU && !even) ? &tmB1 : &tmB0;
      uint64_t pol_a, pol_b;  // the operand that later tiles read again is kept in L2
      l2_policies(sched, &pol_a, &pol_b);
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        int e, nt, mt;
        decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
        const int a_row = seg_lo(offsets, e) + mt * P_BM + static_cast<int>(rank) * 128;
        const int b_row = SWIGLU ? e * b_rows_per_expert + nt * TILE_N
                                 : e * b_rows_per_expert + nt * TILE_N + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + stage * P_STAGE_BYTES;
          const uint32_t full_pair = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
          if (even) ptx::mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
          ptx::tma_load_2d_pair(sa, &tmA, kb * BK, a_row, full_pair, pol_a);
          ptx::tma_load_2d_pair(sa + P_A_BYTES, tmB, kb * BK, b_row, full_pair, pol_b);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (even) {
        // both CTAs' copies into every stage this CTA armed have landed before the pair may exit
        for (int s = 0; s < P_STAGES; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&full[s], (armed_phase >> s) & 1u);
      }
      if (*abort_flag) {
        // copies whose completion is counted in the other CTA cannot be awaited here: give them time
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (even && lane == 0) {
      constexpr uint32_t IDESC = ptx::idesc_bf16_f32(P_BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        if (!wait_cluster_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_cluster_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stages + stage * P_STAGE_BYTES);
          const uint32_t sb = sa + P_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            ptx::mma_bf16_ss_pair(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * UK * 2),
                                  ptx::sdesc_kmajor_sw128(sb + kk * UK * 2), IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair(&empty[stage], 0x3);  // both CTAs' stage is free once these MMAs have read it
          if (++stage == P_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(&tfull[acc], 0x3);  // both halves of the accumulator are complete
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit_pair(drain, 0x1);  // every MMA issued above has completed once this arrives
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const int r_local = static_cast<int>(rank) * 128 + q * 32 + lane;
    uint8_t* ostage = smem + P_OUT_OFF + q * P_OUT_BYTES;  // 1024-byte aligned
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = cid; tile < total; tile += ncl) {
      int e, nt, mt;
      decode_tile(tab, E, NT, tile, &e, &nt, &mt, sched & 1);
      const int seg = seg_lo(offsets, e);
      const int n_e = seg_hi(offsets, e, rows_cap) - seg;
      const bool row_ok = mt * P_BM + r_local < n_e;
      const int64_t row = static_cast<int64_t>(seg) + mt * P_BM + r_local;
      // the tcgen05.ld below is warp-collective: the warp leaves together or not at all
      const bool ready = wait_cluster_bounded(&tfull[acc], acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, ready)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      bf16* orow = out + row * n_out;
      // a warp whose 32 rows all lie inside the segment stages 64-column blocks in shared memory
      // and stores them with the TMA; a warp that straddles the segment's end stores row by row
      const bool warp_full = mt * P_BM + static_cast<int>(rank) * 128 + q * 32 + 32 <= n_e;
      const int row0 = seg + mt * P_BM + static_cast<int>(rank) * 128 + q * 32;
#pragma unroll 1
      for (int c = 0; c < TILE_N; c += 32) {
        uint32_t packed[16];
        if (SWIGLU) {
          uint32_t gv[32], uv[32];
          ptx::tmem_ld_32x32b_x32(tb + c, gv);
          ptx::tmem_ld_32x32b_x32(tb + BN / 2 + c, uv);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = silu_mul(__uint_as_float(gv[2 * i]), __uint_as_float(uv[2 * i]));
            const float a1 = silu_mul(__uint_as_float(gv[2 * i + 1]), __uint_as_float(uv[2 * i + 1]));
            packed[i] = Vec16<bf16>::pack2(a0, a1);
          }
        } else {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(tb + c, v);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = Vec16<bf16>::pack2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        }
        if (!warp_full) {
          if (row_ok) store_32(orow, nt * TILE_N + c, n_out, packed);
          continue;
        }
        const int half = (c >> 5) & 1;  // which 64 bytes of the block's 128-byte rows
        if (half == 0) {
          if (lane == 0) ptx::bulk_wait_read<0>();  // this warp's previous block has been read
          __syncwarp();
        }
        // row `lane`, 16-byte chunks 4 half .. 4 half + 3, at their 128-byte-swizzle positions
        uint4* srow = reinterpret_cast<uint4*>(ostage + lane * 128);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          srow[(4 * half + i) ^ (lane & 7)] =
              make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        if (half == 1) {
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_2d(&tmOut, ostage, nt * TILE_N + c - 32, row0);
            ptx::bulk_commit();
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&tempty[acc]), 0));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) ptx::bulk_wait_all();  // this warp's stores have completed
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // the even CTA's MMAs into this CTA's tensor memory are over
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *abort_flag) set_status(status, MOE_DEV_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Weights as the M operand ("swapped" grouped GEMM on CTA pairs): D^T = W X^T.
//
// A 256-row tile of weight rows (128 per CTA) times up to 256 token rows of one
// expert segment, with the token count N of the last tile of a segment rounded up
// to 16 only.  Row tiles of 128 or 256 tokens waste up to a whole tile per expert
// (11% of the MMA work of a 512-row segment split 4+1, 20% with 256-row pairs);
// with tokens on the N side the waste is under 16 rows per expert, and the CTA
// pair keeps the stage at 32 KB per CTA.
//   A (this CTA)  SwiGLU: 64 W_gate rows then the same 64 W_up rows (output
//                 columns j_base .. j_base + 63, j_base = 128 mt + 64 rank);
//                 plain: 128 W rows (output columns 256 mt + 128 rank + lane quarter).
//   B (this CTA)  token rows seg + 256 nt + rank N/2 .. +N/2 (a 128-row box: the
//                 MMA reads the first N/2 rows of each CTA's B).
//   TMEM lane i of a CTA = its weight row i, column t = token t of the tile.
// SwiGLU epilogue: warps of lane quarters 0/1 hold gate, 2/3 the matching up
// rows.  Per 32-token chunk the two warps of a pair swap halves through shared
// memory (gate of tokens 16..31 one way, up of tokens 0..15 the other), then each
// forms SiLU(g) * u for 16 tokens.  Stores: lane = output column, so each warp
// store writes 32 consecutive columns (64 bytes) of one token row.
constexpr int S_BN = 256;                                  // tokens per tile at most
constexpr int S_STAGES = 6;
constexpr uint32_t S_A_BYTES = 128 * BK * 2;              // 16 KB of weight rows
constexpr uint32_t S_B_BYTES = 128 * BK * 2;              // 16 KB box of token rows
constexpr uint32_t S_STAGE_BYTES = S_A_BYTES + S_B_BYTES;
constexpr uint32_t S_XCH_FLOATS = 2 * 2 * 16 * 32;        // 2 warp pairs x 2 directions x [16][32]
constexpr size_t S_SMEM_BYTES =
    1024 + S_STAGES * S_STAGE_BYTES + S_XCH_FLOATS * 4 + P_BAR_BYTES + sizeof(int) * (MAX_E + 1);
static_assert(S_SMEM_BYTES <= 232448, "shared memory");
static_assert((2 * S_STAGES + 2 + 2 + 1) * 8 + 12 <= P_BAR_BYTES, "barriers fit P_BAR_BYTES");

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// AND of `pred` over the `threads` threads of named barrier `id` (every one of them gets it)
__device__ __forceinline__ bool named_all(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// First row and MMA width N of token tile nt of a segment of n rows: 256-row tiles, the last one
// rounded up to 16 rows.  (Tiles of one balanced size per segment were measured 1-2% slower on the
// 512-row segments of the Mixtral shape: a short last tile costs only its weight reads, which
// the segment's full tiles have already brought into L2.)
__device__ __forceinline__ void swab_tile(int n, int nt, int* t0, int* N) {
  *t0 = nt * S_BN;
  const int rem = n - *t0;
  *N = rem >= S_BN ? S_BN : (rem + 15) / 16 * 16;
}

// SWIGLU: out[row, j] = SiLU((X W0^T)[row, j]) * (X W1^T)[row, j], j < n_out (= d_e), W0/W1 rows per expert = d_e.
// plain:  out[row, m] = (X W0^T)[row, m],                           m < n_out (= h),   W0 rows per expert = h.
// FP8 (SwiGLU only): X, W0, W1 are E4M3 codes (kind::f8f6f4, 128 K-elements per stage row); each
// sum is scaled by x_scale[row] * w_scale[weight row] before SiLU * up.
template <bool SWIGLU, bool FP8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    grouped_gemm_swab(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                      const __grid_constant__ CUtensorMap tmX, const int32_t* __restrict__ offsets, int E, int K,
                      int w_rows_per_expert, int n_out, int64_t rows_cap, bf16* __restrict__ out, int32_t* status,
                      const float* __restrict__ x_scale = nullptr, const float* __restrict__ w0_scale = nullptr,
                      const float* __restrict__ w1_scale = nullptr) {
  static_assert(SWIGLU || !FP8, "the FP8 path is the up-projection");
  constexpr int WT = SWIGLU ? 128 : 256;  // output columns per pair tile
  constexpr int BKE = FP8 ? 2 * BK : BK;  // K elements per stage (128 bytes of every row)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + aligned_1024(smem_raw);
  uint8_t* stages = smem;
  float* xch = reinterpret_cast<float*>(smem + S_STAGES * S_STAGE_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S_STAGES * S_STAGE_BYTES + S_XCH_FLOATS * 4);
  uint64_t* empty = full + S_STAGES;
  uint64_t* tfull = empty + S_STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* bad_flag = reinterpret_cast<int*>(tmem_holder + 2);
  int* tab = reinterpret_cast<int*>(smem + S_STAGES * S_STAGE_BYTES + S_XCH_FLOATS * 4 + P_BAR_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool even = rank == 0;
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  const int MT = (n_out + WT - 1) / WT;  // weight tiles per expert
  const int KB = (K + BKE - 1) / BKE;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *bad_flag = 0;
  }
  __syncthreads();
  // token tiles per expert; both CTAs of a pair reach the same decisions
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
    int m = 0;
    if (lo < 0 || hi < lo || static_cast<int64_t>(hi) > rows_cap)
      *bad_flag = 1;
    else
      m = (hi - lo + S_BN - 1) / S_BN;
    tab[e + 1] = m;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    tab[0] = 0;
    for (int e = 0; e < E; ++e) tab[e + 1] += tab[e];
    if (*bad_flag && blockIdx.x == 0) set_status(status, MOE_DEV_BAD_OFFSETS);
    for (int s = 0; s < S_STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 8);
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbarrier_init();
  }
  __syncthreads();
  if (*bad_flag) return;
  const int total = tab[E] * MT;
  if (cid >= total) return;
  ptx::cluster_sync_all();  // the peer's barriers are initialised before anything arrives on them

  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmW0);
      if (SWIGLU) ptx::prefetch_tmap(&tmW1);
      ptx::prefetch_tmap(&tmX);
      const uint64_t pol_w = ptx::policy_evict_normal();
      const uint64_t pol_x = ptx::policy_evict_last();
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        int e, mt, nt;
        decode_tile(tab, E, MT, tile, &e, &mt, &nt);
        const int seg = seg_lo(offsets, e);
        const int n_e = seg_hi(offsets, e, rows_cap) - seg;
        int t0, N;
        swab_tile(n_e, nt, &t0, &N);
        const int x_row = seg + t0 + static_cast<int>(rank) * (N / 2);
        const int w_row = SWIGLU ? e * w_rows_per_expert + mt * WT + static_cast<int>(rank) * 64
                                 : e * w_rows_per_expert + mt * WT + static_cast<int>(rank) * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* sa = stages + stage * S_STAGE_BYTES;
          const uint32_t full_pair = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
          if (even) ptx::mbar_arrive_expect_tx(&full[stage], 2 * S_STAGE_BYTES);
          if (SWIGLU) {
            ptx::tma_load_2d_pair(sa, &tmW0, kb * BKE, w_row, full_pair, pol_w);
            ptx::tma_load_2d_pair(sa + S_A_BYTES / 2, &tmW1, kb * BKE, w_row, full_pair, pol_w);
          } else {
            ptx::tma_load_2d_pair(sa, &tmW0, kb * BKE, w_row, full_pair, pol_w);
          }
          ptx::tma_load_2d_pair(sa + S_A_BYTES, &tmX, kb * BKE, x_row, full_pair, pol_x);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == S_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (even) {
        for (int s = 0; s < S_STAGES; ++s)
          if ((armed >> s) & 1u) mbar_wait_drain(&full[s], (armed_phase >> s) & 1u);
      }
      if (*abort_flag) {
        // copies whose completion is counted in the other CTA cannot be awaited here: give them time
        const uint64_t t0 = ptx::globaltimer_ns();
        while (ptx::globaltimer_ns() - t0 < 1000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (even && lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        int e, mt, nt;
        decode_tile(tab, E, MT, tile, &e, &mt, &nt);
        const int n_e = seg_hi(offsets, e, rows_cap) - seg_lo(offsets, e);
        int t0, N;
        swab_tile(n_e, nt, &t0, &N);
        const uint32_t idesc = FP8 ? ptx::idesc_e4m3_f32(256, N) : ptx::idesc_bf16_f32(256, N);
        if (!wait_cluster_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!wait_cluster_bounded(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(stages + stage * S_STAGE_BYTES);
          const uint32_t sb = sa + S_A_BYTES;
          // 32 bytes of K per MMA: 16 bf16 or 32 E4M3
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            if (FP8)
              ptx::mma_f8_ss_pair(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * 32), ptx::sdesc_kmajor_sw128(sb + kk * 32),
                                  idesc, (kb | kk) != 0 ? 1u : 0u);
            else
              ptx::mma_bf16_ss_pair(d_tmem, ptx::sdesc_kmajor_sw128(sa + kk * 32),
                                    ptx::sdesc_kmajor_sw128(sb + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair(&empty[stage], 0x3);
          if (++stage == S_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(&tfull[acc], 0x3);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;  // tensor-memory lane quarter this warp may read
    const bool up_half = SWIGLU && q >= 2;
    const int p = q & 1;     // SwiGLU: warps of quarters p and p + 2 hold gate and up of the same columns
    float* xg = xch + p * (2 * 16 * 32);  // gate values of tokens 16..31, [16][32]
    float* xu = xg + 16 * 32;             // up values of tokens 0..15
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = cid; tile < total; tile += ncl) {
      int e, mt, nt;
      decode_tile(tab, E, MT, tile, &e, &mt, &nt);
      const int seg = seg_lo(offsets, e);
      const int n_e = seg_hi(offsets, e, rows_cap) - seg;
      int t_tile, N;
      swab_tile(n_e, nt, &t_tile, &N);
      const int n_valid = n_e - t_tile < N ? n_e - t_tile : N;
      const int col = SWIGLU ? mt * WT + static_cast<int>(rank) * 64 + p * 32 + lane
                             : mt * WT + static_cast<int>(rank) * 128 + q * 32 + lane;
      const bool col_ok = col < n_out;
      bf16* obase = out + (static_cast<int64_t>(seg) + t_tile) * n_out + col;
      // FP8: this lane's weight-row scale (gate rows in quarters 0/1, up rows in 2/3)
      float w_s = 1.f;
      if (FP8 && col_ok) w_s = (up_half ? w1_scale : w0_scale)[static_cast<int64_t>(e) * w_rows_per_expert + col];
      // the tcgen05.ld below is warp-collective, and the SwiGLU exchange pairs two warps: both
      // warps of a pair leave together or not at all
      const bool ready = wait_cluster_bounded(&tfull[acc], acc_phase, abort_flag);
      const bool go = SWIGLU ? named_all(1 + p, 64, ready) : __all_sync(0xffffffffu, ready);
      if (!go) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < n_valid; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tb + c, v);
        // FP8: lane i holds the scale of token c + i, shared by every weight row
        const float my_xs = (FP8 && c + lane < n_valid) ? x_scale[static_cast<int64_t>(seg) + t_tile + c + lane] : 0.f;
        ptx::tmem_wait_ld();
        if (FP8) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) * (w_s * __shfl_sync(0xffffffffu, my_xs, i)));
        }
        if (SWIGLU) {
          // swap halves with the partner warp: keep 16 tokens, hand over the other 16
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (up_half)
              xu[i * 32 + lane] = __uint_as_float(v[i]);
            else
              xg[i * 32 + lane] = __uint_as_float(v[16 + i]);
          }
          named_sync(1 + p, 64);
          const int t0 = c + (up_half ? 16 : 0);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = up_half ? xg[i * 32 + lane] : __uint_as_float(v[i]);
            const float uv = up_half ? __uint_as_float(v[16 + i]) : xu[i * 32 + lane];
            if (col_ok && t0 + i < n_valid) obase[static_cast<int64_t>(t0 + i) * n_out] = __float2bfloat16_rn(silu_mul(gv, uv));
          }
          named_sync(1 + p, 64);  // both have read the exchange before the next chunk writes it
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (col_ok && c + i < n_valid) obase[static_cast<int64_t>(c + i) * n_out] = __float2bfloat16_rn(__uint_as_float(v[i]));
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&tempty[acc]), 0));
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();  // the even CTA's MMAs into this CTA's tensor memory are over
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
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

// Row-major matrix [rows, cols] of bf16 (or of bytes: E4M3 codes) read in boxes of box_rows x
// 128 bytes with the 128-byte swizzle.
static bool make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                      bool bytes = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (bytes ? 1 : 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(bytes ? 2 * BK : BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

// Which kernel runs the two grouped GEMMs.  CTA pairs cut the shared-memory
// operand traffic per MMA by a third.  With row tiles of 256 tokens they pay off
// when the expert segments are long (measured on B300: 0.80 vs 0.67 of the bf16
// peak with 6144-row segments); shorter segments go to the weights-as-M pair
// kernel, whose token tiles end within 16 rows of each segment (measured:
// 1100 vs 1017 TFLOP/s with 512-row segments, 82% vs 76% of HBM bandwidth with
// the 128-row segments of the 256-expert shape).  The single-CTA kernel serves
// the FP8 and gathered up-projections, one-segment products and the override.
// MOE_FFN_TILES=single|pair|swab overrides the choice (for measurement and for
// testing every kernel).
static bool use_pair_tiles(const Plan& p) {
  const char* env = getenv("MOE_FFN_TILES");
  if (env && strcmp(env, "single") == 0) return false;
  if (env && strcmp(env, "pair") == 0) return true;
  return p.Tk >= static_cast<int64_t>(1024) * p.E;  // mean rows per expert >= 1024
}

// The swapped-operand pair kernel (weights as M, tokens as N): segments shorter than 1024 rows
// on average, unless MOE_FFN_TILES names another kernel.
static bool use_swab_tiles(const Plan& p) {
  const char* env = getenv("MOE_FFN_TILES");
  if (env && (strcmp(env, "single") == 0 || strcmp(env, "pair") == 0)) return false;
  if (env && strcmp(env, "swab") == 0) return true;
  return p.Tk < static_cast<int64_t>(1024) * p.E;
}

template <bool SWIGLU, bool FP8 = false>
static cudaError_t launch_swab(int64_t tiles, const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& x,
                               const int32_t* offsets, int E, int K, int w_rows, int n_out, int64_t rows_cap,
                               bf16* out, int32_t* status, cudaStream_t s, const float* x_scale = nullptr,
                               const float* w0_scale = nullptr, const float* w1_scale = nullptr) {
  using namespace tc;
  auto kern = grouped_gemm_swab<SWIGLU, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(S_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  int grid = 2 * static_cast<int>(std::min<int64_t>(current_sm_count() / 2, tiles));
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = S_SMEM_BYTES;
  lc.stream = s;
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &lc) == cudaSuccess && max_clusters > 0 &&
      2 * max_clusters < grid)
    grid = 2 * max_clusters;
  (void)cudaGetLastError();
  kern<<<grid, THREADS, S_SMEM_BYTES, s>>>(w0, w1, x, offsets, E, K, w_rows, n_out, rows_cap, out, status, x_scale,
                                           w0_scale, w1_scale);
  return cudaGetLastError();
}

static cudaError_t launch_ffn_swab(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                                   const void* W_up, const void* W_down, void* act, void* Y, int32_t* status,
                                   cudaStream_t s) {
  using namespace tc;
  CUtensorMap tmX, tmG, tmU, tmAct, tmD;
  const uint64_t Tk = static_cast<uint64_t>(p.Tk);
  if (!make_tmap(&tmX, X, Tk, p.h, 128) ||
      !make_tmap(&tmG, W_gate, static_cast<uint64_t>(p.E) * p.d_e, p.h, 64) ||
      !make_tmap(&tmU, W_up, static_cast<uint64_t>(p.E) * p.d_e, p.h, 64) ||
      !make_tmap(&tmAct, act, Tk, p.d_e, 128) ||
      !make_tmap(&tmD, W_down, static_cast<uint64_t>(p.E) * p.h, p.d_e, 128))
    return cudaErrorNotSupported;
  const int64_t ntiles = (p.Tk + S_BN - 1) / S_BN + p.E;  // token tiles, at most
  const int64_t tiles1 = ntiles * ((p.d_e + 127) / 128);
  const int64_t tiles2 = ntiles * ((p.h + 255) / 256);
  if (tiles1 >= (int64_t(1) << 31) || tiles2 >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  cudaError_t e = launch_swab<true>(tiles1, tmG, tmU, tmX, offsets, p.E, p.h, p.d_e, p.d_e, p.Tk,
                                    static_cast<bf16*>(act), status, s);
  if (e != cudaSuccess) return e;
  return launch_swab<false>(tiles2, tmD, tmD, tmAct, offsets, p.E, p.d_e, p.h, p.h, p.Tk, static_cast<bf16*>(Y),
                            status, s);
}

template <bool SWIGLU, bool GATHER = false>
static cudaError_t launch_gemm(bool pair, int grid, const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                               const int32_t* offsets, int E, int K, int b_rows, int n_out, int64_t rows_cap, bf16* out,
                               int32_t* status, cudaStream_t s, tc::Gather g = tc::Gather{}, int sched = 0) {
  using namespace tc;
  if (pair) {
    // the pair kernel's epilogue stores 32-row x 64-column blocks of `out` through this map
    CUtensorMap tmOut;
    if (!make_tmap(&tmOut, out, static_cast<uint64_t>(rows_cap), static_cast<uint64_t>(n_out), 32))
      return cudaErrorNotSupported;
    auto kern = grouped_gemm_tc_pair<SWIGLU, GATHER>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(P_SMEM_BYTES));
    if (e != cudaSuccess) return e;
    // no more clusters than can be resident at once (SMs that cannot be paired stay idle)
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(THREADS);
    lc.dynamicSmemBytes = P_SMEM_BYTES;
    lc.stream = s;
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &lc) == cudaSuccess && max_clusters > 0 &&
        2 * max_clusters < grid)
      grid = 2 * max_clusters;
    (void)cudaGetLastError();
    kern<<<grid, THREADS, P_SMEM_BYTES, s>>>(a, b0, b1, tmOut, offsets, E, K, b_rows, n_out, rows_cap, out, status, g,
                                             sched);
  } else {
    auto kern = grouped_gemm_tc<SWIGLU, false, GATHER>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    kern<<<grid, THREADS, SMEM_BYTES, s>>>(a, b0, b1, offsets, E, K, b_rows, n_out, rows_cap, out, status, nullptr,
                                           nullptr, nullptr, g, sched);
  }
  return cudaGetLastError();
}

// out[rows, N] = A[rows, K] B[N, K]^T (bf16, both K-major, float32 accumulation, bf16 out), one
// segment of all rows on the single-CTA kernel.
cudaError_t launch_dense_gemm_tc(const void* A, int64_t rows, int K, const void* B, int N, void* out, int32_t* status,
                                 cudaStream_t s) {
  using namespace tc;
  if (rows == 0) return cudaSuccess;
  CUtensorMap tmA, tmB;
  if (!make_tmap(&tmA, A, static_cast<uint64_t>(rows), static_cast<uint64_t>(K), BM) ||
      !make_tmap(&tmB, B, static_cast<uint64_t>(N), static_cast<uint64_t>(K), BN))
    return cudaErrorNotSupported;
  const int64_t tiles = ((rows + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = static_cast<int>(std::min<int64_t>(current_sm_count(), tiles));
  return launch_gemm<false>(false, grid, tmA, tmB, tmB, nullptr, 1, K, N, N, rows, static_cast<bf16*>(out), status, s);
}

cudaError_t launch_ffn_tc(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                          const void* W_up, const void* W_down, void* act, void* Y, int32_t* status,
                          cudaStream_t s, const void* gather_src, const int32_t* gather_rows) {
  using namespace tc;
  if (p.Tk == 0) return cudaSuccess;
  const bool gather = gather_rows != nullptr;  // X[row] = gather_src[gather_rows[row]], read by GEMM1 itself
  if (!gather && offsets != nullptr && use_swab_tiles(p))
    return launch_ffn_swab(p, X, offsets, W_gate, W_up, W_down, act, Y, status, s);
  const bool pair = use_pair_tiles(p);
  const uint32_t a_box = pair ? 128 : BM;           // rows of A each CTA stages
  const uint32_t down_box = pair ? BN / 2 : BN;     // rows of W_down each CTA stages
  CUtensorMap tmX, tmG, tmU, tmAct, tmD;
  const uint64_t Tk = static_cast<uint64_t>(p.Tk);
  // (gathered: the token rows of the source, one-row boxes for the four-row gathers)
  if (!make_tmap(&tmX, gather ? gather_src : X, gather ? static_cast<uint64_t>(p.T) : Tk, p.h, gather ? 1 : a_box) ||
      !make_tmap(&tmG, W_gate, static_cast<uint64_t>(p.E) * p.d_e, p.h, BN / 2) ||
      !make_tmap(&tmU, W_up, static_cast<uint64_t>(p.E) * p.d_e, p.h, BN / 2) ||
      !make_tmap(&tmAct, act, Tk, p.d_e, a_box) ||
      !make_tmap(&tmD, W_down, static_cast<uint64_t>(p.E) * p.h, p.d_e, down_box))
    return cudaErrorNotSupported;
  const int nsm = current_sm_count();
  const int rows_per_tile = pair ? P_BM : BM;
  const int64_t mtiles_max = (p.Tk + rows_per_tile - 1) / rows_per_tile + p.E;
  const int64_t tiles1 = mtiles_max * ((p.d_e + BN / 2 - 1) / (BN / 2));
  const int64_t tiles2 = mtiles_max * ((p.h + BN - 1) / BN);
  if (tiles1 >= (int64_t(1) << 31) || tiles2 >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  // persistent grids: one CTA per SM (pairs: one cluster per two SMs)
  const int units = pair ? nsm / 2 : nsm;
  const int per = pair ? 2 : 1;
  const int grid1 = per * static_cast<int>(std::min<int64_t>(units, tiles1));
  const int grid2 = per * static_cast<int>(std::min<int64_t>(units, tiles2));
  // tile order: the operand re-read per tile of the other is the smaller one of an expert (its mean
  // rows of A against its rows of B, both K wide): on the stress shape the 6144-row segments of X
  // are 50 MB against 23 MB of gate|up weights, and were read from HBM about 2.5 times
  // (MOE_FFN_ORDER=rows|cols overrides the choice for both GEMMs, for measurement and tests)
  const int64_t a_rows = p.Tk / p.E;
  int order1 = a_rows > 2 * static_cast<int64_t>(p.d_e) ? 1 : 0;
  int order2 = a_rows > static_cast<int64_t>(p.h) ? 1 : 0;
  if (const char* env = getenv("MOE_FFN_ORDER")) {
    if (strcmp(env, "rows") == 0) order1 = order2 = 0;
    if (strcmp(env, "cols") == 0) order1 = order2 = 1;
  }
  // L2 hints (MOE_FFN_L2=none|first for measurement): bits 1-2 of the tile schedule
  int l2 = 0;
  if (const char* env = getenv("MOE_FFN_L2")) {
    if (strcmp(env, "none") == 0) l2 = 1;
    if (strcmp(env, "first") == 0) l2 = 2;
  }
  order1 |= l2 << 1;
  order2 |= l2 << 1;
  cudaError_t e =
      gather ? launch_gemm<true, true>(pair, grid1, tmX, tmG, tmU, offsets, p.E, p.h, p.d_e, p.d_e, p.Tk,
                                       static_cast<bf16*>(act), status, s,
                                       Gather{gather_rows, p.T}, order1)
             : launch_gemm<true>(pair, grid1, tmX, tmG, tmU, offsets, p.E, p.h, p.d_e, p.d_e, p.Tk,
                                 static_cast<bf16*>(act), status, s, Gather{}, order1);
  if (e != cudaSuccess) return e;
  return launch_gemm<false>(pair, grid2, tmAct, tmD, tmD, offsets, p.E, p.d_e, p.h, p.h, p.Tk, static_cast<bf16*>(Y),
                            status, s, Gather{}, order2);
}

// The FP8 up-projection (single-CTA kernel, kind::f8f6f4) followed by the usual bf16 down GEMM.
cudaError_t launch_ffn_fp8_tc(const Plan& p, const uint8_t* X8, const float* x_scale, const int32_t* offsets,
                              const uint8_t* W_gate8, const uint8_t* W_up8, const float* s_gate, const float* s_up,
                              const void* W_down, void* act, void* Y, int32_t* status, cudaStream_t s) {
  using namespace tc;
  if (p.Tk == 0) return cudaSuccess;
  const bool pair = use_pair_tiles(p);
  const uint32_t a_box = pair ? 128 : BM;
  const uint32_t down_box = pair ? BN / 2 : BN;
  CUtensorMap tmX, tmG, tmU, tmAct, tmD;
  const uint64_t Tk = static_cast<uint64_t>(p.Tk);
  if (!make_tmap(&tmX, X8, Tk, p.h, BM, true) ||
      !make_tmap(&tmG, W_gate8, static_cast<uint64_t>(p.E) * p.d_e, p.h, BN / 2, true) ||
      !make_tmap(&tmU, W_up8, static_cast<uint64_t>(p.E) * p.d_e, p.h, BN / 2, true) ||
      !make_tmap(&tmAct, act, Tk, p.d_e, a_box) ||
      !make_tmap(&tmD, W_down, static_cast<uint64_t>(p.E) * p.h, p.d_e, down_box))
    return cudaErrorNotSupported;
  const int nsm = current_sm_count();
  const int64_t mt1 = (p.Tk + BM - 1) / BM + p.E;
  const int64_t tiles1 = mt1 * ((p.d_e + BN / 2 - 1) / (BN / 2));
  const int rows_per_tile = pair ? P_BM : BM;
  const int64_t tiles2 = ((p.Tk + rows_per_tile - 1) / rows_per_tile + p.E) * ((p.h + BN - 1) / BN);
  if (tiles1 >= (int64_t(1) << 31) || tiles2 >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int grid1 = static_cast<int>(std::min<int64_t>(nsm, tiles1));
  const int per = pair ? 2 : 1;
  const int grid2 = per * static_cast<int>(std::min<int64_t>(pair ? nsm / 2 : nsm, tiles2));
  if (use_swab_tiles(p)) {
    // both GEMMs on the weights-as-M pair kernel (64-row gate/up boxes, 128-row token boxes)
    CUtensorMap sX, sG, sU, sAct, sD;
    if (!make_tmap(&sX, X8, Tk, p.h, 128, true) ||
        !make_tmap(&sG, W_gate8, static_cast<uint64_t>(p.E) * p.d_e, p.h, 64, true) ||
        !make_tmap(&sU, W_up8, static_cast<uint64_t>(p.E) * p.d_e, p.h, 64, true) ||
        !make_tmap(&sAct, act, Tk, p.d_e, 128) || !make_tmap(&sD, W_down, static_cast<uint64_t>(p.E) * p.h, p.d_e, 128))
      return cudaErrorNotSupported;
    const int64_t nt = (p.Tk + S_BN - 1) / S_BN + p.E;
    cudaError_t e = launch_swab<true, true>(nt * ((p.d_e + 127) / 128), sG, sU, sX, offsets, p.E, p.h, p.d_e, p.d_e,
                                            p.Tk, static_cast<bf16*>(act), status, s, x_scale, s_gate, s_up);
    if (e != cudaSuccess) return e;
    return launch_swab<false>(nt * ((p.h + 255) / 256), sD, sD, sAct, offsets, p.E, p.d_e, p.h, p.h, p.Tk,
                              static_cast<bf16*>(Y), status, s);
  }
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_tc<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  grouped_gemm_tc<true, true><<<grid1, THREADS, SMEM_BYTES, s>>>(tmX, tmG, tmU, offsets, p.E, p.h, p.d_e, p.d_e, p.Tk,
                                                                 static_cast<bf16*>(act), status, x_scale, s_gate,
                                                                 s_up);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_gemm<false>(pair, grid2, tmAct, tmD, tmD, offsets, p.E, p.d_e, p.h, p.h, p.Tk, static_cast<bf16*>(Y),
                            status, s);
}

}  // namespace moe
