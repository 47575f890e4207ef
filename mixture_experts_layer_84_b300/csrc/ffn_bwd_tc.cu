// Backward of the grouped bf16 SwiGLU experts on the 5th-generation tensor cores.
//
// "MoE 与专家并行" (hs-black.github.io/posts/scaling-moe), section 专家计算：
// padding、block-sparse 与 grouped GEMM: the backward of the SwiGLU experts is
// grouped GEMMs as well, one group for the input gradients and one for the
// weight gradients.  Section 从稠密 FFN 到 MoE gives the expert
// y = W_down (SiLU(W_gate x) * W_up x); with G = x W_gate^T, Up = x W_up^T,
// s = sigmoid(G):
//   d_act = dY W_down                      (rows x d_e, K = h)       DACT
//   dG = d_act Up s (1 + G (1 - s)),  dUp = d_act G s                 DGU
//        (G and Up recomputed by the forward gate|up product)
//   dX = dG W_gate + dUp W_up              (rows x h, K = 2 d_e)     DX
//   dW_down = dY^T act,  dW_gate = dG^T X,  dW_up = dUp^T X           WGRAD
//        (K = the expert's rows)
// The weights are stored K-major for the forward, so the input-gradient
// products read them MN-major (the N index contiguous): TMA boxes of 64 N x
// 64 K with the 128-byte swizzle, MMA descriptors with MN-atoms 8 KB apart
// and 8-row K groups 1 KB apart, and the instruction's B-major bit set.  The
// weight gradients read both operands MN-major from the row-major
// activations, their K running over one expert's rows; the rows of a last
// k-block past the expert's segment are zeroed in shared memory before the
// MMA reads them (they hold the next expert's rows).
// Pipeline, roles and bounded waits follow the forward kernel: warp 0 TMA
// producer (4 stages), warp 1 tensor-memory owner and MMA issuer (two
// 128 x 256 float32 accumulators), warps 2-5 epilogue.  The weight gradients'
// epilogue stages each warp's 32 x 32 float32 block in shared memory and writes
// it with one TMA store through an [E, M, N] map, so every store leaves as whole
// 128-byte rows.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace bwd {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int UK = 16;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t ACC_COLS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int THREADS = 192;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr int MAX_E = 1024;
constexpr size_t BAR_BYTES = 128;
constexpr size_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + BAR_BYTES + sizeof(int) * (MAX_E + 1);
static_assert(SMEM_BYTES <= 232448, "shared memory");

constexpr uint32_t ATOM_BYTES = 64 * 128;  // one MN-major atom column: 64 K-rows of 128 bytes
// grouped_wgrad stages each epilogue warp's 32 x 32 float32 block (4 KB, 128-byte swizzle) for a
// TMA store, after the tile table
constexpr size_t W_STAGING_OFFSET = (STAGES * STAGE_BYTES + BAR_BYTES + sizeof(int) * (MAX_E + 1) + 1023) / 1024 * 1024;
constexpr size_t W_SMEM_BYTES = 1024 + W_STAGING_OFFSET + 4 * 4096;
static_assert(W_SMEM_BYTES <= 232448, "shared memory");

enum Mode { DACT = 0, DGU = 1, DX = 2 };

// MN-major operand, 128-byte swizzle: 64 MN elements per 128-byte K-row, 8-row K groups of
// 1024 bytes, MN-atoms `lbo` bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t smem_addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(lbo >> 4) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc(int M, int N, bool a_mn, bool b_mn) {
  return ptx::idesc_bf16_f32(M, N) | (a_mn ? (1u << 15) : 0u) | (b_mn ? (1u << 16) : 0u);
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
  return true;
}

__device__ __forceinline__ void decode_tile(const int* tab, int E, int NT, int tile, int* e, int* nt, int* mt) {
  int lo = 0, hi = E;
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
  *nt = local / m_e;
  *mt = local - (*nt) * m_e;
}

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

// Shared per-CTA setup of the tile table (m-tiles of `rows_per_tile` rows per expert) and barriers.
struct Smem {
  uint8_t* stages;
  uint64_t *full, *empty, *tfull, *tempty, *drain;
  uint32_t* tmem_holder;
  volatile int* abort_flag;
  int* bad_flag;
  int* tab;
};

__device__ __forceinline__ Smem carve(uint8_t* smem_raw) {
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);  // (shared state space kept)
  Smem m;
  m.stages = smem;
  m.full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  m.empty = m.full + STAGES;
  m.tfull = m.empty + STAGES;
  m.tempty = m.tfull + 2;
  m.drain = m.tempty + 2;
  m.tmem_holder = reinterpret_cast<uint32_t*>(m.drain + 1);
  m.abort_flag = reinterpret_cast<volatile int*>(m.tmem_holder + 1);
  m.bad_flag = reinterpret_cast<int*>(m.tmem_holder + 2);
  m.tab = reinterpret_cast<int*>(smem + STAGES * STAGE_BYTES + BAR_BYTES);
  return m;
}

// tab[e + 1] - tab[e] = tiles_per_expert(e) (rows-based, or 1 for every expert when per_expert > 0);
// returns false (and flags the status) when the offsets are inconsistent.
__device__ __forceinline__ bool setup(const Smem& m, const int32_t* offsets, int E, int64_t rows_cap,
                                      int rows_per_tile, int32_t* status) {
  if (threadIdx.x == 0) {
    *m.abort_flag = 0;
    *m.bad_flag = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
    int t = 0;
    if (lo < 0 || hi < lo || static_cast<int64_t>(hi) > rows_cap)
      *m.bad_flag = 1;
    else
      t = rows_per_tile > 0 ? (hi - lo + rows_per_tile - 1) / rows_per_tile : 1;
    m.tab[e + 1] = t;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    m.tab[0] = 0;
    for (int e = 0; e < E; ++e) m.tab[e + 1] += m.tab[e];
    if (*m.bad_flag && blockIdx.x == 0) set_status(status, MOE_DEV_BAD_OFFSETS);
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&m.full[s], 1);
      ptx::mbar_init(&m.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&m.tfull[a], 1);
      ptx::mbar_init(&m.tempty[a], 4);
    }
    ptx::mbar_init(m.drain, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  __syncthreads();
  return !*m.bad_flag;
}

// --------------------------------------------------------------------------------------------
// Row-tiled products: one tile = 128 rows of one expert x up to 256 accumulator columns.
//   DACT: out0 = dY W_down[e]                         A = dY [rows, h]     B = W_down [E h, d_e] MN
//   DGU:  (G | Up) = X W_gate^T | X W_up^T, then dG, dUp from d_act        B K-major as forward
//   DX:   out0 = dG W_gate[e] + dUp W_up[e]           A = dG | dUp        B = W_gate | W_up [E d_e, h] MN
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_bwd_rows(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                     const int32_t* __restrict__ offsets, int E, int K, int b_rows_per_expert, int n_out,
                     int64_t rows_cap, const bf16* __restrict__ d_act, bf16* __restrict__ out0,
                     bf16* __restrict__ out1, int32_t* status) {
  constexpr bool B_MN = MODE != DGU;
  constexpr int TILE_N = MODE == DGU ? BN / 2 : BN;
  extern __shared__ uint8_t smem_raw[];
  const Smem m = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = (n_out + TILE_N - 1) / TILE_N;
  const int KB1 = (K + BK - 1) / BK;           // k-blocks of one product
  const int KB = MODE == DX ? 2 * KB1 : KB1;   // DX: dG W_gate, then dUp W_up

  if (!setup(m, offsets, E, rows_cap, BM, status)) return;
  const int total = m.tab[E] * NT;
  if (static_cast<int>(blockIdx.x) >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(m.tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *m.tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA0);
      ptx::prefetch_tmap(&tmB0);
      if (MODE != DACT) {
        ptx::prefetch_tmap(&tmA1);
        ptx::prefetch_tmap(&tmB1);
      }
      const uint64_t pol_a = ptx::policy_evict_last();
      const uint64_t pol_b = ptx::policy_evict_normal();
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, nt, mt;
        decode_tile(m.tab, E, NT, tile, &e, &nt, &mt);
        const int a_row = seg_lo(offsets, e) + mt * BM;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&m.empty[stage], phase ^ 1u, m.abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* sa = m.stages + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          ptx::mbar_arrive_expect_tx(&m.full[stage], STAGE_BYTES);
          if (MODE == DGU) {
            const int b_row = e * b_rows_per_expert + nt * TILE_N;
            ptx::tma_load_2d(sa, &tmA0, kb * BK, a_row, &m.full[stage], pol_a);
            ptx::tma_load_2d(sb, &tmB0, kb * BK, b_row, &m.full[stage], pol_b);
            ptx::tma_load_2d(sb + B_BYTES / 2, &tmB1, kb * BK, b_row, &m.full[stage], pol_b);
          } else {
            const bool second = MODE == DX && kb >= KB1;
            const int kk = second ? kb - KB1 : kb;
            ptx::tma_load_2d(sa, second ? &tmA1 : &tmA0, kk * BK, a_row, &m.full[stage], pol_a);
            const CUtensorMap* tb = second ? &tmB1 : &tmB0;
            const int k_row = e * b_rows_per_expert + kk * BK;  // K index = weight row
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              ptx::tma_load_2d(sb + i * ATOM_BYTES, tb, nt * TILE_N + i * 64, k_row, &m.full[stage], pol_b);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) wait_drain(&m.full[s], (armed_phase >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc(BM, BN, false, B_MN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        if (!ptx::mbar_wait_bounded(&m.tempty[acc], acc_phase ^ 1u, m.abort_flag, WAIT_LIMIT_NS)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&m.full[stage], phase, m.abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(m.stages + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            const uint64_t ad = ptx::sdesc_kmajor_sw128(sa + kk * UK * 2);
            const uint64_t bd = B_MN ? sdesc_mn_sw128(sb + kk * UK * 128, ATOM_BYTES)
                                     : ptx::sdesc_kmajor_sw128(sb + kk * UK * 2);
            ptx::mma_bf16_ss(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(&m.empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&m.tfull[acc]);
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      ptx::mma_commit(m.drain);
      wait_drain(m.drain, 0);
    }
    __syncwarp();
  } else {
    const int q = warp & 3;
    const int r_local = q * 32 + lane;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, nt, mt;
      decode_tile(m.tab, E, NT, tile, &e, &nt, &mt);
      const int seg = seg_lo(offsets, e);
      const int n_e = seg_hi(offsets, e, rows_cap) - seg;
      const bool row_ok = mt * BM + r_local < n_e;
      const int64_t row = static_cast<int64_t>(seg) + mt * BM + r_local;
      const bool ready = ptx::mbar_wait_bounded(&m.tfull[acc], acc_phase, m.abort_flag, WAIT_LIMIT_NS);
      if (!__all_sync(0xffffffffu, ready)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      if (MODE == DGU) {
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gv[32], uv[32], pg[16], pu[16];
          ptx::tmem_ld_32x32b_x32(tb + c, gv);
          ptx::tmem_ld_32x32b_x32(tb + BN / 2 + c, uv);
          ptx::tmem_wait_ld();
          const int col0 = nt * TILE_N + c;
          float da[32];
          if (row_ok && col0 + 32 <= n_out) {
            const uint4* src = reinterpret_cast<const uint4*>(d_act + row * n_out + col0);
#pragma unroll
            for (int i = 0; i < 4; ++i) Vec16<bf16>::unpack(src[i], da + 8 * i);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) da[i] = (row_ok && col0 + i < n_out) ? to_f32(d_act[row * n_out + col0 + i]) : 0.f;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float dg[2], du[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const float g = __uint_as_float(gv[2 * i + h2]), u = __uint_as_float(uv[2 * i + h2]);
              const float s = __fdividef(1.f, 1.f + __expf(-g));
              const float d = da[2 * i + h2];
              du[h2] = d * g * s;
              dg[h2] = d * u * s * fmaf(g, 1.f - s, 1.f);
            }
            pg[i] = Vec16<bf16>::pack2(dg[0], dg[1]);
            pu[i] = Vec16<bf16>::pack2(du[0], du[1]);
          }
          if (row_ok) {
            store_32(out0 + row * n_out, col0, n_out, pg);
            store_32(out1 + row * n_out, col0, n_out, pu);
          }
        }
      } else {
        bf16* orow = out0 + row * n_out;
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
      if (lane == 0) ptx::mbar_arrive(&m.tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *m.abort_flag) set_status(status, MOE_DEV_TIMEOUT);
}

// --------------------------------------------------------------------------------------------
// Weight gradients: out[e][m][n] = sum over the rows r of expert e of A[r][m] B[r][n]
// (A, B row-major activations, read MN-major), float32 output [E, M, N].  One tile = 128 x 256
// of one expert; every expert has M/128 x N/256 tiles, an expert with no rows writes zeros.
// TMA store of a shared block to a 3D tensor at (x, y, z), tracked in this thread's bulk group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, const void* smem_src, int32_t x, int32_t y,
                                             int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(ptx::smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(THREADS, 1)
    grouped_wgrad(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmOut, const int32_t* __restrict__ offsets, int E, int M,
                  int N, int64_t rows_cap, float* __restrict__ out, bool tma_out, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  const Smem m = carve(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int MT = (M + BM - 1) / BM, NT = (N + BN - 1) / BN;
  if (!setup(m, offsets, E, rows_cap, 0, status)) return;
  const int total = E * MT * NT;
  if (static_cast<int>(blockIdx.x) >= total) return;

  if (warp == 1) {
    ptx::tmem_alloc(m.tmem_holder, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *m.tmem_holder;

  auto decode = [&](int tile, int* e, int* mt, int* nt) {
    *e = tile / (MT * NT);
    const int r = tile - *e * (MT * NT);
    *mt = r / NT;
    *nt = r - *mt * NT;
  };

  if (warp == 0) {
    if (lane == 0) {
      ptx::prefetch_tmap(&tmA);
      ptx::prefetch_tmap(&tmB);
      const uint64_t pol = ptx::policy_evict_normal();
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, mt, nt;
        decode(tile, &e, &mt, &nt);
        const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
        const int KB = (hi - lo + BK - 1) / BK;
        for (int kb = 0; kb < KB; ++kb) {
          if (!ptx::mbar_wait_bounded(&m.empty[stage], phase ^ 1u, m.abort_flag, WAIT_LIMIT_NS)) {
            ok = false;
            break;
          }
          uint8_t* sa = m.stages + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          ptx::mbar_arrive_expect_tx(&m.full[stage], STAGE_BYTES);
          const int r0 = lo + kb * BK;
#pragma unroll
          for (int i = 0; i < BM / 64; ++i)
            ptx::tma_load_2d(sa + i * ATOM_BYTES, &tmA, mt * BM + i * 64, r0, &m.full[stage], pol);
#pragma unroll
          for (int i = 0; i < BN / 64; ++i)
            ptx::tma_load_2d(sb + i * ATOM_BYTES, &tmB, nt * BN + i * 64, r0, &m.full[stage], pol);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((armed >> s) & 1u) wait_drain(&m.full[s], (armed_phase >> s) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // the whole warp: it zeroes the rows past a segment in the last k-block; lane 0 issues the MMAs
    constexpr uint32_t IDESC = idesc(BM, BN, true, true);
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int e, mt, nt;
      decode(tile, &e, &mt, &nt);
      const int lo = seg_lo(offsets, e), hi = seg_hi(offsets, e, rows_cap);
      const int KB = (hi - lo + BK - 1) / BK;
      const bool ready = ptx::mbar_wait_bounded(&m.tempty[acc], acc_phase ^ 1u, m.abort_flag, WAIT_LIMIT_NS);
      if (!__all_sync(0xffffffffu, ready)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
      for (int kb = 0; kb < KB; ++kb) {
        const bool got = ptx::mbar_wait_bounded(&m.full[stage], phase, m.abort_flag, WAIT_LIMIT_NS);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        uint8_t* sa_p = m.stages + stage * STAGE_BYTES;
        const int valid = min(BK, hi - (lo + kb * BK));
        if (valid < BK) {
          // K-row r of every atom is the 128-byte line at r * 128 (the swizzle stays inside the line)
          const int lines = (BK - valid) * (BM / 64 + BN / 64);
          for (int i = lane; i < lines * 8; i += 32) {
            const int li = i >> 3, part = i & 7;
            const int atom = li / (BK - valid), r = valid + li % (BK - valid);
            uint4* dst = reinterpret_cast<uint4*>(sa_p + atom * ATOM_BYTES + r * 128 + part * 16);
            *dst = make_uint4(0u, 0u, 0u, 0u);
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(sa_p);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk)
            ptx::mma_bf16_ss(d_tmem, sdesc_mn_sw128(sa + kk * UK * 128, ATOM_BYTES),
                             sdesc_mn_sw128(sb + kk * UK * 128, ATOM_BYTES), IDESC, (kb | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(&m.empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) ptx::mma_commit(&m.tfull[acc]);
      __syncwarp();
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) {
      ptx::mma_commit(m.drain);
      wait_drain(m.drain, 0);
    }
    __syncwarp();
  } else {
    // Each warp moves its 32 rows x 32 columns of the accumulator through a 4 KB shared block
    // (128-byte swizzle: row r's 16-byte chunk i at r * 128 + ((i ^ (r & 7)) << 4)) and one TMA
    // store writes the block as whole 128-byte rows of dW[e]; the [E, M, N] tensor map clips rows
    // past M and columns past N.  Before a block is refilled, the previous store has read it.
    const int q = warp & 3;
    uint8_t* blk = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u) + W_STAGING_OFFSET + q * 4096;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      int e, mt, nt;
      decode(tile, &e, &mt, &nt);
      const bool empty_seg = seg_hi(offsets, e, rows_cap) == seg_lo(offsets, e);
      const bool ready = ptx::mbar_wait_bounded(&m.tfull[acc], acc_phase, m.abort_flag, WAIT_LIMIT_NS);
      if (!__all_sync(0xffffffffu, ready)) break;
      ptx::tc_fence_after();
      const uint32_t tb = tmem_base + acc * ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(tb + c, v);
        ptx::tmem_wait_ld();
        const int col0 = nt * BN + c;
        if (col0 >= N) break;  // (warp-uniform)
        if (!tma_out) {
          // rows whose length is not a multiple of 4 floats: plain stores
          const int mrow = mt * BM + q * 32 + lane;
          if (mrow < M) {
            float* orow = out + (static_cast<int64_t>(e) * M + mrow) * N;
            for (int i = 0; i < 32 && col0 + i < N; ++i) orow[col0 + i] = empty_seg ? 0.f : __uint_as_float(v[i]);
          }
          continue;
        }
        if (lane == 0) bulk_wait_read0();  // the block's previous store has read it
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 val = empty_seg ? make_float4(0.f, 0.f, 0.f, 0.f)
                                       : make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                                     __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          *reinterpret_cast<float4*>(blk + lane * 128 + ((i ^ (lane & 7)) << 4)) = val;
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&tmOut, blk, col0, mt * BM + q * 32, e);
          bulk_commit();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&m.tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();  // every store of this warp has completed
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  if (threadIdx.x == 0 && *m.abort_flag) set_status(status, MOE_DEV_TIMEOUT);
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

// Row-major bf16 [rows, cols], boxes of box_rows x box_cols (box_cols * 2 bytes = 128: one swizzle line).
static bool make_tmap(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_rows(int grid, const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b0,
                               const CUtensorMap& b1, const int32_t* offsets, int E, int K, int b_rows, int n_out,
                               int64_t rows_cap, const bf16* d_act, bf16* o0, bf16* o1, int32_t* status,
                               cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(grouped_bwd_rows<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  grouped_bwd_rows<MODE><<<grid, THREADS, SMEM_BYTES, s>>>(a0, a1, b0, b1, offsets, E, K, b_rows, n_out, rows_cap,
                                                           d_act, o0, o1, status);
  return cudaGetLastError();
}

// float32 [E, M, N] written in boxes of 32 x 32 with the 128-byte swizzle (TMA stores)
static bool make_tmap_out(CUtensorMap* tm, float* base, int E, int M, int N) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || N % 4 != 0 || reinterpret_cast<uintptr_t>(base) % 16 != 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(E)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(N) * 4, static_cast<cuuint64_t>(M) * N * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static cudaError_t launch_wgrad(int nsm, const CUtensorMap& a, const CUtensorMap& b, const int32_t* offsets, int E,
                                int M, int N, int64_t rows_cap, float* out, int32_t* status, cudaStream_t s) {
  CUtensorMap tm_out = {};
  const bool tma_out = make_tmap_out(&tm_out, out, E, M, N);  // false when N % 4 != 0
  cudaError_t e = cudaFuncSetAttribute(grouped_wgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(W_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>(E) * ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(std::min<int64_t>(nsm, tiles));
  grouped_wgrad<<<grid, THREADS, W_SMEM_BYTES, s>>>(a, b, tm_out, offsets, E, M, N, rows_cap, out, tma_out, status);
  return cudaGetLastError();
}

}  // namespace bwd

// out[M, N] (float32) = A^T B over `rows` rows, A [rows, M] and B [rows, N] bf16 row-major.
cudaError_t launch_dense_wgrad_tc(const void* A, const void* B, int64_t rows, int M, int N, float* out,
                                  int32_t* status, cudaStream_t s) {
  using namespace bwd;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A, static_cast<uint64_t>(rows), static_cast<uint64_t>(M), 64) ||
      !make_tmap(&tb, B, static_cast<uint64_t>(rows), static_cast<uint64_t>(N), 64))
    return cudaErrorNotSupported;
  return launch_wgrad(current_sm_count(), ta, tb, nullptr, 1, M, N, rows, out, status, s);
}

cudaError_t launch_ffn_backward_tc(const Plan& p, const void* X, const int32_t* offsets, const void* W_gate,
                                   const void* W_up, const void* W_down, const void* act, const void* dY,
                                   void* d_act, void* dG, void* dUp, void* dX, float* dW_gate, float* dW_up,
                                   float* dW_down, int32_t* status, cudaStream_t s) {
  using namespace bwd;
  if (p.Tk == 0) return cudaSuccess;
  const uint64_t Tk = static_cast<uint64_t>(p.Tk), E = static_cast<uint64_t>(p.E);
  CUtensorMap tm_dY, tm_X, tm_dact, tm_dG, tm_dUp, tm_Wd, tm_Wg_k, tm_Wu_k, tm_Wg_mn, tm_Wu_mn;
  CUtensorMap tm_dY_mn, tm_dG_mn, tm_dUp_mn, tm_act_mn, tm_X_mn;
  // row-tiled A operands (K-major boxes of 128 rows) and K-major forward weights (boxes of 128 rows)
  if (!make_tmap(&tm_dY, dY, Tk, p.h, BM) || !make_tmap(&tm_X, X, Tk, p.h, BM) ||
      !make_tmap(&tm_dG, dG, Tk, p.d_e, BM) || !make_tmap(&tm_dUp, dUp, Tk, p.d_e, BM) ||
      !make_tmap(&tm_Wg_k, W_gate, E * p.d_e, p.h, BN / 2) || !make_tmap(&tm_Wu_k, W_up, E * p.d_e, p.h, BN / 2) ||
      // MN-major reads (boxes of 64 K-rows x 64 N): the weights as [K rows, N cols], the activations
      !make_tmap(&tm_Wd, W_down, E * p.h, p.d_e, 64) || !make_tmap(&tm_Wg_mn, W_gate, E * p.d_e, p.h, 64) ||
      !make_tmap(&tm_Wu_mn, W_up, E * p.d_e, p.h, 64) || !make_tmap(&tm_dY_mn, dY, Tk, p.h, 64) ||
      !make_tmap(&tm_dG_mn, dG, Tk, p.d_e, 64) || !make_tmap(&tm_dUp_mn, dUp, Tk, p.d_e, 64) ||
      !make_tmap(&tm_act_mn, act, Tk, p.d_e, 64) || !make_tmap(&tm_X_mn, X, Tk, p.h, 64))
    return cudaErrorNotSupported;
  (void)tm_dact;
  const int nsm = current_sm_count();
  const int64_t mtiles = (p.Tk + BM - 1) / BM + p.E;
  auto grid_for = [&](int n_out, int tile_n) {
    const int64_t t = mtiles * ((n_out + tile_n - 1) / tile_n);
    return static_cast<int>(std::min<int64_t>(nsm, t));
  };
  // d_act = dY W_down[e]
  cudaError_t e = launch_rows<DACT>(grid_for(p.d_e, BN), tm_dY, tm_dY, tm_Wd, tm_Wd, offsets, p.E, p.h, p.h, p.d_e,
                                    p.Tk, nullptr, static_cast<bf16*>(d_act), nullptr, status, s);
  if (e != cudaSuccess) return e;
  // dG, dUp from the recomputed gate|up product and d_act
  e = launch_rows<DGU>(grid_for(p.d_e, BN / 2), tm_X, tm_X, tm_Wg_k, tm_Wu_k, offsets, p.E, p.h, p.d_e, p.d_e, p.Tk,
                       static_cast<const bf16*>(d_act), static_cast<bf16*>(dG), static_cast<bf16*>(dUp), status, s);
  if (e != cudaSuccess) return e;
  // dX = dG W_gate[e] + dUp W_up[e]
  e = launch_rows<DX>(grid_for(p.h, BN), tm_dG, tm_dUp, tm_Wg_mn, tm_Wu_mn, offsets, p.E, p.d_e, p.d_e, p.h, p.Tk,
                      nullptr, static_cast<bf16*>(dX), nullptr, status, s);
  if (e != cudaSuccess) return e;
  // weight gradients
  e = launch_wgrad(nsm, tm_dY_mn, tm_act_mn, offsets, p.E, p.h, p.d_e, p.Tk, dW_down, status, s);
  if (e != cudaSuccess) return e;
  e = launch_wgrad(nsm, tm_dG_mn, tm_X_mn, offsets, p.E, p.d_e, p.h, p.Tk, dW_gate, status, s);
  if (e != cudaSuccess) return e;
  return launch_wgrad(nsm, tm_dUp_mn, tm_X_mn, offsets, p.E, p.d_e, p.h, p.Tk, dW_up, status, s);
}

}  // namespace moe
