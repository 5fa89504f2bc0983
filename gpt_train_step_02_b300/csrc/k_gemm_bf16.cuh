// k_gemm_bf16.cuh -- bf16-operand matmul on the 5th-generation tensor cores
// (tcgen05.mma kind::f16 with bf16 inputs, fp32 accumulator in TMEM), fed by
// TMA, persistent over output tiles.
//
//   acc(i,j) = sum_k A(i,k) B(j,k),  i < M, j < N, k < K,
// with each operand stored K-major (row i holds its K values contiguously)
// or MN-major (row k holds the M or N values contiguously), bf16 in global
// memory.  The three products of a linear layer map onto it as
//   forward          A = x  (K-major), B = W   (K-major)
//   input gradient   A = dy (K-major), B = W   (MN-major)
//   weight gradient  A = dy (MN-major), B = x  (MN-major).
// MN-major operands need no transpose pass: the tensor core reads them
// through the matrix descriptor's MN-major layout (instruction-descriptor
// transpose bits).
//
// Work unit = (128 x BN output tile, BN = 128, 192 or 256; K split); a CTA walks the units
// blockIdx.x, blockIdx.x + gridDim.x, ...  Ten or fourteen warps:
//   warp 0      one lane issues the TMA loads into a STAGES-deep ring
//   warp 1      allocates TMEM; one lane issues the MMAs (K = 16 per
//               instruction, four per 64-wide K tile) into one of two TMEM
//               accumulators, so the epilogue of unit u overlaps the MMAs of
//               unit u + 1
//   warps 2..    epilogue (two or three warps per TMEM lane quadrant, a
//               share of the columns each): tcgen05.ld TMEM -> registers -> shared-memory
//               transpose -> fused epilogue -> coalesced global stores; K-split
//               units hand off through partial tiles and an
//               arrival counter, the last unit to arrive reducing in split
//               order (deterministic).
// Shared-memory layouts (128-byte swizzle, as TMA writes them):
//   K-major tile   rows of 64 bf16 (128 B); 8-row atoms of 1024 B (SBO);
//                  the MMA's K step advances the start address by 32 B.
//   MN-major tile  one 64(MN) x 64(K) box per 8 KB: rows of 64 MN values
//                  (128 B) per k; 8-k atoms of 1024 B (SBO); the next 64 MN
//                  values 8 KB further (LBO); the MMA's K step (16 k)
//                  advances the start address by 2048 B.
// Every mbarrier wait is bounded (1 s of global-timer time); on expiry the
// CTA records DEV_ERR_TIMEOUT, lets its copies and MMAs in flight land,
// frees its TMEM and returns.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "k_gemm_tc.cuh"

namespace tcb {
using tc::globaltimer_ns;
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_try_wait;
using tc::mbar_wait;
using tc::mbar_wait_drain;
using tc::mma_commit;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tma_load_2d;
using tc::tmem_ld32;

constexpr int BM = 128;
constexpr int BK = 64;  // bf16 elements per K tile: 128 bytes, one swizzle row
constexpr int UMMA_K = 16;
constexpr int MN_BOX = 64;                   // MN extent of one MN-major TMA box
constexpr int MN_BOX_BYTES = MN_BOX * BK * 2;  // 8 KB

// The epilogues with per-element arithmetic or inputs (GELU, GELU', bias +
// residual) are bound by their instruction issue on the products with few K
// tiles (K = C): there they run with EG = 4 (GELU, GELU') or 3 (residual)
// epilogue warps per TMEM lane quadrant instead of 2, at the cost of one
// operand stage of shared memory (the host picks EG per launch).
__host__ __device__ constexpr bool heavy_epilogue(int op) {
  return op == EPI_BIAS_GELU || op == EPI_DGELU || op == EPI_BIAS_RESID;
}
__host__ __device__ constexpr int heavy_epilogue_groups(int op) { return op == EPI_BIAS_RESID ? 3 : 4; }

template <int BN, int OP = EPI_STORE, int EG = 2>
struct Cfg {
  static constexpr int EPI_GROUPS = EG;            // epilogue warps per TMEM lane quadrant
  static constexpr bool STRIDED = EG != 2;         // chunks dealt round-robin instead of by half tile
  static constexpr int EPI_WARPS = 4 * EPI_GROUPS;
  static constexpr int EPI_THREADS = 32 * EPI_WARPS;
  static constexpr int THREADS = 64 + EPI_THREADS;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // as many 64-wide K tiles in flight (at most 6) as fit 227 KB beside the
  // epilogue's staging, the barriers and the alignment slack
  static constexpr int STAGING_BYTES = EPI_WARPS * EPI_STAGE_FLOATS * 4;
  static constexpr int STAGES_FIT = (232448 - 1024 - 256 - STAGING_BYTES) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT < 6 ? STAGES_FIT : 6;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  // full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], mma_done
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_EPI = (OFF_MISC + 64 + 15) / 16 * 16;  // the epilogue warps' staging
  static constexpr int SMEM_BYTES = OFF_EPI + EPI_WARPS * EPI_STAGE_FLOATS * 4 + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "227 KB of shared memory per CTA");
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // two accumulators (a power of two)
};

struct Params {
  int M, N, K;
  int a_kmajor, b_kmajor;
  int k_tiles, kt_per_split, splits;
  int tiles_m, tiles_n, units;
  EpiArgs epi;
  float* partial;  // split-K partials [splits][M][N] (splits > 1)
  int* tile_ctr;   // split-K arrival counters, one per output tile, zero between launches
  int* err;
};

// Shared-memory matrix descriptor, 128-byte swizzle, version 1.
GPT2_DEV uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 128, N = BN,
// bit 15 / 16 set for an MN-major A / B.
template <int BN>
GPT2_DEV uint32_t idesc_bf16(int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

GPT2_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// unit -> (first row m0, column-tile index tn, K split z, output tile index).
// Consecutive units are the K splits of one tile, then tiles walk down M
// within one N column, so CTAs running at the same time share the B tile
// (the weights, in the forward product).
GPT2_DEV void unit_coords(const Params& p, int unit, int& m0, int& tn, int& z, int& tile) {
  z = unit % p.splits;
  tile = unit / p.splits;
  m0 = (tile % p.tiles_m) * BM;
  tn = tile / p.tiles_m;
}

// Softmax statistics of one row's 32 logits v (columns j0 .. j0+31) merged
// into the running (m, s): m the largest logit of a real column (j < V), s the
// sum of exp(logit - m) over them.  The target column's logit goes to *tl.
GPT2_DEV void logits_row_stats(const float* v, int j0, int V, int tgt, float& m, float& s, float* tl) {
  float cm = -INFINITY;
#pragma unroll
  for (int k = 0; k < 32; k++)
    if (j0 + k < V) cm = fmaxf(cm, v[k]);
  if (cm != -INFINITY) {
    const float L2E = 1.4426950408889634f;
    const float nm = fmaxf(m, cm), nmb = nm * L2E;
    float cs = 0.f;
#pragma unroll
    for (int k = 0; k < 32; k++)
      if (j0 + k < V) cs += ex2f_fast(fmaf(v[k], L2E, -nmb));
    s = s * ex2f_fast((m - nm) * L2E) + cs;  // 0 * 0 while m = -inf
    m = nm;
  }
#pragma unroll
  for (int k = 0; k < 32; k++)
    if (j0 + k == tgt) *tl = v[k];
}

// OP: the epilogue kind (a GemmEpi value), fixed per instantiation
template <int BN, int OP, int EG>
__global__ void __launch_bounds__(Cfg<BN, OP, EG>::THREADS, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ Params p) {
  pdl_launch_dependents();
  using CF = Cfg<BN, OP, EG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + CF::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + CF::STAGES;
  uint64_t* acc_full = bars + 2 * CF::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + CF::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + CF::OFF_MISC + 4);
  volatile int* go_flag = reinterpret_cast<volatile int*>(smem + CF::OFF_MISC + 8);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + CF::OFF_MISC + 12);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < CF::STAGES; s++) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], CF::EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(CF::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the first global-memory access comes after this

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < p.units && ok; unit += gridDim.x) {
        int m0, tn, z, tile;
        unit_coords(p, unit, m0, tn, z, tile);
        const int n0 = tn * BN;
        const int kt0 = z * p.kt_per_split, kt1 = min(p.k_tiles, kt0 + p.kt_per_split);
        for (int kt = kt0; kt < kt1; kt++, it++) {
          const int s = it % CF::STAGES;
          if (!mbar_wait(&empty[s], ((it / CF::STAGES) & 1) ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&full[s], CF::STAGE_BYTES);
          uint8_t* sa = smem + s * CF::STAGE_BYTES;
          uint8_t* sb = sa + CF::A_BYTES;
          const int k = kt * BK;
          if (p.a_kmajor) {
            tma_load_2d(sa, &tmA, k, m0, &full[s]);
          } else {
#pragma unroll
            for (int c = 0; c < BM / MN_BOX; c++) tma_load_2d(sa + c * MN_BOX_BYTES, &tmA, m0 + c * MN_BOX, k, &full[s]);
          }
          if (p.b_kmajor) {
            tma_load_2d(sb, &tmB, k, n0, &full[s]);
          } else {
#pragma unroll
            for (int c = 0; c < BN / MN_BOX; c++) tma_load_2d(sb + c * MN_BOX_BYTES, &tmB, n0 + c * MN_BOX, k, &full[s]);
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        for (int j = max(0, it - CF::STAGES); j < it; j++) mbar_wait_drain(&full[j % CF::STAGES], (j / CF::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16<BN>(!p.a_kmajor, !p.b_kmajor);
      // K step of one MMA (16 bf16): 32 B along a K-major row, 16 rows of 128 B in an MN-major box
      const uint32_t a_kstep = p.a_kmajor ? 32u : 2048u, b_kstep = p.b_kmajor ? 32u : 2048u;
      const uint32_t a_lbo = p.a_kmajor ? 16u : (uint32_t)MN_BOX_BYTES;
      const uint32_t b_lbo = p.b_kmajor ? 16u : (uint32_t)MN_BOX_BYTES;
      int it = 0, lu = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < p.units && ok; unit += gridDim.x, lu++) {
        int m0, tn, z, tile;
        unit_coords(p, unit, m0, tn, z, tile);
        const int kt0 = z * p.kt_per_split, kt1 = min(p.k_tiles, kt0 + p.kt_per_split);
        const int buf = lu & 1;
        if (!mbar_wait(&acc_empty[buf], ((lu >> 1) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
        for (int kt = kt0; kt < kt1; kt++, it++) {
          const int s = it % CF::STAGES;
          if (!mbar_wait(&full[s], (it / CF::STAGES) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * CF::STAGE_BYTES);
          const uint32_t sb = sa + CF::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; kk++) {
            uint64_t da = desc_sw128(sa + kk * a_kstep, a_lbo, 1024);
            uint64_t db = desc_sw128(sb + kk * b_kstep, b_lbo, 1024);
            mma_bf16(d_tmem, da, db, idesc, (kt > kt0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);  // frees the stage once these MMAs have read it
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      // every MMA this thread issued has completed once mma_done fires
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    // ---------------- epilogue ----------------
    const int t = threadIdx.x - 64;          // 0 .. EPI_THREADS-1
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int grp = (warp - 2) / 4;          // which of the quadrant's EPI_GROUPS warps this is
    // its 32-column chunks: with two warps per quadrant the first or second
    // half of the tile (the LM head's row statistics are per half tile); with
    // more, every EG-th chunk
    constexpr int NCH = BN / 32;
    const int cc_first = CF::STRIDED ? grp : grp * (NCH / 2);
    const int cc_end = CF::STRIDED ? NCH : (grp + 1) * (NCH / 2);
    const int cc_step = CF::STRIDED ? CF::EPI_GROUPS : 1;
    int lu = 0;
    for (int unit = blockIdx.x; unit < p.units; unit += gridDim.x, lu++) {
      int m0, tn, z, tile;
      unit_coords(p, unit, m0, tn, z, tile);
      const int n0 = tn * BN;
      const int buf = lu & 1;
      bool ok = mbar_wait(&acc_full[buf], (lu >> 1) & 1, abort_flag, p.err);
      // one decision for all epilogue warps (tcgen05.ld is warp-collective
      // and the split-K hand-off uses a barrier over these threads)
      tc::epi_bar<CF::EPI_THREADS>();
      if (t == 0) *go_flag = (ok && !*abort_flag) ? 1 : 0;
      tc::epi_bar<CF::EPI_THREADS>();
      if (!*go_flag) break;
      tc_fence_after();
      const bool split = p.splits > 1;
      float* stage = reinterpret_cast<float*>(smem + CF::OFF_EPI) + (warp - 2) * EPI_STAGE_FLOATS;
      const int i0 = m0 + q * 32;  // this warp's 32 rows
      const uint32_t tbase = tmem + (uint32_t)(buf * BN) + ((uint32_t)(q * 32) << 16);
      // EPI_LOGITS: row i0 + lane's running (max, sum of exp) over this warp's
      // half of the tile, and its target column
      float xm = -INFINITY, xs = 0.f;
      int xt = -1;
      if constexpr (OP == EPI_LOGITS) xt = (i0 + lane < p.M) ? p.epi.targets[i0 + lane] : -1;
#pragma unroll 1
      for (int cc = cc_first; cc < cc_end; cc += cc_step) {
        float v[32];
        tmem_ld32(tbase + (uint32_t)(cc * 32), v);
        const int j0 = n0 + cc * 32;
        if (j0 >= p.N || i0 >= p.M) continue;  // warp-uniform
        if constexpr (OP == EPI_LOGITS) logits_row_stats(v, j0, p.epi.V, xt, xm, xs, p.epi.tlogit + i0 + lane);
        warp32_stage(stage, v, lane);
        if (split)
          warp32_store_raw(p.partial + (size_t)z * p.M * p.N, p.N, stage, i0, j0, p.M, p.N, lane);
        else
          warp32_epilogue<OP>(p.epi, stage, i0, j0, p.M, p.N, lane);
      }
      if constexpr (OP == EPI_LOGITS) {
        const int blk = tn * 2 + grp;  // this warp's BN/2 columns
        if (i0 + lane < p.M && blk * (BN / 2) < p.N)
          p.epi.xstats[(size_t)(i0 + lane) * p.epi.ldxs + blk] = make_float2(xm, xs);
      }
      // the accumulator is in registers / global memory now: hand it back
      tc_fence_before();
      tc::mbar_arrive_warp(&acc_empty[buf]);
      if (split) {
        __threadfence();
        tc::epi_bar<CF::EPI_THREADS>();
        if (t == 0) *last_flag = (atomicAdd(&p.tile_ctr[tile], 1) == p.splits - 1) ? 1 : 0;
        tc::epi_bar<CF::EPI_THREADS>();
        if (*last_flag) {
          __threadfence();
          const int ew = warp - 2;
          const size_t plane = (size_t)p.M * p.N;
          for (int r = ew; r < BM && m0 + r < p.M; r += CF::EPI_WARPS) {
            const int ii = m0 + r;
            for (int jj = 4 * lane; jj < BN; jj += 128) {
              const int j = n0 + jj;
              if (j >= p.N) break;
              const float* src = p.partial + (size_t)ii * p.N + j;
              if (j + 4 <= p.N && (p.N & 3) == 0) {
                float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
                for (int zz = 1; zz < p.splits; zz++) {
                  float4 b = __ldcg(reinterpret_cast<const float4*>(src + zz * plane));
                  acc.x += b.x; acc.y += b.y; acc.z += b.z; acc.w += b.w;
                }
                epi_store4<OP>(p.epi, ii, j, acc);
              } else {
                for (int c = 0; c < 4 && j + c < p.N; c++) {
                  float a = __ldcg(src + c);
                  for (int zz = 1; zz < p.splits; zz++) a += __ldcg(src + c + zz * plane);
                  epi_store<OP>(p.epi, ii, j + c, a);
                }
              }
            }
          }
          if (t == 0) p.tile_ctr[tile] = 0;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(CF::TMEM_COLS)
                 : "memory");
  }
}

}  // namespace tcb
