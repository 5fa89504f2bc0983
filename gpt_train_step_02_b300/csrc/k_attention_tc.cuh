// k_attention_tc.cuh -- causal attention forward on the tensor cores (bf16
// operands, fp32 softmax), head size 64, T a multiple of 128.
//
// Per (batch b, head h, tile of 128 queries): for each key tile j <= the
// query tile (causal),
//   S   = Q K_j^T * scale                  tcgen05.mma kind::f16 -> TMEM
//   m'  = max(m, rowmax S);  P = exp(S - m');  l = l e^(m-m') + rowsum P
//   O   = O e^(m-m') + P V_j                P (bf16) staged in shared memory,
//                                           P V_j -> TMEM -> registers
// and at the end y = O / l, lse = m + log l (the log-sum-exp of the scaled
// scores, as the backward pass expects).  Keys t2 > t of the diagonal tile
// are masked.  This is the online-softmax form of attention (the page «llm.c：
// Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c», item 1,
// attention_forward computes the same causal softmax(q k^T / sqrt(hs)) v).
//
// Operands come from a bf16 copy of qkv, (B*T, 3C) row-major, through one
// TMA map with 64 x 128 boxes (128-byte swizzle): Q and K tiles are K-major
// (a row of 64 head dims per token); the V tile is read MN-major by the PV
// product (rows of 64 head dims per key = the N dimension contiguous).
// Six warps: warp 0 issues the TMA loads (Q once, K double-buffered, V
// single-buffered so that two CTAs fit one SM);
// warp 1 allocates TMEM and issues the MMAs; warps 2..5 own one query row
// per thread (TMEM lane = row) for the softmax and the output.  Every
// mbarrier wait is bounded (1 s); on expiry the CTA records DEV_ERR_TIMEOUT,
// drains its copies and MMAs and returns.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "k_gemm_bf16.cuh"

namespace tca {
using tc::mbar_arrive;
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_drain;
using tc::mma_commit;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tma_load_2d;
using tc::tmem_ld32;
using tcb::desc_sw128;
using tcb::mma_bf16;

constexpr int BQ = 128;   // queries per CTA
constexpr int BKV = 128;  // keys per tile
constexpr int HS = 64;    // head size
constexpr int THREADS = 192;
constexpr int TILE_BYTES = 128 * HS * 2;  // 16 KB: a Q, K or V tile
namespace fwd {
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;          // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;      // 1 stage (its load waits only on the previous P V)
constexpr int OFF_P = OFF_V + TILE_BYTES;          // 128 x 128 bf16 = two 16 KB K chunks
constexpr int OFF_BAR = OFF_P + 2 * TILE_BYTES;
// q_full, k_full[2], k_empty[2], v_full, v_empty, s_full, p_full, pv_full, mma_done
constexpr int NUM_BARS = 11;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES + 1024 <= 233472 / 2, "two CTAs per SM");
}  // namespace fwd
constexpr int TMEM_COLS = 256;  // forward: S in columns [0, 128), P V in [128, 192)

struct Params {
  int B, T, C, NH;
  float scale;     // 1/sqrt(hs)
  float* y;        // (B, T, C) fp32
  uint16_t* ybf;   // (B, T, C) bf16 copy, or NULL
  float* lse;      // (B, NH, T)
  int* err;
};

// Instruction descriptors: S = Q K^T (M 128, N 128, both K-major);
// O += P V (M 128, N 64, V MN-major).
constexpr uint32_t IDESC_S = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BKV >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);
constexpr uint32_t IDESC_PV =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(HS >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);

__global__ void __launch_bounds__(THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ Params p) {
  pdl_launch_dependents();
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 5;
  uint64_t* v_empty = bars + 6;
  uint64_t* s_full = bars + 7;
  uint64_t* p_full = bars + 8;
  uint64_t* pv_full = bars + 9;
  uint64_t* mma_done = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqt = p.T / BQ;
  const int qt = nqt - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int nkt = qt + 1;                    // key tiles 0..qt
  const int row0 = b * p.T + qt * BQ;        // first query row in (B*T)

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(pv_full, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
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
      mbar_expect_tx(q_full, TILE_BYTES);
      tma_load_2d(smem + OFF_Q, &tmQKV, h * HS, row0, q_full);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < nkt; j++) {
        const int s = j & 1;
        const int krow = b * p.T + j * BKV;
        if (!mbar_wait(&k_empty[s], ((j >> 1) & 1) ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(&k_full[s], TILE_BYTES);
        tma_load_2d(smem + OFF_K + s * TILE_BYTES, &tmQKV, p.C + h * HS, krow, &k_full[s]);
        k_issued = j + 1;
        if (!mbar_wait(v_empty, (j & 1) ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(v_full, TILE_BYTES);
        tma_load_2d(smem + OFF_V, &tmQKV, 2 * p.C + h * HS, krow, v_full);
        v_issued = j + 1;
      }
      if (*abort_flag) {
        mbar_wait_drain(q_full, 0);
        for (int j = max(0, k_issued - 2); j < k_issued; j++) mbar_wait_drain(&k_full[j & 1], (j >> 1) & 1);
        if (v_issued > 0) mbar_wait_drain(v_full, (v_issued - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t sq = smem_u32(smem + OFF_Q), sp = smem_u32(smem + OFF_P);
      const uint32_t t_s = tmem, t_pv = tmem + 128;
      bool ok = mbar_wait(q_full, 0, abort_flag, p.err);
      for (int j = 0; j < nkt && ok; j++) {
        const int s = j & 1;
        if (!mbar_wait(&k_full[s], (j >> 1) & 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t sk = smem_u32(smem + OFF_K + s * TILE_BYTES), sv = smem_u32(smem + OFF_V);
        // S = Q K^T over the 64 head dims (four K = 16 steps along the 128-byte rows)
#pragma unroll
        for (int kk = 0; kk < HS / 16; kk++)
          mma_bf16(t_s, desc_sw128(sq + kk * 32, 16, 1024), desc_sw128(sk + kk * 32, 16, 1024), IDESC_S,
                   kk > 0 ? 1u : 0u);
        mma_commit(s_full);
        mma_commit(&k_empty[s]);
        // P (written by the softmax warps) times V over the 128 keys
        if (!mbar_wait(p_full, j & 1, abort_flag, p.err)) break;
        if (!mbar_wait(v_full, j & 1, abort_flag, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; kk++) {
          const uint32_t pa = sp + (kk >> 2) * TILE_BYTES + (kk & 3) * 32;  // two 64-key chunks
          mma_bf16(t_pv, desc_sw128(pa, 16, 1024), desc_sw128(sv + kk * 2048, 8192, 1024), IDESC_PV,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(pv_full);
        mma_commit(v_empty);
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    // ---------------- softmax + output: one query row per thread ----------------
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // row within the tile = TMEM lane
    const int t = qt * BQ + r;     // query position
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;  // scale * log2(e)
    float o[HS];
#pragma unroll
    for (int d = 0; d < HS; d++) o[d] = 0.f;
    float mrow = -INFINITY, lrow = 0.f;  // running max (of scaled scores) and sum
    bool ok = true;
    uint8_t* prow = smem + OFF_P + r * 128;
    for (int j = 0; j < nkt; j++) {
      if (!tc::epi_bar_and<128>(mbar_wait(s_full, j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = j == qt;
      const int kbase = j * BKV - t;  // key k of this tile lies after the query when kbase + k > 0
      // pass 1: row max of this tile's scores (TMEM read in 32-column chunks)
      float mt = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < BKV / 32; c++) {
        float sv[32];
        tmem_ld32(tmem + lane_off + c * 32, sv);
#pragma unroll
        for (int k = 0; k < 32; k++)
          if (!diag || kbase + c * 32 + k <= 0) mt = fmaxf(mt, sv[k]);
      }
      const float mnew = fmaxf(mrow, mt * p.scale);
      const float corr = exp2f((mrow - mnew) * 1.4426950408889634f);  // 0 on the first tile
      const float mb = mnew * 1.4426950408889634f;
      float lsum = 0.f;
      // pass 2: P = exp(s*scale - mnew) as bf16 into the swizzled K-major P
      // tile (two 64-key chunks of 16 KB; 16-byte groups XOR-swizzled by row)
#pragma unroll 1
      for (int c = 0; c < BKV / 32; c++) {
        float sv[32];
        tmem_ld32(tmem + lane_off + c * 32, sv);
#pragma unroll
        for (int g = 0; g < 4; g++) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; e++) {
            const int k = g * 8 + 2 * e;
            const bool m0 = diag && kbase + c * 32 + k > 0, m1 = diag && kbase + c * 32 + k + 1 > 0;
            float p0 = m0 ? 0.f : exp2f(sv[k] * sl2 - mb), p1 = m1 ? 0.f : exp2f(sv[k + 1] * sl2 - mb);
            uint16_t h0 = to_bf16_bits(p0), h1 = to_bf16_bits(p1);
            // the row sum uses the bf16-rounded weights that the PV product uses
            lsum += __uint_as_float((uint32_t)h0 << 16) + __uint_as_float((uint32_t)h1 << 16);
            w[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
          }
          const int key16 = c * 4 + g;  // 16-byte group of 8 keys, 0..15
          const int chunk = key16 >> 3, grp = key16 & 7;
          *reinterpret_cast<uint4*>(prow + chunk * TILE_BYTES + ((grp ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      lrow = lrow * corr + lsum;
      mrow = mnew;
      // make the generic-proxy P writes visible to the tensor core
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(p_full);
      if (!tc::epi_bar_and<128>(mbar_wait(pv_full, j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < HS / 32; hh++) {
        float pv[32];
        tmem_ld32(tmem + 128 + lane_off + hh * 32, pv);
#pragma unroll
        for (int d = 0; d < 32; d++) o[hh * 32 + d] = o[hh * 32 + d] * corr + pv[d];
      }
    }
    if (tc::epi_bar_and<128>(ok && !*abort_flag)) {
      const float inv = 1.f / lrow;
      const size_t yo = (size_t)(row0 + r) * p.C + h * HS;
#pragma unroll
      for (int d = 0; d < HS; d += 4)
        *reinterpret_cast<float4*>(p.y + yo + d) = make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
      if (p.ybf) {
#pragma unroll
        for (int d = 0; d < HS; d += 8) {
          uint4 w;
          w.x = (uint32_t)to_bf16_bits(o[d] * inv) | ((uint32_t)to_bf16_bits(o[d + 1] * inv) << 16);
          w.y = (uint32_t)to_bf16_bits(o[d + 2] * inv) | ((uint32_t)to_bf16_bits(o[d + 3] * inv) << 16);
          w.z = (uint32_t)to_bf16_bits(o[d + 4] * inv) | ((uint32_t)to_bf16_bits(o[d + 5] * inv) << 16);
          w.w = (uint32_t)to_bf16_bits(o[d + 6] * inv) | ((uint32_t)to_bf16_bits(o[d + 7] * inv) << 16);
          *reinterpret_cast<uint4*>(p.ybf + yo + d) = w;
        }
      }
      p.lse[((size_t)b * p.NH + h) * p.T + t] = mrow + logf(lrow);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}


// ---------------------------------------------------------------------------
// Backward (the page's attention_backward), bf16 operands, head size 64,
// T % 128 == 0.  With P = exp(S*scale - lse) recomputed from the saved
// log-sum-exp, dP = dO V^T, D = rowsum(dO o y) and dS = P o (dP - D):
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// Two kernels, each output row produced by one CTA (no atomics, so the
// result is deterministic):
//   attn_bwd_dkv_tc_kernel  CTA per (key tile, head, batch); walks the query
//       tiles at or after the key tile: S^T = K Q^T, dP^T = V dO^T in TMEM,
//       P^T and dS^T (bf16) staged in shared memory, dV += P^T dO and
//       dK += dS^T Q accumulated in TMEM.
//   attn_bwd_dq_tc_kernel   CTA per (query tile, head, batch); walks the key
//       tiles at or before it: S = Q K^T, dP = dO V^T, dS staged,
//       dQ += dS K in TMEM.
// Operand tiles come from the bf16 copies of qkv and of dO (the gradient of
// the attention output, (B*T, C)), each through a TMA map with 64 x 128
// boxes.  Q, K, V, dO tiles are K-major for the score products and read
// MN-major as the B operand of the accumulating products.
// ---------------------------------------------------------------------------
struct BwdParams {
  int B, T, C, NH;
  float scale;
  const float* lse;  // (B, NH, T)
  const float* D;    // (B, NH, T)
  float* dqkv;       // (B, T, 3C) fp32
  uint16_t* dqkv_bf; // (B, T, 3C) bf16 copy, or NULL
  int* err;
};

// Writes 32 consecutive bf16 values (keys or queries c*32 .. c*32+31 of a
// 128-wide row r) into a K-major, 128-byte-swizzled 128 x 128 tile made of
// two 64-column chunks of 16 KB.
GPT2_DEV void st_row32_sw128(uint8_t* tile, int r, int c, const uint32_t (&w)[16]) {
#pragma unroll
  for (int g = 0; g < 4; g++) {
    const int key16 = c * 4 + g, chunk = key16 >> 3, grp = key16 & 7;
    *reinterpret_cast<uint4*>(tile + chunk * TILE_BYTES + r * 128 + ((grp ^ (r & 7)) << 4)) =
        make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
  }
}

GPT2_DEV uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)to_bf16_bits(a) | ((uint32_t)to_bf16_bits(b) << 16);
}

// 128 x 128 K-major A operand in two 64-column chunks: descriptor of K step kk
GPT2_DEV uint64_t desc_a128(uint32_t base, int kk) {
  return desc_sw128(base + (kk >> 2) * TILE_BYTES + (kk & 3) * 32, 16, 1024);
}

constexpr uint32_t IDESC_SS = IDESC_S;   // 128 x 128 scores, both K-major
constexpr uint32_t IDESC_ACC = IDESC_PV; // 128 x 64 accumulation, B MN-major

namespace dkv {
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + TILE_BYTES;
constexpr int OFF_Q = OFF_V + TILE_BYTES;        // 2 stages
constexpr int OFF_DO = OFF_Q + 2 * TILE_BYTES;   // 2 stages
constexpr int OFF_PT = OFF_DO + 2 * TILE_BYTES;  // P^T, 128 x 128 bf16
constexpr int OFF_DST = OFF_PT + 2 * TILE_BYTES; // dS^T, 128 x 128 bf16
constexpr int OFF_LD = OFF_DST + 2 * TILE_BYTES; // lse and D of one query tile (2 x 128 floats)
constexpr int OFF_BAR = OFF_LD + 2 * 128 * 4;
// kv_full, qd_full[2], qd_empty[2], s_full, st_ready, mma_done
constexpr int NUM_BARS = 8;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
}  // namespace dkv

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                           const __grid_constant__ BwdParams p) {
  pdl_launch_dependents();
  using namespace dkv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* qd_full = bars + 1;
  uint64_t* qd_empty = bars + 3;
  uint64_t* s_full = bars + 5;
  uint64_t* st_ready = bars + 6;
  uint64_t* mma_done = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = p.T / BKV;
  const int kt = (int)blockIdx.x;  // key tile; walks query tiles kt .. nt-1
  const int h = blockIdx.y, b = blockIdx.z;
  const int niter = nt - kt;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(st_ready, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the first global-memory access comes after this
  const uint32_t T_ST = tmem, T_DPT = tmem + 128, T_DV = tmem + 256, T_DK = tmem + 320;

  if (warp == 0) {
    if (lane == 0) {
      const int krow = b * p.T + kt * BKV;
      mbar_expect_tx(kv_full, 2 * TILE_BYTES);
      tma_load_2d(smem + OFF_K, &tmQKV, p.C + h * HS, krow, kv_full);
      tma_load_2d(smem + OFF_V, &tmQKV, 2 * p.C + h * HS, krow, kv_full);
      int issued = 0;
      for (int i = 0; i < niter; i++) {
        const int s = i & 1, qrow = b * p.T + (kt + i) * BQ;
        if (!mbar_wait(&qd_empty[s], ((i >> 1) & 1) ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(&qd_full[s], 2 * TILE_BYTES);
        tma_load_2d(smem + OFF_Q + s * TILE_BYTES, &tmQKV, h * HS, qrow, &qd_full[s]);
        tma_load_2d(smem + OFF_DO + s * TILE_BYTES, &tmDO, h * HS, qrow, &qd_full[s]);
        issued = i + 1;
      }
      if (*abort_flag) {
        mbar_wait_drain(kv_full, 0);
        for (int i = max(0, issued - 2); i < issued; i++) mbar_wait_drain(&qd_full[i & 1], (i >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sk = smem_u32(smem + OFF_K), sv = smem_u32(smem + OFF_V);
      const uint32_t spt = smem_u32(smem + OFF_PT), sdst = smem_u32(smem + OFF_DST);
      bool ok = mbar_wait(kv_full, 0, abort_flag, p.err);
      for (int i = 0; i < niter && ok; i++) {
        const int s = i & 1;
        if (!mbar_wait(&qd_full[s], (i >> 1) & 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t sq = smem_u32(smem + OFF_Q + s * TILE_BYTES), sdo = smem_u32(smem + OFF_DO + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HS / 16; kk++) {
          mma_bf16(T_ST, desc_sw128(sk + kk * 32, 16, 1024), desc_sw128(sq + kk * 32, 16, 1024), IDESC_SS,
                   kk > 0 ? 1u : 0u);
          mma_bf16(T_DPT, desc_sw128(sv + kk * 32, 16, 1024), desc_sw128(sdo + kk * 32, 16, 1024), IDESC_SS,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (!mbar_wait(st_ready, i & 1, abort_flag, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BQ / 16; kk++) {
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          mma_bf16(T_DV, desc_a128(spt, kk), desc_sw128(sdo + kk * 2048, 8192, 1024), IDESC_ACC, acc);
          mma_bf16(T_DK, desc_a128(sdst, kk), desc_sw128(sq + kk * 2048, 8192, 1024), IDESC_ACC, acc);
        }
        mma_commit(&qd_empty[s]);
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row within the tile = TMEM lane
    const int t = threadIdx.x - 64;
    const int k = kt * BKV + r;    // key position
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float l2e = 1.4426950408889634f, sl2 = p.scale * l2e;
    float* lse_s = reinterpret_cast<float*>(smem + OFF_LD);
    float* D_s = lse_s + 128;
    const size_t bh = ((size_t)b * p.NH + h) * p.T;
    bool ok = true;
    for (int i = 0; i < niter; i++) {
      const int qt = kt + i;
      // lse (pre-multiplied by log2 e) and D of this query tile, shared by the 128 rows
      tc::epi_bar<128>();
      lse_s[t] = p.lse[bh + qt * BQ + t] * l2e;
      D_s[t] = p.D[bh + qt * BQ + t];
      tc::epi_bar<128>();
      if (!tc::epi_bar_and<128>(mbar_wait(s_full, i & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = i == 0;  // queries before this key are masked
#pragma unroll 1
      for (int c = 0; c < BQ / 32; c++) {
        float st[32], dpt[32];
        tmem_ld32(T_ST + lane_off + c * 32, st);
        tmem_ld32(T_DPT + lane_off + c * 32, dpt);
        uint32_t wp[16], wd[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          float pv[2], dv[2];
#pragma unroll
          for (int u = 0; u < 2; u++) {
            const int qi = c * 32 + 2 * e + u;
            const bool masked = diag && qt * BQ + qi < k;
            pv[u] = masked ? 0.f : exp2f(st[2 * e + u] * sl2 - lse_s[qi]);
            dv[u] = pv[u] * (dpt[2 * e + u] - D_s[qi]);
          }
          wp[e] = pack_bf16x2(pv[0], pv[1]);
          wd[e] = pack_bf16x2(dv[0], dv[1]);
        }
        st_row32_sw128(smem + OFF_PT, r, c, wp);
        st_row32_sw128(smem + OFF_DST, r, c, wd);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(st_ready);
    }
    if (ok) ok = mbar_wait(mma_done, 0, abort_flag, p.err);
    // one decision for all 128 threads: the TMEM loads below are warp-collective
    if (tc::epi_bar_and<128>(ok && !*abort_flag)) {
      tc_fence_after();
      float dv[64], dk[64];
      tmem_ld32(T_DV + lane_off, dv);
      tmem_ld32(T_DV + lane_off + 32, dv + 32);
      tmem_ld32(T_DK + lane_off, dk);
      tmem_ld32(T_DK + lane_off + 32, dk + 32);
      const size_t o = ((size_t)b * p.T + k) * 3 * p.C + h * HS;
#pragma unroll
      for (int d = 0; d < HS; d += 4) {
        *reinterpret_cast<float4*>(p.dqkv + o + p.C + d) =
            make_float4(dk[d] * p.scale, dk[d + 1] * p.scale, dk[d + 2] * p.scale, dk[d + 3] * p.scale);
        *reinterpret_cast<float4*>(p.dqkv + o + 2 * p.C + d) = make_float4(dv[d], dv[d + 1], dv[d + 2], dv[d + 3]);
      }
      if (p.dqkv_bf) {
#pragma unroll
        for (int d = 0; d < HS; d += 8) {
          uint4 a, c;
          a.x = pack_bf16x2(dk[d] * p.scale, dk[d + 1] * p.scale);
          a.y = pack_bf16x2(dk[d + 2] * p.scale, dk[d + 3] * p.scale);
          a.z = pack_bf16x2(dk[d + 4] * p.scale, dk[d + 5] * p.scale);
          a.w = pack_bf16x2(dk[d + 6] * p.scale, dk[d + 7] * p.scale);
          c.x = pack_bf16x2(dv[d], dv[d + 1]);
          c.y = pack_bf16x2(dv[d + 2], dv[d + 3]);
          c.z = pack_bf16x2(dv[d + 4], dv[d + 5]);
          c.w = pack_bf16x2(dv[d + 6], dv[d + 7]);
          *reinterpret_cast<uint4*>(p.dqkv_bf + o + p.C + d) = a;
          *reinterpret_cast<uint4*>(p.dqkv_bf + o + 2 * p.C + d) = c;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

namespace dqk {
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + TILE_BYTES;
constexpr int OFF_K = OFF_DO + TILE_BYTES;      // 2 stages
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;   // 2 stages
constexpr int OFF_DS = OFF_V + 2 * TILE_BYTES;  // dS, 128 x 128 bf16
constexpr int OFF_BAR = OFF_DS + 2 * TILE_BYTES;
// qd_full, kv_full[2], kv_empty[2], s_full, ds_ready, mma_done
constexpr int NUM_BARS = 8;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
}  // namespace dqk

__global__ void __launch_bounds__(THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmDO,
                          const __grid_constant__ BwdParams p) {
  pdl_launch_dependents();
  using namespace dqk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* qd_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 3;
  uint64_t* s_full = bars + 5;
  uint64_t* ds_ready = bars + 6;
  uint64_t* mma_done = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = p.T / BQ;
  const int qt = nt - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int niter = qt + 1;                 // key tiles 0 .. qt
  const int qrow = b * p.T + qt * BQ;

  if (threadIdx.x == 0) {
    mbar_init(qd_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(ds_ready, 128);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the first global-memory access comes after this
  const uint32_t T_S = tmem, T_DP = tmem + 128, T_DQ = tmem + 256;

  if (warp == 0) {
    if (lane == 0) {
      mbar_expect_tx(qd_full, 2 * TILE_BYTES);
      tma_load_2d(smem + OFF_Q, &tmQKV, h * HS, qrow, qd_full);
      tma_load_2d(smem + OFF_DO, &tmDO, h * HS, qrow, qd_full);
      int issued = 0;
      for (int j = 0; j < niter; j++) {
        const int s = j & 1, krow = b * p.T + j * BKV;
        if (!mbar_wait(&kv_empty[s], ((j >> 1) & 1) ^ 1, abort_flag, p.err)) break;
        mbar_expect_tx(&kv_full[s], 2 * TILE_BYTES);
        tma_load_2d(smem + OFF_K + s * TILE_BYTES, &tmQKV, p.C + h * HS, krow, &kv_full[s]);
        tma_load_2d(smem + OFF_V + s * TILE_BYTES, &tmQKV, 2 * p.C + h * HS, krow, &kv_full[s]);
        issued = j + 1;
      }
      if (*abort_flag) {
        mbar_wait_drain(qd_full, 0);
        for (int j = max(0, issued - 2); j < issued; j++) mbar_wait_drain(&kv_full[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sq = smem_u32(smem + OFF_Q), sdo = smem_u32(smem + OFF_DO), sds = smem_u32(smem + OFF_DS);
      bool ok = mbar_wait(qd_full, 0, abort_flag, p.err);
      for (int j = 0; j < niter && ok; j++) {
        const int s = j & 1;
        if (!mbar_wait(&kv_full[s], (j >> 1) & 1, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t sk = smem_u32(smem + OFF_K + s * TILE_BYTES), sv = smem_u32(smem + OFF_V + s * TILE_BYTES);
#pragma unroll
        for (int kk = 0; kk < HS / 16; kk++) {
          mma_bf16(T_S, desc_sw128(sq + kk * 32, 16, 1024), desc_sw128(sk + kk * 32, 16, 1024), IDESC_SS,
                   kk > 0 ? 1u : 0u);
          mma_bf16(T_DP, desc_sw128(sdo + kk * 32, 16, 1024), desc_sw128(sv + kk * 32, 16, 1024), IDESC_SS,
                   kk > 0 ? 1u : 0u);
        }
        mma_commit(s_full);
        if (!mbar_wait(ds_ready, j & 1, abort_flag, p.err)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BKV / 16; kk++)
          mma_bf16(T_DQ, desc_a128(sds, kk), desc_sw128(sk + kk * 2048, 8192, 1024), IDESC_ACC,
                   (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&kv_empty[s]);
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // query row within the tile = TMEM lane
    const int t = qt * BQ + r;     // query position
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float l2e = 1.4426950408889634f, sl2 = p.scale * l2e;
    const size_t bh = ((size_t)b * p.NH + h) * p.T;
    const float L2 = p.lse[bh + t] * l2e, Dt = p.D[bh + t];
    bool ok = true;
    for (int j = 0; j < niter; j++) {
      if (!tc::epi_bar_and<128>(mbar_wait(s_full, j & 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool diag = j == qt;  // keys after this query are masked
#pragma unroll 1
      for (int c = 0; c < BKV / 32; c++) {
        float sv[32], dp[32];
        tmem_ld32(T_S + lane_off + c * 32, sv);
        tmem_ld32(T_DP + lane_off + c * 32, dp);
        uint32_t wd[16];
#pragma unroll
        for (int e = 0; e < 16; e++) {
          float dv[2];
#pragma unroll
          for (int u = 0; u < 2; u++) {
            const int ki = c * 32 + 2 * e + u;
            const bool masked = diag && j * BKV + ki > t;
            const float pv = masked ? 0.f : exp2f(sv[2 * e + u] * sl2 - L2);
            dv[u] = pv * (dp[2 * e + u] - Dt);
          }
          wd[e] = pack_bf16x2(dv[0], dv[1]);
        }
        st_row32_sw128(smem + OFF_DS, r, c, wd);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(ds_ready);
    }
    if (ok) ok = mbar_wait(mma_done, 0, abort_flag, p.err);
    // one decision for all 128 threads: the TMEM loads below are warp-collective
    if (tc::epi_bar_and<128>(ok && !*abort_flag)) {
      tc_fence_after();
      float dq[64];
      tmem_ld32(T_DQ + lane_off, dq);
      tmem_ld32(T_DQ + lane_off + 32, dq + 32);
      const size_t o = ((size_t)b * p.T + t) * 3 * p.C + h * HS;
#pragma unroll
      for (int d = 0; d < HS; d += 4)
        *reinterpret_cast<float4*>(p.dqkv + o + d) =
            make_float4(dq[d] * p.scale, dq[d + 1] * p.scale, dq[d + 2] * p.scale, dq[d + 3] * p.scale);
      if (p.dqkv_bf) {
#pragma unroll
        for (int d = 0; d < HS; d += 8) {
          uint4 a;
          a.x = pack_bf16x2(dq[d] * p.scale, dq[d + 1] * p.scale);
          a.y = pack_bf16x2(dq[d + 2] * p.scale, dq[d + 3] * p.scale);
          a.z = pack_bf16x2(dq[d + 4] * p.scale, dq[d + 5] * p.scale);
          a.w = pack_bf16x2(dq[d + 6] * p.scale, dq[d + 7] * p.scale);
          *reinterpret_cast<uint4*>(p.dqkv_bf + o + d) = a;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

}  // namespace tca
