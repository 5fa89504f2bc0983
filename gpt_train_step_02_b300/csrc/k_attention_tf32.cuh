// k_attention_tf32.cuh -- causal multi-head attention for short sequences
// (T <= 64) with head size 64 and fp32 operands, its products on the
// 5th-generation tensor cores (tcgen05.mma kind::tf32, accumulators in TMEM)
// at fp32 accuracy: every operand value is split x = hi + lo (hi = x rounded
// to TF32, lo = x - hi) and each product is ah*bh + ah*bl + al*bh, three MMAs
// into one fp32 accumulator (the 3xTF32 scheme of Ootomo & Yokota, 2022),
// as in the fp32 matmul.
//
// Arithmetic (the page «llm.c：Andrej Karpathy带你从零复现LLM», section
// «核心代码解读：train_gpt2.c», item 1: attention_forward / attention_backward):
// scale 1/sqrt(hs), keys t2 <= t; S = q k^T scale, P = softmax(S), y = P v,
// lse = max + log(sum exp); backward through P = exp(S - lse),
// D_t = dy_t . y_t, dS = P o (dy v^T - D), dq = dS k scale, dk = dS^T q scale,
// dv = P^T dy.  Exponentials use expf (the fp32 workloads are compared step
// by step with the oracle).
//
// One CTA of 256 threads per (head, batch).  Thread r < 64 (warps 0-1) owns
// TMEM lane r, i.e. row r of every 128-row accumulator (rows >= T are
// padding; lanes 64..127 are never written or read); all eight warps share
// the shared-memory passes (splits, transposes).  Operands:
//  - A operands (the rows the CTA's threads own) go from registers to TMEM
//    (tcgen05.st; row in the lane, one K value per column);
//  - B operands sit in shared memory as 64 x 64 fp32 tiles, K-major with the
//    128-byte swizzle: K values [32c, 32c + 32) of row n at
//    8 KB * c + 128 n + 16 ((k/4 % 8) ^ (n % 8)) + 4 (k % 4) bytes.  Tiles
//    whose rows are rows of qkv (or dy) come in by TMA in exactly that layout
//    and are split in place (hi) plus a lo copy; transposed tiles (rows =
//    head dimensions) are written by the threads that hold the rows in
//    registers, each thread filling one K position of every tile row.
// One thread issues the MMAs; completion is signalled through an mbarrier.
// Every wait is bounded (tc::mbar_wait) and every stop-or-continue decision
// is taken by the whole CTA at once (__syncthreads_and), so a wait that gives
// up leaves no thread behind at a barrier.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "k_gemm_tc.cuh"

namespace atf {
using tc::mbar_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_drain;
using tc::mma_commit;
using tc::smem_u32;
using tc::tc_fence_after;
using tc::tc_fence_before;
using tc::tf32_hi;
using tc::tma_load_2d;
using tc::tmem_ld32;
using tc::tmem_st16;

constexpr int T_MAX = 64;                 // longest sequence
constexpr int HS = 64;                    // head size
constexpr int THREADS = 256;              // 8 warps share the shared-memory passes
constexpr int TILE_FLOATS = 64 * 64;      // one 64 x 64 fp32 B tile
constexpr int TILE_BYTES = TILE_FLOATS * 4;  // 16 KB
constexpr int BOX_BYTES = TILE_BYTES / 2;    // one 32-column TMA box: 64 rows x 128 B

// Row ownership: warps 0, 1, 4 and 5 (the ones that may access TMEM lanes
// 0..63) own the 64 rows, two threads per row: row 32 (warp % 2) + lane,
// half warp / 4 = columns [32 half, 32 half + 32) of every 64-wide row.  The
// other four warps map onto the rows the same way and, while the owners move
// their rows into TMEM, write the transposed tiles and the hi/lo splits.
GPT2_DEV bool row_owner() { return ((threadIdx.x >> 5) & 2) == 0; }
GPT2_DEV int own_row() { return 32 * ((threadIdx.x >> 5) & 1) + (threadIdx.x & 31); }
GPT2_DEV int own_half() { return threadIdx.x >> 7; }

// float offset of K value k of row n in a swizzled 64 x 64 K-major tile
GPT2_DEV int sw(int n, int k) { return (k >> 5) * 2048 + n * 32 + ((((k & 31) >> 2) ^ (n & 7)) << 2) + (k & 3); }

// Shared-memory descriptor of the 8 K values [8 kc, 8 kc + 8) of a swizzled tile.
GPT2_DEV uint64_t bdesc(const float* tile, int kc) {
  return tc::smem_desc_kmajor_sw128(smem_u32(tile) + (uint32_t)((kc >> 2) * BOX_BYTES + (kc & 3) * 32));
}

// Instruction descriptor: D fp32, A and B tf32 K-major, M = 128, N = n.
GPT2_DEV uint32_t idesc(int n) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

GPT2_DEV void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
      : "memory");
}

// acc (TMEM columns d_col ..) = A B^T over K = 8 ksteps values, 3xTF32: A's
// hi and lo halves in TMEM columns a_hi / a_lo (K value k in column + k), B's
// in swizzled tiles b_hi / b_lo; N = n rows of B.
GPT2_DEV void mma3(uint32_t tmem, int d_col, int a_hi, int a_lo, const float* b_hi, const float* b_lo, int ksteps,
                   int n) {
  const uint32_t id = idesc(n);
  for (int kc = 0; kc < ksteps; kc++) {
    const uint64_t bh = bdesc(b_hi, kc), bl = bdesc(b_lo, kc);
    mma_ta(tmem + d_col, tmem + a_hi + 8 * kc, bh, id, kc > 0 ? 1u : 0u);
    mma_ta(tmem + d_col, tmem + a_hi + 8 * kc, bl, id, 1u);
    mma_ta(tmem + d_col, tmem + a_lo + 8 * kc, bh, id, 1u);
  }
}

// This thread's 32 values of its row (columns [32 half, +32) of a 64-wide
// operand) into TMEM: hi halves at columns col + 32 half .., lo halves at
// col + 64 + 32 half ..
GPT2_DEV void st_half_split(uint32_t tlane, int col, int half, const float* v) {
#pragma unroll
  for (int g = 0; g < 2; g++) {
    float hv[16], lv[16];
#pragma unroll
    for (int k = 0; k < 16; k++) {
      hv[k] = tf32_hi(v[16 * g + k]);
      lv[k] = v[16 * g + k] - hv[k];
    }
    tmem_st16(tlane + (uint32_t)(col + 32 * half + 16 * g), hv);
    tmem_st16(tlane + (uint32_t)(col + 64 + 32 * half + 16 * g), lv);
  }
}

// This thread's 32 values of row r (columns [32 half, +32)) of a TMA-written
// swizzled tile, or zeros when !valid.  The 32 lanes of a warp read 32
// consecutive rows: each 16-byte load touches every bank once per 8 lanes.
GPT2_DEV void ld_tile_half(const float* tile, int r, int half, bool valid, float* v) {
#pragma unroll
  for (int q = 0; q < 8; q++) {
    const float4 x = valid ? *reinterpret_cast<const float4*>(tile + sw(r, 32 * half + 4 * q))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    v[4 * q] = x.x;
    v[4 * q + 1] = x.y;
    v[4 * q + 2] = x.z;
    v[4 * q + 3] = x.w;
  }
}

// 32 floats to dst (16-byte aligned), plus their bf16 copy at dbf when set.
GPT2_DEV void st_half32(float* dst, uint16_t* dbf, const float* v) {
#pragma unroll
  for (int q = 0; q < 8; q++)
    reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  if (dbf) {
#pragma unroll
    for (int q = 0; q < 8; q++)
      reinterpret_cast<uint2*>(dbf)[q] =
          make_uint2(bf16x2_bits(v[4 * q], v[4 * q + 1]), bf16x2_bits(v[4 * q + 2], v[4 * q + 3]));
  }
}

// This thread's 32 values (columns [32 half, +32) of row `row`), split, into
// the transposed tiles: value d goes to row d, K position `row`.  The 32 lanes
// of a warp hold 32 consecutive rows, so each store covers 32 consecutive K
// positions of one tile row: no bank conflicts.
GPT2_DEV void st_half_transposed(float* t_hi, float* t_lo, int row, int half, const float* v) {
#pragma unroll
  for (int k = 0; k < 32; k++) {
    const int d = 32 * half + k;
    const float hi = tf32_hi(v[k]);
    t_hi[sw(d, row)] = hi;
    t_lo[sw(d, row)] = v[k] - hi;
  }
}

// Split of a raw TMA-written tile into hi and lo tiles of the same layout,
// by the 128 threads of the warps that own no TMEM lanes (index nid).
GPT2_DEV void split_tile_to(const float* raw, float* hi, float* lo, int nid) {
  const float4* r4 = reinterpret_cast<const float4*>(raw);
  float4* h4 = reinterpret_cast<float4*>(hi);
  float4* l4 = reinterpret_cast<float4*>(lo);
#pragma unroll 4
  for (int i = nid; i < TILE_FLOATS / 4; i += THREADS / 2) {
    float4 h, l;
    tc::split4(r4[i], h, l);
    h4[i] = h;
    l4[i] = l;
  }
}

// Index of a thread among the warps that own no TMEM lanes (2, 3, 6, 7).
GPT2_DEV int helper_index() { return (threadIdx.x & 63) | ((threadIdx.x >> 7) << 6); }

// Generic-proxy shared-memory writes and TMEM stores made visible to the
// tensor core, then a CTA barrier.
GPT2_DEV void publish_operands() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Shared-memory layout (from a 1024-byte aligned base) of each kernel: NT
// tiles, two mbarriers, the TMEM slot and the abort flag, then the row
// exchange area: xa[2][64], xb[2][64] (per-half partial results of each row)
// and lse_s[64]; + 1 KB alignment slack.
template <int NT>
struct Smem {
  static constexpr int OFF_BAR = NT * TILE_BYTES;
  static constexpr int OFF_VEC = OFF_BAR + 64;
  static constexpr int BYTES = OFF_VEC + 5 * 64 * 4 + 1024;
};
// Every tile of the head's rows comes in raw by TMA; the threads read their
// rows out of the raw tiles, and the B operands are split into hi/lo tiles.
constexpr int FWD_TILES = 7;   // K (hi, lo), V^T (hi, lo), raw K, Q, V
constexpr int DQ_TILES = 11;   // K (hi, lo), V (hi, lo), K^T (hi, lo), raw K, V, Q, dY, Y
constexpr int DKV_TILES = 13;  // Q (hi, lo), dY (hi, lo), Q^T (hi, lo), dY^T (hi, lo), raw Q, dY, K, V, Y
constexpr size_t FWD_SMEM = Smem<FWD_TILES>::BYTES;
constexpr size_t DQ_SMEM = Smem<DQ_TILES>::BYTES;
constexpr size_t DKV_SMEM = Smem<DKV_TILES>::BYTES;

struct Params {
  int B, T, C, NH;
  float scale;
  const float* qkv;    // (B, T, 3C)
  const float* dy;     // (B, T, C) upstream gradient (backward)
  const float* y;      // (B, T, C) attention output (backward: D = dy . y)
  float* out;          // forward: y (B, T, C); backward: dqkv (B, T, 3C)
  uint16_t* out_bf;    // optional bf16 copy of out
  float* lse;          // (B, NH, T): written by the forward, read by the backward
  int* err;
};

// Common prologue: barriers, TMEM allocation (ncols), PDL wait.  The MMA
// completion barrier counts one commit per issuing thread (issuers).
template <int NT>
GPT2_DEV uint32_t prologue(uint8_t* smem, int ncols, int issuers = 1) {
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem<NT>::OFF_BAR);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + Smem<NT>::OFF_BAR + 16);
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);  // TMA
    mbar_init(&bars[1], issuers);  // MMA completion
    *reinterpret_cast<volatile int*>(smem + Smem<NT>::OFF_BAR + 24) = 0;  // abort flag
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t t = *slot;
  pdl_wait();
  return t;
}

GPT2_DEV void epilogue_free(uint32_t tmem, int ncols) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
  }
}

// The two TMA box loads of one tile (rows y0 .. y0+63, columns x0 .. x0+63 of
// map m) onto bar; the caller has set the barrier's expected bytes.
GPT2_DEV void tma_tile(const CUtensorMap* m, float* t, int x0, int y0, uint64_t* bar) {
  tma_load_2d(t, m, x0, y0, bar);
  tma_load_2d(reinterpret_cast<uint8_t*>(t) + BOX_BYTES, m, x0 + 32, y0, bar);
}

// The abort path: the TMA copies and the last committed MMA batch (phase
// mma_phase of the MMA barrier, -1 for none) land before the CTA releases its
// memory.
GPT2_DEV void drain(uint64_t* bars, int mma_phase) {
  if (threadIdx.x == 0) {
    mbar_wait_drain(&bars[0], 0);
    if (mma_phase >= 0) mbar_wait_drain(&bars[1], (uint32_t)(mma_phase & 1));
  }
}

// A bounded wait on bar (phase) by thread 0; the CTA takes the result
// together at the barrier.
GPT2_DEV bool wait_all(uint64_t* bar, uint32_t phase, volatile int* abort_flag, int* err) {
  const bool ok = threadIdx.x == 0 ? mbar_wait(bar, phase, abort_flag, err) : true;
  return __syncthreads_and(ok) != 0;
}

// ---------------------------------------------------------------------------
// forward.  TMEM: S accumulator [0, 64) -> later O; Q hi/lo [64, 192) ->
// later P hi/lo.  tmQKV: qkv as (B*T rows, 3C columns), 32 x 64 boxes, SW128.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS) attn_fwd_tf32_kernel(const __grid_constant__ CUtensorMap tmQKV,
                                                                const __grid_constant__ Params p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  float* k_hi = reinterpret_cast<float*>(smem);
  float* k_lo = k_hi + TILE_FLOATS;
  float* vt_hi = k_lo + TILE_FLOATS;
  float* vt_lo = vt_hi + TILE_FLOATS;
  float* q_raw = vt_lo + TILE_FLOATS;
  float* v_raw = q_raw + TILE_FLOATS;
  float* k_raw = v_raw + TILE_FLOATS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem<FWD_TILES>::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem<FWD_TILES>::OFF_BAR + 24);
  float* xa = reinterpret_cast<float*>(smem + Smem<FWD_TILES>::OFF_VEC);  // [2][64] half-row maxima
  float* xb = xa + 128;                                                      // [2][64] half-row sums
  const uint32_t tmem = prologue<FWD_TILES>(smem, 256);

  const int h = blockIdx.x, b = blockIdx.y, T = p.T, C = p.C;
  const int Tp = (T + 15) & ~15;  // keys padded to the MMA's N granularity
  const bool owner = row_owner();
  const int r = own_row(), hf = own_half();
  const uint32_t tlane = tmem + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16);
  const size_t row0 = (size_t)b * T;
  const bool row_ok = r < T, valid = owner && row_ok;
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bars[0], 3 * TILE_BYTES);
    tma_tile(&tmQKV, k_raw, C + h * HS, b * T, &bars[0]);
    tma_tile(&tmQKV, q_raw, h * HS, b * T, &bars[0]);
    tma_tile(&tmQKV, v_raw, 2 * C + h * HS, b * T, &bars[0]);
  }
  int mma_phase = -1;
  bool ok = wait_all(&bars[0], 0, abort_flag, p.err);
  if (ok) {
    if (owner) {
      float q[32];
      ld_tile_half(q_raw, r, hf, valid, q);
      st_half_split(tlane, 64, hf, q);
    } else {
      float v[32];
      ld_tile_half(v_raw, r, hf, row_ok, v);
      st_half_transposed(vt_hi, vt_lo, r, hf, v);  // V^T: rows d, K values = keys
      split_tile_to(k_raw, k_hi, k_lo, helper_index());
    }
    publish_operands();
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 64, 128, k_hi, k_lo, HS / 8, Tp);  // S = Q K^T
      mma_commit(&bars[1]);
    }
    mma_phase = 0;
    ok = wait_all(&bars[1], 0, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    float s[32];
    float mx = -INFINITY;
    if (owner) {
      tmem_ld32(tlane + (uint32_t)(32 * hf), s);
#pragma unroll
      for (int k = 0; k < 32; k++) {
        const int j = 32 * hf + k;
        s[k] = (j <= r && j < T) ? s[k] * p.scale : -INFINITY;
        mx = fmaxf(mx, s[k]);
      }
      xa[hf * 64 + r] = mx;
    }
    __syncthreads();
    float l = 0.f;
    if (owner) {
      mx = fmaxf(xa[r], xa[64 + r]);
#pragma unroll
      for (int k = 0; k < 32; k++) {
        s[k] = s[k] == -INFINITY ? 0.f : expf(s[k] - mx);
        l += s[k];
      }
      xb[hf * 64 + r] = l;
    }
    __syncthreads();
    if (owner) {
      l = xb[r] + xb[64 + r];
      const float inv = valid ? 1.0f / l : 0.f;
#pragma unroll
      for (int k = 0; k < 32; k++) s[k] *= inv;
      if (valid && hf == 0) p.lse[((size_t)b * p.NH + h) * T + r] = mx + logf(l);
      st_half_split(tlane, 64, hf, s);  // P over Q's columns: the S MMAs have completed
    }
    publish_operands();
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 64, 128, vt_hi, vt_lo, Tp / 8, HS);  // O = P V, over S's columns
      mma_commit(&bars[1]);
    }
    mma_phase = 1;
    ok = wait_all(&bars[1], 1, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    if (owner) {
      float o[32];
      tmem_ld32(tlane + (uint32_t)(32 * hf), o);
      if (valid)
        st_half32(p.out + (row0 + r) * C + h * HS + 32 * hf,
                  p.out_bf ? p.out_bf + (row0 + r) * C + h * HS + 32 * hf : nullptr, o);
    }
  } else {
    drain(bars, mma_phase);  // a copy or MMA still in flight lands before the CTA's memory is released
  }
  epilogue_free(tmem, 256);
}

// ---------------------------------------------------------------------------
// backward, query rows (blockIdx.z == 0 of the backward kernel): dq.  TMEM:
// S [0, 64) -> later dQ; dP [64, 128); Q hi/lo [128, 256) -> later dS hi/lo;
// dY hi/lo [256, 384).
// ---------------------------------------------------------------------------
GPT2_DEV void bwd_dq(const CUtensorMap* tmQKV, const CUtensorMap* tmDY, const CUtensorMap* tmY, const Params& p,
                     uint8_t* smem) {
  float* k_hi = reinterpret_cast<float*>(smem);
  float* k_lo = k_hi + TILE_FLOATS;
  float* v_hi = k_lo + TILE_FLOATS;
  float* v_lo = v_hi + TILE_FLOATS;
  float* kt_hi = v_lo + TILE_FLOATS;
  float* kt_lo = kt_hi + TILE_FLOATS;
  float* q_raw = kt_lo + TILE_FLOATS;
  float* dy_raw = q_raw + TILE_FLOATS;
  float* y_raw = dy_raw + TILE_FLOATS;
  float* k_raw = y_raw + TILE_FLOATS;
  float* v_raw = k_raw + TILE_FLOATS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem<DKV_TILES>::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem<DKV_TILES>::OFF_BAR + 24);
  float* xa = reinterpret_cast<float*>(smem + Smem<DKV_TILES>::OFF_VEC);  // [2][64] half-row D partials
  const uint32_t tmem = prologue<DKV_TILES>(smem, 512, 2);

  const int h = blockIdx.x, b = blockIdx.y, T = p.T, C = p.C;
  const int Tp = (T + 15) & ~15;
  const bool owner = row_owner();
  const int r = own_row(), hf = own_half();
  const uint32_t tlane = tmem + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16);
  const size_t row0 = (size_t)b * T;
  const bool row_ok = r < T, valid = owner && row_ok;
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bars[0], 5 * TILE_BYTES);
    tma_tile(tmQKV, k_raw, C + h * HS, b * T, &bars[0]);
    tma_tile(tmQKV, v_raw, 2 * C + h * HS, b * T, &bars[0]);
    tma_tile(tmQKV, q_raw, h * HS, b * T, &bars[0]);
    tma_tile(tmDY, dy_raw, h * HS, b * T, &bars[0]);
    tma_tile(tmY, y_raw, h * HS, b * T, &bars[0]);
  }
  const float lse_r = valid ? p.lse[((size_t)b * p.NH + h) * T + r] : 0.f;
  int mma_phase = -1;
  bool ok = wait_all(&bars[0], 0, abort_flag, p.err);
  if (ok) {
    if (owner) {
      float dyv[32], yv[32], qv[32];
      ld_tile_half(dy_raw, r, hf, valid, dyv);
      ld_tile_half(y_raw, r, hf, valid, yv);
      ld_tile_half(q_raw, r, hf, valid, qv);
      float D = 0.f;
#pragma unroll
      for (int d = 0; d < 32; d++) D = fmaf(dyv[d], yv[d], D);
      xa[hf * 64 + r] = D;
      st_half_split(tlane, 256, hf, dyv);  // dY
      st_half_split(tlane, 128, hf, qv);   // Q
    } else {
      float kv[32];
      ld_tile_half(k_raw, r, hf, row_ok, kv);
      st_half_transposed(kt_hi, kt_lo, r, hf, kv);  // K^T: row r as a key
      split_tile_to(k_raw, k_hi, k_lo, helper_index());
      split_tile_to(v_raw, v_hi, v_lo, helper_index());
    }
    publish_operands();
    // the two products' 24-MMA chains issued by two threads in different warps
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 128, 192, k_hi, k_lo, HS / 8, Tp);   // S = Q K^T
      mma_commit(&bars[1]);
    } else if (threadIdx.x == 32) {
      mma3(tmem, 64, 256, 320, v_hi, v_lo, HS / 8, Tp);  // dP = dY V^T
      mma_commit(&bars[1]);
    }
    mma_phase = 0;
    ok = wait_all(&bars[1], 0, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    if (owner) {
      const float Dr = xa[r] + xa[64 + r];
      float s[32], dp[32];
      tmem_ld32(tlane + (uint32_t)(32 * hf), s);
      tmem_ld32(tlane + (uint32_t)(64 + 32 * hf), dp);
#pragma unroll
      for (int k = 0; k < 32; k++) {
        const int j = 32 * hf + k;
        // dS, with the scale of S folded in; columns past the MMA's N hold no data
        s[k] = (valid && j <= r) ? expf(s[k] * p.scale - lse_r) * (dp[k] - Dr) * p.scale : 0.f;
      }
      st_half_split(tlane, 128, hf, s);  // dS over Q's columns
    }
    publish_operands();
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 128, 192, kt_hi, kt_lo, Tp / 8, HS);  // dQ = dS K, over S's columns
      mma_commit(&bars[1]);
    } else if (threadIdx.x == 32) {
      mma_commit(&bars[1]);  // the second issuer's arrival (no MMA of its own pending)
    }
    mma_phase = 1;
    ok = wait_all(&bars[1], 1, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    if (owner) {
      float g[32];
      tmem_ld32(tlane + (uint32_t)(32 * hf), g);
      const size_t o = (row0 + r) * 3 * C + h * HS + 32 * hf;
      if (valid) st_half32(p.out + o, p.out_bf ? p.out_bf + o : nullptr, g);
    }
  } else {
    drain(bars, mma_phase);
  }
  epilogue_free(tmem, 512);
}

// ---------------------------------------------------------------------------
// backward, key rows (blockIdx.z == 1): dk and dv.  TMEM: S^T [0, 64) ->
// later dV; dP^T [64, 128) -> later dK; K hi/lo [128, 256) -> later P^T
// hi/lo; V hi/lo [256, 384) -> later dS^T hi/lo.  tmDY: dy as (B*T rows, C
// columns).  Row r also stands for query r: its D_r partials and lse_r are
// shared through shared memory with every key row.
// ---------------------------------------------------------------------------
GPT2_DEV void bwd_dkv(const CUtensorMap* tmQKV, const CUtensorMap* tmDY, const CUtensorMap* tmY, const Params& p,
                      uint8_t* smem) {
  float* q_hi = reinterpret_cast<float*>(smem);
  float* q_lo = q_hi + TILE_FLOATS;
  float* dy_hi = q_lo + TILE_FLOATS;
  float* dy_lo = dy_hi + TILE_FLOATS;
  float* qt_hi = dy_lo + TILE_FLOATS;
  float* qt_lo = qt_hi + TILE_FLOATS;
  float* dyt_hi = qt_lo + TILE_FLOATS;
  float* dyt_lo = dyt_hi + TILE_FLOATS;
  float* k_raw = dyt_lo + TILE_FLOATS;
  float* v_raw = k_raw + TILE_FLOATS;
  float* y_raw = v_raw + TILE_FLOATS;
  float* q_raw = y_raw + TILE_FLOATS;
  float* dy_raw = q_raw + TILE_FLOATS;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem<DKV_TILES>::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem<DKV_TILES>::OFF_BAR + 24);
  float* xa = reinterpret_cast<float*>(smem + Smem<DKV_TILES>::OFF_VEC);  // [2][64] D partials per query
  float* lse_s = xa + 256;                                                  // [64]
  const uint32_t tmem = prologue<DKV_TILES>(smem, 512, 2);

  const int h = blockIdx.x, b = blockIdx.y, T = p.T, C = p.C;
  const int Tp = (T + 15) & ~15;
  const bool owner = row_owner();
  const int r = own_row(), hf = own_half();
  const uint32_t tlane = tmem + ((uint32_t)(32 * ((threadIdx.x >> 5) & 3)) << 16);
  const size_t row0 = (size_t)b * T;
  const bool row_ok = r < T, valid = owner && row_ok;
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bars[0], 5 * TILE_BYTES);
    tma_tile(tmQKV, q_raw, h * HS, b * T, &bars[0]);
    tma_tile(tmDY, dy_raw, h * HS, b * T, &bars[0]);
    tma_tile(tmQKV, k_raw, C + h * HS, b * T, &bars[0]);
    tma_tile(tmQKV, v_raw, 2 * C + h * HS, b * T, &bars[0]);
    tma_tile(tmY, y_raw, h * HS, b * T, &bars[0]);
  }
  const float lse_r = valid ? p.lse[((size_t)b * p.NH + h) * T + r] : 0.f;
  int mma_phase = -1;
  bool ok = wait_all(&bars[0], 0, abort_flag, p.err);
  if (ok) {
    if (owner) {
      float dyv[32], yv[32], kv[32], vv[32];
      ld_tile_half(dy_raw, r, hf, valid, dyv);
      ld_tile_half(y_raw, r, hf, valid, yv);
      ld_tile_half(k_raw, r, hf, valid, kv);
      ld_tile_half(v_raw, r, hf, valid, vv);
      // row r as a query: D_r partial, lse_r, its dY values for the transposed tile
      float D = 0.f;
#pragma unroll
      for (int d = 0; d < 32; d++) D = fmaf(dyv[d], yv[d], D);
      xa[hf * 64 + r] = D;
      if (hf == 0) lse_s[r] = lse_r;
      st_half_transposed(dyt_hi, dyt_lo, r, hf, dyv);  // dY^T
      // row r as a key: K and V into TMEM
      st_half_split(tlane, 128, hf, kv);
      st_half_split(tlane, 256, hf, vv);
    } else {
      float qv[32];
      ld_tile_half(q_raw, r, hf, row_ok, qv);
      st_half_transposed(qt_hi, qt_lo, r, hf, qv);  // Q^T
      split_tile_to(q_raw, q_hi, q_lo, helper_index());
      split_tile_to(dy_raw, dy_hi, dy_lo, helper_index());
    }
    publish_operands();
    // the two products' 24-MMA chains issued by two threads in different warps
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 128, 192, q_hi, q_lo, HS / 8, Tp);     // S^T = K Q^T
      mma_commit(&bars[1]);
    } else if (threadIdx.x == 32) {
      mma3(tmem, 64, 256, 320, dy_hi, dy_lo, HS / 8, Tp);  // dP^T = V dY^T
      mma_commit(&bars[1]);
    }
    mma_phase = 0;
    ok = wait_all(&bars[1], 0, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    if (owner) {
      float pt[32], dst[32];
      tmem_ld32(tlane + (uint32_t)(32 * hf), pt);
      tmem_ld32(tlane + (uint32_t)(64 + 32 * hf), dst);
#pragma unroll
      for (int k = 0; k < 32; k++) {
        const int t = 32 * hf + k;
        // columns past the MMA's N hold no data
        const bool live = valid && t >= r && t < T;
        const float pv = live ? expf(pt[k] * p.scale - lse_s[t]) : 0.f;
        pt[k] = pv;
        dst[k] = live ? pv * (dst[k] - (xa[t] + xa[64 + t])) * p.scale : 0.f;  // dS^T, with the scale folded in
      }
      st_half_split(tlane, 128, hf, pt);   // P^T over K's columns
      st_half_split(tlane, 256, hf, dst);  // dS^T over V's columns
    }
    publish_operands();
    if (threadIdx.x == 0) {
      mma3(tmem, 0, 128, 192, dyt_hi, dyt_lo, Tp / 8, HS);  // dV = P^T dY
      mma_commit(&bars[1]);
    } else if (threadIdx.x == 32) {
      mma3(tmem, 64, 256, 320, qt_hi, qt_lo, Tp / 8, HS);   // dK = dS^T Q
      mma_commit(&bars[1]);
    }
    mma_phase = 1;
    ok = wait_all(&bars[1], 1, abort_flag, p.err);
  }
  if (ok) {
    tc_fence_after();
    if (owner) {
      float g[32];
      const size_t o = (row0 + r) * 3 * C + h * HS + 32 * hf;
      tmem_ld32(tlane + (uint32_t)(64 + 32 * hf), g);
      if (valid) st_half32(p.out + o + C, p.out_bf ? p.out_bf + o + C : nullptr, g);
      tmem_ld32(tlane + (uint32_t)(32 * hf), g);
      if (valid) st_half32(p.out + o + 2 * C, p.out_bf ? p.out_bf + o + 2 * C : nullptr, g);
    }
  } else {
    drain(bars, mma_phase);
  }
  epilogue_free(tmem, 512);
}

// The backward: grid (NH, B, 2); the query-row CTAs (z = 0) and the key-row
// CTAs (z = 1) of every head run side by side.  Both use the larger layout.
constexpr size_t BWD_SMEM = DKV_SMEM;

__global__ void __launch_bounds__(THREADS) attn_bwd_tf32_kernel(const __grid_constant__ CUtensorMap tmQKV,
                                                                const __grid_constant__ CUtensorMap tmDY,
                                                                const __grid_constant__ CUtensorMap tmY,
                                                                const __grid_constant__ Params p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  if (blockIdx.z == 0)
    bwd_dq(&tmQKV, &tmDY, &tmY, p, smem);
  else
    bwd_dkv(&tmQKV, &tmDY, &tmY, p, smem);
}

}  // namespace atf
