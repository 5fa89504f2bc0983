// k_attention_tc.cuh -- causal attention forward on the tensor cores (bf16
// operands, fp32 softmax), head size 64, T a multiple of 128.
//
// Per (batch b, head h, tile of 128 queries): for each key tile j of 64
// keys up to the query tile's end (causal),
//   S   = Q K_j^T * scale                  tcgen05.mma kind::f16 -> TMEM
//   m'  = max(m, rowmax S);  P = exp(S - m');  l = l e^(m-m') + rowsum P
//   O   = O e^(m-m') + P V_j                P (bf16) written to TMEM,
//                                           P V_j -> TMEM -> registers
// and at the end y = O / l, lse = m + log l (the log-sum-exp of the scaled
// scores, as the backward pass expects).  Keys t2 > t of the last two tiles
// are masked.  This is the online-softmax form of attention (the page «llm.c：
// Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c», item 1,
// attention_forward computes the same causal softmax(q k^T / sqrt(hs)) v).
//
// Operands come from a bf16 copy of qkv, (B*T, 3C) row-major, through TMA
// maps with 64 x 128 boxes (Q tiles) and 64 x 64 boxes (K and V tiles),
// 128-byte swizzle: Q and K tiles are K-major (a row of 64 head dims per
// token); the V tile is read MN-major by the PV product (rows of 64 head
// dims per key = the N dimension contiguous).  Six warps: warp 0 issues the
// TMA loads (Q double-buffered per item, K and V through four stages each);
// warp 1 allocates TMEM and issues the MMAs; warps 2..5 own one query row
// per thread (TMEM lane = row) for the softmax and the output.  S and P
// each have two TMEM buffers: the scores of tile j + 2 are issued with the
// P V product of tile j, so the softmax warps find each tile's scores
// computed.
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

// ---- softmax arithmetic, one PTX instruction each ----
// 2^x on the special-function unit (relative error near 2^-22; 2^-inf = 0;
// subnormal results flush to zero, far below what a bf16 weight resolves).
GPT2_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 32 columns from each of two TMEM addresses, one wait for both loads
// lo and hi rounded to bf16 (nearest even) and packed, lo in the low half
GPT2_DEV uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
GPT2_DEV float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// 64 consecutive fp32 TMEM columns of the warp's 32 lanes (one per thread)
GPT2_DEV void tmem_ld64(uint32_t taddr, float* v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; i++) v[i] = __uint_as_float(r[i]);
}
// v[k] = -inf for every k > lim (the keys after the query on the diagonal tile)
GPT2_DEV void mask_after(float* v, int lim) {
#pragma unroll
  for (int k = 0; k < 64; k++)
    if (k > lim) v[k] = -INFINITY;
}

constexpr int BQ = 128;   // queries per CTA
constexpr int BKV = 128;  // keys per tile of the backward
constexpr int HS = 64;    // head size
constexpr int THREADS = 192;  // forward: TMA warp, MMA warp, 4 softmax warps
constexpr int TILE_BYTES = 128 * HS * 2;  // 16 KB: a 128-row Q, K or V tile
namespace fwd {
constexpr int FKV = 64;                      // keys per forward tile
constexpr int KT_BYTES = FKV * HS * 2;       // 8 KB: a 64-row K or V tile
constexpr int NK = 4;                        // K stages
constexpr int NV = 4;                        // V stages
constexpr int OFF_Q = 0;                     // 2 stages (one per item in flight)
constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr int OFF_V = OFF_K + NK * KT_BYTES;
constexpr int OFF_BAR = OFF_V + NV * KT_BYTES;
// q_full[2], q_empty[2], k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
// s_full[2], p_full[2], pv_full[2], mma_done
constexpr int NUM_BARS = 11 + 2 * NK + 2 * NV;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES + 1024 <= 233472 / 2, "two CTAs per SM");
}  // namespace fwd
// forward TMEM: S of tile t in columns [64 (t & 1), +64); P V in [128, 192);
// P of tile t (bf16 pairs) in [192 + 32 (t & 1), +32)
constexpr int TMEM_COLS = 256;

struct Params {
  int B, T, C, NH;
  float scale;     // 1/sqrt(hs)
  float* y;        // (B, T, C) fp32, or NULL
  uint16_t* ybf;   // (B, T, C) bf16 copy, or NULL
  float* lse;      // (B, NH, T)
  int* err;
};

// Instruction descriptors: S = Q K^T (M 128, N 64, both K-major);
// O += P V (M 128, N 64, P from TMEM, V MN-major).
constexpr uint32_t IDESC_FS =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(fwd::FKV >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);
constexpr uint32_t IDESC_PV =
    (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(HS >> 3) << 17) | ((uint32_t)(BQ >> 4) << 24);

// Work item w of B*NH*(T/128): query tile nqt-1 - w / (B*NH) (longest rows
// first) of head/batch w % (B*NH).  The grid is persistent (two CTAs per SM);
// CTA c of G takes item r*G + c in even rounds r and r*G + G-1-c in odd ones,
// a snake order that evens out the causal lengths.
GPT2_DEV bool fwd_item(const Params& p, int r, int& qt, int& h, int& b) {
  const int BH = p.B * p.NH, nitems = (p.T / BQ) * BH, G = gridDim.x, c = blockIdx.x;
  const int w = r * G + ((r & 1) ? G - 1 - c : c);
  if (w >= nitems) return false;
  qt = p.T / BQ - 1 - w / BH;
  h = (w % BH) % p.NH;
  b = (w % BH) / p.NH;
  return true;
}

// D += A B with A (M = 128 rows, K = 16 bf16) in TMEM at a_tmem: row i in
// lane i, two K values per 32-bit column, so 8 columns per MMA.
GPT2_DEV void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of the warp's 32 lanes (one per
// thread), then a wait for the stores to complete
GPT2_DEV void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// The CTA's key tiles in walk order: item n, its key tile j (64 keys), and
// whether j is the item's first / last (item n has 2 (qt + 1) tiles).
struct FwdWalk {
  int n = 0, j = 0, qt = 0, h = 0, b = 0;
  bool valid = false;
  GPT2_DEV void start(const Params& p) { n = 0; j = 0; valid = fwd_item(p, 0, qt, h, b); }
  GPT2_DEV int ntiles() const { return 2 * (qt + 1); }
  GPT2_DEV void next(const Params& p) {
    if (++j == ntiles()) {
      j = 0;
      valid = fwd_item(p, ++n, qt, h, b);
    }
  }
};

__global__ void __launch_bounds__(THREADS, 2)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                       const __grid_constant__ Params p) {
  pdl_launch_dependents();
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 2;
  uint64_t* k_full = bars + 4;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_full = s_full + 4;
  uint64_t* mma_done = s_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; s++) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);  // one arrival per softmax warp
      mbar_init(&pv_full[s], 1);
    }
    for (int s = 0; s < NK; s++) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NV; s++) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
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

  // Counters run on across the CTA's items: item n uses Q stage n & 1; key
  // tile number t (over all items) uses K stage t % NK, V stage t % NV and
  // the S, P and P V buffers t & 1.
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // K runs two tiles ahead of V (the scores of tile t + 2 are issued with
    // the P V product of tile t); Q is loaded with its item's first K.
    if (lane == 0) {
      int nq = 0, nk = 0, nv = 0;  // Q, K and V stage fills issued
      FwdWalk wk, wv;
      wk.start(p);
      wv.start(p);
      auto load_k = [&]() -> bool {
        if (!wk.valid) return true;
        if (wk.j == 0) {
          const int x = wk.n & 1;
          if (!mbar_wait(&q_empty[x], ((wk.n >> 1) & 1) ^ 1, abort_flag, p.err)) return false;
          mbar_expect_tx(&q_full[x], TILE_BYTES);
          tma_load_2d(smem + OFF_Q + x * TILE_BYTES, &tmQ, wk.h * HS, wk.b * p.T + wk.qt * BQ, &q_full[x]);
          nq = wk.n + 1;
        }
        const int s = nk % NK;
        if (!mbar_wait(&k_empty[s], ((nk / NK) & 1) ^ 1, abort_flag, p.err)) return false;
        mbar_expect_tx(&k_full[s], KT_BYTES);
        tma_load_2d(smem + OFF_K + s * KT_BYTES, &tmKV, p.C + wk.h * HS, wk.b * p.T + wk.j * FKV, &k_full[s]);
        nk++;
        wk.next(p);
        return true;
      };
      bool ok = load_k() && load_k();
      for (; ok && wv.valid; wv.next(p)) {
        const int s = nv % NV;
        if (!(ok = mbar_wait(&v_empty[s], ((nv / NV) & 1) ^ 1, abort_flag, p.err))) break;
        mbar_expect_tx(&v_full[s], KT_BYTES);
        tma_load_2d(smem + OFF_V + s * KT_BYTES, &tmKV, 2 * p.C + wv.h * HS, wv.b * p.T + wv.j * FKV, &v_full[s]);
        nv++;
        ok = load_k();
      }
      // the copies still in flight land before the CTA's memory goes away
      // (the latest fill of each stage; on the normal path they have landed)
      for (int i = max(0, nq - 2); i < nq; i++) mbar_wait_drain(&q_full[i & 1], (i >> 1) & 1);
      for (int i = max(0, nk - NK); i < nk; i++) mbar_wait_drain(&k_full[i % NK], (i / NK) & 1);
      for (int i = max(0, nv - NV); i < nv; i++) mbar_wait_drain(&v_full[i % NV], (i / NV) & 1);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // S of tile t + 2 is issued right after P V of tile t, into the S buffer
    // tile t's softmax has just released, so the softmax warps find the next
    // scores computed; P V of tile t waits only for P_t.
    if (lane == 0) {
      const uint32_t sq = smem_u32(smem + OFF_Q);
      FwdWalk ws;  // the tile whose scores are issued next (two ahead of P V)
      ws.start(p);
      int ts = 0;
      auto issue_s = [&]() -> bool {
        if (!ws.valid) return true;
        const int x = ws.n & 1, s = ts % NK;
        if (ws.j == 0 && !mbar_wait(&q_full[x], (ws.n >> 1) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(&k_full[s], (ts / NK) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t qa = sq + x * TILE_BYTES, kb = smem_u32(smem + OFF_K + s * KT_BYTES);
        const uint32_t t_s = tmem + (ts & 1) * FKV;
#pragma unroll
        for (int kk = 0; kk < HS / 16; kk++)
          mma_bf16(t_s, desc_sw128(qa + kk * 32, 16, 1024), desc_sw128(kb + kk * 32, 16, 1024), IDESC_FS,
                   kk > 0 ? 1u : 0u);
        mma_commit(&s_full[ts & 1]);
        mma_commit(&k_empty[s]);
        if (ws.j == ws.ntiles() - 1) mma_commit(&q_empty[x]);  // the item's last scores read Q
        ws.next(p);
        ts++;
        return true;
      };
      bool ok = issue_s() && issue_s();
      FwdWalk w;
      int t = 0;
      for (w.start(p); ok && w.valid; w.next(p), t++) {
        const int s = t % NV;
        ok = mbar_wait(&p_full[t & 1], (t >> 1) & 1, abort_flag, p.err) &&
             mbar_wait(&v_full[s], (t / NV) & 1, abort_flag, p.err);
        if (!ok) break;
        tc_fence_after();
        // P (in TMEM, buffer t & 1) times V (MN-major) into the P V columns,
        // which the softmax warps read out (P_{t-1} V) before releasing P_t
        const uint32_t vb = smem_u32(smem + OFF_V + s * KT_BYTES);
#pragma unroll
        for (int kk = 0; kk < FKV / 16; kk++)
          mma_bf16_ts(tmem + 2 * FKV, tmem + 3 * FKV + (t & 1) * (FKV / 2) + kk * 8, desc_sw128(vb + kk * 2048, 8192, 1024),
                      IDESC_PV, kk > 0 ? 1u : 0u);
        mma_commit(&pv_full[t & 1]);
        mma_commit(&v_empty[s]);
        ok = issue_s();
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    // ---------------- softmax + output: one query row per thread ----------------
    // Scores are kept in base 2: x = s * scale * log2(e), m = running max of x,
    // P = 2^(x - m) rounded to bf16 for the P V product, l = running fp32 sum
    // of P, O accumulated in registers in the basis of m.  Tile t: row max of
    // S_t, P_t written to TMEM, P_{t-1} V folded into O with the correction of
    // tile t-1 (which frees the P V columns), then P_t released to the MMA
    // warp.  Waits are decided per warp (the TMEM loads are warp-collective);
    // the warps meet only at the end of the kernel, so a timeout cannot split
    // a barrier.
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;  // scale * log2(e)
    const float2 sl2v = make_float2(sl2, sl2);
    float o[HS];
    auto fold_pv = [&](int t, float corr) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&pv_full[t & 1], (t >> 1) & 1, abort_flag, p.err))) return false;
      tc_fence_after();
      float pv[HS];
      tmem_ld64(tmem + 2 * FKV + lane_off, pv);
#pragma unroll
      for (int d = 0; d < HS; d += 2) {
        const float2 u = fma2(make_float2(o[d], o[d + 1]), make_float2(corr, corr), make_float2(pv[d], pv[d + 1]));
        o[d] = u.x;
        o[d + 1] = u.y;
      }
      return true;
    };
    int t = 0;
    bool ok = true;
    int qt, h, b;
    for (int it = 0; ok && fwd_item(p, it, qt, h, b); it++) {
      const int nkt = 2 * (qt + 1);
#pragma unroll
      for (int d = 0; d < HS; d++) o[d] = 0.f;
      float m2 = -INFINITY, lrow = 0.f, corr_prev = 0.f;
      for (int j = 0; j < nkt; j++, t++) {
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t & 1], (t >> 1) & 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[FKV];
        tmem_ld64(tmem + (t & 1) * FKV + lane_off, sv);
        // keys of the query tile's own 128 (the last two tiles): key c follows row r when c > lim
        if (j >= nkt - 2) mask_after(sv, r - (j - (nkt - 2)) * FKV);
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < FKV; k += 8) {
          mx[0] = max3(mx[0], sv[k], sv[k + 1]);
          mx[1] = max3(mx[1], sv[k + 2], sv[k + 3]);
          mx[2] = max3(mx[2], sv[k + 4], sv[k + 5]);
          mx[3] = max3(mx[3], sv[k + 6], sv[k + 7]);
        }
        const float mnew = fmaxf(m2, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2);
        const float corr = ex2(m2 - mnew);  // 0 on the first tile (m2 = -inf)
        const float2 nm = make_float2(-mnew, -mnew);
        float2 ls = make_float2(0.f, 0.f);
        uint32_t pw[FKV / 2];  // P of this row, bf16 pairs in key order
#pragma unroll
        for (int k = 0; k < FKV; k += 2) {
          const float2 x = fma2(make_float2(sv[k], sv[k + 1]), sl2v, nm);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          pw[k / 2] = cvt_bf16x2(pp.x, pp.y);
          ls = add2(ls, pp);
        }
        // P buffer t & 1 was last read by P_{t-2} V, folded at tile t - 1
        tmem_st32(tmem + 3 * FKV + (t & 1) * (FKV / 2) + lane_off, pw);
        if (j > 0 && !(ok = fold_pv(t - 1, corr_prev))) break;
        tc_fence_before();
        tc::mbar_arrive_warp(&p_full[t & 1]);
        lrow = lrow * corr + (ls.x + ls.y);
        m2 = mnew;
        corr_prev = corr;
      }
      if (!ok) break;
      if (!(ok = fold_pv(t - 1, corr_prev))) break;
      const float inv = 1.f / lrow;
      const size_t yo = (size_t)(b * p.T + qt * BQ + r) * p.C + h * HS;
      if (p.y) {  // NULL when only the bf16 copy is read downstream
#pragma unroll
        for (int d = 0; d < HS; d += 4)
          *reinterpret_cast<float4*>(p.y + yo + d) = make_float4(o[d] * inv, o[d + 1] * inv, o[d + 2] * inv, o[d + 3] * inv);
      }
      if (p.ybf) {
#pragma unroll
        for (int d = 0; d < HS; d += 8)
          *reinterpret_cast<uint4*>(p.ybf + yo + d) =
              make_uint4(cvt_bf16x2(o[d] * inv, o[d + 1] * inv), cvt_bf16x2(o[d + 2] * inv, o[d + 3] * inv),
                         cvt_bf16x2(o[d + 4] * inv, o[d + 5] * inv), cvt_bf16x2(o[d + 6] * inv, o[d + 7] * inv));
      }
      // log-sum-exp of the scaled scores: (m2 + log2 l) ln 2
      p.lse[((size_t)b * p.NH + h) * p.T + qt * BQ + r] = m2 * 0.6931471805599453f + logf(lrow);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

struct BwdParams {
  int B, T, C, NH;
  float scale;
  const float2* LD;  // (B, NH, T) pairs (-lse * log2 e, -D)
  float* dqkv;       // (B, T, 3C) fp32, or NULL
  uint16_t* dqkv_bf; // (B, T, 3C) bf16 copy, or NULL
  // or NULL: colsum[(b T/128 + tile) 3C + c] = the sum of dqkv(b, t, c) over
  // the 128 positions t of that tile (the first stage of the QKV bias gradient)
  float* colsum;
  int* err;
};

// Column sums of v[0..31] over the 32 lanes of the warp (lane = row): on
// return lane l holds the sum of column l.  Five halving exchange steps,
// 31 shuffles, a fixed order.  v is overwritten.
GPT2_DEV float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; k++) {
      const float send = hi ? v[k] : v[k + w];
      const float keep = hi ? v[k + w] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

constexpr int BWD_SOFTMAX_WARPS = 16;  // four per TMEM lane quarter, 16 columns each
constexpr int BWD_THREADS = 64 + 32 * BWD_SOFTMAX_WARPS;  // + producer warp, MMA warp
constexpr int BWD_CW = 16;  // sub-tile columns per softmax warp
constexpr int SUB = 64;           // queries (dK/dV) or keys (dQ) per sub-tile

// 16 consecutive fp32 TMEM columns of the warp's 32 lanes
GPT2_DEV void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// 16 columns from each of two TMEM addresses, one wait for both loads
GPT2_DEV void tmem_ld16x2(uint32_t a0, uint32_t a1, float* v0, float* v1) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; i++) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[16 + i]);
  }
}

// Column sums of v[0..15] over the 32 lanes of the warp (lane = row): on
// return lane l holds the sum of column l % 16.  Four halving exchange steps
// within each 16-lane half, then the two halves; 16 shuffles, a fixed order.
GPT2_DEV float warp_colsum16(float (&v)[16], int lane) {
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
    const bool hi = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; k++) {
      const float send = hi ? v[k] : v[k + w];
      const float keep = hi ? v[k + w] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Writes 16 bf16 values (8 packed words) at columns 16 qs .. 16 qs + 15 of row
// r of a K-major, 128-byte-swizzled tile with 64-column (128-byte) rows.
GPT2_DEV void st_quarter_row_sw128(uint8_t* tile, int r, int qs, const uint32_t (&w)[8]) {
#pragma unroll
  for (int g = 0; g < 2; g++)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((qs * 2 + g) ^ (r & 7)) << 4)) =
        make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
}

GPT2_DEV void tmem_ld32x2(uint32_t a0, uint32_t a1, float* v0, float* v1) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(a0), "r"(a1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) {
    v0[i] = __uint_as_float(r[i]);
    v1[i] = __uint_as_float(r[32 + i]);
  }
}

// Writes 32 bf16 values (16 packed words) at columns hf*32 .. hf*32+31 of row
// r of a K-major, 128-byte-swizzled tile with 64-column (128-byte) rows.
GPT2_DEV void st_half_row_sw128(uint8_t* tile, int r, int hf, const uint32_t (&w)[16]) {
#pragma unroll
  for (int g = 0; g < 4; g++)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((hf * 4 + g) ^ (r & 7)) << 4)) =
        make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to shared memory, completing on an mbarrier.
GPT2_DEV void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 128 x 64 scores (M = 128 rows, N = 64 columns, both operands K-major)
constexpr uint32_t IDESC_S64 =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(SUB >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
constexpr uint32_t IDESC_ACC = IDESC_PV;  // 128 x 64 accumulation, B MN-major

// Backward (the page's attention_backward), bf16 operands, head size 64,
// T % 128 == 0.  With P = exp(S*scale - lse) recomputed from the saved
// log-sum-exp, dP = dO V^T, D = rowsum(dO o y) and dS = P o (dP - D):
//   dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K.
// Two kernels, each output row produced by one CTA (no atomics, so the
// result is deterministic), both persistent (one CTA per SM walks the work
// items, longest first):
//   attn_bwd_dkv_tc_kernel  item (key tile, head, batch); walks the query
//       tiles at or after the key tile in sub-tiles of 64 queries:
//       S^T = K Q^T, dP^T = V dO^T into one of two TMEM buffers, P^T and
//       dS^T (bf16) into one of two shared-memory buffers, dV += P^T dO and
//       dK += dS^T Q accumulated in TMEM.
//   attn_bwd_dq_tc_kernel   item (query tile, head, batch); walks the key
//       tiles at or before it in sub-tiles of 64 keys: S = Q K^T, dP = dO V^T,
//       dS staged, dQ += dS K in TMEM.
// The scores of sub-tile i+1 are issued before the products of sub-tile i,
// so the tensor core computes the next scores while the sixteen softmax
// warps (four per TMEM lane quarter, 16 columns each) work on the current
// ones.  Operand tiles come from the bf16 copies of qkv and of dO (the
// gradient of the attention output, (B*T, C)) through TMA maps with 64 x 128
// boxes for the item's fixed tile and 64 x 64 boxes for the streamed
// sub-tiles.
// The per-query pairs LD[b,h,t] = (-lse log2 e, -D) with D = sum_d dO y over
// the head's 64 dims (the rowsum the backward subtracts from dP).  One warp
// per token: lane l reads dims 128 k + 4 l .. +3 of dO and y (all loads
// issued before any sum), so each 128-dim chunk holds two heads, summed over
// 16 lanes each.
constexpr int LD_WARPS = 8;
template <int MAXK>  // C <= 128 MAXK
__global__ void __launch_bounds__(LD_WARPS * 32)
    attn_bwd_ld_kernel(float2* __restrict__ LD, const float* __restrict__ lse, const float* __restrict__ dy,
                       const float* __restrict__ y, int B, int T, int C) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * LD_WARPS + (threadIdx.x >> 5);  // token b*T + t
  if (row >= (long long)B * T) return;
  const int b = (int)(row / T), t = (int)(row % T), NH = C / HS;
  const float* dr = dy + row * C;
  const float* yr = y + row * C;
  float sum[MAXK];
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
    const int d = 128 * k + 4 * lane;
    sum[k] = 0.f;
    if (d < C) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(dr + d));
      const float4 c = __ldg(reinterpret_cast<const float4*>(yr + d));
      sum[k] = a.x * c.x + a.y * c.y + a.z * c.z + a.w * c.w;
    }
  }
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum[k] += __shfl_xor_sync(0xffffffffu, sum[k], o);
  }
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
    const int d = 128 * k + 4 * lane, h = 2 * k + (lane >> 4);
    if ((lane & 15) == 0 && d < C) {
      const size_t i = ((size_t)b * NH + h) * T + t;
      LD[i] = make_float2(-lse[i] * 1.4426950408889634f, -sum[k]);
    }
  }
}

// The same pairs from the bf16 copies of dO and y (the model's bf16 path,
// where the fp32 ones are not written): lane l reads 4 bf16 (8 bytes) of each
// at dims 128 k + 4 l .. +3, as above.
template <int MAXK>  // C <= 128 MAXK
__global__ void __launch_bounds__(LD_WARPS * 32)
    attn_bwd_ld_bf16_kernel(float2* __restrict__ LD, const float* __restrict__ lse, const uint16_t* __restrict__ dy,
                            const uint16_t* __restrict__ y, int B, int T, int C) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * LD_WARPS + (threadIdx.x >> 5);  // token b*T + t
  if (row >= (long long)B * T) return;
  const int b = (int)(row / T), t = (int)(row % T), NH = C / HS;
  const uint16_t* dr = dy + row * C;
  const uint16_t* yr = y + row * C;
  float sum[MAXK];
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
    const int d = 128 * k + 4 * lane;
    sum[k] = 0.f;
    if (d < C) {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(dr + d));
      const uint2 c = __ldg(reinterpret_cast<const uint2*>(yr + d));
      sum[k] = __uint_as_float(a.x << 16) * __uint_as_float(c.x << 16) +
               __uint_as_float(a.x & 0xffff0000u) * __uint_as_float(c.x & 0xffff0000u) +
               __uint_as_float(a.y << 16) * __uint_as_float(c.y << 16) +
               __uint_as_float(a.y & 0xffff0000u) * __uint_as_float(c.y & 0xffff0000u);
    }
  }
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum[k] += __shfl_xor_sync(0xffffffffu, sum[k], o);
  }
#pragma unroll
  for (int k = 0; k < MAXK; k++) {
    const int d = 128 * k + 4 * lane, h = 2 * k + (lane >> 4);
    if ((lane & 15) == 0 && d < C) {
      const size_t i = ((size_t)b * NH + h) * T + t;
      LD[i] = make_float2(-lse[i] * 1.4426950408889634f, -sum[k]);
    }
  }
}

// Work item r of this CTA in the persistent backward kernels: items are
// numbered w = 0 .. (T/128) B NH - 1 with rank w / (B NH) (0 = the most
// causal work: key tile 0 for dK/dV, the last query tile for dQ) and
// head/batch w % (B NH); CTA c of G takes w = r G + c in even rounds r and
// r G + G-1-c in odd ones (a snake that evens out the causal lengths).
GPT2_DEV bool bwd_item(const BwdParams& p, int r, int& rank, int& h, int& b) {
  const int BH = p.B * p.NH, nitems = (p.T / BQ) * BH, G = gridDim.x, c = blockIdx.x;
  const int w = r * G + ((r & 1) ? G - 1 - c : c);
  if (w >= nitems) return false;
  rank = w / BH;
  h = (w % BH) % p.NH;
  b = (w % BH) / p.NH;
  return true;
}

namespace dkv {
// The query side streams through a ring of NSQ stages of one 64-query
// sub-tile each (Q, dO and their (-lse log2 e, -D) pairs): a stage is
// refilled as soon as its sub-tile's dV / dK products have read it, so a
// copy has about NSQ - 2 sub-tile periods to land.
constexpr int NSQ = 5;
constexpr int SUBT_BYTES = SUB * HS * 2;           // 8 KB: 64 rows of 64 bf16
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + 2 * TILE_BYTES;      // K and V: 2 stages (one per item in flight)
constexpr int OFF_Q = OFF_V + 2 * TILE_BYTES;      // NSQ stages
constexpr int OFF_DO = OFF_Q + NSQ * SUBT_BYTES;   // NSQ stages
constexpr int SUB_BYTES = 128 * SUB * 2;           // 16 KB: a 128 x 64 bf16 P^T or dS^T
constexpr int OFF_PT = OFF_DO + NSQ * SUBT_BYTES;  // 2 buffers
constexpr int OFF_DST = OFF_PT + 2 * SUB_BYTES;    // 2 buffers
constexpr int LD_BYTES = SUB * 8;                  // (-lse log2 e, -D) of one sub-tile
constexpr int OFF_LD = OFF_DST + 2 * SUB_BYTES;    // NSQ stages
constexpr int RED_BYTES = 2 * 4 * 4 * 16 * 4;      // column-sum partials [dK, dV][qs][q4][16]
constexpr int OFF_RED = OFF_LD + NSQ * LD_BYTES;   // 2 buffers (items alternate)
constexpr int OFF_BAR = OFF_RED + 2 * RED_BYTES;
// kv_full[2], kv_empty[2], qd_full[NSQ], qd_empty[NSQ], s_full[2],
// st_ready[2], pt_free[2], acc_full[2], acc_empty[2], mma_done, s_done
constexpr int NUM_BARS = 16 + 2 * NSQ;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
}  // namespace dkv

// dK/dV: each of the four accumulation chains (S^T, dP^T, dV, dK) is issued
// by its own thread, in its own warp, so that their issue times overlap: a
// 128 x 64 x 16 MMA takes about as long to issue as a 256-wide one.  The
// four threads sit on the four SM sub-partitions (warp w runs on w mod 4:
// dK warp 0, S^T warp 1, dV warp 18, dP^T warp 19), one each: a
// sub-partition that hosted two such polling threads started its softmax
// warps about 0.45 us late on every sub-tile.  So there is no separate
// copy thread: the S^T issuer loads the next item's K and V, the dV issuer
// refills the query-side stages.  The barriers a pair of chains completes
// together (s_full, kv_empty, pt_free, qd_empty, acc_full, mma_done, s_done)
// count two arrivals.
constexpr int DKV_THREADS = BWD_THREADS + 64;
constexpr int DKV_DK_WARP = 0;
constexpr int DKV_DV_WARP = 2 + BWD_SOFTMAX_WARPS;  // 18
constexpr int DKV_DPT_WARP = DKV_DV_WARP + 1;       // 19

// Persistent: one CTA per SM walks the (key tile, head, batch) items (see
// bwd_item).  Counters run on across items: item n uses K/V stage and
// accumulator pair n & 1; sub-tile number g (over all of the CTA's items)
// uses Q/dO/LD stage g % NSQ, score buffer and P^T/dS^T buffer g & 1.  So the
// next item's K and V load, and its first scores compute, while the softmax
// warps finish the current item and read its dV and dK out of tensor memory.
// tmKV: qkv with 128-row boxes (K, V tiles); tmQ, tmDO: qkv and dO with
// 64-row boxes (query sub-tiles).
__global__ void __launch_bounds__(DKV_THREADS, 1)
    attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmQ,
                           const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ BwdParams p) {
  pdl_launch_dependents();
  using namespace dkv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + 2;
  uint64_t* qd_full = bars + 4;
  uint64_t* qd_empty = qd_full + NSQ;
  uint64_t* s_full = qd_empty + NSQ;
  uint64_t* st_ready = s_full + 2;
  uint64_t* pt_free = s_full + 4;
  uint64_t* acc_full = s_full + 6;
  uint64_t* acc_empty = s_full + 8;
  uint64_t* mma_done = s_full + 10;
  uint64_t* s_done = s_full + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = p.T / BKV;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSQ; s++) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 2);                  // the dV and dK issuers
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 2);                  // the S^T and dP^T issuers
      mbar_init(&s_full[s], 2);                    // the S^T and dP^T issuers
      mbar_init(&st_ready[s], BWD_SOFTMAX_WARPS);  // one arrival per softmax warp
      mbar_init(&pt_free[s], 2);                   // the dV and dK issuers
      mbar_init(&acc_full[s], 2);                  // the dV and dK issuers
      mbar_init(&acc_empty[s], BWD_SOFTMAX_WARPS); // one arrival per softmax warp
    }
    mbar_init(mma_done, 2);
    mbar_init(s_done, 2);
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
  // TMEM: score buffer x in columns [128 x, 128 x + 128): S^T then dP^T (64
  // each); accumulator pair a in [256 + 128 a, 384 + 128 a): dV then dK
  auto t_dv = [&](int a) { return tmem + 256 + 128 * a; };

  if (warp == 1 || warp == DKV_DPT_WARP) {
    // ---------------- scores issuers: S^T = K Q^T (warp 1), dP^T = V dO^T ----------------
    // The S^T issuer also loads K and V: item 0's at the start, item n + 1's
    // once item n's first scores are issued (item n - 1's have completed by
    // then, so its stage is free).
    if (lane == 0) {
      const bool dpt = warp == DKV_DPT_WARP;
      int g = 0, nkv = 0;  // nkv: K/V stage fills issued (S^T issuer)
      bool ok = true;
      int kt, h, b;
      auto load_kv = [&](int n) {  // item n's K and V into stage n & 1, if the item exists
        int kt2, h2, b2;
        if (!bwd_item(p, n, kt2, h2, b2)) return true;
        const int y = n & 1, krow = b2 * p.T + kt2 * BKV;
        if (n >= 2 && !mbar_wait(&kv_empty[y], ((n >> 1) & 1) ^ 1, abort_flag, p.err)) return false;
        mbar_expect_tx(&kv_full[y], 2 * TILE_BYTES);
        tma_load_2d(smem + OFF_K + y * TILE_BYTES, &tmKV, p.C + h2 * HS, krow, &kv_full[y]);
        tma_load_2d(smem + OFF_V + y * TILE_BYTES, &tmKV, 2 * p.C + h2 * HS, krow, &kv_full[y]);
        nkv = n + 1;
        return true;
      };
      if (!dpt) ok = load_kv(0);
      for (int n = 0; ok && bwd_item(p, n, kt, h, b); n++) {
        const int x = n & 1;
        if (!(ok = mbar_wait(&kv_full[x], (n >> 1) & 1, abort_flag, p.err))) break;
        const uint32_t sa = smem_u32(smem + (dpt ? OFF_V : OFF_K) + x * TILE_BYTES);
        for (int qt = kt; ok && qt < nt; qt++) {
          for (int u = 0; u < 2; u++, g++) {
            const int s = g % NSQ;
            // score buffer g & 1 was read out by the softmax warps before st_ready(g - 2)
            if (g >= 2 && !(ok = mbar_wait(&st_ready[g & 1], ((g - 2) >> 1) & 1, abort_flag, p.err))) break;
            if (!(ok = mbar_wait(&qd_full[s], (g / NSQ) & 1, abort_flag, p.err))) break;
            tc_fence_after();
            const uint32_t sb = smem_u32(smem + (dpt ? OFF_DO : OFF_Q) + s * SUBT_BYTES);
            const uint32_t t_acc = tmem + (g & 1) * 128 + (dpt ? SUB : 0);
#pragma unroll
            for (int kk = 0; kk < HS / 16; kk++)
              mma_bf16(t_acc, desc_sw128(sa + kk * 32, 16, 1024), desc_sw128(sb + kk * 32, 16, 1024), IDESC_S64,
                       kk > 0 ? 1u : 0u);
            mma_commit(&s_full[g & 1]);
            if (!dpt && qt == kt && u == 0 && !(ok = load_kv(n + 1))) break;
          }
        }
        if (ok) mma_commit(&kv_empty[x]);  // the item's K (V) stage is free once these scores complete
      }
      // the scores these threads issued land before the CTA's resources go,
      // and so do the K/V copies still in flight (the latest fill of each stage)
      mma_commit(s_done);
      mbar_wait_drain(s_done, 0);
      for (int i = max(0, nkv - 2); i < nkv; i++) mbar_wait_drain(&kv_full[i & 1], (i >> 1) & 1);
    }
  } else if (warp == DKV_DV_WARP || warp == DKV_DK_WARP) {
    // ---------------- products issuers: dV += P^T dO, dK += dS^T Q ----------------
    // (a sub-tile's scores have completed by the time its st_ready fires: the
    // softmax warps waited for them, so these commits cover the tile's Q/dO.)
    // The dV issuer also fills the query-side stages: fill f (the CTA's f-th
    // 64-query sub-tile in walk order) goes to stage f % NSQ; the first NSQ at
    // the start, then after sub-tile g's products the fill that reuses the
    // stage of sub-tile g - 1 (whose products have completed by then).
    if (lane == 0) {
      const bool dk = warp == DKV_DK_WARP;
      int g = 0, nfill = 0;
      bool ok = true;
      int kt, h, b;
      int fn = 0, fkt = 0, fh = 0, fb = 0;  // the next fill: item fn, query position fq0
      bool fmore = !dk && bwd_item(p, 0, fkt, fh, fb);
      int fq0 = fkt * BQ;
      auto fill = [&]() {
        const int s = nfill % NSQ;
        const size_t bh = ((size_t)fb * p.NH + fh) * p.T;
        mbar_expect_tx(&qd_full[s], 2 * SUBT_BYTES + LD_BYTES);
        tma_load_2d(smem + OFF_Q + s * SUBT_BYTES, &tmQ, fh * HS, fb * p.T + fq0, &qd_full[s]);
        tma_load_2d(smem + OFF_DO + s * SUBT_BYTES, &tmDO, fh * HS, fb * p.T + fq0, &qd_full[s]);
        bulk_load(smem + OFF_LD + s * LD_BYTES, p.LD + bh + fq0, LD_BYTES, &qd_full[s]);
        nfill++;
        fq0 += SUB;
        if (fq0 >= p.T) {
          fmore = bwd_item(p, ++fn, fkt, fh, fb);
          fq0 = fkt * BQ;
        }
      };
      while (fmore && nfill < NSQ) fill();
      for (int n = 0; ok && bwd_item(p, n, kt, h, b); n++) {
        const int x = n & 1;
        const uint32_t t_acc = t_dv(x) + (dk ? HS : 0);
        // accumulator pair x was read out by the softmax warps of item n - 2
        if (!(ok = mbar_wait(&acc_empty[x], ((n >> 1) & 1) ^ 1, abort_flag, p.err))) break;
        for (int qt = kt; ok && qt < nt; qt++) {
          for (int u = 0; u < 2; u++, g++) {
            const int s = g % NSQ;
            if (!(ok = mbar_wait(&st_ready[g & 1], (g >> 1) & 1, abort_flag, p.err))) break;
            tc_fence_after();
            const uint32_t sb = smem_u32(smem + (dk ? OFF_Q : OFF_DO) + s * SUBT_BYTES);
            const uint32_t sa = smem_u32(smem + (dk ? OFF_DST : OFF_PT) + (g & 1) * SUB_BYTES);
#pragma unroll
            for (int kk = 0; kk < SUB / 16; kk++)
              mma_bf16(t_acc, desc_sw128(sa + kk * 32, 16, 1024), desc_sw128(sb + kk * 2048, 8192, 1024), IDESC_ACC,
                       (qt > kt || u > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&pt_free[g & 1]);
            mma_commit(&qd_empty[s]);
            if (fmore && nfill - NSQ < g) {  // refill the stage of sub-tile nfill - NSQ (= g - 1)
              const int f0 = nfill - NSQ;
              if (!(ok = mbar_wait(&qd_empty[f0 % NSQ], (f0 / NSQ) & 1, abort_flag, p.err))) break;
              fill();
            }
          }
        }
        if (ok) mma_commit(&acc_full[x]);
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
      // the query-side copies still in flight land before the CTA's memory goes
      for (int i = max(0, nfill - NSQ); i < nfill; i++) mbar_wait_drain(&qd_full[i % NSQ], (i / NSQ) & 1);
    }
  } else {
    // ---------------- softmax warps, then each item's dV / dK read-out ----------------
    const int q4 = warp & 3, qs = (warp - 2) >> 2;  // TMEM lane quarter; 16-column slice
    const int r = q4 * 32 + lane;  // key row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    const float2 sl2v = make_float2(sl2, sl2);
    bool ok = true;
    int g = 0;
    int kt, h, b;
    for (int n = 0; bwd_item(p, n, kt, h, b); n++) {
      const int x = n & 1;
      for (int qt = kt; qt < nt; qt++) {
        for (int u = 0; u < 2; u++, g++) {
          if (!ok) continue;  // after a timeout: count through to the item's end
          const int s = g % NSQ;
          // one decision per warp: the TMEM loads below are warp-collective
          const bool got = mbar_wait(&s_full[g & 1], (g >> 1) & 1, abort_flag, p.err) &&
                           mbar_wait(&qd_full[s], (g / NSQ) & 1, abort_flag, p.err) &&
                           (g < 2 || mbar_wait(&pt_free[g & 1], ((g - 2) >> 1) & 1, abort_flag, p.err));
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          float st[BWD_CW], dpt[BWD_CW];
          const uint32_t t_st = tmem + (g & 1) * 128 + lane_off + qs * BWD_CW;
          tmem_ld16x2(t_st, t_st + SUB, st, dpt);
          // queries u*64 + qs*16 + c of this query tile; before the key (masked) only on the diagonal
          const float4* ld = reinterpret_cast<const float4*>(smem + OFF_LD + s * LD_BYTES) + qs * BWD_CW / 2;
          if (qt == kt) {
            const int lim = r - u * SUB - qs * BWD_CW;  // column c is masked when c < lim
#pragma unroll
            for (int c = 0; c < BWD_CW; c++)
              if (c < lim) st[c] = -INFINITY;
          }
          uint32_t wp[BWD_CW / 2], wd[BWD_CW / 2];
#pragma unroll
          for (int e = 0; e < BWD_CW / 2; e++) {
            const float4 v = ld[e];  // (-lse2, -D) of queries 2e, 2e+1
            const float2 xx = fma2(make_float2(st[2 * e], st[2 * e + 1]), sl2v, make_float2(v.x, v.z));
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            const float2 ds = mul2(pp, add2(make_float2(dpt[2 * e], dpt[2 * e + 1]), make_float2(v.y, v.w)));
            wp[e] = cvt_bf16x2(pp.x, pp.y);
            wd[e] = cvt_bf16x2(ds.x, ds.y);
          }
          st_quarter_row_sw128(smem + OFF_PT + (g & 1) * SUB_BYTES, r, qs, wp);
          st_quarter_row_sw128(smem + OFF_DST + (g & 1) * SUB_BYTES, r, qs, wd);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          tc::mbar_arrive_warp(&st_ready[g & 1]);
        }
      }
      // the item's dK then dV (accumulator pair x, one half at a time to
      // keep registers down), then the pair is released
      const bool got = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[x], (n >> 1) & 1, abort_flag, p.err));
      float* red = reinterpret_cast<float*>(smem + OFF_RED + x * RED_BYTES);  // [dK, dV][qs][q4][16]
      if (got) {
        tc_fence_after();
        const size_t o = ((size_t)b * p.T + kt * BKV + r) * 3 * p.C + h * HS + qs * BWD_CW;
#pragma unroll 1
        for (int arr = 0; arr < 2; arr++) {  // 0: dK (scaled), 1: dV
          float v[BWD_CW];
          tmem_ld16(t_dv(x) + (arr == 0 ? HS : 0) + lane_off + qs * BWD_CW, v);
          if (arr == 1) {
            tc_fence_before();
            tc::mbar_arrive_warp(&acc_empty[x]);
          } else {
#pragma unroll
            for (int d = 0; d < BWD_CW; d++) v[d] *= p.scale;
          }
          const size_t oa = o + (1 + arr) * p.C;
          if (p.dqkv) {
#pragma unroll
            for (int d = 0; d < BWD_CW; d += 4)
              *reinterpret_cast<float4*>(p.dqkv + oa + d) = make_float4(v[d], v[d + 1], v[d + 2], v[d + 3]);
          }
          if (p.dqkv_bf) {
#pragma unroll
            for (int d = 0; d < BWD_CW; d += 8)
              *reinterpret_cast<uint4*>(p.dqkv_bf + oa + d) =
                  make_uint4(cvt_bf16x2(v[d], v[d + 1]), cvt_bf16x2(v[d + 2], v[d + 3]),
                             cvt_bf16x2(v[d + 4], v[d + 5]), cvt_bf16x2(v[d + 6], v[d + 7]));
          }
          if (p.colsum) {
            // the 128 key rows' column sums: warp butterflies here, then the
            // four lane quarters in order through this item's partials buffer
            const float sc = warp_colsum16(v, lane);
            if (lane < 16) red[((arr * 4 + qs) * 4 + q4) * 16 + lane] = sc;
          }
        }
      }
      if (p.colsum) {
        // all sixteen warps take every item's barrier; a timeout anywhere ends the walk for all
        if (!tc::epi_bar_and<32 * BWD_SOFTMAX_WARPS>(got)) break;
        const int t2 = threadIdx.x - 64;
        if (t2 < 128) {
          const int arr = t2 >> 6, col = t2 & 63, base = (arr * 4 + (col >> 4)) * 4 * 16 + (col & 15);
          const float sum = ((red[base] + red[base + 16]) + red[base + 32]) + red[base + 48];
          p.colsum[((size_t)b * nt + kt) * 3 * p.C + (1 + arr) * p.C + h * HS + col] = sum;
        }
      } else if (!got) {
        break;
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
// The key side streams through a ring of NSK stages of one 64-key sub-tile
// each (K and V), refilled as soon as the sub-tile's dQ product has read it.
constexpr int NSK = 6;
constexpr int SUBT_BYTES = SUB * HS * 2;          // 8 KB: 64 rows of 64 bf16
constexpr int OFF_Q = 0;                          // 2 stages (one per item in flight)
constexpr int OFF_DO = OFF_Q + 2 * TILE_BYTES;    // 2 stages
constexpr int OFF_K = OFF_DO + 2 * TILE_BYTES;    // NSK stages
constexpr int OFF_V = OFF_K + NSK * SUBT_BYTES;   // NSK stages
constexpr int SUB_BYTES = 128 * SUB * 2;
constexpr int OFF_DS = OFF_V + NSK * SUBT_BYTES;  // dS, 2 buffers of 128 x 64 bf16
constexpr int RED_BYTES = 4 * 4 * 16 * 4;         // column-sum partials [qs][q4][16]
constexpr int OFF_RED = OFF_DS + 2 * SUB_BYTES;   // 2 buffers (items alternate)
constexpr int OFF_BAR = OFF_RED + 2 * RED_BYTES;
// qd_full[2], qd_empty[2], kv_full[NSK], kv_empty[NSK], s_full[2],
// ds_ready[2], ds_free[2], acc_full[2], acc_empty[2], mma_done, s_done
constexpr int NUM_BARS = 16 + 2 * NSK;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
}  // namespace dqk

// dQ: the three accumulation chains (S, dP, dQ) issued by three threads in
// different warps (warp 1 and two warps after the softmax warps), as in the
// dK/dV kernel; s_full, qd_empty and s_done count the two scores issuers.
constexpr int DQ_THREADS = BWD_THREADS + 64;
constexpr int DQ_DQ_WARP = 2 + BWD_SOFTMAX_WARPS;  // 18
constexpr int DQ_DP_WARP = DQ_DQ_WARP + 1;         // 19

// Persistent like the dK/dV kernel: item n of the CTA uses Q/dO stage and dQ
// accumulator n & 1, sub-tile number g (over all of its items) K/V stage
// g % NSK, score buffer and dS buffer g & 1.  tmQ, tmDO: qkv and dO with
// 128-row boxes (query tiles); tmKV: qkv with 64-row boxes (key sub-tiles).
__global__ void __launch_bounds__(DQ_THREADS, 1)
    attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                          const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ BwdParams p) {
  pdl_launch_dependents();
  using namespace dqk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* qd_full = bars;
  uint64_t* qd_empty = bars + 2;
  uint64_t* kv_full = bars + 4;
  uint64_t* kv_empty = kv_full + NSK;
  uint64_t* s_full = kv_empty + NSK;
  uint64_t* ds_ready = s_full + 2;
  uint64_t* ds_free = s_full + 4;
  uint64_t* acc_full = s_full + 6;
  uint64_t* acc_empty = s_full + 8;
  uint64_t* mma_done = s_full + 10;
  uint64_t* s_done = s_full + 11;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = p.T / BQ;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSK; s++) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(&qd_full[s], 1);
      mbar_init(&qd_empty[s], 2);                  // the S and dP issuers
      mbar_init(&s_full[s], 2);                    // the S and dP issuers
      mbar_init(&ds_ready[s], BWD_SOFTMAX_WARPS);  // one arrival per softmax warp
      mbar_init(&ds_free[s], 1);
      mbar_init(&acc_full[s], 1);
      mbar_init(&acc_empty[s], BWD_SOFTMAX_WARPS); // one arrival per softmax warp
    }
    mbar_init(mma_done, 1);
    mbar_init(s_done, 2);
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
  // TMEM: score buffer x in columns [128 x, 128 x + 128): S then dP (64
  // each); dQ accumulator a in [256 + 64 a, 320 + 64 a)
  auto t_dq = [&](int a) { return tmem + 256 + HS * a; };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int nqd = 0, nsub = 0;  // Q/dO and K/V stage fills issued
      bool ok = true;
      int rank, h, b;
      for (int n = 0; ok && bwd_item(p, n, rank, h, b); n++) {
        const int x = n & 1, qt = nt - 1 - rank, qrow = b * p.T + qt * BQ;
        if (!(ok = mbar_wait(&qd_empty[x], ((n >> 1) & 1) ^ 1, abort_flag, p.err))) break;
        mbar_expect_tx(&qd_full[x], 2 * TILE_BYTES);
        tma_load_2d(smem + OFF_Q + x * TILE_BYTES, &tmQ, h * HS, qrow, &qd_full[x]);
        tma_load_2d(smem + OFF_DO + x * TILE_BYTES, &tmDO, h * HS, qrow, &qd_full[x]);
        nqd = n + 1;
        for (int k0 = 0; ok && k0 < (qt + 1) * BKV; k0 += SUB) {  // the item's 64-key sub-tiles
          const int s = nsub % NSK, krow = b * p.T + k0;
          if (!(ok = mbar_wait(&kv_empty[s], ((nsub / NSK) & 1) ^ 1, abort_flag, p.err))) break;
          mbar_expect_tx(&kv_full[s], 2 * SUBT_BYTES);
          tma_load_2d(smem + OFF_K + s * SUBT_BYTES, &tmKV, p.C + h * HS, krow, &kv_full[s]);
          tma_load_2d(smem + OFF_V + s * SUBT_BYTES, &tmKV, 2 * p.C + h * HS, krow, &kv_full[s]);
          nsub++;
        }
      }
      for (int i = max(0, nqd - 2); i < nqd; i++) mbar_wait_drain(&qd_full[i & 1], (i >> 1) & 1);
      for (int i = max(0, nsub - NSK); i < nsub; i++) mbar_wait_drain(&kv_full[i % NSK], (i / NSK) & 1);
    }
  } else if (warp == 1 || warp == DQ_DP_WARP) {
    // ---------------- scores issuers: S = Q K^T (warp 1), dP = dO V^T ----------------
    if (lane == 0) {
      const bool dpr = warp == DQ_DP_WARP;
      int g = 0;
      bool ok = true;
      int rank, h, b;
      for (int n = 0; ok && bwd_item(p, n, rank, h, b); n++) {
        const int x = n & 1, qt = nt - 1 - rank;
        if (!(ok = mbar_wait(&qd_full[x], (n >> 1) & 1, abort_flag, p.err))) break;
        const uint32_t sa = smem_u32(smem + (dpr ? OFF_DO : OFF_Q) + x * TILE_BYTES);
        for (int j = 0; ok && j <= qt; j++) {
          for (int u = 0; u < 2; u++, g++) {
            const int s = g % NSK;
            // score buffer g & 1 was read out by the softmax warps before ds_ready(g - 2)
            if (g >= 2 && !(ok = mbar_wait(&ds_ready[g & 1], ((g - 2) >> 1) & 1, abort_flag, p.err))) break;
            if (!(ok = mbar_wait(&kv_full[s], (g / NSK) & 1, abort_flag, p.err))) break;
            tc_fence_after();
            const uint32_t sb = smem_u32(smem + (dpr ? OFF_V : OFF_K) + s * SUBT_BYTES);
            const uint32_t t_acc = tmem + (g & 1) * 128 + (dpr ? SUB : 0);
#pragma unroll
            for (int kk = 0; kk < HS / 16; kk++)
              mma_bf16(t_acc, desc_sw128(sa + kk * 32, 16, 1024), desc_sw128(sb + kk * 32, 16, 1024), IDESC_S64,
                       kk > 0 ? 1u : 0u);
            mma_commit(&s_full[g & 1]);
          }
        }
        if (ok) mma_commit(&qd_empty[x]);  // the item's Q (dO) stage is free once these scores complete
      }
      mma_commit(s_done);
      mbar_wait_drain(s_done, 0);
    }
  } else if (warp == DQ_DQ_WARP) {
    // ---------------- dQ products issuer ----------------
    // (a sub-tile's scores have completed by the time its ds_ready fires, so
    // these commits cover the key tile's K and V)
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      int rank, h, b;
      for (int n = 0; ok && bwd_item(p, n, rank, h, b); n++) {
        const int x = n & 1, qt = nt - 1 - rank;
        // accumulator x was read out by the softmax warps of item n - 2
        if (!(ok = mbar_wait(&acc_empty[x], ((n >> 1) & 1) ^ 1, abort_flag, p.err))) break;
        for (int j = 0; ok && j <= qt; j++) {
          for (int u = 0; u < 2; u++, g++) {
            const int s = g % NSK;
            if (!(ok = mbar_wait(&ds_ready[g & 1], (g >> 1) & 1, abort_flag, p.err))) break;
            tc_fence_after();
            const uint32_t sk = smem_u32(smem + OFF_K + s * SUBT_BYTES);
            const uint32_t sds = smem_u32(smem + OFF_DS + (g & 1) * SUB_BYTES);
#pragma unroll
            for (int kk = 0; kk < SUB / 16; kk++)
              mma_bf16(t_dq(x), desc_sw128(sds + kk * 32, 16, 1024), desc_sw128(sk + kk * 2048, 8192, 1024),
                       IDESC_ACC, (j > 0 || u > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&ds_free[g & 1]);
            mma_commit(&kv_empty[s]);
          }
        }
        if (ok) mma_commit(&acc_full[x]);
      }
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else {
    // ---------------- softmax warps, then each item's dQ read-out ----------------
    const int q4 = warp & 3, qs = (warp - 2) >> 2;  // TMEM lane quarter; 16-column slice
    const int r = q4 * 32 + lane;  // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const float sl2 = p.scale * 1.4426950408889634f;
    const float2 sl2v = make_float2(sl2, sl2);
    bool ok = true;
    int g = 0;
    int rank, h, b;
    for (int n = 0; bwd_item(p, n, rank, h, b); n++) {
      const int x = n & 1, qt = nt - 1 - rank;
      const int t = qt * BQ + r;  // query position
      const float2 ldr = p.LD[((size_t)b * p.NH + h) * p.T + t];  // (-lse2, -D) of this query
      const float2 nlv = make_float2(ldr.x, ldr.x), ndv = make_float2(ldr.y, ldr.y);
      for (int j = 0; j <= qt; j++) {
        for (int u = 0; u < 2; u++, g++) {
          if (!ok) continue;  // after a timeout: count through to the item's end
          const bool got = mbar_wait(&s_full[g & 1], (g >> 1) & 1, abort_flag, p.err) &&
                           (g < 2 || mbar_wait(&ds_free[g & 1], ((g - 2) >> 1) & 1, abort_flag, p.err));
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            continue;
          }
          tc_fence_after();
          float sv[BWD_CW], dp[BWD_CW];
          const uint32_t t_s = tmem + (g & 1) * 128 + lane_off + qs * BWD_CW;
          tmem_ld16x2(t_s, t_s + SUB, sv, dp);
          if (j == qt) {  // keys after the query are masked: column c when u*64 + qs*16 + c > r
            const int lim = r - u * SUB - qs * BWD_CW;
#pragma unroll
            for (int c = 0; c < BWD_CW; c++)
              if (c > lim) sv[c] = -INFINITY;
          }
          uint32_t wd[BWD_CW / 2];
#pragma unroll
          for (int e = 0; e < BWD_CW / 2; e++) {
            const float2 xx = fma2(make_float2(sv[2 * e], sv[2 * e + 1]), sl2v, nlv);
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            const float2 ds = mul2(pp, add2(make_float2(dp[2 * e], dp[2 * e + 1]), ndv));
            wd[e] = cvt_bf16x2(ds.x, ds.y);
          }
          st_quarter_row_sw128(smem + OFF_DS + (g & 1) * SUB_BYTES, r, qs, wd);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          tc_fence_before();
          tc::mbar_arrive_warp(&ds_ready[g & 1]);
        }
      }
      // the item's dQ (accumulator x), then the accumulator is released
      const bool got = __all_sync(0xffffffffu, ok && mbar_wait(&acc_full[x], (n >> 1) & 1, abort_flag, p.err));
      float dq[BWD_CW];
      if (got) {
        tc_fence_after();
        tmem_ld16(t_dq(x) + lane_off + qs * BWD_CW, dq);
        tc_fence_before();
        tc::mbar_arrive_warp(&acc_empty[x]);
#pragma unroll
        for (int d = 0; d < BWD_CW; d++) dq[d] *= p.scale;
        const size_t o = ((size_t)b * p.T + t) * 3 * p.C + h * HS + qs * BWD_CW;
        if (p.dqkv) {
#pragma unroll
          for (int d = 0; d < BWD_CW; d += 4)
            *reinterpret_cast<float4*>(p.dqkv + o + d) = make_float4(dq[d], dq[d + 1], dq[d + 2], dq[d + 3]);
        }
        if (p.dqkv_bf) {
#pragma unroll
          for (int d = 0; d < BWD_CW; d += 8)
            *reinterpret_cast<uint4*>(p.dqkv_bf + o + d) =
                make_uint4(cvt_bf16x2(dq[d], dq[d + 1]), cvt_bf16x2(dq[d + 2], dq[d + 3]),
                           cvt_bf16x2(dq[d + 4], dq[d + 5]), cvt_bf16x2(dq[d + 6], dq[d + 7]));
        }
      }
      if (p.colsum) {
        // the 128 query rows' column sums, through this item's partials buffer
        float* red = reinterpret_cast<float*>(smem + OFF_RED + x * RED_BYTES);  // [qs][q4][16]
        if (got) {
          const float sq = warp_colsum16(dq, lane);
          if (lane < 16) red[(qs * 4 + q4) * 16 + lane] = sq;
        }
        // all sixteen warps take every item's barrier; a timeout anywhere ends the walk for all
        if (!tc::epi_bar_and<32 * BWD_SOFTMAX_WARPS>(got)) break;
        const int t2 = threadIdx.x - 64;
        if (t2 < 64) {
          const int base = (t2 >> 4) * 4 * 16 + (t2 & 15);
          const float sum = ((red[base] + red[base + 16]) + red[base + 32]) + red[base + 48];
          p.colsum[((size_t)b * nt + qt) * 3 * p.C + h * HS + t2] = sum;
        }
      } else if (!got) {
        break;
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
