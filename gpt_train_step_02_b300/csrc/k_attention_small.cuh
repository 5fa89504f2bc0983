// k_attention_small.cuh -- causal multi-head attention for short sequences
// (T <= 64) with head size 64, on CUDA cores.
//
// The same arithmetic as the streaming CUDA-core kernels (scale 1/sqrt(hs),
// keys t2 <= t; lse = max + log sum exp; backward through P = exp(S - lse),
// D_t = dy_t . y_t, dS = P (dP - D_t)), organised for short sequences: one CTA
// of 256 threads owns a whole (batch, head), loads its q, k, v (and dy) into
// shared memory once -- every global load of the CTA, y's for D included,
// issued before the first store -- and forms every product as a register-tiled
// 64 x 64 matrix product -- each thread a 4 x 4 output block, one 16-byte
// shared-memory load of each operand per 16 FMAs -- instead of one scalar
// load per FMA.  Blocks that lie wholly above the causal diagonal are
// skipped, and the reduction ranges stop at the diagonal.  The backward runs
// in one launch (S, P, dP and dS once; then dV = P^T dy, dK = dS^T q,
// dQ = dS k), with D computed in the kernel.  Every output element is summed
// by one thread in a fixed order, so results are deterministic.  With
// bf16_ops the operands, P entering P V and P^T dy, and dS are rounded to
// bf16 exactly where the streaming kernels round them.  The exponentials use
// expf (not the approximate __expf): these kernels serve the fp32 parity
// workloads, whose loss trajectory is compared step by step.
#pragma once
#include "common.cuh"
#include "k_attention_simt.cuh"

namespace atts {
constexpr int T_MAX = 64;       // longest sequence
constexpr int HS = 64;          // head size
constexpr int P = 68;           // row pitch in floats: rows stay 16-byte aligned, transposing stores spread the banks
constexpr int MAT = T_MAX * P;  // floats per 64 x 64 operand
constexpr int THREADS = 256;
constexpr int FWD_MATS = 4;   // q^T, k^T, v, P^T
constexpr int BWD_MATS = 10;  // q^T, k^T, dy^T, v^T, q, k, dy, P, dS, dS^T
constexpr size_t FWD_SMEM = (size_t)FWD_MATS * MAT * 4;
constexpr size_t BWD_SMEM = (size_t)BWD_MATS * MAT * 4 + 2 * T_MAX * 4;

// Thread -> 4 x 4 output block: rows 4 * ty, columns 4 * tx.  The 16 threads
// of one row block sit in one half-warp; a warp holds row blocks w and 15 - w,
// so under the causal mask every warp has the same number of live blocks.
GPT2_DEV int row_block() {
  const int w = threadIdx.x >> 5;
  return (threadIdx.x & 16) ? 15 - w : w;
}
GPT2_DEV int col_block() { return threadIdx.x & 15; }

// acc[a][c] += sum_{k0 <= k < k1} A(m0 + a, k) B(k, n0 + c), A stored
// transposed (AT[k * P + m]) and B row-major (Bk[k * P + n]).
GPT2_DEV void mm4x4(float (&acc)[4][4], const float* AT, const float* Bk, int m0, int n0, int k0, int k1) {
#pragma unroll 4
  for (int k = k0; k < k1; k++) {
    const float4 a = *reinterpret_cast<const float4*>(AT + k * P + m0);
    const float4 b = *reinterpret_cast<const float4*>(Bk + k * P + n0);
    const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
      for (int j = 0; j < 4; j++) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

GPT2_DEV void zero4x4(float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
}

// One head's 64 columns of rows 0 .. T-1 of a source (row r at src + r * ld),
// to be stored in shared memory row-major (dst[r * P + d]) and/or transposed
// (dT[d * P + r]); rows T .. 63 are stored as zero.
struct HeadCopy {
  const float* src;
  long long ld;
  float* dst;
  float* dT;
};

// All NS copies, every global load issued before the first shared-memory
// store (one round trip to L2 / HBM instead of NS).  Lanes take consecutive
// rows, so the transposing stores hit consecutive words.
template <int NS>
GPT2_DEV void load_heads(const HeadCopy (&cp)[NS], int T, int bf16_ops) {
  constexpr int U = T_MAX * HS / 4 / THREADS;
  float4 v[NS][U];
#pragma unroll
  for (int q = 0; q < NS; q++)
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int e = threadIdx.x + u * THREADS;
      const int r = e & (T_MAX - 1), c = (e >> 6) * 4;
      v[q][u] = r < T ? *reinterpret_cast<const float4*>(cp[q].src + (size_t)r * cp[q].ld + c)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
  for (int q = 0; q < NS; q++)
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int e = threadIdx.x + u * THREADS;
      const int r = e & (T_MAX - 1), c = (e >> 6) * 4;
      const float4 x = make_float4(att_rnd(v[q][u].x, bf16_ops), att_rnd(v[q][u].y, bf16_ops),
                                   att_rnd(v[q][u].z, bf16_ops), att_rnd(v[q][u].w, bf16_ops));
      if (cp[q].dst) *reinterpret_cast<float4*>(cp[q].dst + r * P + c) = x;
      if (cp[q].dT) {
        cp[q].dT[(c + 0) * P + r] = x.x;
        cp[q].dT[(c + 1) * P + r] = x.y;
        cp[q].dT[(c + 2) * P + r] = x.z;
        cp[q].dT[(c + 3) * P + r] = x.w;
      }
    }
}

// max / sum over the 16 threads of a row block (lanes differing in bits 0..3)
GPT2_DEV float rowblock_max(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
GPT2_DEV float rowblock_sum(float v) {
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// grid (NH, B): y (B,T,C), its bf16 copy (optional) and lse (B,NH,T) from qkv (B,T,3C).
__global__ void __launch_bounds__(THREADS)
    attn_fwd_small_kernel(float* __restrict__ y, uint16_t* __restrict__ ybf, float* __restrict__ lse,
                          const float* __restrict__ qkv, int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float4 sm_small4[];
  float* sm = reinterpret_cast<float*>(sm_small4);
  float* QT = sm;
  float* KT = QT + MAT;
  float* V = KT + MAT;
  float* PT = V + MAT;
  const int h = blockIdx.x, b = blockIdx.y;
  const float* base = qkv + (size_t)b * T * 3 * C + (size_t)h * HS;
  const HeadCopy cp[3] = {{base, 3LL * C, nullptr, QT}, {base + C, 3LL * C, nullptr, KT}, {base + 2 * C, 3LL * C, V, nullptr}};
  load_heads(cp, T, bf16_ops);
  __syncthreads();

  const int t0 = 4 * row_block(), j0 = 4 * col_block();
  const float scale = rsqrtf((float)HS);
  float s[4][4];
  zero4x4(s);
  if (j0 <= t0 + 3 && t0 < T) mm4x4(s, QT, KT, t0, j0, 0, HS);
  float mx[4], l[4];
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int t = t0 + a;
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; c++) {
      const int j = j0 + c;
      s[a][c] = (j <= t && t < T) ? s[a][c] * scale : -INFINITY;
      m = fmaxf(m, s[a][c]);
    }
    m = rowblock_max(m);
    mx[a] = t < T ? m : 0.f;  // rows past T have no live entry
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < 4; c++) {
      s[a][c] = expf(s[a][c] - mx[a]);  // exp(-inf) = 0 off the diagonal
      sum += s[a][c];
    }
    l[a] = rowblock_sum(sum);
  }
  // P^T for the weighted sum over keys
#pragma unroll
  for (int c = 0; c < 4; c++)
    *reinterpret_cast<float4*>(PT + (j0 + c) * P + t0) =
        make_float4(att_rnd(s[0][c], bf16_ops), att_rnd(s[1][c], bf16_ops), att_rnd(s[2][c], bf16_ops),
                    att_rnd(s[3][c], bf16_ops));
  __syncthreads();

  float o[4][4];
  zero4x4(o);
  const int d0 = j0;
  if (t0 < T) mm4x4(o, PT, V, t0, d0, 0, min(T, t0 + 4));
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int t = t0 + a;
    if (t >= T) break;
    const float inv = 1.f / l[a];
    const float4 out = make_float4(o[a][0] * inv, o[a][1] * inv, o[a][2] * inv, o[a][3] * inv);
    const size_t off = ((size_t)b * T + t) * C + (size_t)h * HS + d0;
    *reinterpret_cast<float4*>(y + off) = out;
    if (ybf) {
      uint2 pk = make_uint2(bf16x2_bits(out.x, out.y), bf16x2_bits(out.z, out.w));
      *reinterpret_cast<uint2*>(ybf + off) = pk;
    }
    if (col_block() == 0) lse[((size_t)b * NH + h) * T + t] = mx[a] + logf(l[a]);
  }
}

// grid (NH, B): dq, dk, dv of one head into dqkv (B,T,3C) (and its bf16 copy,
// optional) from qkv, dy, y (B,T,C) and lse.
__global__ void __launch_bounds__(THREADS)
    attn_bwd_small_kernel(float* __restrict__ dqkv, uint16_t* __restrict__ dqkv_bf, const float* __restrict__ qkv,
                          const float* __restrict__ dy, const float* __restrict__ y, const float* __restrict__ lse,
                          int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float4 sm_small4[];
  float* sm = reinterpret_cast<float*>(sm_small4);
  float* QT = sm;
  float* KT = QT + MAT;
  float* GT = KT + MAT;  // dy^T
  float* VT = GT + MAT;
  float* Qr = VT + MAT;
  float* Kr = Qr + MAT;
  float* Gr = Kr + MAT;  // dy
  float* Pm = Gr + MAT;
  float* Sm = Pm + MAT;  // dS
  float* ST = Sm + MAT;  // dS^T
  float* Ls = ST + MAT;
  float* Ds = Ls + T_MAX;
  const int h = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* base = qkv + (size_t)b * T * 3 * C + (size_t)h * HS;
  const float* gbase = dy + (size_t)b * T * C + (size_t)h * HS;
  // D_t = dy_t . y_t in fp32 (unrounded; warp w takes rows w + 8u, lane the
  // columns lane and lane + 32) and lse: their loads go out with the head
  // copies' below, so the whole CTA waits for memory once
  constexpr int DR = T_MAX / (THREADS / 32);
  float dyv[DR][2], yv[DR][2];
#pragma unroll
  for (int u = 0; u < DR; u++) {
    const int t = warp + u * (THREADS / 32);
    const size_t off = ((size_t)b * T + t) * C + (size_t)h * HS;
    dyv[u][0] = t < T ? dy[off + lane] : 0.f;
    dyv[u][1] = t < T ? dy[off + lane + 32] : 0.f;
    yv[u][0] = t < T ? y[off + lane] : 0.f;
    yv[u][1] = t < T ? y[off + lane + 32] : 0.f;
  }
  const float lsev = (int)threadIdx.x < T ? lse[((size_t)b * NH + h) * T + threadIdx.x] : 0.f;
  const HeadCopy cp[4] = {{base, 3LL * C, Qr, QT}, {base + C, 3LL * C, Kr, KT}, {base + 2 * C, 3LL * C, nullptr, VT},
                          {gbase, C, Gr, GT}};
  load_heads(cp, T, bf16_ops);
#pragma unroll
  for (int u = 0; u < DR; u++) {
    const float d = warp_sum(dyv[u][0] * yv[u][0] + dyv[u][1] * yv[u][1]);
    if (lane == 0) Ds[warp + u * (THREADS / 32)] = d;
  }
  if (threadIdx.x < T_MAX) Ls[threadIdx.x] = lsev;
  __syncthreads();

  const int t0 = 4 * row_block(), j0 = 4 * col_block();
  const float scale = rsqrtf((float)HS);
  {
    float s[4][4], dp[4][4];
    zero4x4(s);
    zero4x4(dp);
    const bool live = j0 <= t0 + 3 && t0 < T;
    if (live) {
      mm4x4(s, QT, KT, t0, j0, 0, HS);
      mm4x4(dp, GT, VT, t0, j0, 0, HS);
    }
#pragma unroll
    for (int a = 0; a < 4; a++) {
      const int t = t0 + a;
      const float Lt = Ls[t], Dt = Ds[t];
      float pr[4], ds[4];
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const int j = j0 + c;
        const float p = (j <= t && t < T) ? expf(s[a][c] * scale - Lt) : 0.f;
        ds[c] = att_rnd(p * (dp[a][c] - Dt), bf16_ops);
        pr[c] = att_rnd(p, bf16_ops);
      }
      *reinterpret_cast<float4*>(Pm + t * P + j0) = make_float4(pr[0], pr[1], pr[2], pr[3]);
      *reinterpret_cast<float4*>(Sm + t * P + j0) = make_float4(ds[0], ds[1], ds[2], ds[3]);
      s[a][0] = ds[0]; s[a][1] = ds[1]; s[a][2] = ds[2]; s[a][3] = ds[3];
    }
#pragma unroll
    for (int c = 0; c < 4; c++)
      *reinterpret_cast<float4*>(ST + (j0 + c) * P + t0) = make_float4(s[0][c], s[1][c], s[2][c], s[3][c]);
  }
  __syncthreads();

  // second phase: rows m0 = 4 * row block index keys (dk, dv) or queries (dq),
  // columns d0 the head dimensions
  const int m0 = t0, d0 = j0;
  if (m0 >= T) return;
  float acc[4][4];
  // dv[j] = sum_{t >= j} P[t][j] dy[t]
  zero4x4(acc);
  mm4x4(acc, Pm, Gr, m0, d0, m0, T);
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int j = m0 + a;
    if (j >= T) break;
    const size_t o = ((size_t)b * T + j) * 3 * C + 2 * C + (size_t)h * HS + d0;
    const float4 v = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    *reinterpret_cast<float4*>(dqkv + o) = v;
    if (dqkv_bf) *reinterpret_cast<uint2*>(dqkv_bf + o) = make_uint2(bf16x2_bits(v.x, v.y), bf16x2_bits(v.z, v.w));
  }
  // dk[j] = scale sum_{t >= j} dS[t][j] q[t]
  zero4x4(acc);
  mm4x4(acc, Sm, Qr, m0, d0, m0, T);
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int j = m0 + a;
    if (j >= T) break;
    const size_t o = ((size_t)b * T + j) * 3 * C + C + (size_t)h * HS + d0;
    const float4 v = make_float4(acc[a][0] * scale, acc[a][1] * scale, acc[a][2] * scale, acc[a][3] * scale);
    *reinterpret_cast<float4*>(dqkv + o) = v;
    if (dqkv_bf) *reinterpret_cast<uint2*>(dqkv_bf + o) = make_uint2(bf16x2_bits(v.x, v.y), bf16x2_bits(v.z, v.w));
  }
  // dq[t] = scale sum_{j <= t} dS[t][j] k[j]
  zero4x4(acc);
  mm4x4(acc, ST, Kr, m0, d0, 0, min(T, m0 + 4));
#pragma unroll
  for (int a = 0; a < 4; a++) {
    const int t = m0 + a;
    if (t >= T) break;
    const size_t o = ((size_t)b * T + t) * 3 * C + (size_t)h * HS + d0;
    const float4 v = make_float4(acc[a][0] * scale, acc[a][1] * scale, acc[a][2] * scale, acc[a][3] * scale);
    *reinterpret_cast<float4*>(dqkv + o) = v;
    if (dqkv_bf) *reinterpret_cast<uint2*>(dqkv_bf + o) = make_uint2(bf16x2_bits(v.x, v.y), bf16x2_bits(v.z, v.w));
  }
}

}  // namespace atts
