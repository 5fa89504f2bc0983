// k_attention_simt.cuh -- causal multi-head attention on CUDA cores, for the
// shapes neither the tensor-core kernels (bf16, head size 64, T a multiple of
// 128) nor the one-CTA-per-head kernels (head size 64, T <= 64) take.
//
// Forward (online softmax over keys t2 <= t, scale 1/sqrt(hs)) writes the
// output y (B,T,C) and the log-sum-exp lse (B,NH,T) of each score row.
// Backward recomputes P = exp(S - lse):
//   D_t   = dy_t . y_t                (= sum_t2 P dP)
//   dS    = P (dP - D_t),  dP = dy_t . v_t2
//   dq_t  = scale * sum_t2 dS k_t2,   dk_t2 = scale * sum_t dS q_t,
//   dv_t2 = sum_t P dy_t.
// A CTA of 8 warps owns 8 consecutive rows of one (batch, head): query rows
// (forward, dq) or key rows (dk, dv), one row per warp.  The other side --
// keys and values, or queries, dy, lse and D -- streams through shared
// memory in chunks of 64 rows loaded once per CTA.  Within a chunk lane j
// computes the dot products of rows j and j + 32 (rows padded by one float
// so that the lanes hit distinct banks); the weighted sums are then formed
// with lane l holding head dimensions l, l + 32, ... (ND of them,
// hs <= 32 * ND), the weights broadcast by shuffles.  Every output row is
// produced by one warp in a fixed order, so results are deterministic.
// With bf16_ops the operands (and the softmax weights P, dS entering the
// weighted sums) are rounded to bf16, matching the bf16 workloads.
#pragma once
#include "common.cuh"

#define ATT_ROWS 8    // rows per CTA (one per warp)
#define ATT_CHUNK 64  // streamed rows per shared-memory chunk

GPT2_DEV float att_rnd(float x, int bf16_ops) { return bf16_ops ? round_bf16(x) : x; }

// Shared-memory bytes of the forward / dq kernels: K and V chunks (padded
// pitch hs + 1) plus the 8 rows of q and dy.
static inline size_t att_smem_fwd(int hs) { return (size_t)(2 * ATT_CHUNK * (hs + 1) + 2 * ATT_ROWS * hs) * 4; }
// dk/dv kernel: Q and dy chunks, lse and D of the chunk, the 8 rows of k and v.
static inline size_t att_smem_dkv(int hs) {
  return (size_t)(2 * ATT_CHUNK * (hs + 1) + 2 * ATT_CHUNK + 2 * ATT_ROWS * hs) * 4;
}

// Loads rows r0 .. r0+n-1 (n <= ATT_CHUNK; the rest of the chunk is zero) of
// a head's hs columns into dst[ATT_CHUNK][pitch]; source row r at src + r*ld.
// hs % 4 == 0 and the source rows are 16-byte aligned: each thread issues all
// of its 16-byte loads before it stores any of them.
GPT2_DEV void att_load_chunk(float* dst, int pitch, const float* src, long long ld, int r0, int n, int hs,
                             int bf16_ops) {
  constexpr int MAXV = ATT_CHUNK * 128 / 4 / (ATT_ROWS * 32);  // float4 per thread for hs <= 128
  const int hs4 = hs >> 2, total = ATT_CHUNK * hs4;
  float4 v[MAXV];
#pragma unroll
  for (int u = 0; u < MAXV; u++) {
    const int e = threadIdx.x + u * ATT_ROWS * 32;
    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < total) {
      const int r = e / hs4, d4 = e - r * hs4;
      if (r < n) v[u] = *reinterpret_cast<const float4*>(src + (size_t)(r0 + r) * ld + 4 * d4);
    }
  }
#pragma unroll
  for (int u = 0; u < MAXV; u++) {
    const int e = threadIdx.x + u * ATT_ROWS * 32;
    if (e < total) {
      const int r = e / hs4, d = 4 * (e - r * hs4);
      float* o = dst + r * pitch + d;
      o[0] = att_rnd(v[u].x, bf16_ops);
      o[1] = att_rnd(v[u].y, bf16_ops);
      o[2] = att_rnd(v[u].z, bf16_ops);
      o[3] = att_rnd(v[u].w, bf16_ops);
    }
  }
}

template <int ND>
__global__ void __launch_bounds__(ATT_ROWS * 32)
    attn_fwd_simt_kernel(float* __restrict__ y, uint16_t* __restrict__ ybf, float* __restrict__ lse,
                         const float* __restrict__ qkv, int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  const int hs = C / NH, hp = hs + 1;
  float* KS = sm;
  float* VS = KS + ATT_CHUNK * hp;
  float* QS = VS + ATT_CHUNK * hp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * ATT_ROWS, t = t0 + warp;
  const float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  const long long ld = 3LL * C;
  // this CTA's query rows
  for (int e = threadIdx.x; e < ATT_ROWS * hs; e += blockDim.x) {
    int r = e / hs, d = e - r * hs;
    QS[e] = t0 + r < T ? att_rnd(base[(size_t)(t0 + r) * ld + h * hs + d], bf16_ops) : 0.f;
  }
  float o[ND];
#pragma unroll
  for (int k = 0; k < ND; k++) o[k] = 0.f;
  float m = -INFINITY, l = 0.f;
  const int kend = min(T, t0 + ATT_ROWS);  // keys this CTA needs
  for (int c0 = 0; c0 < kend; c0 += ATT_CHUNK) {
    const int n = min(ATT_CHUNK, kend - c0);
    __syncthreads();
    att_load_chunk(KS, hp, base + C + h * hs, ld, c0, n, hs, bf16_ops);
    att_load_chunk(VS, hp, base + 2 * C + h * hs, ld, c0, n, hs, bf16_ops);
    __syncthreads();
    if (t >= T || c0 > t) continue;
    const float* q = QS + warp * hs;
    float s0 = 0.f, s1 = 0.f;
    for (int d = 0; d < hs; d++) {
      s0 += q[d] * KS[lane * hp + d];
      s1 += q[d] * KS[(lane + 32) * hp + d];
    }
    s0 = c0 + lane <= t ? s0 * scale : -INFINITY;
    s1 = c0 + lane + 32 <= t ? s1 * scale : -INFINITY;
    const float mn = fmaxf(m, warp_max(fmaxf(s0, s1)));
    const float corr = __expf(m - mn);  // 0 on the first chunk (m = -inf)
    const float p0 = __expf(s0 - mn), p1 = __expf(s1 - mn);
    l = l * corr + warp_sum(p0 + p1);
    const float q0 = att_rnd(p0, bf16_ops), q1 = att_rnd(p1, bf16_ops);
#pragma unroll
    for (int k = 0; k < ND; k++) o[k] *= corr;
    const int jn = min(ATT_CHUNK, t - c0 + 1);
    for (int j = 0; j < jn; j++) {
      const float pj = __shfl_sync(0xffffffffu, j < 32 ? q0 : q1, j & 31);
#pragma unroll
      for (int k = 0; k < ND; k++) {
        const int d = lane + 32 * k;
        if (d < hs) o[k] += pj * VS[j * hp + d];
      }
    }
    m = mn;
  }
  if (t >= T) return;
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < ND; k++) {
    const int d = lane + 32 * k;
    if (d < hs) {
      const float out = o[k] * inv;
      y[((size_t)b * T + t) * C + h * hs + d] = out;
      if (ybf) ybf[((size_t)b * T + t) * C + h * hs + d] = to_bf16_bits(out);
    }
  }
  if (lane == 0) lse[((size_t)b * NH + h) * T + t] = m + logf(l);
}

// D[b,h,t] = sum_d dy[b,t,h,d] * y[b,t,h,d], into D and/or, for the tensor-core
// kernels, as the pair LD[b,h,t] = (-lse[b,h,t] log2 e, -D[b,h,t]).
__global__ void attn_bwd_D_kernel(float* __restrict__ D, float2* __restrict__ LD, const float* __restrict__ lse,
                                  const float* __restrict__ dy, const float* __restrict__ y, int B, int T, int C,
                                  int NH) {
  pdl_launch_dependents();
  pdl_wait();
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  size_t off = ((size_t)b * T + t) * C + h * hs;
  float s = 0.f;
  for (int d = lane; d < hs; d += 32) s += dy[off + d] * y[off + d];
  s = warp_sum(s);
  if (lane == 0) {
    const size_t i = ((size_t)b * NH + h) * T + t;
    if (D) D[i] = s;
    if (LD) LD[i] = make_float2(-lse[i] * 1.4426950408889634f, -s);
  }
}

// dq for 8 query rows per CTA; keys and values stream through shared memory.
template <int ND>
__global__ void __launch_bounds__(ATT_ROWS * 32)
    attn_bwd_dq_kernel(float* __restrict__ dqkv, uint16_t* __restrict__ dqkv_bf, const float* __restrict__ qkv,
                       const float* __restrict__ dy, const float* __restrict__ lse, const float* __restrict__ D, int B,
                       int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  const int hs = C / NH, hp = hs + 1;
  float* KS = sm;
  float* VS = KS + ATT_CHUNK * hp;
  float* QS = VS + ATT_CHUNK * hp;
  float* GS = QS + ATT_ROWS * hs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * ATT_ROWS, t = t0 + warp;
  const float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  const long long ld = 3LL * C;
  for (int e = threadIdx.x; e < ATT_ROWS * hs; e += blockDim.x) {
    int r = e / hs, d = e - r * hs;
    bool ok = t0 + r < T;
    QS[e] = ok ? att_rnd(base[(size_t)(t0 + r) * ld + h * hs + d], bf16_ops) : 0.f;
    GS[e] = ok ? att_rnd(dy[((size_t)b * T + t0 + r) * C + h * hs + d], bf16_ops) : 0.f;
  }
  const size_t bh = ((size_t)b * NH + h) * T;
  const float L = t < T ? lse[bh + t] : 0.f, Dt = t < T ? D[bh + t] : 0.f;
  float dq[ND];
#pragma unroll
  for (int k = 0; k < ND; k++) dq[k] = 0.f;
  const int kend = min(T, t0 + ATT_ROWS);
  for (int c0 = 0; c0 < kend; c0 += ATT_CHUNK) {
    const int n = min(ATT_CHUNK, kend - c0);
    __syncthreads();
    att_load_chunk(KS, hp, base + C + h * hs, ld, c0, n, hs, bf16_ops);
    att_load_chunk(VS, hp, base + 2 * C + h * hs, ld, c0, n, hs, bf16_ops);
    __syncthreads();
    if (t >= T || c0 > t) continue;
    const float* q = QS + warp * hs;
    const float* g = GS + warp * hs;
    float s0 = 0.f, s1 = 0.f, dp0 = 0.f, dp1 = 0.f;
    for (int d = 0; d < hs; d++) {
      s0 += q[d] * KS[lane * hp + d];
      s1 += q[d] * KS[(lane + 32) * hp + d];
      dp0 += g[d] * VS[lane * hp + d];
      dp1 += g[d] * VS[(lane + 32) * hp + d];
    }
    const float p0 = c0 + lane <= t ? __expf(s0 * scale - L) : 0.f;
    const float p1 = c0 + lane + 32 <= t ? __expf(s1 * scale - L) : 0.f;
    const float ds0 = att_rnd(p0 * (dp0 - Dt), bf16_ops), ds1 = att_rnd(p1 * (dp1 - Dt), bf16_ops);
    const int jn = min(ATT_CHUNK, t - c0 + 1);
    for (int j = 0; j < jn; j++) {
      const float dsj = __shfl_sync(0xffffffffu, j < 32 ? ds0 : ds1, j & 31);
#pragma unroll
      for (int k = 0; k < ND; k++) {
        const int d = lane + 32 * k;
        if (d < hs) dq[k] += dsj * KS[j * hp + d];
      }
    }
  }
  if (t >= T) return;
#pragma unroll
  for (int k = 0; k < ND; k++) {
    const int d = lane + 32 * k;
    if (d < hs) {
      const size_t o = ((size_t)b * T + t) * 3 * C + h * hs + d;
      dqkv[o] = dq[k] * scale;
      if (dqkv_bf) dqkv_bf[o] = to_bf16_bits(dq[k] * scale);
    }
  }
}

// dk, dv for 8 key rows per CTA; queries, dy, lse and D stream through
// shared memory (the queries t >= the CTA's first key).
template <int ND>
__global__ void __launch_bounds__(ATT_ROWS * 32)
    attn_bwd_dkv_kernel(float* __restrict__ dqkv, uint16_t* __restrict__ dqkv_bf, const float* __restrict__ qkv,
                        const float* __restrict__ dy, const float* __restrict__ lse, const float* __restrict__ D, int B,
                        int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sm[];
  const int hs = C / NH, hp = hs + 1;
  float* QS = sm;
  float* GS = QS + ATT_CHUNK * hp;
  float* LS = GS + ATT_CHUNK * hp;
  float* DS = LS + ATT_CHUNK;
  float* KR = DS + ATT_CHUNK;
  float* VR = KR + ATT_ROWS * hs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * ATT_ROWS, t2 = t0 + warp;  // this warp's key row
  const float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  const long long ld = 3LL * C;
  const size_t bh = ((size_t)b * NH + h) * T;
  for (int e = threadIdx.x; e < ATT_ROWS * hs; e += blockDim.x) {
    int r = e / hs, d = e - r * hs;
    bool ok = t0 + r < T;
    KR[e] = ok ? att_rnd(base[(size_t)(t0 + r) * ld + C + h * hs + d], bf16_ops) : 0.f;
    VR[e] = ok ? att_rnd(base[(size_t)(t0 + r) * ld + 2 * C + h * hs + d], bf16_ops) : 0.f;
  }
  float dk[ND], dv[ND];
#pragma unroll
  for (int k = 0; k < ND; k++) dk[k] = dv[k] = 0.f;
  for (int c0 = t0; c0 < T; c0 += ATT_CHUNK) {
    const int n = min(ATT_CHUNK, T - c0);
    __syncthreads();
    att_load_chunk(QS, hp, base + h * hs, ld, c0, n, hs, bf16_ops);
    att_load_chunk(GS, hp, dy + (size_t)b * T * C + h * hs, C, c0, n, hs, bf16_ops);
    for (int e = threadIdx.x; e < ATT_CHUNK; e += blockDim.x) {
      LS[e] = e < n ? lse[bh + c0 + e] : 0.f;
      DS[e] = e < n ? D[bh + c0 + e] : 0.f;
    }
    __syncthreads();
    if (t2 >= T) continue;
    const float* kr = KR + warp * hs;
    const float* vr = VR + warp * hs;
    float s0 = 0.f, s1 = 0.f, dp0 = 0.f, dp1 = 0.f;
    for (int d = 0; d < hs; d++) {
      s0 += QS[lane * hp + d] * kr[d];
      s1 += QS[(lane + 32) * hp + d] * kr[d];
      dp0 += GS[lane * hp + d] * vr[d];
      dp1 += GS[(lane + 32) * hp + d] * vr[d];
    }
    // query c0 + j attends to this key when c0 + j >= t2 (and c0 + j < T)
    const bool v0 = lane < n && c0 + lane >= t2, v1 = lane + 32 < n && c0 + lane + 32 >= t2;
    const float p0 = v0 ? __expf(s0 * scale - LS[lane]) : 0.f;
    const float p1 = v1 ? __expf(s1 * scale - LS[lane + 32]) : 0.f;
    const float ds0 = att_rnd(p0 * (dp0 - DS[lane]), bf16_ops), ds1 = att_rnd(p1 * (dp1 - DS[lane + 32]), bf16_ops);
    const float r0 = att_rnd(p0, bf16_ops), r1 = att_rnd(p1, bf16_ops);
    for (int j = 0; j < n; j++) {
      const float pj = __shfl_sync(0xffffffffu, j < 32 ? r0 : r1, j & 31);
      const float dsj = __shfl_sync(0xffffffffu, j < 32 ? ds0 : ds1, j & 31);
#pragma unroll
      for (int k = 0; k < ND; k++) {
        const int d = lane + 32 * k;
        if (d < hs) {
          dv[k] += pj * GS[j * hp + d];
          dk[k] += dsj * QS[j * hp + d];
        }
      }
    }
  }
  if (t2 >= T) return;
#pragma unroll
  for (int k = 0; k < ND; k++) {
    const int d = lane + 32 * k;
    if (d < hs) {
      const size_t o = ((size_t)b * T + t2) * 3 * C + C + h * hs + d;
      dqkv[o] = dk[k] * scale;
      dqkv[o + C] = dv[k];
      if (dqkv_bf) {
        dqkv_bf[o] = to_bf16_bits(dk[k] * scale);
        dqkv_bf[o + C] = to_bf16_bits(dv[k]);
      }
    }
  }
}
