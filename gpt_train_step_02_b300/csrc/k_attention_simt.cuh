// k_attention_simt.cuh -- causal multi-head attention on CUDA cores, one warp
// per (batch, head, row).  Lanes split the head dimension (hs <= 128).
//
// Forward (online softmax over keys t2 <= t, scale 1/sqrt(hs)) writes the
// output y (B,T,C) and the log-sum-exp lse (B,NH,T) of each score row.
// Backward recomputes P = exp(S - lse):
//   D_t   = dy_t . y_t                (= sum_t2 P dP)
//   dS    = P (dP - D_t),  dP = dy_t . v_t2
//   dq_t  = scale * sum_t2 dS k_t2,   dk_t2 = scale * sum_t dS q_t,
//   dv_t2 = sum_t P dy_t.
// Every output row is produced by one warp, so results are deterministic.
#pragma once
#include "common.cuh"

#define ATT_ND 4  // head dims per lane: hs <= 128

__global__ void attn_fwd_simt_kernel(float* __restrict__ y, float* __restrict__ lse, const float* __restrict__ qkv,
                                     int B, int T, int C, int NH, int bf16_ops) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float q[ATT_ND], o[ATT_ND];
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    float qq = d < hs ? base[(size_t)t * 3 * C + h * hs + d] : 0.f;
    q[k] = bf16_ops ? round_bf16(qq) : qq;
    o[k] = 0.f;
  }
  float mx = -INFINITY, l = 0.f;
  for (int t2 = 0; t2 <= t; t2++) {
    const float* kr = base + (size_t)t2 * 3 * C + C + h * hs;
    const float* vr = kr + C;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) {
      int d = lane + 32 * k;
      if (d < hs) s += q[k] * (bf16_ops ? round_bf16(kr[d]) : kr[d]);
    }
    s = warp_sum(s) * scale;
    float mn = fmaxf(mx, s);
    float corr = __expf(mx - mn), p = __expf(s - mn);
    l = l * corr + p;
    float pp = bf16_ops ? round_bf16(p) : p;
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) {
      int d = lane + 32 * k;
      if (d < hs) o[k] = o[k] * corr + pp * (bf16_ops ? round_bf16(vr[d]) : vr[d]);
    }
    mx = mn;
  }
  float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) y[((size_t)b * T + t) * C + h * hs + d] = o[k] * inv;
  }
  if (lane == 0) lse[((size_t)b * NH + h) * T + t] = mx + logf(l);
}

// D[b,h,t] = sum_d dy[b,t,h,d] * y[b,t,h,d]
__global__ void attn_bwd_D_kernel(float* __restrict__ D, const float* __restrict__ dy, const float* __restrict__ y,
                                  int B, int T, int C, int NH) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  size_t off = ((size_t)b * T + t) * C + h * hs;
  float s = 0.f;
  for (int d = lane; d < hs; d += 32) s += dy[off + d] * y[off + d];
  s = warp_sum(s);
  if (lane == 0) D[gw] = s;
}

__global__ void attn_bwd_dq_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv,
                                   const float* __restrict__ dy, const float* __restrict__ lse,
                                   const float* __restrict__ D, int B, int T, int C, int NH, int bf16_ops) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float q[ATT_ND], g[ATT_ND], dq[ATT_ND];
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    float qq = d < hs ? base[(size_t)t * 3 * C + h * hs + d] : 0.f;
    float gg = d < hs ? dy[((size_t)b * T + t) * C + h * hs + d] : 0.f;
    q[k] = bf16_ops ? round_bf16(qq) : qq;
    g[k] = bf16_ops ? round_bf16(gg) : gg;
    dq[k] = 0.f;
  }
  float L = lse[gw], Dt = D[gw];
  for (int t2 = 0; t2 <= t; t2++) {
    const float* kr = base + (size_t)t2 * 3 * C + C + h * hs;
    const float* vr = kr + C;
    float s = 0.f, dp = 0.f;
    float kk[ATT_ND];
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) {
      int d = lane + 32 * k;
      kk[k] = 0.f;
      if (d < hs) {
        kk[k] = bf16_ops ? round_bf16(kr[d]) : kr[d];
        s += q[k] * kk[k];
        dp += g[k] * (bf16_ops ? round_bf16(vr[d]) : vr[d]);
      }
    }
    s = warp_sum(s) * scale;
    dp = warp_sum(dp);
    float p = __expf(s - L);
    float ds = p * (dp - Dt);
    if (bf16_ops) ds = round_bf16(ds);
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) dq[k] += ds * kk[k];
  }
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) dqkv[((size_t)b * T + t) * 3 * C + h * hs + d] = dq[k] * scale;
  }
}

__global__ void attn_bwd_dkv_kernel(float* __restrict__ dqkv, const float* __restrict__ qkv,
                                    const float* __restrict__ dy, const float* __restrict__ lse,
                                    const float* __restrict__ D, int B, int T, int C, int NH, int bf16_ops) {
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t2 = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float kk[ATT_ND], vv[ATT_ND], dk[ATT_ND], dv[ATT_ND];
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    float a = d < hs ? base[(size_t)t2 * 3 * C + C + h * hs + d] : 0.f;
    float c = d < hs ? base[(size_t)t2 * 3 * C + 2 * C + h * hs + d] : 0.f;
    kk[k] = bf16_ops ? round_bf16(a) : a;
    vv[k] = bf16_ops ? round_bf16(c) : c;
    dk[k] = dv[k] = 0.f;
  }
  const float* lse_bh = lse + ((size_t)b * NH + h) * T;
  const float* D_bh = D + ((size_t)b * NH + h) * T;
  for (int t = t2; t < T; t++) {
    const float* qr = base + (size_t)t * 3 * C + h * hs;
    const float* gr = dy + ((size_t)b * T + t) * C + h * hs;
    float s = 0.f, dp = 0.f;
    float q[ATT_ND], g[ATT_ND];
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) {
      int d = lane + 32 * k;
      q[k] = g[k] = 0.f;
      if (d < hs) {
        q[k] = bf16_ops ? round_bf16(qr[d]) : qr[d];
        g[k] = bf16_ops ? round_bf16(gr[d]) : gr[d];
        s += q[k] * kk[k];
        dp += g[k] * vv[k];
      }
    }
    s = warp_sum(s) * scale;
    dp = warp_sum(dp);
    float p = __expf(s - lse_bh[t]);
    float ds = p * (dp - D_bh[t]);
    if (bf16_ops) {
      ds = round_bf16(ds);
      p = round_bf16(p);
    }
#pragma unroll
    for (int k = 0; k < ATT_ND; k++) {
      dv[k] += p * g[k];
      dk[k] += ds * q[k];
    }
  }
#pragma unroll
  for (int k = 0; k < ATT_ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) {
      dqkv[((size_t)b * T + t2) * 3 * C + C + h * hs + d] = dk[k] * scale;
      dqkv[((size_t)b * T + t2) * 3 * C + 2 * C + h * hs + d] = dv[k];
    }
  }
}
