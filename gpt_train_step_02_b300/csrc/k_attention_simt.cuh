// k_attention_simt.cuh -- causal multi-head attention on CUDA cores, one warp
// per (batch, head, row).  Lane l holds head dimensions l, l+32, ... (ND of
// them, hs <= 32 * ND).
//
// Forward (online softmax over keys t2 <= t, scale 1/sqrt(hs)) writes the
// output y (B,T,C) and the log-sum-exp lse (B,NH,T) of each score row.
// Backward recomputes P = exp(S - lse):
//   D_t   = dy_t . y_t                (= sum_t2 P dP)
//   dS    = P (dP - D_t),  dP = dy_t . v_t2
//   dq_t  = scale * sum_t2 dS k_t2,   dk_t2 = scale * sum_t dS q_t,
//   dv_t2 = sum_t P dy_t.
// Keys (or queries, for dk/dv) are visited in blocks of ATT_KB rows whose
// global loads are all issued before the block's arithmetic, so a warp waits
// about one memory latency per block rather than one per key.  Every output
// row is produced by one warp in a fixed order, so results are deterministic.
#pragma once
#include "common.cuh"

#define ATT_KB 8

template <int ND>
GPT2_DEV void att_load_row(float (&dst)[ND], const float* row, int lane, int hs, bool valid, int bf16_ops) {
#pragma unroll
  for (int k = 0; k < ND; k++) {
    int d = lane + 32 * k;
    float a = 0.f;
    if (valid && d < hs) a = row[d];
    dst[k] = bf16_ops ? round_bf16(a) : a;
  }
}

template <int ND>
__global__ void attn_fwd_simt_kernel(float* __restrict__ y, uint16_t* __restrict__ ybf, float* __restrict__ lse,
                                     const float* __restrict__ qkv, int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float q[ND], o[ND];
  att_load_row<ND>(q, base + (size_t)t * 3 * C + h * hs, lane, hs, true, bf16_ops);
#pragma unroll
  for (int k = 0; k < ND; k++) o[k] = 0.f;
  float mx = -INFINITY, l = 0.f;
  for (int t0 = 0; t0 <= t; t0 += ATT_KB) {
    float kk[ATT_KB][ND], vv[ATT_KB][ND];
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      const float* kr = base + (size_t)(t0 + u) * 3 * C + C + h * hs;
      att_load_row<ND>(kk[u], kr, lane, hs, t0 + u <= t, bf16_ops);
      att_load_row<ND>(vv[u], kr + C, lane, hs, t0 + u <= t, bf16_ops);
    }
    float sc[ATT_KB];
    float mn = mx;
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      float s = 0.f;
#pragma unroll
      for (int k = 0; k < ND; k++) s += q[k] * kk[u][k];
      s = warp_sum(s) * scale;
      sc[u] = t0 + u <= t ? s : -INFINITY;
      mn = fmaxf(mn, sc[u]);
    }
    float corr = __expf(mx - mn);  // 0 on the first block (mx = -inf)
    l *= corr;
#pragma unroll
    for (int k = 0; k < ND; k++) o[k] *= corr;
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      float p = t0 + u <= t ? __expf(sc[u] - mn) : 0.f;
      l += p;
      float pp = bf16_ops ? round_bf16(p) : p;
#pragma unroll
      for (int k = 0; k < ND; k++) o[k] += pp * vv[u][k];
    }
    mx = mn;
  }
  float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) {
      float out = o[k] * inv;
      y[((size_t)b * T + t) * C + h * hs + d] = out;
      if (ybf) ybf[((size_t)b * T + t) * C + h * hs + d] = to_bf16_bits(out);
    }
  }
  if (lane == 0) lse[((size_t)b * NH + h) * T + t] = mx + logf(l);
}

// D[b,h,t] = sum_d dy[b,t,h,d] * y[b,t,h,d]
__global__ void attn_bwd_D_kernel(float* __restrict__ D, const float* __restrict__ dy, const float* __restrict__ y,
                                  int B, int T, int C, int NH) {
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
  if (lane == 0) D[gw] = s;
}

template <int ND>
__global__ void attn_bwd_dq_kernel(float* __restrict__ dqkv, uint16_t* __restrict__ dqkv_bf, const float* __restrict__ qkv,
                                   const float* __restrict__ dy, const float* __restrict__ lse,
                                   const float* __restrict__ D, int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float q[ND], g[ND], dq[ND];
  att_load_row<ND>(q, base + (size_t)t * 3 * C + h * hs, lane, hs, true, bf16_ops);
  att_load_row<ND>(g, dy + ((size_t)b * T + t) * C + h * hs, lane, hs, true, bf16_ops);
#pragma unroll
  for (int k = 0; k < ND; k++) dq[k] = 0.f;
  float L = lse[gw], Dt = D[gw];
  for (int t0 = 0; t0 <= t; t0 += ATT_KB) {
    float kk[ATT_KB][ND], vv[ATT_KB][ND];
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      const float* kr = base + (size_t)(t0 + u) * 3 * C + C + h * hs;
      att_load_row<ND>(kk[u], kr, lane, hs, t0 + u <= t, bf16_ops);
      att_load_row<ND>(vv[u], kr + C, lane, hs, t0 + u <= t, bf16_ops);
    }
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int k = 0; k < ND; k++) {
        s += q[k] * kk[u][k];
        dp += g[k] * vv[u][k];
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      float p = t0 + u <= t ? __expf(s - L) : 0.f;
      float ds = p * (dp - Dt);
      if (bf16_ops) ds = round_bf16(ds);
#pragma unroll
      for (int k = 0; k < ND; k++) dq[k] += ds * kk[u][k];
    }
  }
#pragma unroll
  for (int k = 0; k < ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) {
      size_t o = ((size_t)b * T + t) * 3 * C + h * hs + d;
      dqkv[o] = dq[k] * scale;
      if (dqkv_bf) dqkv_bf[o] = to_bf16_bits(dq[k] * scale);
    }
  }
}

template <int ND>
__global__ void attn_bwd_dkv_kernel(float* __restrict__ dqkv, uint16_t* __restrict__ dqkv_bf, const float* __restrict__ qkv,
                                    const float* __restrict__ dy, const float* __restrict__ lse,
                                    const float* __restrict__ D, int B, int T, int C, int NH, int bf16_ops) {
  pdl_launch_dependents();
  pdl_wait();
  int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (gw >= B * NH * T) return;
  int t2 = gw % T, h = (gw / T) % NH, b = gw / (T * NH);
  int hs = C / NH;
  float scale = rsqrtf((float)hs);
  const float* base = qkv + (size_t)b * T * 3 * C;
  float kk[ND], vv[ND], dk[ND], dv[ND];
  att_load_row<ND>(kk, base + (size_t)t2 * 3 * C + C + h * hs, lane, hs, true, bf16_ops);
  att_load_row<ND>(vv, base + (size_t)t2 * 3 * C + 2 * C + h * hs, lane, hs, true, bf16_ops);
#pragma unroll
  for (int k = 0; k < ND; k++) dk[k] = dv[k] = 0.f;
  const float* lse_bh = lse + ((size_t)b * NH + h) * T;
  const float* D_bh = D + ((size_t)b * NH + h) * T;
  for (int t0 = t2; t0 < T; t0 += ATT_KB) {
    float qq[ATT_KB][ND], gg[ATT_KB][ND], Lt[ATT_KB], Dt[ATT_KB];
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      int t = t0 + u;
      bool valid = t < T;
      att_load_row<ND>(qq[u], base + (size_t)t * 3 * C + h * hs, lane, hs, valid, bf16_ops);
      att_load_row<ND>(gg[u], dy + ((size_t)b * T + t) * C + h * hs, lane, hs, valid, bf16_ops);
      Lt[u] = 0.f;
      Dt[u] = 0.f;
      if (valid) {
        Lt[u] = lse_bh[t];
        Dt[u] = D_bh[t];
      }
    }
#pragma unroll
    for (int u = 0; u < ATT_KB; u++) {
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int k = 0; k < ND; k++) {
        s += qq[u][k] * kk[k];
        dp += gg[u][k] * vv[k];
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      float p = t0 + u < T ? __expf(s - Lt[u]) : 0.f;
      float ds = p * (dp - Dt[u]);
      if (bf16_ops) {
        ds = round_bf16(ds);
        p = round_bf16(p);
      }
#pragma unroll
      for (int k = 0; k < ND; k++) {
        dv[k] += p * gg[u][k];
        dk[k] += ds * qq[u][k];
      }
    }
  }
#pragma unroll
  for (int k = 0; k < ND; k++) {
    int d = lane + 32 * k;
    if (d < hs) {
      size_t o = ((size_t)b * T + t2) * 3 * C + C + h * hs + d;
      dqkv[o] = dk[k] * scale;
      dqkv[o + C] = dv[k];
      if (dqkv_bf) {
        dqkv_bf[o] = to_bf16_bits(dk[k] * scale);
        dqkv_bf[o + C] = to_bf16_bits(dv[k]);
      }
    }
  }
}
