// k_xent.cuh -- fused softmax + cross-entropy + loss gradient, one CTA per
// row of the (BT, Vp) logits.
//
// Pass 1: each thread keeps a running (max, sum of exp) over its strided
// float4 slice of the V real columns; the CTA combines the pairs in a fixed
// tree.  loss = log(sum) + max - logit[target].
// Pass 2: dlogits[v] = (exp(logit[v] - max) / sum - [v == target]) * dloss
// for v < V and 0 for the padded columns [V, Vp), stored in fp32 (dlogits,
// may be NULL) and/or bf16 (dlogits_bf, may be NULL).  Vp % 4 == 0.
#pragma once
#include "common.cuh"

// 1024 threads: at most two CTAs per SM, so the rows being processed
// (2 x 148 x Vp x 4 bytes, 60 MB for GPT-2) stay in the 126 MB L2 and pass 2
// re-reads them from there.  Each thread keeps four float4 loads in flight.
#define XENT_THREADS 1024
#define XENT_UNROLL 4

GPT2_DEV void online_merge(float& m, float& s, float m2, float s2) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = s * __expf(m - mn) + s2 * __expf(m2 - mn);
  m = mn;
}

__global__ void __launch_bounds__(XENT_THREADS) xent_fused_kernel(
    float* __restrict__ dlogits, uint16_t* __restrict__ dlogits_bf, float* __restrict__ losses,
    const float* __restrict__ logits, const int* __restrict__ targets, int V, int Vp, float dloss) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float shm[XENT_THREADS / 32], shs[XENT_THREADS / 32];
  const int row = blockIdx.x;
  const float* lr = logits + (size_t)row * Vp;
  const float4* lr4 = reinterpret_cast<const float4*>(lr);
  float m = -INFINITY, s = 0.f;
  const int V4 = Vp >> 2;
  for (int i0 = threadIdx.x; i0 < V4; i0 += XENT_UNROLL * XENT_THREADS) {
    float4 x[XENT_UNROLL];
#pragma unroll
    for (int u = 0; u < XENT_UNROLL; u++) {
      const int i = i0 + u * XENT_THREADS;
      x[u] = i < V4 ? lr4[i] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < XENT_UNROLL; u++) {
      const int v0 = 4 * (i0 + u * XENT_THREADS);
      float a[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int k = 0; k < 4; k++)
        if (v0 + k >= V) a[k] = -INFINITY;  // padded vocabulary columns
      const float mx = fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
      if (mx == -INFINITY) continue;
      if (mx > m) {
        s *= __expf(m - mx);  // 0 while m = -inf
        m = mx;
      }
      s += __expf(a[0] - m) + __expf(a[1] - m) + __expf(a[2] - m) + __expf(a[3] - m);
    }
  }
  // warp combine
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    shm[warp] = m;
    shs[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < XENT_THREADS / 32 ? shm[lane] : -INFINITY;
    s = lane < XENT_THREADS / 32 ? shs[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      online_merge(m, s, m2, s2);
    }
    if (lane == 0) {
      shm[0] = m;
      shs[0] = s;
    }
  }
  __syncthreads();
  m = shm[0];
  s = shs[0];
  const int tgt = min(max(targets[row], 0), V - 1);
  if (threadIdx.x == 0) losses[row] = logf(s) + m - lr[tgt];
  // pass 2: dlogits[v] = (exp(x_v - m) / s - [v == tgt]) dloss, in base 2:
  // 2^(x_v log2 e - m log2 e) * (dloss / s); 0 for the padded columns
  const float L2E = 1.4426950408889634f, mb = m * L2E, scale = dloss / s;
  const int tgt4 = tgt >> 2, full4 = V >> 2;  // float4 i holds only real columns when i < full4
  float* dr = dlogits + (size_t)row * Vp;
  for (int i0 = threadIdx.x; i0 < V4; i0 += XENT_UNROLL * XENT_THREADS) {
    float4 x[XENT_UNROLL];
#pragma unroll
    for (int u = 0; u < XENT_UNROLL; u++) {
      const int i = i0 + u * XENT_THREADS;
      if (i < V4) x[u] = lr4[i];
    }
#pragma unroll
    for (int u = 0; u < XENT_UNROLL; u++) {
      const int i = i0 + u * XENT_THREADS;
      if (i >= V4) continue;
      float* xv = &x[u].x;
#pragma unroll
      for (int k = 0; k < 4; k++) xv[k] = ex2f_fast(fmaf(xv[k], L2E, -mb)) * scale;
      if (i >= full4) {  // the float4 that straddles V, and the padding
#pragma unroll
        for (int k = 0; k < 4; k++)
          if (4 * i + k >= V) xv[k] = 0.f;
      }
      if (i == tgt4) xv[tgt & 3] -= dloss;
      if (dlogits) reinterpret_cast<float4*>(dr)[i] = x[u];
      if (dlogits_bf)
        reinterpret_cast<uint2*>(dlogits_bf + (size_t)row * Vp)[i] =
            make_uint2(bf16x2_bits(x[u].x, x[u].y), bf16x2_bits(x[u].z, x[u].w));
    }
  }
}

// The cross-entropy of the bf16 workloads.  Their LM-head matmul
// (epilogue EPI_LOGITS) has already left, per row, the softmax statistics of
// each block of columns -- (m, s): the largest real logit and the sum of
// exp(logit - m) -- and the target's logit in fp32, and has stored the logits
// themselves rounded to bf16.  One CTA per row merges the nblk block
// statistics in a fixed order into lse = m + log s, stores
// loss = lse - logit[target], and makes ONE pass over the bf16 row:
// dlogits[v] = (exp(logit[v] - lse) - [v == target]) * dloss for v < V and 0
// for the padded columns [V, Vp), rounded to bf16.  Vp % 8 == 0.
#define XENT_BF_THREADS 512
#define XENT_BF_UNROLL 4

__global__ void __launch_bounds__(XENT_BF_THREADS) xent_bf16_kernel(
    uint16_t* __restrict__ dlogits_bf, float* __restrict__ losses, const uint16_t* __restrict__ logits_bf,
    const float2* __restrict__ xstats, int nblk, int ldxs, const float* __restrict__ tlogit,
    const int* __restrict__ targets, int V, int Vp, float dloss) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float shm[XENT_BF_THREADS / 32], shs[XENT_BF_THREADS / 32];
  const int row = blockIdx.x;
  float m = -INFINITY, s = 0.f;
  const float2* st = xstats + (size_t)row * ldxs;
  for (int b = threadIdx.x; b < nblk; b += XENT_BF_THREADS) {
    const float2 x = st[b];
    online_merge(m, s, x.x, x.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    online_merge(m, s, m2, s2);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    shm[warp] = m;
    shs[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < XENT_BF_THREADS / 32 ? shm[lane] : -INFINITY;
    s = lane < XENT_BF_THREADS / 32 ? shs[lane] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      online_merge(m, s, m2, s2);
    }
    if (lane == 0) {
      shm[0] = m;
      shs[0] = s;
    }
  }
  __syncthreads();
  const float lse = shm[0] + logf(shs[0]);
  const int tgt = min(max(targets[row], 0), V - 1);
  if (threadIdx.x == 0) losses[row] = lse - tlogit[row];
  // dlogits[v] = 2^(x_v log2 e - lse log2 e) * dloss, minus dloss at the target
  const float L2E = 1.4426950408889634f, lb = lse * L2E;
  const uint4* lr = reinterpret_cast<const uint4*>(logits_bf + (size_t)row * Vp);
  uint4* dr = reinterpret_cast<uint4*>(dlogits_bf + (size_t)row * Vp);
  const int n8 = Vp >> 3, full8 = V >> 3;  // uint4 i holds only real columns when i < full8
  for (int i0 = threadIdx.x; i0 < n8; i0 += XENT_BF_UNROLL * XENT_BF_THREADS) {
    uint4 x[XENT_BF_UNROLL];
#pragma unroll
    for (int u = 0; u < XENT_BF_UNROLL; u++) {
      const int i = i0 + u * XENT_BF_THREADS;
      if (i < n8) x[u] = lr[i];
    }
#pragma unroll
    for (int u = 0; u < XENT_BF_UNROLL; u++) {
      const int i = i0 + u * XENT_BF_THREADS;
      if (i >= n8) continue;
      const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
      float d[8];
#pragma unroll
      for (int k = 0; k < 4; k++) {
        d[2 * k] = ex2f_fast(fmaf(__uint_as_float(w[k] << 16), L2E, -lb)) * dloss;
        d[2 * k + 1] = ex2f_fast(fmaf(__uint_as_float(w[k] & 0xffff0000u), L2E, -lb)) * dloss;
      }
      if (i >= full8) {  // the uint4 that straddles V, and the padding
#pragma unroll
        for (int k = 0; k < 8; k++)
          if (8 * i + k >= V) d[k] = 0.f;
      }
      if (i == (tgt >> 3)) {
#pragma unroll
        for (int k = 0; k < 8; k++)
          if (k == (tgt & 7)) d[k] -= dloss;
      }
      dr[i] = make_uint4(bf16x2_bits(d[0], d[1]), bf16x2_bits(d[2], d[3]), bf16x2_bits(d[4], d[5]),
                         bf16x2_bits(d[6], d[7]));
    }
  }
}
