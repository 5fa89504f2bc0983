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

#define XENT_THREADS 512

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
  int row = blockIdx.x;
  const float* lr = logits + (size_t)row * Vp;
  float m = -INFINITY, s = 0.f;
  int V4 = Vp >> 2;
  for (int i = threadIdx.x; i < V4; i += XENT_THREADS) {
    float4 x = reinterpret_cast<const float4*>(lr)[i];
    const float* xv = &x.x;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      int v = i * 4 + k;
      if (v < V) {
        if (xv[k] > m) {
          s = s * __expf(m - xv[k]) + 1.f;
          m = xv[k];
        } else {
          s += __expf(xv[k] - m);
        }
      }
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
  int tgt = min(max(targets[row], 0), V - 1);
  if (threadIdx.x == 0) losses[row] = logf(s) + m - lr[tgt];
  float inv = 1.f / s;
  float* dr = dlogits + (size_t)row * Vp;
  for (int i = threadIdx.x; i < V4; i += XENT_THREADS) {
    float4 x = reinterpret_cast<const float4*>(lr)[i];
    float* xv = &x.x;
#pragma unroll
    for (int k = 0; k < 4; k++) {
      int v = i * 4 + k;
      xv[k] = v < V ? (__expf(xv[k] - m) * inv - (v == tgt ? 1.f : 0.f)) * dloss : 0.f;
    }
    if (dlogits) reinterpret_cast<float4*>(dr)[i] = x;
    if (dlogits_bf) {
      ushort4 hb;
      hb.x = to_bf16_bits(x.x);
      hb.y = to_bf16_bits(x.y);
      hb.z = to_bf16_bits(x.z);
      hb.w = to_bf16_bits(x.w);
      reinterpret_cast<ushort4*>(dlogits_bf + (size_t)row * Vp)[i] = hb;
    }
  }
}
