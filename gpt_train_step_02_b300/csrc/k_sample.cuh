// k_sample.cuh -- one draw from the softmax of a logits row (the page «llm.c：
// Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c», item 5:
// sample_mult picks an index from a probability distribution; the main loop
// generates text with it).
//
// Inverse-CDF sampling with a caller-supplied uniform coin u in [0, 1): the
// token is the first index i < V with  sum_{k <= i} exp(x_k - max) > u * sum_{k < V} exp(x_k - max),
// i.e. the first index whose cumulative softmax probability exceeds u; when
// rounding leaves u * total at or above every prefix, the last index with a
// nonzero weight.  One CTA: every thread owns a contiguous chunk of the row,
// the chunk sums are scanned in thread order (a fixed shuffle tree), and the
// thread whose chunk holds the crossing walks it in index order, so the result
// does not depend on scheduling.  u must lie in [0, 1) (the host checks).
#pragma once
#include "common.cuh"

#define SAMPLE_THREADS 1024

__global__ void __launch_bounds__(SAMPLE_THREADS)
    sample_kernel(int* __restrict__ tokens, int t, const float* __restrict__ row, int V, const float* __restrict__ coins,
                  int coin_index) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[SAMPLE_THREADS / 32], wsum[SAMPLE_THREADS / 32];
  __shared__ float scan[SAMPLE_THREADS];
  __shared__ int last_nonzero[SAMPLE_THREADS / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (V + SAMPLE_THREADS - 1) / SAMPLE_THREADS;
  const int k0 = min(V, tid * chunk), k1 = min(V, k0 + chunk);
  // row max
  float m = -INFINITY;
  for (int k = k0; k < k1; k++) m = fmaxf(m, row[k]);
  m = warp_max(m);
  if (lane == 0) red[warp] = m;
  __syncthreads();
  m = red[0];
  for (int w = 1; w < SAMPLE_THREADS / 32; w++) m = fmaxf(m, red[w]);
  // this thread's chunk sum, in index order
  float s = 0.f;
  int nz = -1;
  for (int k = k0; k < k1; k++) {
    const float e = __expf(row[k] - m);
    s += e;
    if (e > 0.f) nz = k;
  }
  const int nzw = __reduce_max_sync(0xffffffffu, nz);
  // inclusive prefix sums of the chunk sums in thread order: a shuffle scan
  // within each warp, then over the warp totals (a fixed tree)
  float incl = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  if (lane == 0) last_nonzero[warp] = nzw;
  __syncthreads();
  if (warp == 0) {
    float w = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  scan[tid] = incl + (warp > 0 ? wsum[warp - 1] : 0.f);
  __syncthreads();
  const float total = scan[SAMPLE_THREADS - 1];
  const float target = coins[coin_index] * total;
  const float before = tid > 0 ? scan[tid - 1] : 0.f;
  if (before <= target && target < scan[tid] && k0 < k1) {
    // the crossing lies in this chunk: walk it in index order
    float acc = before;
    int pick = k1 - 1;
    for (int k = k0; k < k1; k++) {
      acc += __expf(row[k] - m);
      if (target < acc) {
        pick = k;
        break;
      }
    }
    tokens[t] = pick;
  }
  if (tid == 0 && !(target < total)) {
    // u * total at or above the total (u rounds up to 1): the last nonzero weight
    int last = 0;
    for (int w = 0; w < SAMPLE_THREADS / 32; w++) last = max(last, last_nonzero[w]);
    tokens[t] = last;
  }
}
