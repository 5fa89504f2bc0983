// k_layernorm.cuh -- layernorm forward and backward, one warp per row.
//
// Forward: mean and biased variance over C (two passes over the row held in
// registers), rstd = 1/sqrt(var + 1e-5), y = (x - mean) * rstd * w + b.
// Backward: with n = (x - mean) * rstd and g = dy * w,
//   dx += rstd * (g - mean(g) - n * mean(g * n))     (accumulated in place;
//                                                    optional bf16 copy of dx)
//   dw += sum_rows dy * n,  db += sum_rows dy         (two-stage, fixed order)
// RMS = true gives RMSNorm (the Llama-style variant): no mean is subtracted
// (mean = 0 is stored), rstd = 1/sqrt(mean(x^2) + 1e-5), y = x * rstd * w with
// no shift, and the backward drops the mean(g) term and produces dw only.
// C must be a multiple of 4 and at most 32 * 4 * LN_MAXV4_LIMIT; the kernels
// are instantiated for the per-lane float4 count ceil(C / 128) so that the
// row lives in as few registers as it needs.
#pragma once
#include "common.cuh"

#define LN_MAXV4_LIMIT 10  // float4 elements per lane: C <= 32 * 4 * 10 = 1280
#define LN_EPS 1e-5f

template <int LN_MAXV4, bool RMS>
__global__ void layernorm_fwd_kernel(float* __restrict__ y, uint16_t* __restrict__ ybf, float* __restrict__ mean,
                                     float* __restrict__ rstd, const float* __restrict__ x,
                                     const float* __restrict__ w, const float* __restrict__ b, int N, int C) {
  pdl_launch_dependents();
  pdl_wait();
  int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int lane = threadIdx.x & 31;
  if (warp >= N) return;
  const float* xr = x + (size_t)warp * C;
  float4 v[LN_MAXV4];
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < LN_MAXV4; k++) {
    int c = (lane + 32 * k) * 4;
    if (c < C) {
      v[k] = *reinterpret_cast<const float4*>(xr + c);
      s += (v[k].x + v[k].y) + (v[k].z + v[k].w);
    }
  }
  float mu = RMS ? 0.f : warp_sum(s) / (float)C;
  float q = 0.f;
#pragma unroll
  for (int k = 0; k < LN_MAXV4; k++) {
    int c = (lane + 32 * k) * 4;
    if (c < C) {
      float a = v[k].x - mu, bb = v[k].y - mu, cc = v[k].z - mu, d = v[k].w - mu;
      q += (a * a + bb * bb) + (cc * cc + d * d);
    }
  }
  float var = warp_sum(q) / (float)C;
  float rs = rsqrtf(var + LN_EPS);
#pragma unroll
  for (int k = 0; k < LN_MAXV4; k++) {
    int c = (lane + 32 * k) * 4;
    if (c < C) {
      float4 ww = *reinterpret_cast<const float4*>(w + c);
      const float4 bb = RMS ? make_float4(0.f, 0.f, 0.f, 0.f) : *reinterpret_cast<const float4*>(b + c);
      float4 o;
      o.x = (v[k].x - mu) * rs * ww.x + bb.x;
      o.y = (v[k].y - mu) * rs * ww.y + bb.y;
      o.z = (v[k].z - mu) * rs * ww.z + bb.z;
      o.w = (v[k].w - mu) * rs * ww.w + bb.w;
      if (y) *reinterpret_cast<float4*>(y + (size_t)warp * C + c) = o;
      if (ybf) {
        *reinterpret_cast<uint2*>(ybf + (size_t)warp * C + c) = make_uint2(bf16x2_bits(o.x, o.y), bf16x2_bits(o.z, o.w));
      }
    }
  }
  if (lane == 0) {
    mean[warp] = mu;
    rstd[warp] = rs;
  }
}

// Backward: one row per warp, LNB_WARPS rows per block.  Each warp writes its
// row's contributions dy*n, dy (and, with with_dxsum, the updated dx) to its
// own shared-memory slot; the block then sums the slots column by column in
// warp order and writes partial[blockIdx][0..C) (dw), [C..2C) (db) and
// [2C..3C) (column sums of dx: the bias gradient of the linear layer whose
// output gradient dx is).  Only x and dy of one row live in registers, so
// many warps fit an SM.
#define LNB_WARPS 8
#define LNB_MIN_ROWS LNB_WARPS  // rows per block

template <int LN_MAXV4, bool RMS>
__global__ void __launch_bounds__(LNB_WARPS * 32) layernorm_bwd_kernel(
    float* __restrict__ dx, uint16_t* __restrict__ dxbf, float* __restrict__ partial, const float* __restrict__ dy,
    const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int with_dxsum) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sh[];  // [LNB_WARPS][nout * C]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nout = RMS ? 1 : (with_dxsum ? 3 : 2);  // partial columns: dw [, db [, dx sums]]
  const int r = blockIdx.x * LNB_WARPS + warp;
  float* my = sh + warp * nout * C;
  if (r < N) {
    const float mu = mean[r], rs = rstd[r];
    // every load of the row (x, dy and the dx being accumulated into) is
    // issued before the row reductions
    float4 xv[LN_MAXV4], dv[LN_MAXV4], av[LN_MAXV4];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        xv[k] = *reinterpret_cast<const float4*>(x + (size_t)r * C + c);
        dv[k] = *reinterpret_cast<const float4*>(dy + (size_t)r * C + c);
        av[k] = *reinterpret_cast<const float4*>(dx + (size_t)r * C + c);
      }
    }
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 ww = *reinterpret_cast<const float4*>(w + c);
        const float n0 = (xv[k].x - mu) * rs, n1 = (xv[k].y - mu) * rs, n2 = (xv[k].z - mu) * rs,
                    n3 = (xv[k].w - mu) * rs;
        const float g0 = dv[k].x * ww.x, g1 = dv[k].y * ww.y, g2 = dv[k].z * ww.z, g3 = dv[k].w * ww.w;
        sg += (g0 + g1) + (g2 + g3);
        sgn += (g0 * n0 + g1 * n1) + (g2 * n2 + g3 * n3);
      }
    }
    const float mg = RMS ? 0.f : warp_sum(sg) / (float)C, mgn = warp_sum(sgn) / (float)C;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 ww = *reinterpret_cast<const float4*>(w + c);
        const float4 n = make_float4((xv[k].x - mu) * rs, (xv[k].y - mu) * rs, (xv[k].z - mu) * rs,
                                     (xv[k].w - mu) * rs);
        float4* o = reinterpret_cast<float4*>(dx + (size_t)r * C + c);
        float4 a = av[k];
        a.x += rs * (dv[k].x * ww.x - mg - n.x * mgn);
        a.y += rs * (dv[k].y * ww.y - mg - n.y * mgn);
        a.z += rs * (dv[k].z * ww.z - mg - n.z * mgn);
        a.w += rs * (dv[k].w * ww.w - mg - n.w * mgn);
        *o = a;
        if (dxbf) {
          *reinterpret_cast<uint2*>(dxbf + (size_t)r * C + c) = make_uint2(bf16x2_bits(a.x, a.y), bf16x2_bits(a.z, a.w));
        }
        *reinterpret_cast<float4*>(my + c) = make_float4(dv[k].x * n.x, dv[k].y * n.y, dv[k].z * n.z, dv[k].w * n.w);
        if (!RMS) {
          *reinterpret_cast<float4*>(my + C + c) = dv[k];
          if (with_dxsum) *reinterpret_cast<float4*>(my + 2 * C + c) = a;
        }
      }
    }
  } else {
    for (int c = lane; c < nout * C; c += 32) my[c] = 0.f;
  }
  __syncthreads();
  // column sums of the block's rows, in warp (= row) order
  for (int c = threadIdx.x; c < nout * C; c += blockDim.x) {
    float t = sh[c];
#pragma unroll
    for (int wv = 1; wv < LNB_WARPS; wv++) t += sh[wv * nout * C + c];
    partial[(size_t)blockIdx.x * nout * C + c] = t;
  }
}

// Backward for many rows (the host takes it when there are more row groups
// than twice the SM count): one block per SM, LnbStride::WARPS warps, and
// warp w of block b takes rows b W + w, b W + w + G W, ... (G blocks).  Each
// warp adds its rows' contributions, in row order, into its own
// shared-memory slot; the block then sums its slots in warp order into
// partial[blockIdx][...] (the same three column groups as above), so the
// column finish reads G rows instead of one per eight rows.  The row arithmetic is that of
// layernorm_bwd_kernel.  The warp count fills the register file (x, dy and
// dx of a row live in registers: each of the four schedulers of an SM holds
// a quarter of the warps in its 16K registers) within the shared memory of
// one block.
template <int LN_MAXV4>
struct LnbStride {
  static constexpr int WARPS = LN_MAXV4 >= 8 ? 12 : (LN_MAXV4 >= 6 ? 16 : 20);
};

template <int LN_MAXV4, bool RMS>
__global__ void __launch_bounds__(LnbStride<LN_MAXV4>::WARPS * 32, 1) layernorm_bwd_stride_kernel(
    float* __restrict__ dx, uint16_t* __restrict__ dxbf, float* __restrict__ partial, const float* __restrict__ dy,
    const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int with_dxsum) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int W = LnbStride<LN_MAXV4>::WARPS;
  extern __shared__ float sh[];  // [W][nout * C]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nout = RMS ? 1 : (with_dxsum ? 3 : 2);
  float* my = sh + warp * nout * C;
  for (int c = lane; c < nout * C; c += 32) my[c] = 0.f;
  __syncwarp();
  for (int r = blockIdx.x * W + warp; r < N; r += gridDim.x * W) {
    const float mu = mean[r], rs = rstd[r];
    float4 xv[LN_MAXV4], dv[LN_MAXV4], av[LN_MAXV4];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        xv[k] = *reinterpret_cast<const float4*>(x + (size_t)r * C + c);
        dv[k] = *reinterpret_cast<const float4*>(dy + (size_t)r * C + c);
        av[k] = *reinterpret_cast<const float4*>(dx + (size_t)r * C + c);
      }
    }
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 ww = *reinterpret_cast<const float4*>(w + c);
        const float n0 = (xv[k].x - mu) * rs, n1 = (xv[k].y - mu) * rs, n2 = (xv[k].z - mu) * rs,
                    n3 = (xv[k].w - mu) * rs;
        const float g0 = dv[k].x * ww.x, g1 = dv[k].y * ww.y, g2 = dv[k].z * ww.z, g3 = dv[k].w * ww.w;
        sg += (g0 + g1) + (g2 + g3);
        sgn += (g0 * n0 + g1 * n1) + (g2 * n2 + g3 * n3);
      }
    }
    const float mg = RMS ? 0.f : warp_sum(sg) / (float)C, mgn = warp_sum(sgn) / (float)C;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      const int c = (lane + 32 * k) * 4;
      if (c < C) {
        const float4 ww = *reinterpret_cast<const float4*>(w + c);
        const float4 n = make_float4((xv[k].x - mu) * rs, (xv[k].y - mu) * rs, (xv[k].z - mu) * rs,
                                     (xv[k].w - mu) * rs);
        float4* o = reinterpret_cast<float4*>(dx + (size_t)r * C + c);
        float4 a = av[k];
        a.x += rs * (dv[k].x * ww.x - mg - n.x * mgn);
        a.y += rs * (dv[k].y * ww.y - mg - n.y * mgn);
        a.z += rs * (dv[k].z * ww.z - mg - n.z * mgn);
        a.w += rs * (dv[k].w * ww.w - mg - n.w * mgn);
        *o = a;
        if (dxbf) {
          *reinterpret_cast<uint2*>(dxbf + (size_t)r * C + c) = make_uint2(bf16x2_bits(a.x, a.y), bf16x2_bits(a.z, a.w));
        }
        float4* s0 = reinterpret_cast<float4*>(my + c);
        float4 u = *s0;
        *s0 = make_float4(u.x + dv[k].x * n.x, u.y + dv[k].y * n.y, u.z + dv[k].z * n.z, u.w + dv[k].w * n.w);
        if (!RMS) {
          float4* s1 = reinterpret_cast<float4*>(my + C + c);
          u = *s1;
          *s1 = make_float4(u.x + dv[k].x, u.y + dv[k].y, u.z + dv[k].z, u.w + dv[k].w);
          if (with_dxsum) {
            float4* s2 = reinterpret_cast<float4*>(my + 2 * C + c);
            u = *s2;
            *s2 = make_float4(u.x + a.x, u.y + a.y, u.z + a.z, u.w + a.w);
          }
        }
      }
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nout * C; c += blockDim.x) {
    float t = sh[c];
#pragma unroll 4
    for (int wv = 1; wv < W; wv++) t += sh[wv * nout * C + c];
    partial[(size_t)blockIdx.x * nout * C + c] = t;
  }
}
