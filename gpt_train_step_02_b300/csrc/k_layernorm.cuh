// k_layernorm.cuh -- layernorm forward and backward, one warp per row.
//
// Forward: mean and biased variance over C (two passes over the row held in
// registers), rstd = 1/sqrt(var + 1e-5), y = (x - mean) * rstd * w + b.
// Backward: with n = (x - mean) * rstd and g = dy * w,
//   dx += rstd * (g - mean(g) - n * mean(g * n))     (accumulated in place;
//                                                    optional bf16 copy of dx)
//   dw += sum_rows dy * n,  db += sum_rows dy         (two-stage, fixed order)
// C must be a multiple of 4 and at most 32 * 4 * LN_MAXV4_LIMIT; the kernels
// are instantiated for the per-lane float4 count ceil(C / 128) so that the
// row lives in as few registers as it needs.
#pragma once
#include "common.cuh"

#define LN_MAXV4_LIMIT 10  // float4 elements per lane: C <= 32 * 4 * 10 = 1280
#define LN_EPS 1e-5f

template <int LN_MAXV4>
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
  float mu = warp_sum(s) / (float)C;
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
      float4 bb = *reinterpret_cast<const float4*>(b + c);
      float4 o;
      o.x = (v[k].x - mu) * rs * ww.x + bb.x;
      o.y = (v[k].y - mu) * rs * ww.y + bb.y;
      o.z = (v[k].z - mu) * rs * ww.z + bb.z;
      o.w = (v[k].w - mu) * rs * ww.w + bb.w;
      if (y) *reinterpret_cast<float4*>(y + (size_t)warp * C + c) = o;
      if (ybf) {
        ushort4 h;
        h.x = to_bf16_bits(o.x);
        h.y = to_bf16_bits(o.y);
        h.z = to_bf16_bits(o.z);
        h.w = to_bf16_bits(o.w);
        *reinterpret_cast<ushort4*>(ybf + (size_t)warp * C + c) = h;
      }
    }
  }
  if (lane == 0) {
    mean[warp] = mu;
    rstd[warp] = rs;
  }
}

// Block = LNB_WARPS warps covering `rows` consecutive rows (a multiple of
// LNB_WARPS, at least LNB_MIN_ROWS; the host picks it so that the grid
// covers the SMs).  Writes the block's dw/db partial sums (rows in order,
// warps in order) to partial[blockIdx][0..C) and partial[blockIdx][C..2C).
#define LNB_WARPS 8
#define LNB_MIN_ROWS 8

template <int LN_MAXV4>
__global__ void __launch_bounds__(LNB_WARPS * 32) layernorm_bwd_kernel(
    float* __restrict__ dx, uint16_t* __restrict__ dxbf, float* __restrict__ partial, const float* __restrict__ dy,
    const float* __restrict__ x, const float* __restrict__ w, const float* __restrict__ mean,
    const float* __restrict__ rstd, int N, int C, int rows) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float sh[];  // [2C]
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4 aw[LN_MAXV4], ab[LN_MAXV4];
#pragma unroll
  for (int k = 0; k < LN_MAXV4; k++) aw[k] = ab[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  int r0 = blockIdx.x * rows;
  for (int r = r0 + warp; r < min(N, r0 + rows); r += LNB_WARPS) {
    float mu = mean[r], rs = rstd[r];
    float4 n[LN_MAXV4], g[LN_MAXV4], d[LN_MAXV4];
    float sg = 0.f, sgn = 0.f;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      int c = (lane + 32 * k) * 4;
      if (c < C) {
        float4 xx = *reinterpret_cast<const float4*>(x + (size_t)r * C + c);
        d[k] = *reinterpret_cast<const float4*>(dy + (size_t)r * C + c);
        float4 ww = *reinterpret_cast<const float4*>(w + c);
        n[k] = make_float4((xx.x - mu) * rs, (xx.y - mu) * rs, (xx.z - mu) * rs, (xx.w - mu) * rs);
        g[k] = make_float4(d[k].x * ww.x, d[k].y * ww.y, d[k].z * ww.z, d[k].w * ww.w);
        sg += (g[k].x + g[k].y) + (g[k].z + g[k].w);
        sgn += (g[k].x * n[k].x + g[k].y * n[k].y) + (g[k].z * n[k].z + g[k].w * n[k].w);
      }
    }
    float mg = warp_sum(sg) / (float)C, mgn = warp_sum(sgn) / (float)C;
#pragma unroll
    for (int k = 0; k < LN_MAXV4; k++) {
      int c = (lane + 32 * k) * 4;
      if (c < C) {
        float4* o = reinterpret_cast<float4*>(dx + (size_t)r * C + c);
        float4 a = *o;
        a.x += rs * (g[k].x - mg - n[k].x * mgn);
        a.y += rs * (g[k].y - mg - n[k].y * mgn);
        a.z += rs * (g[k].z - mg - n[k].z * mgn);
        a.w += rs * (g[k].w - mg - n[k].w * mgn);
        *o = a;
        if (dxbf) {
          ushort4 hb;
          hb.x = to_bf16_bits(a.x);
          hb.y = to_bf16_bits(a.y);
          hb.z = to_bf16_bits(a.z);
          hb.w = to_bf16_bits(a.w);
          *reinterpret_cast<ushort4*>(dxbf + (size_t)r * C + c) = hb;
        }
        aw[k].x += d[k].x * n[k].x; aw[k].y += d[k].y * n[k].y;
        aw[k].z += d[k].z * n[k].z; aw[k].w += d[k].w * n[k].w;
        ab[k].x += d[k].x; ab[k].y += d[k].y; ab[k].z += d[k].z; ab[k].w += d[k].w;
      }
    }
  }
  // combine the warps' partials in warp order
  for (int wv = 0; wv < LNB_WARPS; wv++) {
    if (warp == wv) {
#pragma unroll
      for (int k = 0; k < LN_MAXV4; k++) {
        int c = (lane + 32 * k) * 4;
        if (c < C) {
          float4* pw = reinterpret_cast<float4*>(sh + c);
          float4* pb = reinterpret_cast<float4*>(sh + C + c);
          if (wv == 0) {
            *pw = aw[k];
            *pb = ab[k];
          } else {
            float4 a = *pw, bb = *pb;
            *pw = make_float4(a.x + aw[k].x, a.y + aw[k].y, a.z + aw[k].z, a.w + aw[k].w);
            *pb = make_float4(bb.x + ab[k].x, bb.y + ab[k].y, bb.z + ab[k].z, bb.w + ab[k].w);
          }
        }
      }
    }
    __syncthreads();
  }
  for (int c = threadIdx.x; c < 2 * C; c += blockDim.x) partial[(size_t)blockIdx.x * 2 * C + c] = sh[c];
}

