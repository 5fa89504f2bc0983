// k_gemm_simt.cuh -- strided fp32 GEMM on CUDA cores with fused epilogues:
//   acc(i,j) = sum_p A(i,p) B(p,j),  A(i,p) = A[i*a_rs + p*a_cs],
//                                    B(p,j) = B[p*b_rs + j*b_cs].
// One layout-agnostic kernel covers the three matmul shapes of a linear
// layer y = x W^T + b:  forward (A = x, B = W^T), input gradient
// (A = dy, B = W) and weight gradient (A = dy^T, B = x).
#pragma once
#include "common.cuh"
#include "gemm_common.cuh"

struct GemmArgs {
  int M, N, K;
  const float* A;
  long long a_rs, a_cs;
  const float* B;
  long long b_rs, b_cs;
  EpiArgs epi;
  int bf16_ops;  // round both operands to bf16 before multiplying
};

#define SG_BM 64
#define SG_BN 64
#define SG_BK 16

__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs p) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Bs[SG_BK][SG_BN + 4];
  int tid = threadIdx.x;
  int tx = tid & 15, ty = tid >> 4;
  int i0 = blockIdx.y * SG_BM, j0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  bool a_kfast = p.a_cs == 1;  // choose the load order that reads memory contiguously
  bool b_jfast = p.b_cs == 1;
  for (int k0 = 0; k0 < p.K; k0 += SG_BK) {
#pragma unroll
    for (int q = 0; q < 4; q++) {
      int e = tid + 256 * q;
      int ii, kk;
      if (a_kfast) { kk = e % SG_BK; ii = e / SG_BK; } else { ii = e % SG_BM; kk = e / SG_BM; }
      int gi = i0 + ii, gk = k0 + kk;
      float v = (gi < p.M && gk < p.K) ? p.A[(size_t)gi * p.a_rs + (size_t)gk * p.a_cs] : 0.f;
      As[kk][ii] = p.bf16_ops ? round_bf16(v) : v;
      int jj;
      if (b_jfast) { jj = e % SG_BN; kk = e / SG_BN; } else { kk = e % SG_BK; jj = e / SG_BK; }
      int gj = j0 + jj;
      gk = k0 + kk;
      float w = (gj < p.N && gk < p.K) ? p.B[(size_t)gk * p.b_rs + (size_t)gj * p.b_cs] : 0.f;
      Bs[kk][jj] = p.bf16_ops ? round_bf16(w) : w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; kk++) {
      float a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; r++) a[r] = As[kk][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; c++) b[c] = Bs[kk][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; r++)
#pragma unroll
        for (int c = 0; c < 4; c++) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; r++)
#pragma unroll
    for (int c = 0; c < 4; c++) {
      int i = i0 + ty * 4 + r, j = j0 + tx * 4 + c;
      if (i < p.M && j < p.N) epi_store(p.epi, i, j, acc[r][c]);
    }
}

static inline void gemm_simt_launch(const GemmArgs& a, cudaStream_t s) {
  dim3 grid(ceil_div(a.N, SG_BN), ceil_div(a.M, SG_BM));
  gemm_simt_kernel<<<grid, 256, 0, s>>>(a);
}
