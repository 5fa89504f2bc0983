// gemm_common.cuh -- the fused epilogues shared by the matmul kernels.
//
// A linear layer y = x W^T + b needs three products: forward, input
// gradient and weight gradient.  Each output element acc(i,j) of such a
// product is finished by one epilogue:
#pragma once
#include "common.cuh"

enum GemmEpi : int {
  EPI_STORE = 0,       // C = acc
  EPI_BIAS = 1,        // C = acc + bias[j]
  EPI_BIAS_RESID = 2,  // C = acc + bias[j] + R(i,j)            (residual add)
  EPI_BIAS_GELU = 3,   // pre(i,j) = acc + bias[j]; C = gelu(pre) (MLP input projection)
  EPI_DGELU = 4,       // C = acc * gelu'(R(i,j))                (input gradient through GELU)
  EPI_ACCUM = 5,       // C += acc                               (weight gradient accumulation)
};

struct EpiArgs {
  float* C;
  long long ldc;
  const float* bias;
  const float* R;
  long long ldr;
  float* pre;
  long long ldpre;
  int epi;
};

GPT2_DEV void epi_store(const EpiArgs& e, int i, int j, float acc) {
  size_t ci = (size_t)i * e.ldc + j;
  float out;
  switch (e.epi) {
    case EPI_BIAS: out = acc + e.bias[j]; break;
    case EPI_BIAS_RESID: out = acc + e.bias[j] + e.R[(size_t)i * e.ldr + j]; break;
    case EPI_BIAS_GELU: {
      float h = acc + e.bias[j];
      e.pre[(size_t)i * e.ldpre + j] = h;
      out = gelu_fwd(h);
      break;
    }
    case EPI_DGELU: out = acc * gelu_grad(e.R[(size_t)i * e.ldr + j]); break;
    case EPI_ACCUM: out = e.C[ci] + acc; break;
    default: out = acc;
  }
  e.C[ci] = out;
}

// Split-K finish: out(i,j) = epilogue(sum_z partial[z][i][j]), the partials
// summed in split order (deterministic).  One thread per output element.
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int splits, int M, int N, EpiArgs e) {
  long long total = (long long)M * N;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int z = 0; z < splits; z++) s += partial[(size_t)z * total + idx];
    epi_store(e, (int)(idx / N), (int)(idx % N), s);
  }
}
