// gemm_common.cuh -- the fused epilogues shared by the matmul kernels.
//
// A linear layer y = x W^T + b needs three products: forward, input
// gradient and weight gradient.  Each output element acc(i,j) of such a
// product is finished by one epilogue (below).  When Cbf is set, every
// output is also stored, rounded to bf16 (nearest even), at Cbf(i,j): the
// operand copy the next bf16 matmul reads.  C may be NULL when only the bf16
// copy is wanted (not with EPI_ACCUM, which reads C).
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
  int vec4;  // every pointer 16-byte aligned and every leading dimension a multiple of 4 (8 for Cbf)
  uint16_t* Cbf;  // optional bf16 copy of the output
  long long ldcbf;
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
  if (e.C) e.C[ci] = out;
  if (e.Cbf) e.Cbf[(size_t)i * e.ldcbf + j] = to_bf16_bits(out);
}

GPT2_DEV float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
GPT2_DEV void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Finishes 32 consecutive outputs (i, j0 .. j0+31) of one row, nvalid of
// them inside the matrix.  With a full chunk and vec4 set, every global load
// of the chunk (bias, R, C) is issued before any arithmetic or store, as
// 16-byte accesses, so a thread waits about one memory latency per chunk.
GPT2_DEV void epi_store_row32(const EpiArgs& e, int i, int j0, const float* v, int nvalid) {
  if (nvalid < 32 || !e.vec4) {
#pragma unroll
    for (int q = 0; q < 32; q++)
      if (q < nvalid) epi_store(e, i, j0 + q, v[q]);
    return;
  }
  float4 in[8], bs[8];
  float* crow = e.C + (size_t)i * e.ldc + j0;
  const int op = e.epi;
  if (op == EPI_BIAS || op == EPI_BIAS_RESID || op == EPI_BIAS_GELU) {
#pragma unroll
    for (int q = 0; q < 8; q++) bs[q] = ld4(e.bias + j0 + 4 * q);
  }
  if (op == EPI_BIAS_RESID || op == EPI_DGELU) {
    const float* rrow = e.R + (size_t)i * e.ldr + j0;
#pragma unroll
    for (int q = 0; q < 8; q++) in[q] = ld4(rrow + 4 * q);
  } else if (op == EPI_ACCUM) {
#pragma unroll
    for (int q = 0; q < 8; q++) in[q] = ld4(crow + 4 * q);
  }
#pragma unroll
  for (int q = 0; q < 8; q++) {
    float o[4];
    const float* b4 = &bs[q].x;
    const float* r4 = &in[q].x;
#pragma unroll
    for (int c = 0; c < 4; c++) {
      float a = v[4 * q + c];
      switch (op) {
        case EPI_BIAS: o[c] = a + b4[c]; break;
        case EPI_BIAS_RESID: o[c] = a + b4[c] + r4[c]; break;
        case EPI_BIAS_GELU: o[c] = a + b4[c]; break;  // pre-activation; GELU below
        case EPI_DGELU: o[c] = a * gelu_grad(r4[c]); break;
        case EPI_ACCUM: o[c] = r4[c] + a; break;
        default: o[c] = a;
      }
    }
    if (op == EPI_BIAS_GELU) {
      st4(e.pre + (size_t)i * e.ldpre + j0 + 4 * q, make_float4(o[0], o[1], o[2], o[3]));
#pragma unroll
      for (int c = 0; c < 4; c++) o[c] = gelu_fwd(o[c]);
    }
    if (e.C) st4(crow + 4 * q, make_float4(o[0], o[1], o[2], o[3]));
    if (e.Cbf) {
      uint2 h;
      h.x = (uint32_t)to_bf16_bits(o[0]) | ((uint32_t)to_bf16_bits(o[1]) << 16);
      h.y = (uint32_t)to_bf16_bits(o[2]) | ((uint32_t)to_bf16_bits(o[3]) << 16);
      *reinterpret_cast<uint2*>(e.Cbf + (size_t)i * e.ldcbf + j0 + 4 * q) = h;
    }
  }
}

// Finishes 4 consecutive outputs (i, j .. j+3), all inside the matrix.
GPT2_DEV void epi_store4(const EpiArgs& e, int i, int j, float4 acc) {
  if (!e.vec4) {
    epi_store(e, i, j, acc.x);
    epi_store(e, i, j + 1, acc.y);
    epi_store(e, i, j + 2, acc.z);
    epi_store(e, i, j + 3, acc.w);
    return;
  }
  float* cp = e.C + (size_t)i * e.ldc + j;
  float4 o = acc;
  switch (e.epi) {
    case EPI_BIAS: {
      float4 b = ld4(e.bias + j);
      o = make_float4(acc.x + b.x, acc.y + b.y, acc.z + b.z, acc.w + b.w);
      break;
    }
    case EPI_BIAS_RESID: {
      float4 b = ld4(e.bias + j), r = ld4(e.R + (size_t)i * e.ldr + j);
      o = make_float4(acc.x + b.x + r.x, acc.y + b.y + r.y, acc.z + b.z + r.z, acc.w + b.w + r.w);
      break;
    }
    case EPI_BIAS_GELU: {
      float4 b = ld4(e.bias + j);
      float4 h = make_float4(acc.x + b.x, acc.y + b.y, acc.z + b.z, acc.w + b.w);
      st4(e.pre + (size_t)i * e.ldpre + j, h);
      o = make_float4(gelu_fwd(h.x), gelu_fwd(h.y), gelu_fwd(h.z), gelu_fwd(h.w));
      break;
    }
    case EPI_DGELU: {
      float4 r = ld4(e.R + (size_t)i * e.ldr + j);
      o = make_float4(acc.x * gelu_grad(r.x), acc.y * gelu_grad(r.y), acc.z * gelu_grad(r.z), acc.w * gelu_grad(r.w));
      break;
    }
    case EPI_ACCUM: {
      float4 c = ld4(cp);
      o = make_float4(c.x + acc.x, c.y + acc.y, c.z + acc.z, c.w + acc.w);
      break;
    }
    default: break;
  }
  if (e.C) st4(cp, o);
  if (e.Cbf) {
    uint2 h;
    h.x = (uint32_t)to_bf16_bits(o.x) | ((uint32_t)to_bf16_bits(o.y) << 16);
    h.y = (uint32_t)to_bf16_bits(o.z) | ((uint32_t)to_bf16_bits(o.w) << 16);
    *reinterpret_cast<uint2*>(e.Cbf + (size_t)i * e.ldcbf + j) = h;
  }
}
