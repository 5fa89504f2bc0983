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
  EPI_LOGITS = 6,      // C = acc, plus the row softmax statistics below (LM head with targets; bf16 kernel)
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
  int fast;       // GELU / GELU' through the hardware tanh approximation (bf16 products)
  // Optional column sums of the fp32 outputs over each 32-row block:
  // colsum[(i / 32) * ldcs + j] = sum of C(i', j) for i' in that block (the
  // first stage of a bias gradient).  Only on the coalesced warp epilogue
  // (vec4, N a multiple of 32); each block is written by exactly one warp.
  float* colsum;
  long long ldcs;
  // EPI_LOGITS: for row i and column block b (the BN/2 columns one epilogue
  // warp finishes), xstats[i * ldxs + b] = (m, s) with m the largest acc(i, j)
  // and s the sum of exp(acc(i, j) - m) over the block's columns j < V
  // (m = -inf, s = 0 when it has none); tlogit[i] = acc(i, targets[i]), in fp32.
  const int* targets;
  int V;
  float2* xstats;
  int ldxs;
  float* tlogit;
  // bf16 in place of the fp32 pre-activation: EPI_BIAS_GELU stores pre(i,j)
  // at pre_bf (pitch ldpre) instead of (or besides) pre; EPI_DGELU reads R
  // from Rbf (pitch ldr) when it is set.
  uint16_t* pre_bf;
  const uint16_t* Rbf;
};

GPT2_DEV float bf16_bits_to_float(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// The epilogue functions take the kind as a template argument OP when the
// caller knows it at compile time (straight-line code per kernel
// instantiation), or read e.epi at run time (OP = -1).
template <int OP>
GPT2_DEV int epi_kind(const EpiArgs& e) {
  return OP >= 0 ? OP : e.epi;
}

template <int OP = -1>
GPT2_DEV void epi_store(const EpiArgs& e, int i, int j, float acc) {
  size_t ci = (size_t)i * e.ldc + j;
  float out;
  switch (epi_kind<OP>(e)) {
    case EPI_BIAS: out = acc + e.bias[j]; break;
    case EPI_BIAS_RESID: out = acc + e.bias[j] + e.R[(size_t)i * e.ldr + j]; break;
    case EPI_BIAS_GELU: {
      float h = acc + e.bias[j];
      if (e.pre) e.pre[(size_t)i * e.ldpre + j] = h;
      if (e.pre_bf) e.pre_bf[(size_t)i * e.ldpre + j] = to_bf16_bits(h);
      out = e.fast ? gelu_fwd_fast(h) : gelu_fwd(h);
      break;
    }
    case EPI_DGELU: {
      const float r = e.Rbf ? bf16_bits_to_float(e.Rbf[(size_t)i * e.ldr + j]) : e.R[(size_t)i * e.ldr + j];
      out = acc * (e.fast ? gelu_grad_fast(r) : gelu_grad(r));
      break;
    }
    case EPI_ACCUM: out = e.C[ci] + acc; break;
    default: out = acc;
  }
  if (e.C) e.C[ci] = out;
  if (e.Cbf) e.Cbf[(size_t)i * e.ldcbf + j] = to_bf16_bits(out);
}

GPT2_DEV float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
GPT2_DEV void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Whether an epilogue reads a per-column bias / a per-element input (R, or C
// for the accumulating product).
GPT2_DEV bool epi_has_bias(int op) { return op == EPI_BIAS || op == EPI_BIAS_RESID || op == EPI_BIAS_GELU; }
GPT2_DEV bool epi_has_input(int op) { return op == EPI_BIAS_RESID || op == EPI_DGELU || op == EPI_ACCUM; }

// The input of element block (i, j .. j+3) an epilogue reads (R or C).
template <int OP = -1>
GPT2_DEV float4 epi_load_input(const EpiArgs& e, int i, int j) {
  if (epi_kind<OP>(e) == EPI_ACCUM) return ld4(e.C + (size_t)i * e.ldc + j);
  if (e.Rbf) {
    const uint2 h = *reinterpret_cast<const uint2*>(e.Rbf + (size_t)i * e.ldr + j);
    return make_float4(__uint_as_float(h.x << 16), __uint_as_float(h.x & 0xffff0000u), __uint_as_float(h.y << 16),
                       __uint_as_float(h.y & 0xffff0000u));
  }
  return ld4(e.R + (size_t)i * e.ldr + j);
}

// Finishes (i, j .. j+3) from the accumulator, the column bias b and the
// element input in (both already loaded when the epilogue needs them).
// vec4 must hold.
template <int OP = -1>
GPT2_DEV float4 epi_apply4(const EpiArgs& e, int i, int j, float4 acc, float4 b, float4 in) {
  float4 o = acc;
  // paired adds in the order of the scalar expressions (acc + b) + in: the same roundings
  const float2 a01 = make_float2(acc.x, acc.y), a23 = make_float2(acc.z, acc.w);
  switch (epi_kind<OP>(e)) {
    case EPI_BIAS: {
      const float2 o01 = add2(a01, make_float2(b.x, b.y)), o23 = add2(a23, make_float2(b.z, b.w));
      o = make_float4(o01.x, o01.y, o23.x, o23.y);
      break;
    }
    case EPI_BIAS_RESID: {
      const float2 o01 = add2(add2(a01, make_float2(b.x, b.y)), make_float2(in.x, in.y));
      const float2 o23 = add2(add2(a23, make_float2(b.z, b.w)), make_float2(in.z, in.w));
      o = make_float4(o01.x, o01.y, o23.x, o23.y);
      break;
    }
    case EPI_BIAS_GELU: {
      const float2 h01 = add2(a01, make_float2(b.x, b.y)), h23 = add2(a23, make_float2(b.z, b.w));
      const float4 h = make_float4(h01.x, h01.y, h23.x, h23.y);
      if (e.pre) st4(e.pre + (size_t)i * e.ldpre + j, h);
      if (e.pre_bf)
        *reinterpret_cast<uint2*>(e.pre_bf + (size_t)i * e.ldpre + j) = make_uint2(bf16x2_bits(h.x, h.y), bf16x2_bits(h.z, h.w));
      if (e.fast) {
        const float2 g01 = gelu_fwd_fast2(h01), g23 = gelu_fwd_fast2(h23);
        o = make_float4(g01.x, g01.y, g23.x, g23.y);
      } else {
        o = make_float4(gelu_fwd(h.x), gelu_fwd(h.y), gelu_fwd(h.z), gelu_fwd(h.w));
      }
      break;
    }
    case EPI_DGELU:
      if (e.fast) {
        const float2 o01 = mul2(a01, gelu_grad_fast2(make_float2(in.x, in.y)));
        const float2 o23 = mul2(a23, gelu_grad_fast2(make_float2(in.z, in.w)));
        o = make_float4(o01.x, o01.y, o23.x, o23.y);
      } else
        o = make_float4(acc.x * gelu_grad(in.x), acc.y * gelu_grad(in.y), acc.z * gelu_grad(in.z),
                        acc.w * gelu_grad(in.w));
      break;
    case EPI_ACCUM: o = make_float4(in.x + acc.x, in.y + acc.y, in.z + acc.z, in.w + acc.w); break;
    default: break;
  }
  if (e.C) st4(e.C + (size_t)i * e.ldc + j, o);
  if (e.Cbf) {
    uint2 h;
    h.x = bf16x2_bits(o.x, o.y);
    h.y = bf16x2_bits(o.z, o.w);
    *reinterpret_cast<uint2*>(e.Cbf + (size_t)i * e.ldcbf + j) = h;
  }
  return o;
}

// Finishes 4 consecutive outputs (i, j .. j+3), all inside the matrix.
template <int OP = -1>
GPT2_DEV void epi_store4(const EpiArgs& e, int i, int j, float4 acc) {
  if (!e.vec4) {
    epi_store<OP>(e, i, j, acc.x);
    epi_store<OP>(e, i, j + 1, acc.y);
    epi_store<OP>(e, i, j + 2, acc.z);
    epi_store<OP>(e, i, j + 3, acc.w);
    return;
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  const int op = epi_kind<OP>(e);
  epi_apply4<OP>(e, i, j, acc, epi_has_bias(op) ? ld4(e.bias + j) : z, epi_has_input(op) ? epi_load_input<OP>(e, i, j) : z);
}

// ---- coalesced epilogue of a warp's 32 x 32 sub-tile --------------------------
// Thread `lane` holds row i0 + lane, columns j0 .. j0+31 (from tcgen05.ld).
// The sub-tile is transposed through the warp's own staging area so that one
// warp instruction then covers 4 rows of 32 columns: lane l handles columns
// j0 + 4 (l % 8) .. +3 of rows i0 + l / 8 + 4 k, k = 0 .. 7, every access a
// 16-byte piece of a full 128-byte row segment.  All global loads of the
// sub-tile are issued before any store.  The staging area is 32 rows of 32
// floats with the row's 16-byte groups permuted (group u of row r at
// position u ^ (r % 8)), so that the row writes and the column reads each
// touch every bank once per 8 lanes without padding.
#define EPI_STAGE_FLOATS (32 * 32)

// float offset of column c of row r in the staging area
GPT2_DEV int stage_off(int r, int c) { return r * 32 + ((((c >> 2) ^ (r & 7))) << 2) + (c & 3); }

GPT2_DEV void warp32_stage(float* stage, const float* v, int lane) {
#pragma unroll
  for (int u = 0; u < 8; u++)
    st4(stage + stage_off(lane, 4 * u), make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]));
  __syncwarp();
}

// Raw fp32 store of the staged sub-tile into P (row pitch ldp), rows < M, columns < N.
GPT2_DEV void warp32_store_raw(float* P, long long ldp, const float* stage, int i0, int j0, int M, int N, int lane) {
  const int c = 4 * (lane & 7), rs = lane >> 3, j = j0 + c;
#pragma unroll
  for (int k = 0; k < 8; k++) {
    const int r = rs + 4 * k, i = i0 + r;
    if (i < M && j < N) {
      const float4 a = ld4(stage + stage_off(r, c));
      if (j + 4 <= N && (ldp & 3) == 0) {
        st4(P + (size_t)i * ldp + j, a);
      } else {
        const float a4[4] = {a.x, a.y, a.z, a.w};
        for (int q = 0; q < 4 && j + q < N; q++) P[(size_t)i * ldp + j + q] = a4[q];
      }
    }
  }
  __syncwarp();
}

// Fused epilogue of the staged sub-tile into the product's outputs.
template <int OP = -1>
GPT2_DEV void warp32_epilogue(const EpiArgs& e, const float* stage, int i0, int j0, int M, int N, int lane) {
  const int c = 4 * (lane & 7), rs = lane >> 3, j = j0 + c;
  const int op = epi_kind<OP>(e);
  if (j < N) {
    if (e.vec4 && j + 4 <= N) {
      const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 b = epi_has_bias(op) ? ld4(e.bias + j) : z;
      float4 in[8];
#pragma unroll
      for (int k = 0; k < 8; k++) {
        const int i = i0 + rs + 4 * k;
        in[k] = (epi_has_input(op) && i < M) ? epi_load_input<OP>(e, i, j) : z;
      }
      float4 cs = z;
#pragma unroll
      for (int k = 0; k < 8; k++) {
        const int r = rs + 4 * k, i = i0 + r;
        if (i < M) {
          const float4 o = epi_apply4<OP>(e, i, j, ld4(stage + stage_off(r, c)), b, in[k]);
          cs = make_float4(cs.x + o.x, cs.y + o.y, cs.z + o.z, cs.w + o.w);
        }
      }
      if (e.colsum) {
        // lanes l, l^8, l^16, l^24 hold the same 4 columns for 8 rows each;
        // the caller guarantees every lane of the warp is on this path
#pragma unroll
        for (int off = 8; off < 32; off <<= 1) {
          cs.x += __shfl_xor_sync(0xffffffffu, cs.x, off);
          cs.y += __shfl_xor_sync(0xffffffffu, cs.y, off);
          cs.z += __shfl_xor_sync(0xffffffffu, cs.z, off);
          cs.w += __shfl_xor_sync(0xffffffffu, cs.w, off);
        }
        if (lane < 8) st4(e.colsum + (size_t)(i0 >> 5) * e.ldcs + j, cs);
      }
    } else {
      for (int k = 0; k < 8; k++) {
        const int r = rs + 4 * k, i = i0 + r;
        if (i < M)
          for (int q = 0; q < 4 && j + q < N; q++) epi_store<OP>(e, i, j + q, stage[stage_off(r, c + q)]);
      }
    }
  }
  __syncwarp();
}
