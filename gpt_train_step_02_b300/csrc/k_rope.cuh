// k_rope.cuh -- rotary position embedding of q and k for the Llama-style
// variant (the page «千行C代码训完GPT-2» (新智元) names RoPE among the layers
// llm.c adds for Llama2/Gemma-style models).
//
// In the (B*T, 3C) qkv layout, pair (2i, 2i+1) of head h of the q block and of
// the k block of token (b, t) is turned by theta = t * 10000^(-2i/hs):
//   (a, b) -> (a cos - b sin, a sin + b cos);
// inverse != 0 turns by -theta, the transpose, which carries the gradients of
// the rotated q and k back to the matmul outputs.  tab holds (cos, sin) for
// every position and pair, computed once on the host in double precision.
// x is updated in place (fp32); when xbf != NULL the bf16 copy of the same
// elements is rewritten from the rotated fp32 values.
#pragma once
#include "common.cuh"

__global__ void rope_kernel(float* __restrict__ x, uint16_t* __restrict__ xbf, const float2* __restrict__ tab, int B,
                            int T, int C, int NH, int inverse) {
  pdl_launch_dependents();
  pdl_wait();
  const int half = C / NH / 2;                           // pairs per head
  const long long npairs = (long long)B * T * NH * half;  // per block (q or k)
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < npairs;
       e += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(e % half);
    const long long bth = e / half;  // (b*T + t)*NH + h
    const int h = (int)(bth % NH);
    const long long bt = bth / NH;
    const int t = (int)(bt % T);
    const float2 cs = tab[(size_t)t * half + i];
    const float sn = inverse ? -cs.y : cs.y;
#pragma unroll
    for (int part = 0; part < 2; part++) {  // q, then k
      const size_t off = (size_t)bt * 3 * C + (size_t)part * C + (size_t)h * 2 * half + 2 * i;
      const float2 v = *reinterpret_cast<const float2*>(x + off);
      const float2 r = make_float2(v.x * cs.x - v.y * sn, v.x * sn + v.y * cs.x);
      *reinterpret_cast<float2*>(x + off) = r;
      if (xbf) *reinterpret_cast<uint32_t*>(xbf + off) = bf16x2_bits(r.x, r.y);
    }
  }
}
