// common.cuh -- shared device helpers of libgpt2b300: warp reductions,
// bf16 rounding, the device-side error word and bounded waits.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define GPT2_DEV __device__ __forceinline__

// Device-side error codes written into the handle's error word.  The host
// maps them onto the public status codes at the next synchronisation.
enum DevError : int {
  DEV_OK = 0,
  DEV_ERR_TOKEN_RANGE = 1,  // a token id outside [0, V)
  DEV_ERR_TIMEOUT = 2,      // a bounded mbarrier / flag wait gave up
  DEV_ERR_SHAPE = 3,        // a kernel was launched with a shape it cannot handle
};

// Programmatic dependent launch.  pdl_wait blocks until the kernels this one
// depends on in the stream have completed and their memory is visible (a
// no-op when the kernel was launched without the attribute);
// pdl_launch_dependents lets the next kernel's CTAs be scheduled once every
// CTA of this grid has issued it or exited.
GPT2_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
GPT2_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

GPT2_DEV void dev_set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

GPT2_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

GPT2_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Round an fp32 value to the nearest bf16 (ties to even) and return it as
// fp32; NaN stays NaN.
GPT2_DEV float round_bf16(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  u += 0x7fffu + ((u >> 16) & 1u);
  return __uint_as_float(u & 0xffff0000u);
}

// x rounded to bf16 (nearest even; NaN stays NaN) by the conversion
// instruction; the same value round_bf16 gives for every non-NaN x
GPT2_DEV uint16_t to_bf16_bits(float x) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return h;
}

// 2^x on the special-function unit (relative error near 2^-22; subnormal
// results flush to zero)
GPT2_DEV float ex2f_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// lo and hi rounded to bf16 and packed into one word, lo in the low half
GPT2_DEV uint32_t bf16x2_bits(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// tanh-form GELU used by GPT-2 and its derivative.
#define GELU_SQRT_2_OVER_PI 0.7978845608028654f
#define GELU_COEF 0.044715f

GPT2_DEV float gelu_fwd(float x) {
  float u = GELU_SQRT_2_OVER_PI * (x + GELU_COEF * x * x * x);
  return 0.5f * x * (1.0f + tanhf(u));
}

// The same with the hardware tanh approximation (tanh.approx.f32, relative
// error about 2^-11): used where the result is rounded to bf16 anyway.
GPT2_DEV float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

GPT2_DEV float gelu_fwd_fast(float x) {
  float u = GELU_SQRT_2_OVER_PI * (x + GELU_COEF * x * x * x);
  return 0.5f * x * (1.0f + tanh_fast(u));
}

GPT2_DEV float gelu_grad_fast(float x) {
  float u = GELU_SQRT_2_OVER_PI * (x + GELU_COEF * x * x * x);
  float th = tanh_fast(u);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * GELU_SQRT_2_OVER_PI * (1.0f + 3.0f * GELU_COEF * x * x);
}

GPT2_DEV float gelu_grad(float x) {
  float u = GELU_SQRT_2_OVER_PI * (x + GELU_COEF * x * x * x);
  float th = tanhf(u);
  return 0.5f * (1.0f + th) + 0.5f * x * (1.0f - th * th) * GELU_SQRT_2_OVER_PI * (1.0f + 3.0f * GELU_COEF * x * x);
}

static inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }
