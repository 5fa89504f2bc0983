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

// ---- paired fp32 arithmetic (f32x2), one instruction for two elements, rounded as
// the scalar forms (round to nearest even); the compiler's own pair builtins, so
// that operands stay in register pairs without packing moves ----
GPT2_DEV float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }  // (a.x b.x + c.x, a.y b.y + c.y)
GPT2_DEV float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
GPT2_DEV float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }

// The GELU and its derivative on two elements with the hardware tanh, for the
// bf16 products.  With u = x (c + c k x^2) (c = sqrt(2/pi), k = 0.044715) and
// t = tanh(u): gelu = x/2 + (x/2) t and
// gelu' = (1 + t)/2 + x (1 - t^2) (c/2 + (3/2) c k x^2).
GPT2_DEV float2 gelu_fwd_fast2(float2 x) {
  const float c = GELU_SQRT_2_OVER_PI, ck = GELU_SQRT_2_OVER_PI * GELU_COEF;
  const float2 x2 = mul2(x, x);
  const float2 u = mul2(x, fma2(x2, make_float2(ck, ck), make_float2(c, c)));
  const float2 t = make_float2(tanh_fast(u.x), tanh_fast(u.y));
  const float2 hx = mul2(x, make_float2(0.5f, 0.5f));
  return fma2(hx, t, hx);
}

GPT2_DEV float2 gelu_grad_fast2(float2 x) {
  const float c = GELU_SQRT_2_OVER_PI, ck = GELU_SQRT_2_OVER_PI * GELU_COEF;
  const float d0 = 0.5f * GELU_SQRT_2_OVER_PI, d1 = 1.5f * GELU_SQRT_2_OVER_PI * GELU_COEF;
  const float2 x2 = mul2(x, x);
  const float2 u = mul2(x, fma2(x2, make_float2(ck, ck), make_float2(c, c)));
  const float2 t = make_float2(tanh_fast(u.x), tanh_fast(u.y));
  const float2 a = fma2(t, make_float2(0.5f, 0.5f), make_float2(0.5f, 0.5f));  // (1 + t) / 2
  const float2 s = fma2(make_float2(-t.x, -t.y), t, make_float2(1.f, 1.f));     // 1 - t^2
  const float2 d = fma2(x2, make_float2(d1, d1), make_float2(d0, d0));
  return fma2(mul2(x, s), d, a);
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
