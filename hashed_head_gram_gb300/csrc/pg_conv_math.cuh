// Arithmetic of the causal conv + SiLU + residual shared by the kernels that compute it
// (pg_conv.cu's full-sequence and decode kernels and the projection kernel that runs the
// conv behind its tiles), so that every one of them rounds each step the same way.
#pragma once

#include <stdint.h>

#include <type_traits>

namespace pg {
namespace {

// Packed pairs of fp32 (Blackwell f32x2 arithmetic: two lanes per instruction).
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// SiLU(c) = c sigmoid(c) = h + h tanh(h) with h = c / 2 (sigmoid(c) = (1 + tanh(c/2)) / 2):
// from the packed half-argument h, one tanh per element and one packed FMA. The sum
// acc + SiLU(c) is returned as h tanh(h) + (h + acc). Stored in bf16, the outputs take the
// hardware approximation (tanh.approx, one MUFU operation, relative error ~2^-11: far inside
// the bf16 rounding of H); stored in fp32 they take CUDA's tanhf (a few ulp), since the
// approximation alone would put the fp32 result above a 1e-5 relative error.
template <typename T>
__device__ __forceinline__ uint64_t silu2_add(uint64_t h, uint64_t acc) {
  float h0, h1, t0, t1;
  upk(h, h0, h1);
  if constexpr (std::is_same<T, float>::value) {
    t0 = tanhf(h0);
    t1 = tanhf(h1);
  } else {
    asm("tanh.approx.f32 %0, %1;" : "=f"(t0) : "f"(h0));
    asm("tanh.approx.f32 %0, %1;" : "=f"(t1) : "f"(h1));
  }
  return fma2(h, pk(t0, t1), add2(h, acc));
}

// f = alpha / sqrt(alpha^2 mean(v^2) + eps), the RMSNorm factor of u = alpha v, with every
// rounding spelled out so the full-sequence and the decode kernel compute the same value.
__device__ __forceinline__ float tap_scale(float a, float ms, float eps) {
  return __fmul_rn(a, rsqrtf(__fmaf_rn(__fmul_rn(a, a), ms, eps)));
}

}  // namespace
}  // namespace pg
