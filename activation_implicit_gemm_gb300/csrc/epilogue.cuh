// Fused epilogue math shared by every kernel of the library: the activation of a
// pre-activation value v = acc + B[m] + Z[n,m,o], computed in fp32 (README
// "Attributes": the activation list and activation_params). The one rounding to T
// happens after the activation, as the f16 subgroup-matrix variants of the package
// describe it (f32 accumulation, then bias, residual, activation and f16 rounding).
#pragma once

#include <cuda_fp16.h>

#include "fconv_internal.h"

namespace fconv {

__device__ __forceinline__ float gelu_tanh_f(float v) {
  const float k = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * v * (1.0f + tanhf(k * (v + 0.044715f * v * v * v)));
}

// act(v) for the activation ids of fconv_act; alpha/beta are the resolved parameters.
__device__ __forceinline__ float apply_act(int act, float v, float alpha, float beta) {
  switch (act) {
    case FCONV_ACT_NONE: return v;
    case FCONV_ACT_RELU: return fmaxf(v, 0.0f);
    case FCONV_ACT_LEAKYRELU: return v < 0.0f ? alpha * v : v;
    case FCONV_ACT_SIGMOID: return 1.0f / (1.0f + expf(-v));
    case FCONV_ACT_TANH: return tanhf(v);
    case FCONV_ACT_HARDSIGMOID: return fminf(fmaxf(alpha * v + beta, 0.0f), 1.0f);
    case FCONV_ACT_HARDSWISH: return v * fminf(fmaxf(v * (1.0f / 6.0f) + 0.5f, 0.0f), 1.0f);
    case FCONV_ACT_CLIP: return fminf(fmaxf(v, alpha), beta);
    case FCONV_ACT_QUICKGELU: return v / (1.0f + expf(-alpha * v));
    case FCONV_ACT_ELU: return v > 0.0f ? v : alpha * expm1f(v);
    case FCONV_ACT_GELU:
      if (alpha != 0.0f) return gelu_tanh_f(v);
      return 0.5f * v * (1.0f + erff(v * 0.7071067811865476f));
    case FCONV_ACT_FASTGELU: return gelu_tanh_f(v);
    case FCONV_ACT_SOFTPLUS: return fmaxf(v, 0.0f) + log1pf(expf(-fabsf(v)));
    case FCONV_ACT_THRESHOLDEDRELU: return v > alpha ? v : 0.0f;
    case FCONV_ACT_ERF: return erff(v);
    default: return v;
  }
}


// act(v) with the activation fixed at compile time. FAST selects __expf-based
// exponentials (relative error ~1e-7, far below an f16 rounding) for f16 outputs;
// f32 outputs use the accurate library functions. Dispatching once per group of
// outputs (FCONV_ACT_SWITCH) keeps one activation's code in the instruction stream
// instead of all fifteen.
// sigmoid(t) = (1 + tanh(t / 2)) / 2 with the hardware tanh approximation (relative
// error about 2^-11 on tanh, so the sigmoid's error stays below 2.5e-4 absolute and
// 5e-4 relative): one special-function operation instead of an exponential and a
// reciprocal. Used only for f16 outputs.
__device__ __forceinline__ float sigmoid_fast(float t) {
  float th;
  asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * t));
  return fmaf(0.5f, th, 0.5f);
}

// Hardware approximations (PTX rcp.approx / ex2.approx): relative error a few ulp of f32.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Exact (erf) GELU, x * Phi(x), with Phi(x) = 1 - erfc(x / sqrt 2) / 2 for x >= 0 and
// erfc(|x| / sqrt 2) / 2 for x < 0. erfc(z) for z >= 0 is Hastings' rational
// approximation as tabulated in Abramowitz & Stegun, Handbook of Mathematical Functions,
// formula 7.1.26: t = 1 / (1 + p z), erfc(z) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5)
// exp(-z^2), |error| <= 1.5e-7. With the approximate reciprocal and exponential the
// error of Phi stays below 3e-7 absolute, far below an f16 rounding of x * Phi(x).
// Used only for f16 outputs.
__device__ __forceinline__ float gelu_erf_fast(float x) {
  const float z = fabsf(x) * 0.70710678118654752f;
  const float t = rcp_approx(fmaf(0.3275911f, z, 1.0f));
  float p = fmaf(1.061405429f, t, -1.453152027f);
  p = fmaf(p, t, 1.421413741f);
  p = fmaf(p, t, -0.284496736f);
  p = fmaf(p, t, 0.254829592f);
  const float q = p * t * ex2_approx(-1.4426950408889634f * z * z);  // erfc(z)
  const float phi = x >= 0.0f ? fmaf(-0.5f, q, 1.0f) : 0.5f * q;
  return x * phi;
}

template <int ACT, bool FAST>
__device__ __forceinline__ float act_eval(float v, float alpha, float beta) {
  if constexpr (ACT == FCONV_ACT_NONE) {
    return v;
  } else if constexpr (ACT == FCONV_ACT_RELU) {
    return fmaxf(v, 0.0f);
  } else if constexpr (ACT == FCONV_ACT_LEAKYRELU) {
    return v < 0.0f ? alpha * v : v;
  } else if constexpr (ACT == FCONV_ACT_SIGMOID) {
    return FAST ? sigmoid_fast(v) : 1.0f / (1.0f + expf(-v));
  } else if constexpr (ACT == FCONV_ACT_TANH) {
    return tanhf(v);
  } else if constexpr (ACT == FCONV_ACT_HARDSIGMOID) {
    return fminf(fmaxf(alpha * v + beta, 0.0f), 1.0f);
  } else if constexpr (ACT == FCONV_ACT_HARDSWISH) {
    return v * fminf(fmaxf(v * (1.0f / 6.0f) + 0.5f, 0.0f), 1.0f);
  } else if constexpr (ACT == FCONV_ACT_CLIP) {
    return fminf(fmaxf(v, alpha), beta);
  } else if constexpr (ACT == FCONV_ACT_QUICKGELU) {
    return FAST ? v * sigmoid_fast(alpha * v) : v / (1.0f + expf(-alpha * v));
  } else if constexpr (ACT == FCONV_ACT_ELU) {
    return v > 0.0f ? v : alpha * (FAST ? (__expf(v) - 1.0f) : expm1f(v));
  } else if constexpr (ACT == FCONV_ACT_GELU) {
    if (alpha != 0.0f) return gelu_tanh_f(v);
    return FAST ? gelu_erf_fast(v) : 0.5f * v * (1.0f + erff(v * 0.7071067811865476f));
  } else if constexpr (ACT == FCONV_ACT_FASTGELU) {
    return gelu_tanh_f(v);
  } else if constexpr (ACT == FCONV_ACT_SOFTPLUS) {
    return FAST ? fmaxf(v, 0.0f) + __logf(1.0f + __expf(-fabsf(v)))
                : fmaxf(v, 0.0f) + log1pf(expf(-fabsf(v)));
  } else if constexpr (ACT == FCONV_ACT_THRESHOLDEDRELU) {
    return v > alpha ? v : 0.0f;
  } else {
    return erff(v);
  }
}

// Calls BODY(ACT) with ACT a compile-time activation id equal to the runtime `act`.
#define FCONV_ACT_SWITCH(act, BODY)                        \
  switch (act) {                                           \
    case FCONV_ACT_RELU: BODY(FCONV_ACT_RELU); break;      \
    case FCONV_ACT_LEAKYRELU: BODY(FCONV_ACT_LEAKYRELU); break; \
    case FCONV_ACT_SIGMOID: BODY(FCONV_ACT_SIGMOID); break; \
    case FCONV_ACT_TANH: BODY(FCONV_ACT_TANH); break;      \
    case FCONV_ACT_HARDSIGMOID: BODY(FCONV_ACT_HARDSIGMOID); break; \
    case FCONV_ACT_HARDSWISH: BODY(FCONV_ACT_HARDSWISH); break; \
    case FCONV_ACT_CLIP: BODY(FCONV_ACT_CLIP); break;      \
    case FCONV_ACT_QUICKGELU: BODY(FCONV_ACT_QUICKGELU); break; \
    case FCONV_ACT_ELU: BODY(FCONV_ACT_ELU); break;        \
    case FCONV_ACT_GELU: BODY(FCONV_ACT_GELU); break;      \
    case FCONV_ACT_FASTGELU: BODY(FCONV_ACT_FASTGELU); break; \
    case FCONV_ACT_SOFTPLUS: BODY(FCONV_ACT_SOFTPLUS); break; \
    case FCONV_ACT_THRESHOLDEDRELU: BODY(FCONV_ACT_THRESHOLDEDRELU); break; \
    case FCONV_ACT_ERF: BODY(FCONV_ACT_ERF); break;        \
    default: BODY(FCONV_ACT_NONE); break;                  \
  }

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) {
  return __float2half_rn(v);
}

}  // namespace fconv
