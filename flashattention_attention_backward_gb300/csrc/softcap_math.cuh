// tanh for the softcap (logit = c tanh(u), u = tau s / c; "反向传播算法详解"
// §2.1(3)), on pairs of fp32 values through the f32x2 arithmetic.
//
// Two forms with the same accuracy (absolute error about 1e-7 in fp32):
//  * tanh_poly2: u + u^3 Q(u^2) with Q of degree 5, valid for |u| <= 1.
//    Seven f32x2 multiply-adds on the FMA pipe and no MUFU operation. Q is a
//    minimax fit of (tanh(u) - u) / u^3 for the absolute error of tanh
//    (Lawson's iteratively reweighted least squares; csrc/tanh_poly_fit.py
//    reproduces the coefficients and checks the fp32 evaluation: 8.3e-8).
//  * tanh_mufu2: 1 - 2 / (2^(2u log2e) + 1), any u: one exp2 and one
//    reciprocal per value on the MUFU pipe.
// The forward takes the polynomial for a group of scores when every |u| of
// the warp's group is at most 1 (a warp vote), and the MUFU form otherwise.
// The backward kernels keep the MUFU form: their softmax warps issue the
// P and dS phases of a tile back to back, and there the seven FMA-pipe
// instructions measured slower than the two MUFU operations they replace
// (softcap d = 64 workload: 0.135 ms against 0.131 ms; the forward: 0.106
// ms against 0.117 ms).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {
namespace softcap {

constexpr float kPolyMax = 1.0f;  // |u| range of tanh_poly2
constexpr float kC0 = -3.333273530e-01f;
constexpr float kC1 = 1.332349032e-01f;
constexpr float kC2 = -5.338026956e-02f;
constexpr float kC3 = 2.014188841e-02f;
constexpr float kC4 = -6.073148455e-03f;
constexpr float kC5 = 9.981628973e-04f;

__device__ __forceinline__ uint64_t tanh_poly2(uint64_t u2) {
  using namespace ptx;
  const uint64_t x2 = f2_mul(u2, u2);
  uint64_t q = f2_fma(x2, f2_make(kC5, kC5), f2_make(kC4, kC4));
  q = f2_fma(q, x2, f2_make(kC3, kC3));
  q = f2_fma(q, x2, f2_make(kC2, kC2));
  q = f2_fma(q, x2, f2_make(kC1, kC1));
  q = f2_fma(q, x2, f2_make(kC0, kC0));
  return f2_fma(f2_mul(u2, x2), q, u2);
}

// e2u2 = 2u log2e for the pair
__device__ __forceinline__ uint64_t tanh_mufu2(uint64_t e2u2) {
  using namespace ptx;
  const uint64_t e1 = f2_add(f2_make(ex2_approx(f2_lo(e2u2)), ex2_approx(f2_hi(e2u2))),
                             f2_make(1.f, 1.f));
  return f2_fma(f2_make(rcp_approx(f2_lo(e1)), rcp_approx(f2_hi(e1))), f2_make(-2.f, -2.f),
                f2_make(1.f, 1.f));
}

// Largest |x| of n raw fp32 words (to choose the form for a group).
template <int N>
__device__ __forceinline__ float max_abs(const uint32_t (&raw)[N]) {
  float m0 = 0.f, m1 = 0.f;
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    m0 = fmaxf(m0, fabsf(__uint_as_float(raw[j])));
    m1 = fmaxf(m1, fabsf(__uint_as_float(raw[j + 1])));
  }
  return fmaxf(m0, m1);
}

}  // namespace softcap
}  // namespace attn
