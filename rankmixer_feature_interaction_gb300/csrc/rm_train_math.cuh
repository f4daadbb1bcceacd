// GELU and its derivative for the backward pass ("RankMixer 详解（1）" section
// 4.1: Gelu(u) = u Phi(u); section 5.2: Gelu'(u) = Phi(u) + u phi(u)).
//
// Phi comes from the upper tail Q(x) = erfc(x / sqrt 2) / 2 for x = |u|,
// with erfc by Abramowitz & Stegun 7.1.26 (|error of erf| <= 1.5e-7):
//   erfc(y) ~= t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-y^2),  t = 1 / (1 + p y).
// exp(-y^2) with y = |u| / sqrt 2 is exp(-u^2 / 2), which phi(u) shares; it and
// the reciprocal run on the special-function unit (ex2.approx, rcp.approx,
// relative error about 2^-22), far inside the approximation's own 1.5e-7.
#pragma once

#include <cuda_runtime.h>

#include "rm_common.cuh"

namespace rm {

struct GeluPair {
    float value;   // Gelu(u)
    float grad;    // Gelu'(u)
};

__device__ __forceinline__ GeluPair gelu_with_grad(float u) {
    constexpr float p = 0.3275911f;
    constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f, a4 = -1.453152027f,
                    a5 = 1.061405429f;
    constexpr float inv_sqrt2 = 0.70710678118654752f;
    constexpr float inv_sqrt_2pi = 0.39894228040143268f;
    constexpr float half_log2e = 0.72134752044448170f;     // log2(e) / 2
    const float y = fabsf(u) * inv_sqrt2;
    const float e = ex2_approx(-half_log2e * u * u);       // exp(-u^2 / 2) on the MUFU unit
    const float t = rcp_approx(fmaf(p, y, 1.0f));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, a5, a4), a3), a2), a1);
    const float q = 0.5f * poly * e;                       // Q(|u|) = P(N(0,1) > |u|)
    const float Phi = u >= 0.0f ? 1.0f - q : q;
    GeluPair r;
    r.value = u * Phi;
    r.grad = fmaf(u * inv_sqrt_2pi, e, Phi);
    return r;
}

}  // namespace rm
