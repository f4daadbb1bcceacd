// GELU and its derivative for the backward pass ("RankMixer 详解（1）" section
// 4.1: Gelu(u) = u Phi(u); section 5.2: Gelu'(u) = Phi(u) + u phi(u)).
//
// Phi comes from the upper tail Q(x) = erfc(x / sqrt 2) / 2 for x = |u|,
// with erfc by Abramowitz & Stegun 7.1.26 (|error of erf| <= 1.5e-7):
//   erfc(y) ~= t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-y^2),  t = 1 / (1 + p y),
// p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741, -1.453152027, 1.061405429.
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

// Gelu and Gelu' of two values at once in the packed fp32x2 arithmetic
// (one instruction per pair for add, multiply and fused multiply-add), for
// u = acc * s + b.  With Q = Q(|u|) and h = 1/2 - Q, both branch-free:
//   Phi(u) = 1/2 + sgn(u) h          (1 - Q for u >= 0, Q for u < 0)
//   Gelu(u) = u Phi(u) = u / 2 + |u| h
//   Gelu'(u) = Phi(u) + u exp(-u^2 / 2) / sqrt(2 pi).
// The coefficients below are -a_i / 2 and the tail runs as in the scalar
// form: t = 1 / (1 + p |u| / sqrt 2) and exp(-u^2 / 2) = 2^(-(k1 |u|)^2),
// k1 = sqrt(log2(e) / 2), so q t (...) exp(...) = -Q.
__device__ __forceinline__ void gelu_with_grad_x2(uint64_t acc, uint64_t s, uint64_t b, uint64_t& value,
                                                  uint64_t& grad) {
    constexpr float k1 = 0.8493218002880191f;     // sqrt(log2(e) / 2)
    constexpr float pp = 0.27273748087922245f;    // p / (sqrt(2) k1)
    constexpr float nh1 = -0.127414796f, nh2 = 0.142248368f, nh3 = -0.7107068705f, nh4 = 0.7265760135f,
                    nh5 = -0.5307027145f;
    constexpr float inv_sqrt_2pi = 0.39894228040143268f;
    const uint64_t u = f2_fma(acc, s, b);
    const uint64_t a = u & 0x7fffffff7fffffffull;                   // |u|
    const uint64_t xp = f2_mul(a, f2_splat(k1));
    const uint64_t den = f2_fma(f2_splat(pp), xp, f2_splat(1.0f));
    float d0, d1;
    f2_unpack(den, d0, d1);
    const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
    uint64_t q = f2_fma(t, f2_splat(nh5), f2_splat(nh4));
    q = f2_fma(t, q, f2_splat(nh3));
    q = f2_fma(t, q, f2_splat(nh2));
    q = f2_fma(t, q, f2_splat(nh1));
    q = f2_mul(q, t);
    const uint64_t sq = f2_mul(xp, xp);
    float s0, s1;
    f2_unpack(sq, s0, s1);
    const uint64_t e = f2_pack(ex2_approx(-s0), ex2_approx(-s1));   // exp(-u^2 / 2)
    const uint64_t h = f2_fma(q, e, f2_splat(0.5f));                // 1/2 - Q
    value = f2_fma(a, h, f2_mul(u, f2_splat(0.5f)));
    const uint64_t sh = h ^ (u & 0x8000000080000000ull);            // sgn(u) h
    grad = f2_fma(f2_mul(u, f2_splat(inv_sqrt_2pi)), e, f2_add(sh, f2_splat(0.5f)));
}

// Scalar form: the packed arithmetic on (u, u), so that every path computes
// the same values.
__device__ __forceinline__ GeluPair gelu_with_grad(float u) {
    uint64_t v, g;
    gelu_with_grad_x2(f2_splat(u), f2_splat(1.0f), f2_splat(0.0f), v, g);
    float v1, g1;
    GeluPair r;
    f2_unpack(v, r.value, v1);
    f2_unpack(g, r.grad, g1);
    return r;
}

}  // namespace rm
