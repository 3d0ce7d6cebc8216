// situ_math.cuh — fp32 register math of the SiTU-GLU activation and its backward.
//
// Definition ("Frontier-scale RL with Kimi K3", section "Streaming activations"),
// for u = gate, v = linear, β = beta, λ = lbeta:
//   T = tanh(u/β), S = σ(u), G = β·T·S,   W = tanh(v/λ), L = λ·W,   a = G·L
//   G' = (1 − T²)·S + β·T·S·(1 − S),      L' = 1 − W²
//
// Everything is rewritten in terms of three exponentials of non-positive
// arguments, so nothing overflows for any finite input and no derivative is
// formed by cancellation (no 1 − tanh² of a rounded tanh):
//   E1 = e^{−2|u|/β}, E2 = e^{−|u|}, e = e^{−2|v|/λ}            (all in [0, 1])
//   tanh(u/β) = sgn(u)·(1 − E1)/(1 + E1)       1 − T² = 4·E1/(1 + E1)²
//   σ(u) = s/(1 + E2), s = 1 (u ≥ 0) or E2 (u < 0)   σ(1 − σ) = E2/(1 + E2)²
//   tanh(v/λ) = sgn(v)·(1 − e)/(1 + e)         1 − W² = 4·e/(1 + e)²
// With q = 1/((1 + E1)(1 + E2)) and w = 1/(1 + e), both from ONE reciprocal of
// D = (1 + E1)(1 + E2)(1 + e):
//   G  = β·sgn(u)·(1 − E1)·s·q
//   G' = q²·[4·E1·s·(1 + E2) + β·sgn(u)·(1 − E1)(1 + E1)·E2]
//   L  = λ·sgn(v)·(1 − e)·w,   L' = 4·e·w²
// For β = 4, E1 = e^{−|u|/2} and E2 = E1², so one exponential serves the gate:
// 2 ex2 + 1 rcp on the MUFU per element pair, forward and backward alike.
//
// Accuracy: ex2.approx and rcp.approx are within a few fp32 ulp (PTX ISA), so
// every quantity above has a relative error of a few 2^-23, except (1 − E1)
// and (1 − e) for tiny arguments, whose error is absolute (~2^-22). On the
// β = 4 fast path that leaves an absolute error below λ·2^-21 in L and below
// 2^-20 in G: tiny against the bf16 half-ulp or the 1e-3 floor of the outputs.
// The general path replaces (1 − E1) and (1 − e) by a short odd Taylor series
// of tanh below |z| < 1/16 so it stays relatively accurate for any β and λ.
#pragma once

#include <stdint.h>

namespace situ {

// Per-launch constants, computed on the host in double and rounded once.
struct Coef {
    float k_tu;      // −(2/β)·log2(e):  ex2(|u|·k_tu) = e^{−2|u|/β}
    float k_su;      // −log2(e):        ex2(|u|·k_su) = e^{−|u|}
    float k_tv;      // −(2/λ)·log2(e):  ex2(|v|·k_tv) = e^{−2|v|/λ}
    float inv_beta;  // 1/β
    float inv_lbeta; // 1/λ
    float beta;      // β
    float lbeta;     // λ
    float beta_lbeta;// β·λ
};

// MUFU exp2: ex2.approx.ftz.f32 (results below the normal range flush to +0).
__device__ __forceinline__ float ex2(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// MUFU reciprocal: rcp.approx.ftz.f32. Only ever applied to D in [1, 8].
__device__ __forceinline__ float rcp(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// Sign bit of x.
__device__ __forceinline__ uint32_t sign_of(float x) { return __float_as_uint(x) & 0x80000000u; }

// |m| with the sign flipped by the sign bit s (m is non-negative up to rounding).
__device__ __forceinline__ float with_sign(float m, uint32_t s) { return __uint_as_float(__float_as_uint(m) ^ s); }

// tanh(z)·(1 + E) for 0 <= z < 1/16, E = e^{−2z}: the odd Taylor series of tanh,
// z − z³/3 + 2z⁵/15 (next term 17z⁷/315 is < 4e-9 relative here), times (1 + E)
// so that it stands in for the numerator (1 − E) of (1 − E)/(1 + E).
__device__ __forceinline__ float tanh_num_small(float z, float onepE) {
    float z2 = z * z;
    float t = z * fmaf(z2, fmaf(z2, 2.0f / 15.0f, -1.0f / 3.0f), 1.0f);
    return t * onepE;
}

constexpr float kSmallZ = 0.0625f;

// ---------------- forward: a = G·L ----------------

// β == 4 (E2 = E1²). 2 ex2 + 1 rcp.
__device__ __forceinline__ float fwd_b4(float u, float v, const Coef& c) {
    float E = ex2(fabsf(u) * c.k_tu);           // e^{−|u|/2}
    float e = ex2(fabsf(v) * c.k_tv);           // e^{−2|v|/λ}
    float E2 = E * E;                           // e^{−|u|}
    float r = rcp((1.0f + E) * (1.0f + E2) * (1.0f + e));
    float s = (u < 0.0f) ? E2 : 1.0f;
    float m = (1.0f - E) * (1.0f - e) * s * r * c.beta_lbeta;
    return with_sign(m, sign_of(u) ^ sign_of(v));
}

// Any β, λ. 3 ex2 + 1 rcp, small-argument series for both tanh numerators.
__device__ __forceinline__ float fwd_gen(float u, float v, const Coef& c) {
    float au = fabsf(u), av = fabsf(v);
    float E1 = ex2(au * c.k_tu);
    float E2 = ex2(au * c.k_su);
    float e = ex2(av * c.k_tv);
    float pE1 = 1.0f + E1, pe = 1.0f + e;
    float zu = au * c.inv_beta, zv = av * c.inv_lbeta;
    float tn = (zu < kSmallZ) ? tanh_num_small(zu, pE1) : (1.0f - E1);
    float wn = (zv < kSmallZ) ? tanh_num_small(zv, pe) : (1.0f - e);
    float r = rcp(pE1 * (1.0f + E2) * pe);
    float s = (u < 0.0f) ? E2 : 1.0f;
    float m = tn * wn * s * r * c.beta_lbeta;
    return with_sign(m, sign_of(u) ^ sign_of(v));
}

// ---------------- backward: a, dgate, dlinear ----------------
// pg = p·g (dL/da of this element); a is returned unrounded for the dp sum.

struct Bwd {
    float a;
    float dgate;
    float dlin;
};

// β == 4. 2 ex2 + 1 rcp.
__device__ __forceinline__ Bwd bwd_b4(float u, float v, float pg, const Coef& c) {
    float E = ex2(fabsf(u) * c.k_tu);           // e^{−|u|/2}
    float e = ex2(fabsf(v) * c.k_tv);           // e^{−2|v|/λ}
    float E2 = E * E;                           // e^{−|u|}
    float pE = 1.0f + E, pE2 = 1.0f + E2, pe = 1.0f + e;
    float P = pE * pE2;
    float r = rcp(P * pe);
    float q = r * pe;                           // 1/((1+E)(1+E2))
    float w = r * P;                            // 1/(1+e)
    bool neg = u < 0.0f;
    float s = neg ? E2 : 1.0f;
    float omE = 1.0f - E;
    uint32_t su = sign_of(u), sv = sign_of(v);
    float G = with_sign(4.0f * omE * s * q, su);
    float t2 = omE * pE * E2;                   // (1 − E2)·E2
    float br = fmaf(E * s, pE2, neg ? -t2 : t2);
    float Gp = 4.0f * q * q * br;
    float L = with_sign(c.lbeta * (1.0f - e) * w, sv);
    float Lp = 4.0f * e * w * w;
    Bwd o;
    o.a = G * L;
    o.dgate = pg * L * Gp;
    o.dlin = pg * G * Lp;
    return o;
}

// Any β, λ. 3 ex2 + 1 rcp, small-argument series for both tanh numerators.
__device__ __forceinline__ Bwd bwd_gen(float u, float v, float pg, const Coef& c) {
    float au = fabsf(u), av = fabsf(v);
    float E1 = ex2(au * c.k_tu);
    float E2 = ex2(au * c.k_su);
    float e = ex2(av * c.k_tv);
    float pE1 = 1.0f + E1, pE2 = 1.0f + E2, pe = 1.0f + e;
    float zu = au * c.inv_beta, zv = av * c.inv_lbeta;
    float tn = (zu < kSmallZ) ? tanh_num_small(zu, pE1) : (1.0f - E1);
    float wn = (zv < kSmallZ) ? tanh_num_small(zv, pe) : (1.0f - e);
    float P = pE1 * pE2;
    float r = rcp(P * pe);
    float q = r * pe;
    float w = r * P;
    bool neg = u < 0.0f;
    float s = neg ? E2 : 1.0f;
    uint32_t su = sign_of(u), sv = sign_of(v);
    float G = with_sign(c.beta * tn * s * q, su);
    float t2 = c.beta * tn * pE1 * E2;          // β·(1 − E1²)·E2
    float br = fmaf(4.0f * E1 * s, pE2, neg ? -t2 : t2);
    float Gp = q * q * br;
    float L = with_sign(c.lbeta * wn * w, sv);
    float Lp = 4.0f * e * w * w;
    Bwd o;
    o.a = G * L;
    o.dgate = pg * L * Gp;
    o.dlin = pg * G * Lp;
    return o;
}

template <bool BETA4>
__device__ __forceinline__ float fwd(float u, float v, const Coef& c) {
    return BETA4 ? fwd_b4(u, v, c) : fwd_gen(u, v, c);
}

template <bool BETA4>
__device__ __forceinline__ Bwd bwd(float u, float v, float pg, const Coef& c) {
    return BETA4 ? bwd_b4(u, v, pg, c) : bwd_gen(u, v, pg, c);
}

}  // namespace situ
