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
// With q = 1/((1 + E1)(1 + E2)) and w = 1/(1 + e):
//   G  = β·sgn(u)·(1 − E1)·s·q
//   G' = q²·[4·E1·s·(1 + E2) + β·sgn(u)·(1 − E1)(1 + E1)·E2]
//   L  = λ·sgn(v)·(1 − e)·w,   L' = 4·e·w²
// For β = 4, E1 = e^{−|u|/2} and E2 = E1², so one exponential serves the gate. The forward
// needs only a = G·L, whose denominators share ONE reciprocal of (1 + E1)(1 + E2)(1 + e):
// 2 ex2 + 1 rcp on the MUFU per element pair; the backward takes q and w from two reciprocals.
//
// Accuracy: ex2.approx and rcp.approx are within a few fp32 ulp (PTX ISA), so every quantity
// above has a relative error of a few 2^-23, except the numerators 1 - E1 and 1 - e for small
// arguments: E = ex2(t) carries an absolute error ~2^-22.5 near t = 0, so 1 - E computed as a
// difference has a relative error ~2^-22.5 / |t|. The backward (whose dp has a purely relative
// tolerance) therefore takes 1 - 2^t as the larger of two lower bounds of it, the series
// x - x²/2 (x = -t·ln2) and the difference lowered by more than its own error (one_minus_exp2:
// relative error below 5e-5 at every t), and the general path uses an odd Taylor series of tanh
// below |z| < 1/16. The beta = 4 forward keeps the plain difference: its absolute error (below
// 2^-20 in G and lbeta·2^-21 in L) is far inside the 1e-3 absolute floor of a bf16 output.
//
// The backward returns a/16, p·g·L·G' and p·g·G·L' from pg16 = 16·p·g: the factors 4 of G, G'
// and L' (and 1/4 of L) are folded into the caller's per-row 16·p and the final 16·dp, exact
// power-of-two scalings that save three multiplies per element pair.
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
    float beta_4;    // β/4
    float lbeta_4;   // λ/4
};

// MUFU exp2: ex2.approx.ftz.f32 (results below the normal range flush to +0).
__device__ __forceinline__ float ex2(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// MUFU reciprocal: rcp.approx.ftz.f32. Only ever applied to arguments in [1, 8].
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

// 1 - 2^t for t <= 0 given e = ex2(t), relatively accurate at every t. With x = -t·ln2 >= 0 the
// exact value 1 - e^-x lies above both
//   the series x - x²/2 (the alternating series of e^-x cut after a negative term: it undershoots
//   by less than x³/6), and
//   (1 - 2^-21) - e (the difference lowered by 2^-21, more than the absolute error of ex2 there;
//   the subtraction is exact while e >= 1/2),
// so the larger of the two undershoots by at most min(x³/6, 2^-21 + err(e)): a relative error below
// 5e-5 at every x, largest where the two bounds cross (x ~ 0.016). Four instructions; NaN and
// t = -inf pass through (the series is then NaN or -inf and the difference wins or propagates).
__device__ __forceinline__ float one_minus_exp2(float t, float e) {
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kLn2Sq2 = 0.2402265069591007f;  // ln(2)^2 / 2
    constexpr float kOneLow = 1.0f - 0x1p-21f;      // exact in fp32
    const float series = t * fmaf(t, -kLn2Sq2, -kLn2);
    return fmaxf(series, kOneLow - e);
}

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

// ---------------- backward: a/16, dgate, dlinear ----------------
// pg16 = 16·p·g (16 times dL/da of this element); a16 = a/16 is returned unrounded for the dp sum.

struct Bwd {
    float a16;    // a / 16
    float dgate;  // p·g·L·G'
    float dlin;   // p·g·G·L'
};

// β == 4 from the exponent arguments tg = |u|·k_tu, tl = |v|·k_tv and the sign bits of u and v
// (the only ways u and v enter). 2 ex2 + 2 rcp: q = 1/((1+E)(1+E2)) and w = 1/(1+e) each from
// its own reciprocal, which costs one MUFU operation more and three multiplies fewer than
// splitting one reciprocal of the whole product (the backward is issue-bound, not MUFU-bound).
__device__ __forceinline__ Bwd bwd_b4_t(float tg, float tl, uint32_t su, uint32_t sv, float pg16, const Coef& c) {
    const float E = ex2(tg);                    // e^{−|u|/2}
    const float e = ex2(tl);                    // e^{−2|v|/λ}
    const float E2 = E * E;                     // e^{−|u|}
    const float pE = 1.0f + E, pE2 = 1.0f + E2;
    const float q = rcp(pE * pE2);              // 1/((1+E)(1+E2))
    const float w = rcp(1.0f + e);              // 1/(1+e)
    const float s = su ? E2 : 1.0f;             // σ numerator (u = −0 gives E2 = 1 as well)
    const float omE = with_sign(one_minus_exp2(tg, E), su);              // sgn(u)·(1 − E)
    const float G4 = omE * s * q;                                        // G/4
    const float br = fmaf(E * s, pE2, omE * pE * E2);                    // G' = 4·q²·br
    const float L4 = with_sign(one_minus_exp2(tl, e), sv) * (c.lbeta_4 * w);  // L/4
    Bwd o;
    o.a16 = G4 * L4;
    o.dgate = (pg16 * L4) * (q * q * br);
    o.dlin = (pg16 * G4) * (e * (w * w));       // L' = 4·e·w²
    return o;
}

// ---------------- backward on two elements at once (paired fp32 instructions) ----------------
// The same arithmetic as bwd_b4_t for two independent elements, with every multiply, add and
// fused multiply-add issued as one paired fp32 instruction (fma/mul/add .rn.f32x2, sm_100 and
// later) and the MUFU operations, selects and sign flips per element: about two thirds of the
// FMA-pipe instructions of two scalar evaluations. Each paired operation rounds each lane exactly
// as the scalar operation would, so the two lanes return what bwd_b4_t returns.

struct Bwd2 {
    float2 a16, dgate, dlin;
};

__device__ __forceinline__ float2 pair(float a, float b) { return make_float2(a, b); }

// one_minus_exp2 on two lanes.
__device__ __forceinline__ float2 one_minus_exp2_x2(float2 t, float2 e) {
    constexpr float kLn2 = 0.6931471805599453f;
    constexpr float kLn2Sq2 = 0.2402265069591007f;
    constexpr float kOneLow = 1.0f - 0x1p-21f;
    const float2 series = __fmul2_rn(t, __ffma2_rn(t, pair(-kLn2Sq2, -kLn2Sq2), pair(-kLn2, -kLn2)));
    const float2 diff = __ffma2_rn(e, pair(-1.0f, -1.0f), pair(kOneLow, kOneLow));   // kOneLow - e, one rounding
    return pair(fmaxf(series.x, diff.x), fmaxf(series.y, diff.y));
}

// β == 4 for two elements: exponent arguments tg, tl, sign bits su, sv of each lane's u and v.
__device__ __forceinline__ Bwd2 bwd_b4_t2(float2 tg, float2 tl, uint32_t su0, uint32_t su1, uint32_t sv0,
                                          uint32_t sv1, float2 pg16, const Coef& c) {
    const float2 one = pair(1.0f, 1.0f);
    const float2 E = pair(ex2(tg.x), ex2(tg.y));
    const float2 e = pair(ex2(tl.x), ex2(tl.y));
    const float2 E2 = __fmul2_rn(E, E);
    const float2 pE = __fadd2_rn(one, E), pE2 = __fadd2_rn(one, E2);
    const float2 P = __fmul2_rn(pE, pE2);
    const float2 pe = __fadd2_rn(one, e);
    const float2 q = pair(rcp(P.x), rcp(P.y));
    const float2 w = pair(rcp(pe.x), rcp(pe.y));
    const float2 s = pair(su0 ? E2.x : 1.0f, su1 ? E2.y : 1.0f);
    float2 omE = one_minus_exp2_x2(tg, E);
    omE = pair(with_sign(omE.x, su0), with_sign(omE.y, su1));
    const float2 G4 = __fmul2_rn(__fmul2_rn(omE, s), q);
    const float2 br = __ffma2_rn(__fmul2_rn(E, s), pE2, __fmul2_rn(__fmul2_rn(omE, pE), E2));
    float2 ome = one_minus_exp2_x2(tl, e);
    ome = pair(with_sign(ome.x, sv0), with_sign(ome.y, sv1));
    const float2 L4 = __fmul2_rn(ome, __fmul2_rn(pair(c.lbeta_4, c.lbeta_4), w));
    Bwd2 o;
    o.a16 = __fmul2_rn(G4, L4);
    o.dgate = __fmul2_rn(__fmul2_rn(pg16, L4), __fmul2_rn(__fmul2_rn(q, q), br));
    o.dlin = __fmul2_rn(__fmul2_rn(pg16, G4), __fmul2_rn(e, __fmul2_rn(w, w)));
    return o;
}

// fwd_b4 on two elements (u0, v0) and (u1, v1) with paired fp32 instructions; each lane returns
// exactly what fwd_b4 returns for it (the same operations in the same order, each rounded as the
// scalar one).
__device__ __forceinline__ float2 fwd_b4_2(float u0, float u1, float v0, float v1, const Coef& c) {
    const float2 one = pair(1.0f, 1.0f);
    const float2 E = pair(ex2(fabsf(u0) * c.k_tu), ex2(fabsf(u1) * c.k_tu));
    const float2 e = pair(ex2(fabsf(v0) * c.k_tv), ex2(fabsf(v1) * c.k_tv));
    const float2 E2 = __fmul2_rn(E, E);
    const float2 den = __fmul2_rn(__fmul2_rn(__fadd2_rn(one, E), __fadd2_rn(one, E2)), __fadd2_rn(one, e));
    const float2 r = pair(rcp(den.x), rcp(den.y));
    const float2 s = pair((u0 < 0.0f) ? E2.x : 1.0f, (u1 < 0.0f) ? E2.y : 1.0f);
    const float2 omE = __fadd2_rn(one, pair(-E.x, -E.y)), ome = __fadd2_rn(one, pair(-e.x, -e.y));
    const float2 m = __fmul2_rn(__fmul2_rn(__fmul2_rn(__fmul2_rn(omE, ome), s), r), pair(c.beta_lbeta, c.beta_lbeta));
    return pair(with_sign(m.x, sign_of(u0) ^ sign_of(v0)), with_sign(m.y, sign_of(u1) ^ sign_of(v1)));
}

// β == 4. 2 ex2 + 2 rcp.
__device__ __forceinline__ Bwd bwd_b4(float u, float v, float pg16, const Coef& c) {
    return bwd_b4_t(fabsf(u) * c.k_tu, fabsf(v) * c.k_tv, sign_of(u), sign_of(v), pg16, c);
}

// Any β, λ. 3 ex2 + 1 rcp, small-argument series for both tanh numerators.
__device__ __forceinline__ Bwd bwd_gen(float u, float v, float pg16, const Coef& c) {
    const float au = fabsf(u), av = fabsf(v);
    const float E1 = ex2(au * c.k_tu);
    const float E2 = ex2(au * c.k_su);
    const float e = ex2(av * c.k_tv);
    const float pE1 = 1.0f + E1, pE2 = 1.0f + E2, pe = 1.0f + e;
    const float zu = au * c.inv_beta, zv = av * c.inv_lbeta;
    const float tn = (zu < kSmallZ) ? tanh_num_small(zu, pE1) : (1.0f - E1);
    const float wn = (zv < kSmallZ) ? tanh_num_small(zv, pe) : (1.0f - e);
    const float P = pE1 * pE2;
    const float r = rcp(P * pe);
    const float q = r * pe;
    const float w = r * P;
    const float s = (u < 0.0f) ? E2 : 1.0f;
    const uint32_t su = sign_of(u), sv = sign_of(v);
    const float G4 = with_sign(c.beta_4 * tn * s * q, su);                          // G/4
    const float br = fmaf(E1 * s, pE2, with_sign(c.beta_4 * tn * pE1 * E2, su));    // G' = 4·q²·br
    const float L4 = with_sign(c.lbeta_4 * wn * w, sv);                             // L/4
    Bwd o;
    o.a16 = G4 * L4;
    o.dgate = (pg16 * L4) * (q * q * br);
    o.dlin = (pg16 * G4) * (e * (w * w));
    return o;
}

template <bool BETA4>
__device__ __forceinline__ float fwd(float u, float v, const Coef& c) {
    return BETA4 ? fwd_b4(u, v, c) : fwd_gen(u, v, c);
}

template <bool BETA4>
__device__ __forceinline__ Bwd bwd(float u, float v, float pg16, const Coef& c) {
    return BETA4 ? bwd_b4(u, v, pg16, c) : bwd_gen(u, v, pg16, c);
}

}  // namespace situ
