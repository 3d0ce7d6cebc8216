// situ_glu_fp8.cu — SiTU-GLU with x saved block-wise in FP8 (E4M3) for the backward.
//
// "Kimi K3 模型结构（9）：显存", section "统一激活管理器：重算、量化、offload 都是存储策略": most
// activations saved for the backward are stored with block-wise FP8 quantisation, while
// elementwise operators are recomputed. For SiTU-GLU the saved tensor is x, so:
//   situ_glu_fwd_save_fp8    reads bf16 x once and writes out (as situ_glu_fwd) together with
//                            the E4M3 codes of x and one fp32 scale per 128-element block;
//   situ_glu_bwd_router_fp8  the fused backward + router gradient evaluated at the dequantised
//                            x^ = decode(code) * scale.
// Block scheme (the pages do not fix it): 128 consecutive elements of one half of a row;
// a = max(amax, 448 * 2^-126), scale = a / 448, code = E4M3_RNE_satfinite(x * (448 / a)), each
// step one IEEE fp32 operation, so the codes are fully determined.
// Bytes per row: forward 4H read + 2H (out) + 2H (codes) + 8 * ceil(H/128) (scales) written;
// backward 2H (codes) + 8 * ceil(H/128) (scales) + 2H (g) + 4 (p) read, 4H (dx) + 4 (dp) written
// — 8H + 8nb + 8 against 10H + 8 for the bf16-saved backward, and half the saved bytes.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/situ_glu.h"
#include "situ_device.cuh"
#include "situ_host.h"
#include "situ_math.cuh"

namespace {

using namespace situ;
using namespace situ_host;

constexpr int kBlock = SITU_GLU_FP8_BLOCK;          // elements per scale block
constexpr float kE4M3Max = 448.0f;
constexpr float kAmaxFloor = 448.0f * 0x1p-126f;    // keeps the scale a normal fp32, 448/amax finite

// 8 codes of one 8-element chunk as two 32-bit words.
struct Codes8 {
    uint32_t w[2];
};

__device__ __forceinline__ Codes8 ld_codes(const Codes8* p) {
    Codes8 v;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.w[0]), "=r"(v.w[1]) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_codes(Codes8* p, const Codes8& v) {
    asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]) : "memory");
}

// 8 bf16 (one 16-byte chunk) -> 8 E4M3 codes with the block's inverse scale.
__device__ __forceinline__ Codes8 quantize_chunk(const Vec<4>& xv, float inv) {
    uint16_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = e4m3x2_from_f32(__fmul_rn(bf16_lo(xv.w[i]), inv), __fmul_rn(bf16_hi(xv.w[i]), inv));
    Codes8 q;
    q.w[0] = (uint32_t)c[0] | ((uint32_t)c[1] << 16);
    q.w[1] = (uint32_t)c[2] | ((uint32_t)c[3] << 16);
    return q;
}

__device__ __forceinline__ float chunk_amax(const Vec<4>& xv) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(xv.w[i])), fabsf(bf16_hi(xv.w[i]))));
    return m;
}

// ---------------------------------------------------------------------------
// forward that also saves x in FP8
// ---------------------------------------------------------------------------

// Vector path: H % 8 == 0; x, out 16-byte and xq 8-byte aligned. One warp per row; a step of
// the warp covers 32 consecutive 8-element chunks, i.e. two 128-element blocks, so lanes 0-15
// and 16-31 each hold one block and reduce its amax with four half-warp shuffles. PAIRED (β == 4):
// the forward of the two elements of each word with the paired fp32 math (situ::fwd_b4_2), the
// same results in fewer instructions: measured at R = 1.6M, H = 3072, 6.57 -> 6.23 ms (1024
// threads, 2 chunks per lane; 640 x 4 6.47, 768 x 2 6.83, 640 x 3 6.92, 512 x 4 7.06 ms).
template <bool BETA4, int U, int TPB, bool PAIRED = false>
__global__ void __launch_bounds__(TPB, 1) fwd_fp8_vec_kernel(const Vec<4>* __restrict__ x, Vec<4>* __restrict__ out,
                                                             Codes8* __restrict__ xq, float* __restrict__ xs,
                                                             int64_t R, int cpr, int nb, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * TPB + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * TPB) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const Vec<4>* xg = x + r * (2 * (int64_t)cpr);
        const Vec<4>* xl = xg + cpr;
        Vec<4>* o = out + r * (int64_t)cpr;
        Codes8* qg = xq + r * (2 * (int64_t)cpr);
        Codes8* ql = qg + cpr;
        float* sg = xs + r * (2 * (int64_t)nb);
        float* sl = sg + nb;
        for (int c0 = 0; c0 < cpr; c0 += 32 * U) {
            Vec<4> gv[U], lv[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    gv[k] = ld_stream<4, true, true>(xg + ci);
                    lv[k] = ld_stream<4, true, true>(xl + ci);
                } else {
                    gv[k] = Vec<4>{{0u, 0u, 0u, 0u}};
                    lv[k] = Vec<4>{{0u, 0u, 0u, 0u}};
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                const bool valid = ci < cpr;
                // block amax over 16 lanes (absent chunks contribute 0), floored
                const float ag = fmaxf(halfwarp_max(chunk_amax(gv[k])), kAmaxFloor);
                const float al = fmaxf(halfwarp_max(chunk_amax(lv[k])), kAmaxFloor);
                if (valid) {
                    Vec<4> ov;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if constexpr (BETA4 && PAIRED) {
                            const float2 a = situ::fwd_b4_2(bf16_lo(gv[k].w[i]), bf16_hi(gv[k].w[i]),
                                                            bf16_lo(lv[k].w[i]), bf16_hi(lv[k].w[i]), c);
                            ov.w[i] = pack_bf16x2(a.x, a.y);
                        } else {
                            float a0 = situ::fwd<BETA4>(bf16_lo(gv[k].w[i]), bf16_lo(lv[k].w[i]), c);
                            float a1 = situ::fwd<BETA4>(bf16_hi(gv[k].w[i]), bf16_hi(lv[k].w[i]), c);
                            ov.w[i] = pack_bf16x2(a0, a1);
                        }
                    }
                    st_stream<4>(o + ci, ov);
                    st_codes(qg + ci, quantize_chunk(gv[k], __fdiv_rn(kE4M3Max, ag)));
                    st_codes(ql + ci, quantize_chunk(lv[k], __fdiv_rn(kE4M3Max, al)));
                    if ((ci & 15) == 0) {
                        sg[ci >> 4] = __fdiv_rn(ag, kE4M3Max);
                        sl[ci >> 4] = __fdiv_rn(al, kE4M3Max);
                    }
                }
            }
        }
    }
}

constexpr int kElemThreads = 256;

// Element path: any H. One warp per row; blocks of 128 are handled one at a time, four
// elements per lane, amax reduced over the warp.
template <bool BETA4>
__global__ void __launch_bounds__(kElemThreads) fwd_fp8_elem_kernel(const uint16_t* __restrict__ x,
                                                                    uint16_t* __restrict__ out,
                                                                    uint8_t* __restrict__ xq,
                                                                    float* __restrict__ xs, int64_t R, int64_t H,
                                                                    int64_t nb, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kElemThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kElemThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint16_t* xr = x + r * 2 * H;
        uint16_t* orow = out + r * H;
        uint8_t* qr = xq + r * 2 * H;
        float* sr = xs + r * 2 * nb;
        for (int64_t b = 0; b < nb; ++b) {
            float u[kBlock / 32], v[kBlock / 32];
            float au = 0.0f, av = 0.0f;
#pragma unroll
            for (int i = 0; i < kBlock / 32; ++i) {
                const int64_t j = b * kBlock + i * 32 + lane;
                u[i] = 0.0f;
                v[i] = 0.0f;
                if (j < H) {
                    u[i] = bf16_to_f32(xr[j]);
                    v[i] = bf16_to_f32(xr[H + j]);
                    orow[j] = f32_to_bf16(situ::fwd<BETA4>(u[i], v[i], c));
                }
                au = fmaxf(au, fabsf(u[i]));
                av = fmaxf(av, fabsf(v[i]));
            }
            au = fmaxf(warp_max(au), kAmaxFloor);
            av = fmaxf(warp_max(av), kAmaxFloor);
            const float iu = __fdiv_rn(kE4M3Max, au), iv = __fdiv_rn(kE4M3Max, av);
#pragma unroll
            for (int i = 0; i < kBlock / 32; ++i) {
                const int64_t j = b * kBlock + i * 32 + lane;
                if (j < H) {
                    qr[j] = (uint8_t)(e4m3x2_from_f32(__fmul_rn(u[i], iu), 0.0f) & 0xFFu);
                    qr[H + j] = (uint8_t)(e4m3x2_from_f32(__fmul_rn(v[i], iv), 0.0f) & 0xFFu);
                }
            }
            if (lane == 0) {
                sr[b] = __fdiv_rn(au, kE4M3Max);
                sr[nb + b] = __fdiv_rn(av, kE4M3Max);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// backward + router gradient from the FP8-saved x
// ---------------------------------------------------------------------------

// Vector path: H % 8 == 0; xq 8-byte, g and dx 16-byte aligned.
template <bool BETA4, int U, int TPB>
__global__ void __launch_bounds__(TPB, 1) bwd_fp8_vec_kernel(const Codes8* __restrict__ xq,
                                                             const float* __restrict__ xs,
                                                             const Vec<4>* __restrict__ g,
                                                             const float* __restrict__ p, Vec<4>* __restrict__ dx,
                                                             float* __restrict__ dp, int64_t R, int cpr, int nb,
                                                             Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * TPB + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * TPB) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const Codes8* qg = xq + r * (2 * (int64_t)cpr);
        const Codes8* ql = qg + cpr;
        const float* sg = xs + r * (2 * (int64_t)nb);
        const float* sl = sg + nb;
        const Vec<4>* gr = g + r * (int64_t)cpr;
        Vec<4>* dgr = dx + r * (2 * (int64_t)cpr);
        Vec<4>* dlr = dgr + cpr;
        const float pr = 16.0f * p[r];   // 16·p: see situ::Bwd
        float acc = 0.0f;
        for (int c0 = 0; c0 < cpr; c0 += 32 * U) {
            Codes8 qgv[U], qlv[U];
            Vec<4> yv[U];
            float scg[U], scl[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    qgv[k] = ld_codes(qg + ci);
                    qlv[k] = ld_codes(ql + ci);
                    yv[k] = ld_stream<4, true, true>(gr + ci);
                    scg[k] = sg[ci >> 4];
                    scl[k] = sl[ci >> 4];
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    Vec<4> dgo, dlo;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint16_t cgi = (uint16_t)(qgv[k].w[i >> 1] >> (16 * (i & 1)));
                        const uint16_t cli = (uint16_t)(qlv[k].w[i >> 1] >> (16 * (i & 1)));
                        float u0, u1, v0, v1;
                        e4m3x2_to_f32(cgi, u0, u1);
                        e4m3x2_to_f32(cli, v0, v1);
                        u0 = __fmul_rn(u0, scg[k]);
                        u1 = __fmul_rn(u1, scg[k]);
                        v0 = __fmul_rn(v0, scl[k]);
                        v1 = __fmul_rn(v1, scl[k]);
                        const float g0 = bf16_lo(yv[k].w[i]), g1 = bf16_hi(yv[k].w[i]);
                        situ::Bwd b0 = situ::bwd<BETA4>(u0, v0, pr * g0, c);
                        situ::Bwd b1 = situ::bwd<BETA4>(u1, v1, pr * g1, c);
                        acc = fmaf(g0, b0.a16, acc);
                        acc = fmaf(g1, b1.a16, acc);
                        dgo.w[i] = pack_bf16x2(b0.dgate, b1.dgate);
                        dlo.w[i] = pack_bf16x2(b0.dlin, b1.dlin);
                    }
                    st_stream<4>(dgr + ci, dgo);
                    st_stream<4>(dlr + ci, dlo);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) dp[r] = 16.0f * acc;
    }
}

// 16 codes (one 16-element chunk) as four 32-bit words.
struct Codes16 {
    uint32_t w[4];
};

__device__ __forceinline__ Codes16 ld_codes16(const Codes16* p) {
    Codes16 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
        : "l"(p));
    return v;
}

// One 16-element chunk of the wide path: codes of both halves, g, the chunk's two block scales.
// PAIRED (β == 4 only): the two elements of each word through the paired fp32 math (bwd_b4_t2).
template <bool BETA4, bool PAIRED>
__device__ __forceinline__ void fp8_chunk(const Codes16& qgv, const Codes16& qlv, const Vec<8>& yv, float scg,
                                          float scl, float pr, const Coef& c, float2& acc2, Vec<8>& dgo,
                                          Vec<8>& dlo) {
    const float kg = scg * c.k_tu, kl = scl * c.k_tv;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint16_t cgi = (uint16_t)(qgv.w[i >> 1] >> (16 * (i & 1)));
        const uint16_t cli = (uint16_t)(qlv.w[i >> 1] >> (16 * (i & 1)));
        float u0, u1, v0, v1;
        e4m3x2_to_f32(cgi, u0, u1);
        e4m3x2_to_f32(cli, v0, v1);
        const float g0 = bf16_lo(yv.w[i]), g1 = bf16_hi(yv.w[i]);
        if constexpr (BETA4 && PAIRED) {
            const float2 gg = situ::pair(g0, g1);
            const situ::Bwd2 b = situ::bwd_b4_t2(situ::pair(fabsf(u0) * kg, fabsf(u1) * kg),
                                                 situ::pair(fabsf(v0) * kl, fabsf(v1) * kl), sign_of(u0), sign_of(u1),
                                                 sign_of(v0), sign_of(v1), __fmul2_rn(situ::pair(pr, pr), gg), c);
            acc2 = __ffma2_rn(gg, b.a16, acc2);
            dgo.w[i] = pack_bf16x2(b.dgate.x, b.dgate.y);
            dlo.w[i] = pack_bf16x2(b.dlin.x, b.dlin.y);
        } else {
            situ::Bwd b0, b1;
            if constexpr (BETA4) {
                b0 = situ::bwd_b4_t(fabsf(u0) * kg, fabsf(v0) * kl, sign_of(u0), sign_of(v0), pr * g0, c);
                b1 = situ::bwd_b4_t(fabsf(u1) * kg, fabsf(v1) * kl, sign_of(u1), sign_of(v1), pr * g1, c);
            } else {
                b0 = situ::bwd_gen(__fmul_rn(u0, scg), __fmul_rn(v0, scl), pr * g0, c);
                b1 = situ::bwd_gen(__fmul_rn(u1, scg), __fmul_rn(v1, scl), pr * g1, c);
            }
            acc2.x = fmaf(g0, b0.a16, acc2.x);
            acc2.y = fmaf(g1, b1.a16, acc2.y);
            dgo.w[i] = pack_bf16x2(b0.dgate, b1.dgate);
            dlo.w[i] = pack_bf16x2(b0.dlin, b1.dlin);
        }
    }
}

// Wide path: H % 16 == 0; xq 16-byte, g and dx 32-byte aligned. A lane takes 16 elements per
// chunk (16 bytes of codes per half, 32 bytes of g) and loads U chunks before any math; a warp
// chunk covers four scale blocks, one per group of 8 lanes. For beta = 4 the dequantisation
// scale folds into the exponent arguments: u enters the backward only through |u|·k_tu and its
// sign, so t = |value(code)|·(scale·k_tu) replaces value·scale followed by |·|·k_tu (one fp32
// rounding less than the oracle's two). The FP8 row moves fewer bytes per element than the bf16
// one, so the loads in flight per thread (U·64 bytes) set the bandwidth more than the arithmetic.
template <bool BETA4, int TPB, int U, bool PAIRED>
__global__ void __launch_bounds__(TPB, 1) bwd_fp8_wide_kernel(const Codes16* __restrict__ xq,
                                                              const float* __restrict__ xs,
                                                              const Vec<8>* __restrict__ g,
                                                              const float* __restrict__ p, Vec<8>* __restrict__ dx,
                                                              float* __restrict__ dp, int64_t R, int cpr, int nb,
                                                              Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * TPB + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * TPB) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const Codes16* qg = xq + r * (2 * (int64_t)cpr);
        const Codes16* ql = qg + cpr;
        const float* sg = xs + r * (2 * (int64_t)nb);
        const float* sl = sg + nb;
        const Vec<8>* gr = g + r * (int64_t)cpr;
        Vec<8>* dgr = dx + r * (2 * (int64_t)cpr);
        Vec<8>* dlr = dgr + cpr;
        const float pr = 16.0f * p[r];   // 16·p: see situ::Bwd
        float2 acc2 = situ::pair(0.0f, 0.0f);   // the even and the odd elements' sums
        for (int c0 = 0; c0 < cpr; c0 += 32 * U) {
            Codes16 qgv[U], qlv[U];
            Vec<8> yv[U];
            float scg[U], scl[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    qgv[k] = ld_codes16(qg + ci);
                    qlv[k] = ld_codes16(ql + ci);
                    yv[k] = ld_stream<8, true, true>(gr + ci);
                    scg[k] = sg[ci >> 3];
                    scl[k] = sl[ci >> 3];
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    Vec<8> dgo, dlo;
                    fp8_chunk<BETA4, PAIRED>(qgv[k], qlv[k], yv[k], scg[k], scl[k], pr, c, acc2, dgo, dlo);
                    st_stream<8>(dgr + ci, dgo);
                    st_stream<8>(dlr + ci, dlo);
                }
            }
        }
        const float acc = warp_sum(acc2.x + acc2.y);
        if (lane == 0) dp[r] = 16.0f * acc;
    }
}

// Element path: any H.
template <bool BETA4>
__global__ void __launch_bounds__(kElemThreads) bwd_fp8_elem_kernel(const uint8_t* __restrict__ xq,
                                                                    const float* __restrict__ xs,
                                                                    const uint16_t* __restrict__ g,
                                                                    const float* __restrict__ p,
                                                                    uint16_t* __restrict__ dx, float* __restrict__ dp,
                                                                    int64_t R, int64_t H, int64_t nb, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kElemThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kElemThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint8_t* qr = xq + r * 2 * H;
        const float* sr = xs + r * 2 * nb;
        const uint16_t* gr = g + r * H;
        uint16_t* dxr = dx + r * 2 * H;
        const float pr = 16.0f * p[r];   // 16·p: see situ::Bwd
        float acc = 0.0f;
        for (int64_t j = lane; j < H; j += 32) {
            float u, v, unused;
            e4m3x2_to_f32((uint16_t)qr[j], u, unused);
            e4m3x2_to_f32((uint16_t)qr[H + j], v, unused);
            u = __fmul_rn(u, sr[j / kBlock]);
            v = __fmul_rn(v, sr[nb + j / kBlock]);
            const float gj = bf16_to_f32(gr[j]);
            situ::Bwd b = situ::bwd<BETA4>(u, v, pr * gj, c);
            acc = fmaf(gj, b.a16, acc);
            dxr[j] = f32_to_bf16(b.dgate);
            dxr[H + j] = f32_to_bf16(b.dlin);
        }
        acc = warp_sum(acc);
        if (lane == 0) dp[r] = 16.0f * acc;
    }
}

constexpr int kFp8U = 2;
constexpr int kFp8Tpb = 1024;
// Launch shape of the wide backward: threads per CTA, chunks per lane, paired fp32 math. Measured at
// R = 1.6M, H = 3072 (median of 5 x 10 launches, same call): 1024 threads x 1 chunk 7.25 ms
// (scalar) / 7.27 (paired); 768 x 2 7.32 / 6.86; 512 x 2 8.20 / 7.16; 512 x 3 7.96 / 6.97;
// 1024 x 2 7.65 / 7.33; 384 x 4 paired 7.75; 640 x 2 paired 6.79 ms. The row moves fewer bytes per
// element than the bf16 one, so more loads in flight per thread pay, and the paired math frees the
// issue slots they need.
constexpr int kWideTpb = 640, kWideU = 2;
constexpr bool kWidePaired = true;

}  // namespace

extern "C" {

int situ_glu_fwd_save_fp8(const void* x, void* out, uint8_t* xq, float* xs, int64_t R, int64_t H, float beta,
                          float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    if (R == 0) return SITU_GLU_OK;
    if (x == nullptr || out == nullptr || xq == nullptr || xs == nullptr) return SITU_GLU_INVALID_ARG;
    if (!aligned(x, 2) || !aligned(out, 2) || !aligned(xs, 4)) return SITU_GLU_INVALID_ARG;
    const int64_t nb = (H + kBlock - 1) / kBlock;
    const Range rx = range_of(x, R * 2 * H * 2), ro = range_of(out, R * H * 2);
    const Range rq = range_of(xq, R * 2 * H), rs = range_of(xs, R * 2 * nb * 4);
    if (overlap(ro, rx) || overlap(rq, rx) || overlap(rs, rx)) return SITU_GLU_OVERLAP;
    if (overlap(ro, rq) || overlap(ro, rs) || overlap(rq, rs)) return SITU_GLU_OVERLAP;

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    if (H % 8 == 0 && aligned(x, 16) && aligned(out, 16) && aligned(xq, 8)) {
        const int cpr = (int)(H / 8);
        const Vec<4>* xv = (const Vec<4>*)x;
        Vec<4>* ov = (Vec<4>*)out;
        Codes8* qv = (Codes8*)xq;
        if (b4)
            return launch(fwd_fp8_vec_kernel<true, kFp8U, kFp8Tpb, true>, kFp8Tpb, R, stream, xv, ov, qv, xs, R, cpr,
                          (int)nb, c);
        return launch(fwd_fp8_vec_kernel<false, kFp8U, kFp8Tpb>, kFp8Tpb, R, stream, xv, ov, qv, xs, R, cpr, (int)nb, c);
    }
    const uint16_t* xs16 = (const uint16_t*)x;
    uint16_t* os16 = (uint16_t*)out;
    if (b4) return launch(fwd_fp8_elem_kernel<true>, kElemThreads, R, stream, xs16, os16, xq, xs, R, H, nb, c);
    return launch(fwd_fp8_elem_kernel<false>, kElemThreads, R, stream, xs16, os16, xq, xs, R, H, nb, c);
}

int situ_glu_bwd_router_fp8(const uint8_t* xq, const float* xs, const void* g, const float* p, void* dx, float* dp,
                            int64_t R, int64_t H, float beta, float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    if (R == 0) return SITU_GLU_OK;
    if (xq == nullptr || xs == nullptr || g == nullptr || p == nullptr || dx == nullptr || dp == nullptr)
        return SITU_GLU_INVALID_ARG;
    if (!aligned(xs, 4) || !aligned(g, 2) || !aligned(dx, 2) || !aligned(p, 4) || !aligned(dp, 4))
        return SITU_GLU_INVALID_ARG;
    const int64_t nb = (H + kBlock - 1) / kBlock;
    const Range rq = range_of(xq, R * 2 * H), rs = range_of(xs, R * 2 * nb * 4), rg = range_of(g, R * H * 2);
    const Range rp = range_of(p, R * 4), rdx = range_of(dx, R * 2 * H * 2), rdp = range_of(dp, R * 4);
    if (overlap(rdx, rq) || overlap(rdx, rs) || overlap(rdx, rg) || overlap(rdx, rp) || overlap(rdx, rdp))
        return SITU_GLU_OVERLAP;
    if (overlap(rdp, rq) || overlap(rdp, rs) || overlap(rdp, rg) || overlap(rdp, rp)) return SITU_GLU_OVERLAP;

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    if (H % 16 == 0 && aligned(xq, 16) && aligned(g, 32) && aligned(dx, 32)) {
        const int cpr = (int)(H / 16);
        const Codes16* qv = (const Codes16*)xq;
        const Vec<8>* gv = (const Vec<8>*)g;
        Vec<8>* dxv = (Vec<8>*)dx;
        if (b4)
            return launch(bwd_fp8_wide_kernel<true, kWideTpb, kWideU, kWidePaired>, kWideTpb, R, stream, qv, xs, gv, p,
                          dxv, dp, R, cpr, (int)nb, c);
        return launch(bwd_fp8_wide_kernel<false, kWideTpb, kWideU, false>, kWideTpb, R, stream, qv, xs, gv, p, dxv,
                      dp, R, cpr, (int)nb, c);
    }
    if (H % 8 == 0 && aligned(xq, 8) && aligned(g, 16) && aligned(dx, 16)) {
        const int cpr = (int)(H / 8);
        const Codes8* qv = (const Codes8*)xq;
        const Vec<4>* gv = (const Vec<4>*)g;
        Vec<4>* dxv = (Vec<4>*)dx;
        if (b4)
            return launch(bwd_fp8_vec_kernel<true, kFp8U, kFp8Tpb>, kFp8Tpb, R, stream, qv, xs, gv, p, dxv, dp, R, cpr,
                          (int)nb, c);
        return launch(bwd_fp8_vec_kernel<false, kFp8U, kFp8Tpb>, kFp8Tpb, R, stream, qv, xs, gv, p, dxv, dp, R, cpr,
                      (int)nb, c);
    }
    const uint16_t* g16 = (const uint16_t*)g;
    uint16_t* dx16 = (uint16_t*)dx;
    if (b4) return launch(bwd_fp8_elem_kernel<true>, kElemThreads, R, stream, xq, xs, g16, p, dx16, dp, R, H, nb, c);
    return launch(bwd_fp8_elem_kernel<false>, kElemThreads, R, stream, xq, xs, g16, p, dx16, dp, R, H, nb, c);
}

}  // extern "C"
