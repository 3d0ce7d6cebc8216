// situ_glu.cu — SiTU-GLU forward and fused backward + router gradient for GB300 (sm_103a),
// and the C ABI declared in include/situ_glu.h.
//
// The path is elementwise plus a per-row reduction, so it is bound by HBM bandwidth:
//   forward   reads x (4H B/row), writes out (2H B/row)              -> 6H B/row
//   backward  reads x (4H), g (2H), p (4 B); writes dx (4H), dp (4 B) -> 10H + 8 B/row
// There is no contraction, so no tensor cores. Design:
//   * one warp per row, rows distributed grid-stride over a persistent grid sized
//     from the SM count and the kernel's occupancy;
//   * each lane moves 16-byte vectors (8 bf16); a warp instruction covers 512
//     contiguous bytes; UNROLL chunks per lane are loaded before any math so
//     every warp has several KB in flight;
//   * all intermediates (the "constant fp32 workspace" of the pages' custom
//     operator) live in registers: nothing but x, g, p, out, dx, dp touches memory;
//   * dp is a fixed-order per-lane fp32 sum followed by a butterfly shuffle, so
//     results are bit-reproducible.
// Sources: "Frontier-scale RL with Kimi K3", section "Streaming activations";
// "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出".
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "../../include/situ_glu.h"
#include "situ_math.cuh"

namespace {

using situ::Coef;

// ---------------------------------------------------------------------------
// memory helpers (inline PTX)
// ---------------------------------------------------------------------------

// Streaming 16-byte load through the non-coherent path (inputs that no thread writes).
__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Streaming 16-byte load through the coherent path (x may alias dx in the backward).
__device__ __forceinline__ uint4 ld_co(const uint4* p) {
    uint4 v;
    asm("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Streaming (evict-first) 16-byte store.
__device__ __forceinline__ void st_cs(uint4* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// Two fp32 -> packed bf16x2 (round to nearest even); lo goes to the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) { return (uint16_t)(pack_bf16x2(f, 0.0f) & 0xFFFFu); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// forward kernels
// ---------------------------------------------------------------------------

constexpr int kThreads = 256;           // 8 warps per CTA
constexpr int kWarps = kThreads / 32;

// Vector path: H % 8 == 0, x and out 16-byte aligned. cpr = H / 8 chunks per half-row.
template <bool BETA4, int UNROLL>
__global__ void __launch_bounds__(kThreads) fwd_vec_kernel(const uint4* __restrict__ x, uint4* __restrict__ out,
                                                           int64_t R, int cpr, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint4* xg = x + r * (2 * (int64_t)cpr);
        const uint4* xl = xg + cpr;
        uint4* o = out + r * (int64_t)cpr;
        for (int c0 = 0; c0 < cpr; c0 += 32 * UNROLL) {
            uint4 gv[UNROLL], lv[UNROLL];
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    gv[k] = ld_nc(xg + ci);
                    lv[k] = ld_nc(xl + ci);
                }
            }
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    const uint32_t gw[4] = {gv[k].x, gv[k].y, gv[k].z, gv[k].w};
                    const uint32_t lw[4] = {lv[k].x, lv[k].y, lv[k].z, lv[k].w};
                    uint32_t ow[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float a0 = situ::fwd<BETA4>(bf16_lo(gw[i]), bf16_lo(lw[i]), c);
                        float a1 = situ::fwd<BETA4>(bf16_hi(gw[i]), bf16_hi(lw[i]), c);
                        ow[i] = pack_bf16x2(a0, a1);
                    }
                    st_cs(o + ci, make_uint4(ow[0], ow[1], ow[2], ow[3]));
                }
            }
        }
    }
}

// Element path: any H, any 2-byte-aligned pointers.
template <bool BETA4>
__global__ void __launch_bounds__(kThreads) fwd_elem_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                                            int64_t R, int64_t H, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint16_t* xr = x + r * 2 * H;
        uint16_t* orow = out + r * H;
        for (int64_t j = lane; j < H; j += 32) {
            float a = situ::fwd<BETA4>(bf16_to_f32(xr[j]), bf16_to_f32(xr[H + j]), c);
            orow[j] = f32_to_bf16(a);
        }
    }
}

// ---------------------------------------------------------------------------
// backward + router-gradient kernels
// ---------------------------------------------------------------------------

template <bool BETA4>
__device__ __forceinline__ void bwd_chunk(const uint4& gv, const uint4& lv, const uint4& dv, float p, const Coef& c,
                                          float& acc, uint4& dgo, uint4& dlo) {
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
    const uint32_t yw[4] = {dv.x, dv.y, dv.z, dv.w};
    uint32_t dg[4], dl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float g0 = bf16_lo(yw[i]), g1 = bf16_hi(yw[i]);
        situ::Bwd b0 = situ::bwd<BETA4>(bf16_lo(gw[i]), bf16_lo(lw[i]), p * g0, c);
        situ::Bwd b1 = situ::bwd<BETA4>(bf16_hi(gw[i]), bf16_hi(lw[i]), p * g1, c);
        acc = fmaf(g0, b0.a, acc);
        acc = fmaf(g1, b1.a, acc);
        dg[i] = pack_bf16x2(b0.dgate, b1.dgate);
        dl[i] = pack_bf16x2(b0.dlin, b1.dlin);
    }
    dgo = make_uint4(dg[0], dg[1], dg[2], dg[3]);
    dlo = make_uint4(dl[0], dl[1], dl[2], dl[3]);
}

// Vector path: H % 8 == 0; x, g, dx 16-byte aligned. dx may equal x (in place): every
// 16-byte chunk of x is loaded by the lane that later stores the same chunk of dx, and
// no thread reads a chunk after it was written, so x is read through the coherent path.
template <bool BETA4, int UNROLL>
__global__ void __launch_bounds__(kThreads) bwd_vec_kernel(const uint4* x, const uint4* __restrict__ g,
                                                           const float* __restrict__ p, uint4* dx,
                                                           float* __restrict__ dp, int64_t R, int cpr, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint4* xg = x + r * (2 * (int64_t)cpr);
        const uint4* xl = xg + cpr;
        const uint4* gr = g + r * (int64_t)cpr;
        uint4* dgr = dx + r * (2 * (int64_t)cpr);
        uint4* dlr = dgr + cpr;
        const float pr = p[r];
        float acc = 0.0f;
        for (int c0 = 0; c0 < cpr; c0 += 32 * UNROLL) {
            uint4 gv[UNROLL], lv[UNROLL], yv[UNROLL];
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    gv[k] = ld_co(xg + ci);
                    lv[k] = ld_co(xl + ci);
                    yv[k] = ld_nc(gr + ci);
                }
            }
#pragma unroll
            for (int k = 0; k < UNROLL; ++k) {
                const int ci = c0 + k * 32 + lane;
                if (ci < cpr) {
                    uint4 dgo, dlo;
                    bwd_chunk<BETA4>(gv[k], lv[k], yv[k], pr, c, acc, dgo, dlo);
                    st_cs(dgr + ci, dgo);
                    st_cs(dlr + ci, dlo);
                }
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) dp[r] = acc;
    }
}

// Element path: any H, any 2-byte-aligned bf16 pointers. dx may equal x (each element is
// read and then written by the same lane).
template <bool BETA4>
__global__ void __launch_bounds__(kThreads) bwd_elem_kernel(const uint16_t* x, const uint16_t* __restrict__ g,
                                                            const float* __restrict__ p, uint16_t* dx,
                                                            float* __restrict__ dp, int64_t R, int64_t H, Coef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
    for (int64_t r = warp0; r < R; r += nwarps) {
        const uint16_t* xr = x + r * 2 * H;
        const uint16_t* gr = g + r * H;
        uint16_t* dxr = dx + r * 2 * H;
        const float pr = p[r];
        float acc = 0.0f;
        for (int64_t j = lane; j < H; j += 32) {
            float u = bf16_to_f32(xr[j]);
            float v = bf16_to_f32(xr[H + j]);
            float gj = bf16_to_f32(gr[j]);
            situ::Bwd b = situ::bwd<BETA4>(u, v, pr * gj, c);
            acc = fmaf(gj, b.a, acc);
            dxr[j] = f32_to_bf16(b.dgate);
            dxr[H + j] = f32_to_bf16(b.dlin);
        }
        acc = warp_sum(acc);
        if (lane == 0) dp[r] = acc;
    }
}

// ---------------------------------------------------------------------------
// host side: validation, launch configuration, errors
// ---------------------------------------------------------------------------

constexpr int kFwdUnroll = 4;
constexpr int kBwdUnroll = 4;

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return SITU_GLU_CUDA_ERROR;
}

Coef make_coef(float beta, float lbeta) {
    const double log2e = 1.4426950408889634074;
    Coef c;
    c.k_tu = (float)(-(2.0 / (double)beta) * log2e);
    c.k_su = (float)(-log2e);
    c.k_tv = (float)(-(2.0 / (double)lbeta) * log2e);
    c.inv_beta = (float)(1.0 / (double)beta);
    c.inv_lbeta = (float)(1.0 / (double)lbeta);
    c.beta = beta;
    c.lbeta = lbeta;
    c.beta_lbeta = (float)((double)beta * (double)lbeta);
    return c;
}

bool finite_positive(float f) { return isfinite(f) && f > 0.0f; }

// The beta == 4 kernels share one exponential between tanh(u/4) and sigmoid(u) and skip the
// small-argument series; their absolute error in L grows like lbeta * 2^-21, so they are used
// only for lbeta <= 64 (error below 3e-5). Every other (beta, lbeta) takes the general kernels.
constexpr float kFastMaxLbeta = 64.0f;
bool fast_path(float beta, float lbeta) { return beta == 4.0f && lbeta <= kFastMaxLbeta; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void* p, int64_t bytes) {
    uintptr_t lo = (uintptr_t)p;
    return Range{lo, lo + (uintptr_t)bytes};
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Shared checks of R, H, beta, lbeta; sets *elems2 = R*2H when valid.
int check_shape(int64_t R, int64_t H, float beta, float lbeta) {
    if (R < 0 || H <= 0 || H > SITU_GLU_MAX_H) return SITU_GLU_INVALID_ARG;
    if (!finite_positive(beta) || !finite_positive(lbeta)) return SITU_GLU_INVALID_ARG;
    // R * 2H * 2 bytes must fit in int64
    if (R > 0 && R > (INT64_MAX / 4) / H) return SITU_GLU_INVALID_ARG;
    return SITU_GLU_OK;
}

// Per-device launch configuration cache: SM count and resident CTAs per SM for each kernel.
constexpr int kMaxDevices = 64;
constexpr int kNumKernels = 8;
std::mutex g_cfg_mutex;
int g_sm_count[kMaxDevices];
int g_blocks_per_sm[kMaxDevices][kNumKernels];

int grid_for(int kernel_id, const void* fn, int64_t R, int* grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    int sms, per_sm;
    {
        std::lock_guard<std::mutex> lock(g_cfg_mutex);
        if (g_sm_count[dev] == 0) {
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_fail(e);
            g_sm_count[dev] = n;
        }
        if (g_blocks_per_sm[dev][kernel_id] == 0) {
            int b = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, kThreads, 0);
            if (e != cudaSuccess) return cuda_fail(e);
            g_blocks_per_sm[dev][kernel_id] = b > 0 ? b : 1;
        }
        sms = g_sm_count[dev];
        per_sm = g_blocks_per_sm[dev][kernel_id];
    }
    const int64_t persistent = (int64_t)sms * per_sm;
    const int64_t needed = (R + kWarps - 1) / kWarps;  // one warp per row
    *grid = (int)(needed < persistent ? needed : persistent);
    return SITU_GLU_OK;
}

template <typename Kernel, typename... Args>
int launch(int kernel_id, Kernel kernel, int64_t R, cudaStream_t stream, Args... args) {
    int grid = 0;
    int st = grid_for(kernel_id, (const void*)kernel, R, &grid);
    if (st != SITU_GLU_OK) return st;
    kernel<<<grid, kThreads, 0, stream>>>(args...);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // namespace

extern "C" {

int situ_glu_fwd(const void* x, void* out, int64_t R, int64_t H, float beta, float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    if (R == 0) return SITU_GLU_OK;
    if (x == nullptr || out == nullptr) return SITU_GLU_INVALID_ARG;
    if (!aligned(x, 2) || !aligned(out, 2)) return SITU_GLU_INVALID_ARG;
    const int64_t xb = R * 2 * H * 2, ob = R * H * 2;
    if (overlap(range_of(x, xb), range_of(out, ob))) return SITU_GLU_OVERLAP;

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    const bool vec = (H % 8 == 0) && aligned(x, 16) && aligned(out, 16);
    if (vec) {
        const int cpr = (int)(H / 8);
        const uint4* xv = (const uint4*)x;
        uint4* ov = (uint4*)out;
        if (b4) return launch(0, fwd_vec_kernel<true, kFwdUnroll>, R, stream, xv, ov, R, cpr, c);
        return launch(1, fwd_vec_kernel<false, kFwdUnroll>, R, stream, xv, ov, R, cpr, c);
    }
    const uint16_t* xs = (const uint16_t*)x;
    uint16_t* os = (uint16_t*)out;
    if (b4) return launch(2, fwd_elem_kernel<true>, R, stream, xs, os, R, H, c);
    return launch(3, fwd_elem_kernel<false>, R, stream, xs, os, R, H, c);
}

int situ_glu_bwd_router(const void* x, const void* g, const float* p, void* dx, float* dp, int64_t R, int64_t H,
                        float beta, float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    if (R == 0) return SITU_GLU_OK;
    if (x == nullptr || g == nullptr || p == nullptr || dx == nullptr || dp == nullptr) return SITU_GLU_INVALID_ARG;
    if (!aligned(x, 2) || !aligned(g, 2) || !aligned(dx, 2) || !aligned(p, 4) || !aligned(dp, 4))
        return SITU_GLU_INVALID_ARG;
    const Range rx = range_of(x, R * 2 * H * 2), rg = range_of(g, R * H * 2), rp = range_of(p, R * 4);
    const Range rdx = range_of(dx, R * 2 * H * 2), rdp = range_of(dp, R * 4);
    const bool in_place = (dx == x);
    if (!in_place && overlap(rdx, rx)) return SITU_GLU_OVERLAP;
    if (overlap(rdx, rg) || overlap(rdx, rp) || overlap(rdx, rdp)) return SITU_GLU_OVERLAP;
    if (overlap(rdp, rx) || overlap(rdp, rg) || overlap(rdp, rp)) return SITU_GLU_OVERLAP;

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    const bool vec = (H % 8 == 0) && aligned(x, 16) && aligned(g, 16) && aligned(dx, 16);
    if (vec) {
        const int cpr = (int)(H / 8);
        const uint4* xv = (const uint4*)x;
        const uint4* gv = (const uint4*)g;
        uint4* dxv = (uint4*)dx;
        if (b4) return launch(4, bwd_vec_kernel<true, kBwdUnroll>, R, stream, xv, gv, p, dxv, dp, R, cpr, c);
        return launch(5, bwd_vec_kernel<false, kBwdUnroll>, R, stream, xv, gv, p, dxv, dp, R, cpr, c);
    }
    const uint16_t* xs = (const uint16_t*)x;
    const uint16_t* gs = (const uint16_t*)g;
    uint16_t* dxs = (uint16_t*)dx;
    if (b4) return launch(6, bwd_elem_kernel<true>, R, stream, xs, gs, p, dxs, dp, R, H, c);
    return launch(7, bwd_elem_kernel<false>, R, stream, xs, gs, p, dxs, dp, R, H, c);
}

const char* situ_glu_status_string(int status) {
    switch (status) {
        case SITU_GLU_OK: return "ok";
        case SITU_GLU_INVALID_ARG: return "invalid argument (null pointer, bad size, bad beta/lbeta or misaligned pointer)";
        case SITU_GLU_OVERLAP: return "output buffer overlaps an input or another output";
        case SITU_GLU_CUDA_ERROR: return "CUDA error (see situ_glu_last_cuda_error)";
        default: return "unknown status";
    }
}

int situ_glu_last_cuda_error(void) { return t_last_cuda_error; }

int situ_glu_version(void) {
    return SITU_GLU_VERSION_MAJOR * 10000 + SITU_GLU_VERSION_MINOR * 100 + SITU_GLU_VERSION_PATCH;
}

}  // extern "C"
