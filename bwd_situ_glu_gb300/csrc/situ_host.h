// situ_host.h — host-side helpers shared by the library's translation units: argument checks,
// per-launch constants, launch-configuration cache and CUDA error bookkeeping.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "../../include/situ_glu.h"
#include "situ_math.cuh"

namespace situ_host {

using situ::Coef;

// The cudaError_t behind the last SITU_GLU_CUDA_ERROR on this host thread.
inline thread_local int t_last_cuda_error = 0;

inline int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return SITU_GLU_CUDA_ERROR;
}

inline Coef make_coef(float beta, float lbeta) {
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
    c.beta_4 = (float)((double)beta / 4.0);
    c.lbeta_4 = (float)((double)lbeta / 4.0);
    return c;
}

inline bool finite_positive(float f) { return isfinite(f) && f > 0.0f; }

// The beta == 4 kernels share one exponential between tanh(u/4) and sigmoid(u) and skip the
// small-argument series; their absolute error in L grows like lbeta * 2^-21, so they are used
// only for lbeta <= 64 (error below 3e-5). Every other (beta, lbeta) takes the general kernels.
constexpr float kFastMaxLbeta = 64.0f;
inline bool fast_path(float beta, float lbeta) { return beta == 4.0f && lbeta <= kFastMaxLbeta; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

inline bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

inline Range range_of(const void* p, int64_t bytes) {
    uintptr_t lo = (uintptr_t)p;
    return Range{lo, lo + (uintptr_t)bytes};
}

inline bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Shared checks of R, H, beta, lbeta.
inline int check_shape(int64_t R, int64_t H, float beta, float lbeta) {
    if (R < 0 || H <= 0 || H > SITU_GLU_MAX_H) return SITU_GLU_INVALID_ARG;
    if (!finite_positive(beta) || !finite_positive(lbeta)) return SITU_GLU_INVALID_ARG;
    // R * 2H * 2 bytes must fit in int64
    if (R > 0 && R > (INT64_MAX / 4) / H) return SITU_GLU_INVALID_ARG;
    return SITU_GLU_OK;
}

// Per-device launch configuration: SM count and resident CTAs per SM of each kernel.
constexpr int kMaxDevices = 64;

struct LaunchCache {
    std::mutex mu;
    int sm_count[kMaxDevices] = {};
    std::unordered_map<const void*, int> blocks_per_sm[kMaxDevices];
};

inline LaunchCache& launch_cache() {
    static LaunchCache cache;
    return cache;
}

// Persistent grid: SM count x resident CTAs per SM, capped by one warp per row.
inline int grid_for(const void* fn, int tpb, int64_t R, int* grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    LaunchCache& lc = launch_cache();
    int sms, per_sm;
    {
        std::lock_guard<std::mutex> lock(lc.mu);
        if (lc.sm_count[dev] == 0) {
            int n = 0;
            e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return cuda_fail(e);
            lc.sm_count[dev] = n;
        }
        auto it = lc.blocks_per_sm[dev].find(fn);
        if (it == lc.blocks_per_sm[dev].end()) {
            int b = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, fn, tpb, 0);
            if (e != cudaSuccess) return cuda_fail(e);
            it = lc.blocks_per_sm[dev].emplace(fn, b > 0 ? b : 1).first;
        }
        sms = lc.sm_count[dev];
        per_sm = it->second;
    }
    const int64_t persistent = (int64_t)sms * per_sm;
    const int64_t warps_per_cta = tpb / 32;
    const int64_t needed = (R + warps_per_cta - 1) / warps_per_cta;
    *grid = (int)(needed < persistent ? needed : persistent);
    return SITU_GLU_OK;
}

template <typename Kernel, typename... Args>
int launch(Kernel kernel, int tpb, int64_t R, cudaStream_t stream, Args... args) {
    int grid = 0;
    int st = grid_for((const void*)kernel, tpb, R, &grid);
    if (st != SITU_GLU_OK) return st;
    kernel<<<grid, tpb, 0, stream>>>(args...);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // namespace situ_host
