// situ_adam.cu — Adam on host-resident optimizer state, streamed chunk by chunk (host code and
// CUDA copies only; no device kernel).
//
// "Frontier-scale RL with Kimi K3", sections "Memory management" and "Streaming gradients": the
// optimizer state lives in host memory (fp32 master weights and two bf16 moment tensors); the
// gradients computed on the device are brought to the host and the updated weights sent back as
// the bf16 working copy. Moving all gradients in one transfer needs a parameter-sized fp32 host
// gradient buffer (12 bytes of host memory per parameter in total); because Adam updates every
// parameter independently, the update can instead run chunk by chunk with the transfers of the
// next chunks in flight, and only a few chunk-sized staging slots remain (8 bytes per parameter
// plus the slots).
//
// Host arithmetic: one Adam step per element as a fixed sequence of single IEEE fp32 operations
// (this file is compiled without floating-point contraction, and without errno from sqrtf so the
// element loop vectorises; IEEE results are the same), so every result, including the bf16
// codes of the moments, is fully determined:
//   constants (formed in double from the double hyper-parameters, each rounded to fp32 once):
//     b1, b2, eps, c1 = 1 - b1, c2 = 1 - b2, s = lr / (1 - b1^t), r = 1 / sqrt(1 - b2^t),
//     d = 1 - lr·wd
//   w1 = wd > 0 ? w·d : w                      (decoupled weight decay)
//   m1 = b1·m + c1·g                           (two products, then the sum)
//   v1 = b2·v + c2·(g·g)
//   q  = sqrt(v1)·r + eps
//   w2 = w1 - s·(m1 / q)
//   stored: master = w2, m = bf16(m1), v = bf16(v1), working weight = bf16(w2), bf16 rounding to
//   nearest even (NaN -> 0x7FC0).
#include <cuda_runtime.h>
#include <math.h>
#include <sched.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <thread>
#include <vector>

#include "../../include/situ_glu.h"
#include "situ_host.h"

namespace {

using situ_host::cuda_fail;

// ---------------------------------------------------------------- element update

struct Consts {
    float b1, b2, eps, c1, c2, s, r, d;
    bool decay;
};

Consts make_consts(const situ_adam_params& hp) {
    const double bc1 = 1.0 - pow(hp.beta1, (double)hp.step);
    const double bc2 = 1.0 - pow(hp.beta2, (double)hp.step);
    Consts k;
    k.b1 = (float)hp.beta1;
    k.b2 = (float)hp.beta2;
    k.eps = (float)hp.eps;
    k.c1 = (float)(1.0 - hp.beta1);
    k.c2 = (float)(1.0 - hp.beta2);
    k.s = (float)(hp.lr / bc1);
    k.r = (float)(1.0 / sqrt(bc2));
    k.d = (float)(1.0 - hp.lr * hp.weight_decay);
    k.decay = hp.weight_decay > 0.0;
    return k;
}

inline float from_bf16(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// Round to nearest even; carries into the exponent give the next binade or infinity as they
// should. Written without branches (NaN by a select) so the update loop vectorises.
inline uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    const uint32_t rounded = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
    return (uint16_t)(((u & 0x7FFFFFFFu) > 0x7F800000u) ? 0x7FC0u : rounded);
}

template <bool DECAY>
void update_range_t(float* __restrict__ master, uint16_t* __restrict__ m, uint16_t* __restrict__ v,
                    const float* __restrict__ g, uint16_t* __restrict__ w_out, int64_t n, const Consts& k) {
    const float b1 = k.b1, b2 = k.b2, c1 = k.c1, c2 = k.c2, s = k.s, r = k.r, eps = k.eps, d = k.d;
    for (int64_t i = 0; i < n; ++i) {
        float w1 = master[i];
        if constexpr (DECAY) w1 = w1 * d;
        const float gi = g[i];
        const float m1 = b1 * from_bf16(m[i]) + c1 * gi;
        const float v1 = b2 * from_bf16(v[i]) + c2 * (gi * gi);
        const float q = sqrtf(v1) * r + eps;
        const float w2 = w1 - s * (m1 / q);
        master[i] = w2;
        m[i] = to_bf16(m1);
        v[i] = to_bf16(v1);
        w_out[i] = to_bf16(w2);
    }
}

void update_range(float* master, uint16_t* m, uint16_t* v, const float* g, uint16_t* w_out, int64_t n,
                  const Consts& k) {
    if (k.decay)
        update_range_t<true>(master, m, v, g, w_out, n, k);
    else
        update_range_t<false>(master, m, v, g, w_out, n, k);
}

// ---------------------------------------------------------------- validation

bool params_ok(const situ_adam_params* hp) {
    if (!hp) return false;
    const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
    if (!isfinite(lr) || lr < 0.0) return false;
    if (!isfinite(b1) || b1 < 0.0 || b1 >= 1.0) return false;
    if (!isfinite(b2) || b2 < 0.0 || b2 >= 1.0) return false;
    if (!isfinite(eps) || eps <= 0.0) return false;
    if (!isfinite(wd) || wd < 0.0) return false;
    return hp->step >= 1;
}

using situ_host::aligned;
using situ_host::overlap;
using situ_host::Range;
using situ_host::range_of;

int host_threads(int requested) {
    if (requested > 0) return requested;
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        const int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    const unsigned h = std::thread::hardware_concurrency();
    return h > 0 ? (int)h : 1;
}

// Run update_range over [0, n) split into `threads` contiguous slices (the caller's thread takes
// the first).
void update_parallel(float* master, uint16_t* m, uint16_t* v, const float* g, uint16_t* w_out, int64_t n,
                     const Consts& k, int threads) {
    if (threads <= 1 || n < 4096) {
        update_range(master, m, v, g, w_out, n, k);
        return;
    }
    std::vector<std::thread> pool;
    const int64_t per = (n + threads - 1) / threads;
    for (int t = 1; t < threads; ++t) {
        const int64_t a = t * per, b = a + per < n ? a + per : n;
        if (a >= b) break;
        pool.emplace_back(update_range, master + a, m + a, v + a, g + a, w_out + a, b - a, std::cref(k));
    }
    update_range(master, m, v, g, w_out, per < n ? per : n, k);
    for (auto& th : pool) th.join();
}

// Workers for the streamed step: each updates slice `id` of every chunk once the coordinating
// thread has published it (go > c) and reports completion through `done`.
struct Crew {
    std::atomic<int64_t> go{0};
    std::atomic<int64_t> done{0};
    std::atomic<bool> stop{false};
};

}  // namespace

extern "C" {

int situ_adam_update_host(float* master, void* m, void* v, const float* g, void* w_out, int64_t n,
                          const situ_adam_params* hp, int nthreads) {
    if (n < 0 || !params_ok(hp)) return SITU_GLU_INVALID_ARG;
    if (n == 0) return SITU_GLU_OK;
    if (!master || !m || !v || !g || !w_out) return SITU_GLU_INVALID_ARG;
    if (!aligned(master, 4) || !aligned(g, 4) || !aligned(m, 2) || !aligned(v, 2) || !aligned(w_out, 2))
        return SITU_GLU_INVALID_ARG;
    const Range rw = range_of(master, n * 4), rm = range_of(m, n * 2), rv = range_of(v, n * 2);
    const Range rg = range_of(g, n * 4), ro = range_of(w_out, n * 2);
    const Range all[5] = {rw, rm, rv, rg, ro};
    for (int a = 0; a < 5; ++a)
        for (int b = a + 1; b < 5; ++b)
            if (overlap(all[a], all[b])) return SITU_GLU_OVERLAP;
    const Consts k = make_consts(*hp);
    update_parallel(master, (uint16_t*)m, (uint16_t*)v, g, (uint16_t*)w_out, n, k, host_threads(nthreads));
    return SITU_GLU_OK;
}

int situ_adam_stream_step(const float* grad_dev, void* weight_dev, float* master, void* m, void* v, int64_t n,
                          const situ_adam_params* hp, void* staging, int64_t chunk, int nslots, int nthreads,
                          cudaStream_t stream) {
    if (n < 0 || !params_ok(hp) || chunk <= 0 || chunk % 64 != 0 || nslots < 2 || nslots > 64)
        return SITU_GLU_INVALID_ARG;
    if (n == 0) return SITU_GLU_OK;
    if (!grad_dev || !weight_dev || !master || !m || !v || !staging) return SITU_GLU_INVALID_ARG;
    if (!aligned(grad_dev, 4) || !aligned(weight_dev, 2) || !aligned(master, 4) || !aligned(m, 2) ||
        !aligned(v, 2) || !aligned(staging, 16))
        return SITU_GLU_INVALID_ARG;
    if (chunk > (INT64_MAX / 8) / nslots) return SITU_GLU_INVALID_ARG;
    const Range rs = range_of(staging, (int64_t)nslots * chunk * 6);
    const Range host[4] = {range_of(master, n * 4), range_of(m, n * 2), range_of(v, n * 2), rs};
    for (int a = 0; a < 4; ++a)
        for (int b = a + 1; b < 4; ++b)
            if (overlap(host[a], host[b])) return SITU_GLU_OVERLAP;
    if (overlap(range_of(grad_dev, n * 4), range_of(weight_dev, n * 2))) return SITU_GLU_OVERLAP;

    const Consts k = make_consts(*hp);
    float* gslot = (float*)staging;                                  // [nslots][chunk] fp32
    uint16_t* wslot = (uint16_t*)((uint8_t*)staging + (size_t)nslots * chunk * 4);  // [nslots][chunk] bf16
    uint16_t* mh = (uint16_t*)m;
    uint16_t* vh = (uint16_t*)v;
    uint16_t* wd = (uint16_t*)weight_dev;
    const int64_t nchunks = (n + chunk - 1) / chunk;
    auto len_of = [&](int64_t c) { return c + 1 < nchunks ? chunk : n - c * chunk; };

    std::vector<cudaEvent_t> ev_d2h(nslots, nullptr), ev_h2d(nslots, nullptr);
    cudaError_t e = cudaSuccess;
    for (int s = 0; s < nslots && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&ev_d2h[s], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev_h2d[s], cudaEventDisableTiming);
    }

    // the crew: `workers` threads plus this one, each a fixed slice of every chunk
    const int threads = host_threads(nthreads);
    const int workers = threads - 1;
    Crew crew;
    std::vector<std::thread> pool;
    auto slice = [&](int64_t c, int id, int64_t& a, int64_t& b) {
        const int64_t len = len_of(c), per = (len + threads - 1) / threads;
        a = id * per < len ? id * per : len;
        b = a + per < len ? a + per : len;
    };
    auto work = [&](int64_t c, int id) {
        int64_t a, b;
        slice(c, id, a, b);
        if (b <= a) return;
        const int64_t base = c * chunk, s = c % nslots;
        update_range(master + base + a, mh + base + a, vh + base + a, gslot + s * chunk + a,
                     wslot + s * chunk + a, b - a, k);
    };
    if (e == cudaSuccess) {
        for (int id = 1; id <= workers; ++id) {
            pool.emplace_back([&, id] {
                for (int64_t c = 0; c < nchunks; ++c) {
                    while (crew.go.load(std::memory_order_acquire) <= c) {
                        if (crew.stop.load(std::memory_order_acquire)) return;
                        std::this_thread::yield();
                    }
                    if (crew.stop.load(std::memory_order_acquire)) return;
                    work(c, id);
                    crew.done.fetch_add(1, std::memory_order_acq_rel);
                }
            });
        }
    }

    // first nslots gradient chunks in flight
    for (int64_t c = 0; c < nchunks && c < nslots && e == cudaSuccess; ++c) {
        e = cudaMemcpyAsync(gslot + (c % nslots) * chunk, grad_dev + c * chunk, (size_t)len_of(c) * 4,
                            cudaMemcpyDeviceToHost, stream);
        if (e == cudaSuccess) e = cudaEventRecord(ev_d2h[c % nslots], stream);
    }
    for (int64_t c = 0; c < nchunks && e == cudaSuccess; ++c) {
        const int s = (int)(c % nslots);
        e = cudaEventSynchronize(ev_d2h[s]);                        // gradients of chunk c landed
        if (e == cudaSuccess && c >= nslots) e = cudaEventSynchronize(ev_h2d[s]);  // slot's weights sent
        if (e != cudaSuccess) break;
        crew.go.store(c + 1, std::memory_order_release);
        work(c, 0);
        while (crew.done.load(std::memory_order_acquire) < (c + 1) * workers) std::this_thread::yield();
        e = cudaMemcpyAsync(wd + c * chunk, wslot + s * chunk, (size_t)len_of(c) * 2, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaEventRecord(ev_h2d[s], stream);
        if (e == cudaSuccess && c + nslots < nchunks) {
            const int64_t cn = c + nslots;
            e = cudaMemcpyAsync(gslot + s * chunk, grad_dev + cn * chunk, (size_t)len_of(cn) * 4,
                                cudaMemcpyDeviceToHost, stream);
            if (e == cudaSuccess) e = cudaEventRecord(ev_d2h[s], stream);
        }
    }
    // every chunk's weights are on the device; and on an error, no copy this call queued may still
    // be reading or writing the caller's staging slots when it returns
    const cudaError_t es = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = es;

    crew.stop.store(true, std::memory_order_release);
    for (auto& th : pool) th.join();
    for (int s = 0; s < nslots; ++s) {
        if (ev_d2h[s]) cudaEventDestroy(ev_d2h[s]);
        if (ev_h2d[s]) cudaEventDestroy(ev_h2d[s]);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // extern "C"
