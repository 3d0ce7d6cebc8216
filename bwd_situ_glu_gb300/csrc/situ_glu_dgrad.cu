// situ_glu_dgrad.cu — down-projection dgrad grouped GEMM on the 5th-generation tensor cores
// (tcgen05, TMA, TMEM), with the SiTU-GLU backward and the router gradient fused into its epilogue.
//
// "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出": for a routed row of
// expert e, g = (W_down,e)ᵀ·dL/dy is what the backward computes on its way to a_e; from it,
// dL/dp_e = <g, a_e> and dL/da_e = p_e·g. This kernel forms g = dY_e·W_down,e per expert with
// tcgen05.mma into TMEM and, without ever writing g, evaluates in the epilogue
//   dp[r] = Σ_j g[r,j]·a[r,j],  dx[r,j] = p·g·L·G',  dx[r,H+j] = p·g·G·L'
// from the fp32 accumulators and the saved bf16 x ("Frontier-scale RL with Kimi K3", section
// "Streaming activations": the backward keeps only x and recomputes tanh and sigmoid).
//
// Per-CTA pipeline (one CTA per SM, persistent over M-tiles of 128 rows of one expert):
//   warp 0      TMA producer: dY tile [128 x 64] and W_downᵀ tile [256 x 64] (bf16, 128-byte
//               swizzle) into a 4-stage shared-memory ring, completion on mbarriers;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and one thread
//               issues tcgen05.mma (M = 128, N = 256, K = 16), committing to mbarriers that free
//               ring stages and hand finished accumulators to the epilogue;
//   warps 2..   epilogue, EPW warps per 32-lane TMEM quadrant, each with a slice of the 256 columns;
//               a thread owns one row, reads its g with tcgen05.ld, loads the matching x (prefetched
//               one chunk ahead), and writes dx; its dp partial stays in a register across the
//               N-tiles of the row.
// Every mbarrier wait is bounded: on a timeout the CTA records a non-zero status, stops issuing,
// drains what it issued, frees TMEM and returns.
#include <cuda.h>
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

constexpr int BM = 128;                      // rows per tile (TMEM lanes)
constexpr int BN = 256;                      // accumulator columns per job
constexpr int BK = 64;                       // K per ring stage (128 bytes of bf16: one swizzle row)
constexpr int UK = 16;                       // K per tcgen05.mma (kind::f16)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BYTES = BN * BK * 2;         // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPW = 2;                       // epilogue warps per 32-lane TMEM quadrant
constexpr int CW = 32;                       // accumulator columns per tcgen05.ld chunk
constexpr int NUM_EPI_THREADS = 4 * EPW * 32;
constexpr int NUM_THREADS = 64 + NUM_EPI_THREADS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int COLS_PER_WARP = BN / EPW;      // accumulator columns of one job an epilogue warp owns
constexpr int CPJ = COLS_PER_WARP / CW;      // chunks per job per epilogue warp
constexpr int XV = CW / 16;                  // 32-byte vectors (16 bf16) per half-row per chunk
static_assert(CPJ >= 2 && CPJ % 2 == 0, "the x prefetch alternates two register buffers");
constexpr int TMEM_COLS = 512;               // 2 accumulators x 256 columns
constexpr int MAX_EXPERTS = 4096;
constexpr uint32_t WAIT_LIMIT = 1u << 22;    // polls of a try_wait before giving up (~1-2 s)

// Shared memory layout (dynamic, base rounded up to 1024 bytes for the 128-byte swizzle).
struct alignas(8) Barriers {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + (int)sizeof(Barriers) + EPW * BM * 4 +
                           (MAX_EXPERTS + 1) * 4 + 64;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_addr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; on a timeout sets the CTA's abort flag and the caller's status word.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Barriers* bars, int* status) {
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(b, parity)) return true;
        if (i > 64 && *(volatile int*)&bars->abort) return false;
    }
    *(volatile int*)&bars->abort = 1;
    if (status) atomicExch(status, 1);
    return false;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major bf16 tile with 128-byte swizzle: rows of 128 bytes,
// 8-row groups 1024 bytes apart (stride byte offset), version bits 46-47 = 1, swizzle mode 2.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);          // start address
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset: 8 rows x 128 B
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both K-major, N = 256, M = 128.
constexpr uint32_t IDESC = (1u << 4)           // D format fp32
                         | (1u << 7)           // A format bf16
                         | (1u << 10)          // B format bf16
                         | ((uint32_t)(BN >> 3) << 17)
                         | ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// N consecutive fp32 columns (N = 16 or 32) of this thread's TMEM lane, waited for.
template <int N>
__device__ __forceinline__ void tc_ld(uint32_t taddr, float (&v)[N]) {
    uint32_t r[N];
    if constexpr (N == 32) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
            "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
              "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
              "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
              "=r"(r[30]), "=r"(r[31])
            : "r"(taddr));
    } else {
        static_assert(N == 16, "16 or 32 columns");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
            : "r"(taddr));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, %0;" ::"r"(NUM_EPI_THREADS) : "memory"); }

// M-tile t -> (expert, first row, end row of the expert).
__device__ __forceinline__ void tile_rows(const int* tile_start, const int64_t* off, int E, int64_t R, int t,
                                          int& e, int64_t& row0, int64_t& row_end) {
    int lo = 0, hi = E - 1;                 // last e with tile_start[e] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    row0 = off[e] + (int64_t)(t - tile_start[e]) * BM;
    row_end = off[e + 1] < R ? off[e + 1] : R;     // clamped: malformed offsets never index past R
}

// ---------------------------------------------------------------- the kernel

template <bool BETA4>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    dgrad_bwd_kernel(const __grid_constant__ CUtensorMap map_dy, const __grid_constant__ CUtensorMap map_w,
                     const uint16_t* __restrict__ x, const int64_t* __restrict__ offsets, const float* __restrict__ p,
                     uint16_t* __restrict__ dx, float* __restrict__ dp, int* __restrict__ status, int E, int64_t R,
                     int64_t H, int KB, Coef c) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t* ring = smem;                                            // STAGES x (A | B)
    Barriers* bars = (Barriers*)(smem + STAGES * STAGE_BYTES);
    float* dp_part = (float*)(bars + 1);                             // [EPW][BM] per-warp-slot dp partials
    int* tile_start = (int*)(dp_part + EPW * BM);                    // [E + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (int)(H / BN);

    // tile prefix over experts (each CTA builds its own copy): counts in parallel, then one
    // warp scans them (each lane a contiguous segment, shuffles across lanes)
    for (int e = threadIdx.x; e < E; e += NUM_THREADS) {
        const int64_t n = offsets[e + 1] - offsets[e];
        tile_start[e + 1] = n > 0 ? (int)((n + BM - 1) / BM) : 0;
    }
    if (threadIdx.x == 0) {
        tile_start[0] = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->tfull[a], 1);
            mbar_init(&bars->tempty[a], NUM_EPI_THREADS);
        }
        mbar_init(&bars->mma_done, 1);
        bars->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        const int seg = (E + 31) / 32;
        const int b = 1 + lane * seg, en = min(E + 1, b + seg);
        int sum = 0;
        for (int i = b; i < en; ++i) sum += tile_start[i];
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int i = b; i < en; ++i) {
            run += tile_start[i];
            tile_start[i] = run;
        }
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&bars->tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int T = tile_start[E];

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t pending = 0;            // bit s: stage s has a load in flight of parity pend_par
            uint32_t pend_par = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x) {
                int e;
                int64_t row0, row_end;
                tile_rows(tile_start, offsets, E, R, t, e, row0, row_end);
                for (int nt = 0; ok && nt < NT; ++nt) {
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!mbar_wait(&bars->empty[stage], phase ^ 1, bars, status)) { ok = false; break; }
                        mbar_expect_tx(&bars->full[stage], STAGE_BYTES);
                        uint8_t* sa = ring + stage * STAGE_BYTES;
                        tma_load_2d(sa, &map_dy, kb * BK, (int)row0, &bars->full[stage]);
                        tma_load_2d(sa + A_BYTES, &map_w, kb * BK, (int)((int64_t)e * H + (int64_t)nt * BN),
                                    &bars->full[stage]);
                        pending |= 1u << stage;
                        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                }
            }
            // every load issued must land before the CTA exits: wait for each stage's last phase
            for (int s2 = 0; s2 < STAGES; ++s2) {
                if (!(pending & (1u << s2))) continue;
                const uint32_t par = (pend_par >> s2) & 1u;
                for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
                    if (mbar_try_wait(&bars->full[s2], par)) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int job = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < T; t += gridDim.x) {
                for (int nt = 0; ok && nt < NT; ++nt, ++job) {
                    const int acc = job & 1;
                    const uint32_t acc_phase = (uint32_t)((job >> 1) & 1);
                    if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1, bars, status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!mbar_wait(&bars->full[stage], phase, bars, status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t sa = smem_addr(ring + stage * STAGE_BYTES);
                        const uint64_t adesc = smem_desc(sa), bdesc = smem_desc(sa + A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UK; ++kk) {
                            // advance 16 bf16 (32 bytes = 2 descriptor units) along K inside the swizzled rows
                            tc_mma(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2),
                                   (kb > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc_commit(&bars->empty[stage]);          // ring stage free once these MMAs finish
                        if (++stage == STAGES) { stage = 0; phase ^= 1; }
                    }
                    if (ok) tc_commit(&bars->tfull[acc]);        // accumulator complete
                }
            }
            // all MMAs issued by this thread complete before TMEM is freed
            tc_commit(&bars->mma_done);
            for (uint32_t i = 0; i < WAIT_LIMIT; ++i)
                if (mbar_try_wait(&bars->mma_done, 0)) break;
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2 .. 2 + 4·EPW − 1)
        // A warp may read only the TMEM lanes of quadrant warp % 4; the EPW warps of a quadrant split
        // each job's 256 columns into EPW slices of COLS_PER_WARP, read CW columns at a time. One
        // thread owns one row for a whole M-tile: its x is fetched with 32-byte loads one chunk ahead
        // (across job boundaries too, as x does not depend on the accumulator), so the loads are in
        // flight while the previous chunk is computed and while the next accumulator is awaited.
        const int quad = warp & 3;
        const int slot = (warp - 2) >> 2;
        const int lrow = quad * 32 + lane;         // row within the tile
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        int job = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < T; t += gridDim.x) {
            int e;
            int64_t row0, row_end;
            tile_rows(tile_start, offsets, E, R, t, e, row0, row_end);
            const int64_t row = row0 + lrow;
            const bool valid = ok && row >= 0 && row < row_end;
            const float pr16 = valid ? 16.0f * p[row] : 0.0f;
            const uint16_t* xr = x + (valid ? row : 0) * 2 * H + slot * COLS_PER_WARP;
            uint16_t* dxr = dx + (valid ? row : 0) * 2 * H + slot * COLS_PER_WARP;
            float acc_dp = 0.0f;
            Vec<8> xb[2][2][XV];                   // [buffer][gate, linear][32-byte vector]
            if (valid) {
#pragma unroll
                for (int v = 0; v < XV; ++v) {
                    xb[0][0][v] = ld_stream<8, true>((const Vec<8>*)(xr + 16 * v));
                    xb[0][1][v] = ld_stream<8, true>((const Vec<8>*)(xr + H + 16 * v));
                }
            }
            for (int nt = 0; nt < NT; ++nt, ++job) {
                const int acc = job & 1;
                const uint32_t acc_phase = (uint32_t)((job >> 1) & 1);
                if (ok && !mbar_wait(&bars->tfull[acc], acc_phase, bars, status)) ok = false;
                ok = __all_sync(0xffffffffu, ok);                 // tcgen05.ld below is warp-collective
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < CPJ; ++k) {
                    const int cur = k & 1;
                    // prefetch the next chunk of this row: (nt, k + 1), or (nt + 1, 0) after the last
                    const bool last = (k + 1 == CPJ);
                    if (valid && (!last || nt + 1 < NT)) {
                        const int64_t jn = last ? (int64_t)(nt + 1) * BN : (int64_t)nt * BN + (k + 1) * CW;
#pragma unroll
                        for (int v = 0; v < XV; ++v) {
                            xb[cur ^ 1][0][v] = ld_stream<8, true>((const Vec<8>*)(xr + jn + 16 * v));
                            xb[cur ^ 1][1][v] = ld_stream<8, true>((const Vec<8>*)(xr + H + jn + 16 * v));
                        }
                    }
                    float gv[CW];
                    if (ok) tc_ld<CW>(tmem + t_lane + (uint32_t)(acc * BN + slot * COLS_PER_WARP + k * CW), gv);
                    if (last) {
                        tc_fence_before();
                        mbar_arrive(&bars->tempty[acc]);       // accumulator may be overwritten
                    }
                    if (ok && valid) {
                        const int64_t j0 = (int64_t)nt * BN + k * CW;
#pragma unroll
                        for (int v = 0; v < XV; ++v) {
                            Vec<8> dgo, dlo;
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const uint32_t gw = xb[cur][0][v].w[i], lw = xb[cur][1][v].w[i];
                                const float g0 = gv[16 * v + 2 * i], g1 = gv[16 * v + 2 * i + 1];
                                situ::Bwd b0 = situ::bwd<BETA4>(bf16_lo(gw), bf16_lo(lw), pr16 * g0, c);
                                situ::Bwd b1 = situ::bwd<BETA4>(bf16_hi(gw), bf16_hi(lw), pr16 * g1, c);
                                acc_dp = fmaf(g0, b0.a16, acc_dp);
                                acc_dp = fmaf(g1, b1.a16, acc_dp);
                                dgo.w[i] = pack_bf16x2(b0.dgate, b1.dgate);
                                dlo.w[i] = pack_bf16x2(b0.dlin, b1.dlin);
                            }
                            st_stream<8>((Vec<8>*)(dxr + j0 + 16 * v), dgo);
                            st_stream<8>((Vec<8>*)(dxr + H + j0 + 16 * v), dlo);
                        }
                    }
                }
            }
            // combine the EPW column slices of each row
            if (slot > 0) dp_part[slot * BM + lrow] = acc_dp;
            epi_barrier();
            if (slot == 0 && valid) {
                float s = acc_dp;
#pragma unroll
                for (int k = 1; k < EPW; ++k) s += dp_part[k * BM + lrow];
                dp[row] = 16.0f * s;
            }
            epi_barrier();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiled)p;
    });
    return fn;
}

// 2-D bf16 tensor map: rows x cols (cols contiguous), box of box_rows x 64 columns, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int situ_glu_bwd_router_dgrad(const void* x, const void* dy, const void* w_down_t, const int64_t* expert_offsets,
                              int64_t E, const float* p, void* dx, float* dp, int* status, int64_t R, int64_t H,
                              int64_t D, float beta, float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    if (D <= 0 || D % BK != 0 || H % BN != 0 || E < 1 || E > MAX_EXPERTS) return SITU_GLU_INVALID_ARG;
    if (R > INT32_MAX || E * H > INT32_MAX || D > INT32_MAX / 2) return SITU_GLU_INVALID_ARG;
    if (R == 0) return SITU_GLU_OK;
    if (!x || !dy || !w_down_t || !expert_offsets || !p || !dx || !dp) return SITU_GLU_INVALID_ARG;
    if (!aligned(x, 32) || !aligned(dy, 16) || !aligned(w_down_t, 16) || !aligned(dx, 32) ||
        !aligned(expert_offsets, 8) || !aligned(p, 4) || !aligned(dp, 4) || (status && !aligned(status, 4)))
        return SITU_GLU_INVALID_ARG;
    const Range rx = range_of(x, R * 2 * H * 2), ry = range_of(dy, R * D * 2), rw = range_of(w_down_t, E * H * D * 2);
    const Range ro = range_of(expert_offsets, (E + 1) * 8), rp = range_of(p, R * 4);
    const Range rdx = range_of(dx, R * 2 * H * 2), rdp = range_of(dp, R * 4);
    for (Range in : {rx, ry, rw, ro, rp}) {
        if (overlap(rdx, in) || overlap(rdp, in)) return SITU_GLU_OVERLAP;
        if (status && overlap(range_of(status, 4), in)) return SITU_GLU_OVERLAP;
    }
    if (overlap(rdx, rdp)) return SITU_GLU_OVERLAP;
    if (status && (overlap(range_of(status, 4), rdx) || overlap(range_of(status, 4), rdp))) return SITU_GLU_OVERLAP;

    CUtensorMap map_dy, map_w;
    if (!make_map(&map_dy, dy, (uint64_t)R, (uint64_t)D, BM)) return cuda_fail(cudaErrorInvalidValue);
    if (!make_map(&map_w, w_down_t, (uint64_t)(E * H), (uint64_t)D, BN)) return cuda_fail(cudaErrorInvalidValue);

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    auto kernel = b4 ? dgrad_bwd_kernel<true> : dgrad_bwd_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(e);
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return cuda_fail(e);
    // persistent: one CTA per SM, never more CTAs than M-tiles could need
    const int64_t max_tiles = (R + BM - 1) / BM + E;
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(map_dy, map_w, (const uint16_t*)x, expert_offsets, p,
                                                      (uint16_t*)dx, dp, status, (int)E, R, H, (int)(D / BK), c);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // extern "C"
