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
// The GEMM pipeline (persistent CTAs over 128-row M-tiles of one expert, TMA producer warp,
// single-thread tcgen05.mma issuer, two TMEM accumulators, bounded mbarrier waits) is the one in
// situ_tc.cuh, with A = dY and B = W_downᵀ (rows e·H + nt·256 ..). The epilogue here:
//   EPW = 3 warps per 32-lane TMEM quadrant (12 warps: 3 per SM sub-partition, 128 registers),
//   taking a job's 16-column chunks in turn; a thread owns one row, reads its g with tcgen05.ld,
//   loads the matching x (prefetched one chunk ahead, 32-byte loads), and writes dx; its dp
//   partial stays in a register across the N-tiles of the row and the EPW partials of a row are
//   summed through shared memory at the end of the M-tile.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/situ_glu.h"
#include "situ_device.cuh"
#include "situ_host.h"
#include "situ_math.cuh"
#include "situ_tc.cuh"

namespace {

using namespace situ;
using namespace situ_host;
using namespace situ_tc;

constexpr int EPW = 3;                       // epilogue warps per 32-lane TMEM quadrant
constexpr int CW = 16;                       // accumulator columns per tcgen05.ld chunk
constexpr int NUM_EPI_THREADS = 4 * EPW * 32;
constexpr int NUM_THREADS = 64 + NUM_EPI_THREADS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int NCH = BN / CW;                 // chunks of a job; warp slot s takes chunks s, s + EPW, ...
constexpr int MAXC = (NCH + EPW - 1) / EPW;  // chunks of a job for the busiest slot
constexpr int NBUF = 3;                      // x register buffers, rotating; a job's first chunk uses 0
constexpr int XV = CW / 16;                  // 32-byte vectors (16 bf16) per half-row per chunk
static_assert(XV == 1, "one 32-byte vector per half-row per chunk");
constexpr bool buffers_ok() {                // a slot's last chunk of a job never uses buffer 0,
    for (int s = 0; s < EPW; ++s)            // which the prefetch of the next job's first chunk fills
        if (((NCH - s + EPW - 1) / EPW - 1) % NBUF == 0) return false;
    return true;
}
static_assert(buffers_ok(), "x buffer rotation across job boundaries");
// L2 sector promotion of the operand loads. The weight tiles with 128-byte promotion instead of
// 256: 5-6 % faster at both shapes (896 experts x ~292 rows 7.22-7.27 -> 6.85-6.93 ms, 32 x 8192
// rows 4.49-4.51 -> 4.22 ms, same call); for the dY tiles it makes no measurable difference.
constexpr CUtensorMapL2promotion DGRAD_L2_PROMO_A = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;   // dY tiles
constexpr CUtensorMapL2promotion DGRAD_L2_PROMO_B = CU_TENSOR_MAP_L2_PROMOTION_L2_128B;   // weight tiles
constexpr int DGRAD_SPLIT = 4;               // CTAs sharing an M-tile (each every 4th N-tile)
// The CTAs sharing an M-tile form one cluster (their dp partials meet in the leader's shared
// memory) when the experts are large; with small experts they form two clusters of 2, which fill
// all 152 SMs where clusters of 4 leave 8 idle (GPC packing), and the two cluster sums meet in dp.
// Measured at R = 262144, H = 3072, D = 3584: 896 experts of ~292 rows 8.03 ms (one cluster of 4)
// vs 7.25 ms (two of 2); 32 experts of 8192 rows 4.52 vs 4.73 ms.
constexpr int DGRAD_CLUSTER = 2;
constexpr int64_t CLUSTER4_MIN_ROWS = 4 * BM; // experts averaging at least this many rows: clusters of 4
static_assert(DGRAD_SPLIT / DGRAD_CLUSTER <= 2, "at most two dp contributions per row: a + b == b + a");
constexpr int MAX_SPLIT = DGRAD_SPLIT;       // largest cluster
// extra shared memory: dp_part [EPW][BM] | dp_cl [2][MAX_SPLIT][BM] | dp_full[2], dp_free[2]
constexpr int SMEM_BYTES = SMEM_FIXED_BYTES + 16 + EPW * BM * 4 + 2 * MAX_SPLIT * BM * 4 + 4 * 8;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
// dx leaves in per-thread 32-byte stores: staging it in shared memory for TMA tensor stores (as the
// gate/up epilogue does) was measured slower here, where the epilogue also has x loads in flight.

// ---------------------------------------------------------------- the kernel

// W_MN: the weights arrive as W_down,e [D, H] (the nn.Linear layout: N-major for this GEMM),
// loaded as four 64-column boxes per stage and read by the MMA with B transposed; otherwise as
// (W_down,e)ᵀ [H, D] (K-major), one 256-row box per stage.
template <bool BETA4, bool W_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    dgrad_bwd_kernel(const __grid_constant__ CUtensorMap map_dy, const __grid_constant__ CUtensorMap map_w,
                     const uint16_t* __restrict__ x, const int64_t* __restrict__ offsets, const float* __restrict__ p,
                     uint16_t* __restrict__ dx, float* __restrict__ dp, int* __restrict__ status, int E, int64_t R,
                     int64_t H, int KB, int csplit, int ncl, Coef c) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    Barriers* bars = sm.bars;
    float* dp_part = (float*)sm.extra;                               // [EPW][BM] per-warp-slot dp partials
    float* dp_cl = dp_part + EPW * BM;                               // [2][MAX_SPLIT][BM] cluster partials
    uint64_t* dp_full = (uint64_t*)(dp_cl + 2 * MAX_SPLIT * BM);     // [2] leader: partials of all ranks in
    uint64_t* dp_free = dp_full + 2;                                 // [2] other ranks: the leader read them
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (int)((H + BN - 1) / BN);  // the last N-tile may run past H: its extra columns are
                                              // computed (on the next expert's rows, or zeros past the
                                              // tensor) and never used
    const uint32_t crank = cluster_rank();

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&dp_full[b], (uint32_t)((ncl - 1) * BM));
            mbar_init(&dp_free[b], (uint32_t)BM);
        }
    }
    const Sched sc = make_sched(csplit);
    uint32_t tmem;
    const int T = pipeline_setup(sm, offsets, E, R, NUM_EPI_THREADS, &tmem);
    const int* tile_start = sm.tile_start;
    cluster_sync();                          // every CTA's barriers are initialised before any remote use

    if (warp == 0) {
        // ------------------------------------------------ TMA producer: B = W_downᵀ rows e·H + nt·256 ..
        if (lane == 0)
            run_producer(sm, sc, &map_dy, offsets, E, R, T, NT, KB, status,
                         [&](uint8_t* sb, int e, int nt, int kb, uint64_t* bar, uint64_t pol) {
                             if constexpr (W_MN) {
                                 // rows e·D + kb·64 .. of W_down,e, columns nt·256 + 64j ..
                                 const int r = (int)((int64_t)e * (KB * BK) + (int64_t)kb * BK);
#pragma unroll
                                 for (int j = 0; j < BN / 64; ++j)
                                     tma_load_2d_hint(sb + j * BMN_BOX_BYTES, &map_w, nt * BN + 64 * j, r, bar, pol);
                             } else {
                                 tma_load_2d_hint(sb, &map_w, kb * BK, (int)((int64_t)e * H + (int64_t)nt * BN),
                                                  bar, pol);
                             }
                         });
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) run_mma<W_MN>(sm, sc, tmem, T, NT, KB, status);
    } else {
        // ------------------------------------------------ epilogue (warps 2 .. 2 + 4·EPW − 1)
        // A warp may read only the TMEM lanes of quadrant warp % 4; the EPW warps of a quadrant take
        // a job's 16-column chunks in turn (slot s: chunks s, s + EPW, ...). One thread owns one row
        // for a whole M-tile: the x of its next chunk is fetched with 32-byte loads before the
        // current chunk is computed (also across job boundaries, as x does not depend on the
        // accumulator), so the loads are in flight while the previous chunk is computed and while
        // the next accumulator is awaited.
        const int quad = warp & 3;
        const int slot = (warp - 2) >> 2;
        const int lrow = quad * 32 + lane;         // row within the tile
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        int job = 0, it = 0;
        bool ok = true;
        for (int t = sc.t0; t < T; t += sc.tstep, ++it) {
            int e;
            int64_t row0, row_end;
            tile_rows(tile_start, offsets, E, R, t, e, row0, row_end);
            const int64_t row = row0 + lrow;
            const bool valid = ok && row >= 0 && row < row_end;
            const float pr16 = valid ? 16.0f * p[row] : 0.0f;
            const uint16_t* xr = x + (valid ? row : 0) * 2 * H;
            uint16_t* dxr = dx + (valid ? row : 0) * 2 * H;
            float acc_dp = 0.0f;
            Vec<8> xb[NBUF][2];                    // [buffer][gate, linear]
            const int64_t j1 = (int64_t)sc.n0 * BN + slot * CW;
            if (valid && j1 < H) {                 // first chunk: (first N-tile of this CTA, chunk slot)
                xb[0][0] = ld_stream<8, true>((const Vec<8>*)(xr + j1));
                xb[0][1] = ld_stream<8, true>((const Vec<8>*)(xr + H + j1));
            }
            for (int nt = sc.n0; nt < NT; nt += sc.nstep, ++job) {
                const int acc = job & 1;
                const uint32_t acc_phase = (uint32_t)((job >> 1) & 1);
                if (ok && !mbar_wait(&bars->tfull[acc], acc_phase, bars, status)) ok = false;
                ok = __all_sync(0xffffffffu, ok);                 // tcgen05.ld below is warp-collective
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < MAXC; ++i) {
                    const int kk = slot + i * EPW;                // this warp's i-th chunk of the job
                    if (kk < NCH) {
                        const int cur = i % NBUF;
                        const bool last = kk + EPW >= NCH;        // this warp's last chunk of the job
                        // prefetch the next chunk: (nt, kk + EPW), or (next N-tile, slot) after the last
                        if (last) {
                            const int64_t jn = (int64_t)(nt + sc.nstep) * BN + slot * CW;
                            if (valid && nt + sc.nstep < NT && jn < H) {
                                xb[0][0] = ld_stream<8, true>((const Vec<8>*)(xr + jn));
                                xb[0][1] = ld_stream<8, true>((const Vec<8>*)(xr + H + jn));
                            }
                        } else if (valid && (int64_t)nt * BN + (kk + EPW) * CW < H) {
                            const int64_t jn = (int64_t)nt * BN + (kk + EPW) * CW;
                            xb[(i + 1) % NBUF][0] = ld_stream<8, true>((const Vec<8>*)(xr + jn));
                            xb[(i + 1) % NBUF][1] = ld_stream<8, true>((const Vec<8>*)(xr + H + jn));
                        }
                        float gv[CW];
                        if (ok) tc_ld<CW>(tmem + t_lane + (uint32_t)(acc * BN + kk * CW), gv);
                        if (last) {
                            tc_fence_before();
                            mbar_arrive(&bars->tempty[acc]);     // accumulator may be overwritten
                        }
                        if (ok && valid && (int64_t)nt * BN + kk * CW < H) {   // whole chunks: H % 16 == 0
                            const int64_t j0 = (int64_t)nt * BN + kk * CW;
                            Vec<8> dgo, dlo;
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const uint32_t gw = xb[cur][0].w[q], lw = xb[cur][1].w[q];
                                const float g0 = gv[2 * q], g1 = gv[2 * q + 1];
                                situ::Bwd b0 = situ::bwd<BETA4>(bf16_lo(gw), bf16_lo(lw), pr16 * g0, c);
                                situ::Bwd b1 = situ::bwd<BETA4>(bf16_hi(gw), bf16_hi(lw), pr16 * g1, c);
                                acc_dp = fmaf(g0, b0.a16, acc_dp);
                                acc_dp = fmaf(g1, b1.a16, acc_dp);
                                dgo.w[q] = pack_bf16x2(b0.dgate, b1.dgate);
                                dlo.w[q] = pack_bf16x2(b0.dlin, b1.dlin);
                            }
                            st_stream<8>((Vec<8>*)(dxr + j0), dgo);
                            st_stream<8>((Vec<8>*)(dxr + H + j0), dlo);
                        }
                    }
                }
            }
            // combine the EPW column slices of each row, then the ncl CTAs of the cluster: every
            // rank pushes its partial into the leader's shared memory (double-buffered by M-tile
            // parity) and the leader adds them in rank order. When the csplit CTAs of the M-tile form
            // two clusters, each leader adds its cluster's sum into the zeroed dp with one
            // red.global.add: two addends commute exactly, so dp does not depend on timing either way
            if (slot > 0) dp_part[slot * BM + lrow] = acc_dp;
            epi_barrier(NUM_EPI_THREADS);
            if (slot == 0) {
                float s = acc_dp;
#pragma unroll
                for (int k = 1; k < EPW; ++k) s += dp_part[k * BM + lrow];
                if (ncl > 1) {
                    const int b = it & 1;
                    const uint32_t use_par = (uint32_t)((it >> 1) & 1);
                    if (crank != 0) {
                        if (it >= 2) mbar_wait_cluster(&dp_free[b], use_par ^ 1, bars, status);
                        st_cluster_f32(cluster_addr(&dp_cl[(b * MAX_SPLIT + (int)crank) * BM + lrow], 0), s);
                        mbar_arrive_cluster(cluster_addr(&dp_full[b], 0));
                    } else {
                        mbar_wait_cluster(&dp_full[b], use_par, bars, status);
                        for (int k = 1; k < ncl; ++k) s += dp_cl[(b * MAX_SPLIT + k) * BM + lrow];
                        for (int k = 1; k < ncl; ++k) mbar_arrive_cluster(cluster_addr(&dp_free[b], (uint32_t)k));
                    }
                }
                if (crank == 0 && valid) {
                    if (ncl < csplit) atomicAdd(&dp[row], 16.0f * s);
                    else dp[row] = 16.0f * s;
                }
            }
            epi_barrier(NUM_EPI_THREADS);
        }
    }

    cluster_sync();                          // no CTA leaves while another may still access its shared memory
    pipeline_teardown(tmem);
}

}  // namespace

namespace {

// Both entry points: w is (W_down,e)ᵀ [E, H, D] (w_mn false) or W_down,e [E, D, H] (w_mn true).
int dgrad_launch(const void* x, const void* dy, const void* w, bool w_mn, const int64_t* expert_offsets, int64_t E,
                 const float* p, void* dx, float* dp, int* status, int64_t R, int64_t H, int64_t D, float beta,
                 float lbeta, cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    // Any H % 16 == 0 (the epilogue's 16-column chunks are whole) and D % 8 == 0 (16-byte TMA row
    // strides): the last K-block reads zeros past D, the last N-tile computes columns past H that
    // are never used. The nn.Linear layout keeps D % 64 == 0: its K runs along the rows of
    // [E·D, H], so a K tail would read the next expert's rows instead of zeros.
    if (D <= 0 || D % 8 != 0 || H % 16 != 0 || E < 1 || E > MAX_EXPERTS) return SITU_GLU_INVALID_ARG;
    if (w_mn && D % BK != 0) return SITU_GLU_INVALID_ARG;
    if (R > INT32_MAX || E * H > INT32_MAX - BN || E * D > INT32_MAX || D > INT32_MAX / 2) return SITU_GLU_INVALID_ARG;
    if (R == 0) return SITU_GLU_OK;
    if (!x || !dy || !w || !expert_offsets || !p || !dx || !dp) return SITU_GLU_INVALID_ARG;
    if (!aligned(x, 32) || !aligned(dy, 16) || !aligned(w, 16) || !aligned(dx, 32) ||
        !aligned(expert_offsets, 8) || !aligned(p, 4) || !aligned(dp, 4) || (status && !aligned(status, 4)))
        return SITU_GLU_INVALID_ARG;
    const Range rx = range_of(x, R * 2 * H * 2), ry = range_of(dy, R * D * 2), rw = range_of(w, E * H * D * 2);
    const Range ro = range_of(expert_offsets, (E + 1) * 8), rp = range_of(p, R * 4);
    const Range rdx = range_of(dx, R * 2 * H * 2), rdp = range_of(dp, R * 4);
    for (Range in : {rx, ry, rw, ro, rp}) {
        if (overlap(rdx, in) || overlap(rdp, in)) return SITU_GLU_OVERLAP;
        if (status && overlap(range_of(status, 4), in)) return SITU_GLU_OVERLAP;
    }
    if (overlap(rdx, rdp)) return SITU_GLU_OVERLAP;
    if (status && (overlap(range_of(status, 4), rdx) || overlap(range_of(status, 4), rdp))) return SITU_GLU_OVERLAP;

    CUtensorMap map_dy, map_w;
    if (!make_map(&map_dy, dy, (uint64_t)R, (uint64_t)D, BM, BK, true, DGRAD_L2_PROMO_A))
        return cuda_fail(cudaErrorInvalidValue);
    const bool mw = w_mn ? make_map(&map_w, w, (uint64_t)(E * D), (uint64_t)H, BK, 64, true,   // 64 K rows x 64 N
                                    DGRAD_L2_PROMO_B)
                         : make_map(&map_w, w, (uint64_t)(E * H), (uint64_t)D, BN, BK, true,   // 256 N rows x 64 K
                                    DGRAD_L2_PROMO_B);
    if (!mw) return cuda_fail(cudaErrorInvalidValue);

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    auto kernel = b4 ? (w_mn ? dgrad_bwd_kernel<true, true> : dgrad_bwd_kernel<true, false>)
                     : (w_mn ? dgrad_bwd_kernel<false, true> : dgrad_bwd_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(e);
    const int NT = (int)((H + BN - 1) / BN);
    const int csplit = NT < DGRAD_SPLIT ? NT : DGRAD_SPLIT;
    const int ncl = (csplit % DGRAD_CLUSTER != 0 || R / E >= CLUSTER4_MIN_ROWS) ? csplit : DGRAD_CLUSTER;
    if (ncl < csplit) {                      // two clusters per M-tile add into dp
        e = cudaMemsetAsync(dp, 0, (size_t)R * 4, stream);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    e = launch_clusters(kernel, R, E, ncl, csplit, NUM_THREADS, SMEM_BYTES, stream, map_dy, map_w,
                        (const uint16_t*)x, expert_offsets, p, (uint16_t*)dx, dp, status, (int)E, R, H,
                        (int)((D + BK - 1) / BK), csplit, ncl, c);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // namespace

extern "C" {

int situ_glu_bwd_router_dgrad(const void* x, const void* dy, const void* w_down_t, const int64_t* expert_offsets,
                              int64_t E, const float* p, void* dx, float* dp, int* status, int64_t R, int64_t H,
                              int64_t D, float beta, float lbeta, cudaStream_t stream) {
    return dgrad_launch(x, dy, w_down_t, false, expert_offsets, E, p, dx, dp, status, R, H, D, beta, lbeta, stream);
}

int situ_glu_bwd_router_dgrad_wd(const void* x, const void* dy, const void* w_down, const int64_t* expert_offsets,
                                 int64_t E, const float* p, void* dx, float* dp, int* status, int64_t R, int64_t H,
                                 int64_t D, float beta, float lbeta, cudaStream_t stream) {
    return dgrad_launch(x, dy, w_down, true, expert_offsets, E, p, dx, dp, status, R, H, D, beta, lbeta, stream);
}

}  // extern "C"
