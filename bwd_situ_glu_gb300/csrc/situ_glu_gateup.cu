// situ_glu_gateup.cu — gate/up projection grouped GEMM on the 5th-generation tensor cores
// (tcgen05, TMA, TMEM), with the SiTU-GLU forward fused into its epilogue.
//
// "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出": a routed
// row of expert e computes a_e = SiTU(W_gate,e·h, W_up,e·h) from its dispatched input h.
// "Frontier-scale RL with Kimi K3", section "Streaming activations": the backward keeps only the
// bf16 pre-activation x = [W_gate,e·h | W_up,e·h]; the forward reads x and writes a in bf16.
// This kernel computes both projections of a row on the tensor cores and, from the fp32
// accumulators, writes the bf16 x that the backward will read and out = a computed from that
// same bf16 x, so the result equals the unfused projection followed by situ_glu_fwd, with one
// fewer round trip of x through memory.
//
// The GEMM pipeline is the one in situ_tc.cuh — for experts of many rows its two-M-tile form, in
// which two M-tiles of one expert share every weight stage (chosen per launch from the mean rows
// per expert) — with A = h and a B tile made of two 128-row halves: rows nt·128 .. of W_gate,e
// and the same rows of W_up,e, so accumulator column c < 128 holds gate column nt·128 + c and
// column 128 + c the matching linear column. Epilogue: EPW warps
// per 32-lane TMEM quadrant, each owning 128/EPW of a job's 128 column pairs; a thread owns one
// row, reads 32 gate and 32 linear accumulators per chunk, rounds them to bf16 (nearest even),
// evaluates the forward on the rounded values and writes x (both halves) and out with 32-byte
// stores.
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

constexpr int HN = BN / 2;                   // column pairs per job (128 gate + 128 linear columns)
constexpr int EPW = 2;                       // epilogue warps per 32-lane TMEM quadrant
constexpr int CW = 16;                       // column pairs per chunk
constexpr int NUM_EPI_THREADS = 4 * EPW * 32;
constexpr int NUM_THREADS = 64 + NUM_EPI_THREADS;  // warp 0 TMA, warp 1 MMA, then the epilogue
constexpr int PAIRS_PER_WARP = HN / EPW;
constexpr int CPJ = PAIRS_PER_WARP / CW;     // chunks per job per epilogue warp
static_assert(CPJ >= 1 && PAIRS_PER_WARP % CW == 0, "whole chunks per warp");
constexpr int STAGE_TILE = 32 * CW * 2;      // one 32-row x CW-column bf16 output tile in shared memory
constexpr int STAGE_BYTES_EPI = 4 * EPW * 3 * STAGE_TILE;   // [warp][x gate, x linear, out]
constexpr int SMEM_BYTES = SMEM_FIXED_BYTES + 128 + STAGE_BYTES_EPI;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr int CSPLIT = 8;                    // CTAs sharing an M-tile (each every 8th N-tile)

// UNIT = M-tiles per work unit: 1 (two double-buffered accumulators, the next job's MMAs overlap
// this job's epilogue) or 2 (two M-tiles share every weight stage, a third fewer bytes per MMA
// flop, no overlap). The host picks 2 when experts average at least UNIT2_MIN_ROWS rows.
constexpr int64_t UNIT2_MIN_ROWS = 4 * BM;

template <bool BETA4, int UNIT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gateup_fwd_kernel(const __grid_constant__ CUtensorMap map_h, const __grid_constant__ CUtensorMap map_w,
                      const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_out,
                      const int64_t* __restrict__ offsets, uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                      int* __restrict__ status, int E, int64_t R, int64_t H, int KB, int csplit, Coef c) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve_smem(smem_raw);
    Barriers* bars = sm.bars;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = (int)((H + HN - 1) / HN);   // the last N-tile may run past H: the weight rows past
                                               // H read as zeros, those columns are never stored

    const Sched sc = make_sched(csplit);
    uint32_t tmem;
    const int T = pipeline_setup(sm, offsets, E, R, NUM_EPI_THREADS, &tmem, UNIT);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer: B = W_gate,e and W_up,e rows nt·128 ..
        // one 3-D box: K-block kb of rows nt·128 .. of W_gate,e (plane 2e) and of W_up,e (plane 2e + 1)
        auto load_b = [&](uint8_t* sb, int e, int nt, int kb, uint64_t* bar, uint64_t pol) {
            tma_load_3d_hint(sb, &map_w, kb * BK, nt * HN, 2 * e, bar, pol);
        };
        if (lane == 0) {
            if constexpr (UNIT == 2)
                run_producer2(sm, sc, &map_h, offsets, E, R, T, NT, KB, status, load_b);
            else
                run_producer(sm, sc, &map_h, offsets, E, R, T, NT, KB, status, load_b);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            if constexpr (UNIT == 2)
                run_mma2(sm, sc, tmem, offsets, E, R, T, NT, KB, status);
            else
                run_mma(sm, sc, tmem, T, NT, KB, status);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2 .. 2 + 4·EPW − 1)
        const int quad = warp & 3;
        const int slot = (warp - 2) >> 2;
        const int lrow = quad * 32 + lane;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        uint8_t* stage = (uint8_t*)(((uintptr_t)sm.extra + 127) & ~(uintptr_t)127);
        uint8_t* st_g = stage + (warp - 2) * 3 * STAGE_TILE;   // this warp's x gate, x linear, out tiles
        uint8_t* st_l = st_g + STAGE_TILE;
        uint8_t* st_o = st_l + STAGE_TILE;
        bool stores_pending = false;                            // lane 0 has TMA stores in flight
        int job = 0;
        bool ok = true;
        for (int u = sc.t0; u < T; u += sc.tstep) {
            int e, ntiles = 1;
            int64_t urow0, row_end;
            if constexpr (UNIT == 2)
                unit2_rows(sm.tile_start, offsets, E, R, u, e, urow0, row_end, ntiles);
            else
                tile_rows(sm.tile_start, offsets, E, R, u, e, urow0, row_end);
            for (int nt = sc.n0; nt < NT; nt += sc.nstep, ++job) {
                // UNIT 1: accumulator job & 1 through barrier pair job & 1; UNIT 2: both, through pair 0
                const int bi = UNIT == 2 ? 0 : (job & 1);
                const uint32_t par = UNIT == 2 ? (uint32_t)(job & 1) : (uint32_t)((job >> 1) & 1);
                if (ok && !mbar_wait(&bars->tfull[bi], par, bars, status)) ok = false;
                ok = __all_sync(0xffffffffu, ok);                 // tcgen05.ld below is warp-collective
                tc_fence_after();
                for (int m = 0; m < ntiles; ++m) {               // the unit's M-tiles
                    const int acc_col = UNIT == 2 ? m * BN : bi * BN;
                    const int64_t row0 = urow0 + (int64_t)m * BM;
                    const int64_t row = row0 + lrow;
                    const bool valid = ok && row >= 0 && row < row_end;
                    // all 32 rows of this warp's quadrant belong to the expert: x and out leave through TMA stores
                    const bool full_quad = row0 + quad * 32 + 31 < row_end;
                    uint16_t* xr = x + (valid ? row : 0) * 2 * H + slot * PAIRS_PER_WARP;
                    uint16_t* outr = out + (valid ? row : 0) * H + slot * PAIRS_PER_WARP;
#pragma unroll
                    for (int k = 0; k < CPJ; ++k) {
                        uint32_t gr[CW], lr[CW];
                        if (ok) {
                            const uint32_t col = (uint32_t)(acc_col + slot * PAIRS_PER_WARP + k * CW);
                            tc_ld_issue<CW>(tmem + t_lane + col, gr);
                            tc_ld_issue<CW>(tmem + t_lane + col + HN, lr);
                            tc_wait_ld();
                        }
                        if (m + 1 == ntiles && k + 1 == CPJ) {
                            tc_fence_before();
                            mbar_arrive(&bars->tempty[bi]);      // the job's accumulators may be overwritten
                        }
                        static_assert(CW == 16, "one 32-byte vector per output row per chunk");
                        // whole 16-column chunks (H % 16 == 0): a chunk past H is not evaluated or stored
                        const bool chunk_ok = (int64_t)nt * HN + k * CW + slot * PAIRS_PER_WARP < H;
                        Vec<8> xg, xl, o;
                        if (ok && valid && chunk_ok) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                xg.w[i] = pack_bf16x2(__uint_as_float(gr[2 * i]), __uint_as_float(gr[2 * i + 1]));
                                xl.w[i] = pack_bf16x2(__uint_as_float(lr[2 * i]), __uint_as_float(lr[2 * i + 1]));
                                const float a0 = situ::fwd<BETA4>(bf16_lo(xg.w[i]), bf16_lo(xl.w[i]), c);
                                const float a1 = situ::fwd<BETA4>(bf16_hi(xg.w[i]), bf16_hi(xl.w[i]), c);
                                o.w[i] = pack_bf16x2(a0, a1);
                            }
                        }
                        const int64_t jl = (int64_t)nt * HN + k * CW;                        // within the slice
                        const int64_t j0 = jl + slot * PAIRS_PER_WARP;                       // column in [0, H)
                        if (ok && full_quad && chunk_ok) {
                            // the warp's 32 rows x CW columns of x (both halves) and of out: staged, then
                            // one TMA store each
                            if (stores_pending) {
                                if (lane == 0) bulk_wait_read_all();     // the previous tiles have been read out
                                __syncwarp();
                            }
                            st_shared_v4(st_g + lane * 32, xg.w[0], xg.w[1], xg.w[2], xg.w[3]);
                            st_shared_v4(st_g + lane * 32 + 16, xg.w[4], xg.w[5], xg.w[6], xg.w[7]);
                            st_shared_v4(st_l + lane * 32, xl.w[0], xl.w[1], xl.w[2], xl.w[3]);
                            st_shared_v4(st_l + lane * 32 + 16, xl.w[4], xl.w[5], xl.w[6], xl.w[7]);
                            st_shared_v4(st_o + lane * 32, o.w[0], o.w[1], o.w[2], o.w[3]);
                            st_shared_v4(st_o + lane * 32 + 16, o.w[4], o.w[5], o.w[6], o.w[7]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int r0q = (int)(row0 + quad * 32);
                                tma_store_2d(&map_x, (int)j0, r0q, st_g);
                                tma_store_2d(&map_x, (int)(H + j0), r0q, st_l);
                                tma_store_2d(&map_out, (int)j0, r0q, st_o);
                                bulk_commit();
                            }
                            stores_pending = true;
                        } else if (ok && valid && chunk_ok) {
                            // a quadrant crossing the expert's end: only this row, from registers
                            st_stream<8>((Vec<8>*)(xr + jl), xg);
                            st_stream<8>((Vec<8>*)(xr + H + jl), xl);
                            st_stream<8>((Vec<8>*)(outr + jl), o);
                        }
                    }
                }
            }
        }
        if (lane == 0 && stores_pending) bulk_wait_all();           // every x and out tile written
    }

    pipeline_teardown(tmem);
}

}  // namespace

extern "C" {

int situ_glu_fwd_gateup(const void* h, const void* w_gate_up, const int64_t* expert_offsets, int64_t E, void* x,
                        void* out, int* status, int64_t R, int64_t H, int64_t D, float beta, float lbeta,
                        cudaStream_t stream) {
    int st = check_shape(R, H, beta, lbeta);
    if (st != SITU_GLU_OK) return st;
    // Any H % 16 == 0 (whole 16-column epilogue chunks) and D % 8 == 0 (16-byte TMA row strides): the
    // last K-block reads zeros past D, the last N-tile reads zero weight rows past H.
    if (D <= 0 || D % 8 != 0 || H % 16 != 0 || E < 1 || E > MAX_EXPERTS) return SITU_GLU_INVALID_ARG;
    if (R > INT32_MAX || E * 2 * H > INT32_MAX || D > INT32_MAX / 2) return SITU_GLU_INVALID_ARG;
    if (R == 0) return SITU_GLU_OK;
    if (!h || !w_gate_up || !expert_offsets || !x || !out) return SITU_GLU_INVALID_ARG;
    if (!aligned(h, 16) || !aligned(w_gate_up, 16) || !aligned(x, 32) || !aligned(out, 32) ||
        !aligned(expert_offsets, 8) || (status && !aligned(status, 4)))
        return SITU_GLU_INVALID_ARG;
    const Range rh = range_of(h, R * D * 2), rw = range_of(w_gate_up, E * 2 * H * D * 2);
    const Range ro = range_of(expert_offsets, (E + 1) * 8);
    const Range rx = range_of(x, R * 2 * H * 2), rout = range_of(out, R * H * 2);
    for (Range in : {rh, rw, ro}) {
        if (overlap(rx, in) || overlap(rout, in)) return SITU_GLU_OVERLAP;
        if (status && overlap(range_of(status, 4), in)) return SITU_GLU_OVERLAP;
    }
    if (overlap(rx, rout)) return SITU_GLU_OVERLAP;
    if (status && (overlap(range_of(status, 4), rx) || overlap(range_of(status, 4), rout))) return SITU_GLU_OVERLAP;

    CUtensorMap map_h, map_w;
    if (!make_map(&map_h, h, (uint64_t)R, (uint64_t)D, BM)) return cuda_fail(cudaErrorInvalidValue);
    // [W_gate,e; W_up,e] as 2E planes of [H, D]: one box brings 128 rows of both halves (one TMA
    // instruction per weight tile instead of two; 256-byte L2 promotion, which the dgrad's weight
    // tiles measured slower with, is neutral to slightly better here)
    if (!make_map_3d(&map_w, w_gate_up, (uint64_t)D, (uint64_t)H, (uint64_t)(2 * E), (uint64_t)D * 2,
                     (uint64_t)(H * D * 2), BK, HN, 2))
        return cuda_fail(cudaErrorInvalidValue);
    CUtensorMap map_x, map_out;
    if (!make_map(&map_x, x, (uint64_t)R, (uint64_t)(2 * H), 32, CW, false)) return cuda_fail(cudaErrorInvalidValue);
    if (!make_map(&map_out, out, (uint64_t)R, (uint64_t)H, 32, CW, false)) return cuda_fail(cudaErrorInvalidValue);

    const Coef c = make_coef(beta, lbeta);
    const bool b4 = fast_path(beta, lbeta);
    const bool unit2 = R / E >= UNIT2_MIN_ROWS;
    auto kernel = b4 ? (unit2 ? gateup_fwd_kernel<true, 2> : gateup_fwd_kernel<true, 1>)
                     : (unit2 ? gateup_fwd_kernel<false, 2> : gateup_fwd_kernel<false, 1>);
    cudaError_t e = cudaFuncSetAttribute((const void*)kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(e);
    const int NT = (int)((H + HN - 1) / HN);
    const int csplit = NT < CSPLIT ? NT : CSPLIT;
    int grid = 0;
    if ((e = (cudaError_t)persistent_grid(R, E, csplit, &grid)) != cudaSuccess) return cuda_fail(e);
    kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(map_h, map_w, map_x, map_out, expert_offsets, (uint16_t*)x,
                                                      (uint16_t*)out,
                                                      status, (int)E, R, H, (int)((D + BK - 1) / BK), csplit, c);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    return SITU_GLU_OK;
}

}  // extern "C"
