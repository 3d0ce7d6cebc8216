// situ_tc.cuh — the expert-grouped GEMM pipeline on the 5th-generation tensor cores (tcgen05,
// TMA, TMEM, mbarriers) shared by the two fused kernels: the down-projection dgrad with the
// SiTU-GLU backward in its epilogue, and the gate/up projection with the SiTU-GLU forward in its
// epilogue. Each kernel supplies only its B-tile loads and its epilogue.
//
// Problem: rows are grouped by expert (expert e owns rows offsets[e] .. offsets[e+1]-1); for every
// row r of expert e and output column n, C[r, n] = Σ_k A[r, k]·B_e[n, k] with A and B_e bf16 and
// K-major (k contiguous), C accumulated in fp32.
//
// Work decomposition: an M-tile is 128 consecutive rows of ONE expert (an expert with n rows has
// ceil(n/128) M-tiles; the last one is partial and the epilogue skips the rows past the expert's
// end). A job is one M-tile times one 256-column N-tile. CTAs are persistent (one per SM); a
// group of CSPLIT consecutive CTAs takes M-tiles g, g + groups, ... and its k-th CTA the N-tiles
// k, k + CSPLIT, ... of each (see Sched).
//
// Per-CTA roles:
//   warp 0, one thread   TMA producer: per 64-wide K-block, A [128 x 64] and B [256 x 64] (bf16,
//                        128-byte swizzle) into a STAGES-deep shared-memory ring, completion
//                        signalled on the stage's "full" mbarrier (transaction bytes);
//   warp 1               allocates 512 TMEM columns (two 128 x 256 fp32 accumulators); one thread
//                        issues tcgen05.mma (M = 128, N = 256, K = 16) and commits to mbarriers
//                        that free ring stages ("empty") and hand accumulators to the epilogue
//                        ("tfull"); the epilogue hands them back through "tempty";
//   warps 2 ..           the kernel's epilogue.
// Every wait is bounded (2 s by %globaltimer, or WAIT_LIMIT polls): on a timeout the CTA sets its
// abort flag and the caller's status word, stops issuing work, waits (bounded) for what it
// already issued, frees its TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace situ_tc {

constexpr int BM = 128;                      // rows per M-tile (TMEM lanes)
constexpr int BN = 256;                      // accumulator columns per job
constexpr int BK = 64;                       // K per ring stage (128 bytes of bf16: one swizzle row)
constexpr int UK = 16;                       // K per tcgen05.mma (kind::f16)
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BYTES = BN * BK * 2;         // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;               // 2 accumulators x 256 columns
constexpr int MAX_EXPERTS = 1024;           // the per-CTA tile prefix lives in shared memory
constexpr uint64_t WAIT_NS = 2000000000ull;  // a pipeline wait gives up after 2 s (%globaltimer)
constexpr uint32_t WAIT_LIMIT = 1u << 24;    // and in any case after this many polls

struct alignas(8) Barriers {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};

// Dynamic shared memory: [pad to 1024] ring | Barriers | tile_start[MAX_EXPERTS + 1] | extra.
constexpr int SMEM_FIXED_BYTES = 1024 + STAGES * STAGE_BYTES + (int)sizeof(Barriers) + (MAX_EXPERTS + 1) * 4;

struct Smem {
    uint8_t* ring;
    Barriers* bars;
    int* tile_start;
    uint8_t* extra;     // 16-byte aligned kernel-specific area
};

__device__ __forceinline__ Smem carve_smem(uint8_t* raw) {
    Smem s;
    s.ring = (uint8_t*)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    s.bars = (Barriers*)(s.ring + STAGES * STAGE_BYTES);
    s.tile_start = (int*)(s.bars + 1);
    s.extra = (uint8_t*)(((uintptr_t)(s.tile_start + MAX_EXPERTS + 1) + 15) & ~(uintptr_t)15);
    return s;
}

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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait; on a timeout (WAIT_NS, or WAIT_LIMIT polls) sets the CTA's abort flag and the
// caller's status word. Returns early, false, once another role of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, Barriers* bars, int* status) {
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(b, parity)) return true;
        if ((i & 63) == 63) {
            if (*(volatile int*)&bars->abort) return false;
            if (global_ns() - t0 > WAIT_NS) break;
        }
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

// The same with an L2 eviction-priority policy (from make_policy) for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 3-D box load (dims innermost first) with an L2 eviction-priority policy.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

enum class L2Hint { normal, first, last };

template <L2Hint P>
__device__ __forceinline__ uint64_t make_policy() {
    uint64_t pol;
    if constexpr (P == L2Hint::last)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else if constexpr (P == L2Hint::first)
        asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// L2 priorities of the two operands: the A tile (activations, re-read once per N-tile) and the
// B tiles (weights, re-read by every M-tile of their expert). Weights evict-last measured 1-3 %
// faster for both kernels at 896 x ~292 and 32 x 8192 rows (same calls, two rounds each); A
// evict-first was 5-15 % slower, A evict-last mixed.
constexpr L2Hint kHintA = L2Hint::normal;
constexpr L2Hint kHintB = L2Hint::last;

// ---------------------------------------------------------------- TMA stores (epilogue output tiles)

// Order this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Store a box of a 2-D tensor map from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(c0),
                 "r"(c1), "r"(smem_addr(src))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the committed bulk stores of this thread have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until the committed bulk stores of this thread are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_addr(p)), "r"(a), "r"(b), "r"(c), "r"(d)
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

// The same with B stored N-major ("MN-major": bit 16, transpose B).
constexpr uint32_t IDESC_BMN = IDESC | (1u << 16);

// Shared-memory descriptor of an N-major bf16 B tile with 128-byte swizzle, as written by TMA
// boxes of 64 N-elements x 64 K-rows: each K row of a box is 128 bytes (64 consecutive N), 8 K
// rows form a 1024-byte swizzle atom (stride byte offset), and the next 64 N-elements start one
// box (8 KB) further on (leading byte offset).
constexpr uint32_t BMN_BOX_BYTES = 64 * BK * 2;
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((BMN_BOX_BYTES >> 4) & 0x3FFFu) << 16;   // leading byte offset: next 64 N
    d |= (uint64_t)(1024 >> 4) << 32;                         // stride byte offset: next 8 K rows
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

template <bool B_MN = false>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(B_MN ? IDESC_BMN : IDESC), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

// Issue a load of N consecutive fp32 columns (N = 16 or 32) of this thread's TMEM lane; the
// registers are valid after tc_wait_ld().
template <int N>
__device__ __forceinline__ void tc_ld_issue(uint32_t taddr, uint32_t (&r)[N]) {
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
}

__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// N consecutive fp32 columns of this thread's TMEM lane, waited for.
template <int N>
__device__ __forceinline__ void tc_ld(uint32_t taddr, float (&v)[N]) {
    uint32_t r[N];
    tc_ld_issue<N>(taddr, r);
    tc_wait_ld();
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- thread-block clusters

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster; orders shared-memory accesses across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of this CTA's shared variable p in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t caddr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(caddr), "f"(v) : "memory");
}

// Arrive (release at cluster scope) on an mbarrier of any CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// Bounded wait for the completion of work this CTA already issued (its own loads and MMAs), at the
// end of a run or after an abort: no status, since that work completes by itself.
__device__ __forceinline__ void mbar_drain(uint64_t* b, uint32_t parity) {
    if (mbar_try_wait(b, parity)) return;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        if (mbar_try_wait(b, parity)) return;
        if ((i & 63) == 63 && global_ns() - t0 > WAIT_NS) return;
    }
}

// Bounded wait with acquire at cluster scope (data written by other CTAs of the cluster before
// their arrive is visible afterwards); on a timeout sets the abort flag and the status word.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* b, uint32_t parity, Barriers* bars, int* status) {
    uint64_t t0 = 0;
    for (uint32_t i = 0; i < WAIT_LIMIT; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(smem_addr(b)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (i == 0) t0 = global_ns();
        if ((i & 63) == 63) {
            if (*(volatile int*)&bars->abort) return false;
            if (global_ns() - t0 > WAIT_NS) break;
        }
    }
    *(volatile int*)&bars->abort = 1;
    if (status) atomicExch(status, 1);
    return false;
}

// Named barrier over the epilogue warps only (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void epi_barrier(int nthreads) { asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory"); }

// Expert e's rows as [begin, end) clamped into [0, R] (end >= begin): malformed offsets can
// neither index outside the row range nor inflate the number of tiles beyond R/BM + E.
__device__ __forceinline__ void expert_range(const int64_t* off, int e, int64_t R, int64_t& begin, int64_t& end) {
    int64_t a = off[e], b = off[e + 1];
    a = a < 0 ? 0 : (a > R ? R : a);
    b = b < a ? a : (b > R ? R : b);
    begin = a;
    end = b;
}

// M-tile t -> (expert, first row, end row of the expert).
__device__ __forceinline__ void tile_rows(const int* tile_start, const int64_t* off, int E, int64_t R, int t,
                                          int& e, int64_t& row0, int64_t& row_end) {
    int lo = 0, hi = E - 1;                 // last e with tile_start[e] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    e = lo;
    int64_t begin;
    expert_range(off, e, R, begin, row_end);
    row0 = begin + (int64_t)(t - tile_start[e]) * BM;
}

// ---------------------------------------------------------------- work assignment

// CSPLIT consecutive CTAs share each M-tile, CTA rank k taking N-tiles k, k + CSPLIT, ...: at any
// moment only gridDim.x / CSPLIT distinct A tiles (128 rows x K) are being streamed, so each one
// stays in L2 across the N-tiles that re-read it. gridDim.x is a multiple of CSPLIT.
struct Sched {
    int t0, tstep;      // M-tiles t0, t0 + tstep, ...
    int n0, nstep;      // N-tiles n0, n0 + nstep, ... of each M-tile
};

__device__ __forceinline__ Sched make_sched(int csplit) {
    Sched s;
    s.t0 = (int)blockIdx.x / csplit;
    s.tstep = (int)gridDim.x / csplit;
    s.n0 = (int)blockIdx.x % csplit;
    s.nstep = csplit;
    return s;
}

// Work unit u of two M-tiles -> (expert, first row, end row of the expert, M-tiles in the unit:
// 2, or 1 for the last unit of an expert with an odd number of M-tiles).
__device__ __forceinline__ void unit2_rows(const int* unit_start, const int64_t* off, int E, int64_t R, int u,
                                           int& e, int64_t& row0, int64_t& row_end, int& ntiles) {
    int lo = 0, hi = E - 1;                 // last e with unit_start[e] <= u
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit_start[mid] <= u) lo = mid; else hi = mid - 1;
    }
    e = lo;
    int64_t begin;
    expert_range(off, e, R, begin, row_end);
    row0 = begin + (int64_t)(u - unit_start[e]) * 2 * BM;
    ntiles = row_end - row0 > BM ? 2 : 1;
}

// ---------------------------------------------------------------- pipeline phases

// All threads: per-expert prefix of work units of unit_tiles M-tiles each (each CTA builds its own
// copy: counts in parallel, then one warp scans them, each lane a contiguous segment, shuffles
// across lanes), barrier init, TMEM allocation by warp 1. Returns the number of units; *tmem
// receives the TMEM base address.
__device__ __forceinline__ int pipeline_setup(const Smem& sm, const int64_t* offsets, int E, int64_t R,
                                              int num_epi_threads, uint32_t* tmem, int unit_tiles = 1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Barriers* bars = sm.bars;
    int* tile_start = sm.tile_start;             // per expert: its first work unit
    const int64_t unit_rows = (int64_t)unit_tiles * BM;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int64_t begin, end;
        expert_range(offsets, e, R, begin, end);
        tile_start[e + 1] = (int)((end - begin + unit_rows - 1) / unit_rows);
    }
    if (threadIdx.x == 0) {
        tile_start[0] = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&bars->tfull[a], 1);
            mbar_init(&bars->tempty[a], (uint32_t)num_epi_threads);
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
    *tmem = bars->tmem_base;
    return tile_start[E];
}

// One thread of warp 0. load_b(b_smem, e, nt, kb, bar, policy) issues the B-tile TMA loads
// (B_BYTES in total) of expert e, N-tile nt, K-block kb; A comes from map_a at (kb·BK, row0).
template <class LoadB>
__device__ __forceinline__ void run_producer(const Smem& sm, const Sched& sc, const CUtensorMap* map_a,
                                             const int64_t* offsets, int E, int64_t R, int T, int NT, int KB,
                                             int* status, LoadB load_b) {
    Barriers* bars = sm.bars;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0;            // bit s: stage s has a load in flight of parity pend_par
    uint32_t pend_par = 0;
    const uint64_t pol_a = make_policy<kHintA>(), pol_b = make_policy<kHintB>();
    bool ok = true;
    for (int t = sc.t0; ok && t < T; t += sc.tstep) {
        int e;
        int64_t row0, row_end;
        tile_rows(sm.tile_start, offsets, E, R, t, e, row0, row_end);
        for (int nt = sc.n0; ok && nt < NT; nt += sc.nstep) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!mbar_wait(&bars->empty[stage], phase ^ 1, bars, status)) { ok = false; break; }
                mbar_expect_tx(&bars->full[stage], STAGE_BYTES);
                uint8_t* sa = sm.ring + stage * STAGE_BYTES;
                tma_load_2d_hint(sa, map_a, kb * BK, (int)row0, &bars->full[stage], pol_a);
                load_b(sa + A_BYTES, e, nt, kb, &bars->full[stage], pol_b);
                pending |= 1u << stage;
                pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
        }
    }
    // every load issued must land before the CTA exits: wait for each stage's last phase
    for (int s2 = 0; s2 < STAGES; ++s2) {
        if (!(pending & (1u << s2))) continue;
        mbar_drain(&bars->full[s2], (pend_par >> s2) & 1u);
    }
}

// One thread of warp 1: the MMA issuer. B_MN: the B tile is N-major (four 64-column TMA boxes).
template <bool B_MN = false>
__device__ __forceinline__ void run_mma(const Smem& sm, const Sched& sc, uint32_t tmem, int T, int NT, int KB,
                                        int* status) {
    Barriers* bars = sm.bars;
    int stage = 0;
    uint32_t phase = 0;
    int job = 0;
    bool ok = true;
    for (int t = sc.t0; ok && t < T; t += sc.tstep) {
        for (int nt = sc.n0; ok && nt < NT; nt += sc.nstep, ++job) {
            const int acc = job & 1;
            const uint32_t acc_phase = (uint32_t)((job >> 1) & 1);
            if (!mbar_wait(&bars->tempty[acc], acc_phase ^ 1, bars, status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < KB; ++kb) {
                if (!mbar_wait(&bars->full[stage], phase, bars, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_addr(sm.ring + stage * STAGE_BYTES);
                const uint64_t adesc = smem_desc(sa);
                const uint64_t bdesc = B_MN ? smem_desc_mn(sa + A_BYTES) : smem_desc(sa + A_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / UK; ++kk) {
                    // A (K-major): advance 16 bf16 = 32 bytes (2 descriptor units) inside the swizzled
                    // rows; B N-major: advance 16 K rows = 2048 bytes (128 units) to the next two atoms
                    const uint64_t bk = B_MN ? (uint64_t)(kk * 128) : (uint64_t)(kk * 2);
                    tc_mma<B_MN>(d_tmem, adesc + (uint64_t)(kk * 2), bdesc + bk, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&bars->empty[stage]);          // ring stage free once these MMAs finish
                if (++stage == STAGES) { stage = 0; phase ^= 1; }
            }
            if (ok) tc_commit(&bars->tfull[acc]);        // accumulator complete
        }
    }
    // all MMAs issued by this thread complete before TMEM is freed
    tc_commit(&bars->mma_done);
    mbar_drain(&bars->mma_done, 0);
}

// ---------------------------------------------------------------- units of two M-tiles

// A unit of two M-tiles of one expert shares each B (weight) stage between two MMAs into two
// accumulators: a stage holds A0 | A1 | B (64 KB, STAGES2 of them in the same ring memory), a
// third fewer bytes per MMA flop than one M-tile per stage, so the same shared memory covers 1.5x
// the MMA time. Both TMEM accumulators belong to the unit's job (columns 0..255: the first M-tile,
// 256..511: the second), so the epilogue of a job is not overlapped with the next job's MMAs.
constexpr int STAGES2 = 3;
constexpr int STAGE_BYTES2 = 2 * A_BYTES + B_BYTES;
static_assert(STAGES2 * STAGE_BYTES2 <= STAGES * STAGE_BYTES, "the two-tile ring fits the ring memory");
static_assert(STAGES2 <= STAGES, "stage barriers");

template <class LoadB>
__device__ __forceinline__ void run_producer2(const Smem& sm, const Sched& sc, const CUtensorMap* map_a,
                                              const int64_t* offsets, int E, int64_t R, int T, int NT, int KB,
                                              int* status, LoadB load_b) {
    Barriers* bars = sm.bars;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;
    const uint64_t pol_a = make_policy<kHintA>(), pol_b = make_policy<kHintB>();
    bool ok = true;
    for (int u = sc.t0; ok && u < T; u += sc.tstep) {
        int e, ntiles;
        int64_t row0, row_end;
        unit2_rows(sm.tile_start, offsets, E, R, u, e, row0, row_end, ntiles);
        const uint32_t bytes = (uint32_t)(ntiles * A_BYTES + B_BYTES);
        for (int nt = sc.n0; ok && nt < NT; nt += sc.nstep) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!mbar_wait(&bars->empty[stage], phase ^ 1, bars, status)) { ok = false; break; }
                mbar_expect_tx(&bars->full[stage], bytes);
                uint8_t* sa = sm.ring + stage * STAGE_BYTES2;
                tma_load_2d_hint(sa, map_a, kb * BK, (int)row0, &bars->full[stage], pol_a);
                if (ntiles == 2) tma_load_2d_hint(sa + A_BYTES, map_a, kb * BK, (int)(row0 + BM), &bars->full[stage], pol_a);
                load_b(sa + 2 * A_BYTES, e, nt, kb, &bars->full[stage], pol_b);
                pending |= 1u << stage;
                pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES2) { stage = 0; phase ^= 1; }
            }
        }
    }
    for (int s2 = 0; s2 < STAGES2; ++s2)
        if (pending & (1u << s2)) mbar_drain(&bars->full[s2], (pend_par >> s2) & 1u);
}

// One thread of warp 1. The unit's accumulators are handed over through tfull[0] / tempty[0].
__device__ __forceinline__ void run_mma2(const Smem& sm, const Sched& sc, uint32_t tmem, const int64_t* offsets,
                                         int E, int64_t R, int T, int NT, int KB, int* status) {
    Barriers* bars = sm.bars;
    int stage = 0;
    uint32_t phase = 0;
    int job = 0;
    bool ok = true;
    for (int u = sc.t0; ok && u < T; u += sc.tstep) {
        int e, ntiles;
        int64_t row0, row_end;
        unit2_rows(sm.tile_start, offsets, E, R, u, e, row0, row_end, ntiles);
        for (int nt = sc.n0; ok && nt < NT; nt += sc.nstep, ++job) {
            if (!mbar_wait(&bars->tempty[0], (uint32_t)(job & 1) ^ 1, bars, status)) { ok = false; break; }
            tc_fence_after();
            for (int kb = 0; kb < KB; ++kb) {
                if (!mbar_wait(&bars->full[stage], phase, bars, status)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sa = smem_addr(sm.ring + stage * STAGE_BYTES2);
                const uint64_t a0 = smem_desc(sa), a1 = smem_desc(sa + A_BYTES), b = smem_desc(sa + 2 * A_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / UK; ++kk) {
                    const uint32_t accum = (kb > 0 || kk > 0) ? 1u : 0u;
                    tc_mma(tmem, a0 + (uint64_t)(kk * 2), b + (uint64_t)(kk * 2), accum);
                    if (ntiles == 2) tc_mma(tmem + (uint32_t)BN, a1 + (uint64_t)(kk * 2), b + (uint64_t)(kk * 2), accum);
                }
                tc_commit(&bars->empty[stage]);
                if (++stage == STAGES2) { stage = 0; phase ^= 1; }
            }
            if (ok) tc_commit(&bars->tfull[0]);
        }
    }
    tc_commit(&bars->mma_done);
    mbar_drain(&bars->mma_done, 0);
}

// All threads, at the end: TMEM is freed by warp 1 once every role has finished with it.
__device__ __forceinline__ void pipeline_teardown(uint32_t tmem) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiled encode_fn() {
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

// 2-D bf16 tensor map: rows x cols (cols contiguous), box of box_rows x box_cols. Operand tiles use
// 64 columns (128 bytes) with the 128-byte swizzle the MMA descriptors expect; epilogue output
// tiles are unswizzled. Rows past the end read as zero and are not written. promo: the L2 sector
// promotion of the box's reads (256 bytes unless a kernel measured better with less).
inline bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_cols = BK, bool swizzle128 = true,
                     CUtensorMapL2promotion promo = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor map, 128-byte swizzle: d0 (contiguous) x d1 (stride1 bytes) x d2 (stride2
// bytes), box of box0 x box1 x box2 (box0 = 64: one 128-byte swizzle row).
inline bool make_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                        uint64_t stride2, uint32_t box0, uint32_t box1, uint32_t box2) {
    EncodeTiled fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {box0, box1, box2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch of a persistent kernel as clusters of ncl CTAs (ncl = 1: plain CTAs) in groups of csplit
// CTAs (a multiple of ncl; the CTAs sharing an M-tile): as many whole groups as can be resident at
// once, never more groups than there are M-tiles.
template <class... KArgs, class... Args>
inline cudaError_t launch_clusters(void (*kernel)(KArgs...), int64_t R, int64_t E, int ncl, int csplit,
                                   int threads, int smem, cudaStream_t stream, Args... args) {
    if (ncl < 1 || csplit % ncl != 0) return cudaErrorInvalidConfiguration;
    const int per_group = csplit / ncl;      // clusters per group
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(sms / csplit * csplit));
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, (const void*)kernel, &cfg);
    if (e != cudaSuccess) return e;
    int64_t groups = clusters / per_group;
    const int64_t tiles = (R + BM - 1) / BM + E;
    if (groups > tiles) groups = tiles;
    if (groups < 1) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3((unsigned)(groups * csplit));
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Persistent grid: one CTA per SM, a multiple of csplit, never more CTAs than the jobs could need.
inline int persistent_grid(int64_t R, int64_t E, int csplit, int* grid) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    const int64_t max_ctas = ((R + BM - 1) / BM + E) * csplit;
    int64_t g = max_ctas < sms ? max_ctas : sms;
    g = g / csplit * csplit;
    *grid = (int)(g > 0 ? g : csplit);
    return 0;
}

}  // namespace situ_tc
