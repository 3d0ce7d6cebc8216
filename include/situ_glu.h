/*
 * situ_glu.h — C ABI of the GB300 (sm_103a) SiTU-GLU library.
 *
 * Two operations, each one hand-written CUDA kernel launch:
 *
 *   situ_glu_fwd         the SiTU-GLU expert activation over routed rows.
 *                        Defined in "Frontier-scale RL with Kimi K3", section
 *                        "Streaming activations" (the naive situ_and_mul listing):
 *                        split each row of x into gate | linear halves and return
 *                        out = [beta·tanh(gate/beta)·sigmoid(gate)] · [lbeta·tanh(linear/lbeta)],
 *                        computed in fp32 from bf16 x and rounded to bf16.
 *
 *   situ_glu_bwd_router  its backward, which keeps only bf16 x and recomputes
 *                        tanh / sigmoid (same section: the custom operator,
 *                        points 1 and 2), fused with the router-probability
 *                        gradient of "Kimi K3 模型结构（9）：显存", section
 *                        "MoE 反向：推一下为什么可以不存 expert 输出":
 *                        with g = W_downᵀ·dL/dy for a routed row and that row's
 *                        router weight p,
 *                            dp[r]     = Σ_j g[r,j]·a[r,j]         (= dL/dp_e, no stored o_e)
 *                            dx[r,j]   = p[r]·g[r,j]·L·G'          (gate half)
 *                            dx[r,H+j] = p[r]·g[r,j]·G·L'          (linear half)
 *                        where G = beta·tanh(u/beta)·sigmoid(u), L = lbeta·tanh(v/lbeta),
 *                        G' = dG/du, L' = dL/dv, a = G·L, u = x[r,j], v = x[r,H+j].
 *
 * Layouts (all row-major, contiguous, little-endian):
 *   x    bf16 [R, 2H]   gate in columns 0..H-1, linear in columns H..2H-1
 *   out  bf16 [R, H]
 *   g    bf16 [R, H]    NOT pre-scaled by p
 *   p    fp32 [R]
 *   dx   bf16 [R, 2H]   d/dgate in columns 0..H-1, d/dlinear in H..2H-1
 *   dp   fp32 [R]
 * bf16 tensors are passed as raw 16-bit storage (the bits of __nv_bfloat16).
 *
 * Arithmetic: fp32 in registers; the dp reduction uses the unrounded fp32 a,
 * summed per row in a fixed order (results are bit-reproducible run to run).
 * bf16 results are rounded to nearest even.
 *
 * Pointers are DEVICE pointers on the calling thread's current CUDA device.
 * The caller owns every buffer. The library allocates no memory, keeps no
 * workspace and no state beyond per-device launch-configuration caches.
 * Calls are asynchronous on `stream` (0 = the legacy default stream) and never
 * synchronise the host.
 *
 * Fast path: base pointers of x/out (fwd) or x/g/dx (bwd) 16-byte aligned and
 * H % 8 == 0 -> 16-byte vector loads and stores. Anything else still works on a
 * per-element path (slower). Non-finite inputs propagate (NaN in, NaN out);
 * finite inputs of any magnitude give finite results.
 *
 * Return value of every compute entry point: a situ_glu_status. All argument
 * checks happen before any CUDA call; on a non-zero status nothing was enqueued.
 */
#ifndef SITU_GLU_H
#define SITU_GLU_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SITU_GLU_VERSION_MAJOR 1
#define SITU_GLU_VERSION_MINOR 6
#define SITU_GLU_VERSION_PATCH 0

/* Largest H accepted (columns per half). */
#define SITU_GLU_MAX_H (1LL << 30)

typedef enum situ_glu_status {
    SITU_GLU_OK = 0,
    /* a required pointer is NULL while R > 0; R < 0; H <= 0 or H > SITU_GLU_MAX_H;
       beta or lbeta not finite or <= 0; R*2H*2 bytes overflows int64; a bf16
       pointer not 2-byte aligned or an fp32 pointer not 4-byte aligned */
    SITU_GLU_INVALID_ARG = 1,
    /* an output byte range overlaps an input or another output. The single
       exception: situ_glu_bwd_router accepts dx == x exactly (in place). */
    SITU_GLU_OVERLAP = 2,
    /* a CUDA runtime call or the kernel launch failed; see situ_glu_last_cuda_error() */
    SITU_GLU_CUDA_ERROR = 3
} situ_glu_status;

/*
 * Forward: out[r,j] = bf16( G(x[r,j]) · L(x[r,H+j]) ) for r < R, j < H.
 *   x      device, bf16 [R,2H], read only
 *   out    device, bf16 [R,H], written; must not overlap x
 *   R      rows (>= 0; R == 0 is a successful no-op, pointers may then be NULL)
 *   H      columns per half (1 .. SITU_GLU_MAX_H)
 *   beta   gate scale β (finite, > 0; 4 in the pages). β == 4 with λ <= 64 takes a
 *          faster kernel that shares one exponential between tanh(u/4) and sigmoid(u)
 *   lbeta  linear scale λ (finite, > 0; 25 in the pages)
 *   stream CUDA stream to enqueue on
 * Source: "Frontier-scale RL with Kimi K3", section "Streaming activations".
 */
int situ_glu_fwd(const void* x, void* out, int64_t R, int64_t H, float beta, float lbeta,
                 cudaStream_t stream);

/*
 * Fused backward + router gradient (see the file comment for the formulas).
 *   x      device, bf16 [R,2H], read only (the only tensor saved from forward)
 *   g      device, bf16 [R,H], read only: g = W_downᵀ·dL/dy per routed row
 *   p      device, fp32 [R], read only: router weight of each row
 *   dx     device, bf16 [R,2H], written. May be exactly x (in place: each
 *          element of x is read before the same thread overwrites it);
 *          must not otherwise overlap x, g, p or dp
 *   dp     device, fp32 [R], written; must not overlap any other buffer
 *   R, H, beta, lbeta, stream as for situ_glu_fwd
 * Sources: "Frontier-scale RL with Kimi K3", section "Streaming activations"
 * (backward keeps only x and recomputes tanh and sigmoid); "Kimi K3 模型结构（9）：显存",
 * section "MoE 反向：推一下为什么可以不存 expert 输出" (dL/dp_e = <W_downᵀ dL/dy, a_e>,
 * dL/da_e = p_e·W_downᵀ dL/dy).
 */
int situ_glu_bwd_router(const void* x, const void* g, const float* p, void* dx, float* dp,
                        int64_t R, int64_t H, float beta, float lbeta, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Block-wise FP8 saved x.
 *
 * "Kimi K3 模型结构（9）：显存", section "统一激活管理器：重算、量化、offload 都是存储策略": most
 * activations saved for the backward are stored with block-wise FP8 quantisation, while
 * elementwise operators are recomputed. Here the saved tensor x is stored as OCP FP8 E4M3
 * codes with one fp32 scale per block of SITU_GLU_FP8_BLOCK consecutive elements of one half
 * of a row (the last block of a half may be shorter), which halves the saved bytes and cuts
 * the backward's traffic from 10H + 8 to 8H + 8*ceil(H/128) + 8 bytes per row.
 *
 * For each block: a = max(amax(|x|), 448 * 2^-126), scale = a / 448,
 * code = E4M3 round-to-nearest-even, saturated to +-448, of x * (448 / a); each step is one
 * IEEE fp32 operation. Dequantised x^ = value(code) * scale (fp32).
 *
 * Layouts: xq uint8 [R, 2H] (gate codes then linear codes, like x); xs fp32 [R, 2*nb] with
 * nb = ceil(H / SITU_GLU_FP8_BLOCK) (gate blocks, then linear blocks).
 * A non-finite element makes its own code NaN; an infinity also makes its block's scale
 * infinite (so the block dequantises to NaN).
 * --------------------------------------------------------------------------------------- */
#define SITU_GLU_FP8_BLOCK 128

/*
 * Forward that also saves x in FP8: out exactly as situ_glu_fwd, plus xq and xs from one read
 * of x.
 *   x      device, bf16 [R,2H], read only
 *   out    device, bf16 [R,H], written
 *   xq     device, uint8 [R,2H], written (8-byte alignment takes the vector path)
 *   xs     device, fp32 [R,2*nb], written (4-byte aligned)
 *   outputs must not overlap x or each other
 *   R, H, beta, lbeta, stream as for situ_glu_fwd
 */
int situ_glu_fwd_save_fp8(const void* x, void* out, uint8_t* xq, float* xs, int64_t R, int64_t H,
                          float beta, float lbeta, cudaStream_t stream);

/*
 * Fused backward + router gradient from the FP8-saved x: the formulas of situ_glu_bwd_router
 * evaluated at x^ = value(xq) * xs.
 *   xq, xs device, read only, as written by situ_glu_fwd_save_fp8
 *   g, p   as for situ_glu_bwd_router
 *   dx     device, bf16 [R,2H], written; dp device, fp32 [R], written; neither may overlap an
 *          input or the other
 *   R, H, beta, lbeta, stream as for situ_glu_fwd
 */
int situ_glu_bwd_router_fp8(const uint8_t* xq, const float* xs, const void* g, const float* p,
                            void* dx, float* dp, int64_t R, int64_t H, float beta, float lbeta,
                            cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Down-projection dgrad fused with the backward (tensor cores).
 *
 * "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出": the routed row's
 * g = (W_down,e)ᵀ·dL/dy is what the backward computes anyway; the router gradient and dL/da_e
 * follow from it and a_e. This entry point computes g = dY·W_down,e for every expert's rows on
 * the tensor cores (tcgen05, fp32 accumulation in tensor memory) and, in the same kernel, the
 * outputs of situ_glu_bwd_router from that g (fp32, never rounded or written) and x.
 *
 *   x          device, bf16 [R,2H], read only (the saved forward input)
 *   dy         device, bf16 [R,D], read only: dL/dy of each routed row (D = expert output width)
 *   w_down_t   device, bf16 [E,H,D], read only: (W_down,e)ᵀ of each expert, K-major (row j of
 *              expert e holds W_down,e[:, j]), so g[r,j] = Σ_d dy[r,d]·w_down_t[e,j,d]
 *   expert_offsets device, int64 [E+1]: rows of expert e are expert_offsets[e] ..
 *              expert_offsets[e+1]-1 (non-decreasing, from 0 to R; rows grouped by expert).
 *              Malformed offsets (negative, decreasing, beyond R) are clamped into [0, R]: the
 *              results of the rows they cover are undefined, but nothing is accessed outside the
 *              buffers and the work stays bounded (at most ceil(R/128) + E row tiles).
 *   p, dx, dp  as for situ_glu_bwd_router. When H >= 1024 and the experts average fewer than
 *              512 rows, dp is zeroed on the stream first and each row's dp arrives as two
 *              partial sums added with atomics; two addends commute exactly, so dp is still
 *              deterministic (that add flushes a subnormal result, |dp| < 2^-126, to zero).
 *   status     device int (may be NULL), written only on failure: set to 1 if a pipeline wait in
 *              the kernel exceeded its limit (then dx and dp are incomplete). Zero it beforehand.
 *   R, H, D, E sizes: H % 16 == 0, D % 8 == 0, 1 <= E <= 1024, R < 2^31, E*H < 2^31 - 256.
 *              The tensor cores work on 256-column N-tiles and 64-deep K-blocks: a K tail reads
 *              zeros past D, and an N tail computes columns past H that are never used.
 *   Pointers to dy and w_down_t must be 16-byte aligned (TMA), to x and dx 32-byte aligned
 *   (32-byte vector access).
 * Returns SITU_GLU_INVALID_ARG for shapes or alignments outside these limits.
 * --------------------------------------------------------------------------------------- */
int situ_glu_bwd_router_dgrad(const void* x, const void* dy, const void* w_down_t,
                              const int64_t* expert_offsets, int64_t E, const float* p, void* dx,
                              float* dp, int* status, int64_t R, int64_t H, int64_t D, float beta,
                              float lbeta, cudaStream_t stream);

/* The same with the weights in their nn.Linear layout: w_down device, bf16 [E,D,H], row d of
 * expert e holding W_down,e[d, :], so g[r,j] = Σ_d dy[r,d]·w_down[e,d,j] (read N-major by the
 * tensor cores; no transposed copy needed). D % 64 == 0 here (K runs along the rows of [E·D, H],
 * so a K tail would reach the next expert's rows), E*D < 2^31; everything else as above; results
 * are bit-identical to situ_glu_bwd_router_dgrad on the transposed weights. */
int situ_glu_bwd_router_dgrad_wd(const void* x, const void* dy, const void* w_down,
                                 const int64_t* expert_offsets, int64_t E, const float* p, void* dx,
                                 float* dp, int* status, int64_t R, int64_t H, int64_t D,
                                 float beta, float lbeta, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Gate/up projection fused with the forward (tensor cores).
 *
 * "Kimi K3 模型结构（9）：显存", section "MoE 反向：推一下为什么可以不存 expert 输出": a routed row
 * of expert e computes a_e = SiTU(W_gate,e·h, W_up,e·h) from its dispatched input h.
 * "Frontier-scale RL with Kimi K3", section "Streaming activations": only the bf16 pre-activation
 * x = [W_gate,e·h | W_up,e·h] is kept for the backward. This entry point computes both
 * projections of every routed row on the tensor cores (tcgen05, fp32 accumulation in tensor
 * memory) and, in the same kernel, writes x rounded to bf16 (nearest even) and
 * out = G(gate)·L(linear) evaluated on that bf16 x: the same values as the projection followed
 * by situ_glu_fwd, without reading x back.
 *
 *   h          device, bf16 [R,D], read only: each routed row's dispatched input, rows grouped
 *              by expert
 *   w_gate_up  device, bf16 [E,2H,D], read only, K-major: rows 0..H-1 of expert e are W_gate,e
 *              (row j = the weights of gate column j), rows H..2H-1 are W_up,e, so
 *              x[r,n] = Σ_d h[r,d]·w_gate_up[e,n,d]
 *   expert_offsets device, int64 [E+1]: as for situ_glu_bwd_router_dgrad
 *   x          device, bf16 [R,2H], written: the saved pre-activation (gate half, linear half)
 *   out        device, bf16 [R,H], written: SiTU-GLU of x
 *   status     device int (may be NULL), written only on failure: set to 1 if a pipeline wait in
 *              the kernel exceeded its limit (then x and out are incomplete). Zero it beforehand.
 *   R, H, D, E sizes: H % 16 == 0, D % 8 == 0, 1 <= E <= 1024, R < 2^31, E*2H < 2^31 (the
 *              tensor cores work on 128-column pairs of N-tiles and 64-deep K-blocks; the tails
 *              read zeros past H and D, and columns past H are not stored)
 *   Pointers to h and w_gate_up must be 16-byte aligned (TMA), to x and out 32-byte aligned.
 * x and out may not overlap each other or any input (SITU_GLU_OVERLAP). Returns
 * SITU_GLU_INVALID_ARG for shapes or alignments outside these limits.
 * --------------------------------------------------------------------------------------- */
int situ_glu_fwd_gateup(const void* h, const void* w_gate_up, const int64_t* expert_offsets,
                        int64_t E, void* x, void* out, int* status, int64_t R, int64_t H,
                        int64_t D, float beta, float lbeta, cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Adam on host-resident optimizer state, streamed chunk by chunk.
 *
 * "Frontier-scale RL with Kimi K3", sections "Memory management" and "Streaming gradients": the
 * optimizer state lives in host memory (fp32 master weights, two bf16 moment tensors); the
 * device's gradients are brought to the host and the updated weights go back as the bf16
 * working copy. Instead of one parameter-sized fp32 host gradient buffer (12 bytes of host
 * memory per parameter), the update runs chunk by chunk with the transfers of the next chunks
 * in flight: 8 bytes per parameter plus nslots chunk-sized staging slots.
 *
 * One step per element, as single IEEE fp32 operations in this order (no fused multiply-add):
 *   constants formed in double from the fields below and rounded to fp32 once:
 *     b1, b2, eps, c1 = 1 - beta1, c2 = 1 - beta2, s = lr / (1 - beta1^step),
 *     r = 1 / sqrt(1 - beta2^step), d = 1 - lr * weight_decay
 *   w1 = weight_decay > 0 ? w * d : w          (decoupled weight decay, as PyTorch's AdamW)
 *   m1 = b1*m + c1*g;   v1 = b2*v + c2*(g*g);   q = sqrt(v1)*r + eps;   w2 = w1 - s*(m1/q)
 *   stored: master = w2; m, v, working weight = bf16(m1), bf16(v1), bf16(w2), rounded to nearest
 *   even (NaN -> 0x7FC0).
 * --------------------------------------------------------------------------------------- */
typedef struct {
    double lr;            /* >= 0, finite */
    double beta1, beta2;  /* in [0, 1) */
    double eps;           /* > 0 */
    double weight_decay;  /* >= 0; 0 = plain Adam */
    int64_t step;         /* 1-based step count t of this update (bias corrections 1 - beta^t) */
} situ_adam_params;

/* One step over n parameters, all in host memory: master fp32 [n], m and v bf16 [n] updated in
 * place, g fp32 [n] read, w_out bf16 [n] written with the new working weights. nthreads host
 * threads (<= 0: the CPUs this process may run on). No CUDA call. Buffers may not overlap
 * (SITU_GLU_OVERLAP); fp32 pointers 4-byte and bf16 pointers 2-byte aligned. */
int situ_adam_update_host(float* master, void* m, void* v, const float* g, void* w_out, int64_t n,
                          const situ_adam_params* hp, int nthreads);

/* The streamed step: grad_dev device fp32 [n] (read), weight_dev device bf16 [n] (overwritten with
 * the new working weights), master / m / v host as above (any host memory), staging page-locked
 * host memory of nslots * chunk * 6 bytes (16-byte aligned; nslots fp32 gradient slots, then
 * nslots bf16 weight slots), chunk elements per transfer (a positive multiple of 64),
 * 2 <= nslots <= 64. The copies run on `stream` in order after the work already queued there
 * (so after the kernels that produced the gradients), gradient chunk c + nslots in flight while
 * chunk c is updated by nthreads host threads; returns when every chunk's weights are on the
 * device. Creates and destroys 2*nslots CUDA events per call; allocates no memory. On a CUDA
 * error (SITU_GLU_CUDA_ERROR) a prefix of the chunks may have been updated; the call still
 * waits for `stream` (every copy it queued) before returning, so staging may be reused or
 * freed as soon as it returns, whatever the status. */
int situ_adam_stream_step(const float* grad_dev, void* weight_dev, float* master, void* m, void* v,
                          int64_t n, const situ_adam_params* hp, void* staging, int64_t chunk,
                          int nslots, int nthreads, cudaStream_t stream);

/* Self-test of the tensor-core kernels' failure path (faults nothing): launches one CTA that
 * waits, with the same bounded wait as the GEMM pipelines, on an mbarrier nothing completes. The
 * wait gives up after about 2 s and the kernel writes 1 to *status (device int, zeroed by the
 * caller) and returns normally; *elapsed_ns (device, may be NULL) receives how long it waited.
 * Asynchronous on `stream`. */
int situ_glu_selftest_wait_timeout(int* status, unsigned long long* elapsed_ns, cudaStream_t stream);

/* Static, NUL-terminated description of a status code (unknown codes included). */
const char* situ_glu_status_string(int status);

/* The cudaError_t behind the last SITU_GLU_CUDA_ERROR returned on this host thread
   (cudaSuccess if none). */
int situ_glu_last_cuda_error(void);

/* MAJOR*10000 + MINOR*100 + PATCH */
int situ_glu_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SITU_GLU_H */
