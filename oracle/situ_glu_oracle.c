/*
 * SiTU-GLU oracle: a plain, slow, fp64 CPU restatement of what the method
 * computes, written from the two pages below.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline / reference legs may load or run this library. The
 * product path (the CUDA library in bwd_situ_glu_gb300/) never calls it, and the
 * two share no code, header, table or constant.
 *
 * Sources:
 *  [K3-RL]  "Frontier-scale RL with Kimi K3" (appliedcompute.com),
 *           section "Streaming activations": the naive situ_and_mul definition
 *           (split x into gate | linear halves, gate -> beta*tanh(gate/beta)*sigmoid(gate),
 *           linear -> linear_beta*tanh(linear/linear_beta), return their product),
 *           computed in fp32 from a bf16 x, beta = 4, linear_beta = 25; and the
 *           custom operator whose backward keeps only bf16 x and recomputes
 *           tanh and sigmoid.
 *  [K3-MEM] "Kimi K3 模型结构（9）：显存" (blog.javazero.top),
 *           section "MoE 反向：推一下为什么可以不存 expert 输出": the expert equation
 *           a_e = SiTU(W_gate x_e, W_up x_e), o_e = W_down a_e, y = sum_e p_e o_e;
 *           the router gradient dL/dp_e = <dL/dy, o_e>, moved across the inner
 *           product to <W_down^T dL/dy, a_e>; and dL/da_e = p_e W_down^T dL/dy.
 *
 * Notation (u = gate element, v = linear element, beta = β, lbeta = λ):
 *   T = tanh(u/β)   S = σ(u)   G = β·T·S
 *   W = tanh(v/λ)   L = λ·W    a = G·L
 *   G' = dG/du = (1 − T²)·S + β·T·S·(1 − S)        (product and chain rule)
 *   L' = dL/dv = 1 − W²
 * Backward with the router rewrite, for one routed row with upstream
 * g = W_downᵀ·dL/dy (not scaled by p) and router weight p:
 *   dp      = Σ_j g_j·a_j                            ([K3-MEM], rewritten inner product)
 *   dgate   = p·g·L·G'                               (dL/da = p·g, times da/du)
 *   dlinear = p·g·G·L'                               (dL/da = p·g, times da/dv)
 *
 * Everything is evaluated in double with libm tanh/exp; no blocking, fusion or
 * reordering. Rows are independent, so rows are split across threads; the
 * per-row sum runs over j = 0..H-1 in order, so results do not depend on the
 * thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* σ(u) without overflow: 1/(1+e^-u) for u >= 0, e^u/(1+e^u) for u < 0. */
static double sigmoid(double u) {
    if (u >= 0.0) return 1.0 / (1.0 + exp(-u));
    double e = exp(u);
    return e / (1.0 + e);
}

/* One element pair of [K3-RL] "Streaming activations" plus its two partial
 * derivatives. Writes G, L, G', L' (a = G·L). */
void oracle_situ_point(double u, double v, double beta, double lbeta, double res[4]) {
    double T = tanh(u / beta);
    double S = sigmoid(u);
    double G = beta * T * S;
    double W = tanh(v / lbeta);
    double L = lbeta * W;
    double Gp = (1.0 - T * T) * S + beta * T * S * (1.0 - S);
    double Lp = 1.0 - W * W;
    res[0] = G;
    res[1] = L;
    res[2] = Gp;
    res[3] = Lp;
}

/* bf16 storage bits -> double (exact: bf16 is the top half of an fp32). */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* ---------------- row kernels (one row at a time) ---------------- */

/* Forward of one row ([K3-RL] "Streaming activations"): gate = xr[0:H],
 * linear = xr[H:2H], out[j] = G(gate_j)·L(linear_j), unrounded. */
static void fwd_row(const double* xr, double* outr, int64_t H, double beta, double lbeta) {
    double res[4];
    for (int64_t j = 0; j < H; ++j) {
        oracle_situ_point(xr[j], xr[H + j], beta, lbeta, res);
        outr[j] = res[0] * res[1];
    }
}

/* Backward of one row with the router-gradient rewrite ([K3-MEM] section above):
 * dp = <g, a>, dgate = p·g·L·G', dlinear = p·g·G·L'. Also returns Σ|g_j·a_j|
 * (the scale of the dot product, used by the tests' tolerance). */
static void bwd_row(const double* xr, const double* gr, double p, double* dxr, double* dp,
                    double* dp_abs, int64_t H, double beta, double lbeta) {
    double res[4];
    double acc = 0.0, acc_abs = 0.0;
    for (int64_t j = 0; j < H; ++j) {
        oracle_situ_point(xr[j], xr[H + j], beta, lbeta, res);
        double G = res[0], L = res[1], Gp = res[2], Lp = res[3];
        double a = G * L;
        acc += gr[j] * a;
        acc_abs += fabs(gr[j] * a);
        dxr[j] = p * gr[j] * L * Gp;
        dxr[H + j] = p * gr[j] * G * Lp;
    }
    *dp = acc;
    if (dp_abs) *dp_abs = acc_abs;
}

/* ---------------- threading over rows ---------------- */

typedef struct {
    int kind;               /* 0 fwd f64, 1 bwd f64, 2 fwd bf16, 3 bwd bf16 */
    const void* x;
    const void* g;
    const void* p;
    double* out;            /* fwd: out [R,H]; bwd: dx [R,2H] */
    double* dp;
    double* dp_abs;
    int64_t r0, r1, H;
    double beta, lbeta;
} job_t;

static void* run_job(void* arg) {
    job_t* jb = (job_t*)arg;
    int64_t H = jb->H;
    double* xbuf = NULL;
    double* gbuf = NULL;
    if (jb->kind >= 2) {
        xbuf = (double*)malloc(sizeof(double) * (size_t)(2 * H));
        gbuf = (double*)malloc(sizeof(double) * (size_t)H);
        if (!xbuf || !gbuf) {
            free(xbuf);
            free(gbuf);
            return (void*)1;
        }
    }
    for (int64_t r = jb->r0; r < jb->r1; ++r) {
        const double* xr;
        const double* gr = NULL;
        double p = 0.0;
        if (jb->kind < 2) {
            xr = (const double*)jb->x + r * 2 * H;
            if (jb->kind == 1) {
                gr = (const double*)jb->g + r * H;
                p = ((const double*)jb->p)[r];
            }
        } else {
            const uint16_t* xb = (const uint16_t*)jb->x + r * 2 * H;
            for (int64_t j = 0; j < 2 * H; ++j) xbuf[j] = oracle_bf16_to_double(xb[j]);
            xr = xbuf;
            if (jb->kind == 3) {
                const uint16_t* gb = (const uint16_t*)jb->g + r * H;
                for (int64_t j = 0; j < H; ++j) gbuf[j] = oracle_bf16_to_double(gb[j]);
                gr = gbuf;
                p = (double)((const float*)jb->p)[r];
            }
        }
        if (jb->kind == 0 || jb->kind == 2) {
            fwd_row(xr, jb->out + r * H, H, jb->beta, jb->lbeta);
        } else {
            bwd_row(xr, gr, p, jb->out + r * 2 * H, jb->dp + r, jb->dp_abs ? jb->dp_abs + r : NULL,
                    H, jb->beta, jb->lbeta);
        }
    }
    free(xbuf);
    free(gbuf);
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run_rows(job_t proto, int64_t R, int nthreads) {
    if (R < 0 || proto.H <= 0) return 1;
    if (R == 0) return 0;
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if ((int64_t)nthreads > R) nthreads = (int)R;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
    if (!th || !jobs) {
        free(th);
        free(jobs);
        return 2;
    }
    int rc = 0;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].r0 = R * t / nthreads;
        jobs[t].r1 = R * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0) {
            /* fall back to running the remaining rows on this thread */
            job_t rest = proto;
            rest.r0 = jobs[t].r0;
            rest.r1 = R;
            if (run_job(&rest) != NULL) rc = 2;
            break;
        }
        ++started;
    }
    for (int t = 0; t < started; ++t) {
        void* ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = 2;
    }
    free(th);
    free(jobs);
    return rc;
}

/* ---------------- public entry points ---------------- */

/* Forward on an fp64 x [R,2H] -> out [R,H]. Returns 0 on success. */
int oracle_situ_glu_fwd_f64(const double* x, double* out, int64_t R, int64_t H, double beta,
                            double lbeta, int nthreads) {
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 0;
    jb.x = x;
    jb.out = out;
    jb.H = H;
    jb.beta = beta;
    jb.lbeta = lbeta;
    return run_rows(jb, R, nthreads);
}

/* Backward with the router rewrite on fp64 inputs: x [R,2H], g [R,H], p [R]
 * -> dx [R,2H], dp [R], and dp_abs [R] = Σ|g·a| (may be NULL). */
int oracle_situ_glu_bwd_router_f64(const double* x, const double* g, const double* p, double* dx,
                                   double* dp, double* dp_abs, int64_t R, int64_t H, double beta,
                                   double lbeta, int nthreads) {
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 1;
    jb.x = x;
    jb.g = g;
    jb.p = p;
    jb.out = dx;
    jb.dp = dp;
    jb.dp_abs = dp_abs;
    jb.H = H;
    jb.beta = beta;
    jb.lbeta = lbeta;
    return run_rows(jb, R, nthreads);
}

/* Forward on bf16 storage bits (converted exactly to double). */
int oracle_situ_glu_fwd_bf16(const uint16_t* x, double* out, int64_t R, int64_t H, double beta,
                             double lbeta, int nthreads) {
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 2;
    jb.x = x;
    jb.out = out;
    jb.H = H;
    jb.beta = beta;
    jb.lbeta = lbeta;
    return run_rows(jb, R, nthreads);
}

/* Backward on bf16 x and g bits and fp32 p (all converted exactly to double). */
int oracle_situ_glu_bwd_router_bf16(const uint16_t* x, const uint16_t* g, const float* p,
                                    double* dx, double* dp, double* dp_abs, int64_t R, int64_t H,
                                    double beta, double lbeta, int nthreads) {
    job_t jb;
    memset(&jb, 0, sizeof jb);
    jb.kind = 3;
    jb.x = x;
    jb.g = g;
    jb.p = p;
    jb.out = dx;
    jb.dp = dp;
    jb.dp_abs = dp_abs;
    jb.H = H;
    jb.beta = beta;
    jb.lbeta = lbeta;
    return run_rows(jb, R, nthreads);
}

/* ===================================================================================
 * Block-wise FP8 saved x ([K3-MEM], section "统一激活管理器：重算、量化、offload 都是存储策略":
 * most activations saved for backward are stored block-wise in FP8; elementwise operators
 * recompute). The pages leave the format open; the readings taken here:
 *   - FP8 E4M3 as defined by the OCP 8-bit floating point format (bias 7, 3 mantissa bits,
 *     subnormals, largest finite 448, code 0x7F/0xFF is NaN, no infinity);
 *   - blocks of 128 consecutive elements along a row, separately within the gate half and the
 *     linear half (the last block of a half may be shorter); nb = ceil(H / 128) per half;
 *   - one fp32 scale per block from the block's amax floored at 448 * 2^-126 (so the scale is a
 *     normal fp32 and 448 / amax cannot overflow): a = max(amax, 448 * 2^-126), s = a / 448,
 *     codes q = E4M3_RNE_satfinite(x * (448 / a)); dequantised x^ = decode(q) * s. An all-zero
 *     block gets s = 2^-126 and codes 0.
 * Every one of these steps is a single IEEE fp32 operation (amax exact, division and product
 * rounded to nearest), so the integer codes are fixed by the definition itself.
 * =================================================================================== */

/* value of a non-negative E4M3 code 0x00..0x7E (exact in float) */
static float e4m3_mag(int c) {
    int e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0) return ldexpf((float)m, -9);           /* subnormal: m/8 * 2^-6 */
    return ldexpf((float)(8 + m), e - 10);              /* (1 + m/8) * 2^(e-7) */
}

float oracle_e4m3_decode(uint8_t code) {
    int c = code & 0x7F;
    if (c == 0x7F) return NAN;
    float v = e4m3_mag(c);
    return (code & 0x80) ? -v : v;
}

/* Round to nearest E4M3 (ties to the even code), saturating finite values to +-448. */
uint8_t oracle_e4m3_encode(float v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (a >= 448.0f) return sign | 0x7E;
    /* largest code whose value is <= a (codes are monotone in value), by bisection */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_mag(mid) <= a) lo = mid; else hi = mid - 1;
    }
    int c = lo;
    if (c < 0x7E) {
        float below = e4m3_mag(c), above = e4m3_mag(c + 1);
        float d_lo = a - below, d_hi = above - a;       /* exact: both sides are representable steps */
        if (d_hi < d_lo || (d_hi == d_lo && (c & 1))) c = c + 1;
    }
    return (uint8_t)(sign | c);
}

/* One row half (n elements of bf16 bits) -> codes and scales of its blocks. */
static void quantize_half(const uint16_t* xb, int64_t n, uint8_t* q, float* s, int64_t block) {
    for (int64_t b0 = 0, bi = 0; b0 < n; b0 += block, ++bi) {
        int64_t b1 = b0 + block < n ? b0 + block : n;
        float amax = 0.0f;
        for (int64_t j = b0; j < b1; ++j) {
            float v = fabsf((float)oracle_bf16_to_double(xb[j]));
            if (v > amax) amax = v;
        }
        const float floor_amax = 448.0f * 0x1p-126f;     /* exact: 7 * 2^-120 */
        if (amax < floor_amax) amax = floor_amax;
        s[bi] = amax / 448.0f;
        float inv = 448.0f / amax;
        for (int64_t j = b0; j < b1; ++j) q[j] = oracle_e4m3_encode((float)oracle_bf16_to_double(xb[j]) * inv);
    }
}

/* x bf16 [R,2H] -> q uint8 [R,2H], s fp32 [R, 2*nb] (gate blocks, then linear blocks). */
int oracle_quantize_fp8(const uint16_t* x, uint8_t* q, float* s, int64_t R, int64_t H, int64_t block) {
    if (R < 0 || H <= 0 || block <= 0) return 1;
    int64_t nb = (H + block - 1) / block;
    for (int64_t r = 0; r < R; ++r) {
        quantize_half(x + r * 2 * H, H, q + r * 2 * H, s + r * 2 * nb, block);
        quantize_half(x + r * 2 * H + H, H, q + r * 2 * H + H, s + r * 2 * nb + nb, block);
    }
    return 0;
}

/* q, s -> x^ fp32 [R,2H] = decode(q) * s, one fp32 product per element. */
int oracle_dequantize_fp8(const uint8_t* q, const float* s, float* xhat, int64_t R, int64_t H, int64_t block) {
    if (R < 0 || H <= 0 || block <= 0) return 1;
    int64_t nb = (H + block - 1) / block;
    for (int64_t r = 0; r < R; ++r) {
        for (int64_t half = 0; half < 2; ++half) {
            for (int64_t j = 0; j < H; ++j) {
                float sc = s[r * 2 * nb + half * nb + j / block];
                xhat[r * 2 * H + half * H + j] = oracle_e4m3_decode(q[r * 2 * H + half * H + j]) * sc;
            }
        }
    }
    return 0;
}

/* ===================================================================================
 * bf16 rounding of an exact (double) value, for the gate/up projection whose output x is
 * saved in bf16 ([K3-RL] "Streaming activations": x is "the bf16 input tensor"; [K3-MEM]
 * section "MoE 反向…": x_e's two halves are W_gate,e·x_e and W_up,e·x_e). bf16 has 8
 * significant bits, exponents -126..127, subnormals down to 2^-133 and a largest finite value
 * (2 - 2^-7)·2^127. Rounding is to nearest, ties to the even significand (IEEE 754
 * roundTiesToEven), overflowing to infinity exactly when the rounded magnitude would need
 * exponent 128.
 * =================================================================================== */

/* Bits of a bf16 value given exactly as a double (an exact float, so its top 16 bits). */
static uint16_t bf16_bits_of_exact(double r) {
    float f = (float)r;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* The two bf16 values bracketing v: *lo <= v <= *hi, consecutive (or equal when v is a bf16
 * value). Finite v only; magnitudes beyond the largest finite bf16 bracket with infinity. */
void oracle_bf16_neighbours(double v, uint16_t* lo, uint16_t* hi) {
    double a = fabs(v);
    int e;
    frexp(a, &e);                          /* a = m·2^e, m in [0.5, 1) */
    int ex = (a == 0.0) ? -126 : e - 1;    /* a in [2^ex, 2^(ex+1)) */
    if (ex < -126) ex = -126;              /* subnormal range: spacing 2^-133 */
    double ulp = ldexp(1.0, ex - 7);
    double q = floor(a / ulp);             /* a / ulp is exact (power-of-two scaling) */
    double dn = q * ulp, up = (q * ulp == a) ? a : (q + 1.0) * ulp;
    const double maxf = ldexp(255.0, 120); /* (2 - 2^-7)·2^127 */
    uint16_t bdn = dn > maxf ? 0x7F80 : bf16_bits_of_exact(dn);
    uint16_t bup = up > maxf ? 0x7F80 : bf16_bits_of_exact(up);
    if (v < 0.0 || (v == 0.0 && signbit(v))) {
        *lo = (uint16_t)(bup | 0x8000);
        *hi = (uint16_t)(bdn | 0x8000);
    } else {
        *lo = bdn;
        *hi = bup;
    }
}

/* v rounded to the nearest bf16, ties to even; NaN -> the canonical quiet NaN 0x7FC0,
 * +-infinity kept, signed zero kept. */
uint16_t oracle_round_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    if (isinf(v)) return v > 0 ? 0x7F80 : 0xFF80;
    double a = fabs(v);
    int e;
    frexp(a, &e);
    int ex = (a == 0.0) ? -126 : e - 1;
    if (ex < -126) ex = -126;
    double ulp = ldexp(1.0, ex - 7);
    double q = a / ulp;                    /* exact */
    double fl = floor(q), rem = q - fl;    /* rem exact */
    double n = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;
    double r = n * ulp;
    uint16_t b = r > ldexp(255.0, 120) ? 0x7F80 : bf16_bits_of_exact(r);
    return (uint16_t)((signbit(v) ? 0x8000 : 0) | b);
}

int oracle_round_bf16_array(const double* v, uint16_t* out, int64_t n) {
    if (n < 0) return 1;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(v[i]);
    return 0;
}

/* ===================================================================================
 * Adam on host-resident optimizer state ([K3-RL] "Memory management" and "Streaming
 * gradients": the optimizer state lives in host memory as fp32 master weights and two bf16
 * moment tensors; gradients come from the device, the update is applied chunk by chunk
 * because Adam treats every parameter independently, and the updated weights go back to the
 * device as the bf16 working copy).
 *
 * The pages name Adam without formulas; the update is the textbook one (Kingma & Ba, with
 * PyTorch's placement of eps and, when weight_decay > 0, its decoupled AdamW decay):
 *   w  <- w·(1 - lr·wd)                                  (only when wd > 0)
 *   m  <- b1·m + (1 - b1)·g
 *   v  <- b2·v + (1 - b2)·g²
 *   w  <- w - (lr / (1 - b1^t)) · m / (sqrt(v) / sqrt(1 - b2^t) + eps)
 *
 * oracle_adam_f64: that definition in double on double state (the textbook reference).
 * oracle_adam_stored: the same update on the stored precisions the pages give (fp32 master,
 * bf16 moments): each step below is one IEEE fp32 operation, rounded to nearest, in this order
 * (no fused multiply-add), so the bf16 codes of the moments are decided in fp32 like the
 * product's:
 *   b1, b2, eps, c1 = 1 - b1, c2 = 1 - b2, s = lr / bc1, r = 1 / sqrt(bc2), d = 1 - lr·wd:
 *        each formed in double from the double hyper-parameters (bc1 = 1 - b1^t, bc2 = 1 - b2^t)
 *        and rounded to fp32 once (rounding b2 first and then forming 1 - b2 in fp32 would put
 *        a 1e-5 relative error on c2 = 0.001)
 *   w1 = wd > 0 ? fl(w·d) : w
 *   m1 = fl(fl(b1·m) + fl(c1·g))
 *   v1 = fl(fl(b2·v) + fl(c2·fl(g·g)))
 *   q  = fl(fl(sqrt(v1))·r) + eps  -> fl
 *   w2 = fl(w1 - fl(s·fl(m1 / q)))
 *   stored: master = w2, m = RNE_bf16(m1), v = RNE_bf16(v1), working weight = RNE_bf16(w2)
 * =================================================================================== */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
} oracle_adam_hp;

int oracle_adam_f64(double* w, double* m, double* v, const double* g, int64_t n, const oracle_adam_hp* hp) {
    if (n < 0 || !hp || hp->step < 1) return 1;
    const double bc1 = 1.0 - pow(hp->beta1, (double)hp->step);
    const double bc2 = 1.0 - pow(hp->beta2, (double)hp->step);
    for (int64_t i = 0; i < n; ++i) {
        if (hp->weight_decay > 0.0) w[i] = w[i] * (1.0 - hp->lr * hp->weight_decay);
        m[i] = hp->beta1 * m[i] + (1.0 - hp->beta1) * g[i];
        v[i] = hp->beta2 * v[i] + (1.0 - hp->beta2) * g[i] * g[i];
        const double denom = sqrt(v[i]) / sqrt(bc2) + hp->eps;
        w[i] = w[i] - (hp->lr / bc1) * m[i] / denom;
    }
    return 0;
}

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

int oracle_adam_stored(float* master, uint16_t* m, uint16_t* v, const float* g, uint16_t* w_out, int64_t n,
                       const oracle_adam_hp* hp) {
    if (n < 0 || !hp || hp->step < 1) return 1;
    const double bc1 = 1.0 - pow(hp->beta1, (double)hp->step);
    const double bc2 = 1.0 - pow(hp->beta2, (double)hp->step);
    const float b1 = (float)hp->beta1, b2 = (float)hp->beta2, eps = (float)hp->eps;
    const float c1 = (float)(1.0 - hp->beta1), c2 = (float)(1.0 - hp->beta2);
    const float s = (float)(hp->lr / bc1);
    const float r = (float)(1.0 / sqrt(bc2));
    const float d = (float)(1.0 - hp->lr * hp->weight_decay);
    const int decay = hp->weight_decay > 0.0;
    for (int64_t i = 0; i < n; ++i) {
        volatile float t;                 /* one rounding per operation, in this order */
        float w1 = master[i];
        if (decay) { t = w1 * d; w1 = t; }
        float gb = g[i];
        t = b1 * bf16_bits_to_float(m[i]); float ma = t;
        t = c1 * gb; float mb = t;
        t = ma + mb; float m1 = t;
        t = gb * gb; float gg = t;
        t = b2 * bf16_bits_to_float(v[i]); float va = t;
        t = c2 * gg; float vb = t;
        t = va + vb; float v1 = t;
        t = sqrtf(v1); float sq = t;
        t = sq * r; float qa = t;
        t = qa + eps; float q = t;
        t = m1 / q; float u = t;
        t = s * u; float su = t;
        t = w1 - su; float w2 = t;
        master[i] = w2;
        m[i] = oracle_round_bf16((double)m1);
        v[i] = oracle_round_bf16((double)v1);
        w_out[i] = oracle_round_bf16((double)w2);
    }
    return 0;
}
