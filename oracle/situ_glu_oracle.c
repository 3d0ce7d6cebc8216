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
