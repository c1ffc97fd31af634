/*
 * CPU ORACLE -- test infrastructure, not part of the product.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * build, load or call this file. The CUDA library never links it, and it uses
 * nothing from the CUDA library.
 *
 * What it computes: the gated delta rule, one token at a time, in fp64.
 * For every sequence s and value head h (key/query head kh = h / (nv / nk)):
 *
 *     S   <- S_0[s][h]                                   (dk x dv, fp64)
 *     for each token t of s, in order:
 *         S <- exp(g_t) * S                              (decay the whole state)
 *         p <- S^T k_t                                   (what S recalls for k_t)
 *         S <- S + beta_t * k_t (v_t - p)^T              (delta-rule write)
 *         o_t <- S^T q_t / sqrt(dk)                      (read-out after the write)
 *     S_T[s][h] <- S
 *
 * The two middle lines are S <- e^{g}(I - beta k k^T) S + beta k v^T, the
 * recurrence whose chunked evaluation is the GDN prefill op (ssm_gdn_a3.rs,
 * doc comment of `gdn_prefill_fla`: a per-chunk WY triangular solve, a serial
 * state spine over chunks, and a chunk-parallel output stage). The output
 * reads the state after the token's own update, and 1/sqrt(dk) scales the
 * read-out.
 *
 * Inputs may be bf16 bit patterns, fp32 or fp64 (widened exactly to fp64);
 * arithmetic is fp64 throughout. Row addressing follows the op's problem
 * arguments: row r = b*T + t (dense) or cu_seqlens[s] + t (varlen); element
 * (r, head, i) of q/k sits at r*stride + head*dk + i, and of g/beta at
 * r*stride + h.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_F32 = 1, ORC_F64 = 2 };

static double orc_load(const void* base, int dtype, int64_t idx) {
    if (dtype == ORC_BF16) {
        uint32_t u = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    if (dtype == ORC_F32) return (double)((const float*)base)[idx];
    return ((const double*)base)[idx];
}

static void orc_load_row(const void* base, int dtype, int64_t off, int n, double* dst) {
    for (int i = 0; i < n; ++i) dst[i] = orc_load(base, dtype, off + i);
}

/*
 * Runs the recurrence for the (sequence, v-head) pairs selected by `heads`
 * (all nv heads when heads == NULL). Returns 0, or -1 on bad arguments or an
 * allocation failure.
 *
 *   q, k      : [rows][q_stride] / [rows][k_stride], dtype qkv_dtype
 *   v         : [rows][v_stride], dtype qkv_dtype
 *   g, beta   : [rows][g_stride] / [rows][beta_stride], dtype gb_dtype
 *   h0        : [B][nv][dk][dv], dtype h_dtype, or NULL for a zero state
 *   out       : [rows][nv][dv] fp64 (only rows of evaluated heads written)
 *   hT        : [B][nv][dk][dv] fp64 (only evaluated heads written)
 *   cu_seqlens: host [B+1] or NULL (dense: B sequences of T rows)
 */
int gdn_oracle_run(const void* q, const void* k, const void* v, int qkv_dtype,
                   const void* g, const void* beta, int gb_dtype,
                   const void* h0, int h_dtype,
                   double* out, double* hT,
                   int B, int T, int nk, int nv, int dk, int dv,
                   int64_t q_stride, int64_t k_stride, int64_t v_stride,
                   int64_t g_stride, int64_t beta_stride,
                   const int32_t* cu_seqlens,
                   const int32_t* heads, int n_heads, int n_threads) {
    if (B < 0 || nk <= 0 || nv <= 0 || dk <= 0 || dv <= 0 || nv % nk != 0) return -1;
    if (heads == NULL) n_heads = nv;
    const int group = nv / nk;
    const double scale = 1.0 / sqrt((double)dk);
    const int64_t pairs = (int64_t)B * n_heads;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t pi = 0; pi < pairs; ++pi) {
        const int s = (int)(pi / n_heads);
        const int h = heads ? heads[pi % n_heads] : (int)(pi % n_heads);
        const int kh = h / group;
        const int64_t row0 = cu_seqlens ? cu_seqlens[s] : (int64_t)s * T;
        const int64_t len = cu_seqlens ? (int64_t)cu_seqlens[s + 1] - cu_seqlens[s] : T;
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
        double* qt = (double*)malloc(sizeof(double) * (size_t)dk);
        double* kt = (double*)malloc(sizeof(double) * (size_t)dk);
        double* vt = (double*)malloc(sizeof(double) * (size_t)dv);
        double* p = (double*)malloc(sizeof(double) * (size_t)dv);
        if (!S || !qt || !kt || !vt || !p) {
            failed |= 1;
        } else {
            const int64_t sbase = ((int64_t)s * nv + h) * dk * dv;
            for (int64_t i = 0; i < (int64_t)dk * dv; ++i)
                S[i] = h0 ? orc_load(h0, h_dtype, sbase + i) : 0.0;
            for (int64_t t = 0; t < len; ++t) {
                const int64_t r = row0 + t;
                const double a = exp(orc_load(g, gb_dtype, r * g_stride + h));
                const double b = orc_load(beta, gb_dtype, r * beta_stride + h);
                orc_load_row(q, qkv_dtype, r * q_stride + (int64_t)kh * dk, dk, qt);
                orc_load_row(k, qkv_dtype, r * k_stride + (int64_t)kh * dk, dk, kt);
                orc_load_row(v, qkv_dtype, r * v_stride + (int64_t)h * dv, dv, vt);
                /* S <- a S */
                for (int64_t i = 0; i < (int64_t)dk * dv; ++i) S[i] *= a;
                /* p <- S^T k */
                for (int j = 0; j < dv; ++j) p[j] = 0.0;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) p[j] += S[(int64_t)i * dv + j] * kt[i];
                /* S <- S + b k (v - p)^T */
                for (int i = 0; i < dk; ++i) {
                    const double bk = b * kt[i];
                    for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += bk * (vt[j] - p[j]);
                }
                /* o <- S^T q / sqrt(dk) */
                double* o = out + (r * nv + h) * dv;
                for (int j = 0; j < dv; ++j) o[j] = 0.0;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) o[j] += S[(int64_t)i * dv + j] * qt[i];
                for (int j = 0; j < dv; ++j) o[j] *= scale;
            }
            memcpy(hT + sbase, S, sizeof(double) * (size_t)dk * dv);
        }
        free(S);
        free(qt);
        free(kt);
        free(vt);
        free(p);
    }
    return failed ? -1 : 0;
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Backward of the same recurrence (reverse-mode, fp64), for the training pass.
 * Given dO = dL/do_t for every row and dST = dL/dS_T (or NULL for zero), it
 * returns dL/dq, dL/dk, dL/dv, dL/dg, dL/dbeta and dL/dS_0. Per token, with
 * P = S_{t-1}, D = e^{g} P, p = D^T k, S = D + beta k (v - p)^T and G = dL/dS
 * (the future's gradient plus the token's own read-out term q do^T / sqrt(dk)):
 *
 *     dq    = S do / sqrt(dk)
 *     dv    = beta G^T k                    dp = -dv
 *     dbeta = k^T G (v - p)
 *     dD    = G + k dp^T
 *     dk    = beta G (v - p) + D dp
 *     dg    = <dD, D>                       (dL/dg = e^{g} <dD, P>)
 *     dL/dS_{t-1} = e^{g} dD
 *
 * q and k gradients of a key head sum over the value heads of its group. The
 * states S_{t-1} are recomputed forward from checkpoints every 64 tokens.
 *
 *   dout : [rows][nv][dv] fp64          dST : [B][nv][dk][dv] fp64 or NULL
 *   dq, dk : [rows][nk][dk] fp64        dv : [rows][nv][dv] fp64
 *   dg, dbeta : [rows][nv] fp64         dh0 : [B][nv][dk][dv] fp64
 * Rows outside every sequence are left untouched. Returns 0, or -1.
 */
int gdn_oracle_backward(const void* q, const void* k, const void* v, int qkv_dtype,
                        const void* g, const void* beta, int gb_dtype,
                        const void* h0, int h_dtype,
                        const double* dout, const double* dST,
                        double* dq, double* dkk, double* dvv, double* dg, double* dbeta, double* dh0,
                        int B, int T, int nk, int nv, int dk, int dv,
                        int64_t q_stride, int64_t k_stride, int64_t v_stride,
                        int64_t g_stride, int64_t beta_stride,
                        const int32_t* cu_seqlens, int n_threads) {
    if (B < 0 || nk <= 0 || nv <= 0 || dk <= 0 || dv <= 0 || nv % nk != 0) return -1;
    const int group = nv / nk;
    const double scale = 1.0 / sqrt((double)dk);
    const int64_t dd = (int64_t)dk * dv;
    const int blk = 64;
    const int64_t pairs = (int64_t)B * nk;
    int failed = 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t pi = 0; pi < pairs; ++pi) {
        const int s = (int)(pi / nk), kh = (int)(pi % nk);
        const int64_t row0 = cu_seqlens ? cu_seqlens[s] : (int64_t)s * T;
        const int64_t len = cu_seqlens ? (int64_t)cu_seqlens[s + 1] - cu_seqlens[s] : T;
        const int64_t nblk = (len + blk - 1) / blk;
        double* ck = (double*)malloc(sizeof(double) * (size_t)((nblk > 0 ? nblk : 1) * dd));
        double* st = (double*)malloc(sizeof(double) * (size_t)((blk + 1) * dd));
        double* G = (double*)malloc(sizeof(double) * (size_t)dd);
        double* dD = (double*)malloc(sizeof(double) * (size_t)dd);
        double* vec = (double*)malloc(sizeof(double) * (size_t)(4 * dk + 6 * dv));
        if (!ck || !st || !G || !dD || !vec) {
            failed |= 1;
        } else {
            double *qt = vec, *kt = vec + dk, *dkv = vec + 2 * dk, *dqv = vec + 3 * dk;
            double *vt = vec + 4 * dk, *p = vt + dv, *w = p + dv, *gk = w + dv, *dov = gk + dv, *dp = dov + dv;
            for (int hh = 0; hh < group; ++hh) {
                const int h = kh * group + hh;
                const int64_t sbase = ((int64_t)s * nv + h) * dd;
                /* forward: checkpoints of the state entering each block of 64 tokens */
                double* S = st;
                for (int64_t i = 0; i < dd; ++i) S[i] = h0 ? orc_load(h0, h_dtype, sbase + i) : 0.0;
                for (int64_t t = 0; t < len; ++t) {
                    if (t % blk == 0) memcpy(ck + (t / blk) * dd, S, sizeof(double) * (size_t)dd);
                    const int64_t r = row0 + t;
                    const double a = exp(orc_load(g, gb_dtype, r * g_stride + h));
                    const double b = orc_load(beta, gb_dtype, r * beta_stride + h);
                    orc_load_row(k, qkv_dtype, r * k_stride + (int64_t)kh * dk, dk, kt);
                    orc_load_row(v, qkv_dtype, r * v_stride + (int64_t)h * dv, dv, vt);
                    for (int64_t i = 0; i < dd; ++i) S[i] *= a;
                    for (int j = 0; j < dv; ++j) p[j] = 0.0;
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j) p[j] += S[(int64_t)i * dv + j] * kt[i];
                    for (int i = 0; i < dk; ++i)
                        for (int j = 0; j < dv; ++j) S[(int64_t)i * dv + j] += b * kt[i] * (vt[j] - p[j]);
                }
                /* backward, block by block from the end */
                for (int64_t i = 0; i < dd; ++i) G[i] = dST ? dST[sbase + i] : 0.0;
                for (int64_t bi = nblk - 1; bi >= 0; --bi) {
                    const int64_t t0 = bi * blk, t1 = (t0 + blk < len) ? t0 + blk : len;
                    /* st[j] = the state entering token t0 + j */
                    memcpy(st, ck + bi * dd, sizeof(double) * (size_t)dd);
                    for (int64_t t = t0; t < t1; ++t) {
                        const int64_t r = row0 + t;
                        const double a = exp(orc_load(g, gb_dtype, r * g_stride + h));
                        const double b = orc_load(beta, gb_dtype, r * beta_stride + h);
                        orc_load_row(k, qkv_dtype, r * k_stride + (int64_t)kh * dk, dk, kt);
                        orc_load_row(v, qkv_dtype, r * v_stride + (int64_t)h * dv, dv, vt);
                        const double* P = st + (t - t0) * dd;
                        double* N = st + (t - t0 + 1) * dd;
                        for (int j = 0; j < dv; ++j) p[j] = 0.0;
                        for (int i = 0; i < dk; ++i)
                            for (int j = 0; j < dv; ++j) p[j] += a * P[(int64_t)i * dv + j] * kt[i];
                        for (int i = 0; i < dk; ++i)
                            for (int j = 0; j < dv; ++j)
                                N[(int64_t)i * dv + j] = a * P[(int64_t)i * dv + j] + b * kt[i] * (vt[j] - p[j]);
                    }
                    for (int64_t t = t1 - 1; t >= t0; --t) {
                        const int64_t r = row0 + t;
                        const double gg = orc_load(g, gb_dtype, r * g_stride + h);
                        const double a = exp(gg);
                        const double b = orc_load(beta, gb_dtype, r * beta_stride + h);
                        orc_load_row(q, qkv_dtype, r * q_stride + (int64_t)kh * dk, dk, qt);
                        orc_load_row(k, qkv_dtype, r * k_stride + (int64_t)kh * dk, dk, kt);
                        orc_load_row(v, qkv_dtype, r * v_stride + (int64_t)h * dv, dv, vt);
                        const double* P = st + (t - t0) * dd;
                        const double* Sn = st + (t - t0 + 1) * dd;
                        for (int j = 0; j < dv; ++j) dov[j] = dout[(r * nv + h) * dv + j];
                        /* read-out: G += q do^T / sqrt(dk); dq = S do / sqrt(dk) */
                        for (int i = 0; i < dk; ++i) {
                            double acc = 0.0;
                            for (int j = 0; j < dv; ++j) {
                                G[(int64_t)i * dv + j] += scale * qt[i] * dov[j];
                                acc += Sn[(int64_t)i * dv + j] * dov[j];
                            }
                            dqv[i] = scale * acc;
                        }
                        /* p = D^T k (D = a P), w = v - p */
                        for (int j = 0; j < dv; ++j) p[j] = 0.0;
                        for (int i = 0; i < dk; ++i)
                            for (int j = 0; j < dv; ++j) p[j] += a * P[(int64_t)i * dv + j] * kt[i];
                        for (int j = 0; j < dv; ++j) w[j] = vt[j] - p[j];
                        /* gk = G^T k; dv = b gk; dp = -dv; dbeta = gk . w */
                        double db = 0.0;
                        for (int j = 0; j < dv; ++j) gk[j] = 0.0;
                        for (int i = 0; i < dk; ++i)
                            for (int j = 0; j < dv; ++j) gk[j] += G[(int64_t)i * dv + j] * kt[i];
                        for (int j = 0; j < dv; ++j) {
                            dvv[(r * nv + h) * dv + j] = b * gk[j];
                            dp[j] = -b * gk[j];
                            db += gk[j] * w[j];
                        }
                        dbeta[r * nv + h] = db;
                        /* dD = G + k dp^T; dk = b G w + D dp; dg = <dD, D>; G <- a dD */
                        double dgs = 0.0;
                        for (int i = 0; i < dk; ++i) {
                            double gw = 0.0, ddp = 0.0;
                            for (int j = 0; j < dv; ++j) {
                                const double Dij = a * P[(int64_t)i * dv + j];
                                const double x = G[(int64_t)i * dv + j] + kt[i] * dp[j];
                                gw += G[(int64_t)i * dv + j] * w[j];
                                ddp += Dij * dp[j];
                                dgs += x * Dij;
                                dD[(int64_t)i * dv + j] = x;
                            }
                            dkv[i] = b * gw + ddp;
                        }
                        dg[r * nv + h] = dgs;
                        for (int64_t i = 0; i < dd; ++i) G[i] = a * dD[i];
                        for (int i = 0; i < dk; ++i) {
                            double* dqr = dq + (r * nk + kh) * dk;
                            double* dkr = dkk + (r * nk + kh) * dk;
                            if (hh == 0) {
                                dqr[i] = dqv[i];
                                dkr[i] = dkv[i];
                            } else {
                                dqr[i] += dqv[i];
                                dkr[i] += dkv[i];
                            }
                        }
                    }
                }
                memcpy(dh0 + sbase, G, sizeof(double) * (size_t)dd);
            }
        }
        free(ck);
        free(st);
        free(G);
        free(dD);
        free(vec);
    }
    return failed ? -1 : 0;
}
