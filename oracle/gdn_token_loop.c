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
