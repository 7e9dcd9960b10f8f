/*
 * Oracle for the causal multi-head differential-attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, fp64 CPU statement of
 * what the GPU path computes. Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may build, load or call it; the
 * product path never does. It shares no code, header, table or helper with the
 * CUDA library, and includes nothing from it.
 *
 * Every step follows the definition on the pages, in their order, with no
 * blocking, fusion or reordering beyond it:
 *
 *   lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)),  l = 1, 2, ...
 *       ("DiffTransformer.py", class DiffTransformer, __init__: the decaying
 *        lambda_init given to each layer, l counted from 1)
 *   lambda = exp(lambda_q1 . lambda_k1) - exp(lambda_q2 . lambda_k2) + lambda_init
 *       ("DiffTransformer.py", MultiHeadDifferentialAttention.forward,
 *        "Compute lambda using reparameterization")
 *   z_c[j] = s * <Q_c[i], K_c[j]>,  s = d^-0.5 on the component dim d
 *       ("DiffTransformer.py", forward, "Compute attention scores";
 *        "LlamaDiffSdpaAttention.py", forward: scaling = (head_dim // 2) ** -0.5)
 *   causal: key j takes part iff j <= i (positions inside one sequence)
 *       ("DiffTransformer.py", forward, "Causal Mask Implementation")
 *   p_c = softmax_j(z_c)  for c = 1, 2 ("Apply softmax to get attention weights")
 *   D = sum_j p_1[j] V[j] - lambda * sum_j p_2[j] V[j]
 *       (output-difference form of "LlamaDiffSdpaAttention.py", forward:
 *        attn1 - lambda_full * attn2; equal by linearity to the map form
 *        (A1 - lambda A2) V of "DiffTransformer.py")
 *   y = D / sqrt(mean_e D[e]^2 + eps) * w * (1 - lambda_init)
 *       ("DiffTransformer.py", forward, "Normalize each head independently
 *        using RMSNorm" and "Scale the normalized output"; eps = 1e-5 there)
 *   Grouped key/value heads: diff head h reads key/value head h / (H / Hkv),
 *   component matched (Q1 with K1, Q2 with K2), as repeat_kv applied to k1, k2
 *   and the values separately in "LlamaDiffSdpaAttention.py", forward.
 *
 * Layouts (token-major, contiguous, fp64):
 *   q [tokens][H][2d]  (Q1 = first d, Q2 = last d of each head: Q.chunk(2, -1))
 *   k [tokens][Hkv][2d], v [tokens][Hkv][dv], out [rows][dv].
 * Sequence s occupies tokens cu[s] .. cu[s+1]-1; positions restart at 0.
 */
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads an OpenMP parallel region of the oracle uses (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

double oracle_lambda_init(int depth) {
    return 0.8 - 0.6 * exp(-0.3 * (double)(depth - 1));
}

/* lambda for n_sets independent parameter sets; each vector has d entries. */
void oracle_lambda(const double* lq1, const double* lk1, const double* lq2, const double* lk2,
                   int n_sets, int d, double lambda_init, double* out) {
    for (int i = 0; i < n_sets; ++i) {
        double a = 0.0, b = 0.0;
        for (int e = 0; e < d; ++e) {
            a += lq1[(size_t)i * d + e] * lk1[(size_t)i * d + e];
            b += lq2[(size_t)i * d + e] * lk2[(size_t)i * d + e];
        }
        out[i] = exp(a) - exp(b) + lambda_init;
    }
}

/*
 * Computes the rows (row_token[r], row_head[r]) for r < n_rows, or every
 * (token, head) row in token-major order when n_rows < 0 (out is then
 * [tokens][H][dv]). lambda_h holds one reparameterised lambda per diff head.
 * Returns 0, or -1 on an argument the definition does not cover.
 */
int oracle_diffattn_rows(int num_seqs, const int* cu_seqlens,
                         int H, int Hkv, int d, int dv,
                         const double* q, const double* k, const double* v,
                         const double* lambda_h, double lambda_init,
                         const double* w, double eps, int causal,
                         int n_rows, const int* row_token, const int* row_head,
                         double* out) {
    if (num_seqs < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d <= 0 || dv <= 0) return -1;
    const int tokens = cu_seqlens[num_seqs];
    int max_len = 0;
    for (int s = 0; s < num_seqs; ++s) {
        int n = cu_seqlens[s + 1] - cu_seqlens[s];
        if (n < 0) return -1;
        if (n > max_len) max_len = n;
    }
    const long total = n_rows < 0 ? (long)tokens * H : (long)n_rows;
    const int group = H / Hkv;
    const double s_scale = 1.0 / sqrt((double)d);
    int bad = 0;

#pragma omp parallel
    {
        double* z = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double* o1 = (double*)malloc(sizeof(double) * (size_t)dv);
        double* o2 = (double*)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            const int t = n_rows < 0 ? (int)(r / H) : row_token[r];
            const int h = n_rows < 0 ? (int)(r % H) : row_head[r];
            double* y = out + (size_t)r * dv;
            if (t < 0 || t >= tokens || h < 0 || h >= H) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            /* the sequence holding token t, and t's position i inside it */
            int sidx = 0;
            while (!(cu_seqlens[sidx] <= t && t < cu_seqlens[sidx + 1])) ++sidx;
            const int start = cu_seqlens[sidx];
            const int len = cu_seqlens[sidx + 1] - start;
            const int i = t - start;
            const int n_keys = causal ? i + 1 : len;
            const int g = h / group;
            const double* qrow = q + ((size_t)t * H + h) * (size_t)(2 * d);
            for (int e = 0; e < dv; ++e) { o1[e] = 0.0; o2[e] = 0.0; }
            /* component 1: Q1 with K1; component 2: Q2 with K2; one shared V */
            for (int c = 0; c < 2; ++c) {
                double* oc = c == 0 ? o1 : o2;
                double m = -INFINITY;
                for (int j = 0; j < n_keys; ++j) {
                    const double* kr = k + ((size_t)(start + j) * Hkv + g) * (size_t)(2 * d) + (size_t)c * d;
                    const double* qr = qrow + (size_t)c * d;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += qr[e] * kr[e];
                    z[j] = s_scale * dot;
                    if (z[j] > m) m = z[j];
                }
                double sum = 0.0;
                for (int j = 0; j < n_keys; ++j) {
                    z[j] = exp(z[j] - m);
                    sum += z[j];
                }
                for (int j = 0; j < n_keys; ++j) {
                    const double p = z[j] / sum;
                    const double* vr = v + ((size_t)(start + j) * Hkv + g) * (size_t)dv;
                    for (int e = 0; e < dv; ++e) oc[e] += p * vr[e];
                }
            }
            const double lam = lambda_h[h];
            double ms = 0.0;
            for (int e = 0; e < dv; ++e) {
                y[e] = o1[e] - lam * o2[e];
                ms += y[e] * y[e];
            }
            ms /= (double)dv;
            const double inv = 1.0 / sqrt(ms + eps);
            for (int e = 0; e < dv; ++e) y[e] = y[e] * inv * w[e] * (1.0 - lambda_init);
        }
        free(z);
        free(o1);
        free(o2);
    }
    return bad ? -1 : 0;
}
