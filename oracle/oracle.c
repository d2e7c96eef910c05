/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the MoE layer
 * "dispatch -> FFN -> combine".
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * library in dispatch_ffn_combine_gb300/csrc.
 *
 * What the layer computes (mKernel README, kernel table, row "MoE Dispatch +
 * FFN + Combine"): tokens are routed to experts, every expert runs its FFN
 * "gemm1 -> SwiGLU -> gemm2", and the weighted expert outputs are combined
 * back into each token's row.  The pages leave the router, the gating
 * convention and all precisions open; the readings used here are:
 *
 *   R1  gate logit l[t,e] = sum_i x[t,i] * Wg[e,i] (+ bias[e]) in fp32, in a
 *       fixed order: 32 interleaved partial sums s_j (j = 0..31), each a
 *       sequential chain of correctly rounded fmaf over i = j, j+32, j+64, ...;
 *       then a pairwise tree s_j += s_{j+off} for off = 16, 8, 4, 2, 1 (j < off);
 *       the logit is s_0, plus bias[e] (one fp32 add) when a bias is given.
 *   R2  the k experts are chosen on the logits (softmax is monotone).
 *   R3  ties: the lower expert id wins (fp32 ==, so +0 == -0).
 *   R4  slot order j within a token: descending logit, ties lower id first.
 *   R5  inside an expert's block, rows are in ascending token order.
 *   R6  h = silu(x W1^T) * (x W3^T); W1 = gate, W3 = up; W1, W3 are [E][f][d],
 *       W2 is [E][d][f] (out x in, like a linear layer's weight).
 *   w   w_j = exp(l_j - l_0) / sum_j' exp(l_j' - l_0) over the k chosen
 *       (softmax over all E, renormalised over the chosen k: the same number).
 *
 * Precision.  The router logits are fp32 in the R1 order, because they decide
 * integers (which experts) and both sides must take that decision in the same
 * precision.  Everything after the choice (weights, FFN, combine) is fp64 here:
 * the oracle is the exact definition, the GPU's bf16 intermediates are the
 * approximation whose error the parity tolerance bounds.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -fPIC -shared.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> fp32 is exact: the 16 bits are the high half of the fp32 pattern. */
static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* One gate logit in the R1 order. */
static float logit_r1(const uint16_t* xrow, const float* wrow, int d, const float* bias, int e) {
    float s[32];
    for (int j = 0; j < 32; ++j) {
        float acc = 0.0f;
        for (int i = j; i < d; i += 32)
            acc = fmaf(bf16_bits_to_float(xrow[i]), wrow[i], acc);
        s[j] = acc;
    }
    for (int off = 16; off >= 1; off >>= 1)
        for (int j = 0; j < off; ++j)
            s[j] = s[j] + s[j + off];
    float l = s[0];
    if (bias) l = l + bias[e];
    return l;
}

/* logits[t][e], fp32, R1 order.  x: bf16 bits [T][d]; wg: [E][d]; bias: [E] or NULL. */
void oracle_router_logits(const uint16_t* x, const float* wg, const float* bias,
                          int64_t T, int d, int E, float* logits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e)
            logits[t * E + e] = logit_r1(x + t * (int64_t)d, wg + (int64_t)e * d, d, bias, e);
}

/* The same logits in fp64 (exact products, fp64 sums in index order).  Used only
 * to flag near-ties, i.e. tokens whose choice could flip under another order. */
void oracle_router_logits_f64(const uint16_t* x, const float* wg, const float* bias,
                              int64_t T, int d, int E, double* logits) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < d; ++i)
                acc += (double)bf16_bits_to_float(x[t * d + i]) * (double)wg[(int64_t)e * d + i];
            if (bias) acc += (double)bias[e];
            logits[t * E + e] = acc;
        }
}

/* Top-k on one token's logits (R2-R4) by k rounds of "largest remaining,
 * lower id on ties", then the renormalised softmax weights in fp64. */
static void topk_one(const float* l, int E, int k, int32_t* ids, double* w) {
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            int taken = 0;
            for (int q = 0; q < j; ++q)
                if (ids[q] == e) taken = 1;
            if (taken) continue;
            if (best < 0 || l[e] > l[best]) best = e; /* strict >: equal keeps the lower id */
        }
        ids[j] = best;
    }
    double top = (double)l[ids[0]];
    double z = 0.0;
    for (int j = 0; j < k; ++j) z += exp((double)l[ids[j]] - top);
    for (int j = 0; j < k; ++j) w[j] = exp((double)l[ids[j]] - top) / z;
}

void oracle_topk(const float* logits, int64_t T, int E, int k, int32_t* ids, double* w) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        topk_one(logits + t * E, E, k, ids + t * k, w + t * k);
}

/* Dispatch by plain counting (R5): counts, exclusive-scan offsets, then walk the
 * tokens in ascending order and hand out the next free row of each expert. */
void oracle_dispatch(const int32_t* ids, int64_t T, int E, int k,
                     int32_t* counts, int32_t* offsets, int32_t* row_token, int32_t* slot_row) {
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t q = 0; q < T * k; ++q) counts[ids[q]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int64_t t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int e = ids[t * k + j];
            int32_t r = offsets[e] + fill[e];
            fill[e] += 1;
            row_token[r] = (int32_t)t;
            slot_row[t * k + j] = r;
        }
    free(fill);
}

/* One expert's FFN on one token row, fp64 (R6):
 *   g = W1_e x,  u = W3_e x,  h = silu(g) * u,  out = W2_e h.               */
static void expert_ffn_one(const double* xd, const uint16_t* w1e, const uint16_t* w3e,
                           const uint16_t* w2e, int d, int f, double* h, double* out) {
    for (int n = 0; n < f; ++n) {
        double g = 0.0, u = 0.0;
        const uint16_t* r1 = w1e + (int64_t)n * d;
        const uint16_t* r3 = w3e + (int64_t)n * d;
        for (int i = 0; i < d; ++i) {
            g += (double)bf16_bits_to_float(r1[i]) * xd[i];
            u += (double)bf16_bits_to_float(r3[i]) * xd[i];
        }
        double silu = g / (1.0 + exp(-g));
        h[n] = silu * u;
    }
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        const uint16_t* r2 = w2e + (int64_t)c * f;
        for (int n = 0; n < f; ++n) acc += (double)bf16_bits_to_float(r2[n]) * h[n];
        out[c] = acc;
    }
}

/* Expert FFN on given (token, expert) pairs: out[p][d] = FFN_{expert[p]}(x[token[p]]). */
void oracle_expert_ffn(const uint16_t* x, const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                       int d, int f, const int64_t* token, const int32_t* expert, int64_t npairs,
                       double* out) {
#pragma omp parallel
    {
        double* xd = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)f);
#pragma omp for schedule(dynamic, 1)
        for (int64_t p = 0; p < npairs; ++p) {
            int64_t t = token[p];
            int64_t e = expert[p];
            for (int i = 0; i < d; ++i) xd[i] = (double)bf16_bits_to_float(x[t * d + i]);
            expert_ffn_one(xd, w1 + e * f * d, w3 + e * f * d, w2 + e * d * f, d, f, h, out + p * d);
        }
        free(xd);
        free(h);
    }
}

/* Per-expert linear map on given (token, expert) pairs, fp64: the grouped GEMM
 * of the README's "MoE Dispatch + GEMM" row (each expert multiplies the token
 * rows it receives by its weight):
 *   out[p][c] = sum_i W_e[c][i] * x_t[i],  e = expert[p], t = token[p],
 *   W: [E][n][d] (out x in, like a linear layer's weight).                   */
void oracle_expert_linear(const uint16_t* x, const uint16_t* w, int d, int n,
                          const int64_t* token, const int32_t* expert, int64_t npairs, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < npairs; ++p) {
        const uint16_t* xrow = x + token[p] * d;
        const uint16_t* we = w + (int64_t)expert[p] * n * d;
        for (int c = 0; c < n; ++c) {
            const uint16_t* wrow = we + (int64_t)c * d;
            double acc = 0.0;
            for (int i = 0; i < d; ++i) acc += (double)bf16_bits_to_float(wrow[i]) * (double)bf16_bits_to_float(xrow[i]);
            out[p * n + c] = acc;
        }
    }
}

/* The whole layer for a list of tokens (all of them, or a sample: tokens are
 * independent once the weights are fixed).  For each listed token t:
 *   route (R1-R4 + weights), run its k experts, y_t = sum_j w_j * out_j in j
 *   order, fp64.  y: [ntok][d]; ids_out [ntok][k] and w_out [ntok][k] may be NULL. */
void oracle_layer(const uint16_t* x, const float* wg, const float* bias,
                  const uint16_t* w1, const uint16_t* w3, const uint16_t* w2,
                  int64_t T, int d, int E, int k, int f,
                  const int64_t* tokens, int64_t ntok,
                  double* y, int32_t* ids_out, double* w_out) {
    (void)T;
#pragma omp parallel
    {
        float* l = (float*)malloc(sizeof(float) * (size_t)E);
        int32_t ids[64];
        double w[64];
        double* xd = (double*)malloc(sizeof(double) * (size_t)d);
        double* h = (double*)malloc(sizeof(double) * (size_t)f);
        double* out = (double*)malloc(sizeof(double) * (size_t)d);
#pragma omp for schedule(dynamic, 1)
        for (int64_t q = 0; q < ntok; ++q) {
            int64_t t = tokens[q];
            const uint16_t* xrow = x + t * d;
            for (int e = 0; e < E; ++e) l[e] = logit_r1(xrow, wg + (int64_t)e * d, d, bias, e);
            topk_one(l, E, k, ids, w);
            for (int i = 0; i < d; ++i) xd[i] = (double)bf16_bits_to_float(xrow[i]);
            double* yrow = y + q * d;
            for (int c = 0; c < d; ++c) yrow[c] = 0.0;
            for (int j = 0; j < k; ++j) {
                int64_t e = ids[j];
                expert_ffn_one(xd, w1 + e * f * d, w3 + e * f * d, w2 + e * d * f, d, f, h, out);
                for (int c = 0; c < d; ++c) yrow[c] += w[j] * out[c];
            }
            if (ids_out)
                for (int j = 0; j < k; ++j) ids_out[q * k + j] = ids[j];
            if (w_out)
                for (int j = 0; j < k; ++j) w_out[q * k + j] = w[j];
        }
        free(l);
        free(xd);
        free(h);
        free(out);
    }
}
