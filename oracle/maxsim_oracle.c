/*
 * Plain fp64 CPU oracle for late-interaction MaxSim scoring.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do. It shares no code, header, table or
 * helper with the CUDA library: it is a direct, slow, loop-by-loop writing
 * of the definitions, so that a reader can check it against the sources by
 * eye.
 *
 * Sources (web pages; cited by title and section):
 *  - "TileMaxSim: IO-Aware GPU MaxSim Scoring with Dimension Tiling and Fused
 *    Product Quantization", paper-daily deep reading:
 *      §1 (problem and motivation): the operator -- for every query token
 *         take the largest similarity over the document's tokens, then add
 *         these maxima over the query tokens;
 *      §2(3): product-quantised scoring through the per-query table
 *         T[i,m,k] = q_i[subspace m] . C[m,k];
 *      §5: variable-length documents and the fixed-length padding waste.
 *  - "FLASH-MAXSIM: IO-Aware Fused Kernels for Late-Interaction Scoring":
 *      Abstract: the same operator; the backward pass reuses the forward
 *         argmax; INT8 x INT8 scoring; variable-length (padding-free)
 *         documents.
 *      Figure 1 / Algorithm 2: a running maximum initialised to -inf,
 *         one scalar score per (query, document) pair.
 *
 * Readings taken where the sources are silent:
 *  - "cosine similarity" is the plain dot product of the given vectors;
 *    inputs are L2-normalised upstream, the operator does not normalise.
 *  - a token outside the document (padding, a CSR neighbour) takes no part
 *    in the maximum (it is not a 0 similarity);
 *  - the argmax is the lowest token index attaining the maximum;
 *  - a document with no tokens scores 0 and has argmax -1;
 *  - INT8: sim(i,j) = fp32( (float)dot_ij * s_d[j] ), m_i = max_j sim(i,j),
 *    score = sum_i s_q[i] * m_i  (per-token symmetric scales, s > 0);
 *  - PQ: subspace m owns the contiguous dimensions [m*d/M, (m+1)*d/M).
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math).
 * All floating point here is IEEE double, except the one fp32 product the
 * INT8 reading fixes.
 */
#include <stdint.h>
#include <math.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Forward MaxSim over documents given as token ranges of a row-major token
 * matrix D[*, d]: document b owns rows tok_start[b] .. tok_start[b]+tok_len[b]-1.
 * The padded layout (row b*Nd, length L_b) and the CSR layout (row
 * offsets[b], length offsets[b+1]-offsets[b]) are both this form.
 *
 *   score[q,b]  = sum_{i<nq} max_{j<L_b} sum_{k<d} Q[q,i,k] * D[start_b + j, k]
 *   argmax[q,b,i] = lowest j attaining that maximum (-1 for an empty doc)
 *   gap[q,b,i]  = (largest sim) - (second largest sim over the other tokens),
 *                 +inf when the document has fewer than two tokens.
 *
 * Q is [n_queries, nq, d]; out is [n_queries, B]; argmax and gap (either may
 * be NULL) are [n_queries, B, nq].
 */
void oracle_maxsim(const double *Q, int n_queries, int nq, int d,
                   const double *D, const int64_t *tok_start, const int64_t *tok_len,
                   int64_t B, double *out, int32_t *argmax, double *gap)
{
    int64_t b;
#pragma omp parallel for schedule(dynamic, 16)
    for (b = 0; b < B; ++b) {
        const double *doc = D + (size_t)tok_start[b] * (size_t)d;
        int64_t L = tok_len[b];
        for (int q = 0; q < n_queries; ++q) {
            double score = 0.0;
            for (int i = 0; i < nq; ++i) {
                const double *qi = Q + ((size_t)q * nq + i) * (size_t)d;
                double best = -INFINITY, second = -INFINITY;
                int32_t best_j = -1;
                for (int64_t j = 0; j < L; ++j) {
                    const double *dj = doc + (size_t)j * (size_t)d;
                    double s = 0.0;
                    for (int k = 0; k < d; ++k) s += qi[k] * dj[k];
                    if (s > best) {          /* strict: keeps the lowest j */
                        second = best;
                        best = s;
                        best_j = (int32_t)j;
                    } else if (s > second) {
                        second = s;
                    }
                }
                size_t o = ((size_t)q * (size_t)B + (size_t)b) * (size_t)nq + (size_t)i;
                if (argmax) argmax[o] = best_j;
                if (gap) gap[o] = (L >= 2) ? (best - second) : INFINITY;
                if (L > 0) score += best;   /* empty document: contributes 0 */
            }
            out[(size_t)q * (size_t)B + (size_t)b] = score;
        }
    }
}

/*
 * Product-quantisation distance table (TileMaxSim §2(3)):
 *   T[i,m,k] = sum_{t < d/M} Q[i, m*(d/M) + t] * C[m,k,t]
 * Q is [nq, d], C is [M, K, d/M], T is [nq, M, K].
 */
void oracle_pq_table(const double *Q, int nq, int d, const double *C, int M, int K,
                     double *T)
{
    int ds = d / M;
    for (int i = 0; i < nq; ++i)
        for (int m = 0; m < M; ++m)
            for (int k = 0; k < K; ++k) {
                double s = 0.0;
                for (int t = 0; t < ds; ++t)
                    s += Q[(size_t)i * d + (size_t)m * ds + t] *
                         C[((size_t)m * K + k) * ds + t];
                T[((size_t)i * M + m) * K + k] = s;
            }
}

/*
 * PQ scoring by table lookup (TileMaxSim §2(3)):
 *   sim(i,j)  = sum_{m<M} T[i, m, codes[j,m]]
 *   score[b]  = sum_i max_{j in doc b} sim(i,j)
 * codes is [T_tok, M] uint8 (K <= 256); offsets is [B+1].
 */
void oracle_maxsim_pq(const double *T, int nq, int M, int K, const uint8_t *codes,
                      const int64_t *offsets, int64_t B, double *out, int32_t *argmax)
{
    int64_t b;
#pragma omp parallel for schedule(dynamic, 64)
    for (b = 0; b < B; ++b) {
        int64_t j0 = offsets[b], L = offsets[b + 1] - offsets[b];
        double score = 0.0;
        for (int i = 0; i < nq; ++i) {
            double best = -INFINITY;
            int32_t best_j = -1;
            for (int64_t j = 0; j < L; ++j) {
                const uint8_t *c = codes + (size_t)(j0 + j) * (size_t)M;
                double s = 0.0;
                for (int m = 0; m < M; ++m)
                    s += T[((size_t)i * M + m) * K + c[m]];
                if (s > best) { best = s; best_j = (int32_t)j; }
            }
            if (argmax) argmax[(size_t)b * nq + i] = best_j;
            if (L > 0) score += best;
        }
        out[b] = score;
    }
}

/*
 * INT8 x INT8 scoring (FLASH-MAXSIM, Abstract: INT8xINT8 quantisation), with
 * per-token symmetric scales:
 *   dot(i,j) = sum_k Qi8[i,k] * Di8[j,k]                    (exact integer)
 *   sim(i,j) = (float)dot(i,j) * s_d[j]                     (one fp32 multiply, RN)
 *   m_i      = max_j sim(i,j)        (fp32 compare; lowest j on ties)
 *   score[b] = sum_i s_q[i] * m_i    (accumulated here in fp64)
 * maxv, maxdot and argmax (any may be NULL) are [B, nq]: m_i, dot(i, argmax)
 * and argmax. An empty document gives score 0, maxv 0, maxdot 0, argmax -1.
 */
void oracle_maxsim_i8(const int8_t *Q, const float *s_q, int nq, int d,
                      const int8_t *D, const float *s_d, const int64_t *offsets,
                      int64_t B, double *out, float *maxv, int32_t *maxdot,
                      int32_t *argmax)
{
    int64_t b;
#pragma omp parallel for schedule(dynamic, 64)
    for (b = 0; b < B; ++b) {
        int64_t j0 = offsets[b], L = offsets[b + 1] - offsets[b];
        double score = 0.0;
        for (int i = 0; i < nq; ++i) {
            float best = 0.0f;
            int64_t best_dot = 0;
            int32_t best_j = -1;
            for (int64_t j = 0; j < L; ++j) {
                const int8_t *qi = Q + (size_t)i * d;
                const int8_t *dj = D + (size_t)(j0 + j) * (size_t)d;
                int64_t dot = 0;
                for (int k = 0; k < d; ++k) dot += (int64_t)qi[k] * (int64_t)dj[k];
                volatile float prod = (float)dot * s_d[j0 + j];
                float s = prod;
                if (best_j < 0 || s > best) { best = s; best_dot = dot; best_j = (int32_t)j; }
            }
            size_t o = (size_t)b * nq + i;
            if (maxv) maxv[o] = best;
            if (maxdot) maxdot[o] = (int32_t)best_dot;
            if (argmax) argmax[o] = best_j;
            if (L > 0) score += (double)s_q[i] * (double)best;
        }
        out[b] = score;
    }
}

/*
 * Backward pass through the forward argmax (FLASH-MAXSIM, Abstract: the
 * backward reuses the forward argmax). With loss = sum_{q,b} dS[q,b] *
 * score[q,b] and a = argmax[q,b,i] (doc-local; -1 for an empty doc):
 *   dQ[q,i,:]         = sum_b dS[q,b] * D[start_b + a, :]
 *   dD[start_b + j,:] = sum_q dS[q,b] * sum_{i : a(q,b,i) = j} Q[q,i,:]
 * dD has the row layout of D; rows no argmax points at stay 0. The caller
 * zeroes dQ and dD. Written as plain scatter loops over (q, b, i).
 */
void oracle_backward(const double *Q, int n_queries, int nq, int d,
                     const double *D, const int64_t *tok_start, int64_t B,
                     const int32_t *argmax, const double *dS, double *dQ, double *dD)
{
    for (int q = 0; q < n_queries; ++q)
        for (int64_t b = 0; b < B; ++b) {
            double g = dS[(size_t)q * (size_t)B + (size_t)b];
            for (int i = 0; i < nq; ++i) {
                int32_t a = argmax[((size_t)q * (size_t)B + (size_t)b) * (size_t)nq + (size_t)i];
                if (a < 0) continue;
                const double *drow = D + (size_t)(tok_start[b] + a) * (size_t)d;
                const double *qrow = Q + ((size_t)q * nq + i) * (size_t)d;
                double *dq = dQ + ((size_t)q * nq + i) * (size_t)d;
                double *dd = dD + (size_t)(tok_start[b] + a) * (size_t)d;
                for (int k = 0; k < d; ++k) {
                    dq[k] += g * drow[k];
                    dd[k] += g * qrow[k];
                }
            }
        }
}
