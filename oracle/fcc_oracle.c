/*
 * fcc_oracle.c -- CPU fp64 oracle for the fused GEMM + collective operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may call,
 * link or load this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA path.
 *
 * Every routine is the plain definition of its operator written out as loops
 * over the output elements, in double precision, over bfloat16 inputs widened
 * exactly to double.  Products of two bfloat16 values are exact in double;
 * the sums carry at most about K' * 2^-53 relative error, so for the shapes
 * used here the result is the exact real-number result to ~1e-12.
 *
 * Operators (the pages name them; the index formulas are the plain readings):
 *   - GEMM + ReduceScatter and GEMM + AllReduce: the mKernel article (UCCL
 *     project news page), section "A fuzios kernelek hangja", list of the five
 *     fused kernels; also "Optimizing Distributed ML Communication with Fused
 *     Computation-Collective Operations" (SC24), abstract: a computation fused
 *     with the collective that consumes its output.
 *   - GEMV + AllReduce: the SC24 abstract, the Transformer operator.
 *   - AllGather + GEMM: the mKernel article, fused kernel list.
 *   - MoE Dispatch + GEMM: the mKernel article, fused kernel list; the SC24
 *     abstract, GEMM + All-to-All for MoE.
 *   - MoE combine (the return all-to-all and the gate-weighted sum): the SC24
 *     abstract, GEMM + All-to-All for MoE.
 * Rows are row-major and contiguous: A_r is [M,K], B_r is [K,N]; shard j of an
 * M-row result is the contiguous row block [j*M/R, (j+1)*M/R).
 *
 * Parallelism: OpenMP over independent output rows only; the arithmetic of
 * each output element is the sequential sum in the order stated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bfloat16 bit pattern to double. */
static double bf16_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Rank sum of R products, for selected rows of the M x N result:
 *   S[row][n] = sum_{r=0}^{R-1} sum_{k=0}^{K-1} A_r[row][k] * B_r[k][n]
 * summed r-major, then k.  out is [nrows][N]; rows[i] is a row of S in
 * [0, M).  This is the all-reduce result (every rank receives all of S).
 * Returns 0 on success, 1 on a bad argument.
 */
int orc_rank_sum_rows(int R, const uint16_t *const *A, const uint16_t *const *B,
                      int64_t M, int64_t N, int64_t K,
                      const int64_t *rows, int64_t nrows, double *out)
{
    if (R < 1 || M < 0 || N < 0 || K < 0 || nrows < 0)
        return 1;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M)
            return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row = rows[i];
        double *o = out + i * N;
        for (int64_t n = 0; n < N; ++n)
            o[n] = 0.0;
        for (int r = 0; r < R; ++r) {
            const uint16_t *a = A[r] + row * K;
            for (int64_t k = 0; k < K; ++k) {
                const double av = bf16_to_double(a[k]);
                const uint16_t *b = B[r] + k * N;
                for (int64_t n = 0; n < N; ++n)
                    o[n] += av * bf16_to_double(b[n]);
            }
        }
    }
    return 0;
}

/*
 * GEMM + ReduceScatter, shard j: out_j[i][n] = S[j*M/R + i][n] for the
 * shard-local rows listed in local_rows (each in [0, M/R)).
 */
int orc_gemm_rs_rows(int R, const uint16_t *const *A, const uint16_t *const *B,
                     int64_t M, int64_t N, int64_t K, int j,
                     const int64_t *local_rows, int64_t nrows, double *out)
{
    if (R < 1 || M % R != 0 || j < 0 || j >= R || nrows < 0)
        return 1;
    const int64_t Ms = M / R;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows > 0 ? nrows : 1));
    if (rows == NULL)
        return 1;
    for (int64_t i = 0; i < nrows; ++i) {
        if (local_rows[i] < 0 || local_rows[i] >= Ms) {
            free(rows);
            return 1;
        }
        rows[i] = (int64_t)j * Ms + local_rows[i];
    }
    const int rc = orc_rank_sum_rows(R, A, B, M, N, K, rows, nrows, out);
    free(rows);
    return rc;
}

/*
 * AllGather + GEMM for rank r, selected rows:
 *   X = [X_0; X_1; ...; X_{R-1}]  (each X_s is [M/R, K], so X is [M, K])
 *   out_r[row][n] = sum_k X[row][k] * B_r[k][n]
 */
int orc_ag_gemm_rows(int R, const uint16_t *const *X, const uint16_t *const *B,
                     int64_t M, int64_t N, int64_t K, int r,
                     const int64_t *rows, int64_t nrows, double *out)
{
    if (R < 1 || M % R != 0 || r < 0 || r >= R || nrows < 0)
        return 1;
    const int64_t Ms = M / R;
    for (int64_t i = 0; i < nrows; ++i)
        if (rows[i] < 0 || rows[i] >= M)
            return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t row = rows[i];
        const uint16_t *x = X[row / Ms] + (row % Ms) * K;   /* the gather */
        double *o = out + i * N;
        for (int64_t n = 0; n < N; ++n)
            o[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double xv = bf16_to_double(x[k]);
            const uint16_t *b = B[r] + k * N;
            for (int64_t n = 0; n < N; ++n)
                o[n] += xv * bf16_to_double(b[n]);
        }
    }
    return 0;
}

/*
 * MoE router, per token (ntok tokens, E logits each, float32):
 *   idx[t][s], s < topk: the experts with the largest logits, largest first;
 *     among equal logits the lower expert index comes first.  Softmax is
 *     strictly increasing, so ranking by logit is ranking by probability.
 *   gate[t][s] = exp(l_e - max_l) / sum_{e'} exp(l_e' - max_l), the softmax
 *     probability of the chosen expert over all E experts (not renormalised
 *     over the chosen ones).
 * Logits must be finite.
 */
int orc_moe_route(int64_t ntok, int E, int topk, const float *logits,
                  int32_t *idx, double *gate)
{
    if (ntok < 0 || E < 1 || topk < 1 || topk > E || E > 4096)
        return 1;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < ntok; ++t) {
        const float *l = logits + t * E;
        unsigned char taken[4096];
        memset(taken, 0, (size_t)E);
        double mx = (double)l[0];
        for (int e = 1; e < E; ++e)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        double den = 0.0;
        for (int e = 0; e < E; ++e)
            den += exp((double)l[e] - mx);
        for (int s = 0; s < topk; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])   /* strict: ties keep the lower index */
                    best = e;
            }
            taken[best] = 1;
            idx[t * topk + s] = best;
            gate[t * topk + s] = exp((double)l[best] - mx) / den;
        }
    }
    return 0;
}

/*
 * MoE dispatch (the all-to-all), as a stable counting sort by expert.
 *   Assignments a = (s, t, slot) in lexicographic order, s < R source ranks,
 *   t < T tokens, slot < topk; expert e(a) = idx[(s*T + t)*topk + slot].
 *   Expert e lives on rank dest(e) = e / (E/R) (E/R consecutive experts each).
 *   counts[e]          = #{a : e(a) = e}
 *   base[e]            = sum of counts[e'] over dest(e)'s experts e' < e
 *   recv_row[a]        = base[e(a)] + #{a' < a : e(a') = e(a)}
 *   recv_src[d][row]   = s*T + t of the assignment placed at (d, row)
 *   recv_expert[d][row]= e of that assignment
 *   send_counts[s*R+d] = #{a from s : dest(e(a)) = d}
 *   recv_counts[d]     = rows received by d
 * recv_src/recv_expert are [R][cap]; rows past recv_counts[d] are set to -1.
 * Returns 2 when some rank receives more than cap rows.
 */
int orc_moe_dispatch(int R, int64_t T, int E, int topk, const int32_t *idx,
                     int64_t cap, int32_t *counts, int32_t *send_counts,
                     int32_t *recv_counts, int32_t *recv_row,
                     int32_t *recv_src, int32_t *recv_expert)
{
    if (R < 1 || E < R || E % R != 0 || T < 0 || topk < 1 || cap < 0)
        return 1;
    const int Eloc = E / R;
    const int64_t nassign = (int64_t)R * T * topk;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int i = 0; i < R * R; ++i)
        send_counts[i] = 0;
    for (int d = 0; d < R; ++d)
        recv_counts[d] = 0;
    for (int64_t a = 0; a < nassign; ++a) {
        const int e = idx[a];
        if (e < 0 || e >= E)
            return 1;
        counts[e] += 1;
    }
    int64_t base[4096];
    if (E > 4096)
        return 1;
    for (int d = 0; d < R; ++d) {
        int64_t acc = 0;
        for (int e = d * Eloc; e < (d + 1) * Eloc; ++e) {
            base[e] = acc;
            acc += counts[e];
        }
        if (acc > cap)
            return 2;
        recv_counts[d] = (int32_t)acc;
    }
    for (int64_t i = 0; i < (int64_t)R * cap; ++i) {
        recv_src[i] = -1;
        recv_expert[i] = -1;
    }
    int64_t seen[4096];
    for (int e = 0; e < E; ++e)
        seen[e] = 0;
    for (int s = 0; s < R; ++s) {
        for (int64_t t = 0; t < T; ++t) {
            for (int slot = 0; slot < topk; ++slot) {
                const int64_t a = ((int64_t)s * T + t) * topk + slot;
                const int e = idx[a];
                const int d = e / Eloc;
                const int64_t row = base[e] + seen[e];
                seen[e] += 1;
                recv_row[a] = (int32_t)row;
                recv_src[(int64_t)d * cap + row] = (int32_t)((int64_t)s * T + t);
                recv_expert[(int64_t)d * cap + row] = e;
                send_counts[s * R + d] += 1;
            }
        }
    }
    return 0;
}

/*
 * Expert GEMM rows: out[i][f] = sum_h X_{src_rank[i]}[src_tok[i]][h] * W_{expert[i]}[h][f]
 * (the dispatched token row times its expert's weight; no gate applied).
 */
int orc_moe_expert_rows(int R, const uint16_t *const *X, const uint16_t *const *W,
                        int64_t T, int64_t H, int64_t F, int E,
                        const int32_t *src_rank, const int32_t *src_tok,
                        const int32_t *expert, int64_t nrows, double *out)
{
    if (R < 1 || E < 1 || nrows < 0)
        return 1;
    for (int64_t i = 0; i < nrows; ++i)
        if (src_rank[i] < 0 || src_rank[i] >= R || src_tok[i] < 0 || src_tok[i] >= T ||
            expert[i] < 0 || expert[i] >= E)
            return 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        const uint16_t *x = X[src_rank[i]] + (int64_t)src_tok[i] * H;
        const uint16_t *w = W[expert[i]];
        double *o = out + i * F;
        for (int64_t f = 0; f < F; ++f)
            o[f] = 0.0;
        for (int64_t h = 0; h < H; ++h) {
            const double xv = bf16_to_double(x[h]);
            const uint16_t *wr = w + h * F;
            for (int64_t f = 0; f < F; ++f)
                o[f] += xv * bf16_to_double(wr[f]);
        }
    }
    return 0;
}

/*
 * MoE combine: the return all-to-all and the gate-weighted sum of each
 * token's top-k expert outputs (the step after the expert GEMM in the SC24
 * paper's GEMM + All-to-All operator for MoE):
 *   out[i][f] = sum over j < topk with idx[i][j] >= 0 of
 *               gate[i][j] * sum_h X_{src_rank[i]}[src_tok[i]][h] * W_{idx[i][j]}[h][f]
 * with the slots added in order j = 0, 1, ...  idx[i][j] < 0 marks a slot whose
 * row was not received (dropped for capacity): it adds nothing.
 */
int orc_moe_combine_rows(int R, const uint16_t *const *X, const uint16_t *const *W,
                         int64_t T, int64_t H, int64_t F, int E, int topk,
                         const int32_t *src_rank, const int32_t *src_tok,
                         const int32_t *idx, const double *gate, int64_t n, double *out)
{
    if (R < 1 || E < 1 || topk < 1 || n < 0)
        return 1;
    for (int64_t i = 0; i < n; ++i) {
        if (src_rank[i] < 0 || src_rank[i] >= R || src_tok[i] < 0 || src_tok[i] >= T)
            return 1;
        for (int j = 0; j < topk; ++j)
            if (idx[i * topk + j] >= E)
                return 1;
    }
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t *x = X[src_rank[i]] + (int64_t)src_tok[i] * H;
        double *o = out + i * F;
        double *row = (double *)malloc((size_t)F * sizeof(double));
        if (row == NULL) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        for (int64_t f = 0; f < F; ++f)
            o[f] = 0.0;
        for (int j = 0; j < topk; ++j) {
            const int e = idx[i * topk + j];
            if (e < 0)
                continue;
            /* the slot's expert row x . W_e, each element summed over h in order */
            const uint16_t *w = W[e];
            for (int64_t f = 0; f < F; ++f)
                row[f] = 0.0;
            for (int64_t h = 0; h < H; ++h) {
                const double xv = bf16_to_double(x[h]);
                const uint16_t *wr = w + h * F;
                for (int64_t f = 0; f < F; ++f)
                    row[f] += xv * bf16_to_double(wr[f]);
            }
            const double g = gate[i * topk + j];
            for (int64_t f = 0; f < F; ++f)
                o[f] += g * row[f];
        }
        free(row);
    }
    return bad ? 3 : 0;
}

/*
 * Embedding + All-to-All (SC24 abstract: the embedding + All-to-All operator
 * for DLRM).  Table tau is a [V, D] matrix; bag (tau, g) of global sample g
 * is the index list indices_tau[offsets_tau[g] .. offsets_tau[g+1]).  The
 * pooled vector of a bag is the sum of its rows (an empty bag gives zeros):
 *   out[i][d] = sum over k in bag (bag_table[i], bag_sample[i]) of
 *               table_{bag_table[i]}[indices[k]][d]
 * summed in bag order.  The all-to-all that sends sample g's vectors to its
 * rank is a placement of these rows, done by the Python wrapper.
 */
int orc_embedding_bags(int ntables, const uint16_t *const *tables, int64_t V, int64_t D,
                       const int32_t *const *offsets, const int32_t *const *indices,
                       int64_t nsamples, const int32_t *bag_table, const int64_t *bag_sample,
                       int64_t nbags, double *out)
{
    if (ntables < 1 || V < 1 || D < 1 || nbags < 0)
        return 1;
    for (int64_t i = 0; i < nbags; ++i) {
        const int tau = bag_table[i];
        const int64_t g = bag_sample[i];
        if (tau < 0 || tau >= ntables || g < 0 || g >= nsamples)
            return 1;
        const int32_t k0 = offsets[tau][g], k1 = offsets[tau][g + 1];
        if (k0 < 0 || k1 < k0)
            return 1;
        for (int32_t k = k0; k < k1; ++k)
            if (indices[tau][k] < 0 || indices[tau][k] >= V)
                return 1;
    }
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nbags; ++i) {
        const int tau = bag_table[i];
        const int64_t g = bag_sample[i];
        double *o = out + i * D;
        for (int64_t d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int32_t k = offsets[tau][g]; k < offsets[tau][g + 1]; ++k) {
            const uint16_t *row = tables[tau] + (int64_t)indices[tau][k] * D;
            for (int64_t d = 0; d < D; ++d)
                o[d] += bf16_to_double(row[d]);
        }
    }
    return 0;
}

/*
 * Ring attention (the mKernel article's fused kernel list names Ring
 * Attention; read as exact softmax attention of each rank's queries over the
 * keys and values of all R sequence shards, which the ring brings round).
 * The global sequence is shard-major: rank q's row t is position q*S + t.
 *   s_j   = (Q_r[i][h] . K_{j/S}[j%S][h]) / sqrt(d)
 *   O_r[i][h][:] = sum_j exp(s_j - max s) V_{j/S}[j%S][h][:] / sum_j exp(s_j - max s)
 * over all positions j (causal: only j <= r*S + i).  Q, K, V, O rows are
 * [S][H][d].  One output row (rank[i], row[i], head[i]) per entry.
 */
int orc_attention_rows(int R, const uint16_t *const *Q, const uint16_t *const *K,
                       const uint16_t *const *V, int64_t S, int H, int64_t d, int causal,
                       int64_t n, const int32_t *rank, const int64_t *row, const int32_t *head,
                       double *out)
{
    if (R < 1 || S < 1 || H < 1 || d < 1 || n < 0)
        return 1;
    for (int64_t i = 0; i < n; ++i)
        if (rank[i] < 0 || rank[i] >= R || row[i] < 0 || row[i] >= S || head[i] < 0 ||
            head[i] >= H)
            return 1;
    const int64_t L = (int64_t)R * S;
    const double scale = 1.0 / sqrt((double)d);
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        double *s = (double *)malloc((size_t)L * sizeof(double));
        if (s == NULL) {
#pragma omp atomic write
            bad = 1;
            continue;
        }
        const int r = rank[i], h = head[i];
        const uint16_t *q = Q[r] + (row[i] * H + h) * d;
        const int64_t pos = (int64_t)r * S + row[i];
        const int64_t jend = causal ? pos + 1 : L;
        double m = -INFINITY;
        for (int64_t j = 0; j < jend; ++j) {
            const uint16_t *k = K[j / S] + ((j % S) * H + h) * d;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += bf16_to_double(q[c]) * bf16_to_double(k[c]);
            s[j] = dot * scale;
            if (s[j] > m)
                m = s[j];
        }
        double *o = out + i * d;
        for (int64_t c = 0; c < d; ++c)
            o[c] = 0.0;
        double l = 0.0;
        for (int64_t j = 0; j < jend; ++j) {
            const double p = exp(s[j] - m);
            l += p;
            const uint16_t *v = V[j / S] + ((j % S) * H + h) * d;
            for (int64_t c = 0; c < d; ++c)
                o[c] += p * bf16_to_double(v[c]);
        }
        for (int64_t c = 0; c < d; ++c)
            o[c] /= l;
        free(s);
    }
    return bad ? 3 : 0;
}
