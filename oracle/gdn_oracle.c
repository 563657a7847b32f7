/*
 * gdn_oracle.c - fp64 CPU reference ("oracle") for the Gated DeltaNet state scan.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load or run this file.  It shares no code with the
 * CUDA library: it is a plain, slow, obviously-correct statement of what the
 * scan computes, in double precision, one (sequence, head) stream at a time.
 *
 * Sources (web pages on hybrid / recurrent LLM prefix caching):
 *  - "Tail-Replay: Escaping the Curse of Linear Attention in Prefix Caching
 *    for Hybrid LLMs" (notes page), section 2.3, equation (1):
 *        S_i = T_i S_{i-1} + beta_i v_i k_i^T,  T_i = alpha_i (I - beta_i k_i k_i^T),
 *    and the same section's layout remark: with S in R^{d_v x d_k} the key-space
 *    operator multiplies the state from the right,
 *        S_i = alpha_i S_{i-1} (I - beta_i k_i k_i^T) + beta_i v_i k_i^T.
 *  - same page, section 2.1 table: replay length k = ceil(r m), replay start
 *    a = m - k; section 2.2 steps 2-3: zero the state at the tail start and run
 *    the k tail tokens; section 2.2 worked example (m = 10,000, r = 5 % ->
 *    positions 9,501..10,000).
 *  - "Sparse prefix caching in hybrid and recurrent LLM serving", section 3:
 *    exact states stored at 1 <= c_1 < ... < c_M <= N; on overlap depth d
 *    resume from j = argmax{c_i <= d} and recompute c_j+1 .. d (nothing when
 *    c_j = d; d = 0 saves nothing).
 *
 * Readings where the pages are silent:
 *  - readout o_t = S_t q_t with the post-update state, no scaling;
 *  - the checkpoint at c holds the state after token c;
 *  - with no c_i <= d, resume starts from the initial state (c_0 = 0);
 *  - ceil(r m) is exact integer arithmetic on r = r_num / r_den.
 *
 * Parity pins live in tests/test_oracle_pins.py.  Every function below is
 * pinned there against brute force, closed forms or the pages' own numbers.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* Tail-Replay page, section 2.1 table: k = ceil(r*m), a = m - k, with
 * r = r_num / r_den in [0, 1].  ceil(x/y) for x >= 0, y > 0 is (x + y - 1) / y. */
ORACLE_API int gdn_oracle_replay_plan(int64_t m, int32_t r_num, int32_t r_den, int64_t* a, int64_t* k) {
    if (m < 0 || r_den <= 0 || r_num < 0 || r_num > r_den || !a || !k) return 1;
    if (m > ((int64_t)1 << 40)) return 1; /* keep r_num * m far from overflow */
    int64_t num = (int64_t)r_num * m;
    int64_t kk = (num + (int64_t)r_den - 1) / (int64_t)r_den;
    *k = kk;
    *a = m - kk;
    return 0;
}

/* Sparse prefix caching page, section 3: j = argmax{ c_i : c_i <= d }.
 * Returns the 0-based index j, or -1 when no checkpoint lies at or below d
 * (resume then starts from the initial state). */
ORACLE_API int gdn_oracle_select_ckpt(const int64_t* c, int32_t M, int64_t d, int32_t* j) {
    if (M < 0 || (M > 0 && !c) || !j) return 1;
    int32_t best = -1;
    for (int32_t i = 0; i < M; ++i)
        if (c[i] <= d) best = i;
    *j = best;
    return 0;
}

/* Tail-Replay page, section 2.3, equation (1), right-multiplied form:
 * S <- alpha * S (I - beta k k^T) + beta v k^T.
 * The matrix product S (I - beta k k^T) is formed row by row as
 * S - beta (S k) k^T, i.e. with u = S k. */
static void gdn_step(int dk, int dv, double* S, const double* k, const double* v, double alpha,
                     double beta, double* u) {
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * k[j];
        u[i] = acc;
    }
    for (int i = 0; i < dv; ++i)
        for (int j = 0; j < dk; ++j) {
            double sij = S[(size_t)i * dk + j];
            S[(size_t)i * dk + j] = alpha * (sij - beta * u[i] * k[j]) + beta * v[i] * k[j];
        }
}

/* readout o = S q (post-update state) */
static void gdn_readout(int dk, int dv, const double* S, const double* q, double* o) {
    for (int i = 0; i < dv; ++i) {
        double acc = 0.0;
        for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];
        o[i] = acc;
    }
}

/*
 * One (sequence, head) scan over n tokens.
 *   q, k: [n, dk]; v: [n, dv]; alpha, beta: [n]  (q may be NULL when o is NULL)
 *   S0: [dv, dk] initial state, NULL for zeros
 *   o: [n, dv] readout per token, or NULL
 *   ckpt_pos: n_ckpt strictly increasing 1-based positions in [1, n];
 *   ckpt_out: [n_ckpt, dv, dk] the state after each of those tokens
 *   S_final: [dv, dk] the state after token n (S0 when n = 0)
 * Returns 0, or 1 on invalid arguments.
 */
ORACLE_API int gdn_oracle_scan(int dk, int dv, int64_t n, const double* q, const double* k,
                               const double* v, const double* alpha, const double* beta,
                               const double* S0, double* o, int32_t n_ckpt, const int64_t* ckpt_pos,
                               double* ckpt_out, double* S_final) {
    if (dk <= 0 || dv <= 0 || n < 0 || n_ckpt < 0 || !S_final) return 1;
    if (n > 0 && (!k || !v || !alpha || !beta)) return 1;
    if (o && n > 0 && !q) return 1;
    if (n_ckpt > 0 && (!ckpt_pos || !ckpt_out)) return 1;
    for (int32_t i = 0; i < n_ckpt; ++i) {
        if (ckpt_pos[i] < 1 || ckpt_pos[i] > n) return 1;
        if (i > 0 && ckpt_pos[i] <= ckpt_pos[i - 1]) return 1;
    }
    size_t D = (size_t)dv * dk;
    double* S = (double*)malloc(D * sizeof(double));
    double* u = (double*)malloc((size_t)dv * sizeof(double));
    if (!S || !u) {
        free(S);
        free(u);
        return 2;
    }
    if (S0)
        memcpy(S, S0, D * sizeof(double));
    else
        memset(S, 0, D * sizeof(double));
    int32_t next = 0;
    for (int64_t t = 1; t <= n; ++t) {
        const double* kt = k + (size_t)(t - 1) * dk;
        const double* vt = v + (size_t)(t - 1) * dv;
        gdn_step(dk, dv, S, kt, vt, alpha[t - 1], beta[t - 1], u);
        if (o) gdn_readout(dk, dv, S, q + (size_t)(t - 1) * dk, o + (size_t)(t - 1) * dv);
        if (next < n_ckpt && ckpt_pos[next] == t) {
            memcpy(ckpt_out + (size_t)next * D, S, D * sizeof(double));
            ++next;
        }
    }
    memcpy(S_final, S, D * sizeof(double));
    free(S);
    free(u);
    return 0;
}

/* "Sparse prefix caching in hybrid and recurrent LLM serving", section 3 and section 4, Theorem 2:
 * the least expected recompute over placements of min(M, N) checkpoints, by the plain dynamic
 * programme DP[k][t] = min_{k-1 <= s < t} DP[k-1][s] + C(s, t) with DP[0][0] = 0 (the start is the
 * implicit checkpoint c_0 = 0), C(s, t) = sum_{d=s}^{t-1} w[d] (d - s) read from prefix sums, and
 * the last segment [c_M, N] closed by C(c_M, N + 1).  O(M N^2) with exact integer costs; ties go to
 * the smallest s and t.  Returns 0, or 2 when memory runs out. */
int gdn_oracle_place_dp(const int64_t* w, int64_t N, int32_t M, int64_t* pos, int64_t* cost) {
    if (M > N) M = (int32_t)N;
    const size_t n1 = (size_t)N + 2;
    int64_t* W0 = (int64_t*)calloc(n1, sizeof(int64_t));
    int64_t* W1 = (int64_t*)calloc(n1, sizeof(int64_t));
    int64_t* E = (int64_t*)malloc((size_t)(M + 1) * (size_t)(N + 1) * sizeof(int64_t));
    int64_t* par = (int64_t*)malloc((size_t)(M + 1) * (size_t)(N + 1) * sizeof(int64_t));
    if (!W0 || !W1 || !E || !par) {
        free(W0);
        free(W1);
        free(E);
        free(par);
        return 2;
    }
    for (int64_t d = 0; d <= N; ++d) {
        W0[d + 1] = W0[d] + w[d];
        W1[d + 1] = W1[d] + d * w[d];
    }
#define SEG(s, t) ((W1[t] - W1[s]) - (s) * (W0[t] - W0[s]))
#define AT(a, k, t) a[(size_t)(k) * (size_t)(N + 1) + (size_t)(t)]
    const int64_t INF = INT64_MAX;
    for (int64_t t = 0; t <= N; ++t) AT(E, 0, t) = t == 0 ? 0 : INF;
    for (int32_t k = 1; k <= M; ++k) {
        for (int64_t t = 0; t <= N; ++t) {
            AT(E, k, t) = INF;
            AT(par, k, t) = -1;
            if (t < k) continue;
            for (int64_t s = k - 1; s < t; ++s) {
                if (AT(E, k - 1, s) == INF) continue;
                const int64_t v = AT(E, k - 1, s) + SEG(s, t);
                if (v < AT(E, k, t)) {
                    AT(E, k, t) = v;
                    AT(par, k, t) = s;
                }
            }
        }
    }
    int64_t best = INF, best_t = 0;
    for (int64_t t = M; t <= N; ++t) {
        if (AT(E, M, t) == INF) continue;
        const int64_t v = AT(E, M, t) + SEG(t, N + 1);
        if (v < best) {
            best = v;
            best_t = t;
        }
    }
    int64_t t = best_t;
    for (int32_t k = M; k >= 1; --k) {
        pos[k - 1] = t;
        t = AT(par, k, t);
    }
    *cost = best;
#undef SEG
#undef AT
    free(W0);
    free(W1);
    free(E);
    free(par);
    return 0;
}
