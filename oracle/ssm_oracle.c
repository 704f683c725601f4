/*
 * fp64 CPU oracle for the Mamba-layer speculative verify/commit step.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, sequential
 * definition that the CUDA path is checked against. Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load it. It shares no code,
 * header, table or helper with the CUDA library and must never be reached
 * from the product path.
 *
 * What it computes, and where the pages say so. The pages are the paper
 * "The Mamba in the Llama: Distilling and Accelerating Hybrid Models" (its
 * abstract) and two news summaries of it: "Llama 3+Mamba ... 推理速度提升1.6倍"
 * (taipingwang.com, below "the news summary") and the skycaiji.com method
 * overview (below "the method overview").
 *
 *  - The method overview describes Mamba's continuous-time state space model
 *    as producing a discrete-time linear RNN. The discretisation used here is
 *    zero-order hold on A and Euler on B, per head h and draft token t:
 *        a_t       = exp(dt_t * A_h)
 *        S_t[p][n] = a_t * S_{t-1}[p][n] + (dt_t * x_t[p]) * B_t[n]
 *        y_t[p]    = sum_n C_t[n] * S_t[p][n] + D_h * x_t[p]
 *    with C, B, x in the roles of attention's query, key and value (the
 *    attention-to-linear-RNN correspondence in the news summary's
 *    initialisation section and the method overview).
 *    The state S is stored [P][N]: row p is the head-dimension channel, column
 *    n the state channel, so the update is the outer product x_t B_t^T.
 *  - Speculative decoding (news summary, speculative-decoding section): the
 *    Mamba layer processes the K draft tokens one after another from the
 *    cached state; accepted tokens advance the state without storing the
 *    intermediate states; at the first wrong token processing stops and the
 *    state is rolled back to the last accepted token. Here accept_len[b] = j
 *    counts the accepted draft tokens, the committed state is S_j (the state
 *    after tokens 0..j-1), and j = 0 leaves the cached state unchanged.
 *  - y is produced for every one of the K tokens: acceptance is decided from
 *    the verifier's outputs for all of them.
 *
 * Readings where the pages are silent (no formula, shape or dtype is printed):
 *  A and D are per-head scalars; dt is a per-(sequence, token, head) scalar
 *  that is already positive (no softplus, bias or clamp is applied here);
 *  head h uses B/C group g = h / (H / G) (consecutive blocks of heads);
 *  an accept_len outside [0, K] leaves that sequence's state untouched and is
 *  reported in the return value.
 *
 * Arithmetic is IEEE double, in the order written above, compiled without
 * floating-point contraction so that a*S + u*B is two roundings, not an FMA.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BAD_SHAPE (-1)
#define ORACLE_BAD_ACCEPT_LEN 1
#define ORACLE_NO_MEMORY (-2)

/* Index helpers, all row-major, last index fastest. */
static size_t idx_state(int64_t b, int64_t h, int64_t p, int64_t n, int64_t H, int64_t P, int64_t N)
{
    return (size_t)(((b * H + h) * P + p) * N + n);
}

/*
 * One verify/commit pass over a batch of sequences for one layer.
 *
 * state0     [batch][H][P][N]   cached state h_0 (read only)
 * x          [batch][K][H][P]
 * Bm, Cm     [batch][K][G][N]
 * dt         [batch][K][H]      already positive
 * A, D       [H]
 * accept_len [batch] or NULL    NULL means every token is accepted (j = K)
 * y          [batch][K][H][P]   or NULL (commit only)
 * state_out  [batch][H][P][N]   or NULL (verify only): receives h_j
 * trajectory [batch][H][K+1][P][N] or NULL: receives h_0 .. h_K (test aid)
 *
 * Returns 0, ORACLE_BAD_SHAPE, ORACLE_NO_MEMORY, or ORACLE_BAD_ACCEPT_LEN if
 * some accept_len was outside [0, K] (those sequences get state_out = state0).
 */
int ssm_oracle_verify_commit(int64_t batch, int64_t H, int64_t P, int64_t N, int64_t G, int64_t K,
                             const double *state0, const double *x, const double *Bm,
                             const double *Cm, const double *dt, const double *A, const double *D,
                             const int32_t *accept_len, double *y, double *state_out,
                             double *trajectory)
{
    if (batch < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || K < 0 || H % G != 0)
        return ORACLE_BAD_SHAPE;

    const int64_t heads_per_group = H / G;
    const size_t slice = (size_t)(P * N);
    int status = 0;
    double *cur = (double *)malloc(slice * sizeof(double));
    if (!cur)
        return ORACLE_NO_MEMORY;

    for (int64_t b = 0; b < batch; ++b) {
        int64_t j = accept_len ? (int64_t)accept_len[b] : K;
        int valid = (j >= 0 && j <= K);
        if (!valid)
            status |= ORACLE_BAD_ACCEPT_LEN;

        for (int64_t h = 0; h < H; ++h) {
            const int64_t g = h / heads_per_group;
            const double *S0 = state0 + idx_state(b, h, 0, 0, H, P, N);
            double *S = state_out ? state_out + idx_state(b, h, 0, 0, H, P, N) : NULL;
            double *traj = trajectory ? trajectory + (size_t)((b * H + h) * (K + 1)) * slice : NULL;

            /* The running state h_t lives in its own buffer; state_out gets h_j. */
            memcpy(cur, S0, slice * sizeof(double));
            if (traj)
                memcpy(traj, cur, slice * sizeof(double));
            if (S)
                memcpy(S, S0, slice * sizeof(double)); /* j = 0, or invalid j */

            for (int64_t t = 0; t < K; ++t) {
                const double dtv = dt[(b * K + t) * H + h];
                const double a = exp(dtv * A[h]);
                const double *xt = x + ((b * K + t) * H + h) * P;
                const double *Bt = Bm + ((b * K + t) * G + g) * N;
                const double *Ct = Cm + ((b * K + t) * G + g) * N;
                for (int64_t p = 0; p < P; ++p) {
                    const double u = dtv * xt[p];
                    double *row = cur + p * N;
                    double acc = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        row[n] = a * row[n] + u * Bt[n];
                        acc += Ct[n] * row[n];
                    }
                    if (y)
                        y[((b * K + t) * H + h) * P + p] = acc + D[h] * xt[p];
                }
                if (traj)
                    memcpy(traj + (size_t)(t + 1) * slice, cur, slice * sizeof(double));
                if (S && valid && t + 1 == j)
                    memcpy(S, cur, slice * sizeof(double));
            }
        }
    }
    free(cur);
    return status;
}
