/*
 * oracle.c -- plain fp64 CPU oracle for chunkwise gated linear attention with
 * per-segment affine state summaries.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * statement of what the CUDA path computes.  It shares no code, header, table
 * or helper with the CUDA library; only tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Method (per batch row b and head h; q_t, k_t in R^Dk, v_t in R^Dv, g_t scalar):
 *     alpha_t = exp(g_t), or 0 when token t starts a sequence,
 *     S_t     = alpha_t * S_{t-1} + k_t v_t^T          (S_{-1} = 0, Dk x Dv)
 *     o_t     = scale * S_t^T q_t
 * Segment summaries follow the Megatron-Core API docs page
 * "core.ssm.context_parallel.chunkwise":
 *   - CPForwardUnpackedSummary: S_out = M S_in + delta_S, computed by
 *     LinearAttentionCPBackend.cp_forward_prepare "with zero incoming state";
 *   - chunkwise_cp_forward: compose the selected causal prefix of summaries,
 *     then cp_forward_apply computes the local output;
 *   - CPBackwardUnpackedSummary: dS_in = M^T dS_out + gamma, with gamma from
 *     cp_backward_prepare "with zero outgoing-state gradient";
 *   - chunkwise_cp_backward / cp_backward_apply: compose the reverse-causal
 *     suffix and finish the input gradients;
 *   - PackedSequenceCPMetadata / build_packed_sequence_cp_metadata: per-shard
 *     sequence ids, local cu_seqlens, preceding_rank_start (inclusive) and
 *     following_rank_stop (exclusive).
 * Here a "shard" is a contiguous segment of the sequence axis and every
 * segment lives in the same process.
 *
 * Layouts (all contiguous, row-major): q, k [B,T,H,Dk]; v, o, dO [B,T,H,Dv];
 * g, dg [B,T,H]; summaries [nseg,B,H,Dk,Dv]; M [nseg,B,H].  seq_idx is NULL
 * (every row is one sequence) or an int32 [T] array applied to every row.
 * seg_starts is int32 [nseg+1], seg_starts[0] = 0, seg_starts[nseg] = T,
 * strictly increasing (segments need not be equal).
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes):
 *   - the gate is one scalar per (token, head);
 *   - a token that starts a sequence has alpha = 0, so its gate has no effect
 *     and its gate gradient is exactly 0;
 *   - M of a segment is exp(sum of its gates), or 0 if any of its tokens
 *     starts a sequence (its first token included);
 *   - the gate gradient is dg_t = sum_{r >= t, same sequence} (q_r.dq_r - k_r.dk_r),
 *     derived from o_t = scale sum_{s<=t} exp(G_t - G_s)(q_t.k_s) v_s with
 *     G the running sum of g; oracle_backward_direct computes the equivalent
 *     alpha_t <S_{t-1}, D_t> form from stored states for small inputs.
 *
 * Compiled with -ffp-contract=off so the results do not depend on whether
 * the host compiler fuses multiply-adds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

/* ----------------------------------------------------------------------- */
/* helpers                                                                  */
/* ----------------------------------------------------------------------- */

int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Token t starts a sequence: the first token of a row, or a change of id. */
static int starts_sequence(const int32_t* seq_idx, i64 t) {
    if (t == 0) return 1;
    if (seq_idx == NULL) return 0;
    return seq_idx[t] != seq_idx[t - 1];
}

static int same_sequence(const int32_t* seq_idx, i64 s, i64 t) {
    if (seq_idx == NULL) return 1;
    return seq_idx[s] == seq_idx[t];
}

static double gate_alpha(const double* g, const int32_t* seq_idx, i64 row_base_t,
                         i64 t, int H, int h) {
    if (starts_sequence(seq_idx, t)) return 0.0;
    return exp(g[(row_base_t + t) * H + h]);
}

#define IDX_QK(b, t, h) ((((i64)(b) * T + (t)) * H + (h)) * Dk)
#define IDX_V(b, t, h) ((((i64)(b) * T + (t)) * H + (h)) * Dv)
#define IDX_G(b, t, h) (((i64)(b) * T + (t)) * H + (h))

/* S = alpha S + k v^T */
static void state_step(double* S, double alpha, const double* k, const double* v,
                       int Dk, int Dv) {
    for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j)
            S[(i64)i * Dv + j] = alpha * S[(i64)i * Dv + j] + k[i] * v[j];
}

/* o = scale S^T q */
static void state_read(const double* S, const double* q, double scale, double* o,
                       int Dk, int Dv) {
    for (int j = 0; j < Dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < Dk; ++i) acc += S[(i64)i * Dv + j] * q[i];
        o[j] = scale * acc;
    }
}

/* dq = scale S dO */
static void state_apply(const double* S, const double* dO, double scale, double* dq,
                        int Dk, int Dv) {
    for (int i = 0; i < Dk; ++i) {
        double acc = 0.0;
        for (int j = 0; j < Dv; ++j) acc += S[(i64)i * Dv + j] * dO[j];
        dq[i] = scale * acc;
    }
}

/* D = scale q dO^T + beta D */
static void adjoint_step(double* D, double beta, const double* q, const double* dO,
                         double scale, int Dk, int Dv) {
    for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j)
            D[(i64)i * Dv + j] = scale * q[i] * dO[j] + beta * D[(i64)i * Dv + j];
}

/* dk = D v, dv = D^T k */
static void adjoint_read(const double* D, const double* k, const double* v,
                         double* dk, double* dv, int Dk, int Dv) {
    for (int i = 0; i < Dk; ++i) {
        double acc = 0.0;
        for (int j = 0; j < Dv; ++j) acc += D[(i64)i * Dv + j] * v[j];
        dk[i] = acc;
    }
    for (int j = 0; j < Dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < Dk; ++i) acc += D[(i64)i * Dv + j] * k[i];
        dv[j] = acc;
    }
}

static double dot(const double* a, const double* b, int n) {
    double acc = 0.0;
    for (int i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* ----------------------------------------------------------------------- */
/* monolithic recurrence                                                    */
/* ----------------------------------------------------------------------- */

/* Forward: walk t = 0..T-1 with the token recurrence. */
void oracle_forward(int B, int T, int H, int Dk, int Dv, double scale,
                    const double* q, const double* k, const double* v, const double* g,
                    const int32_t* seq_idx, double* o) {
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* S = (double*)calloc((size_t)Dk * Dv, sizeof(double));
        for (i64 t = 0; t < T; ++t) {
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            state_step(S, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_read(S, q + IDX_QK(b, t, h), scale, o + IDX_V(b, t, h), Dk, Dv);
        }
        free(S);
    }
}

/* Backward of L = sum_t dO_t . o_t.
 * Forward sweep: dq_t = scale S_t dO_t.
 * Reverse sweep: D_t = scale q_t dO_t^T + alpha_{t+1} D_{t+1} (alpha_T = 0),
 *                dk_t = D_t v_t, dv_t = D_t^T k_t.
 * Gate: dg_t = sum_{r >= t, same sequence} (q_r.dq_r - k_r.dk_r); 0 at starts. */
void oracle_backward(int B, int T, int H, int Dk, int Dv, double scale,
                     const double* q, const double* k, const double* v, const double* g,
                     const int32_t* seq_idx, const double* dO,
                     double* dq, double* dk, double* dv, double* dg) {
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* S = (double*)calloc((size_t)Dk * Dv, sizeof(double));
        double* qdq = (double*)malloc(sizeof(double) * (size_t)T);
        for (i64 t = 0; t < T; ++t) {
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            state_step(S, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_apply(S, dO + IDX_V(b, t, h), scale, dq + IDX_QK(b, t, h), Dk, Dv);
            qdq[t] = dot(q + IDX_QK(b, t, h), dq + IDX_QK(b, t, h), Dk);
        }
        double* D = S; /* reuse */
        memset(D, 0, sizeof(double) * (size_t)Dk * Dv);
        double run = 0.0;
        for (i64 t = T - 1; t >= 0; --t) {
            const double beta = (t + 1 < T) ? gate_alpha(g, seq_idx, (i64)b * T, t + 1, H, h) : 0.0;
            adjoint_step(D, beta, q + IDX_QK(b, t, h), dO + IDX_V(b, t, h), scale, Dk, Dv);
            adjoint_read(D, k + IDX_QK(b, t, h), v + IDX_V(b, t, h),
                         dk + IDX_QK(b, t, h), dv + IDX_V(b, t, h), Dk, Dv);
            const double kdk = dot(k + IDX_QK(b, t, h), dk + IDX_QK(b, t, h), Dk);
            if (t + 1 < T && !starts_sequence(seq_idx, t + 1))
                run = (qdq[t] - kdk) + run;
            else
                run = qdq[t] - kdk;
            dg[IDX_G(b, t, h)] = starts_sequence(seq_idx, t) ? 0.0 : run;
        }
        free(qdq);
        free(S);
    }
}

/* Backward with the gate gradient in its direct form dg_t = alpha_t <S_{t-1}, D_t>,
 * from all stored states.  Memory O(T Dk Dv): small inputs only. */
void oracle_backward_direct(int B, int T, int H, int Dk, int Dv, double scale,
                            const double* q, const double* k, const double* v, const double* g,
                            const int32_t* seq_idx, const double* dO,
                            double* dq, double* dk, double* dv, double* dg) {
    const i64 SZ = (i64)Dk * Dv;
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* states = (double*)calloc((size_t)(T + 1) * SZ, sizeof(double)); /* states[t+1] = S_t */
        for (i64 t = 0; t < T; ++t) {
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            memcpy(states + (t + 1) * SZ, states + t * SZ, sizeof(double) * (size_t)SZ);
            state_step(states + (t + 1) * SZ, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_apply(states + (t + 1) * SZ, dO + IDX_V(b, t, h), scale, dq + IDX_QK(b, t, h), Dk, Dv);
        }
        double* D = (double*)calloc((size_t)SZ, sizeof(double));
        for (i64 t = T - 1; t >= 0; --t) {
            const double beta = (t + 1 < T) ? gate_alpha(g, seq_idx, (i64)b * T, t + 1, H, h) : 0.0;
            adjoint_step(D, beta, q + IDX_QK(b, t, h), dO + IDX_V(b, t, h), scale, Dk, Dv);
            adjoint_read(D, k + IDX_QK(b, t, h), v + IDX_V(b, t, h),
                         dk + IDX_QK(b, t, h), dv + IDX_V(b, t, h), Dk, Dv);
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            double acc = 0.0;
            for (i64 e = 0; e < SZ; ++e) acc += states[t * SZ + e] * D[e];
            dg[IDX_G(b, t, h)] = a * acc;
        }
        free(D);
        free(states);
    }
}

/* ----------------------------------------------------------------------- */
/* segmented form                                                           */
/* ----------------------------------------------------------------------- */

/* cp_forward_prepare for every segment: with zero incoming state, walk the
 * segment's tokens; delta_S is the state at its end, and M = exp(sum g) over
 * the segment, or 0 when one of its tokens starts a sequence. */
void oracle_forward_prepare(int B, int T, int H, int Dk, int Dv, int nseg,
                            const int32_t* seg_starts,
                            const double* k, const double* v, const double* g,
                            const int32_t* seq_idx, double* M, double* dS) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        double* S = dS + task * SZ; /* task == (j*B + b)*H + h */
        memset(S, 0, sizeof(double) * (size_t)SZ);
        double gsum = 0.0;
        int reset = 0;
        for (i64 t = seg_starts[j]; t < seg_starts[j + 1]; ++t) {
            if (starts_sequence(seq_idx, t)) reset = 1;
            gsum += g[IDX_G(b, t, h)];
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            state_step(S, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
        }
        M[task] = reset ? 0.0 : exp(gsum);
    }
}

/* chunkwise_cp_forward's prefix: S_in[j] = composition of the summaries of
 * segments [pre[j], j), applied in order to a zero state (S <- M_i S + dS_i).
 * pre may be NULL (every prefix starts at segment 0). */
void oracle_compose_prefix(int nseg, int BH, int Dk, int Dv, const double* M,
                           const double* dS, const int32_t* pre, double* S_in) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * BH; ++task) {
        const int j = (int)(task / BH);
        const i64 bh = task % BH;
        double* S = S_in + task * SZ;
        memset(S, 0, sizeof(double) * (size_t)SZ);
        const int start = pre ? pre[j] : 0;
        for (int i = start; i < j; ++i) {
            const double m = M[(i64)i * BH + bh];
            const double* d = dS + ((i64)i * BH + bh) * SZ;
            for (i64 e = 0; e < SZ; ++e) S[e] = m * S[e] + d[e];
        }
    }
}

/* cp_forward_apply: walk each segment from its composed incoming state. */
void oracle_forward_apply(int B, int T, int H, int Dk, int Dv, int nseg,
                          const int32_t* seg_starts, double scale,
                          const double* q, const double* k, const double* v, const double* g,
                          const int32_t* seq_idx, const double* S_in, double* o) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        double* S = (double*)malloc(sizeof(double) * (size_t)SZ);
        memcpy(S, S_in + task * SZ, sizeof(double) * (size_t)SZ);
        for (i64 t = seg_starts[j]; t < seg_starts[j + 1]; ++t) {
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            state_step(S, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_read(S, q + IDX_QK(b, t, h), scale, o + IDX_V(b, t, h), Dk, Dv);
        }
        free(S);
    }
}

/* cp_backward_prepare: gamma_j = dL_local/dS_in with zero outgoing-state
 * gradient: the reverse adjoint sweep over the segment started from D = 0,
 * taken through the first token's transition (gamma = alpha_a D_a). */
void oracle_backward_prepare(int B, int T, int H, int Dk, int Dv, int nseg,
                             const int32_t* seg_starts, double scale,
                             const double* q, const double* g, const int32_t* seq_idx,
                             const double* dO, double* gamma) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        double* D = gamma + task * SZ;
        memset(D, 0, sizeof(double) * (size_t)SZ);
        const i64 a0 = seg_starts[j], e0 = seg_starts[j + 1];
        for (i64 t = e0 - 1; t >= a0; --t) {
            const double beta = (t + 1 < e0) ? gate_alpha(g, seq_idx, (i64)b * T, t + 1, H, h) : 0.0;
            adjoint_step(D, beta, q + IDX_QK(b, t, h), dO + IDX_V(b, t, h), scale, Dk, Dv);
        }
        const double a = gate_alpha(g, seq_idx, (i64)b * T, a0, H, h);
        for (i64 e = 0; e < SZ; ++e) D[e] *= a;
    }
}

/* chunkwise_cp_backward's suffix: dS_out[j] = sum over i in (j, fol[j]) of
 * (M_{j+1} ... M_{i-1}) gamma_i, i.e. D <- M_i D + gamma_i for i = fol[j]-1
 * down to j+1 from D = 0.  fol may be NULL (every suffix ends at nseg). */
void oracle_compose_suffix(int nseg, int BH, int Dk, int Dv, const double* M,
                           const double* gamma, const int32_t* fol, double* dS_out) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * BH; ++task) {
        const int j = (int)(task / BH);
        const i64 bh = task % BH;
        double* D = dS_out + task * SZ;
        memset(D, 0, sizeof(double) * (size_t)SZ);
        const int stop = fol ? fol[j] : nseg;
        for (int i = stop - 1; i > j; --i) {
            const double m = M[(i64)i * BH + bh];
            const double* gi = gamma + ((i64)i * BH + bh) * SZ;
            for (i64 e = 0; e < SZ; ++e) D[e] = m * D[e] + gi[e];
        }
    }
}

/* cp_backward_apply: all four input gradients of one segment, given its true
 * incoming state S_in and the adjoint dS_out of its outgoing state.
 * dg adds <S_out, dS_out> (S_out = the segment's true end state) for tokens of
 * the sequence that is still open at the segment's end. */
void oracle_backward_apply(int B, int T, int H, int Dk, int Dv, int nseg,
                           const int32_t* seg_starts, double scale,
                           const double* q, const double* k, const double* v, const double* g,
                           const int32_t* seq_idx, const double* dO,
                           const double* S_in, const double* dS_out,
                           double* dq, double* dk, double* dv, double* dg) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        const i64 a0 = seg_starts[j], e0 = seg_starts[j + 1];
        double* S = (double*)malloc(sizeof(double) * (size_t)SZ);
        double* qdq = (double*)malloc(sizeof(double) * (size_t)(e0 - a0));
        memcpy(S, S_in + task * SZ, sizeof(double) * (size_t)SZ);
        for (i64 t = a0; t < e0; ++t) {
            const double a = gate_alpha(g, seq_idx, (i64)b * T, t, H, h);
            state_step(S, a, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_apply(S, dO + IDX_V(b, t, h), scale, dq + IDX_QK(b, t, h), Dk, Dv);
            qdq[t - a0] = dot(q + IDX_QK(b, t, h), dq + IDX_QK(b, t, h), Dk);
        }
        const double* dSo = dS_out + task * SZ;
        double ext = 0.0; /* <S_out, dS_out> */
        for (i64 e = 0; e < SZ; ++e) ext += S[e] * dSo[e];
        double* D = S;
        memcpy(D, dSo, sizeof(double) * (size_t)SZ);
        double run = ext;
        for (i64 t = e0 - 1; t >= a0; --t) {
            const double beta = (t + 1 < e0) ? gate_alpha(g, seq_idx, (i64)b * T, t + 1, H, h) : 1.0;
            adjoint_step(D, beta, q + IDX_QK(b, t, h), dO + IDX_V(b, t, h), scale, Dk, Dv);
            adjoint_read(D, k + IDX_QK(b, t, h), v + IDX_V(b, t, h),
                         dk + IDX_QK(b, t, h), dv + IDX_V(b, t, h), Dk, Dv);
            const double kdk = dot(k + IDX_QK(b, t, h), dk + IDX_QK(b, t, h), Dk);
            if (t + 1 < e0 && starts_sequence(seq_idx, t + 1))
                run = qdq[t - a0] - kdk;
            else
                run = (qdq[t - a0] - kdk) + run;
            dg[IDX_G(b, t, h)] = starts_sequence(seq_idx, t) ? 0.0 : run;
        }
        free(qdq);
        free(S);
    }
}

/* ----------------------------------------------------------------------- */
/* packed-sequence metadata, by brute force                                 */
/* ----------------------------------------------------------------------- */

static int segment_of(const int32_t* seg_starts, int nseg, i64 t) {
    for (int j = 0; j < nseg; ++j)
        if (seg_starts[j] <= t && t < seg_starts[j + 1]) return j;
    return -1;
}

/* PackedSequenceCPMetadata for every segment, from cu_seqlens [nseqs+1]:
 *   seq_idx[t]   = i for cu[i] <= t < cu[i+1];
 *   local cu_seqlens of segment j (concatenated, offsets in local_off[nseg+1]):
 *                  0, then every t - a_j for a sequence start t strictly
 *                  inside the segment, then the segment length;
 *   pre[j]       = segment holding the start of the sequence holding a_j;
 *   fol[j]       = 1 + segment holding the last token of the sequence
 *                  holding the segment's last token.
 * Returns 0, or -1 when cu_seqlens is not 0 = cu[0] < cu[1] < ... = T. */
int oracle_packed_metadata(const int32_t* cu, int nseqs, int T, int nseg,
                           const int32_t* seg_starts, int32_t* seq_idx,
                           int32_t* local_cu, int32_t* local_off,
                           int32_t* pre, int32_t* fol) {
    if (nseqs < 1 || cu[0] != 0 || cu[nseqs] != T) return -1;
    for (int i = 0; i < nseqs; ++i)
        if (cu[i + 1] <= cu[i]) return -1;
    for (i64 t = 0; t < T; ++t) {
        seq_idx[t] = -1;
        for (int i = 0; i < nseqs; ++i)
            if (cu[i] <= t && t < cu[i + 1]) seq_idx[t] = i;
    }
    int n = 0;
    for (int j = 0; j < nseg; ++j) {
        const i64 a = seg_starts[j], e = seg_starts[j + 1];
        local_off[j] = n;
        local_cu[n++] = 0;
        for (i64 t = a + 1; t < e; ++t) {
            int is_start = 0;
            for (int i = 0; i <= nseqs; ++i)
                if (cu[i] == t) is_start = 1;
            if (is_start) local_cu[n++] = (int32_t)(t - a);
        }
        local_cu[n++] = (int32_t)(e - a);
        const int s_first = seq_idx[a];
        pre[j] = segment_of(seg_starts, nseg, cu[s_first]);
        const int s_last = seq_idx[e - 1];
        fol[j] = 1 + segment_of(seg_starts, nseg, (i64)cu[s_last + 1] - 1);
    }
    local_off[nseg] = n;
    return 0;
}

/* ----------------------------------------------------------------------- */
/* Mamba2 SSD state passing (the scan this state-summary machinery also     */
/* serves): per row b and head h, with group gi = h / (H / G),              */
/*   a_t = exp(dt_t A_h)  (0 when token t starts a sequence),               */
/*   h_t = a_t h_{t-1} + dt_t B_t x_t^T           (N x P),                  */
/*   y_t = h_t^T C_t + D_h x_t.                                             */
/* x, y [B,T,H,P]; dt [B,T,H]; A, D [H]; Bm, Cm [B,T,G,N].                  */
/* ----------------------------------------------------------------------- */

#define SIDX_X(b, t, h) ((((i64)(b) * T + (t)) * H + (h)) * P)
#define SIDX_BC(b, t, gi) ((((i64)(b) * T + (t)) * G + (gi)) * N)
#define SIDX_DT(b, t, h) (((i64)(b) * T + (t)) * H + (h))

static double ssd_decay(const double* dt, const double* A, const int32_t* seq_idx, int T,
                        int H, int b, i64 t, int h) {
    if (starts_sequence(seq_idx, t)) return 0.0;
    return exp(dt[SIDX_DT(b, t, h)] * A[h]);
}

void oracle_ssd_forward(int B, int T, int H, int G, int N, int P, const double* x,
                        const double* dt, const double* A, const double* Bm, const double* Cm,
                        const double* D, const int32_t* seq_idx, double* y) {
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H), gi = h / (H / G);
        double* hs = (double*)calloc((size_t)N * P, sizeof(double));
        for (i64 t = 0; t < T; ++t) {
            const double a = ssd_decay(dt, A, seq_idx, T, H, b, t, h);
            const double d = dt[SIDX_DT(b, t, h)];
            const double* Bt = Bm + SIDX_BC(b, t, gi);
            const double* Ct = Cm + SIDX_BC(b, t, gi);
            const double* xt = x + SIDX_X(b, t, h);
            for (int n = 0; n < N; ++n)
                for (int p = 0; p < P; ++p)
                    hs[(i64)n * P + p] = a * hs[(i64)n * P + p] + d * Bt[n] * xt[p];
            double* yt = y + SIDX_X(b, t, h);
            for (int p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int n = 0; n < N; ++n) acc += hs[(i64)n * P + p] * Ct[n];
                yt[p] = acc + (D ? D[h] * xt[p] : 0.0);
            }
        }
        free(hs);
    }
}

/* Backward of L = sum_t dy_t . y_t.  Tasks are (row, group) so that the heads
 * of a group, which share B_t and C_t, add into dB and dC in a fixed order.
 *   forward sweep:  dC_t += h_t dy_t;
 *   reverse sweep:  adjoint Q_t = C_t dy_t^T + a_{t+1} Q_{t+1} (a_{t+1} = 0
 *                   past the row or at a sequence start),
 *                   dx_t = dt_t Q_t^T B_t + D_h dy_t,  dB_t += dt_t Q_t x_t,
 *                   ddt_t = B_t . (Q_t x_t) + A_h e_t,  dA_h = sum_t dt_t e_t,
 *                   dD_h = sum_t x_t . dy_t,
 * where e_t = a_t <h_{t-1}, Q_t> is the gradient through the decay's exponent,
 * taken as sum_{r >= t, same sequence} (C_r . dC^h_r - dt_r B_r . (Q_r x_r))
 * (0 at a sequence start) so that no state has to be stored. */
void oracle_ssd_backward(int B, int T, int H, int G, int N, int P, const double* x,
                         const double* dt, const double* A, const double* Bm, const double* Cm,
                         const double* D, const int32_t* seq_idx, const double* dy,
                         double* dx, double* ddt, double* dA, double* dB, double* dC,
                         double* dD) {
    const int hpg = H / G;
    memset(dB, 0, sizeof(double) * (size_t)B * T * G * N);
    memset(dC, 0, sizeof(double) * (size_t)B * T * G * N);
    double* dA_part = (double*)calloc((size_t)B * H, sizeof(double));
    double* dD_part = (double*)calloc((size_t)B * H, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bg = 0; bg < (i64)B * G; ++bg) {
        const int b = (int)(bg / G), gi = (int)(bg % G);
        double* hs = (double*)malloc(sizeof(double) * (size_t)N * P);
        double* Q = (double*)malloc(sizeof(double) * (size_t)N * P);
        double* cdc = (double*)malloc(sizeof(double) * (size_t)T);
        double* dch = (double*)malloc(sizeof(double) * (size_t)N);
        double* qx = (double*)malloc(sizeof(double) * (size_t)N);
        for (int h = gi * hpg; h < (gi + 1) * hpg; ++h) {
            memset(hs, 0, sizeof(double) * (size_t)N * P);
            for (i64 t = 0; t < T; ++t) {
                const double a = ssd_decay(dt, A, seq_idx, T, H, b, t, h);
                const double d = dt[SIDX_DT(b, t, h)];
                const double* Bt = Bm + SIDX_BC(b, t, gi);
                const double* Ct = Cm + SIDX_BC(b, t, gi);
                const double* xt = x + SIDX_X(b, t, h);
                const double* dyt = dy + SIDX_X(b, t, h);
                for (int n = 0; n < N; ++n)
                    for (int p = 0; p < P; ++p)
                        hs[(i64)n * P + p] = a * hs[(i64)n * P + p] + d * Bt[n] * xt[p];
                for (int n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int p = 0; p < P; ++p) acc += hs[(i64)n * P + p] * dyt[p];
                    dch[n] = acc;
                    dC[SIDX_BC(b, t, gi) + n] += acc;
                }
                cdc[t] = dot(Ct, dch, N);
            }
            memset(Q, 0, sizeof(double) * (size_t)N * P);
            double run = 0.0, sa = 0.0, sd = 0.0;
            for (i64 t = T - 1; t >= 0; --t) {
                const double beta = (t + 1 < T) ? ssd_decay(dt, A, seq_idx, T, H, b, t + 1, h) : 0.0;
                const double d = dt[SIDX_DT(b, t, h)];
                const double* Bt = Bm + SIDX_BC(b, t, gi);
                const double* Ct = Cm + SIDX_BC(b, t, gi);
                const double* xt = x + SIDX_X(b, t, h);
                const double* dyt = dy + SIDX_X(b, t, h);
                for (int n = 0; n < N; ++n)
                    for (int p = 0; p < P; ++p)
                        Q[(i64)n * P + p] = Ct[n] * dyt[p] + beta * Q[(i64)n * P + p];
                for (int n = 0; n < N; ++n) {
                    double acc = 0.0;
                    for (int p = 0; p < P; ++p) acc += Q[(i64)n * P + p] * xt[p];
                    qx[n] = acc;
                    dB[SIDX_BC(b, t, gi) + n] += d * acc;
                }
                double* dxt = dx + SIDX_X(b, t, h);
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n) acc += Q[(i64)n * P + p] * Bt[n];
                    dxt[p] = d * acc + (D ? D[h] * dyt[p] : 0.0);
                }
                const double bqx = dot(Bt, qx, N);
                if (t + 1 < T && !starts_sequence(seq_idx, t + 1))
                    run = (cdc[t] - d * bqx) + run;
                else
                    run = cdc[t] - d * bqx;
                const double e = starts_sequence(seq_idx, t) ? 0.0 : run;
                ddt[SIDX_DT(b, t, h)] = bqx + A[h] * e;
                sa += d * e;
                sd += dot(xt, dyt, P);
            }
            dA_part[(i64)b * H + h] = sa;
            dD_part[(i64)b * H + h] = sd;
        }
        free(hs);
        free(Q);
        free(cdc);
        free(dch);
        free(qx);
    }
    for (int h = 0; h < H; ++h) {
        double sa = 0.0, sd = 0.0;
        for (int b = 0; b < B; ++b) {
            sa += dA_part[(i64)b * H + h];
            sd += dD_part[(i64)b * H + h];
        }
        dA[h] = sa;
        dD[h] = sd;
    }
    free(dA_part);
    free(dD_part);
}

/* ----------------------------------------------------------------------- */
/* Vector (per key dimension) gates: the general transition of the summary  */
/* algebra restricted to a diagonal M.  Per row b and head h, with g        */
/* [B,T,H,Dk] fp32 and alpha_t[i] = exp(g_t[i]) (all 0 when token t starts  */
/* a sequence):                                                             */
/*   S_t = diag(alpha_t) S_{t-1} + k_t v_t^T,   o_t = scale S_t^T q_t.      */
/* S0 [B,H,Dk,Dv] (may be NULL) is the state before the first token.        */
/* ----------------------------------------------------------------------- */

#define VG_IDX(b, t, h) ((((i64)(b) * T + (t)) * H + (h)) * Dk)

static void vg_step(double* S, const double* g, int reset, const double* k, const double* v,
                    int Dk, int Dv) {
    for (int i = 0; i < Dk; ++i) {
        const double a = reset ? 0.0 : exp(g[i]);
        for (int j = 0; j < Dv; ++j) S[(i64)i * Dv + j] = a * S[(i64)i * Dv + j] + k[i] * v[j];
    }
}

void oracle_vg_forward(int B, int T, int H, int Dk, int Dv, double scale, const double* q,
                       const double* k, const double* v, const double* g, const int32_t* seq_idx,
                       const double* S0, double* o) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* S = (double*)calloc((size_t)SZ, sizeof(double));
        if (S0) memcpy(S, S0 + bh * SZ, sizeof(double) * (size_t)SZ);
        for (i64 t = 0; t < T; ++t) {
            vg_step(S, g + VG_IDX(b, t, h), starts_sequence(seq_idx, t) && (t > 0 || S0 == NULL),
                    k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
            state_read(S, q + IDX_QK(b, t, h), scale, o + IDX_V(b, t, h), Dk, Dv);
        }
        free(S);
    }
}

/* Backward of L = sum_t dO_t . o_t (S0 = 0).  dq_t = scale S_t dO_t;
 * D_t = scale q_t dO_t^T + diag(alpha_{t+1}) D_{t+1}; dk_t = D_t v_t,
 * dv_t = D_t^T k_t; per dimension i the gate gradient is
 * dg_t[i] = sum_{r >= t, same sequence} (q_r[i] dq_r[i] - k_r[i] dk_r[i]),
 * 0 at sequence starts; direct != 0 takes alpha_t[i] <S_{t-1}[i,:], D_t[i,:]>
 * from stored states instead (small inputs only). */
void oracle_vg_backward(int B, int T, int H, int Dk, int Dv, double scale, const double* q,
                        const double* k, const double* v, const double* g,
                        const int32_t* seq_idx, const double* dO, int direct, double* dq,
                        double* dk, double* dv, double* dg) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* states = (double*)calloc((size_t)(direct ? T + 1 : 1) * SZ, sizeof(double));
        double* S = states;
        double* qdq = (double*)malloc(sizeof(double) * (size_t)T * Dk);
        for (i64 t = 0; t < T; ++t) {
            if (direct) {
                memcpy(states + (t + 1) * SZ, states + t * SZ, sizeof(double) * (size_t)SZ);
                S = states + (t + 1) * SZ;
            }
            vg_step(S, g + VG_IDX(b, t, h), starts_sequence(seq_idx, t), k + IDX_QK(b, t, h),
                    v + IDX_V(b, t, h), Dk, Dv);
            state_apply(S, dO + IDX_V(b, t, h), scale, dq + IDX_QK(b, t, h), Dk, Dv);
            for (int i = 0; i < Dk; ++i) qdq[t * Dk + i] = q[IDX_QK(b, t, h) + i] * dq[IDX_QK(b, t, h) + i];
        }
        double* D = (double*)calloc((size_t)SZ, sizeof(double));
        double* run = (double*)calloc((size_t)Dk, sizeof(double));
        for (i64 t = T - 1; t >= 0; --t) {
            const int next_reset = (t + 1 >= T) || starts_sequence(seq_idx, t + 1);
            const double* gn = (t + 1 < T) ? g + VG_IDX(b, t + 1, h) : NULL;
            const double* qt = q + IDX_QK(b, t, h);
            const double* dOt = dO + IDX_V(b, t, h);
            for (int i = 0; i < Dk; ++i) {
                const double beta = next_reset ? 0.0 : exp(gn[i]);
                for (int j = 0; j < Dv; ++j)
                    D[(i64)i * Dv + j] = scale * qt[i] * dOt[j] + beta * D[(i64)i * Dv + j];
            }
            adjoint_read(D, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), dk + IDX_QK(b, t, h),
                         dv + IDX_V(b, t, h), Dk, Dv);
            double* dgt = dg + VG_IDX(b, t, h);
            const int start = starts_sequence(seq_idx, t);
            for (int i = 0; i < Dk; ++i) {
                if (direct) {
                    double acc = 0.0;
                    for (int j = 0; j < Dv; ++j) acc += states[t * SZ + (i64)i * Dv + j] * D[(i64)i * Dv + j];
                    dgt[i] = start ? 0.0 : exp(g[VG_IDX(b, t, h) + i]) * acc;
                } else {
                    const double c = qdq[t * Dk + i] - k[IDX_QK(b, t, h) + i] * dk[IDX_QK(b, t, h) + i];
                    run[i] = next_reset ? c : c + run[i];
                    dgt[i] = start ? 0.0 : run[i];
                }
            }
        }
        free(run);
        free(D);
        free(qdq);
        free(states);
    }
}

/* cp_forward_prepare with vector gates: per (segment, row, head) the diagonal
 * transition M [Dk] (prod of alpha over the segment, 0 where a token of it
 * starts a sequence) and the local end state dS from S_in = 0. */
void oracle_vg_forward_prepare(int B, int T, int H, int Dk, int Dv, int nseg,
                               const int32_t* seg_starts, const double* k, const double* v,
                               const double* g, const int32_t* seq_idx, double* M, double* dS) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        double* S = dS + task * SZ;
        double* m = M + task * Dk;
        memset(S, 0, sizeof(double) * (size_t)SZ);
        for (int i = 0; i < Dk; ++i) m[i] = 1.0;
        for (i64 t = seg_starts[j]; t < seg_starts[j + 1]; ++t) {
            const int reset = starts_sequence(seq_idx, t);
            const double* gt = g + VG_IDX(b, t, h);
            for (int i = 0; i < Dk; ++i) m[i] = reset ? 0.0 : m[i] * exp(gt[i]);
            vg_step(S, gt, reset, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv);
        }
    }
}

/* ----------------------------------------------------------------------- */
/* Gated delta rule: the matrix-transition case of the summary algebra.     */
/* Per row b and head h, with a scalar gate g_t, a write strength beta_t    */
/* ([B,T,H] each) and A_t = alpha_t (I - beta_t k_t k_t^T), alpha_t =        */
/* exp(g_t) (0 when token t starts a sequence):                              */
/*   S_t = A_t S_{t-1} + beta_t k_t v_t^T,   o_t = scale S_t^T q_t.          */
/* Every state is stored (memory O(T Dk Dv) per task): small inputs only.   */
/* ----------------------------------------------------------------------- */

/* S_out = alpha (S_in - beta k (k^T S_in)) + beta k v^T */
static void gdr_step(double* S, double alpha, double beta, const double* k, const double* v,
                     int Dk, int Dv, double* kS) {
    for (int j = 0; j < Dv; ++j) {
        double acc = 0.0;
        for (int i = 0; i < Dk; ++i) acc += k[i] * S[(i64)i * Dv + j];
        kS[j] = acc;
    }
    for (int i = 0; i < Dk; ++i)
        for (int j = 0; j < Dv; ++j)
            S[(i64)i * Dv + j] = alpha * (S[(i64)i * Dv + j] - beta * k[i] * kS[j]) + beta * k[i] * v[j];
}

void oracle_gdr_forward(int B, int T, int H, int Dk, int Dv, double scale, const double* q,
                        const double* k, const double* v, const double* g, const double* beta,
                        const int32_t* seq_idx, const double* S0, double* o) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* S = (double*)calloc((size_t)SZ, sizeof(double));
        double* kS = (double*)malloc(sizeof(double) * (size_t)Dv);
        if (S0) memcpy(S, S0 + bh * SZ, sizeof(double) * (size_t)SZ);
        for (i64 t = 0; t < T; ++t) {
            const int reset = starts_sequence(seq_idx, t) && (t > 0 || S0 == NULL);
            const double a = reset ? 0.0 : exp(g[IDX_G(b, t, h)]);
            gdr_step(S, a, beta[IDX_G(b, t, h)], k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv, kS);
            state_read(S, q + IDX_QK(b, t, h), scale, o + IDX_V(b, t, h), Dk, Dv);
        }
        free(kS);
        free(S);
    }
}

/* Backward of L = sum_t dO_t . o_t (zero initial state), from the stored
 * states and the adjoint D_t = scale q_t dO_t^T + A_{t+1} D_{t+1} (A is
 * symmetric; A_T = 0):
 *   dq_t    = scale S_t dO_t
 *   dv_t    = beta_t D_t^T k_t
 *   dk_t    = beta_t D_t v_t - alpha_t beta_t (S_{t-1} D_t^T + D_t S_{t-1}^T) k_t
 *   dbeta_t = k_t^T D_t v_t - alpha_t k_t^T D_t S_{t-1}^T k_t
 *   dg_t    = alpha_t <D_t, (I - beta_t k_t k_t^T) S_{t-1}>   (0 at a start) */
void oracle_gdr_backward(int B, int T, int H, int Dk, int Dv, double scale, const double* q,
                         const double* k, const double* v, const double* g, const double* beta,
                         const int32_t* seq_idx, const double* dO, double* dq, double* dk,
                         double* dv, double* dg, double* dbeta) {
    const i64 SZ = (i64)Dk * Dv;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 bh = 0; bh < (i64)B * H; ++bh) {
        const int b = (int)(bh / H), h = (int)(bh % H);
        double* st = (double*)calloc((size_t)(T + 1) * SZ, sizeof(double)); /* st[t+1] = S_t */
        double* kS = (double*)malloc(sizeof(double) * (size_t)Dv);
        double* Dt = (double*)calloc((size_t)SZ, sizeof(double));
        double* tmp = (double*)malloc(sizeof(double) * (size_t)SZ);
        double* u = (double*)malloc(sizeof(double) * (size_t)Dk);
        double* w = (double*)malloc(sizeof(double) * (size_t)Dv);
        for (i64 t = 0; t < T; ++t) {
            const double a = starts_sequence(seq_idx, t) ? 0.0 : exp(g[IDX_G(b, t, h)]);
            memcpy(st + (t + 1) * SZ, st + t * SZ, sizeof(double) * (size_t)SZ);
            gdr_step(st + (t + 1) * SZ, a, beta[IDX_G(b, t, h)], k + IDX_QK(b, t, h), v + IDX_V(b, t, h),
                     Dk, Dv, kS);
            state_apply(st + (t + 1) * SZ, dO + IDX_V(b, t, h), scale, dq + IDX_QK(b, t, h), Dk, Dv);
        }
        for (i64 t = T - 1; t >= 0; --t) {
            /* D_t = scale q_t dO_t^T + A_{t+1} D_{t+1} */
            if (t + 1 < T) {
                const double an = starts_sequence(seq_idx, t + 1) ? 0.0 : exp(g[IDX_G(b, t + 1, h)]);
                const double bn = beta[IDX_G(b, t + 1, h)];
                const double* kn = k + IDX_QK(b, t + 1, h);
                for (int j = 0; j < Dv; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < Dk; ++i) acc += kn[i] * Dt[(i64)i * Dv + j];
                    w[j] = acc;
                }
                for (int i = 0; i < Dk; ++i)
                    for (int j = 0; j < Dv; ++j)
                        tmp[(i64)i * Dv + j] = an * (Dt[(i64)i * Dv + j] - bn * kn[i] * w[j]);
            } else {
                memset(tmp, 0, sizeof(double) * (size_t)SZ);
            }
            const double* qt = q + IDX_QK(b, t, h);
            const double* dOt = dO + IDX_V(b, t, h);
            for (int i = 0; i < Dk; ++i)
                for (int j = 0; j < Dv; ++j) Dt[(i64)i * Dv + j] = scale * qt[i] * dOt[j] + tmp[(i64)i * Dv + j];
            const double* kt = k + IDX_QK(b, t, h);
            const double* vt = v + IDX_V(b, t, h);
            const double* Sp = st + t * SZ; /* S_{t-1} */
            const int start = starts_sequence(seq_idx, t);
            const double a = start ? 0.0 : exp(g[IDX_G(b, t, h)]);
            const double bt = beta[IDX_G(b, t, h)];
            /* w = D_t^T k_t, u = D_t v_t */
            for (int j = 0; j < Dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < Dk; ++i) acc += Dt[(i64)i * Dv + j] * kt[i];
                w[j] = acc;
                dv[IDX_V(b, t, h) + j] = bt * acc;
            }
            for (int i = 0; i < Dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < Dv; ++j) acc += Dt[(i64)i * Dv + j] * vt[j];
                u[i] = acc;
            }
            /* kS = S_{t-1}^T k_t;  (S D^T + D S^T) k = S (D^T k) + D (S^T k) */
            for (int j = 0; j < Dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < Dk; ++i) acc += Sp[(i64)i * Dv + j] * kt[i];
                kS[j] = acc;
            }
            double kDv = 0.0, kDSk = 0.0, dgacc = 0.0;
            for (int i = 0; i < Dk; ++i) {
                double s1 = 0.0, s2 = 0.0;
                for (int j = 0; j < Dv; ++j) {
                    s1 += Sp[(i64)i * Dv + j] * w[j];
                    s2 += Dt[(i64)i * Dv + j] * kS[j];
                }
                dk[IDX_QK(b, t, h) + i] = bt * u[i] - a * bt * (s1 + s2);
                kDv += kt[i] * u[i];
                kDSk += kt[i] * s2;
            }
            for (int i = 0; i < Dk; ++i)
                for (int j = 0; j < Dv; ++j)
                    dgacc += Dt[(i64)i * Dv + j] * (Sp[(i64)i * Dv + j] - bt * kt[i] * kS[j]);
            dbeta[IDX_G(b, t, h)] = kDv - a * kDSk;
            dg[IDX_G(b, t, h)] = start ? 0.0 : a * dgacc;
        }
        free(w);
        free(u);
        free(tmp);
        free(Dt);
        free(kS);
        free(st);
    }
}

/* Segment summaries with matrix transitions: M [nseg,B,H,Dk,Dk] = A_last ... A_first
 * over the segment (A_t = 0 at a sequence start), dS the local end state. */
void oracle_gdr_forward_prepare(int B, int T, int H, int Dk, int Dv, int nseg,
                                const int32_t* seg_starts, const double* k, const double* v,
                                const double* g, const double* beta, const int32_t* seq_idx,
                                double* M, double* dS) {
    const i64 SZ = (i64)Dk * Dv, MZ = (i64)Dk * Dk;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 task = 0; task < (i64)nseg * B * H; ++task) {
        const int j = (int)(task / ((i64)B * H));
        const int b = (int)((task / H) % B), h = (int)(task % H);
        double* S = dS + task * SZ;
        double* Mt = M + task * MZ;
        double* kS = (double*)malloc(sizeof(double) * (size_t)(Dv > Dk ? Dv : Dk));
        double* zero = (double*)calloc((size_t)Dk, sizeof(double));
        memset(S, 0, sizeof(double) * (size_t)SZ);
        memset(Mt, 0, sizeof(double) * (size_t)MZ);
        for (int i = 0; i < Dk; ++i) Mt[(i64)i * Dk + i] = 1.0;
        for (i64 t = seg_starts[j]; t < seg_starts[j + 1]; ++t) {
            const double a = starts_sequence(seq_idx, t) ? 0.0 : exp(g[IDX_G(b, t, h)]);
            const double bt = beta[IDX_G(b, t, h)];
            gdr_step(S, a, bt, k + IDX_QK(b, t, h), v + IDX_V(b, t, h), Dk, Dv, kS);
            gdr_step(Mt, a, bt, k + IDX_QK(b, t, h), zero, Dk, Dk, kS); /* M <- A_t M */
        }
        free(zero);
        free(kS);
    }
}
