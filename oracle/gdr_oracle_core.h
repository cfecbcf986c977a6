/*
 * Precision-generic body of the CPU oracle -- TEST INFRASTRUCTURE ONLY.
 * Included by gdr_oracle.c with REAL (double or float), SFX(name), SQRT, EXP.
 * Every loop below is the definition written out; nothing is blocked, fused or
 * reordered.
 */

static REAL SFX(load_state)(const oracle_problem *p, size_t idx)
{
    if (p->state_bf16)
        return (REAL)bf16_bits_to_double(((const uint16_t *)p->state)[idx]);
    return (REAL)((const float *)p->state)[idx];
}

static void SFX(store_elem)(void *base, int bf16, size_t idx, REAL x)
{
    if (bf16)
        ((uint16_t *)base)[idx] = oracle_round_bf16((double)x);
    else
        ((float *)base)[idx] = (float)x;
}

static REAL SFX(load_elem)(const void *base, int bf16, size_t idx)
{
    if (bf16)
        return (REAL)bf16_bits_to_double(((const uint16_t *)base)[idx]);
    return (REAL)((const float *)base)[idx];
}

/* One token of the recurrence for one (sequence, value head); S is [K][V].
 * "gated_delta_recurrence_fwd_gpu" summary (L2 normalisation, 1/sqrt(K) query
 * scale); "core.ssm.ops.gdp.fused_recurrent" Parameters (log decay g, beta).
 * Outputs: o (V), and the normalised key kh (K) and correction u (V) that a
 * verify record keeps. */
static void SFX(token)(int K, int V, REAL *S, const float *q, const float *k,
                       const float *v, REAL alpha, const float *beta, int beta_stride, int l2,
                       REAL scale, REAL eps, REAL *qh, REAL *kh, REAL *u, REAL *o)
{
    REAL nq = 1, nk = 1;
    if (l2) {
        REAL sq = 0, sk = 0;
        for (int i = 0; i < K; ++i) {
            sq += (REAL)q[i] * (REAL)q[i];
            sk += (REAL)k[i] * (REAL)k[i];
        }
        nq = SQRT(sq + eps);
        nk = SQRT(sk + eps);
    }
    for (int i = 0; i < K; ++i) {
        qh[i] = (REAL)q[i] / nq;
        kh[i] = (REAL)k[i] / nk;
    }
    /* decay the whole state */
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(size_t)i * V + j] = alpha * S[(size_t)i * V + j];
    /* delta rule: u = beta * (v - S^T k^) against the decayed state; beta is
     * one value for the head (beta_stride 0) or one per value column */
    for (int j = 0; j < V; ++j) {
        REAL w = 0;
        for (int i = 0; i < K; ++i)
            w += S[(size_t)i * V + j] * kh[i];
        u[j] = (REAL)beta[(size_t)j * beta_stride] * ((REAL)v[j] - w);
    }
    /* rank-one update S += k^ u^T */
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(size_t)i * V + j] = S[(size_t)i * V + j] + kh[i] * u[j];
    /* readout of the updated state */
    for (int j = 0; j < V; ++j) {
        REAL acc = 0;
        for (int i = 0; i < K; ++i)
            acc += S[(size_t)i * V + j] * qh[i];
        o[j] = scale * acc;
    }
}

/* Shared driver for the forward, verify and snapshot passes.
 *   ring != NULL   : verify -- rows with L <= ring_len write one record per
 *                    token and leave the pool alone; longer rows record
 *                    nothing and commit like the forward pass.
 *   inter != NULL  : snapshots -- after every spt steps of a row the state is
 *                    stored at inter[slot, i, h] (i < n_inter).
 * out is [T, nv*V] in double; padding rows get exact zeros. */
static int SFX(run)(const oracle_problem *p, double *out, void *ring, int ring_bf16, int ring_rows,
                    int ring_len, int record_stride, const int32_t *ring_slot_idx,
                    void *inter, int n_inter, int spt)
{
    if (check_problem(p) != 0 || (p->total_tokens > 0 && !out))
        return -1;
    const int K = p->K, V = p->V, nv = p->nv, nk = p->nk, r = nv / nk;
    const size_t conv_dim = (size_t)2 * nk * K + (size_t)nv * V;
    const size_t value_dim = (size_t)nv * V;
    const REAL scale = p->scale > 0 ? (REAL)p->scale : (REAL)(1.0 / sqrt((double)K));
    const REAL eps = (REAL)p->eps;
    if (ring) {
        if (ring_len <= 0 || ring_rows <= 0 || !ring_slot_idx ||
            record_stride < oracle_ring_record_elements(K, V, r))
            return -1;
    }
    if (inter && (n_inter <= 0 || spt <= 0))
        return -1;

    REAL *S = (REAL *)malloc(sizeof(REAL) * (size_t)K * V);
    REAL *qh = (REAL *)malloc(sizeof(REAL) * K);
    REAL *kh = (REAL *)malloc(sizeof(REAL) * K);
    REAL *u = (REAL *)malloc(sizeof(REAL) * V);
    REAL *o = (REAL *)malloc(sizeof(REAL) * V);
    if (!S || !qh || !kh || !u || !o) {
        free(S); free(qh); free(kh); free(u); free(o);
        return -1;
    }
    int rc = 0;
    for (int b = 0; b < p->batch && rc == 0; ++b) {
        const int64_t t0 = p->offsets[b], t1 = p->offsets[b + 1];
        const int64_t L = t1 - t0;
        const int slot = p->slot_idx[b];
        const int records = ring && L <= ring_len;
        int rs = -1;
        if (ring && slot >= 0) {
            rs = ring_slot_idx[b];
            if (records && L > 0 && (rs < 0 || rs >= ring_rows)) {
                rc = -1;
                break;
            }
        }
        for (int h = 0; h < nv; ++h) {
            if (slot < 0) { /* padding request: zero output, nothing else */
                for (int64_t t = t0; t < t1; ++t)
                    for (int j = 0; j < V; ++j)
                        out[(size_t)t * value_dim + (size_t)h * V + j] = 0.0;
                continue;
            }
            const int hk = h / r, jr = h % r;
            const size_t sbase = (((size_t)slot * nv + h) * K) * V;
            for (size_t e = 0; e < (size_t)K * V; ++e)
                S[e] = SFX(load_state)(p, sbase + e);
            for (int64_t t = t0; t < t1; ++t) {
                const float *row = p->qkv + (size_t)t * conv_dim;
                const float *q = row + (size_t)hk * K;
                const float *k = row + (size_t)nk * K + (size_t)hk * K;
                const float *v = row + (size_t)2 * nk * K + (size_t)h * V;
                const float g = p->decay[(size_t)t * nv + h];
                const REAL alpha = p->decay_is_log ? EXP((REAL)g) : (REAL)g;
                const float *beta = p->beta_per_value
                                         ? p->beta + ((size_t)t * nv + h) * (size_t)V
                                         : p->beta + (size_t)t * nv + h;
                SFX(token)(K, V, S, q, k, v, alpha, beta, p->beta_per_value ? 1 : 0, p->use_l2norm,
                           scale, eps, qh, kh, u, o);
                for (int j = 0; j < V; ++j)
                    out[(size_t)t * value_dim + (size_t)h * V + j] = (double)o[j];
                if (records) {
                    const size_t rec = (((size_t)rs * nk + hk) * ring_len + (size_t)(t - t0)) *
                                       (size_t)record_stride;
                    if (jr == 0)
                        for (int i = 0; i < K; ++i)
                            SFX(store_elem)(ring, ring_bf16, rec + i, kh[i]);
                    SFX(store_elem)(ring, ring_bf16, rec + K + jr, alpha);
                    const size_t ur = rec + K + ((r + 7) / 8) * 8 + (size_t)jr * V;
                    for (int j = 0; j < V; ++j)
                        SFX(store_elem)(ring, ring_bf16, ur + j, u[j]);
                }
                if (inter) {
                    const int64_t s = t - t0;
                    if ((s + 1) % spt == 0) {
                        const int64_t i = (s + 1) / spt - 1;
                        if (i < n_inter) {
                            const size_t ibase =
                                ((((size_t)slot * n_inter + (size_t)i) * nv + h) * K) * V;
                            for (size_t e = 0; e < (size_t)K * V; ++e)
                                SFX(store_elem)(inter, p->state_bf16, ibase + e, S[e]);
                        }
                    }
                }
            }
            if (L > 0 && !records)
                for (size_t e = 0; e < (size_t)K * V; ++e)
                    SFX(store_elem)(p->state, p->state_bf16, sbase + e, S[e]);
        }
    }
    free(S); free(qh); free(kh); free(u); free(o);
    return rc;
}

/* Forward pass: the pool slot of every live row is advanced over the row and
 * written back in place ("gated_delta_recurrence_fwd_gpu", summary and Args). */
int SFX(oracle_fwd)(const oracle_problem *p, double *out)
{
    return SFX(run)(p, out, NULL, 0, 0, 0, 0, NULL, NULL, 0, 0);
}

/* Verify pass ("gated_delta_recurrence_verify_ring_gpu", summary); ring_bf16
 * selects a bfloat16 ring (Parameters: ring_dtype). */
int SFX(oracle_verify_ring)(const oracle_problem *p, double *out, void *ring, int ring_bf16,
                            int ring_rows, int ring_len, int record_stride,
                            const int32_t *ring_slot_idx)
{
    if (!ring)
        return -1;
    return SFX(run)(p, out, ring, ring_bf16, ring_rows, ring_len, record_stride, ring_slot_idx,
                    NULL, 0, 0);
}

/* Forward pass with per-draft-token snapshots ("core.ssm.ops.gdp.fused_recurrent",
 * intermediate_states and steps_per_token). inter is [max_slots, n_inter, nv, K, V]
 * in the pool's dtype. */
int SFX(oracle_fwd_snapshots)(const oracle_problem *p, double *out, void *inter,
                              int n_inter, int spt)
{
    if (!inter)
        return -1;
    return SFX(run)(p, out, NULL, 0, 0, 0, 0, NULL, inter, n_inter, spt);
}

/* Fold: advance each live row's slot over its first counts[b] ring records.
 * counts[b] == 0 or > ring_len leaves the row alone ("gated_delta_recurrence_
 * verify_ring_gpu", summary: the fold skips a row whose count exceeds RING_LEN).
 * Each record applies S = alpha * S; S = S + k^ u^T -- the same two steps the
 * forward pass takes, so in float32 with a float32 ring the result is the
 * forward pass over the accepted prefix, bit for bit. */
int SFX(oracle_fold)(const oracle_problem *p, const void *ring, int ring_bf16, int ring_rows,
                     int ring_len, int record_stride, const int32_t *ring_slot_idx,
                     const int32_t *counts)
{
    if (!p || p->nv <= 0 || p->nk <= 0 || p->nv % p->nk || p->K <= 0 || p->V <= 0 ||
        p->batch < 0 || !ring || !ring_slot_idx || !counts || ring_len <= 0 ||
        ring_rows <= 0 || (p->batch > 0 && !p->slot_idx))
        return -1;
    const int K = p->K, V = p->V, nv = p->nv, nk = p->nk, r = nv / nk;
    if (record_stride < oracle_ring_record_elements(K, V, r))
        return -1;
    REAL *S = (REAL *)malloc(sizeof(REAL) * (size_t)K * V);
    if (!S)
        return -1;
    int rc = 0;
    for (int b = 0; b < p->batch; ++b) {
        const int slot = p->slot_idx[b], c = counts[b];
        if (slot < 0 || c <= 0 || c > ring_len)
            continue;
        const int rs = ring_slot_idx[b];
        if (slot >= p->max_slots || rs < 0 || rs >= ring_rows) {
            rc = -1;
            break;
        }
        for (int h = 0; h < nv; ++h) {
            const int hk = h / r, jr = h % r;
            const size_t sbase = (((size_t)slot * nv + h) * K) * V;
            for (size_t e = 0; e < (size_t)K * V; ++e)
                S[e] = SFX(load_state)(p, sbase + e);
            for (int t = 0; t < c; ++t) {
                const size_t rec =
                    (((size_t)rs * nk + hk) * ring_len + (size_t)t) * (size_t)record_stride;
                const REAL alpha = SFX(load_elem)(ring, ring_bf16, rec + K + jr);
                const size_t ur = rec + K + ((r + 7) / 8) * 8 + (size_t)jr * V;
                for (int i = 0; i < K; ++i)
                    for (int j = 0; j < V; ++j)
                        S[(size_t)i * V + j] = alpha * S[(size_t)i * V + j];
                for (int i = 0; i < K; ++i)
                    for (int j = 0; j < V; ++j)
                        S[(size_t)i * V + j] =
                            S[(size_t)i * V + j] + SFX(load_elem)(ring, ring_bf16, rec + i) *
                                                       SFX(load_elem)(ring, ring_bf16, ur + j);
            }
            for (size_t e = 0; e < (size_t)K * V; ++e)
                SFX(store_elem)(p->state, p->state_bf16, sbase + e, S[e]);
        }
    }
    free(S);
    return rc;
}
