/*
 * CPU oracle for the gated delta rule (GDR) recurrence -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously-correct restatement of what the GPU
 * library computes.  It shares no code, header, table or helper with the CUDA
 * path under gated_deltanet_linear_gdr_gb300/csrc, and nothing in the product
 * path may load it: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg do.
 *
 * Sources restated here (page title, section):
 *   - "gated_delta_recurrence_fwd_gpu" (Modular kernels API), summary and Args:
 *     slot-indexed pool [max_slots, nv, K, V] read and written in place at
 *     slot_idx[b]; qkv_conv_output [T, conv_dim] with Q in [0, key_dim), K in
 *     [key_dim, 2*key_dim), V in [2*key_dim, 2*key_dim + value_dim); per-token
 *     per-head decay and beta [T, nv]; ragged rows [off[b], off[b+1]);
 *     GQA ratio nv/nk; L2 normalisation of q and k; query scale 1/sqrt(K).
 *   - "gated_delta_recurrence_verify_ring_gpu" (Modular Mojo API), summary:
 *     verify writes the same output as the forward pass, leaves the pool
 *     alone, and writes one ring record per token; a row longer than RING_LEN
 *     records nothing and commits like the forward pass; the fold skips a row
 *     whose count exceeds RING_LEN.  Args: ring [ring_rows, nk, RING_LEN,
 *     ring_record_stride] indexed by ring_slot_idx[b].
 *   - "core.ssm.ops.gdp.fused_recurrent" (Megatron-Core), module summary and
 *     Parameters: g is a log decay (alpha = exp(g)); beta is head-wise
 *     [T, HV] or per value element [T, HV, V]; state_indices -1 marks a
 *     padding request (zero output, state untouched, no snapshot writes);
 *     intermediate_states[slot, i] holds the state after draft token i, i.e.
 *     after every steps_per_token recurrence steps.
 *
 * The recurrence, per (sequence, value head h, key head hk = h / (nv/nk)), per
 * token, with S stored [key index, value index]:
 *     q^ = q / sqrt(|q|^2 + eps),  k^ = k / sqrt(|k|^2 + eps)   (if enabled)
 *     S  = alpha * S                                 (gate / decay)
 *     u  = beta * (v - S^T k^)                       (delta-rule correction)
 *     S  = S + k^ u^T                                (rank-one update)
 *     o  = scale * S^T q^                            (readout of the new state)
 *
 * Readings where the pages are silent:
 *   - order decay -> correction -> update -> readout (readout of the updated
 *     state), matching S_t = alpha (I - beta k k^T) S_{t-1} + beta k v^T;
 *   - value head h reads key head h / (nv/nk) (contiguous GQA groups);
 *   - heads are contiguous inside each of the Q, K, V channel ranges and in
 *     the output;
 *   - eps = 1e-6 inside the square root (passed in);
 *   - a bf16 pool is widened exactly on load and rounded to nearest-even once
 *     per call at the end of the row;
 *   - ring record layout, in elements of the ring's dtype (float32, or
 *     bfloat16 rounded to nearest-even from the computed value):
 *       [ k^ (K) | alpha_0 .. alpha_{r-1}, padded to a multiple of 8 |
 *         u_0 (V) | u_1 (V) | ... | u_{r-1} (V) ]
 *     where j = h mod r is the value head's position inside its key head
 *     ("gated_delta_recurrence_verify_ring_gpu" Parameters: ring_dtype; only
 *     a float32 ring keeps the fold bit-exact against the forward pass);
 *   - snapshot i is taken after step (i+1)*steps_per_token - 1 of the row;
 *     a partial trailing draft is not snapshotted.
 *
 * Arithmetic: the core below is compiled twice, once in double (the default
 * oracle) and once in float (the pages' float32 work type, used to check the
 * bit-exact fold contract).  Build with -ffp-contract=off so that no multiply
 * and add are fused behind the source's back.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t batch, nv, nk, K, V;
    int64_t total_tokens;
    const float *qkv;    /* [T, 2*nk*K + nv*V], dense                      */
    const float *decay;  /* [T, nv]: alpha, or g when decay_is_log          */
    const float *beta;   /* [T, nv], or [T, nv, V] when beta_per_value      */
    int32_t decay_is_log, use_l2norm;
    double scale;        /* <= 0 selects K^-0.5                             */
    double eps;
    void *state;         /* [max_slots, nv, K, V]: float32, or bf16 bits    */
    int32_t state_bf16;
    int64_t max_slots;
    const int32_t *slot_idx; /* [batch], -1 = padding                       */
    const int32_t *offsets;  /* [batch + 1]                                 */
    int32_t beta_per_value;
} oracle_problem;

/* ---- storage conversions (shared by both precisions) ------------------- */

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the bfloat16 grid, ties to even.  bfloat16 keeps the
 * float32 exponent range and 8 significant bits, so a finite non-zero value
 * a = m * 2^e (m in [0.5, 1)) is quantised in steps of 2^(e-8), never finer
 * than the subnormal step 2^-133. */
uint16_t oracle_round_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    (void)frexp(a, &e);
    int qexp = e - 8;
    if (qexp < -133)
        qexp = -133;
    double r = rint(ldexp(a, -qexp)); /* default mode: nearest, ties to even */
    double y = ldexp(r, qexp);
    if (y >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)y; /* exact: y lies on the bfloat16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

double oracle_bf16_to_double(uint16_t b) { return bf16_bits_to_double(b); }

/* Minimum ring record length in elements for a GQA ratio r (record layout above). */
int oracle_ring_record_elements(int K, int V, int r)
{
    if (K <= 0 || V <= 0 || r <= 0)
        return -1;
    return K + ((r + 7) / 8) * 8 + r * V;
}

static int check_problem(const oracle_problem *p)
{
    if (!p || p->batch < 0 || p->nv <= 0 || p->nk <= 0 || p->K <= 0 || p->V <= 0)
        return -1;
    if (p->nv % p->nk != 0 || p->total_tokens < 0 || p->max_slots < 0)
        return -1;
    if (p->batch > 0 && (!p->slot_idx || !p->offsets))
        return -1;
    if (p->total_tokens > 0 && (!p->qkv || !p->decay || !p->beta))
        return -1;
    if (p->offsets && p->batch >= 0 && p->offsets[0] < 0)
        return -1;
    for (int b = 0; b < p->batch; ++b) {
        if (p->offsets[b + 1] < p->offsets[b] || p->offsets[b + 1] > p->total_tokens)
            return -1;
        if (p->slot_idx[b] < -1 || p->slot_idx[b] >= p->max_slots)
            return -1;
    }
    return 0;
}

/* ---- the recurrence, once per precision -------------------------------- */

#define REAL double
#define SFX(name) name##_f64
#define SQRT sqrt
#define EXP exp
#include "gdr_oracle_core.h"
#undef REAL
#undef SFX
#undef SQRT
#undef EXP

#define REAL float
#define SFX(name) name##_f32
#define SQRT sqrtf
#define EXP expf
#include "gdr_oracle_core.h"
#undef REAL
#undef SFX
#undef SQRT
#undef EXP

/* ---- Pass-1 causal depthwise convolution ------------------------------- */

/* "gated_delta_recurrence_fwd_gpu", Args: qkv_conv_output is the "Conv1d
 * output from Pass 1".  The pages give only that output's layout; the
 * convolution is taken as the plain causal depthwise one over the conv_dim
 * channels, with every parameter from the caller (readings, each a choice the
 * pages leave open):
 *   - each channel c has its own `width` taps w[c][0..width-1]; for token j of
 *     a row, with xe = (the slot's conv state for c, oldest first) followed by
 *     the row's inputs x[t0 .. t1-1][c],
 *         y[t0+j][c] = bias[c] + sum_m w[c][m] * xe[j + m]
 *     so tap width-1 multiplies the newest input x[t0+j][c];
 *   - bias is optional (none: 0); the activation is none or SiLU,
 *     y / (1 + exp(-y));
 *   - the conv state pool [max_slots, channels, width-1] (float32) is read at
 *     slot_idx[b] and replaced by the last width-1 entries of xe (a row
 *     shorter than width-1 keeps part of the old state);
 *   - a padding row (slot -1) or an empty row leaves the slot alone; its
 *     output rows are set to 0;
 *   - the output is float32, the layout of qkv_conv_output.
 * Computed in double, rounded to float once. */
int oracle_conv1d(int32_t batch, int64_t total_tokens, int32_t channels, int32_t width,
                  const float *x, const float *weight, const float *bias, int32_t silu,
                  float *conv_state, int64_t max_slots, const int32_t *slot_idx,
                  const int32_t *offsets, float *y)
{
    if (batch < 0 || total_tokens < 0 || channels <= 0 || width < 1 || !weight || !slot_idx ||
        !offsets || !y || (total_tokens > 0 && !x) || (width > 1 && !conv_state && batch > 0))
        return -1;
    const int w1 = width - 1;
    double *xe = (double *)malloc(sizeof(double) * (size_t)(w1 + total_tokens + 1));
    if (!xe)
        return -1;
    for (int b = 0; b < batch; ++b) {
        const int t0 = offsets[b], t1 = offsets[b + 1], slot = slot_idx[b];
        if (t0 < 0 || t1 < t0 || t1 > total_tokens || slot < -1 || slot >= max_slots) {
            free(xe);
            return -1;
        }
        const int L = t1 - t0;
        if (slot < 0) {
            for (int t = t0; t < t1; ++t)
                for (int c = 0; c < channels; ++c)
                    y[(size_t)t * channels + c] = 0.0f;
            continue;
        }
        if (L == 0)
            continue;
        for (int c = 0; c < channels; ++c) {
            float *st = conv_state ? conv_state + ((size_t)slot * channels + c) * w1 : NULL;
            for (int i = 0; i < w1; ++i)
                xe[i] = st[i];
            for (int j = 0; j < L; ++j)
                xe[w1 + j] = x[(size_t)(t0 + j) * channels + c];
            for (int j = 0; j < L; ++j) {
                double acc = bias ? (double)bias[c] : 0.0;
                for (int m = 0; m < width; ++m)
                    acc += (double)weight[(size_t)c * width + m] * xe[j + m];
                if (silu)
                    acc = acc / (1.0 + exp(-acc));
                y[(size_t)(t0 + j) * channels + c] = (float)acc;
            }
            for (int i = 0; i < w1; ++i)
                st[i] = (float)xe[L + i];
        }
    }
    free(xe);
    return 0;
}

/* ---- rollback: a plain copy, the same in both precisions --------------- */

/* state[slot, h] <- intermediate[slot, accepted[b], h] for every value head.
 * Padding (slot -1) and accepted -1 are skipped ("core.ssm.ops.gdp.fused_recurrent",
 * intermediate_states: roll back to any accepted prefix). */
int oracle_rollback(const oracle_problem *p, const void *inter, int n_inter,
                    const int32_t *accepted)
{
    if (check_problem(p) != 0 || n_inter <= 0 || !inter || !accepted)
        return -1;
    const size_t esz = p->state_bf16 ? 2 : 4;
    const size_t head = (size_t)p->K * p->V;
    for (int b = 0; b < p->batch; ++b) {
        int slot = p->slot_idx[b], a = accepted[b];
        if (slot < 0 || a < 0)
            continue;
        if (a >= n_inter)
            return -1;
        for (int h = 0; h < p->nv; ++h) {
            const char *src = (const char *)inter +
                esz * ((((size_t)slot * n_inter + a) * p->nv + h) * head);
            char *dst = (char *)p->state + esz * (((size_t)slot * p->nv + h) * head);
            memcpy(dst, src, esz * head);
        }
    }
    return 0;
}
