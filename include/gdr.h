/*
 * gdr.h -- C ABI of the GB300 gated delta rule (GDR) recurrence library (libgdr.so).
 *
 * The library runs the slot-indexed, ragged-batch gated delta rule recurrence
 * and its speculative-decoding variants on one sm_103a GPU.  For every live
 * sequence b and value head h, with key head hk = h / (nv / nk) and the
 * state S = pool[slot_idx[b], h] stored [key index, value index], each token
 * t of the row [offsets[b], offsets[b+1]) does
 *
 *     q^ = q / sqrt(|q|^2 + eps),  k^ = k / sqrt(|k|^2 + eps)   (use_qk_l2norm)
 *     S  = alpha * S,   alpha = decay[t,h]  or  exp(decay[t,h])  (decay_is_log)
 *     u  = beta[t,h] * (v - S^T k^)
 *     S  = S + k^ u^T
 *     out[t, h*V:(h+1)*V] = scale * S^T q^
 *
 * Sources: "gated_delta_recurrence_fwd_gpu" (Modular kernels API), summary and
 * Args; "gated_delta_recurrence_verify_ring_gpu" (Modular Mojo API), summary
 * and Args; "gated_delta_recurrence_fwd_shape" (Modular Mojo API);
 * "core.ssm.ops.gdp.fused_recurrent" (Megatron-Core), module summary and the
 * Parameters of fused_recurrent_gated_delta_rule_update.
 *
 * Conventions shared by every entry point
 *   - Every buffer pointer is a DEVICE pointer owned by the caller (except the
 *     host buffers of gdr_host_io); the library allocates and frees nothing and
 *     keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  They never synchronise and never read device memory on the host;
 *     only gdr_get_status() synchronises.
 *   - Strides are in ELEMENTS.  Arithmetic is float32; per-token inputs and the
 *     output are float32; the pool is bfloat16 or float32.
 *   - Return value: GDR_OK, or a negative code with a message available from
 *     gdr_last_error() (thread-local).  Arguments are checked before anything
 *     is launched; an error launches nothing.
 *   - Problems the host cannot see (slot or ring row out of range, offsets not
 *     monotone, a row longer than max_row_len, a bad count or accepted index)
 *     are detected on the device: the affected (row, head) is skipped -- its
 *     output rows are zeroed where the call writes output -- and a bit is set
 *     in the device status word (GDR_STATUS_*), read with gdr_get_status().
 *   - Results do not depend on how a batch is composed or on which kernel the
 *     library picks: every pass uses one fixed order of float32 operations per
 *     (row, head), so the same row gives the same bits in any call.
 *   - Two live rows of one call must not share a pool slot (they would race).
 *   - Head sizes: K in {16, 32, 64, 128}; V = K, or V = 2K or (for K >= 32)
 *     V = K/2 for the forward, dense and snapshot passes and rollback
 *     ("core.ssm.ops.gdp.fused_recurrent" sizes K and V separately); the verify
 *     ring and fold need V = K, as "gated_delta_recurrence_verify_ring_gpu"
 *     requires.
 */
#ifndef GDR_H
#define GDR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes ------------------------------------------------------- */
#define GDR_OK 0
#define GDR_ERR_INVALID_ARG (-1) /* null pointer, negative size, nv % nk != 0, bad stride */
#define GDR_ERR_UNSUPPORTED (-2) /* head sizes, dtype, misalignment, unsupported mode      */
#define GDR_ERR_CUDA (-3)        /* a CUDA call or kernel launch failed                   */

/* ---- device status bits (sticky until cleared by gdr_get_status) -------- */
#define GDR_STATUS_BAD_SLOT 0x1u          /* slot_idx[b] < -1 or >= max_slots          */
#define GDR_STATUS_BAD_OFFSETS 0x2u       /* offsets not monotone or beyond T          */
#define GDR_STATUS_BAD_RING_SLOT 0x4u     /* ring_slot_idx[b] outside [0, ring_rows)   */
#define GDR_STATUS_BAD_COUNT 0x8u         /* fold count < 0                            */
#define GDR_STATUS_ROW_TOO_LONG 0x10u     /* a row longer than args.max_row_len        */
#define GDR_STATUS_BAD_ACCEPTED 0x20u     /* rollback index outside [-1, n_inter)      */
#define GDR_STATUS_SNAPSHOT_OVERFLOW 0x40u /* a row has more complete drafts than n_inter */

/* ---- dtypes ------------------------------------------------------------- */
typedef enum gdr_dtype { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;

/*
 * Arguments of one recurrence call ("gated_delta_recurrence_fwd_gpu", Args).
 *
 * qkv      [total_tokens, 2*nk*K + nv*V] float32, "qkv_conv_output": Q channels
 *          [0, nk*K), K channels [nk*K, 2*nk*K), V channels [2*nk*K, 2*nk*K + nv*V);
 *          key head hk occupies [hk*K, (hk+1)*K) inside its range, value head h
 *          occupies [h*V, (h+1)*V).  Element (t, c) is at t*qkv_seq_stride +
 *          c*qkv_chan_stride.
 * decay    [total_tokens, nv] float32: alpha, or the log decay g when
 *          decay_is_log != 0 ("core.ssm.ops.gdp.fused_recurrent", g).
 * beta     [total_tokens, nv] float32.  decay and beta share tok_seq_stride /
 *          tok_head_stride ("per_token_seqlen_stride", "per_token_head_stride").
 *          With beta_vdim_stride > 0, beta is per value element instead,
 *          [total_tokens, nv, V] ("core.ssm.ops.gdp.fused_recurrent", beta
 *          [B, T, HV, V]): element (t, h, j) at t*beta_seq_stride +
 *          h*beta_head_stride + j*beta_vdim_stride, and u_j = beta_j (v_j - ...).
 *          Forward and snapshot passes only (the verify pass takes [T, nv]).
 * out      [total_tokens, nv*V] float32; element (t, j) at t*out_seq_stride +
 *          j*out_vdim_stride.  Written for every token of every row.
 * state    [max_slots, nv, K, V] pool of state_dtype, read and written in place at
 *          slot_idx[b]; element (s, h, i, j) at s*state_slot_stride +
 *          h*state_head_stride + i*state_kdim_stride + j*state_vdim_stride.
 *          state_vdim_stride must be 1; the other three strides must keep every
 *          8-element (bf16) / 4-element (f32) group 16-byte aligned, and so must
 *          the base pointer.
 * slot_idx [batch] int32: pool slot of each row, -1 = padding request (output
 *          zeroed, nothing else written).  Same bits as the pages' uint32.
 * offsets  [batch+1] int32: row b spans [offsets[b], offsets[b+1]).
 * scale    query scale; <= 0 selects K^-0.5.
 * eps      added to |q|^2 and |k|^2 under the square root (1e-6 is customary).
 * max_row_len  an upper bound on every row's length, or <= 0 if unknown.  It only
 *          selects the kernel (1 picks the single-token decode kernel); a row
 *          longer than a positive bound is skipped and flagged
 *          GDR_STATUS_ROW_TOO_LONG.
 */
typedef struct gdr_step_args {
    int32_t batch;
    int32_t nv;
    int32_t nk;
    int32_t K;
    int32_t V;
    int32_t decay_is_log;
    int32_t use_qk_l2norm;
    int32_t state_dtype; /* gdr_dtype */
    int64_t total_tokens;
    int64_t max_row_len;
    const float *qkv;
    int64_t qkv_seq_stride;
    int64_t qkv_chan_stride;
    const float *decay;
    const float *beta;
    int64_t tok_seq_stride;
    int64_t tok_head_stride;
    float scale;
    float eps;
    float *out;
    int64_t out_seq_stride;
    int64_t out_vdim_stride;
    void *state;
    int64_t state_slot_stride;
    int64_t state_head_stride;
    int64_t state_kdim_stride;
    int64_t state_vdim_stride;
    int64_t max_slots;
    const int32_t *slot_idx;
    const int32_t *offsets;
    int64_t beta_seq_stride;  /* per-element beta only (beta_vdim_stride > 0) */
    int64_t beta_head_stride;
    int64_t beta_vdim_stride; /* 0: beta is [total_tokens, nv] */
} gdr_step_args;

/* Message for the last error returned on this thread ("" if none). */
const char *gdr_last_error(void);

/* Library version, e.g. 100 for 0.1.0. */
int gdr_version(void);

/* Output shape of a recurrence call: out_shape = {total_tokens, nv*V}
 * ("gated_delta_recurrence_fwd_shape": [total_seq_len, value_dim]). */
int gdr_output_shape(int64_t total_tokens, int32_t nv, int32_t V, int64_t out_shape[2]);

/* Minimum ring record length in elements for GQA ratio `ratio` = nv/nk
 * ("gated_delta_recurrence_verify_ring_gpu", ring_record_stride: at least
 * gated_delta_ring_record_elements(nv // nk)).  Record layout, in elements of
 * the ring's dtype:
 *     [ k^ (K) | alpha_0 .. alpha_{ratio-1}, padded to a multiple of 8 |
 *       u_0 (V) | ... | u_{ratio-1} (V) ]
 * (the padding elements are never written or read) where u_j and alpha_j
 * belong to value head hk*ratio + j.  Returns the length
 * (K + 8*ceil(ratio/8) + ratio*V) or a negative code. */
int gdr_ring_record_elements(int32_t K, int32_t V, int32_t ratio);

/* Forward pass ("gated_delta_recurrence_fwd_gpu"): runs every row over its
 * tokens, writes out for every token and writes each live row's final state
 * back to its slot (bf16 pools are rounded to nearest-even once, at the row
 * end).  Rows of length 0 leave their slot untouched. */
int gdr_fwd(const gdr_step_args *args, void *stream);

/*
 * Token inputs and output in HOST memory, for gdr_fwd_host.  Dense row-major
 * layouts with the shapes of gdr_step_args: qkv [total_tokens, 2*nk*K + nv*V],
 * decay and beta [total_tokens, nv], slot_idx [batch], offsets [batch+1],
 * out [total_tokens, nv*V].  Page-locked memory lets the copies run
 * asynchronously and overlap the compute; other host memory also works, with
 * copies that the CUDA runtime may serialise.
 */
typedef struct gdr_host_io {
    const float *qkv;
    const float *decay;
    const float *beta;
    const int32_t *slot_idx;
    const int32_t *offsets;
    float *out;
} gdr_host_io;

/* Forward pass over host-resident tokens ("gated_delta_recurrence_fwd_gpu",
 * the same computation as gdr_fwd, bit for bit).  `args` names the device
 * buffers the tokens are copied into -- qkv, decay, beta, slot_idx, offsets
 * and out, dense with the shapes above (qkv_seq_stride = 2*nk*K + nv*V,
 * tok_seq_stride = nv, out_seq_stride = nv*V, unit inner strides, head-wise
 * beta) -- and the device pool.  The rows are split into `chunks` groups of
 * consecutive rows (chunks <= 0: the library picks; at most 16 and at most
 * batch), with about equal token counts, except that with three or more groups
 * the first and the last get half as many (their copy in and copy out are the
 * ones no compute overlaps).  Each group's tokens are copied in on
 * h2d_stream, computed on `stream` and its output copied back on d2h_stream,
 * so one group's copies overlap its neighbours' compute (a NULL side stream
 * puts that direction on `stream`, without overlap).  Asynchronous on
 * `stream`: work already queued there precedes the copies, and once `stream`
 * has passed the call host->out holds every row's output and the pool the new
 * states; until then the device buffers and host->out must not be touched.
 * host->offsets is read on the host during the call (it must be monotone,
 * within [0, total_tokens]).  On its first call on a device a host thread
 * creates a few CUDA events that it keeps until exit; no memory is allocated.
 */
int gdr_fwd_host(const gdr_step_args *args, const gdr_host_io *host, int32_t chunks, void *stream,
                 void *h2d_stream, void *d2h_stream);

/* gdr_fwd_host without any device buffers from the caller.  (The pages have
 * no counterpart: this is an entry point for callers that cannot allocate.)
 * Some callers cannot call cudaMalloc or any other allocator: code running
 * where an allocation is not allowed or not wanted (a plug-in that is handed
 * host buffers and a stream only, a stream capture that forbids allocation,
 * a process whose device memory budget belongs to someone else).  This entry
 * point stages the tokens and the output in one fixed device array that the
 * library defines statically: 32 MiB on every GPU that loads the library,
 * held until the process exits.  `args` is read as for gdr_fwd_host except
 * that its qkv, decay, beta, slot_idx, offsets and out pointers and strides
 * are ignored (the library places dense copies in its array); the pool is the
 * caller's, on the device, as always.  A call whose staging would exceed the
 * array (about 4 * T * (2*nk*K + 2*nv*V + 2*nv) bytes) returns
 * GDR_ERR_UNSUPPORTED without launching anything.  Nothing is allocated: the
 * first call on a device looks up the array's device address (keep that first
 * call out of any stream capture); later calls reuse it.  Every call on a
 * device shares the one array and each call overwrites what it reads, so
 * calls that overlap on the GPU (on different streams, or from several host
 * threads without ordering) race: order them on one stream. */
int gdr_fwd_host_noalloc(const gdr_step_args *args, const gdr_host_io *host, int32_t chunks, void *stream,
                         void *h2d_stream, void *d2h_stream);

/*
 * Pass-1 convolution of gdr_fwd_conv ("gated_delta_recurrence_fwd_gpu", Args:
 * qkv_conv_output is the "Conv1d output from Pass 1").  The pages give only
 * the output's layout; the convolution is the causal depthwise one over the
 * conv_dim = 2*nk*K + nv*V channels, every parameter from the caller: for
 * token j of a row and channel c, with xe = the slot's conv state for c
 * (oldest first) followed by the row's raw inputs x[t, c],
 *     y[t0+j, c] = act(bias[c] + sum_m weight[c, m] * xe[j + m]),  m = 0 .. width-1
 * (tap width-1 multiplies the newest input; act is the identity or SiLU
 * y / (1 + exp(-y))), evaluated in float32 as y = bias, then
 * y = fma(weight[c, m], xe[j + m], y) for m = 0, 1, ..., then the activation
 * (with the fast single-precision exponential and division: a few ulp).
 * The conv state pool [max_slots, conv_dim, width-1] is float32, indexed by
 * the args' slot_idx like the recurrence pool, and replaced by the last
 * width-1 entries of xe (a row shorter than width-1 keeps part of it);
 * padding and empty rows leave it alone.
 */
typedef struct gdr_conv_args {
    int32_t width;      /* taps per channel, 1 .. 4                                     */
    int32_t activation; /* 0: none, 1: SiLU                                             */
    const float *weight;          /* [conv_dim, width]: element (c, m) at               */
    int64_t weight_chan_stride;   /*   c*weight_chan_stride + m*weight_tap_stride         */
    int64_t weight_tap_stride;
    const float *bias;            /* [conv_dim], unit stride, or NULL (no bias)          */
    float *conv_state;            /* [max_slots, conv_dim, width-1]; NULL when width == 1 */
    int64_t state_slot_stride;
    int64_t state_chan_stride;
    int64_t state_tap_stride;
} gdr_conv_args;

/* Forward pass on the RAW Pass-1 input ("gated_delta_recurrence_fwd_gpu" with
 * its qkv_conv_output produced in the same call): args->qkv holds the
 * convolution's input x [total_tokens, conv_dim] (same channel layout and
 * strides as qkv_conv_output); the kernel convolves each staged chunk of
 * tokens as it stages them (the convolution output is never written to
 * memory), runs the recurrence exactly as gdr_fwd on the result, and then
 * replaces every live row's conv state.  V = K and head-wise beta only.  A
 * width-1 filter of weight 1, no bias and no activation gives gdr_fwd's
 * results bit for bit.  The conv state must not alias any other buffer. */
int gdr_fwd_conv(const gdr_step_args *args, const gdr_conv_args *conv, void *stream);

/* Forward pass with a dense start and end state ("core.ssm.ops.gdp.fused_recurrent",
 * initial_state [N, HV, K, V] or None for zeros, output_final_state): as gdr_fwd,
 * but row b starts from initial_state[b] (zeros when initial_state is NULL) and
 * its final state is written to final_state[b] (nothing when NULL; at least one
 * of the two must be given).  Both are [batch, nv, K, V] in state_dtype with
 * the args' state strides (state_slot_stride steps between rows) and 16-byte
 * alignment.  args->state, slot_idx and max_slots are ignored; every row is
 * live, and an empty row writes its start state to final_state.  The buffers
 * may be the same (in-place update). */
int gdr_fwd_dense(const gdr_step_args *args, const void *initial_state, void *final_state,
                  void *stream);

/* Verify pass ("gated_delta_recurrence_verify_ring_gpu", summary): writes the
 * same out as gdr_fwd and leaves the pool untouched, except that a row longer
 * than ring_len records nothing and commits its state exactly as gdr_fwd does.
 * A row with L <= ring_len writes record t - offsets[b] of
 *     ring[ring_slot_idx[b], hk, :, :]   (ring is [ring_rows, nk, ring_len, record_stride])
 * for each token, in the layout of gdr_ring_record_elements.  Padding rows
 * write no records.  ring_dtype is GDR_F32 or GDR_BF16 (Parameters: ring_dtype;
 * bfloat16 records are rounded to nearest-even once, and only a float32 ring
 * keeps the fold bit-exact against the forward pass); the ring must be
 * 16-byte aligned; record_stride must be a multiple of 4 (float32) or 8
 * (bfloat16) and at least gdr_ring_record_elements(K, V, nv/nk);
 * 1 <= ring_len <= 32. */
int gdr_verify_ring(const gdr_step_args *args, void *ring, int32_t ring_dtype,
                    int64_t ring_rows, int32_t ring_len, int64_t record_stride,
                    const int32_t *ring_slot_idx, void *stream);

/* Fold ("gated_delta_recurrence_verify_ring_gpu", summary; the pages name the
 * kernel gated_delta_state_fold_gpu): advances each live row's slot over the
 * first counts[b] records of its ring row, S = alpha_t S + k^_t u_t^T, and
 * writes it back.  counts[b] == 0 or counts[b] > ring_len leaves the row alone
 * (a row longer than ring_len was already committed by the verify pass, so a
 * caller passes its full length).  With a float32 ring the result equals
 * gdr_fwd over the accepted prefix bit for bit; a bfloat16 ring is widened
 * exactly.  The ring needs element alignment only (16 bytes for the fast
 * kernel).  Uses from `args`: batch, nv,
 * nk, K, V, state*, max_slots, slot_idx (qkv/decay/beta/out/offsets unused). */
int gdr_fold(const gdr_step_args *args, const void *ring, int32_t ring_dtype,
             int64_t ring_rows, int32_t ring_len, int64_t record_stride,
             const int32_t *ring_slot_idx, const int32_t *counts, void *stream);

/* Forward pass with per-draft-token snapshots ("core.ssm.ops.gdp.fused_recurrent",
 * intermediate_states and steps_per_token): as gdr_fwd, and in addition the
 * state after step (i+1)*steps_per_token - 1 of a row is stored at
 *     inter[slot, i, h, :, :]  = inter + slot*inter_slot_stride +
 *                               i*inter_token_stride + h*inter_head_stride
 * (a dense [K, V] block in the pool's dtype) for every i < n_inter.  inter is
 * indexed by pool slot: it must hold a block row for every slot in
 * [0, max_slots) (a slot the device accepts as valid is never checked against
 * a smaller buffer).  A partial trailing draft is not stored; padding rows
 * store nothing.  A row with more
 * complete drafts than n_inter stores the first n_inter and sets
 * GDR_STATUS_SNAPSHOT_OVERFLOW.  Strides must keep 16-byte alignment. */
int gdr_fwd_snapshots(const gdr_step_args *args, void *inter, int64_t inter_slot_stride,
                      int64_t inter_token_stride, int64_t inter_head_stride,
                      int32_t n_inter, int32_t steps_per_token, void *stream);

/* Rollback ("core.ssm.ops.gdp.fused_recurrent", intermediate_states: roll the
 * recurrence back to any accepted prefix): state[slot_idx[b], h] <-
 * inter[slot_idx[b], accepted[b], h] for every value head.  accepted[b] == -1
 * or slot -1 skips the row.  As for gdr_fwd_snapshots, inter must hold a block
 * row for every slot in [0, max_slots).  Uses from `args`: batch, nv, K, V, state*,
 * max_slots, slot_idx. */
int gdr_rollback(const gdr_step_args *args, const void *inter, int64_t inter_slot_stride,
                 int64_t inter_token_stride, int64_t inter_head_stride, int32_t n_inter,
                 const int32_t *accepted, void *stream);

/* Reads the current device's status word (GDR_STATUS_* bits) into *status and,
 * if clear != 0, resets it.  Synchronises the device. */
int gdr_get_status(uint32_t *status, int32_t clear);

/* Diagnostic, not part of the recurrence: measures how fast the FP32 pipe runs
 * packed float32x2 arithmetic of a given register-operand pattern, every
 * operand already in registers (no memory traffic).  It bounds what the
 * recurrence kernels can reach on the FP32 pipe with their fixed operation
 * order (the per-element decay multiply, rank-1 update and two reductions of
 * "gated_delta_recurrence_fwd_gpu"'s per-token step).  Launches one CTA of
 * 128 * warps_per_subpartition threads on every SM (*ctas receives the CTA
 * count) on `stream`; each thread runs `iterations` iterations of:
 *   pattern 0: the recurrence sweep on 64 rows x 2 columns -- per state
 *              element pair t = alpha x; x = k^ u + t; a += x k'; b += x q'
 *              (8-row chains) -- then a short dependent tail feeding the next
 *              iteration: 256 packed instructions, 512 FP32 operations;
 *   pattern 1: 8 independent packed FMA chains whose multiplier and addend
 *              registers are the same in every instruction: 8 packed, 16 ops;
 *   pattern 2: 8 independent packed FMA chains with three distinct operand
 *              registers per instruction: 8 packed, 16 ops.
 * Every thread writes one float to sink[cta * blockDim + thread]; sink must hold
 * sink_elements >= SMs * 128 * warps_per_subpartition floats.  Time it with
 * events on `stream`.  Returns GDR_ERR_UNSUPPORTED when the pattern's CTA does
 * not fit one SM's registers at that warp count, GDR_ERR_INVALID_ARG for a
 * pattern outside 0..2, warps outside 1..8, iterations < 1 or a null or short
 * sink. */
int gdr_probe_fma(int32_t pattern, int32_t warps_per_subpartition, int32_t iterations, float *sink,
                  int64_t sink_elements, int32_t *ctas, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GDR_H */
