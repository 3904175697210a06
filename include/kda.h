/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library: the chunked
 * forward, the decode step and the backward pass.
 *
 * The operation is the chunked forward pass of Kimi Delta Attention (KDA), as
 * stated by the FlashKDA README ("Kernel API", flash_kda.fwd parameter table)
 * together with the KDA recurrence, per sequence n and head h (K = V = 128 in the
 * README; the shapes this library also takes are listed with kda_shape):
 *
 *   ghat_t  = lower_bound * sigmoid(exp(A_log[h]) * (g_t + dt_bias[h,:]))  (per channel;
 *             the reference call's safe gate, the default; see kda_flags for the others)
 *   S_t     = (I - beta_t k_t k_t^T) Diag(exp(ghat_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t     = scale * S_t^T q_t
 *
 * with beta_t = sigmoid(beta logit) (applied in the kernel, per the README), q_t and
 * k_t L2-normalised per token and head (x / sqrt(|x|^2 + 1e-6)), and the state
 * S (K x V) stored transposed as [.., V, K] (FLA transpose_state_layout=True).
 * The device computes it in 16-token chunks, as FlashKDA does (instagit index); the
 * chunk's unit lower-triangular system is inverted in fp32 by forward
 * substitution (FlashKDA's articles use a Neumann-series product; both give the exact
 * inverse of a 16 x 16 unit lower-triangular matrix).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers to contiguous row-major tensors.
 *    q, k, v, g and the states must be 16-byte aligned, beta and out 2-byte,
 *    A_log 4-byte, and dt_bias 16-byte for kda_fwd and kda_bwd (4-byte for
 *    kda_decode).  The caller owns all memory; the library allocates none and
 *    never synchronises the host (except kda_check_device_error).
 *  - Work is stream-ordered on `stream` (0 = legacy default stream).
 *  - Inputs are never modified; `out` and `final_state` are fully overwritten.
 *  - Errors in the arguments are reported by the return code before anything
 *    is launched.  Errors found on the device (malformed cu_seqlens, a wait
 *    that ran out of time) are recorded in the workspace's error word and read
 *    back with kda_check_device_error; kernels never trap.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kda_stream_t; /* a cudaStream_t */

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, bad size, lower_bound out of range */
    KDA_ERR_UNSUPPORTED_SHAPE = 2,  /* K other than 64 and 128, or V other than 64, 128 and 256 */
    KDA_ERR_WORKSPACE_TOO_SMALL = 3,
    KDA_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    KDA_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed */
    KDA_ERR_TIMEOUT = 6,            /* a device-side wait ran out of time (error word) */
    KDA_ERR_BAD_SEQLENS = 7,        /* cu_seqlens not monotone or not ending at T (error word) */
    KDA_ERR_GATE_RANGE = 8          /* reserved: no longer raised (chunks past 2^-250 are computed) */
} kda_status;

/* State dtype for initial_state / final_state (README: absent, bf16 or fp32). */
typedef enum { KDA_STATE_NONE = 0, KDA_STATE_BF16 = 1, KDA_STATE_FP32 = 2 } kda_state_dtype;

/*
 * Steps the caller has already done, as flags (0 = FlashKDA's fixed behaviour:
 * the gate, the beta sigmoid and the q/k L2 norms are all computed in the
 * kernel).  They mirror the reference call's use_gate_in_kernel,
 * use_beta_sigmoid_in_kernel and use_qk_l2norm_in_kernel switches, set here
 * when the switch is off:
 *   KDA_GATE_PREACTIVATED : g holds the natural-log decay ghat itself; A_log,
 *                           dt_bias and lower_bound are not read (A_log and
 *                           dt_bias may be NULL).  Values must be <= 0.
 *   KDA_BETA_PREACTIVATED : beta holds beta itself, not its logit.
 *   KDA_NO_QK_L2NORM      : q and k are used as given.
 * and one selects the reference call's other gate (its safe_gate switch off):
 *   KDA_GATE_SOFTPLUS     : ghat = -exp(A_log[h]) * softplus(g + dt_bias[h,:]),
 *                           with no lower bound; lower_bound is not read.  Not
 *                           together with KDA_GATE_PREACTIVATED.
 * The chunked form of kda_fwd_ex factors the decay inside each 16-token chunk
 * about half the chunk's total, which is exact while that total stays within
 * 2^-250 (a sum of ghat above -173 over the chunk's 16 tokens on every
 * channel).  The in-kernel safe gate never leaves this range (16 x 5 < 173).
 * With a preactivated or softplus gate, the 32 channels of a chunk that leave
 * it take a direct route instead (every factor 2^G, 2^(G_C - G) and, per token
 * pair, 2^(G_i - G_j), all at most 1), so any decay is computed exactly;
 * KDA_ERR_GATE_RANGE is kept in the status list but kda_fwd_ex no longer
 * raises it.  kda_decode runs the token recurrence itself and takes any gate
 * values.
 *
 * One more flag is not a step of the method but a precision request:
 *   KDA_PRECISE_STATE     : the chunked form reads the carried state as a bf16 pair
 *                           (hi + lo) instead of one bf16 copy, so the rounding of that
 *                           copy (2^-9 relative, fed back every chunk) no longer builds
 *                           up when the gate hardly decays.  Runs one CTA per SM
 *                           (about half the throughput).  kda_fwd_ex turns it on by
 *                           itself for the safe gate with lower_bound > -0.25 and for
 *                           the preactivated and softplus gates, whose decay it cannot
 *                           bound; with a decaying gate the single copy's error fades
 *                           within a few chunks and the flag changes little.
 *                           kda_decode and kda_bwd ignore it.
 * And one selects the backward's form (kda_bwd only):
 *   KDA_BWD_RECURRENT     : the token-by-token fp32 recurrence (gradients exact to fp32
 *                           rounding) instead of the chunked tensor-core form, whose
 *                           bf16 operands put the gradients within 1e-2 relative
 *                           Frobenius of the exact ones.  The preactivated and softplus
 *                           gates always take the recurrent form.
 */
typedef enum {
    KDA_GATE_PREACTIVATED = 1,
    KDA_BETA_PREACTIVATED = 2,
    KDA_NO_QK_L2NORM = 4,
    KDA_GATE_SOFTPLUS = 8,
    KDA_PRECISE_STATE = 16,
    KDA_BWD_RECURRENT = 32
} kda_flags;

/*
 * Problem shape (README parameter table; the README requires K = V = 128, this
 * library also takes V = 256, run as two independent 128-row halves of each
 * state, V = 64, run as one 128-row chain whose last 64 rows stay zero, and
 * K = 64, run with key channels 64-127 held at zero: q = k = 0 and decay 1
 * there, so those state columns stay zero and add nothing to the outputs):
 *   q, k, g : [B, T, H, K] bf16      v, out : [B, T, H, V] bf16
 *   beta    : [B, T, H]    bf16 (logits)
 *   A_log   : [H] fp32               dt_bias : [H, K] fp32
 *   states  : [N, H, V, K]           cu_seqlens : int64 [N + 1]
 * N is the number of sequences: N = B without cu_seqlens (the README treats every
 * batch row as its own sequence); with cu_seqlens B must be 1 and T
 * is the total length across all sequences.
 */
typedef struct {
    int64_t B, T, H, K, V, N;
} kda_shape;

/* Human-readable name of a status code (static storage, never NULL). */
KDA_API const char *kda_status_string(kda_status s);

/*
 * Bytes of device workspace kda_fwd needs for this shape.  The size is linear
 * in the number of heads and of sequence tiles (the instagit workspace-size article
 * states the same growth): it holds the device-side
 * work list and, for sequences split into segments, one pair of 128 x 128
 * fp32 segment transition/carry matrices per (segment, head).
 * Returns KDA_ERR_INVALID_ARGUMENT / KDA_ERR_UNSUPPORTED_SHAPE for bad shapes.
 */
KDA_API kda_status kda_workspace_size(const kda_shape *shape, size_t *bytes);

/*
 * The forward pass (README flash_kda.fwd).
 *   q, k, v, g, beta : bf16 inputs as above.
 *   scale            : output scale (the README's scale argument).
 *   out              : bf16 [B, T, H, V], written for every token.
 *   A_log, dt_bias   : fp32 gate parameters.
 *   lower_bound      : gate lower bound, must lie in [-5, 0] (README range);
 *                      not read with KDA_GATE_PREACTIVATED or KDA_GATE_SOFTPLUS.
 *   initial_state    : NULL (zeros) or [N, H, V, K] of init_dtype.
 *   final_state      : NULL (not written) or [N, H, V, K] of final_dtype;
 *                      when both states are given their dtypes must match
 *                      (README), and final_state may be exactly the same
 *                      buffer as initial_state (in-place update); partial
 *                      overlap is not allowed.
 *   cu_seqlens       : NULL or int64 [N + 1] device array, cu[0] = 0,
 *                      non-decreasing, cu[N] = T (zero-length sequences allowed:
 *                      their final state equals their initial state).
 *   workspace        : device scratch of at least kda_workspace_size bytes,
 *                      256-byte aligned; its contents are undefined afterwards,
 *                      except the error word read by kda_check_device_error.
 * Returns KDA_OK once the kernels are enqueued.
 */
KDA_API kda_status kda_fwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                   const void *g, const void *beta, float scale, void *out, const float *A_log,
                   const float *dt_bias, float lower_bound, const void *initial_state,
                   kda_state_dtype init_dtype, void *final_state, kda_state_dtype final_dtype,
                   const int64_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                   kda_stream_t stream);

/*
 * kda_fwd with `flags` (kda_flags, or-ed): steps the caller has already done.
 * kda_fwd(...) is kda_fwd_ex(..., 0, ...).
 */
KDA_API kda_status kda_fwd_ex(const kda_shape *shape, const void *q, const void *k, const void *v,
                              const void *g, const void *beta, float scale, void *out, const float *A_log,
                              const float *dt_bias, float lower_bound, const void *initial_state,
                              kda_state_dtype init_dtype, void *final_state, kda_state_dtype final_dtype,
                              const int64_t *cu_seqlens, unsigned flags, void *workspace,
                              size_t workspace_bytes, kda_stream_t stream);

/*
 * Synchronises `stream`, reads the error word that the last kda_fwd on this
 * workspace left behind, stores it in *flags (0 = none; bit 0 = a device wait
 * timed out; bit 1 = malformed cu_seqlens; bit 2 = reserved for
 * KDA_ERR_GATE_RANGE, no longer set) and returns KDA_OK, KDA_ERR_TIMEOUT or
 * KDA_ERR_BAD_SEQLENS accordingly.
 */
KDA_API kda_status kda_check_device_error(const void *workspace, kda_stream_t stream, int *flags);

/*
 * Measurement aid (no counterpart in flash_kda): while `events` is non-NULL,
 * every kda_fwd records events[i] (cudaEvent_t handles owned by the caller) on
 * its stream right after its i-th phase -- 0: work-list scheduling, 1: the
 * segment transition runs and the forward runs (two launches, the second
 * overlapping the first), 2: carry composition and the segment corrections (two
 * launches, the second starting beside the first: no event between them), 3:
 * recorded with 2 -- so each phase can be timed with cudaEventElapsedTime
 * (phases a call does not need are recorded empty).  n_events must be 4.
 * Pass NULL to stop.  The setting is process-wide and not thread-safe.
 */
KDA_API kda_status kda_set_profile_events(void *const *events, int n_events);

/*
 * Measurement aid (no counterpart in flash_kda): the number of kernels the
 * calling thread's most recent successful kda_fwd enqueued (2 to 4: work-list
 * scheduling, forward runs, carry composition, segment corrections).
 */
KDA_API int kda_last_launch_count(void);

/*
 * kda_fwd for callers that cannot allocate device memory (no counterpart in
 * flash_kda).  Some callers have no way to hand over scratch memory: code that
 * runs where cudaMalloc is not allowed (a framework that owns every device
 * allocation through its own pool, a runtime that must not grow its footprint
 * after start-up, a plugin without access to the application's allocator).
 * This entry point takes the same arguments as kda_fwd except the workspace,
 * which it takes from a fixed 64 MiB array built into the library; every GPU
 * that loads the library holds that array until the process exits.  The
 * caller still passes all inputs and outputs.
 *   - Problems whose kda_workspace_size exceeds 64 MiB are rejected with
 *     KDA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - It allocates nothing and calls no allocating routine.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, different threads, without ordering between them)
 *     race on it and give undefined results.  Nothing in it needs clearing
 *     between calls.  Its device error word cannot be read back through
 *     kda_check_device_error, which needs a workspace address.
 */
KDA_API kda_status kda_fwd_static_workspace(const kda_shape *shape, const void *q, const void *k,
                                            const void *v, const void *g, const void *beta, float scale,
                                            void *out, const float *A_log, const float *dt_bias,
                                            float lower_bound, const void *initial_state,
                                            kda_state_dtype init_dtype, void *final_state,
                                            kda_state_dtype final_dtype, const int64_t *cu_seqlens,
                                            kda_stream_t stream);

/*
 * The recurrent step for decoding (no counterpart in flash_kda.fwd): the same
 * recurrence as kda_fwd, token by token, for B sequences of T tokens each
 * (T = 1 for one decoding step), with the state updated IN PLACE.  Every
 * (sequence, head) state is read from HBM once and written back once per call,
 * whatever T is; no workspace is needed.
 *   shape            : B sequences, T >= 0 tokens each, H heads, K = 64 or 128,
 *                      V = 64, 128 or 256, N = B.
 *   q, k, g          : bf16 [B, T, H, K]; v : bf16 [B, T, H, V]; beta : bf16 [B, T, H]
 *                      (logits); all 2-byte aligned.
 *   out              : bf16 [B, T, H, V], written for every token, 2-byte aligned.
 *   A_log, dt_bias, lower_bound, scale : as for kda_fwd.
 *   flags            : kda_flags, as for kda_fwd_ex.
 *   state            : [B, H, V, K] of state_dtype (bf16 or fp32), 16-byte aligned;
 *                      read as the state before the first token and overwritten with
 *                      the state after the last (a bf16 state is rounded once, at the
 *                      end of the call).  T = 0 leaves it untouched.
 * Returns KDA_OK once the kernel is enqueued; argument errors as for kda_fwd.
 */
KDA_API kda_status kda_decode(const kda_shape *shape, const void *q, const void *k, const void *v,
                              const void *g, const void *beta, float scale, void *out, const float *A_log,
                              const float *dt_bias, float lower_bound, void *state,
                              kda_state_dtype state_dtype, unsigned flags, kda_stream_t stream);

/*
 * The backward pass: gradients of L = sum(dout * out) + sum(dfinal * final_state) for the
 * forward kda_fwd_ex computes with the same arguments.  FlashKDA's README defines the forward
 * only ("Kernel API"); the gradient is that of its recurrence (above), taken through the
 * gate, the beta sigmoid and the L2 norms the flags leave in the kernel.  K = V = 128.
 *   q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state, init_dtype,
 *   cu_seqlens, flags : the forward's inputs, as for kda_fwd_ex (q, k, v, g 16-byte aligned).
 *   dout             : bf16 [B, T, H, V], dL/d out, 16-byte aligned.
 *   dfinal           : NULL (the final state is not part of L) or fp32 [N, H, V, K],
 *                      dL/d final_state, 16-byte aligned.
 * Outputs, all fp32 and fully overwritten:
 *   dq, dk, dg       : [B, T, H, K], 16-byte aligned.  dg is dL/dg for the raw g the
 *                      caller passed (through the gate unless KDA_GATE_PREACTIVATED).
 *   dv               : [B, T, H, V], 16-byte aligned.
 *   dbeta            : [B, T, H], dL/d beta logits (dL/d beta with KDA_BETA_PREACTIVATED).
 *   dh0              : NULL or [N, H, V, K], dL/d initial_state (defined with or without
 *                      an initial state: the gradient at a zero state).
 *   dA_log, ddt_bias : NULL or [H] and [H, K], summed over every token of every
 *                      sequence; zero with KDA_GATE_PREACTIVATED.
 *   workspace        : device scratch of at least kda_bwd_workspace_size bytes, 256-byte
 *                      aligned; it begins with the error word kda_check_device_error reads
 *                      (malformed cu_seqlens are clamped and flagged, as in kda_fwd).
 * Two forms compute it.  The gate with a lower bound takes the chunked one unless flags
 * has KDA_BWD_RECURRENT: two chains per (sequence, head) run side by side on tcgen05 (the
 * forward storing each 16-token chunk's entering state, and the state gradient carried from
 * the end to the start), then every chunk's gradients are computed independently; bf16
 * operands, gradients within 1e-2 relative Frobenius of the exact ones (dA_log within 1e-3
 * of the sum of its terms' magnitudes).  It stores about 106 KiB per 16 tokens and head.
 * The recurrent form (the other gates, or KDA_BWD_RECURRENT) runs the token recurrence in
 * fp32 and stores the state at every 8th token: (B T / 8 + N + 1) x H x 64 KiB.
 * kda_bwd_workspace_size covers both.  The result is deterministic (fixed-order sums, no
 * atomics on values).  Returns KDA_OK once the kernels are enqueued; argument errors as for
 * kda_fwd (K or V other than 128: KDA_ERR_UNSUPPORTED_SHAPE).
 */
KDA_API kda_status kda_bwd_workspace_size(const kda_shape *shape, size_t *bytes);
KDA_API kda_status kda_bwd(const kda_shape *shape, const void *q, const void *k, const void *v, const void *g,
                           const void *beta, float scale, const float *A_log, const float *dt_bias,
                           float lower_bound, const void *initial_state, kda_state_dtype init_dtype,
                           const int64_t *cu_seqlens, const void *dout, const float *dfinal, float *dq,
                           float *dk, float *dv, float *dg, float *dbeta, float *dh0, float *dA_log,
                           float *ddt_bias, unsigned flags, void *workspace, size_t workspace_bytes,
                           kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
