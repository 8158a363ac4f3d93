/*
 * linattn.h -- C ABI of the GB300 (sm_103a) kernelized linear attention library.
 *
 * The operation (page titles and sections of the sources it follows):
 *
 *   "[Feature] LinearAttention layer for Keras", Mathematical definition:
 *     non-causal  S = sum_j phi(K_j)^T V_j,  Z = sum_j phi(K_j),
 *                 Y_i = phi(Q_i) S / (phi(Q_i) Z + eps)
 *     causal      S_t = S_{t-1} + phi(K_t)^T V_t,  Z_t = Z_{t-1} + phi(K_t),
 *                 Y_t = phi(Q_t) S_t / (phi(Q_t) Z_t + eps)   (token t included)
 *     use_normalizer = 0:  Y = phi(Q) S.
 *   same page, Feature maps:  elu_plus_one  phi(x) = elu(x) + 1 (alpha 1);
 *                              relu          phi(x) = max(x, 0) + eps.
 *   same page, Streaming State: key_value_state S (B, H, Dk, Dv) and
 *     key_state Z (B, H, Dk), kept in the accumulator dtype (float32); chunked
 *     calls that carry the state equal one full-sequence call.
 *   same page, Masking: a (batch, sequence) validity mask.  Causal: an
 *     invalid step leaves S and Z unchanged and outputs zero.  Non-causal:
 *     invalid keys/values leave the sums and invalid queries output zero.
 *   ONNX-light "LinearAttention" operator: packed [B, T, H*D] activations,
 *     grouped KV heads (query head h reads kv head h / (Hq/Hkv)), update rules
 *       linear  S_t = S_{t-1} + k_t (x) v_t
 *       gated   S_t = exp(g_t) S_{t-1} + k_t (x) v_t   (g_t per kv head, log space)
 *               or, per key dimension, row i of S_t scaled by exp(g_t[i])
 *       delta        S_t = S_{t-1} + beta_t k_t (x) (v_t - S_{t-1}^T k_t)
 *       gated_delta  S_t = exp(g_t) S_{t-1} + beta_t k_t (x) (v_t - exp(g_t) S_{t-1}^T k_t)
 *     with o_t = scale * q_t^T S_t and scale 0.0 meaning 1/sqrt(d_k).
 *
 * Conventions shared by every entry point
 *  - All tensor arguments are DEVICE pointers to contiguous row-major memory
 *    owned by the caller.  The library never allocates or frees device
 *    memory; scratch comes from the caller's workspace.
 *  - Activations: q (B, T, Hq, Dk), k (B, T, Hkv, Dk), v (B, T, Hkv, Dv),
 *    y (B, T, Hq, Dv) -- the same bytes as the ONNX packed (B, T, H*D).
 *    decay (B, T, Hkv) in the io dtype, log space; with decay_per_key_dim
 *    (B, T, Hkv, Dk), the ONNX (B, T, H_kv*d_k) layout.
 *  - State: S (B, Hkv, Dk, Dv) float32, Z (B, Hkv, Dk) float32.  S[b,h,i,j]
 *    accumulates phi(k)_i * v_j.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and is asynchronous; the call returns after enqueueing.
 *  - On any status other than LA_OK nothing has been enqueued, except for
 *    LA_ERR_CUDA, which reports a failed launch (cudaGetLastError) and may
 *    follow partially enqueued work.  la_last_error() gives a one-line
 *    description of the last failure on the calling host thread.
 *  - Arithmetic: phi in float32; products on tensor cores (bf16 inputs) or
 *    CUDA cores (float32 inputs); S and Z accumulate in float32; y is
 *    rounded to out_dtype with round-to-nearest-even.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LINATTN_ABI_VERSION 3

typedef enum la_status {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* bad size, null pointer, bad enum, Hq % Hkv != 0 ... */
    LA_ERR_UNSUPPORTED = 2,  /* a valid combination the library does not implement */
    LA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than la_workspace_bytes() */
    LA_ERR_CUDA = 4,         /* a CUDA runtime error while enqueueing */
    LA_ERR_TIMEOUT = 5       /* la_device_status: a kernel gave up on a bounded wait */
} la_status;

typedef enum la_dtype { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

typedef enum la_feature_map {
    LA_FMAP_NONE = 0,          /* identity (ONNX rules) */
    LA_FMAP_ELU_PLUS_ONE = 1,  /* elu(x) + 1 */
    LA_FMAP_RELU_EPS = 2       /* max(x, 0) + epsilon */
} la_feature_map;

typedef enum la_update_rule {
    LA_RULE_LINEAR = 0,
    LA_RULE_GATED = 1,
    LA_RULE_DELTA = 2,       /* la_forward_causal_delta / la_decode_step_delta only */
    LA_RULE_GATED_DELTA = 3  /* idem */
} la_update_rule;

/* The CUDA stream type without the CUDA headers: identical to cudaStream_t. */
typedef struct CUstream_st* la_stream_t;

/* Problem description (the Keras constructor arguments and the ONNX
 * attributes).  Plain data; the library keeps no pointer to it. */
typedef struct la_params {
    int64_t batch;           /* B >= 1 */
    int64_t seq_len;         /* T >= 0; must be 1 for la_decode_step */
    int32_t q_heads;         /* Hq >= 1 */
    int32_t kv_heads;        /* Hkv >= 1, Hq % Hkv == 0 */
    int32_t key_dim;         /* Dk, 1..128 */
    int32_t value_dim;       /* Dv, 1..128 */
    int32_t io_dtype;        /* la_dtype of q, k, v and decay */
    int32_t out_dtype;       /* la_dtype of y */
    int32_t feature_map;     /* la_feature_map, applied to q and k */
    int32_t use_normalizer;  /* 1: divide by phi(q).Z + eps; 0: no Z at all */
    float epsilon;           /* normalization_epsilon >= 0 (also the relu offset) */
    float scale;             /* output scale; 0.0 means 1/sqrt(Dk) (ONNX default) */
    int32_t update_rule;     /* la_update_rule */
    int32_t decay_per_key_dim; /* 0: decay (B,T,Hkv); 1: decay (B,T,Hkv,Dk) (gated rules only).
                                * The tensor-core prefill takes the per-head form; the
                                * per-key-dimension form runs on CUDA cores (token by token). */
} la_params;

/* Zero-filled initial state, Keras get_initial_state / ONNX default
 * past_state ("Streaming State" section of the Keras request).
 * S: (B, Hkv, Dk, Dv) float32, required.  Z: (B, Hkv, Dk) float32, may be
 * NULL (use_normalizer = 0 needs no key_state).  Enqueued memsets. */
la_status la_get_initial_state(const la_params* p, float* S, float* Z, la_stream_t stream);

/* Bytes of device workspace a call needs (0 when none).  causal: 1 for
 * la_forward_causal, 0 for la_forward_noncausal.  The workspace must be at
 * least 256-byte aligned, must not be used by two calls that may run at the
 * same time, and needs no initialisation. */
size_t la_workspace_bytes(const la_params* p, int causal);

/* Causal prefill over T tokens (Keras request, Mathematical definition /
 * Causal; ONNX LinearAttention, prefill T > 1 and decode T = 1).
 *   q, k, v     activations (io_dtype), required when T > 0.
 *   decay       (B, T, Hkv) io_dtype, log space; required iff rule = GATED.
 *   S0, Z0      carried state in (initial_state / past_state); NULL = zeros.
 *               Z0 is ignored when use_normalizer = 0.
 *   y           output (B, T, Hq, Dv) out_dtype, required when T > 0.
 *   S_out,Z_out final state (return_state); NULL = not returned.  S_out may
 *               alias S0 and Z_out may alias Z0 (in-place streaming).
 *   ws          workspace of ws_bytes >= la_workspace_bytes(p, 1).
 * T = 0 copies S0/Z0 (or zeros) to S_out/Z_out.
 * LA_ERR_UNSUPPORTED: gated rule together with a feature map or the
 * normalizer (the pages define neither combination). */
la_status la_forward_causal(const la_params* p, const void* q, const void* k, const void* v,
                            const void* decay, const float* S0, const float* Z0, void* y,
                            float* S_out, float* Z_out, void* ws, size_t ws_bytes,
                            la_stream_t stream);

/* la_forward_causal with a sequence-validity mask (Keras request, Masking):
 *   mask  (B, T) uint8 DEVICE array, nonzero = valid step, row-major; NULL
 *         means every step is valid (the call is then la_forward_causal).
 * An invalid step t of sequence b leaves that sequence's S and Z exactly as
 * they were -- no update and, for the gated rule, no decay -- and its
 * outputs y[b, t, :, :] are zero; later valid steps read the state as the
 * earlier valid steps left it.  Padding (left, right) and interior gaps are
 * all allowed.  Arguments, errors and numerics otherwise as
 * la_forward_causal; masked-out q, k, v values are never used. */
la_status la_forward_causal_masked(const la_params* p, const void* q, const void* k, const void* v,
                                   const void* decay, const uint8_t* mask, const float* S0, const float* Z0,
                                   void* y, float* S_out, float* Z_out, void* ws, size_t ws_bytes,
                                   la_stream_t stream);

/* Size of the scratch built into the library for la_forward_causal_noalloc:
 * 16 MiB of device memory, reserved once per device when the library's
 * device code is loaded there. */
#define LA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* la_forward_causal without a caller workspace.  The methods on the pages
 * have no counterpart to this call: it exists for callers that cannot hand
 * the library device memory -- for example a plug-in inside a host program
 * that owns every device allocation and offers no scratch, or a
 * latency-critical loop that must not call cudaMalloc (which can synchronize
 * the device) or an allocator between steps.
 *
 * Arguments, results and numerics are those of la_forward_causal; the
 * scratch that call would take from `ws` comes from one buffer of
 * LA_NOALLOC_SCRATCH_BYTES compiled into the library (one per device).
 *  - No device memory is allocated or freed by this call, and it calls no
 *    library routine that allocates.
 *  - The first call on a device, made with that device current, looks up the
 *    buffer's address (cudaGetSymbolAddress) and configures the kernels;
 *    make that first call before any stream capture starts on the device.
 *  - Nothing in the buffer has to start at zero: every byte a call reads
 *    was written earlier in the same call.
 *  - The buffer is shared by all calls on one device: two calls that may run
 *    at the same time (different streams, or different host threads without
 *    ordering between them) race on it and give wrong results.  Calls issued
 *    one after another on one stream are safe.
 *  - LA_ERR_WORKSPACE when the problem needs more scratch than
 *    LA_NOALLOC_SCRATCH_BYTES (la_workspace_bytes(p, 1) tells how much);
 *    use la_forward_causal with a caller workspace for those.  On a GPU with
 *    at most 152 SMs every causal problem fits. */
la_status la_forward_causal_noalloc(const la_params* p, const void* q, const void* k, const void* v,
                                    const void* decay, const float* S0, const float* Z0, void* y,
                                    float* S_out, float* Z_out, la_stream_t stream);

/* Non-causal attention with the global state (Keras request, Mathematical
 * definition / Non-causal).  No state in or out ("Non-causal attention does
 * not expose streaming state").  Only the linear rule. */
la_status la_forward_noncausal(const la_params* p, const void* q, const void* k, const void* v,
                               void* y, void* ws, size_t ws_bytes, la_stream_t stream);

/* la_forward_noncausal with a sequence-validity mask (Keras request,
 * Masking, non-causal): mask (B, T) uint8 device array as for
 * la_forward_causal_masked (NULL = all valid).  Invalid positions add
 * nothing to the global S and Z, and their outputs are zero. */
la_status la_forward_noncausal_masked(const la_params* p, const void* q, const void* k, const void* v,
                                      const uint8_t* mask, void* y, void* ws, size_t ws_bytes,
                                      la_stream_t stream);

/* One streaming token per sequence (seq_len must be 1): the recurrent update
 * and read-out ("Causal Linear Attention": S_i = S_{i-1} + phi(k_i) v_i^T,
 * then the read-out with S_i; ONNX LinearAttention decode, T = 1).
 *   q (B,1,Hq,Dk), k (B,1,Hkv,Dk), v (B,1,Hkv,Dv), decay (B,1,Hkv) or NULL.
 *   S (B,Hkv,Dk,Dv) and Z (B,Hkv,Dk) float32 are read and updated IN PLACE;
 *   Z may be NULL when use_normalizer = 0.  y (B,1,Hq,Dv) out_dtype. */
la_status la_decode_step(const la_params* p, const void* q, const void* k, const void* v,
                         const void* decay, float* S, float* Z, void* y, la_stream_t stream);

/* la_decode_step with a validity mask (Keras request, Masking): mask (B,)
 * uint8 device array, one entry per sequence (the (B, T) mask at T = 1);
 * NULL = all valid.  A sequence whose step is invalid keeps S and Z
 * bit-for-bit and gets zero outputs. */
la_status la_decode_step_masked(const la_params* p, const void* q, const void* k, const void* v,
                                const void* decay, const uint8_t* mask, float* S, float* Z, void* y,
                                la_stream_t stream);

/* The delta rules of the ONNX-light "LinearAttention" operator (update_rule
 * "delta" or "gated_delta", its default), causal prefill or chunk of a
 * stream:
 *   delta        S_t = S_{t-1} + beta_t k_t (x) (v_t - S_{t-1}^T k_t)
 *   gated_delta  S_t = exp(g_t) S_{t-1} + beta_t k_t (x) (v_t - exp(g_t) S_{t-1}^T k_t)
 *   o_t = scale * q_t^T S_t
 * p->update_rule is LA_RULE_DELTA or LA_RULE_GATED_DELTA; no feature map and
 * no normalizer (LA_ERR_UNSUPPORTED otherwise: the page defines neither).
 *   decay      (B, T, Hkv) or, with decay_per_key_dim, (B, T, Hkv, Dk) in the
 *              io dtype, log space; required for gated_delta, ignored for delta.
 *   beta       update rate in the io dtype, required: (B, T, Hkv) when
 *              beta_per_head = 1, (B, T, 1) when 0.
 *   mask       (B, T) uint8 validity or NULL (as la_forward_causal_masked).
 *   S0, S_out  as la_forward_causal (Z is not used by these rules).
 * This entry point runs every (batch, kv head) stream as one token-by-token
 * recurrence on CUDA cores and needs no workspace; la_forward_causal_delta_ws
 * is the chunk-parallel tensor-core form. */
la_status la_forward_causal_delta(const la_params* p, const void* q, const void* k, const void* v,
                                  const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                                  const float* S0, void* y, float* S_out, la_stream_t stream);

/* The delta rules in chunk-parallel form on the tensor cores (the operator
 * page's "chunk-parallel WY decomposition during prefill"): arguments,
 * results and errors as la_forward_causal_delta, plus a workspace.  Per
 * chunk of 64 steps the rule is solved in closed form -- a unit
 * lower-triangular system gives the chunk's updates U = U' - W S0, its
 * outputs and its state transition S <- M S + N -- and a scan carries the
 * state from chunk to chunk.  Covers bf16 io with key_dim = value_dim = 128
 * and one decay per kv head (la_delta_workspace_bytes > 0); other shapes run
 * the token-by-token recurrence of la_forward_causal_delta and need no
 * workspace.
 *   ws   workspace of ws_bytes >= la_delta_workspace_bytes(p): about
 *        263 KB per (batch, kv head, 64-step chunk), 256-byte aligned, not
 *        shared with a call that may run at the same time.
 * S_out may alias S0. */
size_t la_delta_workspace_bytes(const la_params* p);
la_status la_forward_causal_delta_ws(const la_params* p, const void* q, const void* k, const void* v,
                                     const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                                     const float* S0, void* y, float* S_out, void* ws, size_t ws_bytes,
                                     la_stream_t stream);

/* One token per sequence with a delta rule (seq_len must be 1): S is read
 * and updated in place; beta (B, 1, Hkv) or (B, 1, 1); mask (B,) or NULL. */
la_status la_decode_step_delta(const la_params* p, const void* q, const void* k, const void* v,
                               const void* decay, const void* beta, int beta_per_head, const uint8_t* mask,
                               float* S, void* y, la_stream_t stream);

/* Gradients of la_forward_causal for the linear rule (the backward pass the
 * Keras request's Test Plan asks to check numerically; no mask, no decay).
 *   q, k, v, S0, Z0  the forward call's inputs (S0/Z0 may be NULL = zeros).
 *   dy               gradient of the output y, (B, T, Hq, Dv) in the io dtype.
 *   dq, dk, dv       outputs in out_dtype, the shapes of q, k, v.
 *   dS0, dZ0         gradients of the initial state (float32), or NULL.
 *   ws               workspace of la_backward_workspace_bytes(p) bytes.
 * bf16 inputs with key_dim == value_dim in {64, 128} and 16-byte aligned
 * pointers run the chunk-parallel form on the tensor cores (five launches:
 * per-chunk key/value products, a forward scan of the chunk start states, a
 * per-chunk kernel for dq and the chunk's reverse-state increment, a reverse
 * scan, a per-chunk kernel for dk and dv); other shapes and float32 inputs
 * run two CUDA-core token scans.  LA_ERR_UNSUPPORTED for the other rules. */
size_t la_backward_workspace_bytes(const la_params* p);
la_status la_backward_causal(const la_params* p, const void* q, const void* k, const void* v, const float* S0,
                             const float* Z0, const void* dy, void* dq, void* dk, void* dv, float* dS0, float* dZ0,
                             void* ws, size_t ws_bytes, la_stream_t stream);

/* Static string for a status code.  la_status_str is the same function
 * under its short name. */
const char* la_status_string(la_status s);
const char* la_status_str(la_status s);

/* One-line description of the last failure on this host thread ("" if none). */
const char* la_last_error(void);

/* LINATTN_ABI_VERSION of the loaded library. */
int la_abi_version(void);

/* Error word of the tensor-core kernels on the current device: 0 when no
 * kernel gave up on a bounded wait (each pipeline wait ends with an error
 * bit instead of hanging); a nonzero value names the wait sites that timed
 * out.  Synchronous (device-to-host copy).  reset != 0 clears it. */
unsigned la_device_error(int reset);

/* The same check as a status: synchronises the current device, then
 * LA_ERR_TIMEOUT when the error word is nonzero (la_last_error names the
 * word), LA_ERR_CUDA when the device reports an error, else LA_OK.
 * reset != 0 clears the word. */
la_status la_device_status(int reset);

/* Bits of the device error word set by la_check_bounded_wait. */
#define LA_SELFTEST_WARP_WAIT (1u << 30)
#define LA_SELFTEST_THREAD_WAIT (1u << 31)

/* Failure-path check of the bounded waits (no counterpart on the pages: it
 * tests the library's own failure detection).  Enqueues one small kernel
 * whose two waits -- the warp-uniform form and the single-thread form that
 * every pipeline wait of the tensor-core kernels uses -- poll an mbarrier
 * that nothing ever completes, give up after limit_us microseconds (1 ..
 * 1000000), set LA_SELFTEST_WARP_WAIT and LA_SELFTEST_THREAD_WAIT in the
 * device error word (read and clear it with la_device_error) and return.
 * The kernel holds no tensor memory and has no copy in flight, so the
 * context stays usable.  LA_ERR_INVALID_ARG for a limit out of range. */
la_status la_check_bounded_wait(uint32_t limit_us, la_stream_t stream);

/* Number of CUDA kernels this library has enqueued in this process so far
 * (memsets and copies are not counted).  For accounting in benchmarks. */
uint64_t la_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
