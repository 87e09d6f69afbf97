/*
 * gdn.h -- C ABI of the gated delta-rule (GDN) linear-attention library for one
 * NVIDIA GB300 (sm_103a).
 *
 * The library computes, per (batch, value head), the recurrence over a state S laid
 * out [Dk, Dv] in fp32:
 *     S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 * with value head h reading key/query head h / (Hv / Hk).
 *
 * Sources (AWS Neuron NKI library API pages):
 *   "GDN CTE Kernel API Reference"  -- the chunked prefill (gdn_prefill).
 *   "GDN TKG Kernel API Reference"  -- the fused single-token decode step
 *                                      (gdn_decode_step; gdn_decode_multi runs T
 *                                      of them with the state kept on chip).
 *   "GDN Block TKG Kernel API Reference" -- the conv1d decode token in front of the
 *                                      decode step (gdn_conv1d_decode).
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers; the caller owns all memory.
 *     The library allocates nothing and frees nothing.
 *   - Tensors are dense, row-major, with the listed shapes. Every pointer must be
 *     non-NULL and 16-byte aligned unless stated otherwise.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream). A GDN_OK return means the work was validated and enqueued.
 *   - Errors are returned, never thrown. On a non-GDN_OK status nothing was enqueued
 *     and gdn_last_error() returns a message for the calling thread.
 *   - Outputs must not overlap inputs, except where aliasing is stated.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_EINVAL = 1,        /* invalid argument: shape, pointer or alignment           */
    GDN_EUNSUPPORTED = 2,  /* valid per the pages but not built here                  */
    GDN_ECUDA = 3,         /* a CUDA runtime/driver call or kernel launch failed       */
    GDN_ETIMEOUT = 4       /* a kernel gave up a bounded wait (gdn_get_device_status) */
} gdn_status;

typedef enum gdn_dtype {
    GDN_DTYPE_F32 = 0,
    GDN_DTYPE_BF16 = 1
} gdn_dtype;

/* Intra-chunk inverse methods of gdn_unit_lower_inverse. */
typedef enum gdn_tril_algorithm {
    GDN_TRIL_SUBSTITUTION = 0, /* forward substitution, fp32                          */
    GDN_TRIL_NEUMANN = 1       /* (I+X)(I+X^2)...(I+X^32), X = -A, tf32 tensor cores  */
} gdn_tril_algorithm;

/* Largest head dimension: "GDN CTE Kernel API Reference", Notes (Dk, Dv <= 128). */
#define GDN_MAX_HEAD_DIM 128

/*
 * gdn_prefill_workspace_bytes -- scratch (device memory) gdn_prefill needs for this
 * shape. Returns 0 when no workspace is needed, or (size_t)-1 if the shape is invalid.
 * The bf16 path with Dk = Dv = 128 (the tensor-core kernels) needs 49680 bytes per
 * (batch, value head, 64-token chunk): B * Hv * ceil(S / 64) * 49680; every other
 * shape needs none.
 */
size_t gdn_prefill_workspace_bytes(int B, int Hk, int Hv, int S, int Dk, int Dv,
                                   gdn_dtype dtype);

/*
 * gdn_prefill -- chunked GDN prefill ("GDN CTE Kernel API Reference": description,
 * parameters, returns and Notes).
 *
 *   q, k       device, [B, Hk, S, Dk], token-major, dtype `dtype` (which sets the
 *              compute dtype of the products and of `out`). Rows must be
 *              L2-normalised (precondition, not checked).
 *   v          device, [B, Hv, S, Dv], dtype `dtype`.
 *   g_log      device, [B, Hv, S] fp32, per-token log decay (<= 0, not checked).
 *   beta       device, [B, Hv, S] fp32, update strength in (0, 1) (not checked).
 *   scale      query scale, applied on the device (typically 1/sqrt(Dk)).
 *   B, Hk, Hv, S, Dk, Dv
 *              B >= 1, Hk >= 1, Hv % Hk == 0, S >= 0, 1 <= Dk, Dv <= 128.
 *              S needs no particular multiple: a ragged last chunk is handled.
 *   state      device, [B, Hv, Dk, Dv] fp32. If state_is_input != 0 its contents are
 *              the initial state and it is overwritten IN PLACE with the final state;
 *              if 0 the initial state is zero, nothing is read from it, and the final
 *              state is written to it.
 *   out        device, [B, Hv, S, Dv], dtype `dtype`, head-major, un-normalised.
 *   workspace  device scratch of gdn_prefill_workspace_bytes(...) bytes, 16-byte
 *              aligned (may be NULL when that is 0), owned by the caller and in use
 *              until the enqueued work completes. Its contents on entry do not matter
 *              and are unspecified on exit.
 *   stream     cudaStream_t to enqueue on.
 *
 * Errors: GDN_EINVAL for a bad shape, a NULL or misaligned pointer, or too little
 * workspace; GDN_ECUDA if a launch fails.
 */
gdn_status gdn_prefill(const void* q, const void* k, const void* v,
                       const float* g_log, const float* beta, float scale,
                       gdn_dtype dtype, int B, int Hk, int Hv, int S, int Dk, int Dv,
                       float* state, int state_is_input, void* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_prefill_varlen_workspace_bytes -- device scratch gdn_prefill_varlen needs for N
 * sequences packed into T tokens: on the bf16 Dk = Dv = 128 path (tensor cores)
 * Hv * (ceil(T / 64) + N) * 49680 bytes rounded up to 256, plus 4 * (N + 2); on every
 * other path 4 * (N + 2) rounded up to 16. (size_t)-1 for an invalid shape.
 */
size_t gdn_prefill_varlen_workspace_bytes(int N, int Hk, int Hv, int T, int Dk, int Dv,
                                          gdn_dtype dtype);

/*
 * gdn_prefill_varlen -- gdn_prefill over a variable-length batch: N independent
 * sequences packed back to back along the token axis, sequence n holding tokens
 * cu_seqlens[n] .. cu_seqlens[n+1] - 1 (the "GDN CTE Kernel API Reference" recurrence
 * per sequence, each from its own state; the pages' kernel takes a dense batch with
 * S % 64 == 0 -- per-sequence offsets are this library's extension).
 *
 *   q, k         device, [Hk, T, Dk] in the compute dtype (one batch row, tokens packed).
 *   v            device, [Hv, T, Dv].
 *   g_log, beta  device, [Hv, T] fp32.
 *   cu_seqlens   device, [N + 1] int32: 0 = cu[0] <= cu[1] <= ... <= cu[N] <= T.
 *                Sequences may be empty; tokens past cu[N] are ignored.
 *   state        device, [N, Hv, Dk, Dv] fp32, one state per sequence, with
 *                state_is_input as in gdn_prefill (an empty sequence leaves its state
 *                unchanged, or writes zeros when state_is_input == 0).
 *   out          device, [Hv, T, Dv]; rows of tokens past cu[N] are not written.
 *   workspace    device scratch of gdn_prefill_varlen_workspace_bytes(...) bytes.
 *   0 <= N <= 65535; N == 0 enqueues nothing.
 *
 * Each sequence's chunks start at its first token, so sequence n gets bit for bit what
 * gdn_prefill returns for it alone (B = 1, S = its length). A malformed cu_seqlens is
 * found on the device: every sequence is then treated as empty and
 * gdn_get_device_status() returns GDN_EINVAL.
 *
 * Errors: as gdn_prefill, plus GDN_EINVAL for N out of range.
 */
gdn_status gdn_prefill_varlen(const void* q, const void* k, const void* v, const float* g_log,
                              const float* beta, float scale, gdn_dtype dtype,
                              const int* cu_seqlens, int N, int Hk, int Hv, int T, int Dk,
                              int Dv, float* state, int state_is_input, void* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * gdn_prefill_noalloc -- gdn_prefill for callers that cannot hand the library device memory:
 * a plug-in inside a host runtime that owns the device memory and gives the plug-in no
 * allocator, or a latency-critical loop in which an allocation (cudaMalloc can synchronise
 * the device) is not allowed. The call takes no workspace and allocates nothing: its scratch
 * is a fixed 128 MiB array in the library's own device memory, which every GPU that loads
 * the library holds until the process exits. (The pages have no counterpart of this call.)
 *
 * Arguments, results and errors as gdn_prefill (the caller still passes inputs, state and
 * out). On the tensor-core path (bf16, Dk = Dv = 128) the sequence is processed in segments
 * of whole 64-token chunks that fit the scratch -- 128 MiB / 49680 bytes per (batch, value
 * head, chunk) unit = 2701 units -- the state carrying over in fp32 from one segment to the
 * next, so the result equals gdn_prefill's. GDN_EUNSUPPORTED, with a message, when B * Hv
 * exceeds 2701 (not even one chunk per head fits). Every other path needs no scratch and
 * runs as gdn_prefill.
 *
 * The first call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture begins. Every call shares the one
 * array, whose contents the next call overwrites before reading: calls that overlap on the
 * GPU (other streams, other threads) race on it, so issue them on one stream or synchronise
 * between them.
 */
gdn_status gdn_prefill_noalloc(const void* q, const void* k, const void* v,
                               const float* g_log, const float* beta, float scale,
                               gdn_dtype dtype, int B, int Hk, int Hv, int S, int Dk,
                               int Dv, float* state, int state_is_input, void* out,
                               void* stream);

/*
 * gdn_decode_step -- one fused decode token ("GDN TKG Kernel API Reference":
 * Background, parameters, returns, Notes and Dimensions).
 *
 *   q, k         device, [BH, K] bf16, RAW (not l2-normalised), already expanded to
 *                the value heads; BH = batch * num_v_heads with heads cycling fastest
 *                (bh = b * num_v_heads + h).
 *   v, z         device, [BH, V] bf16 (z is the RMSNormGated gate input).
 *   b, a         device, [BH] bf16: raw pre-sigmoid beta input and raw gate input.
 *   A_log        device, [num_v_heads] fp32.
 *   dt_bias      device, [num_v_heads] fp32.
 *   norm_weight  device, [V] fp32 (RMSNormGated gamma).
 *   state_in     device, [BH, K, V] fp32, incoming state.
 *   state_out    device, [BH, K, V] fp32, updated state. May equal state_in (in place);
 *                must not otherwise overlap it.
 *   out          device, [BH, V] bf16, the RMSNormGated output.
 *   1 <= K, V <= 128; BH % num_v_heads == 0. BH == 0 enqueues nothing.
 *
 * The step computes, per row: q^ = q/sqrt(|q|^2 + 1e-6), k^ likewise;
 * beta = sigmoid(b); g = -exp(A_log[h]) * softplus(a + dt_bias[h]); alpha = exp(g);
 * S' = alpha (I - beta k^ k^^T) S + beta k^ v^T; o = S'^T q^ / sqrt(K);
 * out = bf16( o / sqrt(mean_V(o^2) + 1e-6) * norm_weight * z * sigmoid(z) ).
 * exp(g) and the 1/sqrt(K) scale are applied inside (Notes). The two eps values and
 * the norm-then-gate order are readings: the pages do not state them.
 *
 * Errors: GDN_EINVAL for a bad shape or a NULL/misaligned pointer; GDN_ECUDA if the
 * launch fails.
 */
gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const void* b,
                           const void* a, const float* A_log, const float* dt_bias,
                           const void* z, const float* norm_weight, const float* state_in,
                           float* state_out, void* out, int BH, int num_v_heads, int K,
                           int V, void* stream);

/*
 * gdn_decode_multi -- T consecutive fused decode tokens of the same BH rows in one call:
 * token t applies the gdn_decode_step formulas to the state left by token t-1.
 * Not on the pages (an extension of the "GDN TKG Kernel API Reference" step): the state
 * is read once and written once, so its HBM traffic is shared by the T tokens.
 * For T >= 2 the tokens run in the equivalent chunk form (blocks of eight), so results
 * agree with T single steps up to rounding, not bit for bit. The state products use
 * two-term tf32 splits, within 2^-21 of fp32; the solve and the state update are fp32.
 * T == 1 is gdn_decode_step bit for bit.
 *
 *   q, k         device, [T, BH, K] bf16 raw (token-major: token t's rows at t * BH).
 *   v, z         device, [T, BH, V] bf16.
 *   b, a         device, [T, BH] bf16.
 *   out          device, [T, BH, V] bf16.
 *   A_log, dt_bias, norm_weight, state_in, state_out: as gdn_decode_step (state_out may
 *                equal state_in). T == 1 is gdn_decode_step; T == 0 or BH == 0 enqueues
 *                nothing.
 *
 * Errors: as gdn_decode_step, plus GDN_EINVAL for T < 0.
 */
gdn_status gdn_decode_multi(const void* q, const void* k, const void* v, const void* b,
                            const void* a, const float* A_log, const float* dt_bias,
                            const void* z, const float* norm_weight, const float* state_in,
                            float* state_out, void* out, int T, int BH, int num_v_heads, int K,
                            int V, void* stream);

/*
 * gdn_unit_lower_inverse -- T = (I + A)^-1 for n strictly lower-triangular C x C fp32
 * matrices, the chunked prefill's intra-chunk inverse, by the method `algorithm` selects
 * ("GDN CTE Kernel API Reference", :param algorithm: -- the pages offer a selectable
 * inverse, "neumann" among them; this call exposes the choice on its own so the two
 * methods can be compared):
 *   GDN_TRIL_SUBSTITUTION  forward substitution in fp32 (rounding only);
 *   GDN_TRIL_NEUMANN       sum_{n<C} X^n with X = -A (nilpotent), as the product
 *                          (I + X)(I + X^2)...(I + X^(C/2)): log2(C) rounds of tf32
 *                          tensor-core products (relative error ~1e-3 for |A| <= 1).
 *
 *   A  device, [n, C, C] fp32, row-major; entries on and above the diagonal are read
 *      as zero by neither method's definition, so they must BE zero.
 *   T  device, [n, C, C] fp32, unit lower triangular. May equal A (in place); must not
 *      otherwise overlap it.
 *   C == 64 (GDN_EUNSUPPORTED otherwise); n == 0 enqueues nothing.
 *
 * Errors: GDN_EINVAL for n < 0, an unknown algorithm, a NULL/misaligned pointer or a
 * partial overlap; GDN_ECUDA if the launch fails.
 */
gdn_status gdn_unit_lower_inverse(const float* A, float* T, int n, int C, int algorithm,
                                  void* stream);

/*
 * gdn_conv1d_decode -- the step in front of the decode step: one token of the q|k|v
 * in_proj output through the depthwise causal convolution with its sliding window,
 * SiLU, then the split into q | k | v with q and k repeated over the value heads
 * ("GDN Block TKG Kernel API Reference": gdn_conv1d_decode -- conv + silu + slide-window
 * state -- and "split conv_out + GQA-repeat q,k"; shapes from its parameters and
 * Dimensions).
 *
 *   x              device, [B, conv_dim] bf16, conv_dim = 2 key_dim + value_dim with
 *                  key_dim = num_k_heads * head_k_dim, value_dim = num_v_heads * head_v_dim
 *                  (channels q | k | v, head-major within each).
 *   conv_weight    device, [conv_dim, K_win] fp32 depthwise taps, oldest tap first.
 *   conv_state_in  device, [B, conv_dim, K_win] bf16, the K_win latest inputs, oldest first.
 *   conv_state_out device, [B, conv_dim, K_win] bf16, the window after this token. May
 *                  equal conv_state_in (in place); must not otherwise overlap it.
 *   q_out, k_out   device, [B * num_v_heads, head_k_dim] bf16 (row b * num_v_heads + h
 *                  holds key head h / (num_v_heads / num_k_heads)): raw, not normalised --
 *                  the form gdn_decode_step takes.
 *   v_out          device, [B * num_v_heads, head_v_dim] bf16.
 *   1 <= head_k_dim, head_v_dim <= 128; 1 <= K_win <= 16; B == 0 enqueues nothing.
 *
 * Per batch and channel: window' = (state[1..K_win-1], x); y = silu(sum_w weight[w]
 * window'[w]) in fp32, rounded to bf16; state' = window'. The page gives the operation
 * and shapes only: the window order and the absence of a bias are readings.
 *
 * Errors: GDN_EINVAL for a bad shape, a NULL/misaligned pointer or a partial overlap of
 * the windows; GDN_ECUDA if the launch fails.
 */
gdn_status gdn_conv1d_decode(const void* x, const float* conv_weight, const void* conv_state_in,
                             void* conv_state_out, void* q_out, void* k_out, void* v_out, int B,
                             int num_k_heads, int num_v_heads, int head_k_dim, int head_v_dim,
                             int K_win, void* stream);

/* Message describing the calling thread's last non-GDN_OK status ("" if none). The
 * pointer stays valid until the thread's next call into the library. */
const char* gdn_last_error(void);

/*
 * gdn_get_device_status -- synchronises `stream`, then reports and clears the
 * device-side status word the kernels set when a bounded wait runs out.
 * Returns GDN_OK, GDN_ETIMEOUT, or GDN_ECUDA if the synchronisation itself failed.
 */
gdn_status gdn_get_device_status(void* stream);

/*
 * gdn_launch_count -- number of CUDA kernels this library has enqueued in this
 * process since it was loaded (diagnostics: lets a caller count the kernels of a
 * timed region). Thread-safe.
 */
unsigned long long gdn_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
