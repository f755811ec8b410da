/*
 * gsdpa.h -- C ABI of the GB300 gated softmax attention library (libgsdpa.so).
 *
 * The operation: for each batch b, query head h and query row i,
 *
 *     O[b,i,h,:] = softmax_j( Q[b,i,h,:] . K[b,j,kv(h),:] / sqrt(d_k)  + causal mask )
 *                  @ V[b,:,kv(h),:]
 *                  (.) sigmoid( X[b,i,:] W_g[:, cols(h)] )
 *
 * Sources (page title and section):
 *   - SDPA, rows non-negative and summing to one:
 *       "GatedAttention [2025]", sec. 1.2.1 (the Attention(Q,K,V) equation).
 *   - The gate Y' = Y (.) sigma(X W_theta), X the hidden state after
 *     pre-normalisation, sigma the logistic sigmoid, multiplicative and
 *     head-specific by default:
 *       "GatedAttention [2025]", sec. 1.2.2.
 *   - Position G1 (on the SDPA output of each head, before the heads are
 *     concatenated), elementwise gate (n x q x d_k) and headwise gate (n x q):
 *       "GatedAttention [2025]", sec. 1.2.2 and 1.3.2; "10 . 门控", sec. 3.2
 *       (position table, Table 1 excerpt rows 5 and 10, and the G1 module with
 *       no bias and head-major gate columns).
 *   - Grouped-query K/V heads: "GatedAttention [2025]", sec. 1.3.1.
 *   - Causal sums over j <= i: "GatedAttention [2025]", sec. 1.4.1.
 *   - First-token attention share: "10 . 门控", sec. 3.4; "GatedAttention
 *     [2025]", sec. 1.4.3 (the F-Attn column).
 *
 * Readings where the pages are silent (the library's choices):
 *   - kv(h) = h / (H_q / H_kv): query heads form contiguous groups.
 *   - When L_q < L_k the causal mask is aligned bottom-right: query i sits at
 *     absolute position L_k - L_q + i and sees keys 0 .. L_k - L_q + i. A single
 *     decode query therefore sees the whole cache (the current token included).
 *   - The gate has no bias. cols(h) = h*d_k .. h*d_k + d_k - 1 (elementwise)
 *     or the single column h (headwise).
 *   - The first-token share is measured on the ungated attention weights and
 *     averaged over query rows: sink[b,h] = mean_i p(i -> key 0).
 *
 * Layouts (all row-major, contiguous, no padding):
 *   X    [B, L_q, d_model]
 *   Q    [B, L_q, H_q,  d_k]
 *   K, V [B, L_k, H_kv, d_k]
 *   W_g  [d_model, H_q*d_k] (elementwise) or [d_model, H_q] (headwise)
 *   O    [B, L_q, H_q,  d_k]  == the concatenated [B, L_q, H_q*d_k]
 *   sink [B, H_q] float32
 * The element type of X, Q, K, V, W_g and O is float32 (GSDPA_F32) or
 * bfloat16 (GSDPA_BF16); sink is always float32.
 *
 * Ownership: the caller owns every buffer (inputs, outputs, workspace) and
 * the stream. All pointers passed to gated_sdpa_fwd are DEVICE pointers of
 * the current device. The library never allocates device memory and never
 * synchronises inside gated_sdpa_fwd: the call enqueues kernels (and small
 * memset nodes on the workspace) on `stream` and returns.
 *
 * Errors: every function returns a gsdpa_status. Argument errors are detected
 * on the host before anything is enqueued. Kernels never wait without a limit:
 * a wait that runs out records a device error word and the kernel returns;
 * gsdpa_check_device_error() reads that word.
 */
#ifndef GSDPA_H_
#define GSDPA_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GSDPA_API __attribute__((visibility("default")))
#else
#define GSDPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GSDPA_GATE_NONE = 0,         /* plain SDPA, W_g and X may be NULL */
    GSDPA_GATE_HEADWISE = 1,     /* one sigmoid per (token, head)     */
    GSDPA_GATE_ELEMENTWISE = 2,  /* one sigmoid per (token, head, c)  */
    /* gated_sdpa_fwd_variant only: */
    GSDPA_GATE_HEADWISE_SHARED = 3,     /* W_g [d_model, 1]: one gate per token, every head */
    GSDPA_GATE_ELEMENTWISE_SHARED = 4,  /* W_g [d_model, d_k]: one gate per (token, c), every head */
    GSDPA_GATE_STATIC = 5,              /* W_g holds theta [H_q, d_k]: the gate does not read X */
    GSDPA_GATE_HEADWISE_AVERAGED = 6,   /* W_g [d_model, H_q]: the H_q heads' gate values averaged,
                                           one gate per token for every head */
    GSDPA_GATE_ELEMENTWISE_AVERAGED = 7 /* W_g [d_model, H_q d_k]: the heads' gate values averaged
                                           over the heads, one gate per (token, c) for every head */
} gsdpa_gate_mode;

/* How the gate's logit gl acts on the SDPA output y (gated_sdpa_fwd_variant). */
typedef enum {
    GSDPA_FN_SIGMOID_MUL = 0,    /* y * sigma(gl)               (gated_sdpa_fwd's gate) */
    GSDPA_FN_NS_SIGMOID_MUL = 1, /* y * (0.5 + 0.5 sigma(gl))                          */
    GSDPA_FN_SIGMOID_ADD = 2,    /* y + sigma(gl)                                      */
    GSDPA_FN_SILU_ADD = 3,       /* y + gl sigma(gl)                                   */
    GSDPA_FN_IDENTITY_ADD = 4,   /* y + gl                                             */
    GSDPA_FN_SILU_SELF = 5,      /* y * sigma(y), no gate (gate_mode NONE)             */
    GSDPA_FN_RMSNORM = 6         /* per head: y / sqrt(mean_c y^2 + eps) * gamma[h, c],
                                    no gate (gate_mode NONE); W_g holds gamma [H_q, d_k]
                                    or is NULL for gamma = 1                            */
} gsdpa_gate_fn;

typedef enum {
    GSDPA_F32 = 0,               /* float32 in/out, float32 arithmetic (SIMT) */
    GSDPA_BF16 = 1               /* bfloat16 in/out, fp32 accumulation (tcgen05) */
} gsdpa_dtype;

typedef enum {
    GSDPA_OK = 0,
    GSDPA_ERR_INVALID_ARG = -1,      /* a size, mode or pointer is invalid      */
    GSDPA_ERR_UNSUPPORTED = -2,      /* valid, but not built (d_k, device, ...) */
    GSDPA_ERR_ALIGNMENT = -3,        /* a pointer is not 16-byte aligned        */
    GSDPA_ERR_WORKSPACE = -4,        /* workspace NULL or smaller than needed   */
    GSDPA_ERR_LAUNCH = -5,           /* the CUDA runtime refused a launch       */
    GSDPA_ERR_DEVICE_TIMEOUT = -6    /* a kernel wait ran out (see below)       */
} gsdpa_status;

/*
 * Bytes of device workspace gated_sdpa_fwd needs for this problem, or 0 if
 * none. Same arguments as gated_sdpa_fwd (want_sink != 0 when a sink pointer
 * will be passed). Returns (size_t)-1 for arguments gated_sdpa_fwd would
 * reject. Host-only; touches no device.
 */
GSDPA_API size_t gsdpa_workspace_bytes(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                             int gate_mode, int want_sink, int dtype);

/*
 * The gated attention forward (prefill when L_q > 1, decode when L_q == 1).
 *
 *   X, Q, K, V, W_g : device inputs in the layouts above. X and W_g may be
 *                     NULL when gate_mode == GSDPA_GATE_NONE.
 *   O               : device output [B, L_q, H_q, d_k], same dtype as inputs.
 *   sink            : device float32 [B, H_q] or NULL (not computed). With
 *                     bf16 prefill the rows' shares are added in fixed point
 *                     with 43 - ceil(log2(L_q + 1)) fraction bits, so the sum
 *                     does not depend on the order of the additions and
 *                     repeated calls give the same bits; there L_q <= 2^24
 *                     (GSDPA_ERR_UNSUPPORTED otherwise).
 *   B, L_q, L_k     : batch, query rows, key rows; 1 <= L_q <= L_k. B, L_q == 0
 *                     is an empty problem: nothing is enqueued, GSDPA_OK.
 *   d_model         : width of X (>= 1 when a gate is used; for bf16 a
 *                     multiple of 8, since every row must start on 16 bytes).
 *   H_q, H_kv       : query and K/V heads, H_q % H_kv == 0 (bf16 headwise
 *                     gate: H_q a multiple of 8, for the same reason).
 *   d_k             : head dimension, 64 or 128.
 *   gate_mode       : gsdpa_gate_mode.
 *   causal          : nonzero for the bottom-right causal mask.
 *   dtype           : gsdpa_dtype. GSDPA_BF16 needs an sm_103 device.
 *   workspace       : device scratch of at least gsdpa_workspace_bytes(...)
 *                     bytes, 256-byte aligned; contents need not be
 *                     initialised and are overwritten. NULL allowed when 0.
 *   stream          : a cudaStream_t (NULL = legacy default stream).
 *
 * X, Q, K, V, W_g and O must be 16-byte aligned and sink 4-byte aligned
 * (GSDPA_ERR_ALIGNMENT otherwise).
 * Calls that share a workspace must not overlap on the device.
 */
GSDPA_API int gated_sdpa_fwd(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                   void* O, float* sink,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The forward with one of the gate variants of "GatedAttention [2025]"
 * (sec. 1.2.2 items (3)-(5): head-shared gates, additive gating with sigmoid
 * or SiLU; sec. 1.4.1: SiLU of the output with no parameters, additive gating
 * without SiLU, per-head RMSNorm before concatenation; sec. 1.4.2: an
 * input-independent gate, NS-sigmoid). The gate shape is gate_mode, how the
 * gate acts on the SDPA output y is gate_fn:
 *   gate_mode HEADWISE, ELEMENTWISE and the two _SHARED shapes: logit
 *     gl = X W_g for the columns the shape gives; gate_fn one of
 *     SIGMOID_MUL .. IDENTITY_ADD;
 *   gate_mode STATIC: gl = theta[h, c] from W_g ([H_q, d_k], same dtype as
 *     the call); X is not read and may be NULL; gate_fn as above;
 *   gate_mode HEADWISE_AVERAGED, ELEMENTWISE_AVERAGED: the head-shared gate
 *     read as an average over the query heads (sec. 1.3.2 (ii)): the
 *     head-specific gate values v_h = f(gl_h) of every head h (gl = X W_g as
 *     for HEADWISE, ELEMENTWISE; f the gate_fn's function of the logit) are
 *     averaged, vbar = (1/H_q) sum_h v_h, and every head combines the same
 *     vbar with its y (multiplied or added as gate_fn says); prefill only
 *     (L_q == 1 decode calls return GSDPA_ERR_UNSUPPORTED);
 *   gate_mode NONE: gate_fn SIGMOID_MUL (plain SDPA), SILU_SELF or RMSNORM
 *     (W_g = gamma [H_q, d_k] or NULL; eps >= 0 is added to the mean square).
 * Other combinations return GSDPA_ERR_INVALID_ARG. The gate's value is kept
 * as fp16 between the gate pass and the attention kernel (bf16 path), as for
 * gated_sdpa_fwd. Workspace: gsdpa_workspace_bytes_variant. All other
 * arguments, alignment and errors as for gated_sdpa_fwd; gate_fn
 * SIGMOID_MUL with gate_mode 0..2 is gated_sdpa_fwd.
 */
GSDPA_API size_t gsdpa_workspace_bytes_variant(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                                               int gate_mode, int gate_fn, int want_sink, int dtype);
GSDPA_API int gated_sdpa_fwd_variant(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                                     void* O, float* sink, int B, int L_q, int L_k, int d_model, int H_q, int H_kv,
                                     int d_k, int gate_mode, int gate_fn, float eps, int causal, int dtype,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * gated_sdpa_fwd that also measures the gate's scores ("GatedAttention
 * [2025]", sec. 1.4.2: the mean gating score of Table 4, the score
 * distribution of Figure 3, and the fraction of scores below a threshold):
 *   stats     : device array of 3 + n_bins unsigned 64-bit counters, 8-byte
 *               aligned, overwritten by the call:
 *               [0] number of scores (B L_q H_q d_k elementwise, B L_q H_q headwise),
 *               [1] the sum of the scores times 2^32 in fixed point: exactly
 *                   the sum of round(score * 2^32) for the headwise gate, the
 *                   decode kernel and the float32 path; the bf16 elementwise
 *                   prefill rounds each thread's float32 partial sums (of at
 *                   most 256 scores) once, so its mean is within 2^-18 of the
 *                   exact mean of the scores,
 *               [2] number of scores < threshold,
 *               [3 + k] scores s with min(floor(s n_bins), n_bins - 1) = k.
 *               Integer counters: the result does not depend on the order in
 *               which threads add them (two calls give the same bits). The
 *               score is the value the call multiplies by (bf16 path: the
 *               fp16 value of the elementwise gate; the fp32 value of the
 *               headwise gate).
 *   n_bins    : 1 .. 64.   threshold : in [0, 1].
 * gate_mode HEADWISE or ELEMENTWISE (GSDPA_ERR_INVALID_ARG otherwise); other
 * arguments, workspace and errors as for gated_sdpa_fwd (an empty problem
 * enqueues nothing and leaves stats as they are).
 */
GSDPA_API int gated_sdpa_fwd_stats(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                                   void* O, float* sink, unsigned long long* stats, int n_bins, float threshold,
                                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k, int gate_mode,
                                   int causal, int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The whole layer around the attention ("GatedAttention [2025]", sec. 1.2.1:
 * Q, K, V projected from the hidden state X; sec. 1.2.2: the gate reads X
 * too; the heads' gated outputs concatenated and projected by W_O):
 *   [Q | K | V | GL] = X W_in                    one GEMM (the four share X)
 *   Y = (softmax(Q K^T / sqrt(d_k) + causal) V (.) sigma(GL)) W_O
 * with the attention of gated_sdpa_fwd in between. Self-attention (L_q = L_k
 * = L) without a cache.
 *   X      : device bf16 [B, L, d_model].
 *   W_in   : device bf16 [d_model, (H_q + 2 H_kv) d_k + G] with G = H_q d_k
 *            (elementwise gate), H_q (headwise gate) or 0 (no gate);
 *            columns: the Q heads, the K heads, the V heads, then the gate's
 *            columns (head-major, like gated_sdpa_fwd's W_g).
 *   W_O    : device bf16 [H_q d_k, d_model].
 *   Y      : device bf16 [B, L, d_model] out.
 *   gate_mode NONE, HEADWISE or ELEMENTWISE (GSDPA_ERR_INVALID_ARG
 *   otherwise); bf16, d_k = 128, L >= 2, d_model a multiple of 8 and >= 256,
 *   H_q a multiple of 8 with the headwise gate (GSDPA_ERR_UNSUPPORTED
 *   otherwise).
 * Q, K, V and the pre-W_O output live in the workspace (bf16), the gate as
 * fp16 values (elementwise) or float32 logits (headwise), as in
 * gated_sdpa_fwd. Pointers 16-byte aligned; asynchronous on `stream`; errors
 * as for gated_sdpa_fwd.
 */
GSDPA_API size_t gsdpa_layer_workspace_bytes(int B, int L, int d_model, int H_q, int H_kv, int d_k, int gate_mode);
GSDPA_API int gated_attention_layer(const void* X, const void* W_in, const void* W_O, void* Y, int B, int L,
                                    int d_model, int H_q, int H_kv, int d_k, int gate_mode, int causal,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * The forward a training step runs: gated_sdpa_fwd, and also, for every
 * batch b, query head h and query row i, the natural log of the softmax
 * denominator, lse[b, h, i] = log sum_j exp(s_j) over the row's visible
 * scores s_j = Q.K / sqrt(d_k) ("GatedAttention [2025]", sec. 1.2.1: the
 * softmax of the SDPA equation; the backward rebuilds the weights from it).
 *
 *   lse : device float32 [B, H_q, L_q] (head-major), 4-byte aligned; required.
 *   Other arguments and the workspace as for gated_sdpa_fwd.
 * bf16 prefill only (L_q != 1): GSDPA_ERR_UNSUPPORTED otherwise.
 */
GSDPA_API int gated_sdpa_fwd_train(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                   void* O, float* sink, float* lse,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * gated_sdpa_fwd_train for the elementwise gate that also saves the gate's
 * values for the backward pass (gated_sdpa_bwd_saved_gate then skips their
 * recomputation, a GEMM of the size of the gate's):
 *   gate_out : device fp16 [B * L_q, H_q * d_k], 16-byte aligned, overwritten
 *              with sigma(X W_g) exactly as the forward multiplied by it.
 * gate_mode ELEMENTWISE and gate_out non-NULL (GSDPA_ERR_INVALID_ARG
 * otherwise); other arguments, workspace and errors as for
 * gated_sdpa_fwd_train. The values are copied from the workspace after the
 * call's kernels, on the same stream.
 */
GSDPA_API int gated_sdpa_fwd_train_save_gate(const void* X, const void* Q, const void* K, const void* V,
                   const void* W_g, void* O, float* sink, float* lse, void* gate_out,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Workspace bytes gated_sdpa_bwd needs for this problem (bf16, d_k = 128);
 * (size_t)-1 for an invalid or unsupported shape, 0 for an empty one.
 */
GSDPA_API size_t gsdpa_bwd_workspace_bytes(int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode);

/*
 * The backward pass of the layer: given dO = dL/dO, the gradients of the
 * loss with respect to Q, K, V and, with a gate, W_g and X (the gate path's
 * share of dX; X also feeds projections this library does not own).
 * The chain rule of the forward ("GatedAttention [2025]", sec. 1.2.1 and
 * 1.2.2); the gate's part as in "解密NeurIPS最佳论文：Gated Attention…",
 * sec. 2.2: the gradient on the gate's input is dO times the ungated output
 * times sigma (1 - sigma).
 *
 *   X, Q, K, V, W_g : the forward's inputs (same layouts as gated_sdpa_fwd).
 *   O, lse          : the forward's output [B, L_q, H_q, d_k] and its
 *                     log-denominators [B, H_q, L_q] (gated_sdpa_fwd_train).
 *   dO              : device [B, L_q, H_q, d_k], same dtype.
 *   dQ              : out, like Q.   dK, dV : out, like K and V (each the sum
 *                     over the query heads of the kv head's group).
 *   dX, dW_g        : out, like X and W_g (gated only; NULL allowed without a gate).
 *   workspace       : gsdpa_bwd_workspace_bytes(...) bytes, 256-byte aligned.
 * Every output is overwritten. bf16, d_k = 128 and gate_mode NONE, HEADWISE
 * or ELEMENTWISE with the sigmoid gate only (GSDPA_ERR_UNSUPPORTED otherwise:
 * the variants of gated_sdpa_fwd_variant have no backward); sm_103 device.
 * Tensors 16-byte aligned, lse 4-byte aligned.
 * Asynchronous on `stream`; errors as for gated_sdpa_fwd.
 */
GSDPA_API int gated_sdpa_bwd(const void* X, const void* Q, const void* K, const void* V, const void* W_g,
                   const void* O, const void* dO, const float* lse,
                   void* dX, void* dQ, void* dK, void* dV, void* dW_g,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * gated_sdpa_bwd for the elementwise gate with the gate's values taken from
 * gate_saved (what gated_sdpa_fwd_train_save_gate wrote: fp16
 * [B * L_q, H_q * d_k], 16-byte aligned) instead of recomputed from X and
 * W_g. With the forward's own values the outputs equal gated_sdpa_bwd's bit
 * for bit. gate_mode ELEMENTWISE and gate_saved non-NULL
 * (GSDPA_ERR_INVALID_ARG otherwise); other arguments, workspace (the same
 * gsdpa_bwd_workspace_bytes) and errors as for gated_sdpa_bwd.
 */
GSDPA_API int gated_sdpa_bwd_saved_gate(const void* X, const void* Q, const void* K, const void* V,
                   const void* W_g, const void* O, const void* dO, const float* lse,
                   const void* gate_saved,
                   void* dX, void* dQ, void* dK, void* dV, void* dW_g,
                   int B, int L_q, int L_k, int d_model, int H_q, int H_kv, int d_k,
                   int gate_mode, int causal, int dtype,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * bounded waits inside the kernels set when they run out. Returns GSDPA_OK,
 * GSDPA_ERR_DEVICE_TIMEOUT, or GSDPA_ERR_LAUNCH if the stream itself reports
 * a CUDA error.
 */
GSDPA_API int gsdpa_check_device_error(void* stream);

/* A static, human-readable name for a gsdpa_status value. */
GSDPA_API const char* gsdpa_status_string(int status);

/*
 * gated_sdpa_decode_noalloc -- the decode call (one query row per sequence,
 * L_q == 1) for callers that cannot allocate device memory. (The pages
 * describe no such entry point; it belongs to this library's interface only.)
 *
 * Some callers cannot hand the library a workspace: code that must never make
 * the device synchronise (cudaMalloc and cudaFree can), plugin or callback
 * hooks that provide no allocator, or processes with a device memory budget
 * fixed in advance. This entry point takes no workspace: its scratch (the
 * split-K partials, the gate-logit partials and the arrival counters) lives
 * in a 16 MiB array inside the library that every GPU loading the library
 * holds until the process exits (see gsdpa_decode_noalloc_max_scratch()).
 *
 *   Arguments are those of gated_sdpa_fwd with L_q = 1, causal, bf16 implied.
 *   Covered gate modes: GSDPA_GATE_NONE, GSDPA_GATE_HEADWISE and
 *   GSDPA_GATE_ELEMENTWISE (sigmoid gate); the head-shared and input-independent
 *   modes return GSDPA_ERR_UNSUPPORTED, values outside gsdpa_gate_mode
 *   GSDPA_ERR_INVALID_ARG. Covered shapes: d_k == 128 and H_q / H_kv a multiple
 *   of 4 (the dedicated decode kernel); others return GSDPA_ERR_UNSUPPORTED. A
 *   problem whose scratch exceeds the fixed array returns GSDPA_ERR_WORKSPACE
 *   (the size a problem needs is gsdpa_workspace_bytes(B, 1, L_k, ...,
 *   dtype = GSDPA_BF16)).
 *
 * The first call on a device resolves the array's device address (a runtime
 * query, no allocation); make that first call before any stream capture. The
 * address is kept for the life of the process: no call may follow a
 * cudaDeviceReset (or any reset of the device's primary context) in the same
 * process. The array is shared by all calls on a device and keeps the last
 * call's contents; counters are cleared at the start of each call. Calls that
 * overlap on the device race on the array: serialise them.
 */
GSDPA_API int gated_sdpa_decode_noalloc(const void* X, const void* Q, const void* K, const void* V,
                                        const void* W_g, void* O, float* sink,
                                        int B, int L_k, int d_model, int H_q, int H_kv, int d_k,
                                        int gate_mode, void* stream);

/* Size in bytes of the fixed scratch array used by gated_sdpa_decode_noalloc. */
GSDPA_API size_t gsdpa_decode_noalloc_max_scratch(void);

/*
 * Test hook, not part of the operation: sets the wait limit, in nanoseconds,
 * that every bounded wait inside the kernels uses from the next launch on
 * (0 restores the default of 2 s). Lets a test make a wait run out quickly.
 */
GSDPA_API int gsdpa_set_wait_limit_ns(unsigned long long ns);

/*
 * Diagnostic, not part of the operation: enqueues on `stream` one thread that
 * waits, with the current wait limit, on a barrier that nothing ever
 * completes. The wait gives up and records the timeout in the device error
 * word, which the next gsdpa_check_device_error() returns as
 * GSDPA_ERR_DEVICE_TIMEOUT (and clears). Lets a test exercise the bounded-wait
 * path without faulting or hanging the device. Returns GSDPA_OK or
 * GSDPA_ERR_LAUNCH.
 */
GSDPA_API int gsdpa_wait_self_test(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GSDPA_H_ */
