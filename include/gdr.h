/*
 * gdr.h -- C ABI of the GB300 (sm_103a) chunked gated delta-rule backward.
 *
 * The method: linear attention with the gated delta rule, per (sequence, head)
 *
 *     qn = q / sqrt(|q|^2 + 1e-6),   kn = k / sqrt(|k|^2 + 1e-6),   beta = sigmoid(b)
 *     S_t = (I - beta_t kn_t kn_t^T) diag(exp g_t) S_{t-1} + beta_t kn_t v_t^T
 *     o_t = scale * S_t^T qn_t
 *
 * with a scalar log gate per token and head (GDN) or a per-channel log gate
 * g = -exp(A_log[h]) * softplus(g_raw + dt_bias[h, :]) (KDA).  The decay is
 * applied before the delta update; for a scalar gate the two orders agree.
 * Sources: the FlashQLA GDN backward page ("FlashQLA ... GDN 反向", §一 for the
 * backward's inputs and outputs: q, k, v, g, beta, h0, dO, optional dht ->
 * dq, dk, dv (bf16), dg, dbeta, dh0 (fp32)) and "FlashKDA之backward（K1）" (the
 * KDA gate parameters, the L2 norm with eps 1e-6, beta in logit space, the
 * atomically reduced dA_log / ddt_bias, varlen through int64 cu_seqlens).
 * The loss whose gradients are returned is  sum_t <dO_t, o_t> + sum <dht, S_T>.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  * All tensor pointers are DEVICE pointers, 16-byte aligned, contiguous:
 *      q, k, v, dO, dq, dk, dv, g_raw, dg_raw : bf16   [T_total, H, D]   (token-major;
 *                                               q, k, dq, dk [T_total, Hk, D] with GQA)
 *      beta_logit, dbeta                      : bf16   [T_total, H]
 *      g, dg  (GDN natural-log gate)          : float  [T_total, H]
 *      A_log, dA_log                          : float  [H]
 *      dt_bias, ddt_bias                      : float  [H, D]
 *      h0, dht, dh0                           : float  [N, H, D, D]  (row = key channel)
 *  * cu_seqlens: device int64 [N + 1], 0 = cu[0] <= cu[1] <= ... <= cu[N] = T_total;
 *    NULL means dense: N sequences of T_total / N tokens each.
 *  * h0 and dht may be NULL (zero).  All outputs are written in full (rows of
 *    every sequence); the library never writes outside the given tensors.
 *  * T_total = 0 (every sequence empty) is a valid call: the token tensors may then be
 *    NULL, dh0 receives dht (or zeros), ht receives h0, dA_log and ddt_bias are zero.
 *  * Ownership: the caller allocates every buffer, including the workspace
 *    (size from gdr_workspace_bytes) and the states buffer (gdr_states_bytes).
 *    The library allocates no device memory and keeps no state besides a
 *    thread-local error string and the optional instrumentation events of
 *    gdr_profile_begin.
 *  * Asynchrony: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and the call returns without synchronising.  Argument
 *    errors are detected on the host before anything is enqueued.  Conditions
 *    only the device can see (inconsistent cu_seqlens, a gate range the
 *    kernels cannot represent) set bits in the workspace status word; read
 *    it with gdr_workspace_status after the work completes.
 *  * Calls that share a workspace must not run concurrently.
 *  * Stream capture: gdr_bwd and kda_bwd enqueue only kernels and memsets on `stream`
 *    and never wait on the host, so a call can be captured into a CUDA graph and
 *    replayed (with the same buffers); the replay gives the same results.
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDR_OK = 0,
    GDR_ERR_INVALID = 1,      /* null / misaligned pointer, bad size or shape (also a problem
                                 whose per-chunk tiles exceed 32-bit row addressing: chunks x
                                 heads x 192 rows must stay below 2^31) */
    GDR_ERR_UNSUPPORTED = 2,  /* head_dim not in {64, 128} */
    GDR_ERR_WORKSPACE = 3,    /* workspace or states buffer too small */
    GDR_ERR_CUDA = 4          /* a CUDA runtime call or kernel launch failed */
} gdr_status;

/* Device-side status bits (gdr_workspace_status). */
#define GDR_DEV_BAD_SEQLENS 1 /* cu_seqlens not non-decreasing from 0 to T_total */
#define GDR_DEV_GATE_RANGE 2  /* a chunk's log-gate span exceeded 160 (or a cumulative gate > 80) */
#define GDR_DEV_TIMEOUT 4     /* a bounded wait for the tensor cores ran out; that CTA's outputs are missing */
#define GDR_DEV_STATES_MISMATCH 8 /* gdr_bwd / kda_bwd got a states buffer written for another variant,
                                     gate function, h0 presence or shape: the main backward wrote none
                                     of dq, dk, dv, dg / dg_raw, dbeta, dA_log, ddt_bias */

typedef struct {
    int32_t num_seqs;          /* N >= 1 */
    int64_t total_tokens;      /* T_total >= 0 */
    int32_t num_heads;         /* H >= 1 */
    int32_t head_dim;          /* D = dk = dv, 64 or 128.  64 runs the 128-channel kernels on
                                * inputs zero-padded to 128 channels in the workspace (zero
                                * channels leave every product, norm and sum of the method
                                * unchanged; the results are the first 64 channels) */
    const int64_t* cu_seqlens; /* device int64 [N + 1], or NULL for dense */
    float scale;               /* output scale, usually 1 / sqrt(D) */
    /* KDA only (ignored by the GDN calls): the per-channel gate function, with
     * x = g_raw + dt_bias[h, :] and a = exp(A_log[h]):
     *   GDR_KDA_GATE_SOFTPLUS (0): g = -a * softplus(x)
     *   GDR_KDA_GATE_SIGMOID  (1): g = ln(2) * gate_scale * sigmoid(a * x), the
     *     sigmoid-bounded gate of "FlashKDA之backward（K1）" §5.2 (whose base-2 log
     *     gate is gate_scale * sigmoid(a x)); gate_scale must be finite and <= 0. */
    int32_t kda_gate;
    float gate_scale;
    /* Grouped q / k heads (GQA): the number Hk of q and k heads, 0 meaning num_heads.
     * num_heads (H) counts the heads of everything else (v, gates, beta, states, o, dO);
     * H must be a multiple of Hk, and value head h reads q / k head h / (H / Hk).  q, k,
     * dq and dk are then [T_total, Hk, D]; dq and dk sum over each group. */
    int32_t num_k_heads;
} gdr_shape;
#define GDR_KDA_GATE_SOFTPLUS 0
#define GDR_KDA_GATE_SIGMOID 1

/* Bytes of the scratch workspace that gdr_fwd_states / gdr_bwd / kda_fwd_states /
 * kda_bwd need for this shape (returns 0 for an invalid shape); for head_dim 64 it
 * includes the zero-padded copies of the inputs and outputs. */
size_t gdr_workspace_bytes(const gdr_shape* shape);

/* Bytes of the per-chunk state buffer written by gdr_fwd_states / kda_fwd_states /
 * gdr_fwd / kda_fwd: a header of GDR_STATES_HEADER_BYTES, then the bf16 chunk-start
 * state of every 64-token chunk and head, stored value-major ([chunk][head][dv][dk],
 * i.e. S^T, the layout the tensor-core products read), with chunks numbered sequence
 * after sequence.
 *
 * head_dim 64 runs on the channels zero-padded to 128 (see gdr_shape.head_dim), and
 * its states keep that padded layout ([chunk][head][128][128]).
 *
 * The header records what the states were computed for: the variant (GDN, KDA with
 * the softplus gate, KDA with the sigmoid-bounded gate and its gate_scale), whether
 * h0 was given, N, H, Hk, D, T_total and dense / varlen.  gdr_bwd and kda_bwd compare
 * it on the device with their own call (the call itself is asynchronous and cannot
 * wait for the buffer): on any difference the main backward writes nothing and
 * raises GDR_DEV_STATES_MISMATCH in the workspace status word.  The header cannot
 * tell two inputs of one shape apart: the caller passes the states of the inputs it
 * differentiates. */
#define GDR_STATES_HEADER_BYTES 256
size_t gdr_states_bytes(const gdr_shape* shape);

/* Forward chunk states for GDN (the "forward workspace" of the FlashKDA
 * pipeline, here the chunk-start state S0 of each chunk, saved so the backward
 * can skip its own recomputation).  Writes `states`. */
gdr_status gdr_fwd_states(const gdr_shape* shape, const void* q, const void* k, const void* v,
                          const float* g, const void* beta_logit, const float* h0,
                          void* states, size_t states_bytes, void* workspace,
                          size_t workspace_bytes, void* stream);

/* Same for KDA (per-channel gate from g_raw, A_log, dt_bias). */
gdr_status kda_fwd_states(const gdr_shape* shape, const void* q, const void* k, const void* v,
                          const void* g_raw, const float* A_log, const float* dt_bias,
                          const void* beta_logit, const float* h0, void* states,
                          size_t states_bytes, void* workspace, size_t workspace_bytes,
                          void* stream);

/* GDN forward: the output o (bf16 [T_total, H, D]) and, if ht is not NULL, the final
 * state of every sequence and head (fp32 [N, H, D, D], row = key channel), from the
 * chunked form of the recurrence (the forward that the backward of
 * "FlashKDA之backward（K1）" undoes, its §0.1: per chunk o = qd S0 + P u with the
 * WY/UT factors).  If `states` is not NULL it also receives
 * the chunk-start states (the buffer of gdr_fwd_states; states_bytes >=
 * gdr_states_bytes), so a following gdr_bwd can skip their recomputation.  Uses the
 * same workspace as gdr_bwd (gdr_workspace_bytes). */
gdr_status gdr_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                   const float* g, const void* beta_logit, const float* h0, void* o, float* ht,
                   void* states, size_t states_bytes, void* workspace, size_t workspace_bytes,
                   void* stream);
/* KDA forward (per-channel gate from g_raw, A_log, dt_bias); as gdr_fwd. */
gdr_status kda_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                   const void* g_raw, const float* A_log, const float* dt_bias,
                   const void* beta_logit, const float* h0, void* o, float* ht, void* states,
                   size_t states_bytes, void* workspace, size_t workspace_bytes, void* stream);
/* GDN backward ("FlashQLA ... GDN 反向", §一-§二: one call returns dq, dk, dv, dg,
 * dbeta, dh0).  `states` is the buffer from gdr_fwd_states for the same inputs,
 * or NULL to recompute the chunk states inside the call.  dg is the gradient
 * w.r.t. the per-token log gate g (the reverse cumsum is done inside); dbeta is
 * w.r.t. the beta logit; dh0 is fp32 and always written. */
gdr_status gdr_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                   const float* g, const void* beta_logit, const float* h0, const void* dO,
                   const float* dht, const void* states, void* workspace, size_t workspace_bytes,
                   void* dq, void* dk, void* dv, float* dg, void* dbeta, float* dh0,
                   void* stream);

/* KDA backward ("FlashKDA之backward（K1）": gate chain per element, dA_log and
 * ddt_bias reduced over all tokens).  dg_raw is w.r.t. g_raw (bf16).  dA_log and
 * ddt_bias are overwritten (zeroed on the stream, then accumulated). */
gdr_status kda_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                   const void* g_raw, const float* A_log, const float* dt_bias,
                   const void* beta_logit, const float* h0, const void* dO, const float* dht,
                   const void* states, void* workspace, size_t workspace_bytes, void* dq,
                   void* dk, void* dv, void* dg_raw, void* dbeta, float* dh0, float* dA_log,
                   float* ddt_bias, void* stream);

/* Allocation-free GDN backward (an addition of this library; the pages have no
 * counterpart).  For callers that cannot allocate device memory where they run
 * the backward: a plug-in whose host framework owns every device allocation,
 * or code where a cudaMalloc (which may synchronise or fail) is not allowed.
 *
 * Same arguments and results as gdr_bwd, without the workspace: the scratch
 * is a static device array of GDR_FIXED_WORKSPACE_BYTES inside this library,
 * which every GPU that loads the library holds until the process exits.
 *  * Problems whose gdr_workspace_bytes exceeds that size are rejected with
 *    GDR_ERR_WORKSPACE (message in gdr_last_error) before anything is enqueued.
 *  * The first call on a device (per process) resolves the array's device
 *    address with cudaGetSymbolAddress, with that device current; make that
 *    first call before any stream capture.  The address is kept for the life of
 *    the process: after a cudaDeviceReset of that device (which unloads the
 *    library's device code and may move the array) this entry point must not be
 *    called again in the same process.
 *  * Every call on a device shares the one array and leaves its contents
 *    behind: calls that overlap on the GPU (different streams, or threads
 *    without ordering) race; serialise them, e.g. on one stream.
 *  * Device-side status bits (gdr_workspace_status) are not reported: the
 *    caller has no handle on the scratch.
 *  * Allocates nothing: no cudaMalloc / cudaFree or allocating library call. */
#define GDR_FIXED_WORKSPACE_BYTES (64u << 20)
#define GDR_FIXED_MAX_DEVICES 64
gdr_status gdr_bwd_fixed(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const void* beta_logit, const float* h0, const void* dO,
                         const float* dht, const void* states, void* dq, void* dk, void* dv,
                         float* dg, void* dbeta, float* dh0, void* stream);

/* Backward of the causal depthwise conv1d (optionally followed by SiLU) that produces
 * q, k and v in a gated delta-rule layer ("第三章 反向传播的完整推导", the
 * causal-convolution page): per channel c with `width` K taps and zero state before
 * each sequence's first token,
 *     z_t = bias[c] + sum_k weight[c, k] x[t-K+1+k, c],   y = silu ? z sigmoid(z) : z.
 * Given dy = dL/dy it writes dx (bf16), dweight (fp32 [C, K]) and, if dbias is not
 * NULL, dbias (fp32 [C]); the pre-activation z is recomputed from x.
 *  * x, dy, dx: bf16 [T_total, C] token-major (C = channels, even);
 *    weight fp32 [C, K], 1 <= K <= 4; bias fp32 [C] or NULL (zero).
 *  * cu_seqlens: device int64 [N + 1] or NULL (dense: N sequences of T_total / N
 *    tokens); no sum crosses a sequence boundary.  Inconsistent cu_seqlens give
 *    meaningless gradients but no access outside the tensors.
 *  * dweight and dbias are overwritten (zeroed on the stream, then accumulated
 *    with atomics, so their last bits depend on the order of the additions). */
gdr_status gdr_conv1d_bwd(int32_t num_seqs, int64_t total_tokens, int32_t channels, int32_t width,
                          const int64_t* cu_seqlens, const void* x, const float* weight,
                          const float* bias, const void* dy, int32_t silu, void* dx,
                          float* dweight, float* dbias, void* stream);
/* Waits for `stream`, then returns in *device_status the OR of the GDR_DEV_*
 * bits raised by the last call that used `workspace` (0 = none). */
gdr_status gdr_workspace_status(const void* workspace, void* stream, int* device_status);

/* Test hook (not part of the method; off unless called).  Makes the next gdr_bwd
 * call on any thread with head_dim 128 hold CTA `cta` of its main backward kernel at
 * its first item on an mbarrier that nothing arrives on, under a short bounded wait
 * (no copy or tensor-core operation is pending on that barrier).  The wait runs out,
 * the CTA records GDR_DEV_TIMEOUT, drains the tile loads it has issued, releases its
 * tensor memory and exits; the other CTAs finish.  It exercises the path every bounded
 * wait of the kernels takes when the tensor cores do not answer, without a GPU fault.
 * cta < 0 clears a pending request.  Not thread-safe with concurrent gdr_bwd calls. */
void gdr_test_stall_next_call(int cta);

/* Message of the last error returned on the calling thread ("" if none). */
const char* gdr_last_error(void);

/* Instrumentation (not part of the method): per-kernel device timing.
 * gdr_profile_begin(n) makes the next n timed sections of this library (one
 * kernel kind of one call; the state recurrences of a call are one section of
 * up to three kernels: two chain phases and the segment boundaries) record a
 * CUDA event pair on their stream (on any thread, not thread-safe);
 * gdr_profile_end waits for them and writes, per kernel kind, the summed
 * milliseconds and the number of kernels launched (arrays of GDR_KERNEL_COUNT). */
#define GDR_KERNEL_CHUNK_TABLE 0 /* varlen chunk table */
#define GDR_KERNEL_PREP 1        /* chunk-parallel intra-chunk preparation */
#define GDR_KERNEL_STATES 2      /* serial state / state-gradient recurrences */
#define GDR_KERNEL_MAIN 3        /* chunk-parallel main backward */
#define GDR_KERNEL_OUT 4         /* chunk-parallel forward output (gdr_fwd / kda_fwd) */
#define GDR_KERNEL_CONV 5        /* causal conv1d backward (gdr_conv1d_bwd) */
#define GDR_KERNEL_COUNT 6
gdr_status gdr_profile_begin(int max_launches);
gdr_status gdr_profile_end(double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
