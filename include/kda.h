/*
 * kda.h -- C ABI of the GB300 (sm_103a) KDA recurrence library, libkda_gb300.so.
 *
 * KDA (Kimi Delta Attention) keeps, per head, a dk x dv fp32 state S and for
 * every token t applies the per-channel gated delta rule
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t                      (read out from the UPDATED state)
 *
 * Defined by: "Colibri Kimi K3 Metal backend" (architecture section, the
 * state update; section 8.2, the two-pass token step and its readout;
 * section 8.4, alpha = exp(g) per element and beta per head), with the model
 * sizes of "Kimi K3 -> TPU v7x feasibility" (section 2 model table: 96 heads,
 * head width 128, decay gate lower bound -5).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless marked "host"; the caller owns all
 *     memory it passes.  The tensor-core prefill (bf16, chunk 64) also needs
 *     a scratch workspace of 59 KB per (64-token chunk, head):
 *     kda_prefill_chunked takes it from a library-owned stream-ordered memory
 *     pool on the current device, which keeps that memory for later calls;
 *     kda_prefill_chunked_ws runs in a buffer the caller passes, and
 *     kda_prefill_chunked_noalloc in a fixed array in the library's device
 *     image.  That pool, that array and the device error word
 *     (kda_device_error) are the library's only global state.
 *   - Layouts are token-major and dense (C order):
 *         q, k, g : [T, H, dk]      v, o : [T, H, dv]      beta : [T, H]
 *         S       : [N, H, dk, dv]  with S[n][h][i][j], i = key channel,
 *                                   j = value channel (the pages' S[i][j],
 *                                   decayed per row i)
 *   - q, k, v are bf16 (KDA_BF16) or fp32 (KDA_F32); g, beta, S and o are
 *     always fp32.  g is the log-decay (decay = exp(g)); beta is already in
 *     [0, 1] (any sigmoid is applied by the caller); q is used as given (any
 *     1/sqrt(dk) scale is folded in by the caller).
 *   - Supported sizes: dk = dv = 128.  Preconditions: -5 <= g <= 0 (the
 *     model's gate bound; the tensor-core prefill's decay folding relies on
 *     it and raises bit 2 of the device error word when it sees a gate
 *     outside that range, or a NaN, in a prefill's input); for the
 *     tensor-core prefill, |q| |k| and |v| far below 65504 (q and k are
 *     L2-normalised in the model, as the layer's prologue makes them; u is
 *     checked, bit 4 below); finite inputs (not checked elsewhere).
 *   - Every pointer must be 16-byte aligned (KDA_ERR_ALIGN otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream); they never synchronise.  Arguments are validated on
 *     the host before any launch; on an argument error nothing is launched.
 *     A launch failure is reported as KDA_ERR_CUDA.  Calls never throw.
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_NULL = 1,        /* a required pointer is NULL */
    KDA_ERR_DIM = 2,         /* unsupported or inconsistent sizes */
    KDA_ERR_CHUNK = 3,       /* chunk not in {16, 32, 64} */
    KDA_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    KDA_ERR_DTYPE = 5,       /* dtype not a kda_dtype_t */
    KDA_ERR_WORKSPACE = 6,   /* the prefill's scratch workspace could not be allocated, or the caller's is too small */
    KDA_ERR_CUDA = 7,        /* the CUDA runtime reported an error at launch */
    KDA_ERR_VALUE = 8        /* a scalar argument is out of range, or buffers alias */
} kda_status_t;

typedef enum {
    KDA_BF16 = 0,            /* q, k, v stored as bfloat16 */
    KDA_F32 = 1              /* q, k, v stored as float32 */
} kda_dtype_t;

/* Library version, major * 10000 + minor * 100 + patch. */
int kda_version(void);

/* Static string naming a status code (never NULL). */
const char *kda_status_string(int status);

/*
 * Chunked prefill over a packed batch of N variable-length sequences.
 *
 * Operation: for every sequence n (tokens cu_seqlens[n] .. cu_seqlens[n+1]-1)
 * and head h, run the recurrence above from S0[n][h] (zeros if S0 == NULL),
 * write o for each token and the final state to S_out[n][h].  The chunked
 * form (chunks of `chunk` tokens, UT transform inside a chunk, fp32 state
 * carried between chunks) computes the same map up to rounding; it follows
 * from unrolling the recurrence inside a chunk.  The varlen packing follows
 * the per-sequence (cu_seqlens) convention of the TPU KDA kernel ("Kimi K3
 * -> TPU v7x feasibility", section 4.2).  Sequences of any length (including
 * 0, and lengths that are not a multiple of `chunk`) are handled in the
 * kernel; an empty sequence copies S0 (or zeros) to S_out.
 *
 *   q, k       [T, H, dk]  bf16 or fp32 (dtype)
 *   v          [T, H, dv]  bf16 or fp32
 *   g          [T, H, dk]  fp32 log-decay
 *   beta       [T, H]      fp32
 *   S0         [N, H, dk, dv] fp32, or NULL for a zero initial state
 *   o          [T, H, dv]  fp32, written
 *   S_out      [N, H, dk, dv] fp32, written; may alias S0 exactly (in place)
 *   cu_seqlens [N + 1]     int32 DEVICE array, cu_seqlens[0] = 0,
 *                          non-decreasing, cu_seqlens[N] = T.  The host
 *                          cannot read it; the kernels check it on the
 *                          device: entries below 0, above T or decreasing
 *                          raise bit 0 of the device error word, and no
 *                          kernel then reads or writes outside the buffers
 *                          sized for T (the outputs are invalid)
 *   N          number of sequences (>= 1); T total tokens (>= 0, < 2^31)
 *   H          heads (>= 1); dk, dv must be 128
 *   chunk      16, 32 or 64.  bf16 inputs with chunk 64 run on the
 *              tensor cores (tcgen05, TMA) in two kernels: an intra-chunk
 *              kernel over every (chunk, head) at once, then an inter-chunk
 *              state pass per (sequence, head); every other combination runs
 *              the fp32 CUDA-core kernel.
 *   dtype      kda_dtype_t of q, k, v
 *   stream     cudaStream_t
 * Returns KDA_OK or a kda_status_t (KDA_ERR_WORKSPACE when the tensor-core
 * path cannot get its workspace).  With T == 0 only S_out is written.
 */
int kda_prefill_chunked(const void *q, const void *k, const void *v,
                        const float *g, const float *beta, const float *S0,
                        float *o, float *S_out, const int32_t *cu_seqlens,
                        int N, int64_t T, int H, int dk, int dv, int chunk,
                        int dtype, void *stream);

/*
 * Measurement form of kda_prefill_chunked for the tensor-core path (bf16,
 * chunk 64, T > 0; KDA_ERR_CHUNK otherwise): the same computation, and it
 * records the caller's four timing events (cudaEvent_t, created by the
 * caller) on `stream` before the chunk-plan kernel, before the intra-chunk
 * kernel, before the state pass and after it, so that each kernel's time can
 * be read with cudaEventElapsedTime.  events: host array of 4 cudaEvent_t.
 */
int kda_prefill_chunked_events(const void *q, const void *k, const void *v,
                               const float *g, const float *beta, const float *S0,
                               float *o, float *S_out, const int32_t *cu_seqlens,
                               int N, int64_t T, int H, int dk, int dv, int chunk,
                               int dtype, void *stream, void *const *events);

/*
 * kda_prefill_chunked without any device allocation during the call.
 *
 * Same operation, arguments, layouts and results as kda_prefill_chunked.
 * The recurrence itself has no such variant (the pages describe no
 * workspace at all); this entry point exists for callers that may not
 * allocate device memory inside a call: runtimes that budget all device
 * memory in a fixed arena up front, where a library pool growing mid-call
 * would break the budget, and latency-critical loops where the first growth
 * of a pool (a driver allocation, which synchronises the device) cannot be
 * afforded.
 *
 * The tensor-core path (bf16, chunk 64, T > 0) takes its workspace from a
 * fixed 64 MiB array in the library's device image instead of the pool.  It
 * needs kda_prefill_workspace_bytes(N, T, H, ...) bytes (about
 * (ceil(T / 64) + N) * H * 60416); larger inputs are rejected with KDA_ERR_WORKSPACE before anything
 * is launched (for H = 96 and one sequence: T <= 640).  Every other dtype /
 * chunk combination runs the CUDA-core kernel, which needs no workspace.
 * Nothing in the array has to be cleared between calls.
 *
 * First call on each device: the library looks up the array's address
 * (cudaGetSymbolAddress, which may load the library's device image); make
 * that first call before any stream capture begins.  The address is cached
 * with the identity of the device's context; after a cudaDeviceReset the
 * next call looks it up again (so that call, too, should come before any
 * capture).  The array is shared by
 * all calls on a device: two calls whose executions overlap (different
 * streams, or different host threads) race on it and must be serialised by
 * the caller.  Returns KDA_OK or a kda_status_t.
 */
int kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v,
                                const float *g, const float *beta, const float *S0,
                                float *o, float *S_out, const int32_t *cu_seqlens,
                                int N, int64_t T, int H, int dk, int dv, int chunk,
                                int dtype, void *stream);

/*
 * Bytes of caller-owned workspace that kda_prefill_chunked_ws needs for these
 * sizes on the tensor-core path (bf16, chunk 64, T > 0): with
 * C = ceil(T / 64) + N chunks (one spare per sequence for a partial tail),
 * 1024 * ceil(4 (N + 2) / 1024) + 1024 * ceil(8 C / 1024) + C * H * 60416
 * (the chunk offsets and a job counter, the chunk table, one record per
 * (chunk, head)); 0 for
 * every other combination (the CUDA-core kernel needs none) and for invalid sizes.
 * Host-only, no CUDA call.
 */
size_t kda_prefill_workspace_bytes(int N, int64_t T, int H, int dk, int dv, int chunk, int dtype);

/*
 * kda_prefill_chunked with a workspace the caller owns (for instance a
 * buffer from the caller's own allocator), so that the library allocates
 * nothing.  Same operation, arguments, layouts and results as
 * kda_prefill_chunked, plus:
 *   workspace  device memory of ws_bytes bytes, 256-byte aligned
 *              (KDA_ERR_ALIGN otherwise), read and written by the call's
 *              kernels on `stream` (the caller keeps it alive and unshared
 *              until they finish); NULL is accepted where
 *              kda_prefill_workspace_bytes gives 0
 *   ws_bytes   at least kda_prefill_workspace_bytes(...) (KDA_ERR_WORKSPACE
 *              otherwise, before anything is launched)
 * Nothing in the workspace has to be initialised or cleared between calls.
 * Returns KDA_OK or a kda_status_t.
 */
int kda_prefill_chunked_ws(const void *q, const void *k, const void *v,
                           const float *g, const float *beta, const float *S0,
                           float *o, float *S_out, const int32_t *cu_seqlens,
                           int N, int64_t T, int H, int dk, int dv, int chunk,
                           int dtype, void *workspace, size_t ws_bytes, void *stream);

/*
 * One decode token for each of B sequences, state updated IN PLACE.
 *
 * Operation: the recurrence above applied once per (b, h) with
 * S = S_inout[b][h]: decay the rows by exp(g), u = S^T k, w = beta (v - u),
 * S += k w^T, o = S^T q (the two passes of "Colibri Kimi K3 Metal backend",
 * section 8.2, fused into one kernel that reads and writes each state once).
 *
 *   q, k      [B, H, dk]  bf16 or fp32 (dtype)
 *   v         [B, H, dv]  bf16 or fp32
 *   g         [B, H, dk]  fp32 log-decay
 *   beta      [B, H]      fp32
 *   S_inout   [B, H, dk, dv] fp32, read and overwritten in place
 *   o         [B, H, dv]  fp32, written (must not alias S_inout)
 *   B, H      >= 1 (B = 0 is a no-op returning KDA_OK); dk, dv must be 128
 * Returns KDA_OK or a kda_status_t.
 */
int kda_decode_step(const void *q, const void *k, const void *v,
                    const float *g, const float *beta, float *S_inout, float *o,
                    int B, int H, int dk, int dv, int dtype, void *stream);

/*
 * One decode token for each of B sequences whose states live in a pool:
 * sequence b reads and updates pool row state_indices[b] in place (the
 * decode-side interface of continuous batching: the TPU KDA decode kernel
 * indexes its state the same way, "Kimi K3 -> TPU v7x feasibility", section
 * 4.2), and the pool may be stored in bf16 to halve the state traffic (the
 * pages list a bf16 state as not yet evaluated for stability, same review,
 * section 6; the recurrence is computed in fp32 and each state value is
 * rounded to nearest-even bf16 when it is stored).
 *
 *   q, k, v, g, beta, o   as for kda_decode_step ([B, H, ...])
 *   S_pool        [P, H, dk, dv], fp32 (state_dtype KDA_F32) or bf16
 *                 (KDA_BF16), read and overwritten in place
 *   state_indices [B] int32 DEVICE array of pool rows, or NULL for the
 *                 identity (then P >= B).  A negative entry marks a padding
 *                 row: its o is written as zeros and no state is touched.
 *                 Entries must be distinct (two sequences on one row race);
 *                 an entry >= P is skipped like padding and sets bit 1 of
 *                 the device error word.
 *   P             pool rows (>= 0)
 * Returns KDA_OK or a kda_status_t; B = 0 is a no-op.
 */
int kda_decode_step_pool(const void *q, const void *k, const void *v,
                         const float *g, const float *beta, void *S_pool,
                         int state_dtype, const int32_t *state_indices, int P,
                         float *o, int B, int H, int dk, int dv, int dtype,
                         void *stream);

/* ---------------------------------------------------------------------------
 * The layer around the recurrence.  "Colibri Kimi K3 Metal backend",
 * section 8 introduction: per token the KDA layer runs conv1d + SiLU on its
 * q, k, v projections, L2-normalises q and k per head, steps the state, then
 * applies a per-head RMSNorm and a sigmoid of its full-rank gate projection
 * to o.  Section 8.3 gives the conv (a per-channel window of the last four
 * raw inputs, shifted left by one per token with the new input in the last
 * slot, dotted with the channel's four taps, then SiLU(x) = x / (1 + e^-x))
 * and the L2 norm (n = 1 / sqrt(sum x^2 + eps) over a head's 128 channels,
 * eps = 1e-6; q is scaled by n * q_scale, the pages' q_scale being
 * 1/sqrt(128); k by n; v is not normalised).  Section 8.4 gives the gated
 * norm: out = o / sqrt(mean_j o_j^2 + eps) * norm_w_j * sigmoid(gate_j).
 *
 * Conv windows ("conv states") are bf16 [rows, 3, 3, H, 128]: index 1 is the
 * projection (0 = q, 1 = k, 2 = v), index 2 the window slot, oldest first
 * (slot 2 = the input just before the next token).  They hold raw bf16
 * projections, so they are exact.  Conv taps are fp32 [3, H, 128, 4]: tap m
 * multiplies window slot m, tap 3 the newest input (y_t = sum_m w_m
 * x_{t-3+m}).
 * ------------------------------------------------------------------------- */

/*
 * conv1d + SiLU + L2-norm prologue of a packed varlen prefill: turns the raw
 * projections into the q, k, v that kda_prefill_chunked takes.
 *
 *   xq, xk, xv [T, H, 128] bf16 raw projections
 *   conv_w     [3, H, 128, 4] fp32 taps
 *   conv_in    [N, 3, 3, H, 128] bf16 window before each sequence, or NULL
 *              (zeros: every sequence starts fresh)
 *   conv_out   [N, 3, 3, H, 128] bf16, written: the window after each
 *              sequence's last token (conv_in's, or zeros, for an empty
 *              sequence), to carry into a later call or the decode step; or
 *              NULL.  Must not be conv_in (KDA_ERR_VALUE).
 *   q, k, v    [T, H, 128] bf16, written (rounded to nearest even)
 *   cu_seqlens [N + 1] int32 device array as for kda_prefill_chunked
 *   d          must be 128; q_scale finite; eps >= 0 (the pages' 1e-6)
 * Returns KDA_OK or a kda_status_t.
 */
int kda_conv_prologue(const void *xq, const void *xk, const void *xv, const float *conv_w,
                      const void *conv_in, void *conv_out, void *q, void *k, void *v,
                      const int32_t *cu_seqlens, int N, int64_t T, int H, int d,
                      float q_scale, float eps, void *stream);

/*
 * kda_prefill_chunked with the layer's gated RMSNorm applied to o: writes
 * out = o / sqrt(mean_j o_j^2 + eps) * norm_w_j * sigmoid(gate_j) per
 * (token, head) instead of o.  On the tensor-core path (bf16, chunk 64) the
 * norm runs inside the inter-chunk state pass on each chunk of o before it
 * is stored; other configurations run the CUDA-core prefill into `out`, then
 * the norm in place.
 *
 *   gate     [T, H, 128] bf16 gate projection (before its sigmoid)
 *   norm_w   [128] fp32 RMSNorm weight, shared by the heads
 *   eps      >= 0
 *   out      [T, H, 128] fp32, written
 *   every other argument as for kda_prefill_chunked (S_out gets the final
 *   states, unchanged by the norm)
 * Returns KDA_OK or a kda_status_t.
 */
int kda_prefill_chunked_gated(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, const float *S0, const void *gate,
                              const float *norm_w, float eps, float *out, float *S_out,
                              const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                              int chunk, int dtype, void *stream);

/*
 * The whole layer's prefill in one call ("Colibri Kimi K3 Metal backend",
 * sections 8.3 and 8.4: the conv + L2-norm prologue feeds the recurrence, the
 * gated RMSNorm follows it): kda_conv_prologue followed by
 * kda_prefill_chunked_gated on the tensor-core path, with q, k, v kept in the
 * call's workspace, so a caller needs no buffers for them.  The results are
 * those two calls' bit for bit.
 *
 *   xq, xk, xv [T, H, 128] bf16 raw projections
 *   conv_w     [3, H, 128, 4] fp32 taps
 *   conv_in    [N, 3, 3, H, 128] bf16 windows before each sequence, or NULL
 *   conv_out   [N, 3, 3, H, 128] bf16, written, or NULL; not conv_in
 *   g, beta, S0, S_out, cu_seqlens   as for kda_prefill_chunked
 *   gate       [T, H, 128] bf16; norm_w [128] fp32
 *   out        [T, H, 128] fp32, written: the gated RMSNorm of o
 *   q_scale    finite; l2_eps, norm_eps >= 0
 *   dk, dv     must be 128
 * The workspace (q, k, v in bf16, 768 bytes per token-head, and the records
 * of kda_prefill_chunked) comes from the library's pool (KDA_ERR_WORKSPACE if
 * it cannot grow).  Returns KDA_OK or a kda_status_t.
 */
int kda_layer_prefill(const void *xq, const void *xk, const void *xv, const float *conv_w,
                      const void *conv_in, void *conv_out, const float *g, const float *beta,
                      const float *S0, const void *gate, const float *norm_w, float q_scale,
                      float l2_eps, float norm_eps, float *out, float *S_out,
                      const int32_t *cu_seqlens, int N, int64_t T, int H, int dk, int dv,
                      void *stream);

/*
 * One token of the whole layer for each of B sequences on slot-indexed
 * pools, in one kernel: conv1d + SiLU + L2 norm of the raw projections (the
 * window of pool row state_indices[b] is read and shifted in place), the
 * state step of kda_decode_step_pool (its q, k, v kept in fp32, not rounded
 * to bf16), and the gated RMSNorm of o.
 *
 *   xq, xk, xv    [B, H, 128] bf16 raw projections of the token
 *   conv_w        [3, H, 128, 4] fp32 taps
 *   conv_pool     [P, 3, 3, H, 128] bf16 windows, read and updated in place
 *   g, beta       [B, H, 128] / [B, H] fp32 as for kda_decode_step
 *   gate          [B, H, 128] bf16; norm_w [128] fp32
 *   S_pool        [P, H, 128, 128] fp32 (state_dtype KDA_F32) or bf16
 *                 (KDA_BF16), updated in place
 *   state_indices [B] int32 device array of pool rows, or NULL (rows 0..B-1;
 *                 then P >= B).  Negative = padding: out row zero, neither
 *                 pool touched.  Entries must be distinct; an entry >= P is
 *                 skipped like padding and sets bit 1 of the device error
 *                 word.
 *   out           [B, H, 128] fp32, written
 *   q_scale       finite; l2_eps, norm_eps >= 0
 * Returns KDA_OK or a kda_status_t; B = 0 is a no-op.
 */
int kda_decode_layer_step(const void *xq, const void *xk, const void *xv, const float *conv_w,
                          void *conv_pool, const float *g, const float *beta, const void *gate,
                          const float *norm_w, void *S_pool, int state_dtype,
                          const int32_t *state_indices, int P, float *out, int B, int H,
                          int dk, int dv, float q_scale, float l2_eps, float norm_eps,
                          void *stream);

/*
 * Gives back the memory that the library's workspace pool on the current
 * device keeps between kda_prefill_chunked / _events / _gated /
 * kda_layer_prefill calls (one 60,416-byte record per (chunk, head) of the
 * largest call so far: about 6 GB after a 66,048-token, 96-head batch).
 * Memory still held by a call in flight is kept: synchronise the streams
 * those calls ran on first.  The next call grows the pool again (a driver
 * allocation).  Host-only bookkeeping plus cudaMemPoolTrimTo; returns KDA_OK
 * (also when the device has no pool yet) or KDA_ERR_CUDA.
 */
int kda_workspace_release(void);

/*
 * Device-side error word of the library.  The outputs of a call that raised
 * a bit are invalid.
 *   Bit 0: the tensor-core prefill kernels never wait without bound: if one
 *          of their waits on an asynchronous copy or on the tensor cores
 *          runs past its iteration limit they set this bit, release their
 *          tensor memory and exit.  Also set when cu_seqlens breaks its
 *          precondition (an entry below 0 or above T, or a decrease), by
 *          the prefill paths and the conv prologue, which then touch no
 *          memory outside their buffers.
 *   Bit 1: a kda_decode_step_pool or kda_decode_layer_step slot index was
 *          past the end of the pool.
 *   Bit 2: the tensor-core prefill saw a gate g outside [-5, 0] or a NaN
 *          (its decay folding is sized for the model's gate bound).
 *   Bit 3: debug builds only (libkda_gb300_debug.so, built with
 *          python -m kda_linear_attention_gb300.build --debug and loaded by
 *          the Python binding when KDA_GB300_DEBUG=1): an index check on a
 *          kernel's global-memory addressing failed; the access was kept
 *          inside its buffer.
 *   Bit 4: the tensor-core prefill's intermediate u = beta (v - ...) (the
 *          delta-rule correction of each token, carried into its second
 *          state-pass product in fp16) reached 65504 in magnitude or NaN:
 *          v far outside a model's activation range.
 *
 *   code   host pointer, receives the word (0 = no error since the last reset)
 *   reset  nonzero: clear the word after reading it
 * Synchronous with respect to the device (a cudaMemcpyFromSymbol).  Returns
 * KDA_OK, KDA_ERR_NULL or KDA_ERR_CUDA.
 */
int kda_device_error(unsigned int *code, int reset);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
