/*
 * kda.h -- C ABI of the Kimi Delta Attention (KDA) library for one GB300 GPU
 * (sm_103a).
 *
 * The layer.  Per head, a state S of shape dk x dv (fp32) is carried along the
 * sequence.  Token t with query q_t, key k_t (dk), value v_t (dv), per-channel
 * log-decay log_alpha_t (dk) and write strength beta_t does
 *
 *     alpha_t = exp(clamp(log_alpha_t, -5, 0))                 (per key channel)
 *     S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t     = S_t^T q_t                                        (updated state)
 *
 * Sources: lecture "Inside Kimi K3: Architecture of an Open Frontier Model",
 * sequence paragraph (a fixed-size state rewritten by every token: diagonal
 * forget gate first, then the beta-weighted k v correction; log-decay bounded
 * below at -5); meridianbulletin.com article on Kimi K3, section "Handling One
 * Million Tokens with a Fixed-Size State Matrix" (alpha kept in [e^-5, 1]).
 * No 1/sqrt(dk) scale, output gate or normalisation is applied: a caller that
 * wants one scales q or post-processes out.
 *
 * Conventions common to every entry point
 * ----------------------------------------
 * - All tensor pointers are DEVICE pointers of the current CUDA device, dense
 *   row-major (innermost index last, no padding) and 16-byte aligned.
 * - bf16 tensors are IEEE bfloat16; f32 tensors are IEEE binary32.
 * - Supported head sizes: dk == dv, and dk in {64, 128}.  Anything else
 *   returns KDA_ERR_UNSUPPORTED.  The prefill entry points also take at most
 *   65535 heads (n_heads); more return KDA_ERR_UNSUPPORTED.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call is asynchronous with respect to the host and ordered
 *   on `stream`; calls on different streams may run concurrently.  The device
 *   entry points never synchronise the host and allocate only stream-ordered,
 *   so they can be captured into a CUDA graph (make one uncaptured call per
 *   device first: it creates the library's per-device state).
 * - The caller owns every buffer.  The library keeps no caller pointer after
 *   a call returns.  Inputs are never written.
 * - Errors found on the host (null pointer, bad size, misalignment,
 *   unsupported shape) are returned synchronously before anything is launched;
 *   outputs are then untouched and kda_last_error_message() explains.
 *   A failed launch or allocation returns KDA_ERR_CUDA / KDA_ERR_OUT_OF_MEMORY.
 *   Errors only the GPU can see (a malformed cu_seqlens array) make the
 *   kernels skip their work and raise a device error word, which
 *   kda_get_device_error() reports.  No kernel traps or asserts.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 1

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARGUMENT = 1, /* null pointer, negative size, misaligned, ... */
    KDA_ERR_UNSUPPORTED = 2,      /* valid but not implemented (e.g. dk = 96)     */
    KDA_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed         */
    KDA_ERR_OUT_OF_MEMORY = 4,    /* the stream-ordered workspace allocation failed */
    KDA_ERR_DEVICE_INPUT = 5      /* the GPU rejected an input (bad cu_seqlens)   */
} kda_status;

/*
 * kda_chunk_fwd -- chunk-parallel prefill.
 *
 * Evaluates the recurrence above for every token of every sequence and head,
 * starting from S0, and writes every output o_t and each sequence's final
 * state.  Tokens of a 64-token chunk are processed together and only the
 * state is handed from chunk to chunk (meridianbulletin.com article, section
 * "Parallelizing Sequential State Updates"); the cumulative decay inside a
 * chunk is handled in 16-token tiles whose accumulated log-decay the clamp
 * keeps within [-80, 0] (orkas.ai close read, section "A lower bound that
 * deleted a GPU code path").  When there are too few (sequence, head) chains
 * to fill the GPU, long sequences are split into segments whose zero-start
 * state and transition are combined by a prefix scan (same section of the
 * meridianbulletin.com article; orkas.ai close read, section "The bill comes
 * due in the serving stack").  Results equal the token-by-token recurrence up
 * to floating-point rounding.
 *
 * Tensors (T = total_tokens, N = n_seqs, H = n_heads):
 *   q, k        bf16 [T, H, dk]       read
 *   v           bf16 [T, H, dv]       read
 *   log_alpha   f32  [T, H, dk]       read; clamped to [-5, 0] on load
 *   beta        f32  [T, H]           read; expected in [0, 1]
 *   S0          f32  [N, H, dk, dv]   read; NULL = zero initial state
 *   cu_seqlens  i32  [N + 1]          read; NULL = N sequences of equal length
 *                                     T / N (T must be divisible by N).
 *                                     Otherwise cu_seqlens[0] = 0,
 *                                     non-decreasing, cu_seqlens[N] = T;
 *                                     sequence n owns tokens
 *                                     cu_seqlens[n] .. cu_seqlens[n+1]-1.
 *                                     Empty sequences are allowed (their
 *                                     S_final is S0).  Checked on the GPU.
 *   out         bf16 [T, H, dv]       written (every row)
 *   S_final     f32  [N, H, dk, dv]   written; NULL = not produced.
 *                                     May alias S0 exactly (in-place
 *                                     continuation); no other overlap allowed.
 * A uniform batch [B, T_b, H, d] is passed as T = B * T_b, N = B,
 * cu_seqlens = NULL.  T = 0 or N = 0 is a valid no-op (S_final = S0).
 *
 * Memory: a uniform batch (cu_seqlens = NULL) whose sequences are not split
 * allocates nothing and is one kernel launch.  Otherwise the call allocates a
 * temporary workspace stream-ordered on `stream` and frees it there: the
 * segment plan (40 bytes per segment) and, when sequences are split,
 * (N + T / segment) * H * dk * (2 dv + dk) * 4 bytes of segment summaries and
 * entry states, plus about (N + T / segment) * H * (segment / 64) * 32 KiB
 * (some 512 bytes per token and head) of T records, which the call leaves out
 * (recomputing T instead) when the pool cannot provide them.
 */
kda_status kda_chunk_fwd(const void *q, const void *k, const void *v,
                         const float *log_alpha, const float *beta,
                         const float *S0, const int32_t *cu_seqlens, void *out,
                         float *S_final, int64_t total_tokens, int32_t n_seqs,
                         int32_t n_heads, int32_t dk, int32_t dv, void *stream);

/*
 * Tensor descriptors: kda_chunk_fwd_t, kda_decode_step_t.
 *
 * The same two layer calls with each tensor passed as a descriptor: device
 * pointer, element type, rank, extents and strides (in elements).  The
 * library then checks on the host, before anything is launched, what the
 * pointer form must take on trust: every tensor's dtype (q, k, v, out bf16;
 * log_alpha, beta, S0, S_final, S_inout f32; cu_seqlens i32), its rank, that
 * its extents agree with q's (and v's for the value side), and that it is
 * dense row-major (stride of the last dimension 1, each other stride the
 * product of the extents after it; a dimension of extent 1 may have any
 * stride).  A wrong dtype, a shape mismatch or a non-dense layout returns
 * KDA_ERR_INVALID_ARGUMENT with kda_last_error_message() naming the tensor.
 * Every other rule (alignment, overlaps, supported head sizes, ownership,
 * streams, device-side errors) is the pointer form's; results are identical.
 *
 * kda_chunk_fwd_t: q is [T, H, dk] (packed; N = cu_seqlens' length - 1, or,
 * without cu_seqlens, S0's or S_final's leading extent, else 1) or
 * [B, T_b, H, dk] (a uniform batch of N = B sequences; cu_seqlens must then
 * be NULL).  k, log_alpha have q's shape; v and out q's shape with dv last;
 * beta q's shape without the last dimension; S0, S_final [N, H, dk, dv];
 * cu_seqlens [N + 1].  S0, cu_seqlens and S_final may be NULL descriptors.
 * kda_decode_step_t: q, k, log_alpha [N, H, dk]; v, out [N, H, dv]; beta
 * [N, H]; S_inout [N, H, dk, dv].
 * The descriptors are read during the call only.
 */
typedef enum { KDA_BF16 = 0, KDA_F32 = 1, KDA_I32 = 2 } kda_dtype;

typedef struct {
    void *data;         /* device pointer to element [0, 0, ...] */
    kda_dtype dtype;
    int32_t ndim;       /* 1 .. 4 */
    int64_t shape[4];   /* extents, outermost first */
    int64_t stride[4];  /* in elements */
} kda_tensor;

kda_status kda_chunk_fwd_t(const kda_tensor *q, const kda_tensor *k,
                           const kda_tensor *v, const kda_tensor *log_alpha,
                           const kda_tensor *beta, const kda_tensor *S0,
                           const kda_tensor *cu_seqlens, kda_tensor *out,
                           kda_tensor *S_final, void *stream);
kda_status kda_decode_step_t(const kda_tensor *q, const kda_tensor *k,
                             const kda_tensor *v, const kda_tensor *log_alpha,
                             const kda_tensor *beta, kda_tensor *S_inout,
                             kda_tensor *out, void *stream);

/*
 * kda_chunk_fwd_split -- kda_chunk_fwd with an explicit segment length.
 *
 * segment_tokens = 0 chooses automatically (what kda_chunk_fwd does).
 * segment_tokens > 0 must be a multiple of 64: every sequence longer than it
 * is cut into segments of that many tokens (the last may be shorter).  A
 * first launch computes the zero-start increment B and the transition M of
 * every segment but each sequence's last, the entry states S_in(j+1) =
 * M_j S_in(j) + B_j are scanned, and a second launch replays every segment
 * from its entry state.  In a uniform batch (cu_seqlens NULL) the first launch
 * replays segment 0 from S0 instead of summarising it (its exit state is
 * S_in(1)), so the second replays segments 1 .. last only.  The first launch
 * also keeps each summarised chunk's UT transform T (32 KiB per chunk and
 * head, in the call's workspace), and the second launch's replay of that
 * segment loads it instead of recomputing it, bit for bit the same; if the
 * workspace pool cannot hold those records, every replay computes its own.
 * segment_tokens < 0 disables splitting.  The result is the same up to
 * rounding; this is the scheduling knob behind the automatic choice.
 */
kda_status kda_chunk_fwd_split(const void *q, const void *k, const void *v,
                               const float *log_alpha, const float *beta,
                               const float *S0, const int32_t *cu_seqlens,
                               void *out, float *S_final, int64_t total_tokens,
                               int32_t n_seqs, int32_t n_heads, int32_t dk,
                               int32_t dv, int64_t segment_tokens, void *stream);

/*
 * kda_auto_segment_tokens -- the segment length segment_tokens = 0 chooses.
 *
 * Host only: touches no device.  sm_count is the device's multiprocessor
 * count (kda_chunk_fwd uses the current device's); uniform is 1 for a uniform
 * batch (cu_seqlens NULL), 0 for a packed one.  Returns a multiple of 64, or
 * -1 for no split.  The choice models each chunk kernel pass as waves of one
 * (segment, head) unit per SM, a unit of c chunks taking c chunk-times:
 * unsplit, ceil(N H / SMs) waves of the whole sequence.  Split at L chunks
 * into s segments per sequence (the last one of l = n - (s - 1) L chunks):
 *   - uniform batch: a first pass of ceil(N H (s - 1) / SMs) waves of L
 *     (replays of segment 0, summaries of segments 1 .. s - 2), and a second
 *     of as many waves of max(0.77 L, l) (replays of segments 1 .. s - 1:
 *     those that load their T records take 0.77 chunk-times per chunk, the
 *     last one computes its own; 0.77 L counts only when s > 2);
 *   - packed batch: ceil(N H (s - 1) / SMs) waves of L, then ceil(N H s / SMs)
 *     waves of L (summaries of segments 0 .. s - 2, then replays of every
 *     segment; the lengths, which only the device reads, may make any
 *     segment a full-length last one).
 * Plus the scan (one chunk-time per segment) and a fixed start of two
 * chunk-times per wave, with sequences taken as total_tokens / n_seqs tokens
 * (n chunks), segments of at least 4 chunks and at most 8 waves of replay
 * units.  It returns the length with the least modelled time, or -1 when no
 * split beats the unsplit pass (always when N H >= sm_count).  Invalid sizes
 * (any of them <= 0) return -1.
 */
int64_t kda_auto_segment_tokens(int64_t total_tokens, int32_t n_seqs, int32_t n_heads,
                                int32_t sm_count, int32_t uniform);

/*
 * kda_chunk_fwd_noalloc -- kda_chunk_fwd without any device allocation.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory during a call: runtimes that hand all
 * device memory to their own allocator at start-up, and callers that must
 * not touch a memory pool or take allocator locks in the middle of a step.
 * It computes the same result as kda_chunk_fwd (same arguments, layouts and
 * error rules) but keeps its working data -- the per-sequence schedule -- in
 * a fixed 256 KiB array inside the library's device memory, which every GPU
 * that loads the library holds until the process exits.  It never splits
 * long sequences across SMs, so with few (sequence, head) chains it can be
 * slower than kda_chunk_fwd.
 *
 * Limit: n_seqs <= 8184; larger batches return KDA_ERR_UNSUPPORTED (use
 * kda_chunk_fwd).  Every other argument is checked exactly as kda_chunk_fwd
 * checks it, with the same status codes.
 *
 * First call on a device: it sets up the library's per-device state -- the
 * SM count and the device addresses of the error word and of the fixed array
 * (cudaDeviceGetAttribute, cudaGetSymbolAddress), under a host mutex, with
 * that device current -- and nothing else: it creates no memory pool (only
 * the entry points that take a workspace do, on their own first use).  Make
 * that first call before any stream capture.  All calls share the one array:
 * calls that overlap on the GPU (different streams, or different host threads
 * without ordering) race and may produce wrong results; order them on one
 * stream.  Each call rebuilds the schedule it needs, so nothing carries over
 * from the previous call.
 */
kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                 const float *log_alpha, const float *beta,
                                 const float *S0, const int32_t *cu_seqlens,
                                 void *out, float *S_final, int64_t total_tokens,
                                 int32_t n_seqs, int32_t n_heads, int32_t dk,
                                 int32_t dv, void *stream);

/*
 * kda_decode_step -- one recurrent step for a batch of N sequences.
 *
 * Per (sequence n, head h): S' = Diag(alpha) S; a = S'^T k; b = S'^T q;
 * u = beta (v - a); S = S' + k u^T (written back IN PLACE); o = S^T q
 * = b + (q . k) u.  The cost per token is constant: one pass over the state
 * (lecture "Inside Kimi K3...", sequence paragraph; orkas.ai close read,
 * section "The bill comes due in the serving stack": the state is updated in
 * place, so a step cannot be undone -- keep a copy to roll back).
 *
 * Tensors:
 *   q, k       bf16 [N, H, dk]        read
 *   v          bf16 [N, H, dv]        read
 *   log_alpha  f32  [N, H, dk]        read; clamped to [-5, 0]
 *   beta       f32  [N, H]            read
 *   S_inout    f32  [N, H, dk, dv]    read and overwritten with the new state
 *   out        bf16 [N, H, dv]        written
 * out must not overlap any other argument.  N = 0 is a no-op.
 * Allocates nothing.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           float *S_inout, void *out, int32_t n_seqs,
                           int32_t n_heads, int32_t dk, int32_t dv,
                           void *stream);

/*
 * kda_chunk_fwd_host -- kda_chunk_fwd for a uniform batch whose tensors are
 * in HOST memory (pinned memory makes the copies asynchronous).
 *
 * Nothing on the pages; it serves callers whose inputs and outputs live on
 * the host.  The batch is processed in time slices of `slice_tokens` tokens
 * per sequence (0 = 512; otherwise a multiple of 64).  Internal streams
 * overlap three things: the host-to-device copy of slice i+1, the prefill
 * of slice i, and the device-to-host copy of slice i-1.  The state stays
 * on the device and carries from slice to slice (the in-place continuation
 * of kda_chunk_fwd), so the results equal one kda_chunk_fwd call on the whole
 * batch up to rounding.
 *
 *   q, k, v, log_alpha, beta, out   HOST pointers, layouts of kda_chunk_fwd
 *                                   with cu_seqlens = NULL (N sequences of
 *                                   total_tokens / N tokens each)
 *   S0, S_final                     HOST pointers or NULL, as kda_chunk_fwd
 * The call is ordered on `stream` like every entry point and returns before
 * the work is done: the host buffers must stay valid, and out / S_final must
 * not be read, until `stream` has been synchronised.  Device staging (two
 * slices of inputs and outputs, plus the state) is allocated stream-ordered
 * on `stream` and released at the end.
 */
kda_status kda_chunk_fwd_host(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const float *S0, void *out, float *S_final,
                              int64_t total_tokens, int32_t n_seqs,
                              int32_t n_heads, int32_t dk, int32_t dv,
                              int64_t slice_tokens, void *stream);

/*
 * kda_chunk_fwd_checkpoints -- kda_chunk_fwd that also emits the state at
 * regular token boundaries of every sequence, for a prefix cache.
 *
 * A fixed-size state at a token boundary is all a later call needs to
 * continue from that prefix (orkas.ai close read, section "The bill comes
 * due in the serving stack": to reuse a prefix, the recurrent state is
 * checkpointed at a sparse subset of the token boundaries the cache hashes,
 * e.g. every 1024 tokens when it hashes every 512).  For sequence n of length len_n and
 * each j = 1 .. floor(len_n / interval), the state after the sequence's first
 * j * interval tokens is written, f32 [dk][dv] per head (the layout of
 * S_final), to
 *     checkpoints[c_n + j - 1, h],   c_n = sum over m < n of floor(len_m / interval),
 * so the checkpoints are packed sequence by sequence in token order.  A
 * sequence whose length is a multiple of interval gets its final state as
 * its last checkpoint too.
 *
 *   interval        > 0, a multiple of 64
 *   checkpoints     f32 [max_checkpoints, H, dk, dv], written; must not
 *                   overlap any other argument (may be NULL if
 *                   max_checkpoints = 0)
 *   max_checkpoints >= 0.  If the sequences have more checkpoints, the
 *                   excess is dropped and kda_get_device_error reports
 *                   KDA_ERR_DEVICE_INPUT; out and S_final are still written.
 * Everything else as kda_chunk_fwd (including the automatic split of long
 * sequences: checkpoints come from the replay, which starts every segment
 * from its exact entry state).
 */
kda_status kda_chunk_fwd_checkpoints(const void *q, const void *k, const void *v,
                                     const float *log_alpha, const float *beta,
                                     const float *S0, const int32_t *cu_seqlens,
                                     void *out, float *S_final,
                                     int64_t total_tokens, int32_t n_seqs,
                                     int32_t n_heads, int32_t dk, int32_t dv,
                                     int64_t interval, float *checkpoints,
                                     int64_t max_checkpoints, void *stream);

/*
 * kda_decode_tokens -- several tokens per sequence in one call, with a commit
 * count: the form speculative decoding needs.
 *
 * For each sequence n, the n_tokens tokens t = 0 .. n_tokens-1 are applied in
 * order starting from S_inout[n], exactly as n_tokens kda_decode_step calls
 * would.  out receives every token's output.  S_inout[n] is then overwritten
 * with the state after the first commit[n] tokens only: commit[n] = 0 leaves
 * it untouched, commit = NULL commits all n_tokens.  The state is updated in
 * place and cannot be rolled back (orkas.ai close read, section "The bill
 * comes due in the serving stack"). So a draft of k tokens is verified with
 * a call that commits nothing. A second call over the same cached inputs
 * then commits the accepted prefix: the state is rebuilt from the inputs,
 * not undone.  The state is read once and written at most once per call, so
 * a call costs about one decode step of memory traffic for all its tokens.
 *
 * Tensors (N = n_seqs, K = n_tokens; token t of sequence n is row n*K + t):
 *   q, k        bf16 [N*K, H, dk]   read
 *   v           bf16 [N*K, H, dv]   read
 *   log_alpha   f32  [N*K, H, dk]   read; clamped to [-5, 0]
 *   beta        f32  [N*K, H]       read
 *   S_inout     f32  [N, H, dk, dv] read; written as described
 *   out         bf16 [N*K, H, dv]   written
 *   commit      i32  [N] on the device, each in [0, K], or NULL.  A value
 *               outside [0, K] is reported through kda_get_device_error
 *               (KDA_ERR_DEVICE_INPUT); that sequence's out and state are
 *               then left unwritten.
 * n_tokens >= 1; n_tokens = 1 with commit = NULL is kda_decode_step.  Other
 * rules as kda_decode_step (commit must not overlap S_inout or out).
 * Allocates nothing.
 */
kda_status kda_decode_tokens(const void *q, const void *k, const void *v,
                             const float *log_alpha, const float *beta,
                             float *S_inout, void *out, const int32_t *commit,
                             int32_t n_seqs, int32_t n_tokens, int32_t n_heads,
                             int32_t dk, int32_t dv, void *stream);

/*
 * kda_chunk_fwd_fused, kda_decode_step_fused, kda_decode_tokens_fused -- the
 * same layer with the input
 * preparation done on load, so a caller passes projections straight through.
 *
 * The pages bound the forget gate's log-decay below at -5 by changing the
 * decay curve itself (lecture "Inside Kimi K3: Architecture of an Open
 * Frontier Model", sequence paragraph; orkas.ai close read, section "A lower
 * bound that deleted a GPU code path": the activation is bounded below).
 * These entry points take that curve's input, a gate logit x per key
 * channel, and form log alpha = -5 * sigmoid(x) = -5 / (1 + e^-x) in fp32,
 * then apply the same clamp to [-5, 0].  q and k arrive unnormalised; each
 * (token, head) vector is scaled to unit L2 norm over its dk channels,
 * x / max(||x||_2, 1e-12), in fp32 and rounded to bf16 (nearest even) before
 * use -- the same values a caller would pass to kda_chunk_fwd /
 * kda_decode_step after normalising itself.
 *
 * Arguments, layouts, ownership and errors are those of kda_chunk_fwd
 * (respectively kda_decode_step, kda_decode_tokens), except:
 *   q_raw, k_raw  bf16 [T, H, dk]   (decode: [N, H, dk])  unnormalised
 *   gate          bf16 [T, H, dk]   (decode: [N, H, dk])  logits, in place of
 *                                   log_alpha
 * Prefill reads 2 * dk fewer bytes per token and head than kda_chunk_fwd
 * (bf16 gate instead of f32 log_alpha).
 */
kda_status kda_chunk_fwd_fused(const void *q_raw, const void *k_raw, const void *v,
                               const void *gate, const float *beta,
                               const float *S0, const int32_t *cu_seqlens,
                               void *out, float *S_final, int64_t total_tokens,
                               int32_t n_seqs, int32_t n_heads, int32_t dk,
                               int32_t dv, void *stream);
kda_status kda_decode_tokens_fused(const void *q_raw, const void *k_raw, const void *v,
                                   const void *gate, const float *beta,
                                   float *S_inout, void *out, const int32_t *commit,
                                   int32_t n_seqs, int32_t n_tokens, int32_t n_heads,
                                   int32_t dk, int32_t dv, void *stream);
kda_status kda_decode_step_fused(const void *q_raw, const void *k_raw, const void *v,
                                 const void *gate, const float *beta,
                                 float *S_inout, void *out, int32_t n_seqs,
                                 int32_t n_heads, int32_t dk, int32_t dv,
                                 void *stream);

/*
 * kda_get_device_error -- synchronise `stream`, then return and clear the
 * device error word of the current device: KDA_OK, or KDA_ERR_DEVICE_INPUT
 * when a kernel rejected an input (kda_last_error_message() names it), or
 * KDA_ERR_CUDA when the synchronisation itself failed.
 */
kda_status kda_get_device_error(void *stream);

/*
 * kda_debug_chunk_dump -- kda_chunk_fwd (never split) that also writes the
 * intermediates of one 64-token chunk: sequence `seq`, head `head`, chunk
 * `chunk` (0-based within the sequence).  A debugging aid: the chunked form
 * of the recurrence goes through these steps, and comparing each with an
 * independent evaluation locates a wrong one.  Tokens of a chunk are
 * processed together and only the state is handed on (meridianbulletin.com
 * article, section "Parallelizing Sequential State Updates").
 *
 *   dump  f32 device buffer of 45056 floats, written:
 *         [0, 8192)        g      [64 tokens][128 key channels]: the
 *                                 chunk-local cumulative clamped log-decay
 *         [8192, 12288)    A_kk   [64][64]: beta_r sum_c k_rc k_ic e^{g_rc - g_ic}, i < r
 *         [12288, 16384)   A_qk   [64][64]: sum_c q_rc k_ic e^{g_rc - g_ic}, i <= r
 *         [16384, 20480)   T      [64][64]: (I + A_kk)^{-1} Diag(beta), as
 *                                 the tensor core reads it (tf32)
 *         [20480, 28672)   U      [64 tokens][128 value channels]:
 *                                 T (V - (k e^g) S), before its tf32 rounding
 *         [28672, 45056)   S      [128][128] (row = key channel): the state
 *                                 at the chunk's start
 *   Rows of tokens past the sequence's end hold the kernel's identity rows.
 *   d = 64 runs zero-padded: channels 64..127 are zero.  Every other argument,
 *   and out and S_final, as kda_chunk_fwd.  Slower than kda_chunk_fwd (extra
 *   barriers in the dumping unit).  The dump must not overlap any other
 *   argument; a chunk past the sequence's end leaves it unwritten.
 */
kda_status kda_debug_chunk_dump(const void *q, const void *k, const void *v,
                                const float *log_alpha, const float *beta,
                                const float *S0, const int32_t *cu_seqlens,
                                void *out, float *S_final, int64_t total_tokens,
                                int32_t n_seqs, int32_t n_heads, int32_t dk,
                                int32_t dv, int32_t seq, int32_t head,
                                int64_t chunk, float *dump, void *stream);

/*
 * kda_workspace_pool_bytes -- memory accounting: the bytes the library's
 * workspace pool currently reserves on the current device, or -1 when the
 * library has created no pool there.  The pool is created by the first call
 * that needs a workspace (kda_chunk_fwd on a packed batch, a split or
 * checkpoints); it keeps freed workspace cached for the next call.
 */
int64_t kda_workspace_pool_bytes(void);

/* Static description of a status code. */
const char *kda_status_string(kda_status status);

/* Detail of the last failure on the calling host thread ("" if none). */
const char *kda_last_error_message(void);

/* KDA_ABI_VERSION of the compiled library. */
int kda_abi_version(void);

/*
 * kda_selftest_bounded_wait -- launch, on `stream`, one wait of the kind every
 * kernel of the library makes on its own asynchronous copies and tensor-core
 * work, on an mbarrier that nothing ever arrives on.  The wait gives up after
 * `polls` polls (each blocks for a hardware-chosen interval, so 1000 polls end
 * within milliseconds) and records a timeout in the device error word, which
 * the next kda_get_device_error(stream) returns as KDA_ERR_DEVICE_INPUT with
 * a message naming the timeout.  Shows that a kernel whose work never arrives
 * reports it instead of hanging, and that the context stays usable.
 * polls in [1, 2^20], else KDA_ERR_INVALID_ARGUMENT.
 */
kda_status kda_selftest_bounded_wait(uint32_t polls, void *stream);

/*
 * The bounds-checked build.  Compiled with -DKDA_BOUNDS_CHECK (the binding's
 * build(checked=True) makes _build/checked/libkda.so), every plain
 * global-memory load and store of the kernels first checks that its elements
 * lie inside the buffer they index (extents from the call's sizes); an access
 * outside is skipped and recorded in the device error word, which the next
 * kda_get_device_error returns as KDA_ERR_DEVICE_INPUT naming the violation.
 * No kernel traps.  TMA copies are bounded by their tensor maps in both builds.
 *
 * kda_bounds_checked -- 1 in the bounds-checked build, 0 otherwise (host only).
 * kda_selftest_bounds_check -- launch, on `stream`, one guard on an index
 * outside a one-element buffer, with no memory access: afterwards
 * kda_get_device_error reports the violation in the bounds-checked build and
 * KDA_OK in the normal one.
 */
int kda_bounds_checked(void);
kda_status kda_selftest_bounds_check(void *stream);

/*
 * Launch timing (tracing aid).  While enabled, every kernel the library
 * launches is bracketed by CUDA events on its launch stream.
 * kda_profile_read() synchronises the device, then reports per kernel name
 * the launch count and the summed event time in milliseconds, and clears the
 * record.  Returns the number of entries written (at most max_entries).
 * Disabled by default; enabling costs two event records per launch.
 */
typedef struct {
    char name[48];
    int64_t launches;
    double total_ms;
} kda_kernel_time;

void kda_profile_enable(int enable);
int kda_profile_read(kda_kernel_time *entries, int max_entries);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
