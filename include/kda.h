/*
 * kda.h -- C ABI of libkda: the Kimi Delta Attention (KDA) state recurrence
 * on one GB300 GPU (sm_103a).
 *
 * The recurrence (GLM-5.3-Flash Architecture Mastery, course index, "Course
 * Outcomes": the closed form (I - beta k k^T) D S + beta k v^T; Lecture 11,
 * section 2, KDA row: the operator order is (I - beta k k^T) D, not
 * D (I - beta k k^T)):
 *
 *     S_t = (I - beta_t k_t k_t^T) D_t S_{t-1} + beta_t k_t v_t^T,
 *     o_t = S_t^T q_t,             D_t = diag(exp(g_t)),
 *
 * per (sequence, head), with S a d_k x d_v fp32 matrix.  Lecture 04,
 * section 2 asks for two kernel families, selected by request phase: a
 * chunked prefill kernel (kda_prefill_chunked) and a fused recurrent decode
 * step (kda_decode_step).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers, contiguous, row-major, and
 *     16-byte aligned; anything else returns KDA_ERR_INVALID_ARG.
 *   - The caller owns every buffer.  The library allocates no device memory
 *     and keeps no global state; prefill scratch comes from the caller
 *     through `workspace` (size from kda_prefill_workspace_size).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  No call synchronises.
 *   - Argument errors are returned before anything is launched; a failed
 *     launch returns KDA_ERR_CUDA.  No exception crosses this boundary.
 *   - Results are deterministic: the same inputs give the same bits, and a
 *     document inside a packed batch gives the same bits as that document
 *     run alone.
 *   - Supported sizes: d_k == d_v in {16, 64, 128}; chunk_size in
 *     {16, 32, 64} (0 selects 64).  bf16 inputs with d = 128 and chunk 64
 *     take the tensor-core (tcgen05) prefill; every other combination takes
 *     the fp32 CUDA-core prefill.
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

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, negative size, bad cu_seqlens, small workspace */
    KDA_ERR_UNSUPPORTED = 2, /* a size or dtype outside the supported set */
    KDA_ERR_CUDA = 3,        /* a CUDA launch or driver call failed */
    KDA_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (reported by kda_prefill_check) */
    KDA_ERR_BOUNDS = 5       /* debug build only: a checked index was out of bounds (kda_prefill_check) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Human-readable name of a status code (static storage, never NULL). */
KDA_API const char *kda_status_string(kda_status status);

/*
 * Bytes of device scratch that kda_prefill_chunked needs for these sizes
 * (0 when the sizes are invalid).  The bound depends only on the arguments,
 * not on the document lengths inside cu_seqlens.
 */
KDA_API size_t kda_prefill_workspace_size(int32_t total_tokens, int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v,
                                  kda_dtype in_dtype, int32_t chunk_size);

/*
 * Chunked prefill over packed documents (Lecture 04, sections 1 and 2: each
 * chunk of L tokens reduces to one affine update in structured
 * diagonal-plus-rank-one form -- a triangular (WY/UT) solve plus dense
 * intra-chunk q k^T, k k^T and k S contractions -- and the chunk updates are
 * then composed in order).
 *
 *   q, k       [total_tokens, H, d_k]  in_dtype
 *   v          [total_tokens, H, d_v]  in_dtype
 *   g          [total_tokens, H, d_k]  fp32 natural-log decay (D_t = diag(exp(g_t)))
 *   beta       [total_tokens, H]       fp32 write strength
 *   cu_seqlens [num_seqs + 1]          int32, device; cu[0] = 0, non-decreasing,
 *                                      cu[num_seqs] = total_tokens.  The state
 *                                      restarts at every document start
 *                                      (Lecture 11, section 2, packing row).
 *   S0         [num_seqs, H, d_k, d_v] fp32 initial state, or NULL for zeros
 *   o          [total_tokens, H, d_v]  in_dtype output, o_t = S_t^T q_t
 *   S_final    [num_seqs, H, d_k, d_v] fp32 state after each document, or NULL.
 *              S_final may alias S0 (in-place continuation); o must not alias
 *              any input.
 *   workspace  device scratch of at least kda_prefill_workspace_size(...) bytes,
 *              256-byte aligned; its contents on entry do not matter.
 *
 * cu_seqlens is read on the device only.  If it is not monotone or does not
 * end at total_tokens, the kernels write nothing to o or S_final (the call
 * itself has already returned KDA_OK; kda_prefill_check reports it).
 */
KDA_API kda_status kda_prefill_chunked(const void *q, const void *k, const void *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t H,
                               int32_t d_k, int32_t d_v, kda_dtype in_dtype, int32_t chunk_size, const float *S0,
                               void *o, float *S_final, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Profiling variant: does exactly what kda_prefill_chunked does and, in
 * addition, records CUDA events on `stream` around its kernels.  events[i]
 * (a cudaEvent_t passed as void*, or NULL to skip it) is recorded just
 * before kernel i, and events[n] just after the last kernel; n is written to
 * *num_kernels and never exceeds KDA_PREFILL_MAX_KERNELS, so `events` must
 * hold KDA_PREFILL_MAX_KERNELS + 1 entries.  kernel_names, if not NULL,
 * receives n static strings naming the kernels in launch order.
 */
#define KDA_PREFILL_MAX_KERNELS 4
KDA_API kda_status kda_prefill_chunked_profiled(const void *q, const void *k, const void *v, const float *g,
                                        const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                        int32_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                        kda_dtype in_dtype, int32_t chunk_size, const float *S0, void *o,
                                        float *S_final, void *workspace, size_t workspace_bytes, void *stream,
                                        void *const *events, int32_t *num_kernels, const char **kernel_names);

/*
 * Reports how the last kda_prefill_chunked call that used this workspace
 * ended on the device.  It copies one status word back and SYNCHRONISES
 * `stream` (the stream the call was enqueued on).  Returns
 *   KDA_OK               the call completed;
 *   KDA_ERR_INVALID_ARG  cu_seqlens was not valid: o and S_final were left
 *                        unwritten;
 *   KDA_ERR_TIMEOUT      a bounded wait inside a kernel gave up (a CTA of a
 *                        cooperative launch, or an asynchronous copy, never
 *                        arrived within its time bound of one to two
 *                        seconds): o and S_final may be partly written.  The
 *                        context stays usable and the next call starts afresh;
 *   KDA_ERR_BOUNDS       (the debug build, libkda_debug.so, only) a checked
 *                        index was out of bounds; the access was skipped and
 *                        the source line of the first failing check is the
 *                        workspace's second int32 word;
 *   KDA_ERR_CUDA         the copy or the synchronisation failed.
 */
KDA_API kda_status kda_prefill_check(const void *workspace, void *stream);

/*
 * One fused recurrent decode step for num_seqs independent sequences
 * (Lecture 04, section 2: one new token per sequence, the state already in
 * memory, one fused step):
 *
 *   q, k     [num_seqs, H, d_k] in_dtype     v [num_seqs, H, d_v] in_dtype
 *   g        [num_seqs, H, d_k] fp32         beta [num_seqs, H] fp32
 *   S_inout  [num_seqs, H, d_k, d_v] fp32, read and overwritten with S_t
 *   o        [num_seqs, H, d_v] in_dtype, o_t = S_t^T q_t
 */
KDA_API kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                           float *S_inout, void *o, void *stream);

/*
 * The steps on either side of the recurrence, fused into its kernels
 * (Lecture 04, section 3: the sublayer runs Q/K normalisation before the
 * recurrence and a gated normalisation on its output; fusing them saves a
 * round trip of q, k and o through memory).  The pages name the two steps
 * without formulas; libkda computes, per (token, head):
 *   qk_l2norm != 0:  q <- q / sqrt(sum_c q_c^2 + qk_eps), and the same for k,
 *                    in fp32 from the input values;
 *   out_gate != NULL: o <- o / sqrt(mean_c o_c^2 + out_eps) * w_c * sigmoid(z_c),
 *                    with z = out_gate [T, H, d_v] in_dtype and w = out_weight
 *                    [d_v] fp32 (NULL: all ones); the stored o is this value.
 * All pointers are device pointers with the alignment rules of the entry
 * points (out_gate and out_weight 16-byte aligned).
 */
typedef struct {
    int32_t qk_l2norm;
    float qk_eps;            /* >= 0 */
    const void *out_gate;    /* NULL: o is the recurrence output as it is */
    const float *out_weight; /* NULL: ones */
    float out_eps;           /* > 0 when out_gate is given */
} kda_fusion_opts;

/* kda_prefill_chunked with the fused prologue and epilogue above (opts NULL: exactly kda_prefill_chunked). */
KDA_API kda_status kda_prefill_chunked_ex(const void *q, const void *k, const void *v, const float *g,
                                          const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                          int32_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                          kda_dtype in_dtype, int32_t chunk_size, const float *S0, void *o,
                                          float *S_final, void *workspace, size_t workspace_bytes, void *stream,
                                          const kda_fusion_opts *opts);

/* kda_decode_step with the fused prologue and epilogue above (out_gate is [num_seqs, H, d_v]). */
KDA_API kda_status kda_decode_step_ex(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                      int32_t num_seqs, int32_t H, int32_t d_k, int32_t d_v, kda_dtype in_dtype,
                                      float *S_inout, void *o, void *stream, const kda_fusion_opts *opts);

/*
 * Decode step for a batch that mixes request phases (Lecture 04, section 2:
 * the fused recurrent kernel serves the sequences that are generating, while
 * others are still in their chunked prefill).  The states live in a pool of
 * num_slots slots; the i-th active sequence's token updates slot
 * seq_idx[i].  Slots that are not listed are not touched.
 *
 *   q, k       [num_active, H, d_k] in_dtype   v [num_active, H, d_v] in_dtype
 *   g          [num_active, H, d_k] fp32       beta [num_active, H] fp32
 *   seq_idx    [num_active] int32, device: distinct slots in [0, num_slots)
 *              (listing a slot twice makes the two updates race)
 *   S_pool     [num_slots, H, d_k, d_v] fp32, the listed slots read and
 *              overwritten with S_t
 *   o          [num_active, H, d_v] in_dtype, o_t = S_t^T q_t
 *   status     optional device int32 (NULL to skip), 4-byte aligned: a slot
 *              outside [0, num_slots) is skipped (its state and o rows are not
 *              written) and sets *status to KDA_ERR_INVALID_ARG if it was 0.
 */
KDA_API kda_status kda_decode_step_indexed(const void *q, const void *k, const void *v, const float *g,
                                           const float *beta, const int32_t *seq_idx, int32_t num_active,
                                           int32_t num_slots, int32_t H, int32_t d_k, int32_t d_v,
                                           kda_dtype in_dtype, float *S_pool, void *o, int32_t *status,
                                           void *stream);

/*
 * State snapshot and restore for rollback (Lecture 11, section 2, "Serving
 * state" row: speculative rollback must reconcile the KDA state; section 3:
 * a run after rollback must equal a from-scratch run).  Each copies whole
 * slots (all H heads) bit for bit:
 *   kda_state_snapshot  S_saved[i] = S_pool[seq_idx[i]]   (i < n)
 *   kda_state_restore   S_pool[seq_idx[i]] = S_saved[i]
 * S_pool is [num_slots, H, d_k, d_v] fp32, S_saved [n, H, d_k, d_v] fp32, both
 * device and 16-byte aligned; seq_idx and status as for
 * kda_decode_step_indexed (a restore that lists a slot twice races).
 */
KDA_API kda_status kda_state_snapshot(const float *S_pool, const int32_t *seq_idx, int32_t n, int32_t num_slots,
                                      int32_t H, int32_t d_k, int32_t d_v, float *S_saved, int32_t *status,
                                      void *stream);
KDA_API kda_status kda_state_restore(const float *S_saved, const int32_t *seq_idx, int32_t n, int32_t num_slots,
                                     int32_t H, int32_t d_k, int32_t d_v, float *S_pool, int32_t *status,
                                     void *stream);

/*
 * Short causal convolution on the inputs of the recurrence (Lecture 04,
 * section 3: a small local mixing step on Q, K and/or V before the Q/K
 * normalisation; Lecture 11, section 2, "Serving state" row: the
 * convolution state must survive continuation and rollback like S does).
 * The pages give no formula; libkda computes, per channel c,
 *     y_t[c] = sum_{j < W} w[c, j] x_{t-j}[c]
 * inside each document, positions before a document's first token reading
 * its carried state.  fp32 arithmetic; 1 <= W <= KDA_SHORT_CONV_MAX_W.
 *
 *   x, y            [total_tokens, C] in_dtype (e.g. C = H * d for q laid out
 *                   [T, H, d]); y must not alias x
 *   w               [C, W] fp32
 *   cu_seqlens      [num_seqs + 1] int32, device, valid as for the prefill
 *                   (not checked here: an invalid table gives wrong values
 *                   but no out-of-bounds access)
 *   conv_state      [num_seqs, W - 1, C] fp32, each document's previous W - 1
 *                   inputs, oldest first, or NULL for zeros
 *   conv_state_out  [num_seqs, W - 1, C] fp32 or NULL: each document's last
 *                   W - 1 inputs (older carried entries when it is shorter);
 *                   must not alias conv_state
 * The decode step takes one token per sequence (x, y [N, C]) and rolls
 * conv_state [N, W - 1, C] in place.  All pointers are device pointers aligned
 * to their element size.
 */
#define KDA_SHORT_CONV_MAX_W 8
KDA_API kda_status kda_short_conv_prefill(const void *x, const float *w, const int32_t *cu_seqlens, int32_t num_seqs,
                                          int32_t total_tokens, int32_t C, int32_t W, kda_dtype in_dtype,
                                          const float *conv_state, void *y, float *conv_state_out, void *stream);
KDA_API kda_status kda_short_conv_decode(const void *x, const float *w, int32_t N, int32_t C, int32_t W,
                                         kda_dtype in_dtype, float *conv_state, void *y, void *stream);

/*
 * Chunked prefill that allocates nothing.  The course pages have no
 * counterpart to this entry point; it repackages kda_prefill_chunked for
 * callers that cannot give the library device scratch: code that runs while a
 * stream is being captured into a graph, serving loops whose device memory is
 * pooled up front and must never see a cudaMalloc (an allocation can also
 * synchronise the device), and plugins that are handed only their inputs and
 * outputs.
 *
 * Arguments and results are those of kda_prefill_chunked without the
 * workspace.  The scratch is a static device array of
 * KDA_NOALLOC_SCRATCH_BYTES inside the library; every GPU that loads the
 * library's device code holds it until the process exits.  Limit: a call
 * whose kda_prefill_workspace_size(...) exceeds KDA_NOALLOC_SCRATCH_BYTES
 * returns KDA_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - All calls on one device share the array: calls whose kernels overlap on
 *     the GPU (unordered streams) race and corrupt each other's results.
 *     Calls ordered on one stream are safe.  Nothing in the array needs to
 *     start at zero.
 *   - Their device-side status (invalid cu_seqlens, a wait that ran out) is
 *     read with kda_prefill_noalloc_check; invalid cu_seqlens leave o and
 *     S_final unwritten.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
/*
 * kda_prefill_check for the no-allocation entry point: reads the status word
 * of the static scratch on the current device and SYNCHRONISES `stream`.  The
 * word describes the last kda_prefill_chunked_noalloc call on this device and
 * is valid until the next such call.  Same return values as
 * kda_prefill_check.
 */
KDA_API kda_status kda_prefill_noalloc_check(void *stream);
KDA_API kda_status kda_prefill_chunked_noalloc(const void *q, const void *k, const void *v, const float *g,
                                               const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                               int32_t total_tokens, int32_t H, int32_t d_k, int32_t d_v,
                                               kda_dtype in_dtype, int32_t chunk_size, const float *S0, void *o,
                                               float *S_final, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
