/*
 * dsa_indexer.h -- C ABI of the GB300 (sm_103a) DSA lightning-indexer forward.
 *
 * The operation follows the DeepSeek-V4 SBHD indexer interface documented on
 * the NeMo AutoModel page
 * "nemo_automodel.components.models.deepseek_v4.kernels.tilelang_indexer":
 *   - `V4IndexerFunction` / `v4_lighting_indexer(index_q, index_k, weights,
 *     compress_ratio, topk, topk_indices=None)`: inputs in SBHD layout,
 *     q [seqlen, batch, heads, dim] bf16, k [seqlen_kv, batch, dim] bf16,
 *     weights [seqlen, batch, heads] fp32, `compress_ratio` (4 on C4
 *     layers), `topk`, optional pre-computed `topk_indices [batch, seqlen,
 *     topk] int32`; result `[batch, seqlen, topk] fp32` ("Returns").
 *   - `pytorch_extract_topk_scores(logits, topk_indices, dim=-1)`: the
 *     given-indices path gathers the scores at caller-supplied indices.
 *   - causal masking (module summary).
 * and the index conventions of the metrale.ai page "Module glm5next_dsa"
 * ("-1 = invalid", section "Shape of the pipeline"; the whole index row is
 * written, -1 first, section "Checkpoint and kernel facts"; kernels refuse
 * shapes they cannot hold instead of dropping data, section "Constants").
 *
 * Score of query t against compressed key j (DSA lightning indexer):
 *     I[t, j] = sum_h w[t, h] * ReLU( q[t, h, :] . k[j, :] )
 * Key j is visible to a query at position t iff (j + 1) * compress_ratio - 1
 * <= t (a key counts only when its whole compressed block is at or before
 * t).  A prefill row s sits at position s; with `q_pos`, row s of sequence b
 * sits at q_pos[b] + s.
 *
 * Memory: every pointer argument is DEVICE memory owned by the caller,
 * dense and contiguous in the stated layout (the varlen entry points'
 * cu_seqlens and the host-buffer entry points dsa_indexer_fwd_host() and
 * dsa_indexer_host_plan() take HOST arrays, as stated there); q and k must
 * be 16-byte aligned.  The library allocates no device memory: it works in the
 * caller's workspace (dsa_indexer_fwd_static_scratch() instead uses a fixed
 * array inside the library).  Every call is asynchronous on `cuda_stream` (a
 * cudaStream_t; NULL = the legacy default stream): outputs are valid once
 * that stream has synchronised.  Calls that share a workspace must be
 * ordered on one stream.
 *
 * Errors: argument problems are returned synchronously, before anything is
 * enqueued, and leave the outputs untouched.  Problems only the device can
 * see (a given index outside [-1, S_kv), a bounded wait that expired) are
 * recorded in the workspace's status word; read them with
 * dsa_indexer_check().
 */
#ifndef DSA_INDEXER_H
#define DSA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,    /* NULL pointer, size <= 0, misaligned q/k */
    DSA_ERR_UNSUPPORTED = 2,    /* shape outside the compiled envelope, or
                                   the current device is not sm_103 */
    DSA_ERR_WORKSPACE = 3,      /* workspace NULL or smaller than required */
    DSA_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    DSA_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait expired */
    DSA_ERR_INDEX_RANGE = 6     /* a given index was outside [-1, S_kv) */
} dsa_status;

/* Compiled envelope (shapes outside it return DSA_ERR_UNSUPPORTED):
 *   H in {1, 2, 4, 8, 16, 32, 64, 128}; 8 <= D <= 128 with D % 8 == 0;
 *   1 <= topk <= DSA_MAX_TOPK; B * S < 2^31; S_kv < 2^31; and the
 *   per-row selection must fit in shared memory (S_kv * 4 + pow2(topk) * 8
 *   bytes plus a few KB, checked against the device limit). */
#define DSA_MAX_TOPK 8192
#define DSA_MAX_D 128

/*
 * Bytes of device workspace dsa_indexer_fwd() needs for this shape
 * (has_in_idx != 0 selects the given-indices path).  Returns 0 when the
 * shape is invalid.  The workspace starts with a 256-byte status header.
 * Top-k path, one kernel (scores and selection in the same kernel, chosen by
 * the prefill policy below): the header is followed by the kernel's per-CTA
 * scratch, 160 x 2 x (256 / H) x (S_kv rounded up to 32, plus 32) fp32,
 * whatever S.
 * Top-k path, two kernels: the header is followed by the fp32 logits of one
 * chunk of query rows, [B, rows, S_kv] with B * rows * S_kv * 4 <= 64 MiB
 * (all S rows when they fit, else a multiple of 256 / H rows, at least one
 * scoring tile), whatever S.
 * Given-indices path: H in {16, 32, 64, 128} scores the gathered keys
 * directly and needs the header only; other H take the header plus the
 * full logits [B, S, S_kv].
 * The result depends on the prefill policy in force when it is called.
 */
DSA_API size_t dsa_indexer_workspace_size(int S, int B, int H, int D,
                                          int S_kv, int compress_ratio,
                                          int topk, int has_in_idx);

/*
 * Prefill top-k path policy (process-wide; the default is
 * DSA_PREFILL_AUTO).  Both paths give the same indices and scores.
 *   DSA_PREFILL_AUTO        the one-kernel forward for rows of at least 8192
 *                           compressed keys (S_kv >= 8192), where its
 *                           selection keeps pace with the scoring; the
 *                           two-kernel forward (scores, then selection, one
 *                           L2-sized chunk of query rows at a time) below.
 *   DSA_PREFILL_ONE_KERNEL  the one-kernel forward whenever the shape fits it
 *                           (H in {32, 64, 128}, S >= 256 / H, topk <= 2048,
 *                           S_kv < 2^20).
 *   DSA_PREFILL_TWO_KERNELS always the two-kernel forward.
 * Decode-shaped rows (S < 256 / H, with H in {32, 64, 128}, D <= 128 and
 * w 16-byte aligned) always take the split-over-keys decode kernel and the
 * selection kernel; other small shapes take the two-kernel forward.  Set the policy before sizing a
 * workspace: the size depends on it.  Returns DSA_OK or
 * DSA_ERR_INVALID_ARG.
 */
#define DSA_PREFILL_AUTO 0
#define DSA_PREFILL_ONE_KERNEL 1
#define DSA_PREFILL_TWO_KERNELS 2
DSA_API int dsa_set_prefill_policy(int policy);

/*
 * Number of kernels dsa_indexer_fwd() launches for this shape under the
 * current policy (1 for the one-kernel forward and the direct given-indices
 * path; 2 per chunk of query rows for the two-kernel forward); 0 for an
 * invalid shape.  dsa_indexer_fwd_profiled() records one event after each.
 */
DSA_API int dsa_indexer_fwd_launches(int S, int B, int H, int D, int S_kv,
                                     int compress_ratio, int topk,
                                     int has_in_idx);

/*
 * The indexer forward (v4_lighting_indexer / V4IndexerFunction.forward).
 *
 *   q        [S, B, H, D] bf16          (index_q)
 *   k        [S_kv, B, D] bf16          (index_k, already compressed)
 *   w        [S, B, H] fp32             (weights)
 *   q_pos    [B] int32 or NULL          (first query position per sequence)
 *   in_idx   [B, S, topk] int32 or NULL (topk_indices)
 *   out_idx  [B, S, topk] int32
 *   out_scores [B, S, topk] fp32
 *
 * in_idx == NULL: per row, the min(topk, n_visible) visible keys with the
 * largest score, sorted by descending score, equal scores by ascending key
 * index; remaining slots hold -1 and -inf.  Scores compare as IEEE values
 * with -0.0 equal to +0.0 (the score written is +0.0).  With non-finite
 * inputs a score may be +-inf or NaN: a NaN orders by its bits (positive
 * NaN above +inf, negative NaN below -inf), and any kept slot whose score
 * is -inf holds index -1.  Only finite inputs are covered by the parity
 * tests.
 * in_idx != NULL: out_idx is a copy of in_idx; out_scores holds the score at
 * each given index, or -inf where the index is -1, not visible, or outside
 * [0, S_kv) (the latter also sets DSA_ERR_INDEX_RANGE in the status word).
 * Each slot is scored on its own: repeated indices repeat the score, order
 * is kept.  No alignment is asked of w or in_idx beyond their element size.
 *
 * Returns DSA_OK once the work is enqueued, else the synchronous error.
 */
DSA_API int dsa_indexer_fwd(const void *q, const void *k, const float *w,
                            int S, int B, int H, int D, int S_kv,
                            int compress_ratio, int topk,
                            const int32_t *q_pos, const int32_t *in_idx,
                            int32_t *out_idx, float *out_scores,
                            void *workspace, size_t workspace_bytes,
                            void *cuda_stream);

/*
 * Packed variable-length sequences (the packed-sequence dispatch of the V4
 * indexer adaptation on the NeMo AutoModel "tilelang_indexer" page).
 * N sequences share one token axis: sequence i owns query rows
 * [cu_seqlens_q[i], cu_seqlens_q[i+1]) and compressed keys
 * [cu_seqlens_k[i], cu_seqlens_k[i+1]).  cu_seqlens_q / cu_seqlens_k are
 * HOST arrays of N + 1 int32, starting at 0, non-decreasing.
 *
 *   q        [T, H, D] bf16       (T = cu_seqlens_q[N])
 *   k        [T_kv, D] bf16       (T_kv = cu_seqlens_k[N])
 *   w        [T, H] fp32
 *   q_pos    [N] int32 or NULL    (device; row s of sequence i sits at
 *                                  q_pos[i] + s, NULL: at s)
 *   in_idx   [T, topk] int32 or NULL (device; indices local to the row's
 *                                  sequence)
 *   out_idx, out_scores [T, topk] (device; indices local to the sequence)
 *
 * Per row the result is that of dsa_indexer_fwd() on the row's sequence
 * alone (B = 1).  Rows of a sequence with no keys get -1 / -inf (given
 * indices are copied through unchecked).  Sequences run on up to 4 streams
 * at once, each with its own slice of the workspace; a workspace smaller
 * than dsa_indexer_varlen_workspace_size() but at least one slice (the
 * largest sequence's need) runs fewer at once.  Asynchronous on
 * `cuda_stream`, which the library's other streams join before the call's
 * work ends; dsa_indexer_check(workspace) reports the device status of all
 * sequences.  Calls on one device are serialised.
 */
DSA_API size_t dsa_indexer_varlen_workspace_size(int N,
                                                 const int32_t *cu_seqlens_q,
                                                 const int32_t *cu_seqlens_k,
                                                 int H, int D,
                                                 int compress_ratio, int topk,
                                                 int has_in_idx);
DSA_API int dsa_indexer_fwd_varlen(const void *q, const void *k,
                                   const float *w, int N,
                                   const int32_t *cu_seqlens_q,
                                   const int32_t *cu_seqlens_k, int H, int D,
                                   int compress_ratio, int topk,
                                   const int32_t *q_pos, const int32_t *in_idx,
                                   int32_t *out_idx, float *out_scores,
                                   void *workspace, size_t workspace_bytes,
                                   void *cuda_stream);

/*
 * How dsa_indexer_fwd_host() splits and orders the query rows of a call of
 * this shape (for inspection; no device work).  Writes the chunk starts
 * (chunks + 1 values, increasing, the last one S) to `starts` and the
 * processing order (a permutation of 0..chunks-1) to `order`, both
 * caller-owned host arrays of at least 17 ints.  q_pos: host [B] or NULL,
 * as in dsa_indexer_fwd_host().  `sms`: the SM count the wave alignment
 * assumes (0 or less: the current device's; none without a device).
 * Returns the chunk count (1..16), or 0 for an invalid shape or a NULL
 * array.
 */
DSA_API int dsa_indexer_host_plan(int S, int B, int H, int D, int S_kv,
                                  int compress_ratio, int topk,
                                  const int32_t *q_pos, int has_in_idx,
                                  int sms, int *starts, int *order);

/*
 * Bytes of DEVICE memory dsa_indexer_fwd_host() needs for this shape: room
 * for the inputs, the outputs and the workspace of its chunked pipeline.
 * Returns 0 when the shape is invalid.
 */
DSA_API size_t dsa_indexer_host_buffer_size(int S, int B, int H, int D,
                                            int S_kv, int compress_ratio,
                                            int topk, int has_in_idx);

/*
 * The forward on HOST buffers (the end-to-end call): q, k, w, q_pos,
 * in_idx are host inputs and out_idx / out_scores host outputs, with the
 * layouts and meaning of dsa_indexer_fwd().  The call copies the inputs to
 * `device_buf` (caller-owned device memory of dsa_indexer_host_buffer_size()
 * bytes, 256-byte aligned), runs the forward there and copies the results
 * back, pipelining the copies against the kernels: the query rows are split
 * along S into up to 16 chunks of at least 512 rows (none for S < 1024),
 * whose starts fall on whole waves of work items of the current device when
 * the chunks hold at least one; the next chunk's rows are copied in while
 * one chunk is scored, and its results are copied out while the following
 * ones are scored.  Chunks run last rows first, or, when the kernels
 * outweigh the copies (many visible keys per copied byte), alternately
 * from the costliest and the cheapest end.  Results are identical to one
 * dsa_indexer_fwd() call whatever the chunking.  The copies overlap only
 * when the host buffers are page-locked (pinned); pageable buffers work but
 * serialise.  dsa_indexer_host_buffer_size() and this call must see the
 * same current device (the chunking reads its SM count).
 *
 * The work is ordered after everything already queued on `cuda_stream` and
 * the call returns once the results are in the host outputs (it
 * synchronises `cuda_stream`).  Calls on one device are serialised.
 * Returns DSA_OK; a synchronous argument error (DSA_ERR_INVALID_ARG,
 * DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE); DSA_ERR_CUDA; or the device
 * status of the run (DSA_ERR_INDEX_RANGE, DSA_ERR_DEVICE_TIMEOUT).  The
 * library keeps two copy streams, a few events and a small page-locked
 * staging buffer per device for the life of the process.
 */
DSA_API int dsa_indexer_fwd_host(const void *q, const void *k, const float *w,
                                 int S, int B, int H, int D, int S_kv,
                                 int compress_ratio, int topk,
                                 const int32_t *q_pos, const int32_t *in_idx,
                                 int32_t *out_idx, float *out_scores,
                                 void *device_buf, size_t device_buf_bytes,
                                 void *cuda_stream);

/*
 * dsa_indexer_fwd() with stage timing: `stage_events` holds `n_events`
 * (0..1024) caller-created cudaEvent_t handles, recorded on `cuda_stream`:
 * event 0 before the first kernel, then one event after each kernel launch
 * in launch order (dsa_indexer_fwd_launches() of them: scores and selection
 * alternate for the two-kernel forward, chunk by chunk); events past the
 * last launch are recorded after it, events past n_events not at all.  Same
 * work, outputs and errors as dsa_indexer_fwd() (plus DSA_ERR_INVALID_ARG
 * for a NULL event or n_events outside 0..1024).
 */
DSA_API int dsa_indexer_fwd_profiled(const void *q, const void *k,
                                     const float *w, int S, int B, int H,
                                     int D, int S_kv, int compress_ratio,
                                     int topk, const int32_t *q_pos,
                                     const int32_t *in_idx, int32_t *out_idx,
                                     float *out_scores, void *workspace,
                                     size_t workspace_bytes,
                                     void *cuda_stream,
                                     void *const *stage_events, int n_events);

/*
 * The scoring step alone: logits [B, S, S_kv] fp32 (`logits`, caller-owned
 * device memory), I[t, j] at visible keys and -inf elsewhere -- the
 * `logits` tensor that pytorch_extract_topk_scores() gathers from.
 * `workspace` needs dsa_indexer_logits_workspace_size() bytes (the status
 * header only).
 */
DSA_API size_t dsa_indexer_logits_workspace_size(void);
DSA_API int dsa_indexer_logits(const void *q, const void *k, const float *w,
                               int S, int B, int H, int D, int S_kv,
                               int compress_ratio, const int32_t *q_pos,
                               float *logits, void *workspace,
                               size_t workspace_bytes, void *cuda_stream);

/*
 * Synchronises `cuda_stream`, then reads and clears the device status word
 * of `workspace`.  Returns DSA_OK, DSA_ERR_INDEX_RANGE,
 * DSA_ERR_DEVICE_TIMEOUT or DSA_ERR_CUDA (a sticky CUDA error).
 */
DSA_API int dsa_indexer_check(void *workspace, void *cuda_stream);

/* Static description of a status code. */
DSA_API const char *dsa_status_string(int status);

/*
 * Self-test of the device wait limit: launches one block that waits on a
 * barrier nothing will complete, with a limit of `limit_us` microseconds
 * (clamped to [1, 1000000]), and records DSA_ERR_DEVICE_TIMEOUT in the
 * status word of `workspace` when the limit expires.  Used by the tests to
 * show a hung wait ends with an error the host can read.
 */
DSA_API int dsa_selftest_wait_limit(int limit_us, void *workspace,
                                    size_t workspace_bytes,
                                    void *cuda_stream);

/*
 * Allocation-free variant of dsa_indexer_fwd() (the pages have no
 * counterpart; this is a library convenience).
 *
 * For callers that cannot call cudaMalloc -- code running while a caching
 * allocator holds all free device memory, plugin hosts that only hand out
 * the tensors they own, or paths where an allocation would synchronise the
 * device.  The forward's scratch (status header, then the one-kernel
 * prefill's per-CTA score rows or the written logits) comes from a fixed
 * array of DSA_STATIC_SCRATCH_BYTES inside the library instead of a caller
 * workspace; the caller still passes every input and output.
 *
 *   - Limit: every top-k shape runs.  A prefill whose one-kernel scratch
 *     (dsa_indexer_workspace_size(); it grows with S_kv: it fits up to
 *     S_kv = 6496, 13056 and 26176 for H = 32, 64 and 128) exceeds
 *     DSA_STATIC_SCRATCH_BYTES (64 MiB plus a 256-byte header) runs scores
 *     then selection instead, whose logits chunk is at
 *     most 64 MiB whatever S (the same results; slower on long rows).  A
 *     given-indices shape that reads scores back from written logits (H not
 *     in {16, 32, 64, 128}) and needs more than the array (B*S*S_kv >
 *     16,777,216) is refused with DSA_ERR_UNSUPPORTED before any device
 *     work.  Other argument errors are those of dsa_indexer_fwd().
 *   - Memory: every GPU that loads this part of the library holds one copy
 *     of the array until the process exits.  No call allocates or frees
 *     device memory.
 *   - Set-up: every call looks up the current device's copy of the array
 *     (cudaGetSymbolAddress, which allocates nothing), so a device reset or
 *     module reload between calls is harmless.  The first call on a device
 *     may also load the library's kernels onto it; make that first call
 *     before any stream capture.
 *   - Sharing: all calls on a device share the one array, which keeps the
 *     last call's contents.  Calls that overlap on the GPU (different
 *     streams, or threads without ordering) race on it; order them on one
 *     stream.  Each call clears the status word it uses; the rest of the
 *     array needs no clearing (every entry read was written earlier in the
 *     same call).
 *   - out_status: NULL, or one device int32 that receives this call's device
 *     status bits (0 = ok; bit 0 = a given index outside [-1, S_kv); bit 1 =
 *     a bounded wait expired), written asynchronously on `cuda_stream`.
 * Asynchronous on `cuda_stream` like dsa_indexer_fwd().
 */
#define DSA_STATIC_SCRATCH_BYTES ((size_t)64 * 1024 * 1024 + 256)
DSA_API int dsa_indexer_fwd_static_scratch(
    const void *q, const void *k, const float *w, int S, int B, int H, int D,
    int S_kv, int compress_ratio, int topk, const int32_t *q_pos,
    const int32_t *in_idx, int32_t *out_idx, float *out_scores,
    int32_t *out_status, void *cuda_stream);

/*
 * Backward of the given-slots scores (V4IndexerFunction.backward(grad_scores,
 * grad_indices) on the NeMo AutoModel "tilelang_indexer" page; the indices
 * are integers and get no gradient).  With s_h = q[t,h,:] . k[j,:] and
 * g = grad_scores[b, s, i] for each slot i of row (b, s) whose key
 * j = idx[b, s, i] is valid (0 <= j < S_kv) and visible to the row:
 *     grad_w[s, b, h] += g * ReLU(s_h)
 *     grad_q[s, b, h] += g * w[s, b, h] * [s_h > 0] * k[j, b]
 *     grad_k[j, b]    += g * w[s, b, h] * [s_h > 0] * q[s, b, h]
 * (ReLU'(0) taken as 0).  Slots holding -1, an invisible key or an index
 * outside [-1, S_kv) contribute nothing; the last also sets
 * DSA_ERR_INDEX_RANGE in the status word.  Duplicate indices in a row
 * contribute once per slot.
 *
 *   q [S, B, H, D] bf16, k [S_kv, B, D] bf16, w [S, B, H] fp32 and q_pos
 *   (nullable) as for dsa_indexer_fwd(); idx [B, S, topk] int32;
 *   grad_scores [B, S, topk] fp32.
 *   Outputs (fp32, caller-owned device memory, every element written):
 *   grad_q [S, B, H, D], grad_k [S_kv, B, D] (cleared by the call, then
 *   accumulated with atomics, so its low-order bits vary from run to run),
 *   grad_w [S, B, H].
 *   Precision: the scores are accumulated in fp32; g * w is rounded to bf16
 *   as an operand of the two gradient products, which accumulate in fp32.
 *   Envelope: H = 64, D a multiple of 8 up to 128, S_kv * B * D < 2^31;
 *   otherwise DSA_ERR_UNSUPPORTED.  q, k and grad_k 16-byte aligned.
 *   workspace: dsa_indexer_bwd_workspace_size() bytes, 256-byte aligned
 *   (the status header; read it with dsa_indexer_check()).
 * Asynchronous on `cuda_stream`; argument errors are returned before any
 * work is enqueued.
 */
DSA_API size_t dsa_indexer_bwd_workspace_size(void);
DSA_API int dsa_indexer_bwd(const void *q, const void *k, const float *w,
                            int S, int B, int H, int D, int S_kv,
                            int compress_ratio, int topk,
                            const int32_t *q_pos, const int32_t *idx,
                            const float *grad_scores, float *grad_q,
                            float *grad_k, float *grad_w, void *workspace,
                            size_t workspace_bytes, void *cuda_stream);

/*
 * The pool variant (metrale.ai page "Module glm5next_dsa", section "Shape
 * of the pipeline": k, gate, valid, ape -> kpool_compress -> index_scores ->
 * topk_pools -> expand_selection -> token ids, -1 = invalid; section
 * "Checkpoint and kernel facts": the pool softmax runs over the slot axis
 * per channel, pooling starts at first_key, a pool counts only if all of its
 * slots are valid, expand_selection writes every slot of the row).
 *
 * Pool p of sequence b covers tokens first_key + p*kpool + s (s < kpool);
 * P = (T - first_key) / kpool whole pools (an incomplete pool at the end is
 * dropped).  Pooled key, per channel c, with z_s = gate[token_s, b, c] +
 * ape[s, c]:  key[p, b, c] = sum_s softmax_s(z)_s * k[token_s, b, c]
 * (fp32, stored bf16).  A pool is a candidate iff every token's valid flag
 * is nonzero (valid NULL: all valid).  Query row s of sequence b at position
 * t = (q_pos ? q_pos[b] : 0) + s sees pool p iff its last token is at or
 * before t.
 *
 *   k [T, B, D] bf16 (per-token indexer keys), gate [T, B, D] fp32,
 *   ape [kpool, D] fp32, valid [T, B] uint8 or NULL; 1 <= kpool <= 8,
 *   D a multiple of 8; k, gate and ape 16-byte aligned.
 */

/* The compression alone: out_keys [P, B, D] bf16 (16-byte aligned),
 * out_valid [P, B] uint8 (nullable).  Asynchronous on cuda_stream. */
DSA_API int dsa_kpool_compress(const void *k, const float *gate,
                               const float *ape, const uint8_t *valid, int T,
                               int B, int D, int kpool, int first_key,
                               void *out_keys, uint8_t *out_valid,
                               void *cuda_stream);

/* The expansion alone: pools [rows, select_k] int32 (pool ids or -1) ->
 * out_tokens [rows, select_k * kpool], slot i*kpool + s = first_key +
 * pool_i*kpool + s, or -1 when pool_i is -1. */
DSA_API int dsa_expand_selection(const int32_t *pools, long long rows,
                                 int select_k, int kpool, int first_key,
                                 int32_t *out_tokens, void *cuda_stream);

/* Workspace bytes of dsa_indexer_fwd_pooled (0 = invalid or unsupported
 * shape). */
DSA_API size_t dsa_indexer_pooled_workspace_size(int S, int B, int H, int D,
                                                 int T, int kpool,
                                                 int first_key,
                                                 int index_topk);

/*
 * The whole variant: compression, the indexer forward over the pools (q
 * [S, B, H, D] bf16, w [S, B, H] fp32 as for dsa_indexer_fwd; the
 * index_topk / kpool best candidate pools per row, descending score, ties
 * to the lower pool), and expansion to index_topk token ids.
 *   index_topk: a nonzero multiple of kpool ("index_topk is a nonzero
 *   multiple of index_kpool").
 *   out_tokens [B, S, index_topk] int32; out_pools [B, S, index_topk/kpool]
 *   int32 (-1 for empty slots); out_scores [B, S, index_topk/kpool] fp32
 *   (-inf for empty slots).
 *   workspace: dsa_indexer_pooled_workspace_size() bytes, 256-byte aligned;
 *   its status word is read by dsa_indexer_check().
 * Asynchronous on cuda_stream; argument errors return before any work.
 */
DSA_API int dsa_indexer_fwd_pooled(
    const void *q, const void *k, const float *gate, const float *ape,
    const uint8_t *valid, const float *w, int S, int B, int H, int D, int T,
    int kpool, int first_key, int index_topk, const int32_t *q_pos,
    int32_t *out_tokens, int32_t *out_pools, float *out_scores,
    void *workspace, size_t workspace_bytes, void *cuda_stream);

/*
 * Sparse MLA forward over selected tokens (page "Module glm5next_dsa",
 * "Shape of the pipeline": the selected tokens feed an MLA attention
 * without the rotary part, over those tokens only; the
 * latent width is kv_lora_rank).  Attention in the latent space, no rotary
 * part, the latent row of a selected token being both key and value: for
 * row (b, s), head h and the slots i whose token j_i = idx[b, s, i] is in
 * [0, T),
 *     x_i = scale * q[s, b, h, :] . c[j_i, b, :]
 *     out_o[s, b, h, :] = sum_i softmax(x)_i * c[j_i, b, :]
 *     out_lse[s, b, h]  = ln sum_i exp(x_i)
 * (-1 slots skipped, repeated tokens counted once per slot; a row with no
 * valid slot gets o = 0 and lse = -inf; an index outside [-1, T) also sets
 * DSA_ERR_INDEX_RANGE in the status word).
 *   q [S, B, H, Dc] bf16 (latent-space queries), c [T, B, Dc] bf16 (latent
 *   cache), idx [B, S, topk] int32 (e.g. the pool variant's token ids);
 *   out_o [S, B, H, Dc] fp32, out_lse [S, B, H] fp32.
 *   Envelope: H a multiple of 64, Dc in {128, 256, 384, 512}, scale > 0;
 *   q and c 16-byte aligned.  Precision: scores and outputs accumulate in
 *   fp32; the softmax weights enter the output product as bf16.
 *   workspace: dsa_sparse_mla_workspace_size() bytes, 256-byte aligned.
 */
DSA_API size_t dsa_sparse_mla_workspace_size(void);
DSA_API int dsa_sparse_mla_fwd(const void *q, const void *c,
                               const int32_t *idx, int S, int B, int H,
                               int Dc, int T, int topk, float scale,
                               float *out_o, float *out_lse, void *workspace,
                               size_t workspace_bytes, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_INDEXER_H */
