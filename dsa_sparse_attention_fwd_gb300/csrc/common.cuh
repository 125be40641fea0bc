// Shared definitions of the CUDA library: problem description, the causal
// visibility rule and the launchers each kernel file provides.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsa {

// Bits of the device status word at the start of the workspace.
constexpr int kStatusIndexRange = 1;  // a given index outside [-1, S_kv)
constexpr int kStatusTimeout = 2;     // a bounded wait expired

// One indexer problem, as the C ABI receives it (device pointers).
struct Problem {
  const void *q;         // [S, B, H, D] bf16
  const void *k;         // [S_kv, B, D] bf16
  const float *w;        // [S, B, H] fp32
  const int32_t *q_pos;  // [B] or nullptr: row s of sequence b at q_pos[b]+s
  int S, B, H, D, S_kv, ratio;
  // [S_kv, B] or nullptr: a key whose flag is 0 is not a candidate (its
  // logit is -inf; the selection turns a selected -inf into -1)
  const uint8_t *kv_valid = nullptr;
};

// Position of query row s of sequence b.
__device__ __forceinline__ long long row_pos(const int32_t *q_pos, int b,
                                             int s) {
  return q_pos ? (long long)__ldg(q_pos + b) + s : (long long)s;
}

// Causal rule over compressed keys (DeepSeek-V4 indexer, causal masking;
// a compressed key stands for source tokens [j*r, (j+1)*r) and is visible
// only when the whole block is at or before the query): (j+1)*r - 1 <= pos.
// Returns how many keys (a prefix 0..n-1) are visible.
__host__ __device__ __forceinline__ int n_visible(long long pos, int ratio,
                                                  int S_kv) {
  if (pos < 0) return 0;
  long long n = (pos + 1) / ratio;
  return n < (long long)S_kv ? (int)n : S_kv;
}

// Programmatic dependent launch: a kernel launched with programmatic
// stream serialization may start while the previous kernel in the stream is
// still running; pdl_wait() blocks until that kernel has completed and its
// memory is visible.  pdl_allow_dependents() lets the next such kernel be
// scheduled before this one finishes.  Both are no-ops without a dependency.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Order-preserving unsigned key of an fp32 score (larger float <-> larger
// key; -0.0 folded onto +0.0 so the index tie-break decides between them).
__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Twice ReLU(x): x + |x| is 2x for x >= 0 and +0 otherwise, exactly unless
// 2x overflows.  The scoring epilogues pair it with halved weights (exact
// unless a weight is subnormal: w/2 * (x + |x|) is the same product as
// w * ReLU(x)) or halve the finished sum (every term and partial sum was
// exactly doubled), and it runs on the FMA pipe instead of the integer/ALU
// one.
__device__ __forceinline__ float relu2(float x) { return x + fabsf(x); }
// relu2 of two values with one packed add (the same result lane by lane).
__device__ __forceinline__ float2 relu2x2(float a, float b) {
  return __fadd2_rn(make_float2(a, b), make_float2(fabsf(a), fabsf(b)));
}

// Scoring kernel tile geometry.
constexpr int kTileKeys = 128;      // MMA M: compressed keys per tile
constexpr int kTileCols = 256;      // MMA N: (query, head) columns per tile
constexpr int kChunk = 64;          // bf16 per 128-byte swizzled row
constexpr int kScoreThreads = 320;  // TMA warp, MMA warp, 8 epilogue warps
constexpr int kDecChunkTiles = 4;   // decode: key tiles per work item

// Top-k selection: a sort pass handles up to 256 threads x (this + 2)
// elements, i.e. topk + 256 candidates with topk <= 256 * DSA_SEL_MAX_EPT
// (= DSA_MAX_TOPK).
#define DSA_SEL_MAX_EPT 32

// Launchers (return cudaSuccess or the launch error).  The scoring and
// selection launches cover query rows [s0, s0 + Sc) of every sequence;
// `logits` is [B, Sc, S_kv] fp32 for those rows (only visible entries are
// written), the outputs are the full [B, S, topk].
cudaError_t launch_index_scores(const Problem &p, const CUtensorMap &tm_q,
                                const CUtensorMap &tm_k, float *logits,
                                int *status, int num_sms, cudaStream_t st,
                                int s0, int Sc);
size_t index_scores_smem_bytes(int H, int D);

cudaError_t launch_topk_select(const Problem &p, const float *logits, int topk,
                               int32_t *out_idx, float *out_scores,
                               int num_sms, cudaStream_t st, int s0, int Sc);
size_t topk_select_smem_bytes(int S_kv, int topk);

// Given indices, scores read from written logits (any H).
cudaError_t launch_gather_logits(const Problem &p, const float *logits,
                                 const int32_t *in_idx, int topk,
                                 int32_t *out_idx, float *out_scores,
                                 int *status, int num_sms, cudaStream_t st);

// Given indices, scores computed from the gathered keys on the tensor cores
// (no logits).  tm_q: q with a box of one query.  Returns
// cudaErrorNotSupported when (H, D) has no instantiation.
cudaError_t launch_gather_scores(const Problem &p, const CUtensorMap &tm_q,
                                 const int32_t *in_idx, int topk,
                                 int32_t *out_idx, float *out_scores,
                                 int *status, int num_sms, cudaStream_t st);
bool gather_supported(int H, int D);
size_t gather_smem_bytes(int H, int D);

// Decode scoring (one MMA column per head of a single query); returns
// cudaErrorNotSupported when (H, D) has no decode instantiation.
cudaError_t launch_decode_scores(const Problem &p, const CUtensorMap &tm_q,
                                 const CUtensorMap &tm_k, float *logits,
                                 int *status, int num_sms, cudaStream_t st);
bool decode_supported(int H, int D);
size_t decode_smem_bytes(int H, int D);

cudaError_t launch_fill_masked(float *logits, size_t n, cudaStream_t st);

// Prefill forward in one kernel: scores and per-row top-k, the scores kept
// in a per-CTA scratch (two work-item slots of 256/H rows of S_kv fp32,
// for at most kIndexTopkMaxCtas CTAs) instead of [B, S, S_kv] logits.
constexpr int kIndexTopkMaxCtas = 160;
constexpr int kIndexTopkMaxTopk = 2048;
constexpr size_t kIndexTopkMaxSmem = 232448;  // 227 KB opt-in per block
bool index_topk_supported(int S, int H, int D, int S_kv, int topk);
size_t index_topk_smem_bytes(int H, int D, int topk);
size_t index_topk_scratch_bytes(int H, int S_kv);
int index_topk_row_stride(int S_kv);
// tm_q: q with a box of 256/H queries (as for launch_index_scores).
cudaError_t launch_index_topk(const Problem &p, const CUtensorMap &tm_q,
                              const CUtensorMap &tm_k, int topk,
                              float *scratch, int32_t *out_idx,
                              float *out_scores, int *status, int num_sms,
                              cudaStream_t st);

// TMA map of q [S, B, H, D] bf16 as (d, h, b, s) with a box of 64 d x H
// heads x 1 x `queries` (returns a dsa_status code).
int encode_q(CUtensorMap *m, const Problem &p, int queries);
int encode_q_heads(CUtensorMap *m, const Problem &p, int queries, int heads);

// Multiprocessor count of the current device (a dsa_status code).
int device_num_sms(int *num_sms);

// The forward behind the C entry points (arguments and return codes of
// dsa_indexer_fwd_profiled); clear_status = false keeps the workspace's
// status word, so forwards sharing a workspace accumulate device errors.
// kv_valid ([S_kv, B] or nullptr): keys whose flag is 0 are not candidates
// (top-k path only).
int forward_core(const void *q, const void *k, const float *w, int S, int B,
                 int H, int D, int S_kv, int compress_ratio, int topk,
                 const int32_t *q_pos, const int32_t *in_idx, int32_t *out_idx,
                 float *out_scores, void *workspace, size_t workspace_bytes,
                 void *cuda_stream, void *const *stage_events, int n_events,
                 bool clear_status, const uint8_t *kv_valid = nullptr,
                 bool one_kernel_ok = true);

// Workspace bytes of a top-k prefill that runs scores then selection over
// row chunks (at most the header plus a 64 MiB logits chunk).
size_t two_kernel_workspace_bytes(int S, int B, int H, int S_kv);

cudaError_t launch_wait_selftest(int limit_us, int *status, cudaStream_t st);

}  // namespace dsa
