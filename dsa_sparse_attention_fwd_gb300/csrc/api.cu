// C ABI of the lightning-indexer forward: argument validation, workspace
// layout, TMA tensor-map encoding and dispatch onto the caller's stream.
// Interface: DeepSeek-V4 SBHD indexer ("tilelang_indexer" page of NeMo
// AutoModel: V4IndexerFunction / v4_lighting_indexer /
// pytorch_extract_topk_scores).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "dsa_indexer.h"
#include "ptx.cuh"

namespace {

using dsa::Problem;

constexpr size_t kHeaderBytes = 256;  // status word + padding
constexpr int kMaxStageEvents = 1024;  // dsa_indexer_fwd_profiled

struct DeviceInfo {
  bool valid = false;
  int num_sms = 0;
  int max_smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

int current_device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo &d = g_dev[dev];
  if (!d.valid) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin,
                               cudaDevAttrMaxSharedMemoryPerBlockOptin,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor,
                               dev) != cudaSuccess)
      return DSA_ERR_CUDA;
    d.valid = true;
  }
  *out = d;
  // The kernels are built for sm_103a only.
  if (d.cc_major != 10 || d.cc_minor != 3) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool is_pow2_heads(int H) {
  return H == 1 || H == 2 || H == 4 || H == 8 || H == 16 || H == 32 ||
         H == 64 || H == 128;
}

// Shape checks shared by every entry point (no device access).
int check_shape(int S, int B, int H, int D, int S_kv, int ratio) {
  if (S <= 0 || B <= 0 || H <= 0 || D <= 0 || S_kv <= 0 || ratio <= 0)
    return DSA_ERR_INVALID_ARG;
  if (!is_pow2_heads(H)) return DSA_ERR_UNSUPPORTED;
  if (D % 8 != 0 || D > DSA_MAX_D) return DSA_ERR_UNSUPPORTED;
  if ((long long)B * S >= (1ll << 31)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

size_t logits_bytes(int S, int B, int S_kv) {
  return (size_t)B * (size_t)S * (size_t)S_kv * sizeof(float);
}

// The two-kernel prefill writes the logits of at most this many bytes of
// query rows at a time (scores, then their selection, chunk after chunk),
// so the buffer stays in L2 and does not grow with S.
constexpr size_t kLogitsChunkBytes = (size_t)64 << 20;

// Query rows per chunk of the two-kernel top-k path (a multiple of the
// scoring tile's 256/H rows, or all S rows).
int logits_chunk_rows(int S, int B, int H, int S_kv) {
  const size_t per_row = (size_t)B * (size_t)S_kv * sizeof(float);
  if ((size_t)S * per_row <= kLogitsChunkBytes) return S;
  const long long tq = dsa::kTileCols / H;
  long long rows = (long long)(kLogitsChunkBytes / per_row) / tq * tq;
  if (rows < tq) rows = tq;
  return rows < S ? (int)rows : S;
}

// Prefill top-k path policy (dsa_set_prefill_policy).
std::atomic<int> g_prefill_policy{DSA_PREFILL_AUTO};

// Whether a top-k call of this shape runs the one-kernel forward: the
// shape must fit it, and under the automatic policy the rows must be long
// (at least 8192 compressed keys), where the selection keeps pace with the
// scoring; shorter rows run scores then selection in two kernels.
bool use_one_kernel(int S, int H, int D, int S_kv, int topk) {
  if (!dsa::index_topk_supported(S, H, D, S_kv, topk)) return false;
  const int pol = g_prefill_policy.load(std::memory_order_relaxed);
  if (pol == DSA_PREFILL_TWO_KERNELS) return false;
  if (pol == DSA_PREFILL_ONE_KERNEL) return true;
  return S_kv >= 8192;
}

bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

namespace dsa {
// q [S, B, H, D] bf16 viewed as the 4-D tensor (d, h, b, s); one box is
// 64 d x H heads x 1 sequence x `queries` queries (256/H for the prefill
// tile = 256 rows of 128 bytes; 1 for decode, given indices and backward).
int encode_q(CUtensorMap *m, const Problem &p, int queries) {
  return encode_q_heads(m, p, queries, p.H);
}

// As encode_q with a box of `heads` heads (a divisor of H).
int encode_q_heads(CUtensorMap *m, const Problem &p, int queries, int heads) {
  auto fn = encode_fn();
  if (!fn) return DSA_ERR_CUDA;
  const cuuint64_t dims[4] = {(cuuint64_t)p.D, (cuuint64_t)p.H,
                              (cuuint64_t)p.B, (cuuint64_t)p.S};
  const cuuint64_t strides[3] = {(cuuint64_t)p.D * 2,
                                 (cuuint64_t)p.H * p.D * 2,
                                 (cuuint64_t)p.B * p.H * p.D * 2};
  const cuuint32_t box[4] = {(cuuint32_t)dsa::kChunk, (cuuint32_t)heads, 1,
                             (cuuint32_t)queries};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                  const_cast<void *>(p.q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_UNSUPPORTED;
}

// Multiprocessor count of the current device (DSA_ERR_UNSUPPORTED unless
// it is an sm_103 device).
int device_num_sms(int *num_sms) {
  DeviceInfo d;
  const int rc = current_device_info(&d);
  if (rc == DSA_OK) *num_sms = d.num_sms;
  return rc;
}

}  // namespace dsa

namespace {
using dsa::encode_q;

// k [S_kv, B, D] bf16 viewed as (d, b, j); one box is 64 d x 1 x 128 keys.
int encode_k(CUtensorMap *m, const Problem &p) {
  auto fn = encode_fn();
  if (!fn) return DSA_ERR_CUDA;
  const cuuint64_t dims[3] = {(cuuint64_t)p.D, (cuuint64_t)p.B,
                              (cuuint64_t)p.S_kv};
  const cuuint64_t strides[2] = {(cuuint64_t)p.D * 2,
                                 (cuuint64_t)p.B * p.D * 2};
  const cuuint32_t box[3] = {(cuuint32_t)dsa::kChunk, 1,
                             (cuuint32_t)dsa::kTileKeys};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void *>(p.k), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_UNSUPPORTED;
}

// Given indices are scored from the gathered keys (no logits) when the
// gather kernel has an instantiation for (H, D); otherwise the logits are
// written and read back.
bool gather_direct_shape(int B, int H, int D, int S_kv) {
  (void)B;
  (void)S_kv;
  return dsa::gather_supported(H, D);
}

// Rows with fewer queries per sequence than one prefill tile packs (256/H)
// go to the decode kernel, which splits each row over its keys instead.
bool decode_shape(int S, int H, int D) {
  return S < dsa::kTileCols / H && dsa::decode_supported(H, D);
}

bool use_decode_path(const Problem &p, const DeviceInfo &dev) {
  return decode_shape(p.S, p.H, p.D) && aligned16(p.w) &&
         (size_t)dev.max_smem_optin >= dsa::decode_smem_bytes(p.H, p.D);
}

// Device checks + tensor maps + the scoring launch.
int run_scores(const Problem &p, float *logits, int *status,
               const DeviceInfo &dev, cudaStream_t st, int s0, int Sc) {
  const bool decode = use_decode_path(p, dev);
  if (!decode &&
      (size_t)dev.max_smem_optin < dsa::index_scores_smem_bytes(p.H, p.D))
    return DSA_ERR_UNSUPPORTED;
  CUtensorMap tm_q, tm_k;
  int rc = encode_q(&tm_q, p, decode ? 1 : dsa::kTileCols / p.H);
  if (rc != DSA_OK) return rc;
  rc = encode_k(&tm_k, p);
  if (rc != DSA_OK) return rc;
  const cudaError_t e =
      decode ? dsa::launch_decode_scores(p, tm_q, tm_k, logits, status,
                                         dev.num_sms, st)
             : dsa::launch_index_scores(p, tm_q, tm_k, logits, status,
                                        dev.num_sms, st, s0, Sc);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported shape or device";
    case DSA_ERR_WORKSPACE: return "workspace missing or too small";
    case DSA_ERR_CUDA: return "CUDA error";
    case DSA_ERR_DEVICE_TIMEOUT: return "device wait limit expired";
    case DSA_ERR_INDEX_RANGE: return "given index outside [-1, S_kv)";
    default: return "unknown status";
  }
}

size_t dsa_indexer_workspace_size(int S, int B, int H, int D, int S_kv,
                                  int compress_ratio, int topk,
                                  int has_in_idx) {
  if (check_shape(S, B, H, D, S_kv, compress_ratio) != DSA_OK) return 0;
  if (topk <= 0 || topk > DSA_MAX_TOPK) return 0;
  if (has_in_idx)
    return gather_direct_shape(B, H, D, S_kv)
               ? kHeaderBytes
               : kHeaderBytes + logits_bytes(S, B, S_kv);
  // scores and selection in one kernel need only its per-CTA scratch; the
  // two-kernel path needs the logits of one chunk of query rows
  if (use_one_kernel(S, H, D, S_kv, topk))
    return kHeaderBytes + dsa::index_topk_scratch_bytes(H, S_kv);
  return dsa::two_kernel_workspace_bytes(S, B, H, S_kv);
}

int dsa_set_prefill_policy(int policy) {
  if (policy != DSA_PREFILL_AUTO && policy != DSA_PREFILL_ONE_KERNEL &&
      policy != DSA_PREFILL_TWO_KERNELS)
    return DSA_ERR_INVALID_ARG;
  g_prefill_policy.store(policy, std::memory_order_relaxed);
  return DSA_OK;
}

int dsa_indexer_fwd_launches(int S, int B, int H, int D, int S_kv,
                             int compress_ratio, int topk, int has_in_idx) {
  if (check_shape(S, B, H, D, S_kv, compress_ratio) != DSA_OK) return 0;
  if (topk <= 0 || topk > DSA_MAX_TOPK) return 0;
  if (has_in_idx) return gather_direct_shape(B, H, D, S_kv) ? 1 : 2;
  if (use_one_kernel(S, H, D, S_kv, topk)) return 1;
  const int rows = logits_chunk_rows(S, B, H, S_kv);
  return 2 * ((S + rows - 1) / rows);
}

size_t dsa_indexer_logits_workspace_size(void) { return kHeaderBytes; }

int dsa_indexer_fwd_profiled(const void *q, const void *k, const float *w,
                             int S, int B, int H, int D, int S_kv,
                             int compress_ratio, int topk,
                             const int32_t *q_pos, const int32_t *in_idx,
                             int32_t *out_idx, float *out_scores,
                             void *workspace, size_t workspace_bytes,
                             void *cuda_stream, void *const *stage_events,
                             int n_events) {
  return dsa::forward_core(q, k, w, S, B, H, D, S_kv, compress_ratio, topk,
                           q_pos, in_idx, out_idx, out_scores, workspace,
                           workspace_bytes, cuda_stream, stage_events,
                           n_events, true);
}

}  // extern "C"

namespace dsa {

size_t two_kernel_workspace_bytes(int S, int B, int H, int S_kv) {
  return kHeaderBytes + logits_bytes(logits_chunk_rows(S, B, H, S_kv), B, S_kv);
}

// The forward behind every entry point.  clear_status = false keeps the
// workspace's status word (several forwards sharing one workspace then
// accumulate their device errors).  one_kernel_ok = false makes a top-k
// prefill run scores then selection whatever the policy (for a scratch too
// small for the one-kernel forward).
int forward_core(const void *q, const void *k, const float *w, int S, int B,
                 int H, int D, int S_kv, int compress_ratio, int topk,
                 const int32_t *q_pos, const int32_t *in_idx, int32_t *out_idx,
                 float *out_scores, void *workspace, size_t workspace_bytes,
                 void *cuda_stream, void *const *stage_events, int n_events,
                 bool clear_status, const uint8_t *kv_valid,
                 bool one_kernel_ok) {
  if (!q || !k || !w || !out_idx || !out_scores) return DSA_ERR_INVALID_ARG;
  if (kv_valid && in_idx) return DSA_ERR_UNSUPPORTED;
  int rc = check_shape(S, B, H, D, S_kv, compress_ratio);
  if (rc != DSA_OK) return rc;
  if (topk <= 0) return DSA_ERR_INVALID_ARG;
  if (topk > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k)) return DSA_ERR_INVALID_ARG;
  if (n_events < 0 || n_events > kMaxStageEvents ||
      (n_events > 0 && !stage_events))
    return DSA_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i)
    if (!stage_events[i]) return DSA_ERR_INVALID_ARG;
  const bool fused =
      !in_idx && one_kernel_ok && use_one_kernel(S, H, D, S_kv, topk);
  const size_t need =
      !in_idx && !fused
          ? two_kernel_workspace_bytes(S, B, H, S_kv)
          : dsa_indexer_workspace_size(S, B, H, D, S_kv, compress_ratio, topk,
                                       in_idx != nullptr);
  if (!workspace || workspace_bytes < need) return DSA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return DSA_ERR_INVALID_ARG;

  DeviceInfo dev;
  rc = current_device_info(&dev);
  if (rc != DSA_OK) return rc;
  if (!in_idx && !fused) {
    const size_t sel = dsa::topk_select_smem_bytes(S_kv, topk) + 4096;
    if (sel > (size_t)dev.max_smem_optin) return DSA_ERR_UNSUPPORTED;
  }

  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int *status = static_cast<int *>(workspace);
  float *logits = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                            kHeaderBytes);
  Problem p{q, k, w, q_pos, S, B, H, D, S_kv, compress_ratio};
  p.kv_valid = kv_valid;
  auto mark = [&](int i) {
    return i < n_events
               ? cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st)
               : cudaSuccess;
  };
  // after the last launch: every remaining event
  auto mark_rest = [&](int from) {
    for (int i = from; i < n_events; ++i)
      if (mark(i) != cudaSuccess) return cudaErrorUnknown;
    return cudaSuccess;
  };

  // Workspace: status header, then the logits.
  if (clear_status &&
      cudaMemsetAsync(status, 0, kHeaderBytes, st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (in_idx && gather_direct_shape(B, H, D, S_kv)) {
    // one kernel: gathered keys -> scores at the given slots
    if ((size_t)dev.max_smem_optin < dsa::gather_smem_bytes(H, D))
      return DSA_ERR_UNSUPPORTED;
    CUtensorMap tm_q;
    rc = encode_q(&tm_q, p, 1);
    if (rc != DSA_OK) return rc;
    if (mark(0) != cudaSuccess) return DSA_ERR_CUDA;
    if (dsa::launch_gather_scores(p, tm_q, in_idx, topk, out_idx,
                                  out_scores, status, dev.num_sms,
                                  st) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (mark_rest(1) != cudaSuccess) return DSA_ERR_CUDA;
    return DSA_OK;
  }
  if (fused) {
    // one kernel: scores into the per-CTA scratch, selection beside them
    if ((size_t)dev.max_smem_optin < dsa::index_topk_smem_bytes(H, D, topk))
      return DSA_ERR_UNSUPPORTED;
    CUtensorMap tm_q, tm_k;
    rc = encode_q(&tm_q, p, dsa::kTileCols / H);
    if (rc != DSA_OK) return rc;
    rc = encode_k(&tm_k, p);
    if (rc != DSA_OK) return rc;
    if (mark(0) != cudaSuccess) return DSA_ERR_CUDA;
    if (dsa::launch_index_topk(p, tm_q, tm_k, topk, logits, out_idx,
                               out_scores, status, dev.num_sms,
                               st) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (mark_rest(1) != cudaSuccess) return DSA_ERR_CUDA;
    return DSA_OK;
  }
  if (mark(0) != cudaSuccess) return DSA_ERR_CUDA;
  if (in_idx) {
    // other H: the given indices read the scores back from full logits
    rc = run_scores(p, logits, status, dev, st, 0, S);
    if (rc != DSA_OK) return rc;
    if (mark(1) != cudaSuccess) return DSA_ERR_CUDA;
    if (dsa::launch_gather_logits(p, logits, in_idx, topk, out_idx,
                                  out_scores, status, dev.num_sms,
                                  st) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (mark_rest(2) != cudaSuccess) return DSA_ERR_CUDA;
    return DSA_OK;
  }
  // scores then selection, one chunk of query rows at a time: the chunk's
  // logits are read back while they are still in L2
  const int rows = logits_chunk_rows(S, B, H, S_kv);
  int ev = 1;
  for (int s0 = 0; s0 < S; s0 += rows) {
    const int sc = S - s0 < rows ? S - s0 : rows;
    rc = run_scores(p, logits, status, dev, st, s0, sc);
    if (rc != DSA_OK) return rc;
    if (mark(ev++) != cudaSuccess) return DSA_ERR_CUDA;
    if (dsa::launch_topk_select(p, logits, topk, out_idx, out_scores,
                                dev.num_sms, st, s0, sc) != cudaSuccess)
      return DSA_ERR_CUDA;
    if (mark(ev++) != cudaSuccess) return DSA_ERR_CUDA;
  }
  if (mark_rest(ev) != cudaSuccess) return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // namespace dsa

extern "C" {

int dsa_indexer_fwd(const void *q, const void *k, const float *w, int S,
                    int B, int H, int D, int S_kv, int compress_ratio,
                    int topk, const int32_t *q_pos, const int32_t *in_idx,
                    int32_t *out_idx, float *out_scores, void *workspace,
                    size_t workspace_bytes, void *cuda_stream) {
  return dsa_indexer_fwd_profiled(q, k, w, S, B, H, D, S_kv, compress_ratio,
                                  topk, q_pos, in_idx, out_idx, out_scores,
                                  workspace, workspace_bytes, cuda_stream,
                                  nullptr, 0);
}

int dsa_indexer_logits(const void *q, const void *k, const float *w, int S,
                       int B, int H, int D, int S_kv, int compress_ratio,
                       const int32_t *q_pos, float *logits, void *workspace,
                       size_t workspace_bytes, void *cuda_stream) {
  if (!q || !k || !w || !logits) return DSA_ERR_INVALID_ARG;
  int rc = check_shape(S, B, H, D, S_kv, compress_ratio);
  if (rc != DSA_OK) return rc;
  if (!aligned16(q) || !aligned16(k)) return DSA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kHeaderBytes) return DSA_ERR_WORKSPACE;
  DeviceInfo dev;
  rc = current_device_info(&dev);
  if (rc != DSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int *status = static_cast<int *>(workspace);
  const Problem p{q, k, w, q_pos, S, B, H, D, S_kv, compress_ratio};
  if (cudaMemsetAsync(status, 0, kHeaderBytes, st) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (dsa::launch_fill_masked(logits, logits_bytes(S, B, S_kv) / 4, st) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  return run_scores(p, logits, status, dev, st, 0, S);
}

int dsa_indexer_check(void *workspace, void *cuda_stream) {
  if (!workspace) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return DSA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  if (word != 0 && cudaMemset(workspace, 0, sizeof word) != cudaSuccess)
    return DSA_ERR_CUDA;
  if (word & dsa::kStatusTimeout) return DSA_ERR_DEVICE_TIMEOUT;
  if (word & dsa::kStatusIndexRange) return DSA_ERR_INDEX_RANGE;
  return DSA_OK;
}

int dsa_selftest_wait_limit(int limit_us, void *workspace,
                            size_t workspace_bytes, void *cuda_stream) {
  if (!workspace || workspace_bytes < kHeaderBytes) return DSA_ERR_WORKSPACE;
  DeviceInfo dev;
  int rc = current_device_info(&dev);
  if (rc != DSA_OK) return rc;
  if (limit_us < 1) limit_us = 1;
  if (limit_us > 1000000) limit_us = 1000000;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int *status = static_cast<int *>(workspace);
  if (cudaMemsetAsync(status, 0, kHeaderBytes, st) != cudaSuccess)
    return DSA_ERR_CUDA;
  return dsa::launch_wait_selftest(limit_us, status, st) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

}  // extern "C"

// ---- wait-limit self-test kernel ---------------------------------------------
namespace dsa {
namespace {

// One warp waits on a barrier that expects an arrival nobody makes; the wait
// gives up after `limit_ns` and records the timeout bit.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(a, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t t0 = globaltimer_ns();
  bool done = false;
  for (uint64_t it = 0; it < kWaitMaxPolls; ++it) {
    if (mbar_try_wait(a, 0)) {
      done = true;
      break;
    }
    if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) break;
  }
  if (!done && threadIdx.x == 0) atomicOr(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(int limit_us, int *status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>((uint64_t)limit_us * 1000ull, status);
  return cudaGetLastError();
}

}  // namespace dsa
