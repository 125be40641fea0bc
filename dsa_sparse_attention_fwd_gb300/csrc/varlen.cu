// dsa_indexer_fwd_varlen: the forward over packed variable-length sequences
// (the "packed-sequence dispatch" of the DeepSeek-V4 indexer adaptation on
// the NeMo AutoModel "tilelang_indexer" page; the pages give no layout, so
// this is the usual packed one: cu_seqlens offsets into one token axis).
//
// Sequence i owns query rows [cu_q[i], cu_q[i+1]) of q [T, H, D], w [T, H]
// and the outputs [T, topk], and compressed keys [cu_k[i], cu_k[i+1]) of
// k [T_kv, D].  Its query row s sits at position q_pos[i] + s (s without
// q_pos), and the indices it returns are local to its own keys.
//
// Each sequence is one B = 1 forward at offset pointers, so every kernel
// is the batched path's.  Sequences run on up to kVarlenSlices streams at
// once (the caller's stream and library-owned ones), each with its own
// slice of the workspace; sequences are assigned longest first to the least
// loaded slice.  The caller's workspace size sets how many slices there
// are.  Every slice's status word is cleared once and then accumulates; at
// the end a one-thread kernel ORs them into the first slice's word, which
// dsa_indexer_check() reads.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "dsa_indexer.h"

namespace {

constexpr int kVarlenSlices = 4;

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Checks the offsets (host arrays of N + 1 entries, starting at 0,
// non-decreasing) and returns the largest per-sequence workspace (0 when
// the shapes are invalid) and the number of sequences with query rows.
int varlen_plan(int N, const int32_t *cu_q, const int32_t *cu_k, int H, int D,
                int ratio, int topk, bool has_in_idx, size_t *slice_bytes,
                int *busy) {
  if (N <= 0 || !cu_q || !cu_k) return DSA_ERR_INVALID_ARG;
  if (cu_q[0] != 0 || cu_k[0] != 0) return DSA_ERR_INVALID_ARG;
  size_t mx = 256;
  int n = 0;
  for (int i = 0; i < N; ++i) {
    const int S = cu_q[i + 1] - cu_q[i], S_kv = cu_k[i + 1] - cu_k[i];
    if (S < 0 || S_kv < 0) return DSA_ERR_INVALID_ARG;
    if (S == 0) continue;
    ++n;
    if (S_kv == 0) continue;  // rows without keys are filled, not scored
    const size_t ws = dsa_indexer_workspace_size(S, 1, H, D, S_kv, ratio,
                                                 topk, has_in_idx ? 1 : 0);
    if (ws == 0) return DSA_ERR_UNSUPPORTED;
    mx = std::max(mx, ws);
  }
  *slice_bytes = up256(mx);
  *busy = n;
  return DSA_OK;
}

struct VarlenStreams {
  bool ready = false;
  cudaStream_t side[kVarlenSlices] = {};
  cudaEvent_t start = nullptr, done[kVarlenSlices] = {};
  std::mutex call;  // one varlen call per device at a time
};

std::mutex g_varlen_mu;
VarlenStreams g_varlen[64];

int get_varlen_streams(VarlenStreams **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_varlen_mu);
  VarlenStreams &v = g_varlen[dev];
  if (!v.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaEventCreateWithFlags(&v.start, ef) != cudaSuccess)
      return DSA_ERR_CUDA;
    for (int i = 1; i < kVarlenSlices; ++i)
      if (cudaStreamCreateWithFlags(&v.side[i], cudaStreamNonBlocking) !=
              cudaSuccess ||
          cudaEventCreateWithFlags(&v.done[i], ef) != cudaSuccess)
        return DSA_ERR_CUDA;
    v.ready = true;
  }
  *out = &v;
  return DSA_OK;
}

// ORs the status words of slices 1.. into slice 0's.
__global__ void merge_status_kernel(char *ws, int slices, size_t slice_bytes) {
  int word = 0;
  for (int s = 0; s < slices; ++s)
    word |= *reinterpret_cast<const int *>(ws + (size_t)s * slice_bytes);
  *reinterpret_cast<int *>(ws) = word;
}

}  // namespace

extern "C" {

size_t dsa_indexer_varlen_workspace_size(int N, const int32_t *cu_seqlens_q,
                                         const int32_t *cu_seqlens_k, int H,
                                         int D, int compress_ratio, int topk,
                                         int has_in_idx) {
  size_t slice = 0;
  int busy = 0;
  if (varlen_plan(N, cu_seqlens_q, cu_seqlens_k, H, D, compress_ratio, topk,
                  has_in_idx != 0, &slice, &busy) != DSA_OK)
    return 0;
  const int slices = std::max(1, std::min(kVarlenSlices, busy));
  return (size_t)slices * slice;
}

int dsa_indexer_fwd_varlen(const void *q, const void *k, const float *w,
                           int N, const int32_t *cu_seqlens_q,
                           const int32_t *cu_seqlens_k, int H, int D,
                           int compress_ratio, int topk, const int32_t *q_pos,
                           const int32_t *in_idx, int32_t *out_idx,
                           float *out_scores, void *workspace,
                           size_t workspace_bytes, void *cuda_stream) {
  if (!q || !k || !w || !out_idx || !out_scores) return DSA_ERR_INVALID_ARG;
  if (topk <= 0 || compress_ratio <= 0) return DSA_ERR_INVALID_ARG;
  size_t slice = 0;
  int busy = 0;
  int rc = varlen_plan(N, cu_seqlens_q, cu_seqlens_k, H, D, compress_ratio,
                       topk, in_idx != nullptr, &slice, &busy);
  if (rc != DSA_OK) return rc;
  if (!workspace || workspace_bytes < slice) return DSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return DSA_ERR_INVALID_ARG;
  const int slices = (int)std::max<size_t>(
      1, std::min<size_t>({(size_t)kVarlenSlices, (size_t)std::max(1, busy),
                           workspace_bytes / slice}));
  VarlenStreams *vp = nullptr;
  rc = get_varlen_streams(&vp);
  if (rc != DSA_OK) return rc;
  std::lock_guard<std::mutex> call_lock(vp->call);
  VarlenStreams &V = *vp;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  char *ws = static_cast<char *>(workspace);
  auto stream_of = [&](int s) { return s == 0 ? st : V.side[s]; };

  // every slice's status word starts at zero and then accumulates
  for (int s = 0; s < slices; ++s)
    if (cudaMemsetAsync(ws + (size_t)s * slice, 0, 256, st) != cudaSuccess)
      return DSA_ERR_CUDA;
  if (slices > 1) {
    if (cudaEventRecord(V.start, st) != cudaSuccess) return DSA_ERR_CUDA;
    for (int s = 1; s < slices; ++s)
      if (cudaStreamWaitEvent(V.side[s], V.start, 0) != cudaSuccess)
        return DSA_ERR_CUDA;
  }

  // longest (most scoring work) first, each to the least loaded slice
  std::vector<int> order;
  for (int i = 0; i < N; ++i)
    if (cu_seqlens_q[i + 1] > cu_seqlens_q[i]) order.push_back(i);
  auto cost = [&](int i) {
    return (double)(cu_seqlens_q[i + 1] - cu_seqlens_q[i]) *
           (double)std::max(1, cu_seqlens_k[i + 1] - cu_seqlens_k[i]);
  };
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return cost(a) > cost(b); });
  std::vector<double> load(slices, 0.0);
  const size_t q_row = (size_t)H * D * 2, k_row = (size_t)D * 2;
  for (int i : order) {
    const int s = (int)(std::min_element(load.begin(), load.end()) -
                        load.begin());
    load[s] += cost(i);
    cudaStream_t ss = stream_of(s);
    const int r0 = cu_seqlens_q[i], S = cu_seqlens_q[i + 1] - r0;
    const int k0 = cu_seqlens_k[i], S_kv = cu_seqlens_k[i + 1] - k0;
    int32_t *oi = out_idx + (size_t)r0 * topk;
    float *os = out_scores + (size_t)r0 * topk;
    const int32_t *gi = in_idx ? in_idx + (size_t)r0 * topk : nullptr;
    if (S_kv == 0) {
      // no keys: every slot is -1 / -inf (given indices are copied through)
      const size_t n = (size_t)S * topk;
      const cudaError_t e =
          gi ? cudaMemcpyAsync(oi, gi, n * 4, cudaMemcpyDeviceToDevice, ss)
             : cudaMemsetAsync(oi, 0xFF, n * 4, ss);
      if (e != cudaSuccess || dsa::launch_fill_masked(os, n, ss) != cudaSuccess)
        return DSA_ERR_CUDA;
      continue;
    }
    rc = dsa::forward_core(
        static_cast<const char *>(q) + (size_t)r0 * q_row,
        static_cast<const char *>(k) + (size_t)k0 * k_row,
        w + (size_t)r0 * H, S, 1, H, D, S_kv, compress_ratio, topk,
        q_pos ? q_pos + i : nullptr, gi, oi, os, ws + (size_t)s * slice,
        slice, ss, nullptr, 0, false);
    if (rc != DSA_OK) break;
  }
  // join the slices back into the caller's stream, then merge the status
  for (int s = 1; s < slices; ++s)
    if (cudaEventRecord(V.done[s], V.side[s]) != cudaSuccess ||
        cudaStreamWaitEvent(st, V.done[s], 0) != cudaSuccess)
      return DSA_ERR_CUDA;
  if (rc != DSA_OK) return rc;
  if (slices > 1) {
    merge_status_kernel<<<1, 1, 0, st>>>(ws, slices, slice);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // extern "C"
