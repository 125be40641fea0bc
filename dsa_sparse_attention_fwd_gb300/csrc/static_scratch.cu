// An indexer forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs while a caching
// allocator owns all free memory, plugin hosts that hand out only the
// tensors they manage, and hot paths where an allocation would synchronise
// the device.  For them this entry point runs the same forward as
// dsa_indexer_fwd() with its scratch (the status header, then per-CTA score
// rows of the one-kernel prefill or the fp32 logits of the other shapes)
// taken from a fixed array in this file instead of a caller workspace.
//
// A top-k prefill whose one-kernel scratch (per-CTA score rows, which grow
// with S_kv) does not fit the array runs scores then selection instead:
// that path's logits chunk is at most 64 MiB, so every top-k prefill fits.
//
// The array is a file-scope __device__ variable: each GPU on which this
// library's module is loaded holds its own copy until the process exits.
// Host code cannot use the array's name as a device address (on the host
// the name is only a stand-in), so the device address is looked up with
// cudaGetSymbolAddress on every call, with the caller's device current.  The
// lookup allocates nothing and is cheap; not caching it keeps the address
// right after a device reset or a reload of the module, where the array may
// move.
#include "common.cuh"
#include "dsa_indexer.h"

namespace {

static __device__ __align__(256) unsigned char
    g_static_scratch[DSA_STATIC_SCRATCH_BYTES];

// Device address of the current device's copy of the scratch array.
int static_scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p)
    return DSA_ERR_CUDA;
  *out = p;
  return DSA_OK;
}

}  // namespace

extern "C" int dsa_indexer_fwd_static_scratch(
    const void *q, const void *k, const float *w, int S, int B, int H, int D,
    int S_kv, int compress_ratio, int topk, const int32_t *q_pos,
    const int32_t *in_idx, int32_t *out_idx, float *out_scores,
    int32_t *out_status, void *cuda_stream) {
  size_t need = dsa_indexer_workspace_size(
      S, B, H, D, S_kv, compress_ratio, topk, in_idx != nullptr);
  if (need == 0)  // invalid shape: report the forward's own argument error
    return dsa_indexer_fwd(q, k, w, S, B, H, D, S_kv, compress_ratio, topk,
                           q_pos, in_idx, out_idx, out_scores, nullptr, 0,
                           cuda_stream);
  bool one_kernel_ok = true;
  if (need > (size_t)DSA_STATIC_SCRATCH_BYTES && !in_idx) {
    // too long for the one-kernel forward's score rows: scores then
    // selection, a bounded chunk of rows at a time
    need = dsa::two_kernel_workspace_bytes(S, B, H, S_kv);
    one_kernel_ok = false;
  }
  if (need > (size_t)DSA_STATIC_SCRATCH_BYTES) return DSA_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  int rc = static_scratch_address(&scratch);
  if (rc != DSA_OK) return rc;
  // The forward clears the status header itself before its kernels run;
  // the rest of the array needs no clearing (every entry that is read was
  // written earlier in the same call).
  rc = dsa::forward_core(q, k, w, S, B, H, D, S_kv, compress_ratio, topk,
                         q_pos, in_idx, out_idx, out_scores, scratch,
                         (size_t)DSA_STATIC_SCRATCH_BYTES, cuda_stream,
                         nullptr, 0, true, nullptr, one_kernel_ok);
  if (rc != DSA_OK) return rc;
  if (out_status &&
      cudaMemcpyAsync(out_status, scratch, sizeof(int32_t),
                      cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(cuda_stream)) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}
