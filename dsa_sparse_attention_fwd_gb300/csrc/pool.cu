// The pool variant of the indexer (page "Module glm5next_dsa", "Shape of
// the pipeline": k, gate, valid, ape -> kpool_compress -> index_scores ->
// topk_pools -> expand_selection -> token ids, -1 = invalid).
//
//   kpool_compress: pool p of sequence b covers tokens first_key + p*kpool
//     + s (s < kpool); only whole pools count (an incomplete pool at the
//     end is dropped), and a pool is a candidate only if all its tokens are
//     valid.  Per channel c, with slot logits z_s = gate[token_s, b, c] +
//     ape[s, c], the pooled key is sum_s softmax_s(z)_s * k[token_s, b, c]
//     (the softmax runs across a pool's slots, separately per channel),
//     computed in fp32 and stored as bf16 (the indexer's key format).
//   index_scores + topk_pools: the lightning-indexer forward over the pools
//     with compress_ratio = kpool at positions shifted by first_key (pool p
//     is visible once its last token is), invalid pools masked out.
//   expand_selection: each row's index_topk / kpool pool ids become
//     index_topk token ids, -1 for the slots of an empty pool slot (the
//     whole output row is filled with -1 first, so no slot is left
//     unwritten).
//
// kpool <= 8: the page's compression kernel holds at most 8 slots
// (KERNEL_MAX_KPOOL) and its configuration refuses more.
#include <cuda_runtime.h>

#include "common.cuh"
#include "dsa_indexer.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kMaxKpool = 8;

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

long long pool_count(int T, int kpool, int first_key) {
  return T > first_key ? (long long)(T - first_key) / kpool : 0;
}

// One thread per (pool, sequence, 4 channels): the KP slots' gate, k and
// position-embedding values are read once (every load issued before the
// first use), the softmax over slots is taken per channel in registers.
// Consecutive threads cover consecutive channels, so every load and store
// is coalesced.
template <int KP>
__global__ void kpool_compress_kernel(
    const uint16_t *__restrict__ k, const float *__restrict__ gate,
    const float *__restrict__ ape, const uint8_t *__restrict__ valid, int B,
    int D, int first_key, long long P, uint16_t *__restrict__ keys,
    uint8_t *__restrict__ pool_valid, const int32_t *__restrict__ q_pos,
    int32_t *__restrict__ q_pos_shifted) {
  constexpr int kpool = KP;  // slots per pool
  if (q_pos_shifted && blockIdx.x == 0)
    for (int b = threadIdx.x; b < B; b += blockDim.x)
      q_pos_shifted[b] = (q_pos ? __ldg(q_pos + b) : 0) - first_key;
  const int D4 = D / 4;
  const long long total = P * B * D4;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       e < total; e += (long long)gridDim.x * blockDim.x) {
    const int c4 = (int)(e % D4);
    const long long pb = e / D4;
    const int b = (int)(pb % B);
    const long long p = pb / B;
    const long long tok0 = first_key + p * kpool;
    float z[KP][4], kv[KP][4];
    float zmax[4] = {-__int_as_float(0x7f800000), -__int_as_float(0x7f800000),
                     -__int_as_float(0x7f800000), -__int_as_float(0x7f800000)};
    bool all_valid = true;
#pragma unroll
    for (int s = 0; s < KP; ++s) {
      const size_t row = (size_t)(tok0 + s) * B + b;
      const float4 g4 =
          __ldg(reinterpret_cast<const float4 *>(gate + row * D) + c4);
      const float4 a4 =
          __ldg(reinterpret_cast<const float4 *>(ape + (size_t)s * D) + c4);
      const uint2 k4 =
          __ldg(reinterpret_cast<const uint2 *>(k + row * D) + c4);
      z[s][0] = g4.x + a4.x;
      z[s][1] = g4.y + a4.y;
      z[s][2] = g4.z + a4.z;
      z[s][3] = g4.w + a4.w;
      kv[s][0] = __uint_as_float(k4.x << 16);
      kv[s][1] = __uint_as_float(k4.x & 0xFFFF0000u);
      kv[s][2] = __uint_as_float(k4.y << 16);
      kv[s][3] = __uint_as_float(k4.y & 0xFFFF0000u);
#pragma unroll
      for (int q = 0; q < 4; ++q) zmax[q] = fmaxf(zmax[q], z[s][q]);
      if (valid && c4 == 0) all_valid &= __ldg(valid + row) != 0;
    }
    float num[4] = {0.f, 0.f, 0.f, 0.f}, den[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < KP; ++s) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float ex = expf(z[s][q] - zmax[q]);
        den[q] += ex;
        num[q] = fmaf(ex, kv[s][q], num[q]);
      }
    }
    uint2 out;
    out.x = pack_bf16x2(num[0] / den[0], num[1] / den[1]);
    out.y = pack_bf16x2(num[2] / den[2], num[3] / den[3]);
    reinterpret_cast<uint2 *>(keys + (size_t)pb * D)[c4] = out;
    if (pool_valid && c4 == 0) pool_valid[pb] = all_valid ? 1 : 0;
  }
}

// Token ids of the selected pools: consecutive threads write consecutive
// slots of a row.
__global__ void expand_selection_kernel(const int32_t *__restrict__ pools,
                                        long long rows, int select_k,
                                        int kpool, int first_key,
                                        int32_t *__restrict__ tokens) {
  const long long width = (long long)select_k * kpool;
  const long long total = rows * width;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       e < total; e += (long long)gridDim.x * blockDim.x) {
    const long long r = e / width;
    const int within = (int)(e % width);
    const int32_t pool = __ldg(pools + r * select_k + within / kpool);
    tokens[e] = pool < 0 ? -1
                         : (int32_t)(first_key + (long long)pool * kpool +
                                     within % kpool);
  }
}

__global__ void fill_neg_inf_f32(float *p, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = -__int_as_float(0x7f800000);
}

int grid_for(long long work) {
  long long g = (work + 255) / 256;
  if (g > 152LL * 16) g = 152LL * 16;
  return g < 1 ? 1 : (int)g;
}

cudaError_t launch_compress(const uint16_t *k, const float *gate,
                            const float *ape, const uint8_t *valid, int B,
                            int D, int kpool, int first_key, long long P,
                            uint16_t *keys, uint8_t *pool_valid,
                            const int32_t *q_pos, int32_t *q_pos_shifted,
                            cudaStream_t st) {
  const int grid = grid_for(P * B * (D / 4));
#define DSA_KP_CASE(N)                                                       \
  case N:                                                                    \
    kpool_compress_kernel<N><<<grid, 256, 0, st>>>(                          \
        k, gate, ape, valid, B, D, first_key, P, keys, pool_valid, q_pos,    \
        q_pos_shifted);                                                      \
    break;
  switch (kpool) {
    DSA_KP_CASE(1)
    DSA_KP_CASE(2)
    DSA_KP_CASE(3)
    DSA_KP_CASE(4)
    DSA_KP_CASE(5)
    DSA_KP_CASE(6)
    DSA_KP_CASE(7)
    DSA_KP_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef DSA_KP_CASE
  return cudaGetLastError();
}

bool al(const void *p, unsigned a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

int check_compress_args(const void *k, const float *gate, const float *ape,
                        int T, int B, int D, int kpool, int first_key) {
  if (!k || !gate || !ape) return DSA_ERR_INVALID_ARG;
  if (T <= 0 || B <= 0 || D <= 0 || kpool <= 0 || first_key < 0)
    return DSA_ERR_INVALID_ARG;
  if (kpool > kMaxKpool || D % 8 != 0 || D > DSA_MAX_D)
    return DSA_ERR_UNSUPPORTED;
  if (!al(k, 16) || !al(gate, 16) || !al(ape, 16)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

}  // namespace
}  // namespace dsa

extern "C" {

int dsa_kpool_compress(const void *k, const float *gate, const float *ape,
                       const uint8_t *valid, int T, int B, int D, int kpool,
                       int first_key, void *out_keys, uint8_t *out_valid,
                       void *cuda_stream) {
  int rc = dsa::check_compress_args(k, gate, ape, T, B, D, kpool, first_key);
  if (rc != DSA_OK) return rc;
  const long long P = dsa::pool_count(T, kpool, first_key);
  if (P == 0) return DSA_OK;
  if (!out_keys || !dsa::al(out_keys, 16)) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  return dsa::launch_compress(static_cast<const uint16_t *>(k), gate, ape,
                              valid, B, D, kpool, first_key, P,
                              static_cast<uint16_t *>(out_keys), out_valid,
                              nullptr, nullptr, st) == cudaSuccess
             ? DSA_OK
             : DSA_ERR_CUDA;
}

int dsa_expand_selection(const int32_t *pools, long long rows, int select_k,
                         int kpool, int first_key, int32_t *out_tokens,
                         void *cuda_stream) {
  if (!pools || !out_tokens || rows < 0 || select_k <= 0 || kpool <= 0 ||
      first_key < 0)
    return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  dsa::expand_selection_kernel<<<dsa::grid_for(rows * select_k * kpool), 256,
                                 0, st>>>(pools, rows, select_k, kpool,
                                          first_key, out_tokens);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_indexer_pooled_workspace_size(int S, int B, int H, int D, int T,
                                         int kpool, int first_key,
                                         int index_topk) {
  if (kpool <= 0 || index_topk <= 0 || index_topk % kpool != 0 ||
      first_key < 0 || T <= 0 || B <= 0 || D <= 0)
    return 0;
  const long long P = dsa::pool_count(T, kpool, first_key);
  if (P == 0) return 256;
  if (P >= (1ll << 31)) return 0;
  const size_t fw = dsa_indexer_workspace_size(S, B, H, D, (int)P, kpool,
                                               index_topk / kpool, 0);
  if (fw == 0) return 0;
  return dsa::up256(fw) + dsa::up256((size_t)P * B * D * 2) +
         dsa::up256((size_t)P * B) + dsa::up256((size_t)B * 4);
}

int dsa_indexer_fwd_pooled(const void *q, const void *k, const float *gate,
                           const float *ape, const uint8_t *valid,
                           const float *w, int S, int B, int H, int D, int T,
                           int kpool, int first_key, int index_topk,
                           const int32_t *q_pos, int32_t *out_tokens,
                           int32_t *out_pools, float *out_scores,
                           void *workspace, size_t workspace_bytes,
                           void *cuda_stream) {
  if (!q || !w || !out_tokens || !out_pools || !out_scores)
    return DSA_ERR_INVALID_ARG;
  int rc = dsa::check_compress_args(k, gate, ape, T, B, D, kpool, first_key);
  if (rc != DSA_OK) return rc;
  if (S <= 0 || H <= 0 || index_topk <= 0) return DSA_ERR_INVALID_ARG;
  if (index_topk % kpool != 0) return DSA_ERR_INVALID_ARG;
  const size_t need = dsa_indexer_pooled_workspace_size(
      S, B, H, D, T, kpool, first_key, index_topk);
  if (need == 0) return DSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need) return DSA_ERR_WORKSPACE;
  if (!dsa::al(workspace, 256)) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int select_k = index_topk / kpool;
  const long long rows = (long long)B * S;
  const long long P = dsa::pool_count(T, kpool, first_key);
  if (P == 0) {
    // no whole pool: every slot is empty
    if (cudaMemsetAsync(workspace, 0, 256, st) != cudaSuccess ||
        cudaMemsetAsync(out_pools, 0xFF, (size_t)rows * select_k * 4, st) !=
            cudaSuccess ||
        cudaMemsetAsync(out_tokens, 0xFF, (size_t)rows * index_topk * 4,
                        st) != cudaSuccess)
      return DSA_ERR_CUDA;
    dsa::fill_neg_inf_f32<<<dsa::grid_for(rows * select_k), 256, 0, st>>>(
        out_scores, rows * select_k);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }
  // workspace: the forward's own (status word first), pooled keys, pool
  // flags, shifted query positions
  const size_t fw = dsa_indexer_workspace_size(S, B, H, D, (int)P, kpool,
                                               select_k, 0);
  char *ws = static_cast<char *>(workspace);
  uint16_t *keys = reinterpret_cast<uint16_t *>(ws + dsa::up256(fw));
  uint8_t *pool_valid = reinterpret_cast<uint8_t *>(
      ws + dsa::up256(fw) + dsa::up256((size_t)P * B * D * 2));
  int32_t *qp = reinterpret_cast<int32_t *>(
      ws + dsa::up256(fw) + dsa::up256((size_t)P * B * D * 2) +
      dsa::up256((size_t)P * B));
  if (dsa::launch_compress(static_cast<const uint16_t *>(k), gate, ape, valid,
                           B, D, kpool, first_key, P, keys, pool_valid, q_pos,
                           qp, st) != cudaSuccess)
    return DSA_ERR_CUDA;
  rc = dsa::forward_core(q, keys, w, S, B, H, D, (int)P, kpool, select_k, qp,
                         nullptr, out_pools, out_scores, workspace, fw, st,
                         nullptr, 0, true, pool_valid);
  if (rc != DSA_OK) return rc;
  dsa::expand_selection_kernel<<<dsa::grid_for(rows * index_topk), 256, 0,
                                 st>>>(out_pools, rows, select_k, kpool,
                                       first_key, out_tokens);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
