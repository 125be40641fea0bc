// dsa_indexer_fwd_host: the forward on host buffers, with the host<->device
// copies pipelined against the kernels.
//
// The query rows are split into chunks along S (rows [s0, s1) of every
// sequence).  One stream copies the inputs in (k and w first, then the q
// rows of each chunk), the caller's stream runs each chunk's forward as
// soon as its rows have landed, and a third stream copies each chunk's
// indices and scores back while the next chunks are scored.  Under the
// causal mask a chunk's cost grows with its rows' positions while its
// copies do not, so the chunk order matters:
//  - link-bound shapes (few visible keys per copied byte) take the last
//    rows first, so the chunk left after the last copy is the cheapest;
//  - compute-bound shapes alternate the costliest and the cheapest chunk
//    left (last, first, second last, second, ...): taken last rows first,
//    their cheap chunks at the end finish scoring faster than their results
//    can be copied out and the copies back up behind the kernels.
// Chunk starts fall on whole waves of work items where the chunks hold at
// least one.  Every row's result is bit-identical to one unchunked call: no
// row's arithmetic depends on the other rows.  A chunk after the first
// sees its rows through per-chunk query positions (q_pos[b] + s0, or s0 for
// prefill).
//
// Device memory is the caller's buffer (dsa_indexer_host_buffer_size()
// bytes): [k][q][w][positions][given indices][indices][scores][status]
// [workspace], each region 256-byte aligned; per-chunk index, output and
// status regions are contiguous [B, rows of the chunk, topk] blocks.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "dsa_indexer.h"

namespace {

constexpr int kMaxChunks = 16;
constexpr int kMinChunkRows = 512;  // keeps each chunk's launch busy

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Chunks along S: as many as there are kMinChunkRows-row blocks, at most
// kMaxChunks (chunk_start places them).
int plan_chunks(int S) {
  int c = S / kMinChunkRows;
  if (c > kMaxChunks) c = kMaxChunks;
  return c < 1 ? 1 : c;
}

// Query rows per wave of prefill work items on a GPU of `sms` SMs (the
// current device's when sms <= 0; one item is 256/H rows of one sequence,
// one CTA per SM): chunk starts on whole waves leave no part-filled last
// wave in each chunk's launch.  4 when unknown.
int wave_rows(int B, int H, int sms) {
  int dev = 0;
  if (sms <= 0 &&
      (cudaGetDevice(&dev) != cudaSuccess ||
       cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
           cudaSuccess))
    sms = 0;
  if (sms <= 0 || H <= 0 || B <= 0) return 4;
  const long long tq = H < 256 ? 256 / H : 1;
  const long long u = ((long long)sms * tq / B) & ~3ll;
  return u < 4 ? 4 : (u > (1 << 20) ? (1 << 20) : (int)u);
}

// Start of chunk i: an even split, on a multiple of 4 rows, moved to the
// nearest whole wave of `unit` rows when the chunks hold at least one
// (starts then still increase and stay below S).
int chunk_start(int S, int chunks, int i, int unit) {
  if (i >= chunks) return S;
  long long s = (long long)S * i / chunks;
  if (unit > 4 && S / chunks >= unit)
    s = (s + unit / 2) / unit * unit;
  else
    s &= ~3ll;
  return (int)s;
}

// Tensor-core FLOPs the kernels run per byte crossing the host link, above
// which the pipeline is compute-bound: about the one-kernel forward's rate
// (1.3 PFLOP/s) over the link's rate with copies both ways (0.34 TB/s),
// discounted.
constexpr double kComputeBoundFlopPerByte = 3000.0;

// Processing order of the chunks (see the file comment): ord[n] is the
// n-th chunk to copy in, score and copy out.  The cost estimate takes each
// chunk's middle row per sequence as its average row.
void chunk_order(int S, int B, int H, int D, int S_kv, int ratio, int topk,
                 const int32_t *q_pos, bool has_in_idx, int C, int unit,
                 int *ord) {
  double flops = 0.0;
  for (int i = 0; i < C; ++i) {
    const int s0 = chunk_start(S, C, i, unit);
    const int s1 = chunk_start(S, C, i + 1, unit);
    const int mid = s0 + (s1 - s0) / 2;
    for (int b = 0; b < B; ++b) {
      const long long pos = (q_pos ? (long long)q_pos[b] : 0) + mid;
      int n = dsa::n_visible(pos, ratio, S_kv);
      if (has_in_idx && n > topk) n = topk;
      flops += 2.0 * H * D * (double)n * (s1 - s0);
    }
  }
  // q and w in, indices and scores out (and given indices in)
  const double bytes = (double)S * B * ((double)H * D * 2 + (double)H * 4 +
                                        (double)topk * (has_in_idx ? 12 : 8));
  const bool alternate = flops > kComputeBoundFlopPerByte * bytes;
  int lo = 0, hi = C - 1;
  for (int n = 0; n < C; ++n) {
    if (!alternate || (n & 1) == 0)
      ord[n] = hi--;
    else
      ord[n] = lo++;
  }
}

struct HostLayout {
  int chunks = 1, max_rows = 0, unit = 4;
  size_t k = 0, q = 0, w = 0, pos = 0, in_idx = 0, out_idx = 0, out_sc = 0,
         status = 0, ws = 0, ws_bytes = 0, total = 0;
};

HostLayout host_layout(int S, int B, int H, int D, int S_kv, int ratio,
                       int topk, bool has_in_idx, int sms = 0) {
  HostLayout L;
  L.chunks = plan_chunks(S);
  L.unit = wave_rows(B, H, sms);
  for (int i = 0; i < L.chunks; ++i) {
    const int r = chunk_start(S, L.chunks, i + 1, L.unit) -
                  chunk_start(S, L.chunks, i, L.unit);
    if (r > L.max_rows) L.max_rows = r;
  }
  L.ws_bytes = dsa_indexer_workspace_size(L.max_rows, B, H, D, S_kv, ratio,
                                          topk, has_in_idx ? 1 : 0);
  if (L.ws_bytes == 0) return HostLayout{};
  const size_t rows_topk = (size_t)B * S * topk * 4;
  size_t o = 0;
  L.k = o;       o += up256((size_t)S_kv * B * D * 2);
  L.q = o;       o += up256((size_t)S * B * H * D * 2);
  L.w = o;       o += up256((size_t)S * B * H * 4);
  L.pos = o;     o += up256((size_t)L.chunks * B * 4);
  L.in_idx = o;  o += has_in_idx ? up256(rows_topk) : 0;
  L.out_idx = o; o += up256(rows_topk);
  L.out_sc = o;  o += up256(rows_topk);
  L.status = o;  o += 256;
  L.ws = o;      o += up256(L.ws_bytes);
  L.total = o;
  return L;
}

struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_done[kMaxChunks] = {},
              fwd_done[kMaxChunks] = {}, out_done = nullptr;
  // page-locked staging for the per-chunk query positions and the status
  // words (so their copies stay asynchronous); grows to the largest call
  int32_t *staging = nullptr;
  size_t staging_ints = 0;
  std::mutex call;  // one host-buffer call per device at a time
};

// Page-locked staging with room for n ints (reused: calls are synchronous).
int staging_for(Pipe &p, size_t n) {
  if (p.staging_ints >= n) return DSA_OK;
  if (p.staging && cudaFreeHost(p.staging) != cudaSuccess) return DSA_ERR_CUDA;
  p.staging = nullptr;
  p.staging_ints = 0;
  size_t cap = 1024;
  while (cap < n) cap *= 2;
  void *h = nullptr;
  if (cudaHostAlloc(&h, cap * sizeof(int32_t), cudaHostAllocDefault) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  p.staging = static_cast<int32_t *>(h);
  p.staging_ints = cap;
  return DSA_OK;
}

std::mutex g_pipes_mu;
Pipe g_pipes[64];

// The device's copy streams and events, created on first use.
int get_pipe(Pipe **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_pipes_mu);
  Pipe &p = g_pipes[dev];
  if (!p.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) !=
            cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) !=
            cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.out_done, ef) != cudaSuccess)
      return DSA_ERR_CUDA;
    for (int i = 0; i < kMaxChunks; ++i)
      if (cudaEventCreateWithFlags(&p.in_done[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.fwd_done[i], ef) != cudaSuccess)
        return DSA_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_indexer_host_plan(int S, int B, int H, int D, int S_kv,
                          int compress_ratio, int topk, const int32_t *q_pos,
                          int has_in_idx, int sms, int *starts, int *order) {
  if (!starts || !order) return 0;
  if (dsa_indexer_workspace_size(S, B, H, D, S_kv, compress_ratio, topk,
                                 has_in_idx) == 0)
    return 0;
  const HostLayout L = host_layout(S, B, H, D, S_kv, compress_ratio, topk,
                                   has_in_idx != 0, sms);
  for (int i = 0; i <= L.chunks; ++i)
    starts[i] = chunk_start(S, L.chunks, i, L.unit);
  chunk_order(S, B, H, D, S_kv, compress_ratio, topk, q_pos, has_in_idx != 0,
              L.chunks, L.unit, order);
  return L.chunks;
}

size_t dsa_indexer_host_buffer_size(int S, int B, int H, int D, int S_kv,
                                    int compress_ratio, int topk,
                                    int has_in_idx) {
  if (dsa_indexer_workspace_size(S, B, H, D, S_kv, compress_ratio, topk,
                                 has_in_idx) == 0)
    return 0;
  return host_layout(S, B, H, D, S_kv, compress_ratio, topk, has_in_idx != 0)
      .total;
}

int dsa_indexer_fwd_host(const void *q, const void *k, const float *w, int S,
                         int B, int H, int D, int S_kv, int compress_ratio,
                         int topk, const int32_t *q_pos,
                         const int32_t *in_idx, int32_t *out_idx,
                         float *out_scores, void *device_buf,
                         size_t device_buf_bytes, void *cuda_stream) {
  if (!q || !k || !w || !out_idx || !out_scores) return DSA_ERR_INVALID_ARG;
  const size_t need = dsa_indexer_host_buffer_size(
      S, B, H, D, S_kv, compress_ratio, topk, in_idx != nullptr);
  if (need == 0) {
    // the forward's own checks name the problem
    return S <= 0 || B <= 0 || H <= 0 || D <= 0 || S_kv <= 0 ||
                   compress_ratio <= 0 || topk <= 0
               ? DSA_ERR_INVALID_ARG
               : DSA_ERR_UNSUPPORTED;
  }
  if (!device_buf || device_buf_bytes < need) return DSA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(device_buf) & 255u) != 0)
    return DSA_ERR_INVALID_ARG;
  const HostLayout L = host_layout(S, B, H, D, S_kv, compress_ratio, topk,
                                   in_idx != nullptr);
  Pipe *pp = nullptr;
  int rc = get_pipe(&pp);
  if (rc != DSA_OK) return rc;
  std::lock_guard<std::mutex> call_lock(pp->call);
  Pipe &P = *pp;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  char *base = static_cast<char *>(device_buf);
  const int C = L.chunks;
  const size_t q_row = (size_t)B * H * D * 2, w_row = (size_t)B * H * 4;
  const size_t topk4 = (size_t)topk * 4;

  // staging: [0, kMaxChunks) status words, then C x B query positions
  const bool chunk_pos = C > 1 || q_pos != nullptr;
  rc = staging_for(P, kMaxChunks + (size_t)C * B);
  if (rc != DSA_OK) return rc;
  int32_t *words = P.staging, *pos_h = P.staging + kMaxChunks;
  if (chunk_pos)
    for (int i = 0; i < C; ++i)
      for (int b = 0; b < B; ++b)
        pos_h[(size_t)i * B + b] =
            (q_pos ? q_pos[b] : 0) + chunk_start(S, C, i, L.unit);
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  int ord[kMaxChunks];
  chunk_order(S, B, H, D, S_kv, compress_ratio, topk, q_pos,
              in_idx != nullptr, C, L.unit, ord);

  // inputs: k, w, positions, then each chunk's q rows (and given indices)
  chk(cudaEventRecord(P.start, st));
  chk(cudaStreamWaitEvent(P.in, P.start, 0));
  chk(cudaMemcpyAsync(base + L.k, k, (size_t)S_kv * B * D * 2,
                      cudaMemcpyHostToDevice, P.in));
  chk(cudaMemcpyAsync(base + L.w, w, (size_t)S * w_row,
                      cudaMemcpyHostToDevice, P.in));
  if (chunk_pos)
    chk(cudaMemcpyAsync(base + L.pos, pos_h, (size_t)C * B * 4,
                        cudaMemcpyHostToDevice, P.in));
  for (int n = 0; n < C && ok; ++n) {
    const int i = ord[n];
    const int s0 = chunk_start(S, C, i, L.unit);
    const int rows = chunk_start(S, C, i + 1, L.unit) - s0;
    chk(cudaMemcpyAsync(base + L.q + (size_t)s0 * q_row,
                        static_cast<const char *>(q) + (size_t)s0 * q_row,
                        (size_t)rows * q_row, cudaMemcpyHostToDevice, P.in));
    if (in_idx)  // [B, S, topk] rows s0.. -> a contiguous [B, rows, topk]
      chk(cudaMemcpy2DAsync(base + L.in_idx + (size_t)B * s0 * topk4,
                            (size_t)rows * topk4, in_idx + (size_t)s0 * topk,
                            (size_t)S * topk4, (size_t)rows * topk4, B,
                            cudaMemcpyHostToDevice, P.in));
    chk(cudaEventRecord(P.in_done[i], P.in));
  }

  // each chunk's forward on the caller's stream, then its results out
  for (int n = 0; n < C && ok; ++n) {
    const int i = ord[n];
    const int s0 = chunk_start(S, C, i, L.unit);
    const int rows = chunk_start(S, C, i + 1, L.unit) - s0;
    chk(cudaStreamWaitEvent(st, P.in_done[i], 0));
    if (!ok) break;
    const size_t oo = (size_t)B * s0 * topk4;  // chunk block offset
    const int32_t *pos_d =
        chunk_pos
            ? reinterpret_cast<const int32_t *>(base + L.pos) + (size_t)i * B
            : nullptr;
    rc = dsa_indexer_fwd(
        base + L.q + (size_t)s0 * q_row, base + L.k,
        reinterpret_cast<const float *>(base + L.w + (size_t)s0 * w_row),
        rows, B, H, D, S_kv, compress_ratio, topk, pos_d,
        in_idx ? reinterpret_cast<const int32_t *>(base + L.in_idx + oo)
               : nullptr,
        reinterpret_cast<int32_t *>(base + L.out_idx + oo),
        reinterpret_cast<float *>(base + L.out_sc + oo), base + L.ws,
        L.ws_bytes, st);
    if (rc != DSA_OK) break;
    // keep the chunk's device status (the next chunk clears the header)
    chk(cudaMemcpyAsync(base + L.status + 4 * i, base + L.ws, 4,
                        cudaMemcpyDeviceToDevice, st));
    chk(cudaEventRecord(P.fwd_done[i], st));
    chk(cudaStreamWaitEvent(P.out, P.fwd_done[i], 0));
    chk(cudaMemcpy2DAsync(out_idx + (size_t)s0 * topk, (size_t)S * topk4,
                          base + L.out_idx + oo, (size_t)rows * topk4,
                          (size_t)rows * topk4, B, cudaMemcpyDeviceToHost,
                          P.out));
    chk(cudaMemcpy2DAsync(out_scores + (size_t)s0 * topk, (size_t)S * topk4,
                          base + L.out_sc + oo, (size_t)rows * topk4,
                          (size_t)rows * topk4, B, cudaMemcpyDeviceToHost,
                          P.out));
  }
  // join the copy streams back into the caller's stream and wait
  chk(cudaEventRecord(P.out_done, P.out));
  chk(cudaStreamWaitEvent(st, P.out_done, 0));
  chk(cudaMemcpyAsync(words, base + L.status, (size_t)C * 4,
                      cudaMemcpyDeviceToHost, st));
  chk(cudaStreamSynchronize(st));
  if (rc != DSA_OK) return rc;
  if (!ok) return DSA_ERR_CUDA;
  int word = 0;
  for (int i = 0; i < C; ++i) word |= words[i];
  if (word & dsa::kStatusTimeout) return DSA_ERR_DEVICE_TIMEOUT;
  if (word & dsa::kStatusIndexRange) return DSA_ERR_INDEX_RANGE;
  return DSA_OK;
}

}  // extern "C"
