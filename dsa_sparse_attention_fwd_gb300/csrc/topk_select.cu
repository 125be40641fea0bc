// topk_select: per query row, the `topk` visible keys with the largest score,
// sorted by descending score with equal scores ordered by ascending key
// index; the rest of the row is -1 / -inf.
//
// One CTA (8 warps) per row.  The row's n visible fp32 scores are staged in
// shared memory as order-preserving unsigned keys (larger float <-> larger
// key; -0.0 folded onto +0.0 so the index tie-break decides between them).
//   1. When n > topk, a most-significant-digit-first radix select (four 8-bit
//      digits; histogram updates aggregated per warp with match_any) finds T,
//      the topk-th largest key, and an ordered two-walk compaction keeps every
//      key > T and the lowest-index keys == T, in index order.
//   2. A stable least-significant-digit radix sort (four 8-bit digits,
//      descending) orders the m = min(n, topk) survivors, packed as
//      (key << 32 | j).  Stability keeps equal keys in index order, which is
//      exactly the "lower index first" tie rule.  A pass whose digit is the
//      same for every element is skipped.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kMaxEpt = DSA_SEL_MAX_EPT;  // elements per lane per sort pass

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 -> +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

struct SelShared {
  uint32_t whist[kSelWarps][256];  // per-warp digit counts / offsets
  uint32_t hist[256];              // block histogram / digit bases
  uint32_t wsum[kSelWarps];
  uint32_t wgt[kSelWarps], weq[kSelWarps];
  uint32_t sel_digit, sel_above;
  int skip;
};

// Exclusive prefix sum of one value per thread over the 256-thread block.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  uint32_t pre = 0;
#pragma unroll
  for (int w = 0; w < kSelWarps; ++w)
    if (w < warp) pre += sh.wsum[w];
  return pre + incl - v;
}

// One stable counting-sort pass on digit (key >> shift) & 255, descending.
// Returns true when the pass moved data into dst, false when every element
// has the same digit (then src already holds the pass's result).
__device__ __forceinline__ bool lsd_pass(const uint64_t *src, uint64_t *dst,
                                         int m, int shift, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int tid = threadIdx.x;
  const int per_warp = ((m + kSelThreads - 1) / kSelThreads) * 32;
  const int ept = per_warp / 32;
  const int seg = warp * per_warp;
  uint32_t *wh = sh.whist[warp];
  const uint32_t lt = lanemask_lt();
  for (int i = lane; i < 256; i += 32) wh[i] = 0;
  __syncwarp();
  uint32_t off[kMaxEpt];
#pragma unroll
  for (int it = 0; it < kMaxEpt; ++it) {
    if (it < ept) {
      const int e = seg + it * 32 + lane;
      const bool valid = e < m;
      const uint64_t v = valid ? src[e] : 0ull;
      const uint32_t d =
          valid ? 255u - (uint32_t)((v >> (32 + shift)) & 255u) : 256u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      const uint32_t rank = __popc(peers & lt);
      const uint32_t base = valid ? wh[d] : 0u;
      __syncwarp();
      if (valid && rank == 0) wh[d] = base + __popc(peers);
      __syncwarp();
      off[it] = base + rank;
    }
  }
  if (tid == 0) sh.skip = 0;
  __syncthreads();
  {
    const int d = tid;  // 256 threads, one digit each
    uint32_t run = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      const uint32_t c = sh.whist[w][d];
      sh.whist[w][d] = run;
      run += c;
    }
    if (run == (uint32_t)m) sh.skip = 1;
    const uint32_t b = block_excl_scan(run, sh);
    sh.hist[d] = b;
  }
  __syncthreads();
  const bool skip = sh.skip != 0;
  __syncthreads();  // everyone has read the flag before it is reset
  if (skip) return false;  // block-uniform
#pragma unroll
  for (int it = 0; it < kMaxEpt; ++it) {
    if (it < ept) {
      const int e = seg + it * 32 + lane;
      if (e < m) {
        const uint64_t v = src[e];
        const uint32_t d = 255u - (uint32_t)((v >> (32 + shift)) & 255u);
        dst[sh.hist[d] + wh[d] + off[it]] = v;
      }
    }
  }
  __syncthreads();
  return true;
}

__global__ void __launch_bounds__(kSelThreads)
    topk_select_kernel(const float *__restrict__ logits,
                       const int32_t *__restrict__ q_pos, int S, int S_kv,
                       int ratio, int topk, int mcap,
                       int32_t *__restrict__ out_idx,
                       float *__restrict__ out_scores) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t *bufA = reinterpret_cast<uint64_t *>(smem);      // [mcap]
  uint64_t *bufB = bufA + mcap;                              // [mcap]
  uint32_t *keys = reinterpret_cast<uint32_t *>(bufB + mcap);  // [S_kv]
  __shared__ SelShared sh;

  const int row = blockIdx.x;  // row id = b * S + s, the output order
  const int b = row / S, s = row % S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = n_visible(row_pos(q_pos, b, s), ratio, S_kv);
  const float *L = logits + (size_t)row * S_kv;
  const int m = nv < topk ? nv : topk;
  const uint32_t lt = lanemask_lt();

  if (nv <= topk) {
    for (int j = tid; j < nv; j += kSelThreads)
      bufA[j] = ((uint64_t)ordered_key(__ldg(L + j)) << 32) | (uint32_t)j;
    __syncthreads();
  } else {
    for (int j = tid; j < nv; j += kSelThreads)
      keys[j] = ordered_key(__ldg(L + j));
    __syncthreads();
    // ---- radix select of T, the topk-th largest key ----
    uint32_t prefix = 0, pmask = 0;
    int need = topk;  // still to take among keys matching prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
      sh.hist[tid] = 0;
      __syncthreads();
      for (int c0 = 0; c0 < nv; c0 += kSelThreads) {
        const int j = c0 + tid;
        const uint32_t u = j < nv ? keys[j] : 0u;
        const bool ok = j < nv && (u & pmask) == prefix;
        const uint32_t d = ok ? (u >> shift) & 255u : 256u;
        const uint32_t peers = __match_any_sync(0xffffffffu, d);
        if (ok && (peers & lt) == 0) atomicAdd(&sh.hist[d], __popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits [8l, 8l+8); find the largest digit d with
        // count(digit >= d) >= need
        uint32_t c[8];
        uint32_t lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = sh.hist[lane * 8 + i];
          lsum += c[i];
        }
        uint32_t incl = lsum;  // inclusive suffix sum over lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t o = __shfl_down_sync(0xffffffffu, incl, off);
          if (lane + off < 32) incl += o;
        }
        const uint32_t above = incl - lsum;
        if (above < (uint32_t)need && (uint32_t)need <= incl) {
          uint32_t run = above;
          for (int i = 7; i >= 0; --i) {
            if (run + c[i] >= (uint32_t)need) {
              sh.sel_digit = (uint32_t)(lane * 8 + i);
              sh.sel_above = run;
              break;
            }
            run += c[i];
          }
        }
      }
      __syncthreads();
      need -= (int)sh.sel_above;
      prefix |= sh.sel_digit << shift;
      pmask |= 255u << shift;
      __syncthreads();
    }
    const uint32_t T = prefix;
    const int n_gt = topk - need;  // keys strictly above T, all kept

    // ---- ordered compaction, two walks over contiguous warp segments ----
    const int seg = ((nv + kSelThreads - 1) / kSelThreads) * 32;
    const int lo = warp * seg, hi = min(nv, lo + seg);
    uint32_t cgt = 0, ceq = 0;
    for (int c = lo; c < lo + seg; c += 32) {
      const int j = c + lane;
      const uint32_t u = j < hi ? keys[j] : 0u;
      cgt += __popc(__ballot_sync(0xffffffffu, j < hi && u > T));
      ceq += __popc(__ballot_sync(0xffffffffu, j < hi && u == T));
    }
    if (lane == 0) {
      sh.wgt[warp] = cgt;
      sh.weq[warp] = ceq;
    }
    __syncthreads();
    uint32_t gpos = 0, epos = 0;
    for (int w = 0; w < warp; ++w) {
      gpos += sh.wgt[w];
      epos += sh.weq[w];
    }
    for (int c = lo; c < lo + seg; c += 32) {
      const int j = c + lane;
      const uint32_t u = j < hi ? keys[j] : 0u;
      const bool is_gt = j < hi && u > T, is_eq = j < hi && u == T;
      const uint32_t bgt = __ballot_sync(0xffffffffu, is_gt);
      const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
      const uint64_t comp = ((uint64_t)u << 32) | (uint32_t)j;
      if (is_gt) bufA[gpos + __popc(bgt & lt)] = comp;
      if (is_eq) {
        const uint32_t r = epos + __popc(beq & lt);
        if (r < (uint32_t)need) bufA[n_gt + r] = comp;
      }
      gpos += __popc(bgt);
      epos += __popc(beq);
    }
    __syncthreads();
  }

  // ---- stable LSD radix sort of the m survivors, descending ----
  uint64_t *cur = bufA, *alt = bufB;
  for (int shift = 0; shift < 32; shift += 8) {
    if (lsd_pass(cur, alt, m, shift, sh)) {
      uint64_t *t = cur;
      cur = alt;
      alt = t;
    }
  }

  int32_t *oi = out_idx + (size_t)row * topk;
  float *os = out_scores + (size_t)row * topk;
  for (int i = tid; i < topk; i += kSelThreads) {
    if (i < m) {
      const uint64_t c = cur[i];
      oi[i] = (int32_t)(uint32_t)c;
      os[i] = key_to_float((uint32_t)(c >> 32));
    } else {
      oi[i] = -1;
      os[i] = -__int_as_float(0x7f800000);
    }
  }
}

__global__ void gather_scores_kernel(const float *__restrict__ logits,
                                     const int32_t *__restrict__ in_idx,
                                     const int32_t *__restrict__ q_pos, int S,
                                     int S_kv, int ratio, int topk,
                                     long long total,
                                     int32_t *__restrict__ out_idx,
                                     float *__restrict__ out_scores,
                                     int *status) {
  const float neg_inf = -__int_as_float(0x7f800000);
  bool bad = false;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       e < total; e += (long long)gridDim.x * blockDim.x) {
    const long long row = e / topk;
    const int b = (int)(row / S), s = (int)(row % S);
    const int nv = n_visible(row_pos(q_pos, b, s), ratio, S_kv);
    const int32_t j = __ldg(in_idx + e);
    out_idx[e] = j;
    float v = neg_inf;
    if (j >= 0 && j < nv) v = __ldg(logits + row * S_kv + j);
    if (j < -1 || j >= S_kv) bad = true;
    out_scores[e] = v;
  }
  if (bad) atomicOr(status, kStatusIndexRange);
}

__global__ void fill_neg_inf_kernel(float *p, size_t n) {
  const float neg_inf = -__int_as_float(0x7f800000);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    p[i] = neg_inf;
}

}  // namespace

size_t topk_select_smem_bytes(int S_kv, int topk) {
  const int mcap = topk < S_kv ? topk : S_kv;
  return (size_t)mcap * 16 + (size_t)S_kv * 4 + sizeof(SelShared);
}

cudaError_t launch_topk_select(const Problem &p, const float *logits, int topk,
                               int32_t *out_idx, float *out_scores,
                               cudaStream_t st) {
  const int mcap = topk < p.S_kv ? topk : p.S_kv;
  const size_t smem = (size_t)mcap * 16 + (size_t)p.S_kv * 4;
  cudaError_t e = cudaFuncSetAttribute(
      topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.S;
  topk_select_kernel<<<(unsigned)rows, kSelThreads, smem, st>>>(
      logits, p.q_pos, p.S, p.S_kv, p.ratio, topk, mcap, out_idx, out_scores);
  return cudaGetLastError();
}

cudaError_t launch_gather_scores(const Problem &p, const float *logits,
                                 const int32_t *in_idx, int topk,
                                 int32_t *out_idx, float *out_scores,
                                 int *status, int num_sms, cudaStream_t st) {
  const long long total = (long long)p.B * p.S * topk;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  gather_scores_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      logits, in_idx, p.q_pos, p.S, p.S_kv, p.ratio, topk, total, out_idx,
      out_scores, status);
  return cudaGetLastError();
}

cudaError_t launch_fill_masked(float *logits, size_t n, cudaStream_t st) {
  size_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  fill_neg_inf_kernel<<<(unsigned)blocks, 256, 0, st>>>(logits, n);
  return cudaGetLastError();
}

}  // namespace dsa
