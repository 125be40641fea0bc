// topk_select: per query row, the `topk` visible keys with the largest score,
// sorted by descending score with equal scores ordered by ascending key
// index; the rest of the row is -1 / -inf.
//
// One CTA per row.  The row's n visible fp32 scores are staged in shared
// memory as order-preserving unsigned keys (larger float <-> larger key;
// -0.0 folded onto +0.0 so the index tie-break decides between them).  A
// most-significant-digit-first radix select (four 8-bit digits, block
// histograms in shared memory) finds T, the k-th largest key.  One ordered
// pass then keeps every key > T and the lowest-index keys == T, and a
// bitonic sort over 64-bit (key << 32 | ~j) composites orders the survivors;
// the composite makes every key distinct, so the sort realises the
// "lower index first" tie rule exactly.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ uint32_t ordered_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0.0 -> +0.0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__host__ __device__ inline int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

__global__ void __launch_bounds__(kSelThreads)
    topk_select_kernel(const float *__restrict__ logits,
                       const int32_t *__restrict__ q_pos, int S, int S_kv,
                       int ratio, int topk, int kpad,
                       int32_t *__restrict__ out_idx,
                       float *__restrict__ out_scores) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t *cand = reinterpret_cast<uint64_t *>(smem);         // [kpad]
  uint32_t *keys = reinterpret_cast<uint32_t *>(cand + kpad);  // [S_kv]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t warp_gt[kSelWarps], warp_eq[kSelWarps];
  __shared__ uint32_t sel_digit, sel_above;

  const int row = blockIdx.x;  // row id = b * S + s, the output order
  const int b = row / S, s = row % S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = n_visible(row_pos(q_pos, b, s), ratio, S_kv);
  const float *L = logits + (size_t)row * S_kv;
  const int m = nv < topk ? nv : topk;

  for (int j = tid; j < nv; j += kSelThreads) keys[j] = ordered_key(L[j]);
  __syncthreads();

  if (nv <= topk) {
    for (int j = tid; j < nv; j += kSelThreads)
      cand[j] = ((uint64_t)keys[j] << 32) | (uint32_t)(~(uint32_t)j);
  } else {
    // ---- radix select of T, the topk-th largest key ----
    uint32_t prefix = 0, pmask = 0;
    int need = topk;  // how many still to take among keys matching prefix
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kSelThreads) hist[i] = 0;
      __syncthreads();
      for (int j = tid; j < nv; j += kSelThreads) {
        const uint32_t u = keys[j];
        if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits [8l, 8l+8); find the largest digit d with
        // count(digit >= d) >= need
        uint32_t c[8];
        uint32_t lsum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = hist[lane * 8 + i];
          lsum += c[i];
        }
        // inclusive suffix sum over lanes
        uint32_t incl = lsum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const uint32_t o = __shfl_down_sync(0xffffffffu, incl, off);
          if (lane + off < 32) incl += o;
        }
        const uint32_t above = incl - lsum;  // digits owned by higher lanes
        // the owning lane: above < need <= incl
        if (above < (uint32_t)need && (uint32_t)need <= incl) {
          uint32_t run = above;
          for (int i = 7; i >= 0; --i) {
            if (run + c[i] >= (uint32_t)need) {
              sel_digit = (uint32_t)(lane * 8 + i);
              sel_above = run;
              break;
            }
            run += c[i];
          }
        }
      }
      __syncthreads();
      need -= (int)sel_above;
      prefix |= sel_digit << shift;
      pmask |= 255u << shift;
      __syncthreads();
    }
    const uint32_t T = prefix;
    const int n_gt = topk - need;  // keys strictly above T, all kept

    // ---- ordered compaction: keys > T, then the `need` lowest-j ties ----
    uint32_t gt_base = 0, eq_base = 0;
    for (int c0 = 0; c0 < nv; c0 += kSelThreads) {
      const int j = c0 + tid;
      const uint32_t u = j < nv ? keys[j] : 0u;
      const bool is_gt = j < nv && u > T;
      const bool is_eq = j < nv && u == T;
      const uint32_t bgt = __ballot_sync(0xffffffffu, is_gt);
      const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
      if (lane == 0) {
        warp_gt[warp] = __popc(bgt);
        warp_eq[warp] = __popc(beq);
      }
      __syncthreads();
      uint32_t pre_gt = 0, pre_eq = 0, tot_gt = 0, tot_eq = 0;
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) {
        const uint32_t g = warp_gt[w], e = warp_eq[w];
        if (w < warp) {
          pre_gt += g;
          pre_eq += e;
        }
        tot_gt += g;
        tot_eq += e;
      }
      const uint32_t lt_mask = (1u << lane) - 1u;
      const uint64_t comp = ((uint64_t)u << 32) | (uint32_t)(~(uint32_t)j);
      if (is_gt) cand[gt_base + pre_gt + __popc(bgt & lt_mask)] = comp;
      if (is_eq) {
        const uint32_t r = eq_base + pre_eq + __popc(beq & lt_mask);
        if (r < (uint32_t)need) cand[n_gt + r] = comp;
      }
      gt_base += tot_gt;
      eq_base += tot_eq;
      __syncthreads();
    }
  }
  // pad to a power of two with the smallest composite (below any real key)
  for (int i = m + tid; i < kpad; i += kSelThreads) cand[i] = 0ull;
  __syncthreads();

  // ---- bitonic sort, descending ----
  const int n2 = pow2_at_least(m < 1 ? 1 : m);
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < n2 / 2; i += kSelThreads) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = cand[lo], c = cand[hi];
        if ((a < c) == desc) {
          cand[lo] = c;
          cand[hi] = a;
        }
      }
      __syncthreads();
    }
  }

  int32_t *oi = out_idx + (size_t)row * topk;
  float *os = out_scores + (size_t)row * topk;
  for (int i = tid; i < topk; i += kSelThreads) {
    if (i < m) {
      const uint64_t c = cand[i];
      oi[i] = (int32_t)(~(uint32_t)c);
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
  const int kpad = pow2_at_least(topk < S_kv ? topk : S_kv);
  return (size_t)kpad * 8 + (size_t)S_kv * 4;
}

cudaError_t launch_topk_select(const Problem &p, const float *logits, int topk,
                               int32_t *out_idx, float *out_scores,
                               cudaStream_t st) {
  const int kpad = pow2_at_least(topk < p.S_kv ? topk : p.S_kv);
  const size_t smem = topk_select_smem_bytes(p.S_kv, topk);
  cudaError_t e = cudaFuncSetAttribute(
      topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.B * p.S;
  topk_select_kernel<<<(unsigned)rows, kSelThreads, smem, st>>>(
      logits, p.q_pos, p.S, p.S_kv, p.ratio, topk, kpad, out_idx, out_scores);
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
