// topk_select: per query row, the `topk` visible keys with the largest score,
// sorted by descending score with equal scores ordered by ascending key
// index; the rest of the row is -1 / -inf.
//
// One CTA per row: 256 threads when there are many rows, 512 when there
// are fewer rows than SMs.  Scores are compared as order-preserving unsigned
// keys (larger float <-> larger key; -0.0 folded onto +0.0 so the index
// tie-break decides between them).
//
// Bucket route (every row first): the row -- in registers up to 4096 keys
// (8192 in a 512-thread CTA), else staged in shared memory when it fits,
// else read from L2 -- is counted into fine buckets spread linearly over
// its finite value range (4096, or for a row held in registers as many as
// it has keys rounded up to 1024, 2048 or 4096).  A
// scan of the counts gives the bucket holding the topk-th key and each
// kept bucket's start; the kept keys are scattered to their buckets and
// each key's final position is its bucket start plus the number of keys of
// the same bucket that precede it (larger key, or equal key and lower
// index).  Three passes over the row, no sort.  A row where a bucket
// holding kept keys has more than 32 keys (heavy ties, a tight cluster, a
// far outlier) continues on the radix route:
//   1. n <= topk: every visible key is a candidate.
//      n > topk: a 4096-bin histogram of the top 12 key bits (the sign, the
//      exponent and three mantissa bits) gives the bucket holding the
//      topk-th largest key.  If the keys in and above that
//      bucket fit topk plus a slack, one pass keeps them all (in any
//      order); otherwise two more passes (12 and 8 bits) find the exact
//      threshold T and an ordered compaction keeps every key > T and the
//      lowest-index keys == T.
//   2. A stable least-significant-digit radix sort (8-bit digits,
//      descending) orders the m candidates, packed as (key << 32 | j), on
//      key bits 8..31.  Within a warp, equal digits are ranked from a peer
//      mask (eight ballots or one match instruction), so ranks follow
//      element order and the sort is stable.  Digit positions on which every
//      candidate agrees (an AND/OR reduction) are skipped.
//   3. Runs of equal top 24 bits (a few elements for real score
//      distributions) are ordered by (low 8 bits desc, index asc) by
//      counting inside the run, which also fixes the order of candidates
//      kept out of index order in step 1.  If a run is longer than 32
//      (heavily tied inputs), the candidates are rebuilt and sorted on all
//      four digits instead.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kSelThreads = 256;       // threads per row, many rows
constexpr int kSelThreadsWide = 512;   // threads per row, few rows
constexpr int kSelMaxWarps = kSelThreadsWide / 32;
constexpr int kHistBins = 4096;  // 12-bit select digit
constexpr int kSelSlack = 256;   // extra candidates a one-pass select keeps

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Lanes of this warp whose 8-bit digit equals mine (0 for invalid lanes).
__device__ __forceinline__ uint32_t digit_peers(uint32_t d, bool valid) {
  uint32_t m = __ballot_sync(0xffffffffu, valid);
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    const bool bit = (d >> b) & 1u;
    const uint32_t bal = __ballot_sync(0xffffffffu, bit);
    m &= bit ? bal : ~bal;
  }
  return valid ? m : 0u;
}

// The same mask from one match instruction (a different execution pipe
// from the ballots, so alternating the two keeps both busy).
__device__ __forceinline__ uint32_t digit_peers_match(uint32_t d, bool valid) {
  const uint32_t key = valid ? d : 0x100u;  // invalid lanes group apart
  const uint32_t m = __match_any_sync(0xffffffffu, key);
  return valid ? m : 0u;
}

struct SelShared {
  uint32_t (*whist)[256];          // per-warp digit counts / offsets; lives
                                   // in the row-key buffer, dead by then
  uint32_t dbase[256];             // digit bases of a sort pass
  uint32_t wsum[kSelMaxWarps];
  uint32_t wgt[kSelMaxWarps], weq[kSelMaxWarps];
  uint32_t wand[kSelMaxWarps], wor[kSelMaxWarps];
  uint32_t sel_digit, sel_above, sel_count;
  uint32_t cursor;
  int overflow;
};

// Exclusive prefix sum of one value per thread over the NT-thread block.
template <int NT>
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
  for (int w = 0; w < NT / 32; ++w)
    if (w < warp) pre += sh.wsum[w];
  __syncthreads();  // wsum may be rewritten by the next scan
  return pre + incl - v;
}

// One stable counting-sort pass of src[0..m) into dst on digit
// (key >> shift) & 255, descending.  Warp w ranks the contiguous elements
// [32*E*w, 32*E*(w+1)); E is the smallest instantiated count that covers m,
// so no iteration runs past the data (warps past the end skip the loops).
template <int E, int NT>
__device__ __forceinline__ void lsd_pass(const uint64_t *src, uint64_t *dst,
                                         int m, int shift, SelShared &sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = warp * 32 * E;
  const bool active = seg < m;  // warp-uniform
  uint32_t *wh = sh.whist[warp];
  const uint32_t lt = lanemask_lt();
  for (int i = lane; i < 256; i += 32) wh[i] = 0;
  __syncwarp();
  uint32_t off[E];
  if (active) {
#pragma unroll
    for (int it = 0; it < E; ++it) {
      const int e = seg + it * 32 + lane;
      const bool valid = e < m;
      const uint64_t v = valid ? src[e] : 0ull;
      const uint32_t d = 255u - (uint32_t)((v >> (32 + shift)) & 255u);
      const uint32_t peers = ((it + warp) & 1) ? digit_peers_match(d, valid)
                                                : digit_peers(d, valid);
      const uint32_t rank = __popc(peers & lt);
      const uint32_t base = valid ? wh[d] : 0u;
      __syncwarp();
      if (valid && rank == 0) wh[d] = base + __popc(peers);
      __syncwarp();
      off[it] = base + rank;
    }
  }
  __syncthreads();
  {
    const int d = threadIdx.x;  // the first 256 threads, one digit each
    uint32_t run = 0;
    if (d < 256) {
#pragma unroll
      for (int w = 0; w < NT / 32; ++w) {
        const uint32_t c = sh.whist[w][d];
        sh.whist[w][d] = run;
        run += c;
      }
    }
    const uint32_t dbase = block_excl_scan<NT>(run, sh);
    if (d < 256) sh.dbase[d] = dbase;
  }
  __syncthreads();
  if (active) {
#pragma unroll
    for (int it = 0; it < E; ++it) {
      const int e = seg + it * 32 + lane;
      if (e < m) {
        const uint64_t v = src[e];
        const uint32_t d = 255u - (uint32_t)((v >> (32 + shift)) & 255u);
        dst[sh.dbase[d] + wh[d] + off[it]] = v;
      }
    }
  }
  __syncthreads();
}

// Runs one pass with the smallest element count per lane that covers m
// (at most EMAX, the kernel's instantiation limit).
template <int EMAX, int NT>
__device__ __forceinline__ void lsd_dispatch(const uint64_t *src,
                                             uint64_t *dst, int m, int shift,
                                             SelShared &sh) {
  const int ept = (m + NT - 1) / NT;
  if (ept <= 1) return lsd_pass<1, NT>(src, dst, m, shift, sh);
  if (ept <= 2) return lsd_pass<2, NT>(src, dst, m, shift, sh);
  if (ept <= 4) return lsd_pass<4, NT>(src, dst, m, shift, sh);
  if (EMAX <= 8 || ept <= 8) return lsd_pass<(EMAX < 8 ? EMAX : 8), NT>(src, dst, m, shift, sh);
  // covers the topk + slack candidates of a one-pass select (2304 for
  // topk 2048)
  if (EMAX <= 10 || ept <= 10) return lsd_pass<(EMAX < 10 ? EMAX : 10), NT>(src, dst, m, shift, sh);
  if (EMAX <= 16 || ept <= 16) return lsd_pass<(EMAX < 16 ? EMAX : 16), NT>(src, dst, m, shift, sh);
  if (EMAX <= 24 || ept <= 24) return lsd_pass<(EMAX < 24 ? EMAX : 24), NT>(src, dst, m, shift, sh);
  return lsd_pass<EMAX, NT>(src, dst, m, shift, sh);
}

// Fix-up after sorting on the top 24 key bits: inside each run of equal top
// 24 bits, order by the low 8 bits, descending, and equal keys by ascending
// index (compared explicitly, so the run may arrive in any order).  Writes the result to dst.  Returns
// true (block-uniform) when some run is longer than kRunLimit, in which case
// dst is incomplete and the caller falls back to a full sort.
constexpr int kRunLimit = 32;

template <int NT>
__device__ __forceinline__ bool run_fixup(const uint64_t *src, uint64_t *dst,
                                          int m, SelShared &sh) {
  if (threadIdx.x == 0) sh.overflow = 0;
  __syncthreads();
  bool over = false;
  for (int i = threadIdx.x; i < m; i += NT) {
    const uint64_t v = src[i];
    const uint32_t top = (uint32_t)(v >> 40);
    const uint32_t low = (uint32_t)(v >> 32) & 0xFFu;
    const uint32_t jv = (uint32_t)v;
    // does candidate u come before v in the final order?
    auto before = [&](uint64_t u) -> int {
      const uint32_t lu = (uint32_t)(u >> 32) & 0xFFu;
      return lu > low || (lu == low && (uint32_t)u < jv);
    };
    int cnt = 0, r = i - 1, steps = 0;
    while (r >= 0 && steps < kRunLimit) {
      const uint64_t u = src[r];
      if ((uint32_t)(u >> 40) != top) break;
      cnt += before(u);
      --r;
      ++steps;
    }
    if (steps == kRunLimit && r >= 0 && (uint32_t)(src[r] >> 40) == top)
      over = true;
    const int start = r + 1;
    r = i + 1;
    steps = 0;
    while (r < m && steps < kRunLimit) {
      const uint64_t u = src[r];
      if ((uint32_t)(u >> 40) != top) break;
      cnt += before(u);
      ++r;
      ++steps;
    }
    if (steps == kRunLimit && r < m && (uint32_t)(src[r] >> 40) == top)
      over = true;
    if (!over) dst[start + cnt] = v;
  }
  if (over) sh.overflow = 1;
  __syncthreads();
  const bool any = sh.overflow != 0;
  __syncthreads();
  return any;
}

// ---- bucket route ----
// One histogram of kBucketBins fine buckets over the row's finite value
// range [lo, hi] both finds the threshold and groups the kept keys; keys
// inside a bucket are then ordered by counting.  The bucket of a key is a
// non-decreasing function of the key (keys at or below the smallest finite
// key go to the lowest bucket, keys at or above the largest to the highest,
// the rest linearly in their float value), so every key of a higher bucket
// comes before every key of a lower one and the count inside the bucket
// gives the exact position.  Rows where a bucket holding kept keys has more
// than kBucketLimit keys (ties, clusters, outliers) take the radix route.
constexpr int kBucketBins = 4096;
constexpr int kBucketLimit = 32;
// (start << 16 | count) packing of the kept bins needs topk + 31 < 2^16
constexpr int kBucketMaxTopk = 32768;

struct BucketMap {
  uint32_t kmin, kmax;  // order keys of the smallest / largest finite value
  float lo, sc;         // lo = value of kmin, sc = bins per unit value
  // descending bin: 0 holds the largest keys
  __device__ __forceinline__ uint32_t desc(uint32_t k) const {
    if (k <= kmin) return kBucketBins - 1;
    if (k >= kmax) return 0u;
    // cvt.rzi saturates; (v - lo) * sc is finite and >= 0 here
    const uint32_t b = __float2uint_rz((key_to_float(k) - lo) * sc);
    return b < kBucketBins - 1 ? (kBucketBins - 1) - b : 0u;
  }
};

// Bank spread for the scan, where thread t reads bins [16t, 16t + 16):
// a permutation inside each aligned group of 16 bins.
__device__ __forceinline__ uint32_t bin_slot(uint32_t b) {
  return b ^ ((b >> 4) & 15u);
}

// Selects and orders the row's top min(nv, topk) keys and writes the output
// row.  Returns false (block-uniform, before writing anything) when a
// bucket holding kept keys is too full; nothing the radix route reads has
// been changed then except the staged keys, which it reloads.
// stage: [stage_cap] u32 (the row's keys when nv fits); bins:
// [kBucketBins] u32; grouped: [>= min(nv, topk) + kBucketLimit] u64.
template <int NT>
__device__ __forceinline__ bool bucket_topk(const float *__restrict__ L, int nv,
                                         int topk, uint32_t *stage,
                                         int stage_cap, uint32_t *bins,
                                         uint64_t *grouped, SelShared &sh,
                                         int32_t *__restrict__ oi,
                                         float *__restrict__ os) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int per = kBucketBins / NT;
  const bool staged = nv <= stage_cap;
  const float neg_inf = -__int_as_float(0x7f800000);

  for (int i = tid; i < kBucketBins; i += NT) bins[i] = 0u;
  // row keys (staged when they fit) and the finite value range
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  for (int j0 = tid; j0 < nv; j0 += 4 * NT) {
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * NT;
      v[u] = j < nv ? __ldg(L + j) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * NT;
      if (j < nv) {
        const uint32_t k = ordered_key(v[u]);
        if (staged) stage[j] = k;
        if (fabsf(v[u]) <= 3.402823466e38f) {
          kmn = min(kmn, k);
          kmx = max(kmx, k);
        }
      }
    }
  }
  kmn = __reduce_min_sync(0xffffffffu, kmn);
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  if (lane == 0) {
    sh.wand[warp] = kmn;
    sh.wor[warp] = kmx;
  }
  if (tid == 0) sh.overflow = 0;
  __syncthreads();
  BucketMap map;
  map.kmin = 0xffffffffu;
  map.kmax = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    map.kmin = min(map.kmin, sh.wand[w]);
    map.kmax = max(map.kmax, sh.wor[w]);
  }
  map.lo = key_to_float(map.kmin);
  map.sc = 0.f;
  if (map.kmin < map.kmax) {
    const float span = key_to_float(map.kmax) - map.lo;
    if (span > 0.f && span <= 3.402823466e38f)
      map.sc = fminf((float)kBucketBins / span, 1e30f);
  }
  auto key_of = [&](int j) -> uint32_t {
    return staged ? stage[j] : ordered_key(__ldg(L + j));
  };

  for (int j = tid; j < nv; j += NT)
    atomicAdd(&bins[bin_slot(map.desc(key_of(j)))], 1u);
  __syncthreads();

  // thread t owns descending bins [t*per, t*per + per)
  uint32_t c[per];
  uint32_t lsum = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    c[i] = bins[bin_slot(tid * per + i)];
    lsum += c[i];
  }
  const uint32_t above = block_excl_scan<NT>(lsum, sh);
  const uint32_t want = (uint32_t)min(nv, topk);
  if (tid == 0 && want == 0) {
    sh.sel_digit = 0xffffffffu;  // no bin holds a kept key
    sh.sel_count = 0;
  }
  if (want > 0 && above < want && want <= above + lsum) {
    uint32_t run = above;
#pragma unroll
    for (int i = 0; i < per; ++i) {
      if (run + c[i] >= want) {
        sh.sel_digit = (uint32_t)(tid * per + i);
        sh.sel_count = run + c[i];
        break;
      }
      run += c[i];
    }
  }
  __syncthreads();
  const uint32_t thr = sh.sel_digit;  // last bin holding kept keys
  const int m = (int)sh.sel_count;    // keys in bins 0..thr
  // kept bins become (start << 16 | count); the scatter advances start
  uint32_t occ = 0, run = above;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    const uint32_t b = (uint32_t)(tid * per + i);
    if (thr != 0xffffffffu && b <= thr) {
      bins[bin_slot(b)] = (run << 16) | c[i];
      occ = max(occ, c[i]);
    }
    run += c[i];
  }
  occ = __reduce_max_sync(0xffffffffu, occ);
  if (lane == 0 && occ > (uint32_t)kBucketLimit) sh.overflow = 1;
  __syncthreads();
  if (sh.overflow) {
    __syncthreads();  // every thread has read the flag
    return false;
  }

  for (int j = tid; j < nv; j += NT) {
    const uint32_t k = key_of(j);
    const uint32_t b = map.desc(k);
    if (b <= thr) {
      const uint32_t pos = atomicAdd(&bins[bin_slot(b)], 1u << 16) >> 16;
      grouped[pos] = ((uint64_t)k << 32) | (uint32_t)j;
    }
  }
  __syncthreads();

  for (int p = tid; p < m; p += NT) {
    const uint64_t cv = grouped[p];
    const uint32_t k = (uint32_t)(cv >> 32), j = (uint32_t)cv;
    const uint32_t e = bins[bin_slot(map.desc(k))];
    const int end = (int)(e >> 16), start = end - (int)(e & 0xffffu);
    int r = start;
    for (int q = start; q < end; ++q) {
      const uint64_t u = grouped[q];
      const uint32_t uk = (uint32_t)(u >> 32);
      r += (uk > k) || (uk == k && (uint32_t)u < j);
    }
    if (r < topk) {
      const float v = key_to_float(k);
      oi[r] = v == neg_inf ? -1 : (int32_t)j;
      os[r] = v;
    }
  }
  for (int i = m + tid; i < topk; i += NT) {
    oi[i] = -1;
    os[i] = neg_inf;
  }
  return true;
}

// The same route for rows of at most R * NT keys, held in registers: thread
// t owns keys 4(t + NT i) + c (c < 4, i < R/4), read as float4 when the row
// is 16-byte aligned, over NB buckets (1024, 2048 or 4096: R * NT, or half
// of it for rows of up to 8192 keys in a 512-thread CTA).
// The bucket map here is a clamped fused multiply-add whose result lands in
// [2^23, 2^23 + NB - 1], where the float's low mantissa bits are the
// bucket; rows holding a NaN take the radix route.  A kept key
// is stored as (key << 32 | bucket << 20 | (2^20 - 1 - j)), so inside a
// bucket "comes before" is one unsigned 64-bit comparison.
template <int NB>
struct RegMap {
  float sc, off;  // t = sat(v * sc + off) in [0, 1]
  // descending bucket of a value among NB: t * (NB - 1) + 2^23 rounds to an
  // integer whose low mantissa bits are the ascending bucket; monotone
  // non-increasing in v, both steps on the FMA pipe; -inf (and, with sc = 0,
  // everything) lands in the last bucket
  __device__ __forceinline__ uint32_t desc(float v) const {
    float t;
    asm("fma.rn.sat.f32 %0, %1, %2, %3;"
      : "=f"(t)
      : "f"(v), "f"(sc), "f"(off));
    const float u = fmaf(t, (float)(NB - 1), 8388608.0f);
    return ~__float_as_uint(u) & (uint32_t)(NB - 1);
  }
};

// vec: the row is 16-byte aligned and its length a multiple of four.
// The keys stay floats until they are kept: the range and the buckets are
// computed on the values, and only the kept keys get their order key.
template <int NT, int R, int NB>
__device__ __forceinline__ bool bucket_topk_reg(
    const float *__restrict__ L, int nv, int topk, bool vec, uint32_t *bins,
    uint64_t *grouped, SelShared &sh, int32_t *__restrict__ oi,
    float *__restrict__ os) {
  static_assert(R % 4 == 0, "keys are read four at a time");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int per = NB / NT;
  const float neg_inf = -__int_as_float(0x7f800000);
  const float pos_inf = __int_as_float(0x7f800000);

  {
    // bins follow a u64 buffer of any length: 8-byte aligned only
    uint2 *b2 = reinterpret_cast<uint2 *>(bins);
#pragma unroll
    for (int i = tid; i < NB / 2; i += NT) b2[i] = make_uint2(0u, 0u);
  }
  // the loops over a thread's key groups skip, block-uniformly, the groups
  // past the row's end (a short row runs a fraction of the unrolled code)
  float kv[R];
  float lo = pos_inf, hi = neg_inf;  // range of the finite values
  bool nan = false;
#pragma unroll
  for (int i = 0; i < R / 4; ++i) {
    if (4 * NT * i >= nv) {
#pragma unroll
      for (int c = 0; c < 4; ++c) kv[4 * i + c] = neg_inf;
      continue;
    }
    const int j0 = 4 * (tid + NT * i);
    float v[4] = {neg_inf, neg_inf, neg_inf, neg_inf};
    if (vec) {
      // j0 < nv <= row length, both multiples of four: the group of four
      // lies inside the row
      if (j0 < nv) {
        const float4 f = __ldg(reinterpret_cast<const float4 *>(L + j0));
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (j0 + c < nv) v[c] = __ldg(L + j0 + c);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      kv[4 * i + c] = v[c];
      // keys past the row's end are -inf here and never counted
      nan |= v[c] != v[c];
      if (fabsf(v[c]) <= 3.402823466e38f) {
        lo = fminf(lo, v[c]);
        hi = fmaxf(hi, v[c]);
      }
    }
  }
  // block range through order-preserving integers (+-inf when no value is
  // finite)
  uint32_t kmn = __reduce_min_sync(0xffffffffu, ordered_key(lo));
  uint32_t kmx = __reduce_max_sync(0xffffffffu, ordered_key(hi));
  nan = __any_sync(0xffffffffu, nan);
  if (lane == 0) {
    sh.wand[warp] = kmn;
    sh.wor[warp] = kmx;
    sh.wgt[warp] = nan ? 1u : 0u;
  }
  if (tid == 0) sh.overflow = 0;
  __syncthreads();
  uint32_t kmin = 0xffffffffu, kmax = 0u, anynan = 0u;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    kmin = min(kmin, sh.wand[w]);
    kmax = max(kmax, sh.wor[w]);
    anynan |= sh.wgt[w];
  }
  if (anynan) return false;  // block-uniform; nothing written yet
  RegMap<NB> map;
  map.sc = 0.f;
  map.off = 0.f;
  if (kmin < kmax) {
    const float flo = key_to_float(kmin);
    const float span = key_to_float(kmax) - flo;
    if (span > 0.f && span <= 3.402823466e38f) {
      map.sc = fminf(1.f / span, 1e30f);
      // v * sc - lo * sc lands within a rounding of [0, 1]; the saturation
      // absorbs the error and keeps the map monotone
      map.off = -flo * map.sc;
    }
  }

  // each key's bucket, two to a register, for the scatter below
  uint32_t bk[R / 2];
#pragma unroll
  for (int i = 0; i < R / 2; ++i) bk[i] = 0u;
#pragma unroll
  for (int i = 0; i < R / 4; ++i) {
    if (4 * NT * i >= nv) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t b = map.desc(kv[4 * i + c]);
      bk[2 * i + (c >> 1)] |= b << (16 * (c & 1));
      if (4 * (tid + NT * i) + c < nv) atomicAdd(&bins[bin_slot(b)], 1u);
    }
  }
  __syncthreads();

  // counts are re-read from shared memory rather than held across the
  // scan (the row's keys already take R registers)
  uint32_t lsum = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) lsum += bins[bin_slot(tid * per + i)];
  const uint32_t above = block_excl_scan<NT>(lsum, sh);
  const uint32_t want = (uint32_t)min(nv, topk);
  if (tid == 0 && want == 0) {
    sh.sel_digit = 0xffffffffu;  // no bin holds a kept key
    sh.sel_count = 0;
  }
  // a bin holds kept keys iff fewer than `want` keys lie in the bins
  // before it; the one where the running count reaches `want` is the last
  uint32_t occ = 0, run = above;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    const uint32_t b = (uint32_t)(tid * per + i);
    const uint32_t c = bins[bin_slot(b)];
    if (run < want) {
      bins[bin_slot(b)] = (run << 16) | c;
      occ = max(occ, c);
      if (run + c >= want) {
        sh.sel_digit = b;
        sh.sel_count = run + c;
      }
    }
    run += c;
  }
  occ = __reduce_max_sync(0xffffffffu, occ);
  if (lane == 0 && occ > (uint32_t)kBucketLimit) sh.overflow = 1;
  __syncthreads();
  const uint32_t thr = sh.sel_digit;  // last bin holding kept keys
  const int m = (int)sh.sel_count;    // keys in bins 0..thr
  if (sh.overflow) {
    __syncthreads();
    return false;
  }

#pragma unroll
  for (int i = 0; i < R / 4; ++i) {
    if (4 * NT * i >= nv) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = 4 * (tid + NT * i) + c;
      const uint32_t b = (bk[2 * i + (c >> 1)] >> (16 * (c & 1))) & 0xffffu;
      if (j < nv && b <= thr) {
        const uint32_t pos = atomicAdd(&bins[bin_slot(b)], 1u << 16) >> 16;
        grouped[pos] = ((uint64_t)ordered_key(kv[4 * i + c]) << 32) |
                       (b << 20) | (0xfffffu - (uint32_t)j);
      }
    }
  }
  __syncthreads();

  for (int p = tid; p < m; p += NT) {
    const uint64_t cv = grouped[p];
    const uint32_t lo32 = (uint32_t)cv;
    const uint32_t e = bins[bin_slot(lo32 >> 20)];
    const int end = (int)(e >> 16), start = end - (int)(e & 0xffffu);
    int r = start;
    for (int q = start; q < end; ++q) r += grouped[q] > cv;
    if (r < topk) {
      const float v = key_to_float((uint32_t)(cv >> 32));
      oi[r] = v == neg_inf ? -1 : (int32_t)(0xfffffu - (lo32 & 0xfffffu));
      os[r] = v;
    }
  }
  for (int i = m + tid; i < topk; i += NT) {
    oi[i] = -1;
    os[i] = neg_inf;
  }
  return true;
}

template <int EPT, int NT>
__global__ void __launch_bounds__(NT, NT == kSelThreads ? 4 : 1)
    topk_select_kernel(const float *__restrict__ logits,
                       const int32_t *__restrict__ q_pos, int s0, int S,
                       int S_out, int S_kv, int ratio, int topk, int mcap,
                       int bcap, int keys_cap, int region_u32,
                       int32_t *__restrict__ out_idx,
                       float *__restrict__ out_scores) {
  // the logits come from the scoring kernel, which this launch may overlap
  // (programmatic dependent launch)
  pdl_wait();
  // the next chunk's scoring kernel may be scheduled once every CTA of this
  // grid has started; it waits for this grid to finish before it writes
  pdl_allow_dependents();
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t *bufA = reinterpret_cast<uint64_t *>(smem);  // [mcap]
  uint64_t *bufB = bufA + mcap;                          // [bcap] (>= 4096 u32)
  uint32_t *hist = reinterpret_cast<uint32_t *>(bufB);   // select histogram
  uint32_t *keys = reinterpret_cast<uint32_t *>(bufB + bcap);  // [S_kv]
  __shared__ SelShared sh;
  if (threadIdx.x == 0)
    sh.whist = reinterpret_cast<uint32_t(*)[256]>(keys);

  // this launch covers rows [s0, s0 + S) of every sequence; the logits hold
  // just those rows, the outputs every row ([B, S_out, topk])
  const int row = blockIdx.x;  // b * S + (s - s0)
  const int b = row / S, s = s0 + row % S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = n_visible(row_pos(q_pos, b, s), ratio, S_kv);
  const float *L = logits + (size_t)row * S_kv;
  const uint32_t lt = lanemask_lt();
  int32_t *oi = out_idx + ((size_t)b * S_out + s) * topk;
  float *os = out_scores + ((size_t)b * S_out + s) * topk;

  // (one pass of a do-while: the routes leave it when the row is done)
  do {
  // the bucket route first; the radix route takes the rows it declines
  if (topk <= kBucketMaxTopk) {
    constexpr int R = kBucketBins / NT;  // keys per thread in registers
    // a 512-thread CTA holds rows of up to 8192 keys, 16 per thread
    constexpr int RW = NT == kSelThreadsWide ? 2 * R : R;
    if (nv <= RW * NT) {
      const bool vec = (S_kv & 3) == 0 &&
                       (reinterpret_cast<uintptr_t>(L) & 15u) == 0;
      // as many buckets as the row has keys, rounded up to 1024, 2048 or
      // 4096: the clear and the scan cost per bucket
      uint32_t *bins = reinterpret_cast<uint32_t *>(bufB);
      bool done;
      if constexpr (R % 16 == 0) {
        if (nv <= kBucketBins / 4)
          done = bucket_topk_reg<NT, R / 4, kBucketBins / 4>(
              L, nv, topk, vec, bins, bufA, sh, oi, os);
        else if (nv <= kBucketBins / 2)
          done = bucket_topk_reg<NT, R / 2, kBucketBins / 2>(
              L, nv, topk, vec, bins, bufA, sh, oi, os);
        else
          done = bucket_topk_reg<NT, R, kBucketBins>(L, nv, topk, vec, bins,
                                                     bufA, sh, oi, os);
      } else if constexpr (RW != R) {
        if (nv <= R * NT)
          done = bucket_topk_reg<NT, R, kBucketBins>(L, nv, topk, vec, bins,
                                                     bufA, sh, oi, os);
        else
          done = bucket_topk_reg<NT, RW, kBucketBins>(L, nv, topk, vec, bins,
                                                      bufA, sh, oi, os);
      } else {
        done = bucket_topk_reg<NT, R, kBucketBins>(L, nv, topk, vec, bins,
                                                   bufA, sh, oi, os);
      }
      if (done) break;
    } else if (bucket_topk<NT>(L, nv, topk, keys, region_u32,
                               reinterpret_cast<uint32_t *>(bufB), bufA, sh,
                               oi, os)) {
      break;
    }
  }

  // the candidates, (key << 32 | j) in index order (within each of the
  // "above T" and "equal to T" groups), into bufA
  uint32_t T = 0;
  int need = 0, n_gt = 0;
  // without a row-key buffer (long rows, many of them) keys come straight
  // from the logits in L2
  const bool staged = keys_cap >= nv;
  auto key_at = [&](int j) -> uint32_t {
    return staged ? keys[j] : ordered_key(__ldg(L + j));
  };
  // row loads keep four independent global loads in flight per thread
  auto load_keys = [&]() {
    if (!staged) return;
    for (int j0 = tid; j0 < nv; j0 += 4 * NT) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
        v[u] = j < nv ? __ldg(L + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
        if (j < nv && staged) keys[j] = ordered_key(v[u]);
      }
    }
  };
  auto load_all = [&]() {
    for (int j0 = tid; j0 < nv; j0 += 4 * NT) {
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
        v[u] = j < nv ? __ldg(L + j) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = j0 + u * NT;
        if (j < nv)
          bufA[j] = ((uint64_t)ordered_key(v[u]) << 32) | (uint32_t)j;
      }
    }
    __syncthreads();
  };
  // ordered compaction, two walks over contiguous warp segments
  auto compact = [&]() {
    __syncthreads();
    const int seg = ((nv + NT - 1) / NT) * 32;
    const int lo = warp * seg, hi = min(nv, lo + seg);
    uint32_t cgt = 0, ceq = 0;
    for (int c = lo; c < lo + seg; c += 32) {
      const int j = c + lane;
      const uint32_t u = j < hi ? key_at(j) : 0u;
      cgt += __popc(__ballot_sync(0xffffffffu, j < hi && (u > T || (need == 0 && u == T))));
      ceq += __popc(__ballot_sync(0xffffffffu, j < hi && need > 0 && u == T));
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
      const uint32_t u = j < hi ? key_at(j) : 0u;
      const bool is_gt = j < hi && (u > T || (need == 0 && u == T));
      const bool is_eq = j < hi && need > 0 && u == T;
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
  };

  int m = nv < topk ? nv : topk;  // candidates to sort
  bool done = false;
  if (nv <= topk) {
    load_all();
    done = true;
  }
  if (!done) {
    load_keys();
    // ---- radix select: 12 + 12 + 8 bits, usually only the first ----
    uint32_t prefix = 0, pmask = 0;
    bool one_pass = false;
    need = topk;  // still to take among keys matching prefix
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
      const int bits = pass == 2 ? 8 : 12;
      const int nb = 1 << bits;
      // bins per owning thread; with fewer bins than threads, the first nb
      // threads own one bin each
      const int per = nb >= NT ? nb / NT : 1, owners = nb / per;
      const uint32_t dmask = (uint32_t)nb - 1u;
      for (int i = tid; i < nb; i += NT) hist[i] = 0;
      __syncthreads();
      for (int j = tid; j < nv; j += NT) {
        const uint32_t u = key_at(j);
        if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & dmask], 1u);
      }
      __syncthreads();
      // thread t < owners owns bins [o*per, o*per+per) with
      // o = owners - 1 - t, so an exclusive scan in thread order counts the
      // bins above its own
      const int o = owners - 1 - tid;
      uint32_t lsum = 0;
      if (o >= 0)
        for (int i = 0; i < per; ++i) lsum += hist[o * per + i];
      const uint32_t above = block_excl_scan<NT>(lsum, sh);
      if (o >= 0 && above < (uint32_t)need &&
          (uint32_t)need <= above + lsum) {
        uint32_t run = above;
        for (int i = per - 1; i >= 0; --i) {
          const uint32_t c = hist[o * per + i];
          if (run + c >= (uint32_t)need) {
            sh.sel_digit = (uint32_t)(o * per + i);
            sh.sel_above = run;
            sh.sel_count = c;
            break;
          }
          run += c;
        }
      }
      __syncthreads();
      const uint32_t dsel = sh.sel_digit, dabove = sh.sel_above;
      const uint32_t dcount = sh.sel_count;
      if (pass == 0 && dabove + dcount <= (uint32_t)mcap) {
        // keep every key whose top 12 bits reach the threshold bucket; the
        // exact sort below settles the boundary (and its ties)
        T = dsel << shift;
        need = 0;
        n_gt = (int)(dabove + dcount);
        m = n_gt;
        one_pass = true;
        break;
      }
      need -= (int)dabove;
      prefix |= dsel << shift;
      pmask |= dmask << shift;
      __syncthreads();
    }
    if (!one_pass) {
      // full select ran: keep keys > T plus the `need` lowest-index ties
      T = prefix;
      n_gt = topk - need;
      m = topk;
    }
    compact();
  }

  // ---- bits on which the survivors differ ----
  uint32_t kand = 0xffffffffu, kor = 0u;
  for (int i = tid; i < m; i += NT) {
    const uint32_t k = (uint32_t)(bufA[i] >> 32);
    kand &= k;
    kor |= k;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    kand &= __shfl_xor_sync(0xffffffffu, kand, off);
    kor |= __shfl_xor_sync(0xffffffffu, kor, off);
  }
  if (lane == 0) {
    sh.wand[warp] = kand;
    sh.wor[warp] = kor;
  }
  __syncthreads();
  uint32_t all_and = 0xffffffffu, all_or = 0u;
#pragma unroll
  for (int w = 0; w < (NT / 32); ++w) {
    all_and &= sh.wand[w];
    all_or |= sh.wor[w];
  }
  const uint32_t diff = all_and ^ all_or;  // block-uniform

  // ---- stable LSD radix sort on the top 24 key bits, then a run fix-up
  // on the low 8 bits; a full four-digit sort when runs are long ----
  uint64_t *cur = bufA, *alt = bufB;
  for (int shift = 8; shift < 32; shift += 8) {
    if (((diff >> shift) & 255u) == 0u) continue;  // every digit equal
    lsd_dispatch<EPT, NT>(cur, alt, m, shift, sh);
    uint64_t *t = cur;
    cur = alt;
    alt = t;
  }
  if ((diff & 0xFFu) != 0u) {
    if (!run_fixup<NT>(cur, alt, m, sh)) {
      uint64_t *t = cur;
      cur = alt;
      alt = t;
    } else {
      // long runs of equal top bits: rebuild the candidates, sort all digits
      if (nv <= topk) {
        load_all();
      } else {
        load_keys();  // the sort reused the key buffer
        compact();
      }
      cur = bufA;
      alt = bufB;
      for (int shift = 0; shift < 32; shift += 8) {
        if (((diff >> shift) & 255u) == 0u) continue;
        lsd_dispatch<EPT, NT>(cur, alt, m, shift, sh);
        uint64_t *t = cur;
        cur = alt;
        alt = t;
      }
    }
  }

  for (int i = tid; i < topk; i += NT) {
    if (i < m) {  // m >= topk or m = n_visible < topk
      const uint64_t c = cur[i];
      const float v = key_to_float((uint32_t)(c >> 32));
      // -inf marks a key that is not a candidate (it sorts last)
      oi[i] = v == -__int_as_float(0x7f800000) ? -1 : (int32_t)(uint32_t)c;
      os[i] = v;
    } else {
      oi[i] = -1;
      os[i] = -__int_as_float(0x7f800000);
    }
  }
  } while (0);

  // the row's logits are dead: drop the L2 lines that lie wholly inside
  // the row instead of letting them be written back
  __syncthreads();
  {
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(L);
    const uintptr_t r1 = r0 + (uintptr_t)S_kv * sizeof(float);
    const uintptr_t first = (r0 + 127) & ~(uintptr_t)127;
    for (uintptr_t a = first + (uintptr_t)tid * 128; a + 128 <= r1;
         a += (uintptr_t)NT * 128)
      discard_l2_line(reinterpret_cast<const void *>(a));
  }
}

__global__ void gather_logits_kernel(const float *__restrict__ logits,
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

// Dynamic shared memory of one selection CTA: bufA [mcap] u64, bufB
// [bcap] u64 (also the 4096-bin select histogram), keys [S_kv] u32 (at least
// 8 KB: the sort's per-warp histograms reuse it once the keys are dead).
struct SelLayout {
  int mcap, bcap, keys_cap;
  int region_u32;  // u32 slots of the key region (the bucket route stages
                   // rows that fit)
  size_t dyn;
};

SelLayout sel_layout(int S_kv, int topk, bool unstaged, int threads) {
  SelLayout l;
  // room for the candidates of a one-pass select: topk plus the rest of
  // the threshold bucket (up to kSelSlack keys, twice that for small topk)
  const int slack = topk < 1024 ? 2 * kSelSlack : kSelSlack;
  l.mcap = topk + slack < S_kv ? topk + slack : S_kv;
  l.bcap = l.mcap > kHistBins / 2 ? l.mcap : kHistBins / 2;
  // unstaged rows are never copied to shared memory whole (their keys are
  // read from L2); the region then holds the sort's per-warp counters, or
  // a row short enough to fit
  const size_t key_bytes = unstaged ? 0 : (size_t)S_kv * 4;
  const size_t whist_bytes = (size_t)(threads / 32) * 256 * 4;
  l.keys_cap = unstaged ? 0 : S_kv;
  const size_t region = key_bytes > whist_bytes ? key_bytes : whist_bytes;
  l.region_u32 = (int)(region / 4);
  l.dyn = (size_t)(l.mcap + l.bcap) * 8 + region;
  return l;
}

// Rows longer than 4096 keys (past the register route) skip the
// shared-memory copy when there are enough rows that more CTAs per SM pay
// off; a few rows (decode) keep it, so their passes stay in shared memory.
bool unstaged_rows(const Problem &p, int rows_per_seq) {
  return p.S_kv > 4096 && (long long)p.B * rows_per_seq >= 2048;
}

template <int EPT, int NT>
cudaError_t launch_sel(const Problem &p, const float *logits, int topk,
                       int32_t *out_idx, float *out_scores, cudaStream_t st,
                       int s0, int Sc) {
  const SelLayout l = sel_layout(p.S_kv, topk, unstaged_rows(p, Sc), NT);
  auto kern = topk_select_kernel<EPT, NT>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)l.dyn);
  if (e != cudaSuccess) return e;
  const long long rows = (long long)p.B * Sc;
  // launched with programmatic stream serialization: the CTAs are queued
  // while the scoring kernel runs and wait for it inside the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = l.dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, logits, p.q_pos, s0, Sc, p.S,
                            p.S_kv, p.ratio, topk, l.mcap, l.bcap, l.keys_cap,
                            l.region_u32, out_idx, out_scores);
}

}  // namespace

size_t topk_select_smem_bytes(int S_kv, int topk) {
  return sel_layout(S_kv, topk, false, kSelThreads).dyn + sizeof(SelShared);
}

// Shared memory the wide (512-thread) variant may take: its per-warp sort
// counters need 16 KB, which the key region usually covers already.
constexpr size_t kWideSmemCap = 160 * 1024;

cudaError_t launch_topk_select(const Problem &p, const float *logits, int topk,
                               int32_t *out_idx, float *out_scores,
                               int num_sms, cudaStream_t st, int s0, int Sc) {
  const bool unstaged = unstaged_rows(p, Sc);
  const int mcap = sel_layout(p.S_kv, topk, unstaged, kSelThreads).mcap;
  // Fewer rows than SMs: each row gets 512 threads, so a row's passes
  // take half the iterations (the rows run side by side anyway).
  const long long rows = (long long)p.B * Sc;
  if (rows < num_sms && mcap <= kSelThreadsWide * 8 &&
      sel_layout(p.S_kv, topk, unstaged, kSelThreadsWide).dyn <= kWideSmemCap)
    return launch_sel<8, kSelThreadsWide>(p, logits, topk, out_idx,
                                          out_scores, st, s0, Sc);
  if (mcap <= kSelThreads * 8)
    return launch_sel<8, kSelThreads>(p, logits, topk, out_idx,
                                      out_scores, st, s0, Sc);
  if (mcap <= kSelThreads * 16)
    return launch_sel<16, kSelThreads>(p, logits, topk, out_idx,
                                       out_scores, st, s0, Sc);
  return launch_sel<DSA_SEL_MAX_EPT + 2, kSelThreads>(
      p, logits, topk, out_idx, out_scores, st, s0, Sc);
}

cudaError_t launch_gather_logits(const Problem &p, const float *logits,
                                 const int32_t *in_idx, int topk,
                                 int32_t *out_idx, float *out_scores,
                                 int *status, int num_sms, cudaStream_t st) {
  const long long total = (long long)p.B * p.S * topk;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  gather_logits_kernel<<<(unsigned)blocks, 256, 0, st>>>(
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
