// index_topk: the prefill lightning-indexer forward in one persistent kernel.
// It computes the score I[t, j] = sum_h w[t,h] * ReLU(q[t,h,:] . k[j,:]) of
// every visible (query, compressed key) pair on the tcgen05 tensor cores and
// selects each row's top-k in the same CTA, so the [S, S_kv] scores never go
// to device memory: a work item's score rows live in a small per-CTA scratch
// (two item slots, a few hundred KB per SM) that stays in L2 and is reused
// item after item.
//
// Scoring is the index_scores design: one MMA tile is 128 keys (M, tensor
// memory lanes) x 256 (query, head) columns (N) x D, K-major operands with
// the 128-byte swizzle staged by TMA, two fp32 accumulators in tensor memory,
// and an epilogue in which each thread owns one key and reduces over the
// heads in its own registers.  Here the K ring is kept at 64-column chunk
// granularity (16 KB stages) so that the selection's shared memory fits next
// to two Q tiles.
//
// Warp roles (576 threads, one CTA per SM):
//   warp 0       TMA producer (Q tile per work item, K chunks through a ring)
//   warp 1       tensor-memory allocator and MMA issuer (one thread)
//   warps 2..9   epilogue: tensor memory -> registers (a tile's 128 columns
//                per warp in four 32-column quarters, the next quarter's
//                load in flight while one is reduced), ReLU, weighted head
//                sum, causal mask; each visible score goes to the item's
//                scratch row, and each row's finite value range [lo, hi] and
//                a non-finite flag are kept on the side
//   warps 10..17 selection: once an item's rows are complete they pick each
//                row's top-k from the scratch while the epilogue fills the
//                other slot with the next item
//
// Selection of one row (n visible scores, k = topk):
//   fast route  the scores are counted into NB buckets spread linearly over
//               [lo, hi] (higher score -> lower bucket; NB = 1024, 2048 or
//               4096, the smallest that holds a row of up to 4096 keys, else
//               4096).  A scan gives the
//               last bucket holding kept keys and each kept bucket's start;
//               the kept keys are scattered to their buckets, and a key's
//               final rank is its bucket's start plus the keys of the same
//               bucket that precede it (larger score, or equal score and
//               lower index).  Rows of up to 4096 keys are read once into
//               registers, longer ones twice from L2 (four 16-byte reads
//               in flight per thread).
//   exact route rows with a non-finite score, or where a kept bucket holds
//               more than 32 keys (ties, clusters, outliers): a radix select
//               over the order-preserving 32-bit keys (12 + 12 + 8 bits) finds
//               the k-th key T, every key above T and the lowest-index keys
//               equal to T are gathered, and a bitonic sort orders them by
//               (score descending, index ascending).
// Scores compare as IEEE values with -0.0 equal to +0.0 (written as +0.0);
// a kept -inf (a key masked out by the validity flags) is written as -1 /
// -inf.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kFusedThreads = 576;
constexpr int kEpiBar = 1;     // named barrier of the 8 epilogue warps
constexpr int kSelBar = 2;     // named barrier of the 8 selection warps
constexpr int kSelT = 256;     // selection threads
constexpr int kSelFirstThread = 320;
constexpr int kBins = 4096;    // fast-route buckets
constexpr int kCrowd = 32;     // most keys a kept bucket may hold
constexpr int kRegGroups = 4;  // float4 groups per thread held in registers
constexpr int kRegKeys = 4 * kRegGroups * kSelT;  // 4096
// order-preserving int of a float (for min / max with integer atomics)
constexpr int kOrdPosInf = 0x7f800000;
constexpr int kOrdNegInf = (int)(0xff800000u ^ 0x7fffffffu);

__device__ __forceinline__ int float_ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord_float(int i) {
  return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff);
}

// Bank spread for the scan, where thread t reads bins [16t, 16t + 16).
__device__ __forceinline__ uint32_t bslot(uint32_t b) {
  return b ^ ((b >> 4) & 15u);
}

// Descending bucket among NB of a score: t = sat(v * sc + off) in [0, 1]
// (sc = 1 / span, off = -lo / span), then t * (NB - 1) + 2^23 rounds to an
// integer in [2^23, 2^23 + NB - 1] whose low mantissa bits count up with v;
// their complement counts down.  Monotone (non-increasing) in v; both steps
// run on the FMA pipe.
template <int NB = kBins>
__device__ __forceinline__ uint32_t bucket_desc(float v, float sc, float off) {
  float t;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;"
      : "=f"(t)
      : "f"(v), "f"(sc), "f"(off));
  const float u = fmaf(t, (float)(NB - 1), 8388608.0f);
  return ~__float_as_uint(u) & (uint32_t)(NB - 1);
}

__host__ __device__ __forceinline__ int pow2_ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// u64 entries of the candidate buffer: the fast route needs topk + 31 (the
// kept keys of every kept bucket), the exact route pow2(topk) for its sort.
__host__ __device__ __forceinline__ int group_cap(int topk) {
  const int a = topk + kCrowd, b = pow2_ceil(topk);
  return a > b ? a : b;
}

// Selection scalars in shared memory.
struct SelMisc {
  uint32_t wsum[8];
  uint32_t weq[8];
  uint32_t sel_bin, sel_cnt;
  uint32_t flag;
  uint32_t cnt;
};

template <int H, int KC>
struct FusedSmem {
  static constexpr int kTQ = kTileCols / H;
  static constexpr int kNS = KC == 1 ? 6 : 4;  // 16 KB chunk stages
  static constexpr int kQBytes = KC * kTileCols * 128;
  static constexpr int kChunkBytes = kTileKeys * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQBytes;
  static constexpr int kOffW = kOffK + kNS * kChunkBytes;
  static constexpr int kOffBins = kOffW + kTileCols * 4;
  // per slot and row: lo, hi (order-preserving ints) and a flag
  static constexpr int kOffStats = kOffBins + kBins * 4;
  static constexpr int kStatsBytes = 2 * kTQ * 3 * 4;
  static constexpr int kOffBar = kOffStats + ((kStatsBytes + 127) / 128) * 128;
  // k_full[NS], k_empty[NS], q_full[2], q_empty[2], acc_full[2],
  // acc_empty[2], slot_full[2], slot_empty[2]
  static constexpr int kNumBars = 2 * kNS + 12;
  static constexpr int kOffMisc = kOffBar + ((kNumBars * 8 + 127) / 128) * 128;
  static constexpr int kMiscBytes = 16 + ((int)sizeof(SelMisc) + 15) / 16 * 16;
  static constexpr int kOffGroup = kOffMisc + kMiscBytes;
  static size_t bytes(int topk) {
    // + room to align the base to 1024 bytes
    return (size_t)kOffGroup + (size_t)group_cap(topk) * 8 + 1024;
  }
};

struct ItemInfo {
  int b, t0, ntiles;
};

template <int H>
__device__ __forceinline__ ItemInfo item_info(int item, int S, int B,
                                              int S_kv, int ratio,
                                              const int32_t *q_pos) {
  constexpr int TQ = kTileCols / H;
  const int n_qb = (S + TQ - 1) / TQ;
  ItemInfo it;
  const int qb = n_qb - 1 - item / B;  // longest (latest) query blocks first
  it.b = item % B;
  it.t0 = qb * TQ;
  const int t_last = min(it.t0 + TQ - 1, S - 1);
  const int nv = n_visible(row_pos(q_pos, it.b, t_last), ratio, S_kv);
  it.ntiles = (nv + kTileKeys - 1) / kTileKeys;
  return it;
}

// Zig-zag deal of items to CTAs (round r: item r*G + c, or r*G + G-1-c on
// odd rounds); -1 past the end.
__device__ __forceinline__ int item_for(int round, int n_items) {
  const int G = gridDim.x, c = blockIdx.x;
  const int idx = round * G + ((round & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

// First item with work at or after round r (ntiles = -1: none left).
template <int H>
__device__ __forceinline__ ItemInfo next_item(int r, int &round, int n_items,
                                              int S, int B, int S_kv,
                                              int ratio, const int32_t *q_pos) {
  for (;; ++r) {
    const int item = item_for(r, n_items);
    if (item < 0) break;
    const ItemInfo it = item_info<H>(item, S, B, S_kv, ratio, q_pos);
    if (it.ntiles > 0) {
      round = r;
      return it;
    }
  }
  ItemInfo none;
  none.b = 0;
  none.t0 = 0;
  none.ntiles = -1;
  round = r;
  return none;
}

// ---- selection (warps 10..17) ------------------------------------------------

__device__ __forceinline__ void sel_sync() { named_bar_sync(kSelBar, kSelT); }

// Exclusive prefix sum of one value per selection thread; `total` gets the
// sum over all of them.
__device__ __forceinline__ uint32_t sel_excl_scan(uint32_t v, int st,
                                                  SelMisc &sm,
                                                  uint32_t &total) {
  const int lane = st & 31, warp = st >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sm.wsum[warp] = incl;
  sel_sync();
  uint32_t pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSelT / 32; ++w) {
    const uint32_t c = sm.wsum[w];
    pre += w < warp ? c : 0u;
    tot += c;
  }
  sel_sync();  // wsum is rewritten by the next scan
  total = tot;
  return pre + incl - v;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void write_padding(int from, int topk, int st,
                                              int32_t *oi, float *os) {
  const float neg_inf = -__int_as_float(0x7f800000);
  for (int i = from + st; i < topk; i += kSelT) {
    __stcs(oi + i, -1);
    __stcs(os + i, neg_inf);
  }
}

// Bitonic sort of g[0..P) (P a power of two) into descending order.
__device__ __forceinline__ void sel_bitonic_desc(uint64_t *g, int P, int st) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = st; i < P / 2; i += kSelT) {
        const int lo = ((i & ~(stride - 1)) << 1) | (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t a = g[lo], b = g[hi];
        if ((a < b) == desc) {
          g[lo] = b;
          g[hi] = a;
        }
      }
      sel_sync();
    }
  }
}

// Exact route: any scores (ordered by their order-preserving keys).  Ends
// with a selection barrier.
__device__ __noinline__ void select_exact(const float *R, int n, int topk,
                                          int st, uint32_t *bins,
                                          uint64_t *grouped, SelMisc &sm,
                                          int32_t *oi, float *os) {
  const int lane = st & 31, warp = st >> 5;
  const int want = n < topk ? n : topk;
  if (n <= topk) {
    // every key is kept: gather them in any order, the sort orders them
    if (st == 0) sm.cnt = 0;
    sel_sync();
    for (int j = st; j < n; j += kSelT) {
      const uint32_t u = ordered_key(__ldcg(R + j));
      const uint32_t pos = atomicAdd(&sm.cnt, 1u);
      grouped[pos] = ((uint64_t)u << 32) | (0xffffffffu - (uint32_t)j);
    }
    sel_sync();
  } else {
    // radix select of the topk-th largest key: 12, 12 and 8 bits
    uint32_t prefix = 0, pmask = 0;
    int need = topk;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 20 : (pass == 1 ? 8 : 0);
      const int nb = pass == 2 ? 256 : kBins;
      const uint32_t dmask = (uint32_t)nb - 1u;
      for (int i = st; i < nb; i += kSelT) bins[i] = 0u;
      sel_sync();
      for (int j = st; j < n; j += kSelT) {
        const uint32_t u = ordered_key(__ldcg(R + j));
        if ((u & pmask) == prefix) atomicAdd(&bins[(u >> shift) & dmask], 1u);
      }
      sel_sync();
      // thread t owns digits [o*per, o*per + per) with o = 255 - t, so the
      // exclusive scan in thread order counts the keys above its digits
      const int per = nb / kSelT;
      const int o = kSelT - 1 - st;
      uint32_t lsum = 0;
      for (int i = 0; i < per; ++i) lsum += bins[o * per + i];
      uint32_t total;
      const uint32_t above = sel_excl_scan(lsum, st, sm, total);
      if (above < (uint32_t)need && (uint32_t)need <= above + lsum) {
        uint32_t run = above;
        for (int i = per - 1; i >= 0; --i) {
          const uint32_t c = bins[o * per + i];
          if (run + c >= (uint32_t)need) {
            sm.sel_bin = (uint32_t)(o * per + i);
            sm.sel_cnt = run;
            break;
          }
          run += c;
        }
      }
      sel_sync();
      need -= (int)sm.sel_cnt;
      prefix |= sm.sel_bin << shift;
      pmask |= dmask << shift;
      sel_sync();  // the digit is read before the bins are cleared again
    }
    const uint32_t T = prefix;
    const int n_gt = topk - need;
    // keys above T in any order; keys equal to T by ascending index, the
    // first `need` of them.  Warp w walks the contiguous range
    // [w * seg, (w + 1) * seg).
    const int seg = ((n + kSelT - 1) / kSelT) * 32;
    const int lo = warp * seg, hi = min(n, lo + seg);
    const uint32_t lt = lanemask_lt();
    uint32_t ceq = 0;
    for (int c = lo; c < lo + seg; c += 32) {
      const int j = c + lane;
      const uint32_t u = j < hi ? ordered_key(__ldcg(R + j)) : 0u;
      ceq += __popc(__ballot_sync(0xffffffffu, j < hi && u == T));
    }
    if (lane == 0) sm.weq[warp] = ceq;
    if (st == 0) sm.cnt = 0;
    sel_sync();
    uint32_t epos = 0;
    for (int w = 0; w < warp; ++w) epos += sm.weq[w];
    for (int c = lo; c < lo + seg; c += 32) {
      const int j = c + lane;
      const uint32_t u = j < hi ? ordered_key(__ldcg(R + j)) : 0u;
      const bool is_gt = j < hi && u > T;
      const bool is_eq = j < hi && u == T;
      const uint32_t beq = __ballot_sync(0xffffffffu, is_eq);
      const uint64_t e = ((uint64_t)u << 32) | (0xffffffffu - (uint32_t)j);
      if (is_gt) grouped[atomicAdd(&sm.cnt, 1u)] = e;
      if (is_eq) {
        const uint32_t r = epos + __popc(beq & lt);
        if (r < (uint32_t)need) grouped[n_gt + r] = e;
      }
      epos += __popc(beq);
    }
    sel_sync();
  }
  const int P = pow2_ceil(want);
  for (int i = want + st; i < P; i += kSelT) grouped[i] = 0ull;
  sel_sync();
  sel_bitonic_desc(grouped, P, st);
  const float neg_inf = -__int_as_float(0x7f800000);
  for (int i = st; i < topk; i += kSelT) {
    if (i < want) {
      const uint64_t e = grouped[i];
      const float v = key_to_float((uint32_t)(e >> 32));
      __stcs(oi + i, v == neg_inf ? -1 : (int32_t)(0xffffffffu - (uint32_t)e));
      __stcs(os + i, v);
    } else {
      __stcs(oi + i, -1);
      __stcs(os + i, neg_inf);
    }
  }
  sel_sync();
}

// Fast route after the histogram: scan, threshold bucket and kept buckets'
// starts.  Returns false (block-uniform) when a kept bucket is crowded.
// On return m = keys in the kept buckets, thr = last kept bucket (or -1).
template <int NB = kBins>
__device__ __forceinline__ bool bucket_scan(int topk, int st, uint32_t *bins,
                                            SelMisc &sm, int &m, int &thr) {
  constexpr int per = NB / kSelT;  // buckets per thread
  const int lane = st & 31;
  uint32_t c[per];
  uint32_t lsum = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    c[i] = bins[bslot(st * per + i)];
    lsum += c[i];
  }
  uint32_t total;
  const uint32_t above = sel_excl_scan(lsum, st, sm, total);
  const uint32_t want = total < (uint32_t)topk ? total : (uint32_t)topk;
  uint32_t occ = 0, run = above;
#pragma unroll
  for (int i = 0; i < per; ++i) {
    const uint32_t b = (uint32_t)(st * per + i);
    if (run < want) {
      bins[bslot(b)] = (run << 16) | c[i];
      occ = max(occ, c[i]);
      if (run + c[i] >= want) {
        sm.sel_bin = b;
        sm.sel_cnt = run + c[i];
      }
    }
    run += c[i];
  }
  occ = __reduce_max_sync(0xffffffffu, occ);
  if (lane == 0 && occ > (uint32_t)kCrowd) sm.flag = 1u;
  sel_sync();
  const bool crowded = sm.flag != 0u;
  if (want == 0) {
    m = 0;
    thr = -1;
  } else {
    m = (int)sm.sel_cnt;
    thr = (int)sm.sel_bin;
  }
  sel_sync();  // every thread has read sel_* and the flag
  return !crowded;
}

// Rank of each kept key inside its bucket and the output row.
__device__ __forceinline__ void bucket_rank_write(int m, int topk, int st,
                                                  const uint32_t *bins,
                                                  const uint64_t *grouped,
                                                  int32_t *oi, float *os) {
  for (int p = st; p < m; p += kSelT) {
    const uint64_t cv = grouped[p];
    const uint32_t lo32 = (uint32_t)cv;
    const uint32_t e = bins[bslot(lo32 >> 20)];
    const int end = (int)(e >> 16), start = end - (int)(e & 0xffffu);
    int r = start;
    for (int q = start; q < end; ++q) r += grouped[q] > cv;
    if (r < topk) {
      __stcs(oi + r, (int32_t)(0xfffffu - (lo32 & 0xfffffu)));
      __stcs(os + r, key_to_float((uint32_t)(cv >> 32)));
    }
  }
  write_padding(m, topk, st, oi, os);
}

// The register route of select_row() for a row of n <= NB scores, over NB
// buckets (NB = 1024, 2048 or 4096, the smallest that holds the row: the
// clear and the scan cost per bucket).  Ends with a selection barrier.
template <int NB>
__device__ __forceinline__ void select_reg(const float *R, int n, int topk,
                                           float lo, float hi, int st,
                                           uint32_t *bins, uint64_t *grouped,
                                           SelMisc &sm, int32_t *oi,
                                           float *os) {
  constexpr int G = NB / (4 * kSelT);  // float4 groups per thread
  const float neg_inf = -__int_as_float(0x7f800000);
  float sc = 0.f, off = 0.f;  // bucket map, see bucket_desc
  if (hi > lo) {
    const float span = hi - lo;
    if (span <= 3.402823466e38f) {
      sc = fminf(1.f / span, 1e30f);
      off = -lo * sc;
    }
  }
  {
    uint2 *b2 = reinterpret_cast<uint2 *>(bins);
    for (int i = st; i < NB / 2; i += kSelT) b2[i] = make_uint2(0u, 0u);
  }
  if (st == 0) sm.flag = 0u;
  int m, thr;
  // thread st owns keys 4 (st + 256 i) + c, i < G
  float kv[4 * G];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const int j0 = 4 * (st + kSelT * i);
    float4 f = make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
    if (4 * kSelT * i < n && j0 < n)
      f = __ldcg(reinterpret_cast<const float4 *>(R + j0));
    kv[4 * i + 0] = j0 + 0 < n ? f.x : neg_inf;
    kv[4 * i + 1] = j0 + 1 < n ? f.y : neg_inf;
    kv[4 * i + 2] = j0 + 2 < n ? f.z : neg_inf;
    kv[4 * i + 3] = j0 + 3 < n ? f.w : neg_inf;
  }
  sel_sync();  // bins cleared
#pragma unroll
  for (int i = 0; i < G; ++i) {
    if (4 * kSelT * i >= n) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float v = kv[4 * i + c];
      if (v != neg_inf)
        atomicAdd(&bins[bslot(bucket_desc<NB>(v, sc, off))], 1u);
    }
  }
  sel_sync();
  if (!bucket_scan<NB>(topk, st, bins, sm, m, thr)) {
    select_exact(R, n, topk, st, bins, grouped, sm, oi, os);
    return;
  }
#pragma unroll
  for (int i = 0; i < G; ++i) {
    if (4 * kSelT * i >= n) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float v = kv[4 * i + c];
      if (v == neg_inf) continue;
      const uint32_t b = bucket_desc<NB>(v, sc, off);
      if ((int)b <= thr) {
        const int j = 4 * (st + kSelT * i) + c;
        const uint32_t pos = atomicAdd(&bins[bslot(b)], 1u << 16) >> 16;
        grouped[pos] = ((uint64_t)ordered_key(v) << 32) | (b << 20) |
                       (0xfffffu - (uint32_t)j);
      }
    }
  }
  sel_sync();
  bucket_rank_write(m, topk, st, bins, grouped, oi, os);
  sel_sync();
}

// One row's selection.  R: the row's n scores (scratch, 16-byte aligned,
// readable up to n rounded up to 4); [lo, hi]: the range of its finite
// unmasked scores; bad: some score is non-finite.  Ends with a selection
// barrier.
__device__ __forceinline__ void select_row(const float *R, int n, int topk,
                                           float lo, float hi, bool bad,
                                           int st, uint32_t *bins,
                                           uint64_t *grouped, SelMisc &sm,
                                           int32_t *oi, float *os) {
  const float neg_inf = -__int_as_float(0x7f800000);
  if (n == 0) {
    write_padding(0, topk, st, oi, os);
    sel_sync();
    return;
  }
  if (bad) {
    select_exact(R, n, topk, st, bins, grouped, sm, oi, os);
    return;
  }
  if (n <= kRegKeys / 4) {
    select_reg<kBins / 4>(R, n, topk, lo, hi, st, bins, grouped, sm, oi, os);
    return;
  }
  if (n <= kRegKeys / 2) {
    select_reg<kBins / 2>(R, n, topk, lo, hi, st, bins, grouped, sm, oi, os);
    return;
  }
  if (n <= kRegKeys) {
    select_reg<kBins>(R, n, topk, lo, hi, st, bins, grouped, sm, oi, os);
    return;
  }
  float sc = 0.f, off = 0.f;  // bucket map, see bucket_desc
  if (hi > lo) {
    const float span = hi - lo;
    if (span <= 3.402823466e38f) {
      sc = fminf(1.f / span, 1e30f);
      off = -lo * sc;
    }
  }
  {
    uint2 *b2 = reinterpret_cast<uint2 *>(bins);
    for (int i = st; i < kBins / 2; i += kSelT) b2[i] = make_uint2(0u, 0u);
  }
  if (st == 0) sm.flag = 0u;
  int m, thr;
  sel_sync();  // bins cleared
  // both passes over the row keep four 16-byte L2 reads in flight per
  // thread before using them
  const float4 ninf4 = make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
  for (int g0 = st; 4 * g0 < n; g0 += 4 * kSelT) {
    float4 f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSelT;
      f[u] = 4 * g < n ? __ldcg(reinterpret_cast<const float4 *>(R) + g)
                       : ninf4;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSelT;
      const float vv[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (4 * g + c < n && vv[c] != neg_inf)
          atomicAdd(&bins[bslot(bucket_desc(vv[c], sc, off))], 1u);
    }
  }
  sel_sync();
  if (!bucket_scan(topk, st, bins, sm, m, thr)) {
    select_exact(R, n, topk, st, bins, grouped, sm, oi, os);
    return;
  }
  for (int g0 = st; 4 * g0 < n; g0 += 4 * kSelT) {
    float4 f[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSelT;
      f[u] = 4 * g < n ? __ldcg(reinterpret_cast<const float4 *>(R) + g)
                       : ninf4;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * kSelT;
      const float vv[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = 4 * g + c;
        if (j >= n || vv[c] == neg_inf) continue;
        const uint32_t b = bucket_desc(vv[c], sc, off);
        if ((int)b <= thr) {
          const uint32_t pos = atomicAdd(&bins[bslot(b)], 1u << 16) >> 16;
          grouped[pos] = ((uint64_t)ordered_key(vv[c]) << 32) | (b << 20) |
                         (0xfffffu - (uint32_t)j);
        }
      }
    }
  }
  sel_sync();
  bucket_rank_write(m, topk, st, bins, grouped, oi, os);
  sel_sync();
}

// ---- the kernel ----------------------------------------------------------------

template <int H, int KC, bool KV>
__global__ void __launch_bounds__(kFusedThreads, 1)
    index_topk_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const float *__restrict__ w,
                      const int32_t *__restrict__ q_pos,
                      const uint8_t *__restrict__ kv_valid,
                      float *__restrict__ scratch, int row_stride, int S,
                      int B, int S_kv, int ratio, int topk,
                      int32_t *__restrict__ out_idx,
                      float *__restrict__ out_scores, int *status) {
  using L = FusedSmem<H, KC>;
  constexpr int NS = L::kNS;
  constexpr int TQ = kTileCols / H;  // query rows per work item
  constexpr int QH = TQ / 2;         // rows per epilogue column half
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileKeys, kTileCols);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);

  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sK = base + L::kOffK;
  float *sW = reinterpret_cast<float *>(smem + L::kOffW);
  uint32_t *bins = reinterpret_cast<uint32_t *>(smem + L::kOffBins);
  int *stats = reinterpret_cast<int *>(smem + L::kOffStats);
  const uint32_t bars = base + L::kOffBar;
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (NS + s); };
  auto q_full = [&](int i) { return bars + 8u * (2 * NS + i); };
  auto q_empty = [&](int i) { return bars + 8u * (2 * NS + 2 + i); };
  auto acc_full = [&](int i) { return bars + 8u * (2 * NS + 4 + i); };
  auto acc_empty = [&](int i) { return bars + 8u * (2 * NS + 6 + i); };
  auto slot_full = [&](int i) { return bars + 8u * (2 * NS + 8 + i); };
  auto slot_empty = [&](int i) { return bars + 8u * (2 * NS + 10 + i); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);
  SelMisc &sm = *reinterpret_cast<SelMisc *>(smem + L::kOffMisc + 16);
  uint64_t *grouped = reinterpret_cast<uint64_t *>(smem + L::kOffGroup);
  // stats of slot s, row r: lo, hi, flag
  auto stat = [&](int s, int r) { return stats + (s * TQ + r) * 3; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = ((S + TQ - 1) / TQ) * B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(q_full(a), 1);
      mbar_init(q_empty(a), 1);
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 8);   // one arrival per epilogue warp
      mbar_init(slot_full(a), 8);   // one arrival per epilogue warp
      mbar_init(slot_empty(a), 1);  // the selection, once per item
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // q is read once: keep it from pushing the score scratch out of L2
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t kst = 0, kph = 0, nq = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_for(r, n_items);
        if (item < 0) break;
        const ItemInfo it = item_info<H>(item, S, B, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq & 1;
        const uint32_t qph = (nq >> 1) & 1u;
        ++nq;
        if (!(ok = wait_bar(q_empty(qs), qph ^ 1u, abort_flag, status))) break;
        mbar_arrive_expect_tx(q_full(qs), L::kQBytes);
        for (int c = 0; c < KC; ++c)
          tma_load_4d_hint(sQ + qs * L::kQBytes + c * (kTileCols * 128),
                           &tm_q, q_full(qs), c * kChunk, 0, it.b, it.t0,
                           pol_q);
        for (int tile = 0; tile < it.ntiles && ok; ++tile) {
          for (int c = 0; c < KC; ++c) {
            if (!(ok = wait_bar(k_empty(kst), kph ^ 1u, abort_flag, status)))
              break;
            mbar_arrive_expect_tx(k_full(kst), L::kChunkBytes);
            tma_load_3d(sK + kst * L::kChunkBytes, &tm_k, k_full(kst),
                        c * kChunk, it.b, tile * kTileKeys);
            if (++kst == NS) {
              kst = 0;
              kph ^= 1u;
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t kst = 0, kph = 0, nq = 0, acc = 0, aph = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_for(r, n_items);
        if (item < 0) break;
        const ItemInfo it = item_info<H>(item, S, B, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq & 1;
        const uint32_t qph = (nq >> 1) & 1u;
        ++nq;
        if (!(ok = wait_bar(q_full(qs), qph, abort_flag, status))) break;
        const uint32_t sQi = sQ + qs * L::kQBytes;
        for (int tile = 0; tile < it.ntiles && ok; ++tile) {
          if (!(ok = wait_bar(acc_empty(acc), aph ^ 1u, abort_flag, status)))
            break;
          const uint32_t d_tmem = tmem + acc * kTileCols;
          for (int c = 0; c < KC; ++c) {
            if (!(ok = wait_bar(k_full(kst), kph, abort_flag, status))) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk) {
              const uint64_t ad =
                  sdesc_k_sw128(sK + kst * L::kChunkBytes + kk * 32);
              const uint64_t bd =
                  sdesc_k_sw128(sQi + c * (kTileCols * 128) + kk * 32);
              mma_bf16(d_tmem, ad, bd, kIdesc, (c | kk) != 0);
            }
            mma_commit(k_empty(kst));  // chunk stage reusable when done
            if (++kst == NS) {
              kst = 0;
              kph ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(acc_full(acc));  // accumulator ready
          if (tile == it.ntiles - 1) mma_commit(q_empty(qs));
          acc ^= 1u;
          if (acc == 0) aph ^= 1u;
        }
      }
    }
  } else if (warp < 10) {
    // ---------------- epilogue (warps 2..9) ----------------
    const int ew = warp - 2;          // 0..7
    const int sp = warp & 3;          // tensor-memory lane quarter
    const int half = ew >> 2;         // which 128 columns
    const int et = threadIdx.x - 64;  // 0..255
    uint32_t acc = 0, aph = 0;
    bool ok = true;
    const int tq_mine = et / H, h_mine = et % H;  // the weight this thread loads
    auto weight_of = [&](const ItemInfo &it) -> float {
      const int t = it.t0 + tq_mine;
      return t < S ? __ldg(w + ((size_t)t * B + it.b) * H + h_mine) : 0.f;
    };
    int r = 0;
    ItemInfo it =
        next_item<H>(0, r, n_items, S, B, S_kv, ratio, q_pos);
    float w_next = it.ntiles > 0 ? weight_of(it) : 0.f;
    const float neg_inf = -__int_as_float(0x7f800000);
    for (uint32_t n_it = 0; it.ntiles > 0; ++n_it) {
      const int slot = (int)(n_it & 1u);
      // the selection has finished with this slot's previous item
      bool got = wait_bar(slot_empty(slot), ((n_it >> 1) & 1u) ^ 1u,
                          abort_flag, status);
      if (named_bar_or(kEpiBar, 256, !(ok && got))) break;
      sW[et] = 0.5f * w_next;  // halved: see the ReLU below
      if (et < TQ) {
        int *s3 = stat(slot, et);
        s3[0] = kOrdPosInf;
        s3[1] = kOrdNegInf;
        s3[2] = 0;
      }
      named_bar_sync(kEpiBar, 256);
      int r_next;
      const ItemInfo nx =
          next_item<H>(r + 1, r_next, n_items, S, B, S_kv, ratio, q_pos);
      if (nx.ntiles > 0) w_next = weight_of(nx);
      const long long qbase = row_pos(q_pos, it.b, 0);
      float *srow = scratch + (size_t)(blockIdx.x * 2 + slot) * TQ * row_stride;
      // keys visible to the half's rows (none past the last row): key j of
      // a row counts iff j < nvq
      int nvq[QH];
#pragma unroll
      for (int qq = 0; qq < QH; ++qq) {
        const int t = it.t0 + half * QH + qq;
        nvq[qq] = t < S ? n_visible(qbase + t, ratio, S_kv) : 0;
      }

      float lo[QH], hi[QH];
#pragma unroll
      for (int i = 0; i < QH; ++i) {
        lo[i] = __int_as_float(0x7f800000);
        hi[i] = neg_inf;
      }
      float chk = 0.f;  // becomes NaN once a score is non-finite

      for (int tile = 0; tile < it.ntiles; ++tile) {
        bool g = wait_bar(acc_full(acc), aph, abort_flag, status);
        g = __all_sync(0xffffffffu, g);
        if (!g) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int j = tile * kTileKeys + sp * 32 + lane;
        const bool kv_ok = !KV || j >= S_kv ||
                           __ldg(kv_valid + (size_t)j * B + it.b) != 0;
        // This warp's 128 columns in four quarters of 32, double-buffered:
        // quarter qt + 1 is loaded while quarter qt is reduced.  Quarter qt
        // holds heads [32 qt mod H, +32) of the half's row 32 qt / H; a row's
        // sum runs over its heads in increasing order whatever the split
        // (the same order as the two-kernel scorer).
        static_assert(H >= 32, "a quarter holds one row's heads");
        const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16) +
                               acc * kTileCols + half * 128;
        uint32_t v[2][32];
        tmem_ld32(taddr, v[0]);
        tmem_ld_wait();
        reg_fence32(v[0]);
        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int qt = 0; qt < 4; ++qt) {
          const int cur = qt & 1;
          if (qt < 3) tmem_ld32(taddr + 32 * (qt + 1), v[cur ^ 1]);
          const int qq = (32 * qt) / H;  // row within the half
          const int h0 = (32 * qt) % H;  // first head of the quarter
          const int tq = half * QH + qq;
          if (h0 == 0) acc2 = make_float2(0.f, 0.f);
          const float4 *wq4 =
              reinterpret_cast<const float4 *>(sW + tq * H + h0);
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 wv = wq4[h >> 2];
            const float2 r01 = relu2x2(__uint_as_float(v[cur][h]),
                                       __uint_as_float(v[cur][h + 1]));
            const float2 r23 = relu2x2(__uint_as_float(v[cur][h + 2]),
                                       __uint_as_float(v[cur][h + 3]));
            acc2 = __ffma2_rn(make_float2(wv.x, wv.y), r01, acc2);
            acc2 = __ffma2_rn(make_float2(wv.z, wv.w), r23, acc2);
          }
          if (qt < 3) {
            tmem_ld_wait();
            reg_fence32(v[cur ^ 1]);
          }
          if (qt == 2) {
            // the last quarter has landed: the accumulator is free
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty(acc));
          }
          if (h0 + 32 < H) continue;  // the row goes on in the next quarter
          const float score = acc2.x + acc2.y;
          if (j < nvq[qq]) {
            float *dst = srow + (size_t)tq * row_stride + j;
            if (kv_ok) {
              *dst = score;
              lo[qq] = fminf(lo[qq], score);
              hi[qq] = fmaxf(hi[qq], score);
              chk = fmaf(score, 0.f, chk);
            } else {
              *dst = neg_inf;  // not a candidate: sorts last
            }
          }
        }
        acc ^= 1u;
        if (acc == 0) aph ^= 1u;
      }
      if (ok) {
        // the item's rows are complete: publish their ranges and hand the
        // slot to the selection.  (A warp whose wait gave up publishes
        // nothing; the slot never fills, the selection's bounded wait sees
        // the abort flag, and every epilogue warp stops together at the
        // next item's barrier.)
        __threadfence_block();
        const bool bad = __any_sync(0xffffffffu, chk != chk);
#pragma unroll
        for (int qq = 0; qq < QH; ++qq) {
          const int tq = half * QH + qq;
          const int lo_i = __reduce_min_sync(0xffffffffu, float_ord(lo[qq]));
          const int hi_i = __reduce_max_sync(0xffffffffu, float_ord(hi[qq]));
          if (lane == 0) {
            int *s3 = stat(slot, tq);
            atomicMin(s3 + 0, lo_i);
            atomicMax(s3 + 1, hi_i);
            if (bad) atomicOr(s3 + 2, 1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(slot_full(slot));
      }
      it = nx;
      r = r_next;
    }
  } else {
    // ---------------- selection (warps 10..17) ----------------
    const int st = threadIdx.x - kSelFirstThread;  // 0..255
    uint32_t n_it = 0;  // items with work so far (they take the slots)
    for (int r = 0;; ++r) {
      const int item = item_for(r, n_items);
      if (item < 0) break;
      const ItemInfo it = item_info<H>(item, S, B, S_kv, ratio, q_pos);
      if (it.ntiles == 0) {
        // no row of the item sees a key: nothing was scored, every slot of
        // its rows is padding
        for (int tq = 0; tq < TQ; ++tq) {
          const int t = it.t0 + tq;
          if (t >= S) break;
          const size_t orow = ((size_t)it.b * S + t) * topk;
          write_padding(0, topk, st, out_idx + orow, out_scores + orow);
        }
        continue;
      }
      const int slot = (int)(n_it & 1u);
      const bool got =
          wait_bar(slot_full(slot), (n_it >> 1) & 1u, abort_flag, status);
      if (named_bar_or(kSelBar, kSelT, !got)) break;
      const float *srow =
          scratch + (size_t)(blockIdx.x * 2 + slot) * TQ * row_stride;
      for (int tq = 0; tq < TQ; ++tq) {
        const int t = it.t0 + tq;
        if (t >= S) break;
        const int nv = n_visible(row_pos(q_pos, it.b, t), ratio, S_kv);
        const int *s3 = stat(slot, tq);
        const float lo = ord_float(s3[0]), hi = ord_float(s3[1]);
        const bool bad = s3[2] != 0;
        const size_t orow = ((size_t)it.b * S + t) * topk;
        select_row(srow + (size_t)tq * row_stride, nv, topk, lo, hi, bad, st,
                   bins, grouped, sm, out_idx + orow, out_scores + orow);
      }
      // the slot's score rows are dead: drop their L2 lines instead of
      // letting them be written back (rows start on 128-byte lines)
      for (int tq = 0; tq < TQ; ++tq) {
        const int t = it.t0 + tq;
        if (t >= S) break;
        const int nv = n_visible(row_pos(q_pos, it.b, t), ratio, S_kv);
        const float *row = srow + (size_t)tq * row_stride;
        for (int l = st; l < (nv + 31) / 32; l += kSelT)
          discard_l2_line(row + 32 * l);
      }
      sel_sync();  // every read and discard of the slot precedes its reuse
      if (st == 0) mbar_arrive(slot_empty(slot));
      ++n_it;
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int H, int KC, bool KV>
cudaError_t launch_hk(const Problem &p, const CUtensorMap &tm_q,
                      const CUtensorMap &tm_k, int topk, float *scratch,
                      int32_t *out_idx, float *out_scores, int *status,
                      int num_sms, cudaStream_t st) {
  constexpr int TQ = kTileCols / H;
  auto kern = index_topk_kernel<H, KC, KV>;
  const size_t smem = FusedSmem<H, KC>::bytes(topk);
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long n_items = (long long)((p.S + TQ - 1) / TQ) * p.B;
  long long grid = n_items < num_sms ? n_items : num_sms;
  if (grid > kIndexTopkMaxCtas) grid = kIndexTopkMaxCtas;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, kFusedThreads, smem, st>>>(
      tm_q, tm_k, p.w, p.q_pos, p.kv_valid, scratch,
      index_topk_row_stride(p.S_kv), p.S, p.B, p.S_kv, p.ratio, topk, out_idx,
      out_scores, status);
  return cudaGetLastError();
}

template <int H, int KC>
cudaError_t launch_h(const Problem &p, const CUtensorMap &tm_q,
                     const CUtensorMap &tm_k, int topk, float *scratch,
                     int32_t *out_idx, float *out_scores, int *status,
                     int num_sms, cudaStream_t st) {
  return p.kv_valid
             ? launch_hk<H, KC, true>(p, tm_q, tm_k, topk, scratch, out_idx,
                                      out_scores, status, num_sms, st)
             : launch_hk<H, KC, false>(p, tm_q, tm_k, topk, scratch, out_idx,
                                       out_scores, status, num_sms, st);
}

template <int KC>
cudaError_t launch_kc(const Problem &p, const CUtensorMap &tm_q,
                      const CUtensorMap &tm_k, int topk, float *scratch,
                      int32_t *out_idx, float *out_scores, int *status,
                      int num_sms, cudaStream_t st) {
  switch (p.H) {
    case 32:
      return launch_h<32, KC>(p, tm_q, tm_k, topk, scratch, out_idx,
                              out_scores, status, num_sms, st);
    case 64:
      return launch_h<64, KC>(p, tm_q, tm_k, topk, scratch, out_idx,
                              out_scores, status, num_sms, st);
    case 128:
      return launch_h<128, KC>(p, tm_q, tm_k, topk, scratch, out_idx,
                               out_scores, status, num_sms, st);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

// Score rows start on 128-byte lines, and one line more than S_kv needs
// keeps rows of power-of-two length from falling into the same L2 sets.
int index_topk_row_stride(int S_kv) { return (S_kv + 31) / 32 * 32 + 32; }

size_t index_topk_smem_bytes(int H, int D, int topk) {
  const bool k1 = D <= kChunk;
  switch (H) {
    case 32: return k1 ? FusedSmem<32, 1>::bytes(topk) : FusedSmem<32, 2>::bytes(topk);
    case 64: return k1 ? FusedSmem<64, 1>::bytes(topk) : FusedSmem<64, 2>::bytes(topk);
    case 128: return k1 ? FusedSmem<128, 1>::bytes(topk) : FusedSmem<128, 2>::bytes(topk);
    default: return 0;
  }
}

bool index_topk_supported(int S, int H, int D, int S_kv, int topk) {
  if (H != 32 && H != 64 && H != 128) return false;
  if (S < kTileCols / H) return false;  // decode-shaped rows
  if (topk > kIndexTopkMaxTopk || S_kv >= (1 << 20)) return false;
  return index_topk_smem_bytes(H, D, topk) <= kIndexTopkMaxSmem;
}

size_t index_topk_scratch_bytes(int H, int S_kv) {
  const int TQ = kTileCols / H;
  return (size_t)kIndexTopkMaxCtas * 2 * TQ * index_topk_row_stride(S_kv) *
         sizeof(float);
}

cudaError_t launch_index_topk(const Problem &p, const CUtensorMap &tm_q,
                              const CUtensorMap &tm_k, int topk,
                              float *scratch, int32_t *out_idx,
                              float *out_scores, int *status, int num_sms,
                              cudaStream_t st) {
  if (p.D <= kChunk)
    return launch_kc<1>(p, tm_q, tm_k, topk, scratch, out_idx, out_scores,
                        status, num_sms, st);
  return launch_kc<2>(p, tm_q, tm_k, topk, scratch, out_idx, out_scores,
                      status, num_sms, st);
}

}  // namespace dsa
