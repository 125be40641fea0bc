// gather_scores: lightning-indexer scores at caller-given key indices
// (DeepSeek-V4 SBHD indexer, "tilelang_indexer" page: the optional
// topk_indices input of v4_lighting_indexer, whose scores are taken at the
// given positions instead of selected), computed on the tensor cores from
// the gathered keys, without the dense logits.
//
// A work item is (query row r = b*S + s, chunk of `tpi` tiles), a tile being
// 128 consecutive index slots of the row.  For each tile the gather warps
// copy the 128 key rows the slots name into one K stage, in the layout a
// 128-byte-swizzled TMA box of 128 dense keys would have, and the MMA
// multiplies them with the row's query: M = 128 gathered keys, N = H heads,
// K = D.  The epilogue reduces the weighted ReLU over the heads for its
// slot, masks slots whose index is -1, out of range or not visible to the
// row, and writes score and index straight to the outputs.
//
// The key rows are scattered 256-byte reads (L2-resident for the long
// contexts this path serves), so the copies are 16-byte cp.async from
// several warps: many requests in flight from the load/store units move
// scattered rows several times faster than TMA row gathers issued by one
// thread each.  Every gather lane arrives on the stage's barrier once its
// copies have landed (cp.async.mbarrier.arrive), so the gather warps never
// wait on their own copies; the MMA thread, having observed the full
// stage, issues a generic-to-async proxy fence before the tensor core reads
// it.
//
// The slots' indices reach shared memory through a ring of 4-byte cp.async
// copies that the fetch warp runs up to kIdxSlots tiles ahead of the
// epilogue, so index-load latency does not stall the gathers; the epilogue
// reads the same ring for masking and for the copied-through indices.
//
// Warp roles (one CTA per SM, persistent): warp 0 index and query fetch,
// warps 1..W key gathers (W = 8, or 4 for H = 128), warp W+1 TMEM
// allocator and MMA issuer, warps W+2..W+5 epilogue.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

// Key-gather warps: as many as the register file allows next to the
// epilogue's H accumulator registers per thread (the copies are bound by
// how fast the warps issue them).
template <int H>
struct GatRoles {
  static constexpr int kGatWarps = H <= 64 ? 8 : 4;
  static constexpr int kThreads = 32 * (kGatWarps + 6);
  static constexpr int kMmaWarp = kGatWarps + 1;
  static constexpr int kEpiWarp0 = kGatWarps + 2;  // first of four
  static_assert(kTileKeys % kGatWarps == 0, "rows split evenly over warps");
};
constexpr int kIdxSlots = 32;  // index ring, in tiles of 128 slots
constexpr int kGatAcc = 4;     // TMEM accumulators

template <int H, int KC>
struct GatSmem {
  static constexpr int kStages = KC == 1 ? 8 : (H <= 64 ? 5 : 4);
  static constexpr int kQSlots = 2;
  static constexpr int kQBytes = KC * H * 128;          // one Q tile
  static constexpr int kKBytes = KC * kTileKeys * 128;  // one gathered stage
  static constexpr int kIdxBytes = kTileKeys * 4;       // one index tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kQBytes;
  static constexpr int kOffIdx = kOffK + kStages * kKBytes;
  static constexpr int kOffW = kOffIdx + kIdxSlots * kIdxBytes;
  static constexpr int kOffBar = kOffW + 2 * H * 4;
  // k_full[S], k_empty[S], q_full[Q], q_empty[Q], i_full[I], i_empty[I],
  // acc_full[A], acc_empty[A]
  static constexpr int kNumBars =
      2 * kStages + 2 * kQSlots + 2 * kIdxSlots + 2 * kGatAcc;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
  // TMEM columns: kGatAcc accumulators of H columns, a power of two >= 32
  static constexpr uint32_t kTmemCols =
      kGatAcc * H < 32 ? 32u : (uint32_t)(kGatAcc * H);
};

// Walks this CTA's tiles in order: items round by round (zig-zag over the
// CTAs), each item's tiles in order.  Every role walks the same sequence.
struct GatCursor {
  int round, item, row, b, s, tile, tile_end;
  bool valid;
};

struct GatGeom {
  int rows, S, ntiles, tpi, nchunks, n_items;
};

__device__ __forceinline__ int gat_item_for(int round, int n_items) {
  const int G = gridDim.x, c = blockIdx.x;
  const long long idx =
      (long long)round * G + ((round & 1) ? (G - 1 - c) : c);
  return idx < n_items ? (int)idx : -1;
}

// Item i covers chunk (i / rows) of row (i % rows).
__device__ __forceinline__ void gat_set_item(GatCursor &c, const GatGeom &g) {
  c.item = gat_item_for(c.round, g.n_items);
  c.valid = c.item >= 0;
  if (!c.valid) return;
  c.row = c.item % g.rows;
  const int chunk = c.item / g.rows;
  c.b = c.row / g.S;
  c.s = c.row % g.S;
  c.tile = chunk * g.tpi;
  const int e = c.tile + g.tpi;
  c.tile_end = e < g.ntiles ? e : g.ntiles;
}

__device__ __forceinline__ GatCursor gat_begin(const GatGeom &g) {
  GatCursor c;
  c.round = 0;
  gat_set_item(c, g);
  return c;
}

// Advances by one tile; returns true when a new item starts.
__device__ __forceinline__ bool gat_next(GatCursor &c, const GatGeom &g) {
  if (++c.tile < c.tile_end) return false;
  ++c.round;
  gat_set_item(c, g);
  return true;
}

template <int H, int KC>
__global__ void __launch_bounds__(GatRoles<H>::kThreads, 1)
    gather_scores_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const uint8_t *__restrict__ k,
                         const float *__restrict__ w,
                         const int32_t *__restrict__ q_pos,
                         const int32_t *__restrict__ in_idx, GatGeom g,
                         int B, int D, int S_kv, int ratio, int topk,
                         int32_t *__restrict__ out_idx,
                         float *__restrict__ out_scores, int *status) {
  using L = GatSmem<H, KC>;
  constexpr int kGatWarps = GatRoles<H>::kGatWarps;
  constexpr int kMmaWarp = GatRoles<H>::kMmaWarp;
  constexpr int kEpiWarp0 = GatRoles<H>::kEpiWarp0;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileKeys, H);
  constexpr int NS = L::kStages, NQ = L::kQSlots;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sK = base + L::kOffK;
  const int32_t *sIdx = reinterpret_cast<const int32_t *>(smem + L::kOffIdx);
  float *sW = reinterpret_cast<float *>(smem + L::kOffW);  // [2][H]
  const uint32_t bars = base + L::kOffBar;
  auto k_full = [&](int i) { return bars + 8u * i; };
  auto k_empty = [&](int i) { return bars + 8u * (NS + i); };
  auto q_full = [&](int i) { return bars + 8u * (2 * NS + i); };
  auto q_empty = [&](int i) { return bars + 8u * (2 * NS + NQ + i); };
  auto i_full = [&](int i) { return bars + 8u * (2 * NS + 2 * NQ + i); };
  auto i_empty = [&](int i) {
    return bars + 8u * (2 * NS + 2 * NQ + kIdxSlots + i);
  };
  auto acc_full = [&](int i) {
    return bars + 8u * (2 * NS + 2 * NQ + 2 * kIdxSlots + i);
  };
  auto acc_empty = [&](int i) {
    return bars + 8u * (2 * NS + 2 * NQ + 2 * kIdxSlots + kGatAcc + i);
  };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(k_full(i), 32 * kGatWarps);  // one per gather lane
      mbar_init(k_empty(i), 1);  // the epilogue, once the MMA is done
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), 1);
    }
    for (int i = 0; i < kIdxSlots; ++i) {
      mbar_init(i_full(i), 32);  // one cp.async arrival per fetch lane
      mbar_init(i_empty(i), 4);  // one arrival per epilogue warp
    }
    for (int i = 0; i < kGatAcc; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(acc_empty(i), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- index + query fetch ----------------
    GatCursor f = gat_begin(g);
    uint32_t nf = 0, nq = 0;
    bool ok = true, item_start = true;
    while (f.valid) {
      if (item_start) {
        // the row's query tile (H x D) into the next Q slot
        const int qs = nq % NQ;
        const uint32_t qph = (nq / NQ) & 1u;
        ++nq;
        ok = __all_sync(
            0xffffffffu,
            wait_bar_inl(q_empty(qs), qph ^ 1u, abort_flag, status));
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full(qs), L::kQBytes);
          for (int cc = 0; cc < KC; ++cc)
            tma_load_4d(sQ + qs * L::kQBytes + cc * (H * 128), &tm_q,
                        q_full(qs), cc * kChunk, 0, f.b, f.s);
        }
      }
      const int slot = nf % kIdxSlots;
      const uint32_t ph = (nf / kIdxSlots) & 1u;
      ok = __all_sync(0xffffffffu,
                      wait_bar_inl(i_empty(slot), ph ^ 1u, abort_flag, status));
      if (!ok) break;
      const int32_t *src =
          in_idx + (size_t)f.row * topk + (size_t)f.tile * kTileKeys;
      const int cnt = topk - f.tile * kTileKeys;
      const uint32_t dst = base + L::kOffIdx + slot * L::kIdxBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = lane + 32 * u;
        if (i < cnt) cp_async4(dst + 4 * i, src + i);
      }
      cp_async_arrive_noinc(i_full(slot));
      ++nf;
      item_start = gat_next(f, g);
    }
    // nothing may land in shared memory after the CTA is gone
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp <= kGatWarps) {
    // ---------------- key gathers ----------------
    constexpr int kSegs = KC * 8;           // 16-byte pieces of a stage row
    constexpr int kRowsPerOp = 32 / kSegs;  // rows one warp-wide copy covers
    constexpr int kRows = kTileKeys / kGatWarps;  // rows of a tile per warp
    static_assert(kRows % kRowsPerOp == 0, "whole copies per warp");
    const int gw = warp - 1;
    const int seg = lane % kSegs, sub = lane / kSegs;
    const int c = seg >> 3, s8 = seg & 7;
    // D is a multiple of 8, so every 16-byte piece is all key or all padding
    const uint32_t seg_bytes = seg * 16 < D * 2 ? 16u : 0u;
    const size_t seg_off = seg_bytes ? (size_t)seg * 16 : 0;
    const size_t key_stride = (size_t)B * D * 2;  // bytes from key j to j+1
    GatCursor cur = gat_begin(g);
    uint32_t ng = 0, kst = 0, kph = 0;
    while (cur.valid) {
      const int slot = ng % kIdxSlots;
      const uint32_t iph = (ng / kIdxSlots) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(i_full(slot), iph, abort_flag, status)))
        break;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(k_empty(kst), kph ^ 1u, abort_flag, status)))
        break;
      const uint32_t stage = sK + kst * L::kKBytes + c * (kTileKeys * 128);
      const uint8_t *kb = k + (size_t)cur.b * D * 2 + seg_off;
      const int r0 = gw * kRows + sub;
      const int live = topk - cur.tile * kTileKeys;  // slots of the tile
      constexpr int kOps = kRows / kRowsPerOp;
      int js[kOps];
#pragma unroll
      for (int u = 0; u < kOps; ++u) {
        const int rr = r0 + u * kRowsPerOp;
        const int j = rr < live ? sIdx[slot * kTileKeys + rr] : -1;
        js[u] = (j < 0 || j >= S_kv) ? -1 : j;
      }
#pragma unroll
      for (int u = 0; u < kOps; ++u) {
        const int rr = r0 + u * kRowsPerOp;
        // masked slots read nothing (zero fill); the epilogue discards them
        const bool valid = js[u] >= 0;
        cp_async16_zfill(stage + rr * 128 + ((s8 ^ (rr & 7)) << 4),
                         kb + (valid ? (size_t)js[u] * key_stride : 0),
                         valid ? seg_bytes : 0u);
      }
      // the stage fills up once every gather lane's copies have landed
      cp_async_arrive_noinc(k_full(kst));
      if (++kst == NS) {
        kst = 0;
        kph ^= 1u;
      }
      ++ng;
      gat_next(cur, g);
    }
    // nothing may land in shared memory after the CTA is gone
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      GatCursor cur = gat_begin(g);
      uint32_t kst = 0, kph = 0, nq = 0, acc = 0, aph = 0;
      bool item_start = true;
      int qs = 0;
      while (cur.valid) {
        if (item_start) {
          qs = nq % NQ;
          const uint32_t qph = (nq / NQ) & 1u;
          ++nq;
          if (!wait_bar_inl(q_full(qs), qph, abort_flag, status)) break;
        }
        if (!wait_bar_inl(acc_empty(acc), aph ^ 1u, abort_flag, status)) break;
        if (!wait_bar_inl(k_full(kst), kph, abort_flag, status)) break;
        // the stage was written by cp.async (generic proxy); order those
        // writes, observed through the barrier, before the tensor core's
        // operand reads (async proxy)
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * H;
        const uint32_t sQi = sQ + qs * L::kQBytes;
#pragma unroll
        for (int cc = 0; cc < KC; ++cc) {
#pragma unroll
          for (int kk = 0; kk < kChunk / 16; ++kk) {
            const uint64_t ad = sdesc_k_sw128(
                sK + kst * L::kKBytes + cc * (kTileKeys * 128) + kk * 32);
            const uint64_t bd = sdesc_k_sw128(sQi + cc * (H * 128) + kk * 32);
            mma_bf16(d_tmem, ad, bd, kIdesc, (cc | kk) != 0);
          }
        }
        // one commit per tile: the epilogue, once it sees the accumulator
        // full, also hands the stage back to the gather warps
        mma_commit(acc_full(acc));
        if (cur.tile + 1 == cur.tile_end) mma_commit(q_empty(qs));
        if (++kst == NS) {
          kst = 0;
          kph ^= 1u;
        }
        if (++acc == kGatAcc) {
          acc = 0;
          aph ^= 1u;
        }
        item_start = gat_next(cur, g);
      }
    }
  } else {
    // ---------------- epilogue (warps kEpiWarp0 .. kEpiWarp0 + 3) ----------
    const int sp = warp & 3;                    // TMEM sub-partition
    const int et = threadIdx.x - 32 * kEpiWarp0;  // 0..127
    const float neg_inf = -__int_as_float(0x7f800000);
    GatCursor cur = gat_begin(g);
    uint32_t acc = 0, aph = 0, nt = 0, ni = 0, est = 0;
    bool ok = true;
    // the first item's weight of head `et`, staged through a register so
    // the next item's load overlaps this item's tiles
    float w_next = 0.f;
    if (cur.valid && et < H)
      w_next = __ldg(w + ((size_t)cur.s * B + cur.b) * H + et);
    while (cur.valid) {
      float *sWi = sW + (ni & 1u) * H;
      if (et < H) sWi[et] = w_next;
      // every epilogue warp stored its weights, or one of them gave up
      if (named_bar_or(1, 128, !ok)) break;
      ++ni;
      const int row = cur.row;
      const int nv = n_visible(row_pos(q_pos, cur.b, cur.s), ratio, S_kv);
      bool bad = false, item_end = false;
      while (!item_end) {
        const int tile = cur.tile;
        const int slot = nt % kIdxSlots;
        const uint32_t iph = (nt / kIdxSlots) & 1u;
        ++nt;
        const bool got = wait_bar_inl(acc_full(acc), aph, abort_flag, status) &&
                         wait_bar_inl(i_full(slot), iph, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        // the tile's MMAs are complete, so its key stage is free again
        if (sp == 0 && lane == 0) mbar_arrive(k_empty(est));
        if (++est == NS) est = 0;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16) + acc * H;
        // weighted ReLU over the heads: weights four at a time, even heads
        // in .x and odd heads in .y of two packed accumulators
        const float4 *w4 = reinterpret_cast<const float4 *>(sWi);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        if constexpr (H >= 32) {
          uint32_t v[H / 32][32];
#pragma unroll
          for (int cc = 0; cc < H / 32; ++cc)
            tmem_ld32(taddr + cc * 32, v[cc]);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < H / 32; ++cc) reg_fence32(v[cc]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(acc));
#pragma unroll
          for (int h = 0; h < H; h += 4) {
            const float4 wv = w4[h >> 2];
            const float2 r01 =
                relu2x2(__uint_as_float(v[h >> 5][h & 31]),
                        __uint_as_float(v[(h + 1) >> 5][(h + 1) & 31]));
            const float2 r23 =
                relu2x2(__uint_as_float(v[(h + 2) >> 5][(h + 2) & 31]),
                        __uint_as_float(v[(h + 3) >> 5][(h + 3) & 31]));
            a0 = __ffma2_rn(make_float2(wv.x, wv.y), r01, a0);
            a1 = __ffma2_rn(make_float2(wv.z, wv.w), r23, a1);
          }
        } else {
          uint32_t v[16];
          tmem_ld16(taddr, v);
          tmem_ld_wait();
          reg_fence16(v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty(acc));
#pragma unroll
          for (int h = 0; h < 16; h += 4) {
            const float4 wv = w4[h >> 2];
            const float2 r01 = relu2x2(__uint_as_float(v[h]),
                                       __uint_as_float(v[h + 1]));
            const float2 r23 = relu2x2(__uint_as_float(v[h + 2]),
                                       __uint_as_float(v[h + 3]));
            a0 = __ffma2_rn(make_float2(wv.x, wv.y), r01, a0);
            a1 = __ffma2_rn(make_float2(wv.z, wv.w), r23, a1);
          }
        }
        const float s0 = a0.x + a0.y, s1 = a1.x + a1.y;
        if (++acc == kGatAcc) {
          acc = 0;
          aph ^= 1u;
        }
        const int i = sp * 32 + lane;
        const int e = tile * kTileKeys + i;  // slot within the row
        const bool in_row = e < topk;
        const int j = in_row ? sIdx[slot * kTileKeys + i] : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(i_empty(slot));
        if (in_row) {
          const size_t o = (size_t)row * topk + e;
          out_idx[o] = j;
          // the sums are of w * 2 ReLU (x + |x|): halving them is exact
          out_scores[o] = (j >= 0 && j < nv) ? 0.5f * (s0 + s1) : neg_inf;
          bad |= j < -1 || j >= S_kv;
        }
        item_end = gat_next(cur, g);
        // prefetch the next item's weight while its first tile is in flight
        if (item_end && cur.valid && et < H)
          w_next = __ldg(w + ((size_t)cur.s * B + cur.b) * H + et);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(status, kStatusIndexRange);
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int H, int KC>
cudaError_t launch_gat(const Problem &p, const CUtensorMap &tm_q,
                       const int32_t *in_idx,
                       int topk, int32_t *out_idx, float *out_scores,
                       int *status, int num_sms, cudaStream_t st) {
  auto kern = gather_scores_kernel<H, KC>;
  constexpr int kThreads = GatRoles<H>::kThreads;
  const int smem = GatSmem<H, KC>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  GatGeom g;
  g.rows = p.B * p.S;
  g.S = p.S;
  g.ntiles = (topk + kTileKeys - 1) / kTileKeys;
  // whole rows per item when there are enough of them to keep every SM
  // busy; otherwise rows split into chunks of tiles (the row's query tile
  // is loaded once per item)
  const long long target = 4ll * num_sms;
  int want = 1;
  if (g.rows < target) {
    const long long c = (target + g.rows - 1) / g.rows;
    want = (int)(c < g.ntiles ? c : g.ntiles);
  }
  g.tpi = (g.ntiles + want - 1) / want;
  g.nchunks = (g.ntiles + g.tpi - 1) / g.tpi;
  const long long n_items = (long long)g.rows * g.nchunks;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  g.n_items = (int)n_items;
  const int grid = (int)(n_items < num_sms ? n_items : num_sms);
  kern<<<grid, kThreads, smem, st>>>(
      tm_q, static_cast<const uint8_t *>(p.k), p.w, p.q_pos, in_idx, g, p.B,
      p.D, p.S_kv, p.ratio, topk, out_idx, out_scores, status);
  return cudaGetLastError();
}

}  // namespace

bool gather_supported(int H, int D) {
  return (H == 16 || H == 32 || H == 64 || H == 128) && D <= 2 * kChunk;
}

size_t gather_smem_bytes(int H, int D) {
  const bool k1 = D <= kChunk;
  switch (H) {
    case 16: return k1 ? GatSmem<16, 1>::kAlloc : GatSmem<16, 2>::kAlloc;
    case 32: return k1 ? GatSmem<32, 1>::kAlloc : GatSmem<32, 2>::kAlloc;
    case 64: return k1 ? GatSmem<64, 1>::kAlloc : GatSmem<64, 2>::kAlloc;
    case 128: return k1 ? GatSmem<128, 1>::kAlloc : GatSmem<128, 2>::kAlloc;
    default: return 0;
  }
}

cudaError_t launch_gather_scores(const Problem &p, const CUtensorMap &tm_q,
                                 const int32_t *in_idx, int topk,
                                 int32_t *out_idx, float *out_scores,
                                 int *status, int num_sms, cudaStream_t st) {
  const bool k1 = p.D <= kChunk;
#define DSA_GAT_CASE(HH)                                                     \
  case HH:                                                                   \
    return k1 ? launch_gat<HH, 1>(p, tm_q, in_idx, topk, out_idx,  \
                                  out_scores, status, num_sms, st)           \
              : launch_gat<HH, 2>(p, tm_q, in_idx, topk, out_idx,  \
                                  out_scores, status, num_sms, st);
  switch (p.H) {
    DSA_GAT_CASE(16)
    DSA_GAT_CASE(32)
    DSA_GAT_CASE(64)
    DSA_GAT_CASE(128)
    default:
      return cudaErrorNotSupported;
  }
#undef DSA_GAT_CASE
}

}  // namespace dsa
