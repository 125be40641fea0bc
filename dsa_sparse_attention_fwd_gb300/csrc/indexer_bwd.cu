// indexer_bwd: gradients of the lightning-indexer scores taken at given
// slots (the backward of V4IndexerFunction, "tilelang_indexer" page of NeMo
// AutoModel: backward(grad_scores, grad_indices); the indices carry no
// gradient).  For every slot (t, i) with a valid, visible key j = idx[t, i]
// and upstream gradient g = grad_scores[t, i], the score
//     I[t, j] = sum_h w[t, h] * ReLU(q[t, h, :] . k[j, :])
// gives
//     grad_w[t, h] += g * ReLU(s_h),                 s_h = q[t, h, :] . k[j, :]
//     grad_q[t, h] += g * w[t, h] * [s_h > 0] * k[j]
//     grad_k[j]    += g * w[t, h] * [s_h > 0] * q[t, h]
// with ReLU'(0) = 0.
//
// Factored form.  With G'[slot, h] = g * [s_h > 0] (no weight) and the
// row's A[h, :] = sum over slots of G'[slot, h] * k[j_slot]:
//     grad_q[t, h] = w[t, h] * A[h, :]
//     grad_w[t, h] = q[t, h, :] . A[h, :]        (= sum g * [s_h > 0] * s_h)
//     grad_k[j]   += sum_h G'[slot, h] * (w[t, h] q[t, h, :])
// so the per-slot work is a select, the weights enter once per row (a
// scaled copy Q' = w * Q of the row's query tile), and grad_w needs no
// per-slot accumulation.
//
// A work item is one query row (all of its slots), a tile 128 consecutive
// slots.  Per tile, on the tensor cores:
//   MMA1   S[slot, h]   = K_g . Q^T        M = 128 slots, N = H, K = D
//   (epilogue: G'[slot, h] = bf16(g) * [S > 0], into shared memory)
//   MMA2   A^T[d, h]   += K_g^T . G'       M = 128 (d), N = H, K = 128 slots
//   MMA3   dK[slot, d]  = G' . Q'          M = 128 slots, N = 128 (d), K = H
// K_g (the gathered keys) and G' are read twice, once K-major and once
// MN-major, from the same shared-memory tiles.  A^T accumulates in tensor
// memory over the row's tiles; dK rows are added into grad_k with vector
// atomics straight from tensor memory (a key is shared by many rows), each
// 4-thread group covering one 32-byte sector.  D <= 128 runs as D = 128
// with zero padding; H = 64 (one 128-byte G' row per slot).
//
// Warp roles (one CTA per SM, persistent, 16 warps): warp 0 index/gradient
// and query fetch, warp 1 TMEM allocator and MMA issuer, warps 4..7
// epilogue, eight warps of key gathers (16-byte cp.async, zero fill for
// masked slots), two idle.
// The MMA thread issues MMA1 of tile n + 1 before MMA2/MMA3 of tile n, so
// the tensor core works on the next scores while the epilogue forms G'.
//
// grad_q and grad_w are plain stores in a fixed order (deterministic);
// grad_k accumulates with atomics, so its rounding depends on their order.
#include "common.cuh"
#include "dsa_indexer.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kBwdH = 64;
// Warp roles.  Warps w and w + 4k share a sub-partition (scheduler); the
// MMA warp's sub-partition holds only it and one epilogue warp, so the
// issue of the tensor-core instructions does not queue behind gather
// copies.  Warps 9 and 13 (that sub-partition's other two) stay idle.
constexpr int kBwdGatWarps = 8;
constexpr int kBwdThreads = 512;
constexpr int kBwdMmaWarp = 1;
constexpr int kBwdEpiWarp0 = 4;  // warps 4..7, one per sub-partition
__device__ __forceinline__ int gather_index(int warp) {
  switch (warp) {
    case 2: return 0;
    case 3: return 1;
    case 8: return 2;
    case 10: return 3;
    case 11: return 4;
    case 12: return 5;
    case 14: return 6;
    case 15: return 7;
    default: return -1;
  }
}
constexpr int kBwdStages = 4;                   // gathered key stages
constexpr int kBwdRing = 8;                     // index/gradient ring (tiles)

struct BwdSmem {
  static constexpr int kQBytes = 2 * kBwdH * 128;      // two d-chunks of 64
  static constexpr int kKBytes = 2 * kTileKeys * 128;  // two d-chunks of 64
  static constexpr int kGBytes = kTileKeys * 128;      // 128 slots x 64 heads
  static constexpr int kRingBytes = kTileKeys * 8;     // indices, gradients
  static constexpr int kOffQ = 0;                      // [2] query slots
  static constexpr int kOffQw = kOffQ + 2 * kQBytes;   // w-scaled query
  static constexpr int kOffK = kOffQw + kQBytes;
  static constexpr int kOffG = kOffK + kBwdStages * kKBytes;
  static constexpr int kOffRing = kOffG + 2 * kGBytes;
  static constexpr int kOffW = kOffRing + kBwdRing * kRingBytes;  // [2][H]
  static constexpr int kOffGW = kOffW + 2 * kBwdH * 4;            // [4][H]
  static constexpr int kOffBar = kOffGW + 4 * kBwdH * 4;
  // k_full[4] k_empty[4] q_full[2] q_empty[2] r_full[8] r_empty[8]
  // s_full[2] g_full[2] dk_full[2] dq_full[2] dq_empty[2] qw_full qw_empty
  static constexpr int kNumBars = 2 * kBwdStages + 4 + 2 * kBwdRing + 10 + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(BwdSmem::kAlloc <= 227 * 1024, "fits one CTA per SM");

// TMEM columns: S x2 (64 each), A^T x2 (64 each), dK x2 (128 each).
constexpr uint32_t kTmemS = 0, kTmemDq = 128, kTmemDk = 256;
constexpr uint32_t kBwdTmemCols = 512;

struct BwdGeom {
  int rows, S, ntiles;
};

// Walks this CTA's tiles: rows round by round (zig-zag over the CTAs), each
// row's tiles in order.  Every role walks the same sequence.
struct BwdCursor {
  int round, row, b, s, tile;
  bool valid;
};

__device__ __forceinline__ void bwd_set_row(BwdCursor &c, const BwdGeom &g) {
  const int G = gridDim.x, cta = blockIdx.x;
  const long long r =
      (long long)c.round * G + ((c.round & 1) ? (G - 1 - cta) : cta);
  c.valid = r < g.rows;
  if (!c.valid) return;
  c.row = (int)r;
  c.b = c.row / g.S;
  c.s = c.row % g.S;
  c.tile = 0;
}

__device__ __forceinline__ BwdCursor bwd_begin(const BwdGeom &g) {
  BwdCursor c;
  c.round = 0;
  bwd_set_row(c, g);
  return c;
}

// Advances by one tile; returns true when a new row starts.
__device__ __forceinline__ bool bwd_next(BwdCursor &c, const BwdGeom &g) {
  if (++c.tile < g.ntiles) return false;
  ++c.round;
  bwd_set_row(c, g);
  return true;
}

// The MMA2/MMA3 half of a tile, issued after the next tile's MMA1.
struct BwdPending {
  uint32_t n;     // the tile's sequence number in this CTA
  int kst, qs;    // its key stage and query slot
  int dq;         // A^T accumulator of its row (row parity)
  uint32_t dqph;  // phase of that accumulator's barriers
  bool first, last;
};

__global__ void __launch_bounds__(kBwdThreads, 1)
    indexer_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const uint8_t *__restrict__ k,
                       const float *__restrict__ w,
                       const int32_t *__restrict__ q_pos,
                       const int32_t *__restrict__ idx,
                       const float *__restrict__ grad_scores, BwdGeom g,
                       int B, int D, int S_kv, int ratio, int topk,
                       float *__restrict__ grad_q, float *__restrict__ grad_k,
                       float *__restrict__ grad_w, int *status) {
  using L = BwdSmem;
  constexpr int H = kBwdH;
  constexpr int NS = kBwdStages;
  // MMA1: both K-major.  MMA2: A = gathered keys read d-major, B = G' read
  // head-major.  MMA3: A = G' K-major (heads), B = Q' read d-major.
  constexpr uint32_t kIdescS = idesc_bf16_f32(kTileKeys, H);
  constexpr uint32_t kIdescDq = idesc_bf16_f32_mn(128, H, true, true);
  constexpr uint32_t kIdescDk = idesc_bf16_f32_mn(kTileKeys, 128, false, true);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sQw = base + L::kOffQw;
  const uint32_t sK = base + L::kOffK;
  const uint32_t sG = base + L::kOffG;
  const uint8_t *sRing = smem + L::kOffRing;
  float *sW = reinterpret_cast<float *>(smem + L::kOffW);
  float *sGW = reinterpret_cast<float *>(smem + L::kOffGW);
  const uint32_t bars = base + L::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  auto k_full = [&](int i) { return bar(i); };
  auto k_empty = [&](int i) { return bar(NS + i); };
  auto q_full = [&](int i) { return bar(2 * NS + i); };
  auto q_empty = [&](int i) { return bar(2 * NS + 2 + i); };
  auto r_full = [&](int i) { return bar(2 * NS + 4 + i); };
  auto r_empty = [&](int i) { return bar(2 * NS + 4 + kBwdRing + i); };
  constexpr int kB2 = 2 * NS + 4 + 2 * kBwdRing;
  // The S, G' and dK buffers need no "empty" barriers: the epilogue reads
  // S(n) and drains dK(n - 2) before it signals G'(n), and drains dK(n)
  // (waiting for MMA2/MMA3 of tile n) before it writes G'(n + 2).
  auto s_full = [&](int i) { return bar(kB2 + i); };
  auto g_full = [&](int i) { return bar(kB2 + 2 + i); };
  auto dk_full = [&](int i) { return bar(kB2 + 4 + i); };
  auto dq_full = [&](int i) { return bar(kB2 + 6 + i); };
  auto dq_empty = [&](int i) { return bar(kB2 + 8 + i); };
  const uint32_t qw_full = bar(kB2 + 10), qw_empty = bar(kB2 + 11);
  static_assert(kB2 + 11 < L::kNumBars, "every barrier has its slot");
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Q chunks the fetch warp loads; with D <= 64 the second chunk of both Q
  // slots stays zero (written once here), so the padded d never contributes
  const int q_chunks = D > kChunk ? 2 : 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(k_full(i), 32 * kBwdGatWarps);  // one per gather lane
      mbar_init(k_empty(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(q_full(i), 1);
      // the row's last MMAs, then each epilogue warp once it is done with Q
      mbar_init(q_empty(i), 1 + 4);
      mbar_init(s_full(i), 1);
      mbar_init(g_full(i), 4);  // epilogue warps
      mbar_init(dk_full(i), 1);
      mbar_init(dq_full(i), 1);
      mbar_init(dq_empty(i), 4);
    }
    mbar_init(qw_full, 4);
    mbar_init(qw_empty, 1);
    for (int i = 0; i < kBwdRing; ++i) {
      mbar_init(r_full(i), 32);  // one cp.async arrival per fetch lane
      mbar_init(r_empty(i), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
  }
  if (q_chunks == 1) {
    for (int o = threadIdx.x * 16; o < 2 * H * 128; o += kBwdThreads * 16) {
      const int slot = o / (H * 128), off = o % (H * 128);
      *reinterpret_cast<uint4 *>(smem + L::kOffQ + slot * L::kQBytes +
                                 H * 128 + off) = make_uint4(0, 0, 0, 0);
    }
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- index, gradient and query fetch ----------------
    BwdCursor f = bwd_begin(g);
    uint32_t nr = 0, nq = 0;
    bool row_start = true;
    while (f.valid) {
      if (row_start) {
        const int qs = nq & 1;
        const uint32_t qph = (nq >> 1) & 1u;
        ++nq;
        if (!__all_sync(
                0xffffffffu,
                wait_bar_inl(q_empty(qs), qph ^ 1u, abort_flag, status)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full(qs), q_chunks * H * 128);
          for (int cc = 0; cc < q_chunks; ++cc)
            tma_load_4d(sQ + qs * L::kQBytes + cc * (H * 128), &tm_q,
                        q_full(qs), cc * kChunk, 0, f.b, f.s);
        }
      }
      const int slot = nr % kBwdRing;
      const uint32_t ph = (nr / kBwdRing) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(r_empty(slot), ph ^ 1u, abort_flag, status)))
        break;
      const size_t off = (size_t)f.row * topk + (size_t)f.tile * kTileKeys;
      const int cnt = topk - f.tile * kTileKeys;
      const uint32_t dst = base + L::kOffRing + slot * L::kRingBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = lane + 32 * u;
        if (i < cnt) {
          cp_async4(dst + 4 * i, idx + off + i);
          cp_async4(dst + 4 * (kTileKeys + i), grad_scores + off + i);
        }
      }
      cp_async_arrive_noinc(r_full(slot));
      ++nr;
      row_start = bwd_next(f, g);
    }
    // nothing may land in shared memory after the CTA is gone
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (gather_index(warp) >= 0) {
    // ---------------- key gathers ----------------
    constexpr int kSegs = 16;               // 16-byte pieces of a stage row
    constexpr int kRowsPerOp = 32 / kSegs;  // rows one warp-wide copy covers
    constexpr int kRows = kTileKeys / kBwdGatWarps;
    constexpr int kOps = kRows / kRowsPerOp;
    const int gw = gather_index(warp);
    const int seg = lane % kSegs, sub = lane / kSegs;
    const int c = seg >> 3, s8 = seg & 7;
    // D is a multiple of 8, so every 16-byte piece is all key or all padding
    const uint32_t seg_bytes = seg * 16 < D * 2 ? 16u : 0u;
    const size_t seg_off = seg_bytes ? (size_t)seg * 16 : 0;
    const size_t key_stride = (size_t)B * D * 2;
    BwdCursor cur = bwd_begin(g);
    uint32_t ng = 0, kst = 0, kph = 0;
    while (cur.valid) {
      const int slot = ng % kBwdRing;
      const uint32_t rph = (ng / kBwdRing) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(r_full(slot), rph, abort_flag, status)))
        break;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(k_empty(kst), kph ^ 1u, abort_flag, status)))
        break;
      const int32_t *sIdx =
          reinterpret_cast<const int32_t *>(sRing + slot * L::kRingBytes);
      const uint32_t stage = sK + kst * L::kKBytes + c * (kTileKeys * 128);
      const uint8_t *kb = k + (size_t)cur.b * D * 2 + seg_off;
      const int r0 = gw * kRows + sub;
      const int live = topk - cur.tile * kTileKeys;
      int js[kOps];
#pragma unroll
      for (int u = 0; u < kOps; ++u) {
        const int rr = r0 + u * kRowsPerOp;
        const int j = rr < live ? sIdx[rr] : -1;
        js[u] = (j < 0 || j >= S_kv) ? -1 : j;
      }
#pragma unroll
      for (int u = 0; u < kOps; ++u) {
        const int rr = r0 + u * kRowsPerOp;
        const bool valid = js[u] >= 0;
        cp_async16_zfill(stage + rr * 128 + ((s8 ^ (rr & 7)) << 4),
                         kb + (valid ? (size_t)js[u] * key_stride : 0),
                         valid ? seg_bytes : 0u);
      }
      cp_async_arrive_noinc(k_full(kst));
      if (++kst == NS) {
        kst = 0;
        kph ^= 1u;
      }
      ++ng;
      bwd_next(cur, g);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kBwdMmaWarp) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs the control flow (converged, waits taken
    // together); lane 0 alone issues the tcgen05 instructions, through a
    // predicate rather than a branch.
    const uint32_t lead = lane == 0;
    auto wait_all = [&](uint32_t b, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bar_inl(b, ph, abort_flag, status));
    };
    // MMA2 and MMA3 of a finished tile: A^T += K_g^T G', dK = G' Q'
    auto issue_back = [&](const BwdPending &p) -> bool {
      const int gb = p.n & 1;
      const uint32_t gph = (p.n >> 1) & 1u;
      // G'(n) is written.  The epilogue forms G'(n) only after it has read
      // S(n) and drained dK(n - 2), so this one wait also frees the dK
      // accumulator MMA3 overwrites and the S buffer of tile n (reused by
      // tile n + 2's MMA1, issued after this).
      if (!wait_all(g_full(gb), gph)) return false;
      // a row's first tile: its A^T accumulator is free and its Q' written
      if (p.first && (!wait_all(dq_empty(p.dq), p.dqph ^ 1u) ||
                      !wait_all(qw_full, (uint32_t)p.dq)))
        return false;
      tc_fence_after();
      // rolled loops, the start address advanced inside the descriptor
      // (its low field counts 16-byte units): the issue loop stays small
      const uint32_t sGb = sG + gb * L::kGBytes;
      // K = 128 slots in steps of 16 (two 8-slot atoms, 2048 bytes)
      // N = 64 is one atom, so G's atom stride along N is never used
      const uint64_t a2 =
          sdesc_mn_sw128(sK + p.kst * L::kKBytes, kTileKeys * 128, 1024);
      const uint64_t b2 = sdesc_mn_sw128(sGb, 1024, 1024);
      const uint32_t d2 = tmem + kTmemDq + p.dq * H;
#pragma unroll 1
      for (int ks = 0; ks < kTileKeys / 16; ++ks)
        mma_bf16_by(d2, a2 + ks * (2048 >> 4), b2 + ks * (2048 >> 4),
                    kIdescDq, (p.first && ks == 0) ? 0u : 1u, lead);
      // K = 64 heads in steps of 16
      const uint64_t a3 = sdesc_k_sw128(sGb);
      const uint64_t b3 = sdesc_mn_sw128(sQw, H * 128, 1024);
      const uint32_t d3 = tmem + kTmemDk + gb * 128;
#pragma unroll 1
      for (int kk = 0; kk < H / 16; ++kk)
        mma_bf16_by(d3, a3 + kk * (32 >> 4), b3 + kk * (2048 >> 4), kIdescDk,
                    kk != 0 ? 1u : 0u, lead);
      // dk_full also tells the epilogue that G' buffer gb is free again
      mma_commit_by(k_empty(p.kst), lead);
      mma_commit_by(dk_full(gb), lead);
      if (p.last) {
        mma_commit_by(dq_full(p.dq), lead);
        mma_commit_by(q_empty(p.qs), lead);
        mma_commit_by(qw_empty, lead);
      }
      return true;
    };

    BwdCursor cur = bwd_begin(g);
    uint32_t kst = 0, kph = 0, nq = 0, n = 0, nrow = 0;
    bool row_start = true, ok = true, pend = false;
    BwdPending pd{};
    int qs = 0;
    while (cur.valid) {
      if (row_start) {
        qs = nq & 1;
        const uint32_t qph = (nq >> 1) & 1u;
        ++nq;
        if (!wait_all(q_full(qs), qph)) {
          ok = false;
          break;
        }
      }
      const int sa = n & 1;
      // S buffer sa was read by the epilogue before it signalled G'(n - 2),
      // which the previous iteration waited for
      if (!wait_all(k_full(kst), kph)) {
        ok = false;
        break;
      }
      // the stage was written by cp.async (generic proxy)
      fence_proxy_async_smem();
      tc_fence_after();
      const uint64_t a1 = sdesc_k_sw128(sK + kst * L::kKBytes);
      const uint64_t b1 = sdesc_k_sw128(sQ + qs * L::kQBytes);
      const uint32_t d1 = tmem + kTmemS + sa * H;
      // two d-chunks of four K = 16 steps (32 bytes each)
#pragma unroll 1
      for (int t = 0; t < 8; ++t) {
        const uint32_t ao = ((t >> 2) * (kTileKeys * 128) + (t & 3) * 32) >> 4;
        const uint32_t bo = ((t >> 2) * (H * 128) + (t & 3) * 32) >> 4;
        mma_bf16_by(d1, a1 + ao, b1 + bo, kIdescS, t != 0 ? 1u : 0u, lead);
      }
      mma_commit_by(s_full(sa), lead);
      if (pend && !issue_back(pd)) {
        ok = false;
        break;
      }
      pd.n = n;
      pd.kst = kst;
      pd.qs = qs;
      pd.dq = nrow & 1;
      pd.dqph = (nrow >> 1) & 1u;
      pd.first = cur.tile == 0;
      pd.last = cur.tile + 1 == g.ntiles;
      pend = true;
      if (pd.last) ++nrow;
      ++n;
      if (++kst == NS) {
        kst = 0;
        kph ^= 1u;
      }
      row_start = bwd_next(cur, g);
    }
    if (ok && pend) issue_back(pd);
  } else if (warp >= kBwdEpiWarp0 && warp < kBwdEpiWarp0 + 4) {
    // ---------------- epilogue (warps kBwdEpiWarp0 .. kBwdEpiWarp0 + 3) ------
    const int sp = warp & 3;                         // TMEM sub-partition
    const int et = threadIdx.x - 32 * kBwdEpiWarp0;  // 0..127
    const int i = sp * 32 + lane;  // TMEM lane: the slot, or d for A^T
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    BwdCursor cur = bwd_begin(g);
    uint32_t n = 0, nrow = 0;
    bool ok = true;
    float w_next = 0.f;
    if (cur.valid && et < H)
      w_next = __ldg(w + ((size_t)cur.s * B + cur.b) * H + et);
    // the previous tile's dK rows, added into grad_k after this tile's G'
    bool dk_pend = false, dk_live = false;
    uint32_t dk_n = 0;
    int dk_off = 0;  // element offset of this lane's dK row in grad_k
    auto drain_dk = [&]() -> bool {
      const int db = dk_n & 1;
      const uint32_t dph = (dk_n >> 1) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(dk_full(db), dph, abort_flag, status)))
        return false;
      tc_fence_after();
      const uint32_t live = __ballot_sync(0xffffffffu, dk_live);
      if (live) {
        // 16 rows per load; 4 consecutive lanes hold 8 consecutive d of a
        // row, so every red covers whole 32-byte sectors
        const int t4 = lane >> 2, c2 = (lane & 3) * 2;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const int ra = hf * 16 + t4, rb = ra + 8;
          const int offa = __shfl_sync(0xffffffffu, dk_off, ra);
          const int offb = __shfl_sync(0xffffffffu, dk_off, rb);
          const bool la = (live >> ra) & 1u, lb = (live >> rb) & 1u;
          const uint32_t ta = tmem + ((uint32_t)(sp * 32 + hf * 16) << 16) +
                              kTmemDk + db * 128;
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t v[16];
            __syncwarp();
            tmem_ld16x256b_x4(ta + c4 * 32, v);
            tmem_ld_wait();
            reg_fence16(v);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
              const int d = c4 * 32 + kb * 8 + c2;
              if (d < D) {
                if (la)
                  red_add_v2(grad_k + offa + d, __uint_as_float(v[4 * kb]),
                             __uint_as_float(v[4 * kb + 1]));
                if (lb)
                  red_add_v2(grad_k + offb + d,
                             __uint_as_float(v[4 * kb + 2]),
                             __uint_as_float(v[4 * kb + 3]));
              }
            }
          }
        }
      }
      // the MMA thread learns that dK buffer db is free from the next G'
      // signal (g_full), which this warp gives only after this drain
      tc_fence_before();
      return true;
    };

    while (cur.valid) {
      float *sWi = sW + (nrow & 1u) * H;
      if (et < H) sWi[et] = w_next;
      // every epilogue warp stored its weights, or one of them gave up
      if (named_bar_or(1, 128, !ok)) break;
      const int b = cur.b, s = cur.s;
      const int nv = n_visible(row_pos(q_pos, b, s), ratio, S_kv);
      // the fetch warp loads one query tile per row, in this order
      const int qs = nrow & 1;
      const uint32_t qph = (nrow >> 1) & 1u;
      const uint32_t sQs = sQ + qs * L::kQBytes;
      // Q' = w * Q for this row's MMA3s, once the previous row's are done
      ok = __all_sync(0xffffffffu,
                      wait_bar_inl(q_full(qs), qph, abort_flag, status) &&
                          wait_bar_inl(qw_empty, (nrow & 1u) ^ 1u, abort_flag,
                                   status));
      if (ok) {
#pragma unroll 2
        for (int u8 = 0; u8 < 8; ++u8) {
          const uint32_t o = (uint32_t)(u8 * 128 + et) * 16u;
          const float wh = sWi[(o & (H * 128 - 1)) >> 7];  // the unit's head
          const float4 x = ld_shared_v4f(sQs + o);
          const uint32_t xs[4] = {__float_as_uint(x.x), __float_as_uint(x.y),
                                  __float_as_uint(x.z), __float_as_uint(x.w)};
          uint32_t y[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            y[e] = pack_bf16x2(__uint_as_float(xs[e] << 16) * wh,
                               __uint_as_float(xs[e] & 0xFFFF0000u) * wh);
          st_shared_v4(sQw + o, y);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(qw_full);
      }
      bool bad = false, row_end = false;
      while (ok && !row_end) {
        const int slot = n % kBwdRing;
        const uint32_t rph = (n / kBwdRing) & 1u;
        const int sa = n & 1;
        const uint32_t sph = (n >> 1) & 1u;
        const bool got = wait_bar_inl(s_full(sa), sph, abort_flag, status) &&
                         wait_bar_inl(r_full(slot), rph, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int e = cur.tile * kTileKeys + i;  // slot within the row
        const bool in_row = e < topk;
        const uint8_t *rs = sRing + slot * L::kRingBytes;
        const int j = in_row ? reinterpret_cast<const int32_t *>(rs)[i] : -1;
        const float gs =
            in_row ? reinterpret_cast<const float *>(rs + kTileKeys * 4)[i]
                   : 0.f;
        __syncwarp();
        if (lane == 0) mbar_arrive(r_empty(slot));
        bad |= in_row && (j < -1 || j >= S_kv);
        const bool valid = j >= 0 && j < nv;
        const float ge = valid ? gs : 0.f;
        // this G' buffer was last read by MMA2/MMA3 of tile n - 2, whose
        // completion the drain of dK(n - 2) has already waited for
        // G'[slot, h] = bf16(g) where S > 0, else 0: a mask on the packed
        // pair (bf16 row of 128 bytes, 16-byte units rotated by the row)
        const uint32_t gg = pack_bf16x2(ge, ge);
        const uint32_t grow = sG + sa * L::kGBytes + i * 128;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(tmem + lane_off + kTmemS + sa * H + half * 32, v);
          tmem_ld_wait();
          reg_fence32(v);
          if (half == 1) tc_fence_before();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t pk[4];
#pragma unroll
            for (int p2 = 0; p2 < 4; ++p2) {
              const int h = u * 8 + p2 * 2;
              const uint32_t m =
                  (__uint_as_float(v[h]) > 0.f ? 0x0000FFFFu : 0u) |
                  (__uint_as_float(v[h + 1]) > 0.f ? 0xFFFF0000u : 0u);
              pk[p2] = gg & m;
            }
            const int uu = half * 4 + u;
            st_shared_v4(grow + ((uu ^ (i & 7)) << 4), pk);
          }
        }
        // the tensor core (async proxy) reads G' next
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(g_full(sa));
        if (dk_pend && !drain_dk()) {
          ok = false;
          break;
        }
        dk_pend = true;
        dk_n = n;
        dk_live = valid && ge != 0.f;
        dk_off = dk_live ? (j * B + b) * D : 0;
        ++n;
        row_end = bwd_next(cur, g);
      }
      // every warp finished the row's tiles, or one of them gave up
      if (named_bar_or(2, 128, !ok)) break;
      // the row's last dK rows, then grad_q = w * A and grad_w = q . A
      dk_pend = false;
      ok = drain_dk();
      const int dq = nrow & 1;
      const uint32_t dqph = (nrow >> 1) & 1u;
      if (ok)
        ok = __all_sync(0xffffffffu,
                        wait_bar_inl(dq_full(dq), dqph, abort_flag, status));
      // this warp's share of grad_w: zero unless the row completes
      sGW[sp * H + lane] = 0.f;
      sGW[sp * H + 32 + lane] = 0.f;
      if (ok) {
        tc_fence_after();
        float *gq = grad_q + ((size_t)s * B + b) * H * D;
        // q[h, d] of this lane's d in the row's (swizzled) query tile
        const int dd = i & (kChunk - 1);
        const uint32_t qcol = sQs + (i >> 6) * (H * 128) + (dd & 7) * 2;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld32(tmem + lane_off + kTmemDq + dq * H + c * 32, v);
          tmem_ld_wait();
          reg_fence32(v);
          float gp[32];
#pragma unroll
          for (int hh = 0; hh < 32; ++hh) {
            const int h = c * 32 + hh;
            const float a = __uint_as_float(v[hh]);
            const uint32_t qa =
                qcol + h * 128 + ((((dd >> 3) ^ (h & 7))) << 4);
            gp[hh] = a * __uint_as_float((uint32_t)ld_shared_u16(qa) << 16);
            // lane = d: each store instruction writes 32 consecutive d
            if (i < D) gq[(size_t)h * D + i] = sWi[h] * a;
          }
          // sum over the lanes' d: halve the 32 sums five times (each lane
          // keeps the half its lane bit selects), leaving head c*32 + lane
#pragma unroll
          for (int o = 16, m = 32; o >= 1; o >>= 1, m >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int h = 0; h < m / 2; ++h) {
              const float send = up ? gp[h] : gp[h + m / 2];
              const float keep = up ? gp[h + m / 2] : gp[h];
              gp[h] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          sGW[sp * H + c * 32 + lane] = gp[0];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(dq_empty(dq));
          mbar_arrive(q_empty(qs));
        }
      }
      named_bar_sync(3, 128);
      if (ok && et < H)
        grad_w[((size_t)s * B + b) * H + et] =
            ((sGW[et] + sGW[H + et]) + sGW[2 * H + et]) + sGW[3 * H + et];
      if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(status, kStatusIndexRange);
      ++nrow;
      // the next row's weight (cur already points at it)
      if (cur.valid && et < H)
        w_next = __ldg(w + ((size_t)cur.s * B + cur.b) * H + et);
    }
  }

  __syncthreads();
  if (warp == kBwdMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

}  // namespace

cudaError_t launch_indexer_bwd(const Problem &p, const CUtensorMap &tm_q,
                               const int32_t *idx, const float *grad_scores,
                               int topk, float *grad_q, float *grad_k,
                               float *grad_w, int *status, int num_sms,
                               cudaStream_t st) {
  if (p.H != kBwdH || p.D > 2 * kChunk) return cudaErrorNotSupported;
  const int smem = BwdSmem::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(
      indexer_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  BwdGeom g;
  g.rows = p.B * p.S;
  g.S = p.S;
  g.ntiles = (topk + kTileKeys - 1) / kTileKeys;
  if (g.rows <= 0) return cudaSuccess;
  const int grid = g.rows < num_sms ? g.rows : num_sms;
  indexer_bwd_kernel<<<grid, kBwdThreads, smem, st>>>(
      tm_q, static_cast<const uint8_t *>(p.k), p.w, p.q_pos, idx, grad_scores,
      g, p.B, p.D, p.S_kv, p.ratio, topk, grad_q, grad_k, grad_w, status);
  return cudaGetLastError();
}

}  // namespace dsa

extern "C" {

size_t dsa_indexer_bwd_workspace_size(void) { return 256; }

int dsa_indexer_bwd(const void *q, const void *k, const float *w, int S,
                    int B, int H, int D, int S_kv, int compress_ratio,
                    int topk, const int32_t *q_pos, const int32_t *idx,
                    const float *grad_scores, float *grad_q, float *grad_k,
                    float *grad_w, void *workspace, size_t workspace_bytes,
                    void *cuda_stream) {
  if (!q || !k || !w || !idx || !grad_scores || !grad_q || !grad_k ||
      !grad_w)
    return DSA_ERR_INVALID_ARG;
  if (S <= 0 || B <= 0 || H <= 0 || D <= 0 || S_kv <= 0 ||
      compress_ratio <= 0 || topk <= 0)
    return DSA_ERR_INVALID_ARG;
  if (H != 64 || D % 8 != 0 || D > 128) return DSA_ERR_UNSUPPORTED;
  if ((long long)B * S >= (1ll << 31) || topk > (1 << 30) ||
      (long long)S_kv * B * D >= (1ll << 31))
    return DSA_ERR_UNSUPPORTED;
  auto al = [](const void *p, unsigned a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
  };
  if (!al(q, 16) || !al(k, 16) || !al(grad_k, 16) || !al(w, 4) ||
      !al(idx, 4) || !al(grad_scores, 4) || !al(grad_q, 4) ||
      !al(grad_w, 4) || (q_pos && !al(q_pos, 4)))
    return DSA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < dsa_indexer_bwd_workspace_size())
    return DSA_ERR_WORKSPACE;
  if (!al(workspace, 256)) return DSA_ERR_INVALID_ARG;
  int num_sms = 0;
  int rc = dsa::device_num_sms(&num_sms);
  if (rc != DSA_OK) return rc;
  dsa::Problem p{q, k, w, q_pos, S, B, H, D, S_kv, compress_ratio};
  CUtensorMap tm_q;
  rc = dsa::encode_q(&tm_q, p, 1);
  if (rc != DSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int *status = static_cast<int *>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess ||
      cudaMemsetAsync(grad_k, 0, (size_t)S_kv * B * D * sizeof(float), st) !=
          cudaSuccess)
    return DSA_ERR_CUDA;
  if (dsa::launch_indexer_bwd(p, tm_q, idx, grad_scores, topk, grad_q, grad_k,
                              grad_w, status, num_sms, st) != cudaSuccess)
    return DSA_ERR_CUDA;
  return DSA_OK;
}

}  // extern "C"
