// sparse_mla: attention over the tokens the indexer selected, in the MLA
// latent space with no rotary part (page "Module glm5next_dsa", "Shape of
// the pipeline": the selected tokens feed an MLA attention without the
// rotary part, over those tokens only; the latent width
// is kv_lora_rank, section "Constants").  The latent row of a selected
// token is both key and value:
//     x_i = scale * q[t, h, :] . c[j_i, :]       (j_i = idx[t, i], valid)
//     o[t, h, :] = sum_i softmax(x)_i * c[j_i, :],   lse[t, h] = ln sum e^x
//
// A work item is one query row and 64 of its heads; a tile is 128
// consecutive slots, its latent rows gathered into shared memory (cp.async,
// zero fill for -1 slots) one block of 128 latent dims at a time, each
// block with its own full/empty barriers: the next tile's block b is
// gathered as soon as the output product has read block b, and the score
// product consumes blocks as they land.  One pass over the row's tiles:
//   S^T[slot, h] = C_g . Q^T on the tensor cores (M = 128 slots, N = 64
//   heads, K = Dc); the epilogue takes each head's tile maximum, moves the
//   running maximum m when a tile exceeds it by more than 2^8 (rescaling
//   the accumulated O^T and l by the change), forms P^T = exp2(S *
//   scale*log2(e) - m) in bf16 (0 for invalid slots; at most 2^8) and each
//   head's sum l; O^T[d, h] += C_g^T . P^T (M = 128 latent dims per block,
//   N = 64, K = 128 slots; the gathered tile read d-major and P^T
//   head-major), accumulated in tensor memory over the row.
// The row ends with o = O^T / l and lse = (m + log2 l) * ln 2; a row
// without a valid slot gets o = 0 and lse = -inf.
//
// Warp roles (one CTA per SM, persistent): warp 0 fetch (index ring, query
// tile), warps 1..8 gathers, warp 9 TMEM allocator and MMA issuer, warps
// 10..17 epilogue (warp w reads TMEM lanes 32 (w % 4) .. + 31 and heads
// 32 ((w - 10) / 4) .. + 31).
#include <cuda_runtime.h>

#include "common.cuh"
#include "dsa_indexer.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kMlaH = 64;  // heads per item
constexpr int kMlaGatWarps = 8;
constexpr int kMlaEpiWarps = 8;  // two per TMEM lane quarter, 32 heads each
constexpr int kMlaThreads = 32 * (kMlaGatWarps + 2 + kMlaEpiWarps);
constexpr int kMlaMmaWarp = kMlaGatWarps + 1;
constexpr int kMlaEpiWarp0 = kMlaGatWarps + 2;
constexpr int kMlaRing = 8;  // index ring (tile visits)

// NB = Dc / 128 latent blocks.
template <int NB>
struct MlaSmem {
  static constexpr int kDc = NB * 128;
  static constexpr int kCh = kDc / 64;                   // 128-byte chunks
  static constexpr int kQBytes = kCh * kMlaH * 128;      // 64 heads x Dc
  static constexpr int kCBytes = kCh * kTileKeys * 128;  // 128 slots x Dc
  static constexpr int kPBytes = kTileKeys * 128;        // 128 slots x 64 h
  static constexpr int kRingBytes = kTileKeys * 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffC = kOffQ + kQBytes;
  static constexpr int kOffP = kOffC + kCBytes;
  static constexpr int kOffRing = kOffP + kPBytes;
  static constexpr int kOffRed = kOffRing + kMlaRing * kRingBytes;  // [4][64]
  static constexpr int kOffM = kOffRed + 4 * kMlaH * 4;             // [64]
  static constexpr int kOffL = kOffM + kMlaH * 4;                   // [64]
  static constexpr int kOffF = kOffL + kMlaH * 4;  // [64] factors + flag
  static constexpr int kOffBar = kOffF + (kMlaH + 4) * 4;
  // k_full[NB] k_empty[NB] q_full q_empty r_full[8] r_empty[8] s_full[2]
  // s_empty[2] p_full p_empty o_full o_empty
  static constexpr int kNumBars = 2 * NB + 2 + 2 * kMlaRing + 4 + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(MlaSmem<4>::kAlloc <= 227 * 1024, "fits one CTA per SM");

constexpr uint32_t kTmemSm = 0;   // S^T x2, 64 columns each
constexpr uint32_t kTmemO = 128;  // O^T: NB blocks of 64 columns

struct MlaGeom {
  int items, S, HG, ntiles;
};

// Walks this CTA's tiles: items round by round (zig-zag over the CTAs),
// each item's tiles in order.
struct MlaCursor {
  int round, row, b, s, hg, tile;
  bool valid;
};

__device__ __forceinline__ void mla_set_item(MlaCursor &c, const MlaGeom &g) {
  const int G = gridDim.x, cta = blockIdx.x;
  const long long it =
      (long long)c.round * G + ((c.round & 1) ? (G - 1 - cta) : cta);
  c.valid = it < g.items;
  if (!c.valid) return;
  c.row = (int)(it / g.HG);
  c.hg = (int)(it % g.HG);
  c.b = c.row / g.S;
  c.s = c.row % g.S;
  c.tile = 0;
}

__device__ __forceinline__ MlaCursor mla_begin(const MlaGeom &g) {
  MlaCursor c;
  c.round = 0;
  mla_set_item(c, g);
  return c;
}

// Advances one tile; returns 0 (same item) or 2 (a new item starts).
__device__ __forceinline__ int mla_next(MlaCursor &c, const MlaGeom &g) {
  if (++c.tile < g.ntiles) return 0;
  ++c.round;
  mla_set_item(c, g);
  return 2;
}

// Sum (MAX = false) or maximum (MAX = true) of N per-lane values over the
// warp's 32 lanes: halve the set five times, each lane keeping the half its
// lane bit selects; lane l ends with values N/32 l .. N/32 l + N/32 - 1 in
// v[0 .. N/32).
template <int N, bool MAX>
__device__ __forceinline__ void warp_fold(float (&v)[N], int lane) {
#pragma unroll
  for (int o = 16, m = N; o >= 1; o >>= 1, m >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int h = 0; h < m / 2; ++h) {
      const float send = up ? v[h] : v[h + m / 2];
      const float keep = up ? v[h + m / 2] : v[h];
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[h] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
}

template <int NB>
__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const uint8_t *__restrict__ cache,
                      const int32_t *__restrict__ idx, MlaGeom g, int B,
                      int H, int T, int topk, float scale_log2e,
                      float *__restrict__ out_o, float *__restrict__ out_lse,
                      int *status) {
  using L = MlaSmem<NB>;
  constexpr int Hg = kMlaH;
  constexpr int Dc = L::kDc, CH = L::kCh;
  constexpr uint32_t kIdescS = idesc_bf16_f32(kTileKeys, Hg);
  constexpr uint32_t kIdescO = idesc_bf16_f32_mn(128, Hg, true, true);
  const float neg_inf = -__int_as_float(0x7f800000);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sC = base + L::kOffC;
  const uint32_t sP = base + L::kOffP;
  const uint8_t *sRing = smem + L::kOffRing;
  float *sRed = reinterpret_cast<float *>(smem + L::kOffRed);
  float *sM = reinterpret_cast<float *>(smem + L::kOffM);
  float *sL = reinterpret_cast<float *>(smem + L::kOffL);
  const uint32_t bars = base + L::kOffBar;
  auto bar = [&](int i) { return bars + 8u * i; };
  // block b of the gathered tile: latent dims [128 b, 128 b + 128)
  auto k_full = [&](int b_) { return bar(b_); };
  auto k_empty = [&](int b_) { return bar(NB + b_); };
  const uint32_t q_full = bar(2 * NB), q_empty = bar(2 * NB + 1);
  auto r_full = [&](int i) { return bar(2 * NB + 2 + i); };
  auto r_empty = [&](int i) { return bar(2 * NB + 2 + kMlaRing + i); };
  constexpr int kB2 = 2 * NB + 2 + 2 * kMlaRing;
  auto s_full = [&](int i) { return bar(kB2 + i); };
  auto s_empty = [&](int i) { return bar(kB2 + 2 + i); };
  const uint32_t p_full = bar(kB2 + 4), p_empty = bar(kB2 + 5);
  const uint32_t o_full = bar(kB2 + 6), o_empty = bar(kB2 + 7);
  static_assert(kB2 + 7 < L::kNumBars, "every barrier has its slot");
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b_ = 0; b_ < NB; ++b_) {
      mbar_init(k_full(b_), 32 * kMlaGatWarps);  // one per gather lane
      mbar_init(k_empty(b_), 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < kMlaRing; ++i) {
      mbar_init(r_full(i), 32);
      mbar_init(r_empty(i), kMlaEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full(i), 1);
      mbar_init(s_empty(i), kMlaEpiWarps);
    }
    mbar_init(p_full, kMlaEpiWarps);
    mbar_init(p_empty, 1);
    mbar_init(o_full, 1);
    mbar_init(o_empty, kMlaEpiWarps);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kMlaMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    // ---------------- index and query fetch ----------------
    MlaCursor f = mla_begin(g);
    uint32_t nr = 0, nq = 0;
    int step = 2;
    while (f.valid) {
      if (step == 2) {
        const uint32_t qph = nq & 1u;
        ++nq;
        if (!__all_sync(0xffffffffu,
                        wait_bar_inl(q_empty, qph ^ 1u, abort_flag, status)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full, L::kQBytes);
          for (int cc = 0; cc < CH; ++cc)
            tma_load_4d(sQ + cc * (Hg * 128), &tm_q, q_full, cc * kChunk,
                        f.hg * Hg, f.b, f.s);
        }
      }
      const int slot = nr % kMlaRing;
      const uint32_t ph = (nr / kMlaRing) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(r_empty(slot), ph ^ 1u, abort_flag, status)))
        break;
      const size_t off = ((size_t)f.b * g.S + f.s) * topk +
                         (size_t)f.tile * kTileKeys;
      const int cnt = topk - f.tile * kTileKeys;
      const uint32_t dst = base + L::kOffRing + slot * L::kRingBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = lane + 32 * u;
        if (i < cnt) cp_async4(dst + 4 * i, idx + off + i);
      }
      cp_async_arrive_noinc(r_full(slot));
      ++nr;
      step = mla_next(f, g);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp <= kMlaGatWarps) {
    // ---------------- latent-row gathers ----------------
    constexpr int kSegs = 16;  // 16-byte pieces of a row's 128-dim block
    constexpr int kRows = kTileKeys / kMlaGatWarps;  // rows per warp
    constexpr int kPer = kRows * kSegs / 32;         // copies per lane
    const int gw = warp - 1;
    const size_t row_bytes = (size_t)Dc * 2;
    MlaCursor cur = mla_begin(g);
    uint32_t nv = 0;
    while (cur.valid) {
      const int slot = nv % kMlaRing;
      const uint32_t rph = (nv / kMlaRing) & 1u;
      if (!__all_sync(0xffffffffu,
                      wait_bar_inl(r_full(slot), rph, abort_flag, status)))
        break;
      const int32_t *sIdx =
          reinterpret_cast<const int32_t *>(sRing + slot * L::kRingBytes);
      const int live = topk - cur.tile * kTileKeys;
      const uint8_t *cb = cache + (size_t)cur.b * row_bytes;
      const size_t tok_stride = (size_t)B * row_bytes;
      // this lane's rows (2u + lane/16 of the warp's 16) and their tokens,
      // the same for every block; -1 for a slot with no valid token
      int jr[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int rr = gw * kRows + (u * 32 + lane) / kSegs;
        const int j = rr < live ? sIdx[rr] : -1;
        jr[u] = j >= 0 && j < T ? j : -1;
      }
      bool stop = false;
#pragma unroll 1
      for (int blk = 0; blk < NB; ++blk) {
        if (!__all_sync(0xffffffffu, wait_bar_inl(k_empty(blk), (nv & 1u) ^ 1u,
                                              abort_flag, status))) {
          stop = true;
          break;
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int flat = u * 32 + lane;
          const int rr = gw * kRows + flat / kSegs;
          const int seg = flat % kSegs;  // 0..15 within the block
          const int c = 2 * blk + (seg >> 3), s8 = seg & 7;
          const int j = jr[u];
          cp_async16_zfill(sC + c * (kTileKeys * 128) + rr * 128 +
                               ((s8 ^ (rr & 7)) << 4),
                           cb + (j >= 0 ? (size_t)j * tok_stride : 0) +
                               (blk * kSegs + seg) * 16,
                           j >= 0 ? 16u : 0u);
        }
        cp_async_arrive_noinc(k_full(blk));
      }
      if (stop) break;
      ++nv;
      mla_next(cur, g);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kMlaMmaWarp) {
    // ---------------- MMA issuer (whole warp; lane 0 issues) ----------------
    const uint32_t lead = lane == 0;
    auto wall = [&](uint32_t b_, uint32_t ph) -> bool {
      return __all_sync(0xffffffffu, wait_bar_inl(b_, ph, abort_flag, status));
    };
    MlaCursor cur = mla_begin(g);
    uint32_t nv = 0, nq = 0, nb = 0, nitem = 0;
    int step = 2;
    while (cur.valid) {
      if (step == 2) {
        if (!wall(q_full, nq & 1u)) break;
        ++nq;
      }
      const int sa = nv & 1;
      const uint32_t sph = (nv >> 1) & 1u;
      if (!wall(s_empty(sa), sph ^ 1u)) break;
      // S^T = C_g . Q^T: CH chunks of four K = 16 steps, two chunks per
      // gathered block, each block as soon as it lands
      const uint64_t a1 = sdesc_k_sw128(sC), b1 = sdesc_k_sw128(sQ);
      const uint32_t d1 = tmem + kTmemSm + sa * Hg;
      bool stop = false;
#pragma unroll 1
      for (int blk = 0; blk < NB; ++blk) {
        if (!wall(k_full(blk), nv & 1u)) {
          stop = true;
          break;
        }
        // the block was written by cp.async (generic proxy)
        fence_proxy_async_smem();
        tc_fence_after();
#pragma unroll 1
        for (int t = blk * 8; t < blk * 8 + 8; ++t) {
          const uint32_t ao =
              ((t >> 2) * (kTileKeys * 128) + (t & 3) * 32) >> 4;
          const uint32_t bo = ((t >> 2) * (Hg * 128) + (t & 3) * 32) >> 4;
          mma_bf16_by(d1, a1 + ao, b1 + bo, kIdescS, t != 0 ? 1u : 0u, lead);
        }
      }
      if (stop) break;
      mma_commit_by(s_full(sa), lead);
      {
        const bool first = cur.tile == 0, last = cur.tile + 1 == g.ntiles;
        if (!wall(p_full, nb & 1u)) break;
        if (first && !wall(o_empty, (nitem & 1u) ^ 1u)) break;
        tc_fence_after();
        // O^T += C_g^T . P^T: NB blocks of 128 latent dims (two chunks,
        // 16 KB apart), K = 128 slots in steps of 16 (2048 bytes)
        const uint64_t a2 = sdesc_mn_sw128(sC, kTileKeys * 128, 1024);
        const uint64_t b2 = sdesc_mn_sw128(sP, 1024, 1024);
#pragma unroll 1
        for (int blk = 0; blk < NB; ++blk) {
#pragma unroll 1
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_by(tmem + kTmemO + blk * Hg,
                        a2 + ((blk * 2 * kTileKeys * 128 + ks * 2048) >> 4),
                        b2 + ((ks * 2048) >> 4), kIdescO,
                        (first && ks == 0) ? 0u : 1u, lead);
          // the next tile's block blk may be gathered once these are done
          mma_commit_by(k_empty(blk), lead);
        }
        mma_commit_by(p_empty, lead);
        if (last) {
          mma_commit_by(o_full, lead);
          mma_commit_by(q_empty, lead);
          ++nitem;
        }
        ++nb;
      }
      ++nv;
      step = mla_next(cur, g);
    }
  } else {
    // ---------------- epilogue (warps kMlaEpiWarp0 .. + 7) ----------------
    constexpr int kEpiThreads = 32 * kMlaEpiWarps;
    const int sp = warp & 3;                         // TMEM lane quarter
    const int hh = (warp - kMlaEpiWarp0) >> 2;       // head half
    const int et = threadIdx.x - 32 * kMlaEpiWarp0;  // 0..255
    const int i = sp * 32 + lane;  // TMEM lane: the slot, or the latent dim
    const int hl = hh * 32 + lane;  // the head this lane folds to
    const uint32_t lane_off = (uint32_t)(sp * 32) << 16;
    float *sF = reinterpret_cast<float *>(smem + L::kOffF);  // [64] factors
    // the running maximum moves only when a tile exceeds it by more than
    // 2^kSlack, so a weight is at most 2^kSlack and rescales stay rare
    constexpr float kSlack = 8.f;
    MlaCursor cur = mla_begin(g);
    uint32_t nv = 0, nitem = 0;
    bool ok = true;
    // this thread's 32 heads of its TMEM lane
    auto load32 = [&](uint32_t taddr, float (&v)[32]) {
      uint32_t u[32];
      __syncwarp();
      tmem_ld32(taddr, u);
      tmem_ld_wait();
      reg_fence32(u);
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(u[q]);
    };

    while (cur.valid) {
      if (named_bar_or(1, kEpiThreads, !ok)) break;
      const int b = cur.b, s = cur.s, hg = cur.hg;
      if (et < 64) sM[et] = neg_inf;  // running maximum (log2 domain)
      named_bar_sync(3, kEpiThreads);
      float lp = 0.f;  // l of head hl (this warp's slots)
      bool bad = false;
      int step = 0;
      while (ok && step == 0) {
        const int slot = nv % kMlaRing;
        const uint32_t rph = (nv / kMlaRing) & 1u;
        const int sa = nv & 1;
        const uint32_t sph = (nv >> 1) & 1u;
        const bool got = wait_bar_inl(s_full(sa), sph, abort_flag, status) &&
                         wait_bar_inl(r_full(slot), rph, abort_flag, status);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sS = tmem + lane_off + kTmemSm + sa * Hg + hh * 32;
        const int e = cur.tile * kTileKeys + i;
        const bool in_row = e < topk;
        const int j =
            in_row ? reinterpret_cast<const int32_t *>(sRing +
                                                       slot * L::kRingBytes)[i]
                   : -1;
        __syncwarp();
        if (lane == 0) mbar_arrive(r_empty(slot));
        const bool valid = j >= 0 && j < T;
        bad |= in_row && (j < -1 || j >= T);
        // each head's largest scaled score in the tile
        float v[32];
        load32(sS, v);
#pragma unroll
        for (int h = 0; h < 32; ++h)
          v[h] = valid ? v[h] * scale_log2e : neg_inf;
        warp_fold<32, true>(v, lane);
        sRed[sp * 64 + hl] = v[0];
        named_bar_sync(3, kEpiThreads);
        bool moved = false;
        if (et < 64) {
          const float tmax = fmaxf(fmaxf(sRed[et], sRed[64 + et]),
                                   fmaxf(sRed[128 + et], sRed[192 + et]));
          const float mold = sM[et];
          float f = 1.f;
          if (tmax > mold + kSlack) {
            f = exp2f(mold - tmax);  // 0 while nothing is accumulated
            sM[et] = tmax;
            moved = true;
          }
          sF[et] = f;
        }
        // every thread sees the new maxima and factors, and whether any moved
        const bool rescale = named_bar_or(3, kEpiThreads, moved);
        // the accumulator is idle once MMA2 of the previous tile is done
        if (!__all_sync(0xffffffffu, wait_bar_inl(p_empty, (nv & 1u) ^ 1u,
                                              abort_flag, status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (rescale) {
          lp *= sF[hl];
          if (cur.tile > 0) {
            // O^T[d, h] *= f[h]: this warp's 32 latent dims and 32 heads of
            // every block
#pragma unroll 1
            for (int blk = 0; blk < NB; ++blk) {
              const uint32_t ta = tmem + lane_off + kTmemO + blk * Hg + hh * 32;
              uint32_t u[32];
              __syncwarp();
              tmem_ld32(ta, u);
              tmem_ld_wait();
              reg_fence32(u);
#pragma unroll
              for (int q = 0; q < 32; ++q)
                u[q] = __float_as_uint(__uint_as_float(u[q]) * sF[hh * 32 + q]);
              tmem_st32(ta, u);
            }
            tmem_st_wait();
          }
        }
        // P^T = exp2(x - m) for the tensor core (the fold consumed v)
        load32(sS, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty(sa));
        const float4 *m4 = reinterpret_cast<const float4 *>(sM + hh * 32);
        const uint32_t prow = sP + i * 128;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          uint32_t pk[4];
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const int h = k8 * 8 + hq * 4;
            const float4 mv = m4[h >> 2];
            const float p0 = valid ? exp2f(fmaf(v[h], scale_log2e, -mv.x)) : 0.f;
            const float p1 =
                valid ? exp2f(fmaf(v[h + 1], scale_log2e, -mv.y)) : 0.f;
            const float p2 =
                valid ? exp2f(fmaf(v[h + 2], scale_log2e, -mv.z)) : 0.f;
            const float p3 =
                valid ? exp2f(fmaf(v[h + 3], scale_log2e, -mv.w)) : 0.f;
            v[h] = p0;
            v[h + 1] = p1;
            v[h + 2] = p2;
            v[h + 3] = p3;
            pk[2 * hq] = pack_bf16x2(p0, p1);
            pk[2 * hq + 1] = pack_bf16x2(p2, p3);
          }
          // 16-byte chunk u8 of the 128-byte P^T row holds heads 8 u8 .. + 7
          const int u8 = hh * 4 + k8;
          st_shared_v4(prow + ((u8 ^ (i & 7)) << 4), pk);
        }
        // the tensor core (async proxy) reads P^T and the rescaled O^T next
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        warp_fold<32, false>(v, lane);
        lp += v[0];
        ++nv;
        step = mla_next(cur, g);
      }
      if (named_bar_or(2, kEpiThreads, !ok)) break;
      sRed[sp * 64 + hl] = lp;
      named_bar_sync(3, kEpiThreads);
      if (et < 64)
        sL[et] = ((sRed[et] + sRed[64 + et]) + sRed[128 + et]) + sRed[192 + et];
      named_bar_sync(3, kEpiThreads);
      // ---- o = O^T / l, lse = (m + log2 l) ln 2 ----
      ok = __all_sync(0xffffffffu,
                      wait_bar_inl(o_full, nitem & 1u, abort_flag, status));
      if (ok) {
        tc_fence_after();
        float *orow = out_o + (((size_t)s * B + b) * H + hg * Hg) * Dc;
#pragma unroll 1
        for (int blk = 0; blk < NB; ++blk) {
          uint32_t u[32];
          __syncwarp();
          tmem_ld32(tmem + lane_off + kTmemO + blk * Hg + hh * 32, u);
          tmem_ld_wait();
          reg_fence32(u);
          // lane = latent dim: each store covers 32 consecutive dims
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const int h = hh * 32 + q;
            const float l = sL[h];
            orow[(size_t)h * Dc + blk * 128 + i] =
                l > 0.f ? __uint_as_float(u[q]) / l : 0.f;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty);
        if (et < 64) {
          const float l = sL[et];
          out_lse[((size_t)s * B + b) * H + hg * Hg + et] =
              l > 0.f ? (sM[et] + log2f(l)) * 0.69314718055994531f : neg_inf;
        }
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(status, kStatusIndexRange);
      ++nitem;
    }
  }

  __syncthreads();
  if (warp == kMlaMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int NB>
cudaError_t launch_mla(const CUtensorMap &tm_q, const void *cache,
                       const int32_t *idx, int S, int B, int H, int T,
                       int topk, float scale_log2e, float *out_o,
                       float *out_lse, int *status, int num_sms,
                       cudaStream_t st) {
  auto kern = sparse_mla_kernel<NB>;
  const int smem = MlaSmem<NB>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  MlaGeom g;
  g.S = S;
  g.HG = H / kMlaH;
  g.items = B * S * g.HG;
  g.ntiles = (topk + kTileKeys - 1) / kTileKeys;
  if (g.items <= 0) return cudaSuccess;
  const int grid = g.items < num_sms ? g.items : num_sms;
  kern<<<grid, kMlaThreads, smem, st>>>(
      tm_q, static_cast<const uint8_t *>(cache), idx, g, B, H, T, topk,
      scale_log2e, out_o, out_lse, status);
  return cudaGetLastError();
}

}  // namespace
}  // namespace dsa

extern "C" {

size_t dsa_sparse_mla_workspace_size(void) { return 256; }

int dsa_sparse_mla_fwd(const void *q, const void *c, const int32_t *idx,
                       int S, int B, int H, int Dc, int T, int topk,
                       float scale, float *out_o, float *out_lse,
                       void *workspace, size_t workspace_bytes,
                       void *cuda_stream) {
  if (!q || !c || !idx || !out_o || !out_lse) return DSA_ERR_INVALID_ARG;
  if (S <= 0 || B <= 0 || H <= 0 || Dc <= 0 || T <= 0 || topk <= 0)
    return DSA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || scale > 1e30f) return DSA_ERR_INVALID_ARG;
  if (H % 64 != 0 || Dc % 128 != 0 || Dc > 512) return DSA_ERR_UNSUPPORTED;
  if ((long long)B * S * (H / 64) >= (1ll << 31) || topk > (1 << 30))
    return DSA_ERR_UNSUPPORTED;
  auto al = [](const void *p, unsigned a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
  };
  if (!al(q, 16) || !al(c, 16) || !al(idx, 4) || !al(out_o, 4) ||
      !al(out_lse, 4))
    return DSA_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < dsa_sparse_mla_workspace_size())
    return DSA_ERR_WORKSPACE;
  if (!al(workspace, 256)) return DSA_ERR_INVALID_ARG;
  int num_sms = 0;
  int rc = dsa::device_num_sms(&num_sms);
  if (rc != DSA_OK) return rc;
  dsa::Problem p{q, c, nullptr, nullptr, S, B, H, Dc, T, 1};
  CUtensorMap tm_q;
  rc = dsa::encode_q_heads(&tm_q, p, 1, dsa::kMlaH);
  if (rc != DSA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  int *status = static_cast<int *>(workspace);
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess)
    return DSA_ERR_CUDA;
  const float sl2 = scale * 1.4426950408889634f;  // scale * log2(e)
  cudaError_t e;
  switch (Dc / 128) {
    case 1:
      e = dsa::launch_mla<1>(tm_q, c, idx, S, B, H, T, topk, sl2, out_o,
                             out_lse, status, num_sms, st);
      break;
    case 2:
      e = dsa::launch_mla<2>(tm_q, c, idx, S, B, H, T, topk, sl2, out_o,
                             out_lse, status, num_sms, st);
      break;
    case 3:
      e = dsa::launch_mla<3>(tm_q, c, idx, S, B, H, T, topk, sl2, out_o,
                             out_lse, status, num_sms, st);
      break;
    default:
      e = dsa::launch_mla<4>(tm_q, c, idx, S, B, H, T, topk, sl2, out_o,
                             out_lse, status, num_sms, st);
      break;
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // extern "C"
