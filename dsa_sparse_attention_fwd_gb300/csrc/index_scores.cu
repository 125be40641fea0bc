// index_scores: the lightning-indexer score I[t, j] = sum_h w[t,h] *
// ReLU(q[t,h,:] . k[j,:]) for every visible (query, compressed key) pair,
// on the sm_103a tensor cores.
//
// Orientation: one MMA tile is 128 keys (M) x 256 (query, head) columns (N),
// K = D.  A = a K tile [128 keys x D] and B = a Q tile [256/H queries x H
// heads x D], both K-major in shared memory with the 128-byte swizzle, staged
// by TMA.  The fp32 accumulator lives in tensor memory: TMEM lane = key,
// column = (query, head).  Each epilogue thread owns one key, so the per-head
// weighted ReLU sum runs along its own registers with no cross-thread
// reduction.  Two accumulators (2 x 256 TMEM columns) let the epilogue of
// tile i overlap the MMA of tile i+1.
//
// Warp roles (320 threads, one CTA per SM, persistent):
//   warp 0      TMA producer: Q tile once per work item into one of two Q
//               buffers (so the next item's Q lands while the current one is
//               multiplied), K tiles through a 3- or 4-stage ring.
//   warp 1      TMEM allocator and MMA issuer (one thread).
//   warps 2..9  epilogue: TMEM -> registers, ReLU, weight multiply-reduce over
//               heads, causal mask, store of the visible scores.
// A work item is (sequence b, block of 256/H consecutive queries); its key
// tiles stop at the last tile any of its queries can see, so fully masked
// tiles are never loaded or multiplied.  Items are dealt to CTAs in a
// zig-zag over a longest-first order to balance the causal triangle.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

template <int H, int KC>
struct ScoreSmem {
  static constexpr int kTQ = kTileCols / H;              // queries per item
  static constexpr int kQSlots = 2;
  static constexpr int kStages = KC == 1 ? 4 : 3;        // K ring depth
  static constexpr int kQBytes = KC * kTileCols * 128;  // one Q tile
  static constexpr int kKBytes = KC * kTileKeys * 128;  // one K stage
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kQBytes;
  static constexpr int kOffW = kOffK + kStages * kKBytes;
  static constexpr int kOffBar = kOffW + kTileCols * 4;
  // barriers: k_full[S], k_empty[S], q_full[2], q_empty[2], acc_full[2],
  // acc_empty[2]
  static constexpr int kNumBars = 2 * kStages + 4 + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  // room to align the base; at least 120 KB so that only one CTA fits on
  // an SM (each CTA allocates all 512 TMEM columns)
  static constexpr int kAlloc =
      kBytes + 1024 > 120 * 1024 ? kBytes + 1024 : 120 * 1024;
};

struct ItemInfo {
  int b, t0, ntiles;
};

// Rows [s0, s0 + S) of every sequence (one chunk of the query rows).
template <int H>
__device__ __forceinline__ ItemInfo item_info(int item, int s0, int S, int B,
                                              int S_kv, int ratio,
                                              const int32_t *q_pos) {
  constexpr int TQ = kTileCols / H;
  const int n_qb = (S + TQ - 1) / TQ;
  ItemInfo it;
  const int qb = n_qb - 1 - item / B;  // longest (latest) query blocks first
  it.b = item % B;
  it.t0 = s0 + qb * TQ;
  const int t_last = min(it.t0 + TQ - 1, s0 + S - 1);
  const int nv = n_visible(row_pos(q_pos, it.b, t_last), ratio, S_kv);
  it.ntiles = (nv + kTileKeys - 1) / kTileKeys;
  return it;
}

// Zig-zag deal of items to CTAs: round r gives CTA c item r*G + c (r even) or
// r*G + G-1-c (r odd).  Returns -1 past the end.
__device__ __forceinline__ int item_for(int round, int n_items) {
  const int G = gridDim.x, c = blockIdx.x;
  const int idx = round * G + ((round & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

template <int H, int KC, bool KV>
__global__ void __launch_bounds__(kScoreThreads, 1)
    index_scores_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const float *__restrict__ w,
                        const int32_t *__restrict__ q_pos,
                        const uint8_t *__restrict__ kv_valid,
                        float *__restrict__ logits, int s0, int S, int B,
                        int S_kv, int ratio, int *status) {
  using L = ScoreSmem<H, KC>;
  constexpr int NQ = L::kQSlots;
  constexpr int kStages = L::kStages;
  constexpr int TQ = kTileCols / H;  // queries per work item
  constexpr int QH = TQ / 2;         // queries per epilogue column half
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileKeys, kTileCols);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);

  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sK = base + L::kOffK;
  float *sW = reinterpret_cast<float *>(smem + L::kOffW);
  const uint32_t bars = base + L::kOffBar;
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (kStages + s); };
  auto q_full = [&](int qs) { return bars + 8u * (2 * kStages + qs); };
  auto q_empty = [&](int qs) { return bars + 8u * (2 * kStages + 2 + qs); };
  auto acc_full = [&](int a) { return bars + 8u * (2 * kStages + 4 + a); };
  auto acc_empty = [&](int a) { return bars + 8u * (2 * kStages + 6 + a); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_items = ((S + TQ - 1) / TQ) * B;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(q_full(a), 1);
      mbar_init(q_empty(a), 1);
      mbar_init(acc_full(a), 1);
      mbar_init(acc_empty(a), 8);  // one arrival per epilogue warp
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
  // launched behind the previous chunk's selection, which still reads the
  // logits buffer: wait for it before anything is written (the setup above
  // overlapped its tail)
  pdl_wait();
  // the selection kernel may be scheduled now; it waits for this grid to
  // finish before it reads anything
  pdl_allow_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // q is read once: keep it from pushing the logits out of L2
      const uint64_t pol_q = l2_policy_evict_first();
      uint32_t kst = 0, kph = 0, nq = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_for(r, n_items);
        if (item < 0) break;
        const ItemInfo it = item_info<H>(item, s0, S, B, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq % NQ;
        const uint32_t qph = (nq / NQ) & 1u;
        ++nq;
        if (!(ok = wait_bar(q_empty(qs), qph ^ 1u, abort_flag, status))) break;
        mbar_arrive_expect_tx(q_full(qs), L::kQBytes);
        for (int c = 0; c < KC; ++c)
          tma_load_4d_hint(sQ + qs * L::kQBytes + c * (kTileCols * 128),
                           &tm_q, q_full(qs), c * kChunk, 0, it.b, it.t0,
                           pol_q);
        for (int tile = 0; tile < it.ntiles; ++tile) {
          if (!(ok = wait_bar(k_empty(kst), kph ^ 1u, abort_flag, status)))
            break;
          mbar_arrive_expect_tx(k_full(kst), L::kKBytes);
          for (int c = 0; c < KC; ++c)
            tma_load_3d(sK + kst * L::kKBytes + c * (kTileKeys * 128), &tm_k,
                        k_full(kst), c * kChunk, it.b, tile * kTileKeys);
          if (++kst == kStages) {
            kst = 0;
            kph ^= 1u;
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
        const ItemInfo it = item_info<H>(item, s0, S, B, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq % NQ;
        const uint32_t qph = (nq / NQ) & 1u;
        ++nq;
        if (!(ok = wait_bar(q_full(qs), qph, abort_flag, status))) break;
        const uint32_t sQi = sQ + qs * L::kQBytes;
        for (int tile = 0; tile < it.ntiles; ++tile) {
          if (!(ok = wait_bar(acc_empty(acc), aph ^ 1u, abort_flag, status)))
            break;
          if (!(ok = wait_bar(k_full(kst), kph, abort_flag, status))) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + acc * kTileCols;
#pragma unroll
          for (int c = 0; c < KC; ++c) {
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk) {
              const uint64_t ad = sdesc_k_sw128(
                  sK + kst * L::kKBytes + c * (kTileKeys * 128) + kk * 32);
              const uint64_t bd =
                  sdesc_k_sw128(sQi + c * (kTileCols * 128) + kk * 32);
              mma_bf16(d_tmem, ad, bd, kIdesc, (c | kk) != 0);
            }
          }
          mma_commit(k_empty(kst));   // K stage reusable when done
          mma_commit(acc_full(acc));  // accumulator ready
          if (tile == it.ntiles - 1) mma_commit(q_empty(qs));
          if (++kst == kStages) {
            kst = 0;
            kph ^= 1u;
          }
          acc ^= 1u;
          if (acc == 0) aph ^= 1u;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..9) ----------------
    const int ew = warp - 2;          // 0..7
    const int sp = warp & 3;          // TMEM sub-partition of this warp
    const int half = ew >> 2;         // which 128 columns
    const int et = threadIdx.x - 64;  // 0..255
    uint32_t acc = 0, aph = 0;
    bool ok = true;
    const int tq_mine = et / H, h_mine = et % H;  // the weight this thread loads
    auto weight_of = [&](const ItemInfo &it) -> float {
      const int t = it.t0 + tq_mine;
      return t < s0 + S ? __ldg(w + ((size_t)t * B + it.b) * H + h_mine)
                        : 0.f;
    };
    // first item with work at or after round r (ntiles = -1: none)
    auto next_item = [&](int r, int &round) -> ItemInfo {
      for (;; ++r) {
        const int item = item_for(r, n_items);
        if (item < 0) break;
        const ItemInfo it = item_info<H>(item, s0, S, B, S_kv, ratio, q_pos);
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
    };
    int r = 0;
    ItemInfo it = next_item(0, r);
    // the weights of the next item are loaded one item ahead, so their
    // global-memory latency hides behind the current item's tiles
    float w_next = it.ntiles > 0 ? weight_of(it) : 0.f;
    while (it.ntiles > 0) {
      // everyone is done with the previous weights; stop together if any
      // epilogue warp gave up on a wait
      if (named_bar_or(1, 256, !ok)) break;
      sW[et] = 0.5f * w_next;  // halved: see the ReLU below
      named_bar_sync(1, 256);
      int r_next;
      const ItemInfo nx = next_item(r + 1, r_next);
      if (nx.ntiles > 0) w_next = weight_of(nx);
      // position of query row t is qbase + t
      const long long qbase = row_pos(q_pos, it.b, 0);
      // keys visible to the half's rows (none past the chunk's last row),
      // kept in registers when the half has at most four rows: key j of a
      // row counts iff j < nvq
      constexpr int NQ = QH <= 4 ? QH : 1;
      int nvq[NQ];
#pragma unroll
      for (int qq = 0; qq < NQ; ++qq) {
        const int t = it.t0 + half * QH + qq;
        nvq[qq] = t < s0 + S ? n_visible(qbase + t, ratio, S_kv) : 0;
      }

      for (int tile = 0; tile < it.ntiles; ++tile) {
        bool got = wait_bar(acc_full(acc), aph, abort_flag, status);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(sp * 32) << 16) +
                               acc * kTileCols + half * 128;
        uint32_t v[4][32];
        tmem_ld32(taddr + 0, v[0]);
        tmem_ld32(taddr + 32, v[1]);
        tmem_ld32(taddr + 64, v[2]);
        tmem_ld32(taddr + 96, v[3]);
        tmem_ld_wait();
        reg_fence32(v[0]);
        reg_fence32(v[1]);
        reg_fence32(v[2]);
        reg_fence32(v[3]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(acc));

        const int j = tile * kTileKeys + sp * 32 + lane;
        // a key that is not a candidate scores -inf (pool variant)
        // (only the masked instantiation reads the mask: the load costs the
        // unmasked epilogue ~8% even when the pointer is null)
        const bool kv_ok = !KV || j >= S_kv ||
                           __ldg(kv_valid + (size_t)j * B + it.b) != 0;
#pragma unroll
        for (int qq = 0; qq < QH; ++qq) {
          const int tq = half * QH + qq;
          const float *wq = sW + tq * H;
          float score;
          if constexpr (H % 4 == 0) {
            // even heads in .x, odd heads in .y; weights four at a time
            float2 acc2 = make_float2(0.f, 0.f);
            const float4 *wq4 = reinterpret_cast<const float4 *>(wq);
#pragma unroll
            for (int h = 0; h < H; h += 4) {
              const float4 wv = wq4[h >> 2];
              const int c = qq * H + h;
              const float2 r01 =
                  relu2x2(__uint_as_float(v[c >> 5][c & 31]),
                          __uint_as_float(v[(c + 1) >> 5][(c + 1) & 31]));
              const float2 r23 =
                  relu2x2(__uint_as_float(v[(c + 2) >> 5][(c + 2) & 31]),
                          __uint_as_float(v[(c + 3) >> 5][(c + 3) & 31]));
              acc2 = __ffma2_rn(make_float2(wv.x, wv.y), r01, acc2);
              acc2 = __ffma2_rn(make_float2(wv.z, wv.w), r23, acc2);
            }
            score = acc2.x + acc2.y;
          } else {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int h = 0; h < H; h += 2) {
              const int c0 = qq * H + h;
              s0 = fmaf(wq[h],
                        relu2(__uint_as_float(v[c0 >> 5][c0 & 31])), s0);
              if (h + 1 < H) {
                const int c1 = c0 + 1;
                s1 = fmaf(wq[h + 1],
                          relu2(__uint_as_float(v[c1 >> 5][c1 & 31])),
                          s1);
              }
            }
            score = s0 + s1;
          }
          const int t = it.t0 + tq;
          bool vis;
          if constexpr (QH <= 4) {
            vis = j < nvq[qq];
          } else {
            vis = t < s0 + S && j < S_kv &&
                  (long long)(j + 1) * ratio - 1 <= qbase + t;
          }
          if (vis) {
            const float sv = kv_ok ? score : -__int_as_float(0x7f800000);
            logits[((size_t)it.b * S + (t - s0)) * S_kv + j] = sv;
          }
        }
        acc ^= 1u;
        if (acc == 0) aph ^= 1u;
      }
      it = nx;
      r = r_next;
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
cudaError_t launch_h(const Problem &p, const CUtensorMap &tm_q,
                     const CUtensorMap &tm_k, float *logits, int *status,
                     int num_sms, cudaStream_t st, int s0, int Sc) {
  constexpr int TQ = kTileCols / H;
  auto kern = index_scores_kernel<H, KC, KV>;
  const int smem = ScoreSmem<H, KC>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long n_items = (long long)((Sc + TQ - 1) / TQ) * p.B;
  const int grid = (int)(n_items < num_sms ? n_items : num_sms);
  if (grid <= 0) return cudaSuccess;
  // programmatic stream serialization: the CTAs may start while the
  // previous kernel (a selection) drains, and wait for it in the kernel
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kScoreThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tm_q, tm_k, p.w, p.q_pos, p.kv_valid,
                            logits, s0, Sc, p.B, p.S_kv, p.ratio, status);
}

template <int H, int KC>
cudaError_t launch_t(const Problem &p, const CUtensorMap &tm_q,
                     const CUtensorMap &tm_k, float *logits, int *status,
                     int num_sms, cudaStream_t st, int s0, int Sc) {
  return p.kv_valid ? launch_h<H, KC, true>(p, tm_q, tm_k, logits, status,
                                            num_sms, st, s0, Sc)
                    : launch_h<H, KC, false>(p, tm_q, tm_k, logits, status,
                                             num_sms, st, s0, Sc);
}

template <int KC>
cudaError_t launch_kc(const Problem &p, const CUtensorMap &tm_q,
                      const CUtensorMap &tm_k, float *logits, int *status,
                      int num_sms, cudaStream_t st, int s0, int Sc) {
  switch (p.H) {
    case 1: return launch_t<1, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 2: return launch_t<2, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 4: return launch_t<4, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 8: return launch_t<8, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 16:
      return launch_t<16, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 32:
      return launch_t<32, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 64:
      return launch_t<64, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    case 128:
      return launch_t<128, KC>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t index_scores_smem_bytes(int H, int D) {
  size_t m = 0;
#define DSA_SMEM_CASE(HH)                                           \
  if (H == HH)                                                      \
    m = D <= kChunk ? ScoreSmem<HH, 1>::kAlloc : ScoreSmem<HH, 2>::kAlloc;
  DSA_SMEM_CASE(1) DSA_SMEM_CASE(2) DSA_SMEM_CASE(4) DSA_SMEM_CASE(8)
  DSA_SMEM_CASE(16) DSA_SMEM_CASE(32) DSA_SMEM_CASE(64) DSA_SMEM_CASE(128)
#undef DSA_SMEM_CASE
  return m;
}

cudaError_t launch_index_scores(const Problem &p, const CUtensorMap &tm_q,
                                const CUtensorMap &tm_k, float *logits,
                                int *status, int num_sms, cudaStream_t st,
                                int s0, int Sc) {
  if (p.D <= kChunk)
    return launch_kc<1>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
  return launch_kc<2>(p, tm_q, tm_k, logits, status, num_sms, st, s0, Sc);
}

}  // namespace dsa
