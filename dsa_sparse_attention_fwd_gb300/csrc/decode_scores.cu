// decode_scores: lightning-indexer scores for rows with few queries per
// sequence (decode), split over the keys so that every SM streams its share
// of k from HBM.
//
// A work item is (query row r = b*S + s, chunk of kDecChunkTiles x 128 keys).
// One MMA tile is 128 keys (M) x H heads of the row's single query (N = H),
// K = D, so no MMA column is padding.  The K ring (5 or 6 x 128 keys) is
// filled by TMA; the row's Q tile (H x D) is loaded once per item into one of
// two buffers.  The fp32 accumulator sits in TMEM (lane = key, column =
// head); each of the four epilogue warps owns 32 keys and reduces the
// weighted ReLU over the heads in its own registers, then stores the visible
// scores.  Items whose chunk starts past the row's last visible key are
// skipped, so masked keys are never read.
//
// Warp roles (192 threads, one CTA per SM, persistent): warp 0 TMA producer,
// warp 1 TMEM allocator and MMA issuer, warps 2..5 epilogue.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kDecThreads = 192;

template <int H, int KC>
struct DecSmem {
  // K ring stages: six where two Q/weight slots leave room (H <= 64; 3.5%
  // faster on the decode batch than five stages and four Q slots), else
  // five.  Two Q slots keep the next item's Q tile in flight.
  static constexpr int kStages = H <= 64 ? 6 : 5;
  static constexpr int kQSlots = 2;
  static_assert(kDecChunkTiles <= kStages,
                "an item's K tiles are issued before its Q and must fit the "
                "ring");
  static constexpr int kQBytes = KC * H * 128;           // one Q tile
  static constexpr int kKBytes = KC * kTileKeys * 128;   // one K stage
  static constexpr int kWBytes = H * 4;                  // one weight row
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQSlots * kQBytes;
  static constexpr int kOffW = kOffK + kStages * kKBytes;
  static constexpr int kOffBar = kOffW + kQSlots * kWBytes;
  // k_full[S], k_empty[S], q_full[Q], q_empty[Q], acc_full[2], acc_empty[2]
  static constexpr int kNumBars = 2 * kStages + 2 * kQSlots + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

struct DecItem {
  int row, b, s, tile0, ntiles;
};

// Item i covers chunk (i / rows) of row (i % rows): consecutive items are
// different rows, so the long rows' chunks spread over all CTAs.
__device__ __forceinline__ DecItem dec_item(int item, int rows, int S,
                                            int S_kv, int ratio,
                                            const int32_t *q_pos) {
  DecItem it;
  it.row = item % rows;
  const int chunk = item / rows;
  it.b = it.row / S;
  it.s = it.row % S;
  const int nv = n_visible(row_pos(q_pos, it.b, it.s), ratio, S_kv);
  const int tiles = (nv + kTileKeys - 1) / kTileKeys;
  it.tile0 = chunk * kDecChunkTiles;
  const int left = tiles - it.tile0;
  it.ntiles = left <= 0 ? 0 : (left < kDecChunkTiles ? left : kDecChunkTiles);
  return it;
}

__device__ __forceinline__ int dec_item_for(int round, int n_items) {
  const int G = gridDim.x, c = blockIdx.x;
  const int idx = round * G + ((round & 1) ? (G - 1 - c) : c);
  return idx < n_items ? idx : -1;
}

template <int H, int KC, bool KV>
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_scores_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const float *__restrict__ w,
                         const int32_t *__restrict__ q_pos,
                         const uint8_t *__restrict__ kv_valid,
                         float *__restrict__ logits,
                         int S, int B,
                         int S_kv, int ratio, int n_items, int *status) {
  using L = DecSmem<H, KC>;
  constexpr int kDecStages = L::kStages;
  constexpr uint32_t kIdesc = idesc_bf16_f32(kTileKeys, H);
  constexpr int kAccCols = H;  // TMEM columns per accumulator

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const uint32_t sQ = base + L::kOffQ;
  const uint32_t sK = base + L::kOffK;
  float *sW = reinterpret_cast<float *>(smem + L::kOffW);  // [slots][H]
  const uint32_t bars = base + L::kOffBar;
  auto k_full = [&](int i) { return bars + 8u * i; };
  auto k_empty = [&](int i) { return bars + 8u * (kDecStages + i); };
  constexpr int NQ = L::kQSlots;
  auto q_full = [&](int i) { return bars + 8u * (2 * kDecStages + i); };
  auto q_empty = [&](int i) {
    return bars + 8u * (2 * kDecStages + NQ + i);
  };
  auto acc_full = [&](int i) {
    return bars + 8u * (2 * kDecStages + 2 * NQ + i);
  };
  auto acc_empty = [&](int i) {
    return bars + 8u * (2 * kDecStages + 2 * NQ + 2 + i);
  };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
  volatile int *abort_flag = reinterpret_cast<int *>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = B * S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(k_full(i), 1);
      mbar_init(k_empty(i), 1);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(q_full(i), 1);
      mbar_init(q_empty(i), 5);  // the MMA issuer + four epilogue warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(acc_empty(i), 4);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), 2 * kAccCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // the selection kernel may be scheduled now; it waits for this grid to
  // finish before it reads anything
  pdl_allow_dependents();

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t kst = 0, kph = 0, nq = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = dec_item_for(r, n_items);
        if (item < 0) break;
        const DecItem it = dec_item(item, rows, S, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq % NQ;
        const uint32_t qph = (nq / NQ) & 1u;
        ++nq;
        // K tiles first, then the Q/weights slot: the tiles only need free
        // ring stages (an item has at most kDecChunkTiles <= kDecStages of
        // them, and every older item already has its Q), so the ring keeps
        // streaming while the Q slot waits for the item two back to finish.
        for (int t = 0; t < it.ntiles; ++t) {
          if (!(ok = wait_bar(k_empty(kst), kph ^ 1u, abort_flag, status)))
            break;
          mbar_arrive_expect_tx(k_full(kst), L::kKBytes);
          for (int c = 0; c < KC; ++c)
            tma_load_3d(sK + kst * L::kKBytes + c * (kTileKeys * 128), &tm_k,
                        k_full(kst), c * kChunk, it.b,
                        (it.tile0 + t) * kTileKeys);
          if (++kst == kDecStages) {
            kst = 0;
            kph ^= 1u;
          }
        }
        if (!ok) break;
        if (!(ok = wait_bar(q_empty(qs), qph ^ 1u, abort_flag, status))) break;
        mbar_arrive_expect_tx(q_full(qs), L::kQBytes + L::kWBytes);
        for (int c = 0; c < KC; ++c)
          tma_load_4d(sQ + qs * L::kQBytes + c * (H * 128), &tm_q, q_full(qs),
                      c * kChunk, 0, it.b, it.s);
        bulk_load(smem_u32(sW) + qs * L::kWBytes,
                  w + ((size_t)it.s * B + it.b) * H, L::kWBytes, q_full(qs));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t kst = 0, kph = 0, nq = 0, acc = 0, aph = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = dec_item_for(r, n_items);
        if (item < 0) break;
        const DecItem it = dec_item(item, rows, S, S_kv, ratio, q_pos);
        if (it.ntiles == 0) continue;
        const int qs = nq % NQ;
        const uint32_t qph = (nq / NQ) & 1u;
        ++nq;
        if (!(ok = wait_bar(q_full(qs), qph, abort_flag, status))) break;
        const uint32_t sQi = sQ + qs * L::kQBytes;
        for (int t = 0; t < it.ntiles; ++t) {
          if (!(ok = wait_bar(acc_empty(acc), aph ^ 1u, abort_flag, status)))
            break;
          if (!(ok = wait_bar(k_full(kst), kph, abort_flag, status))) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + acc * kAccCols;
#pragma unroll
          for (int c = 0; c < KC; ++c) {
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk) {
              const uint64_t ad = sdesc_k_sw128(
                  sK + kst * L::kKBytes + c * (kTileKeys * 128) + kk * 32);
              const uint64_t bd = sdesc_k_sw128(sQi + c * (H * 128) + kk * 32);
              mma_bf16(d_tmem, ad, bd, kIdesc, (c | kk) != 0);
            }
          }
          mma_commit(k_empty(kst));
          mma_commit(acc_full(acc));
          if (t == it.ntiles - 1) mma_commit(q_empty(qs));
          if (++kst == kDecStages) {
            kst = 0;
            kph ^= 1u;
          }
          acc ^= 1u;
          if (acc == 0) aph ^= 1u;
        }
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int sp = warp & 3;            // TMEM sub-partition of this warp
    uint32_t acc = 0, aph = 0, nq = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = dec_item_for(r, n_items);
      if (item < 0) break;
      const DecItem it = dec_item(item, rows, S, S_kv, ratio, q_pos);
      if (it.ntiles == 0) continue;
      // the row's weights arrive with its Q tile (same slot, same barrier)
      const int qs = nq % NQ;
      const uint32_t qph = (nq / NQ) & 1u;
      ++nq;
      bool wok = wait_bar(q_full(qs), qph, abort_flag, status);
      if (!__all_sync(0xffffffffu, wok)) break;
      const float *wq = sW + qs * H;
      const long long pos = row_pos(q_pos, it.b, it.s);
      float *out = logits + (size_t)it.row * S_kv;
      for (int t = 0; t < it.ntiles; ++t) {
        bool got = wait_bar(acc_full(acc), aph, abort_flag, status);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr =
            tmem + ((uint32_t)(sp * 32) << 16) + acc * kAccCols;
        uint32_t v[H / 32][32];
#pragma unroll
        for (int c = 0; c < H / 32; ++c) tmem_ld32(taddr + c * 32, v[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < H / 32; ++c) reg_fence32(v[c]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(acc));
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < H; h += 2) {
          s0 = fmaf(wq[h], relu2(__uint_as_float(v[h >> 5][h & 31])), s0);
          s1 = fmaf(wq[h + 1],
                    relu2(__uint_as_float(v[(h + 1) >> 5][(h + 1) & 31])),
                    s1);
        }
        const int j = (it.tile0 + t) * kTileKeys + sp * 32 + lane;
        if ((long long)(j + 1) * ratio - 1 <= pos && j < S_kv) {
          // a key that is not a candidate scores -inf (pool variant)
          const bool kv_ok = !KV ||
                             __ldg(kv_valid + (size_t)j * B + it.b) != 0;
          // the sums are of w * 2 ReLU (x + |x|): halving them is exact
          const float sc =
              kv_ok ? 0.5f * (s0 + s1) : -__int_as_float(0x7f800000);
          out[j] = sc;
        }
        acc ^= 1u;
        if (acc == 0) aph ^= 1u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty(qs));  // done with this Q/w slot
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kAccCols);
  }
}

template <int H, int KC>
cudaError_t launch_dec(const Problem &p, const CUtensorMap &tm_q,
                       const CUtensorMap &tm_k, float *logits,
                       int *status, int num_sms, cudaStream_t st) {
  // only the masked instantiation reads the key-validity mask
  auto kern = p.kv_valid ? decode_scores_kernel<H, KC, true>
                         : decode_scores_kernel<H, KC, false>;
  const int smem = DecSmem<H, KC>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int rows = p.B * p.S;
  const int tiles = (p.S_kv + kTileKeys - 1) / kTileKeys;
  const int chunks = (tiles + kDecChunkTiles - 1) / kDecChunkTiles;
  const long long n_items = (long long)rows * chunks;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = (int)(n_items < num_sms ? n_items : num_sms);
  kern<<<grid, kDecThreads, smem, st>>>(tm_q, tm_k, p.w, p.q_pos,
                                        p.kv_valid, logits, p.S,
                                        p.B, p.S_kv, p.ratio, (int)n_items,
                                        status);
  return cudaGetLastError();
}

}  // namespace

bool decode_supported(int H, int D) {
  return (H == 32 || H == 64 || H == 128) && D <= 2 * kChunk;
}

size_t decode_smem_bytes(int H, int D) {
  const int kc = D <= kChunk ? 1 : 2;
  if (H == 32) return kc == 1 ? DecSmem<32, 1>::kAlloc : DecSmem<32, 2>::kAlloc;
  if (H == 64) return kc == 1 ? DecSmem<64, 1>::kAlloc : DecSmem<64, 2>::kAlloc;
  return kc == 1 ? DecSmem<128, 1>::kAlloc : DecSmem<128, 2>::kAlloc;
}

cudaError_t launch_decode_scores(const Problem &p, const CUtensorMap &tm_q,
                                 const CUtensorMap &tm_k, float *logits,
                                 int *status, int num_sms, cudaStream_t st) {
  const bool k1 = p.D <= kChunk;
  switch (p.H) {
    case 32:
      return k1 ? launch_dec<32, 1>(p, tm_q, tm_k, logits, status, num_sms, st)
                : launch_dec<32, 2>(p, tm_q, tm_k, logits, status, num_sms, st);
    case 64:
      return k1 ? launch_dec<64, 1>(p, tm_q, tm_k, logits, status, num_sms, st)
                : launch_dec<64, 2>(p, tm_q, tm_k, logits, status, num_sms, st);
    case 128:
      return k1 ? launch_dec<128, 1>(p, tm_q, tm_k, logits, status, num_sms, st)
                : launch_dec<128, 2>(p, tm_q, tm_k, logits, status, num_sms, st);
    default:
      return cudaErrorNotSupported;
  }
}

}  // namespace dsa
