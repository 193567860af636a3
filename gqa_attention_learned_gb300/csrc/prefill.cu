// Causal prefill (ragged, or appended to a paged KV prefix) with learned
// sinks on the 5th-generation tensor cores (tcgen05 + tensor memory).
//
// Operation: "GPT-OSS on day 0" (Perplexity blog), section "Kernels for
// GPT-OSS / Sink Attention" -- each head's running max starts at its sink and
// its running sum at 1, so the sink joins the softmax denominator without a
// value row.  Query i of a request with kv_len keys and q_len new queries
// sees keys j <= kv_len - q_len + i (for plain prefill kv_len = q_len).
//
// Persistent kernel, one CTA per SM.  A work item is 256 consecutive query
// rows of one query head, held as two 128-row tiles A and B that share every
// K/V tile.  Roles (10 warps):
//   warp 8      TMA producer: Q_A, Q_B per item, then K/V tiles of 128 keys
//               into a 4-stage ring (contiguous: one 16 KB box each; paged:
//               eight 2 KB page boxes each), 128-byte swizzle.  It runs ahead
//               into the next item as soon as buffers free up.
//   warp 9      MMA issuer (one thread), ping-pong over the two tiles:
//                 QK_A(0) QK_B(0) | PV_A(j) QK_A(j+1) PV_B(j) QK_B(j+1) | ...
//               S = Q K^T: tcgen05.mma, A and B from shared memory, M=128
//               N=128 K=16 x4, into tensor memory; O += P V: A = P from
//               tensor memory, B = V from shared memory (MN-major), N=64.
//   warps 0..3  softmax for tile A, warps 4..7 for tile B: one thread per
//               query row (= tensor-memory lane).  S is read once per tile,
//               the online softmax runs in base 2 started at the sink, P
//               (bf16) goes back into tensor memory, and O accumulates in
//               tensor memory, rescaled only when a row max grows by more
//               than 2^8.  While softmax A works, the tensor core runs tile
//               B's MMAs and vice versa.
// Tensor memory (512 columns): per tile S 128, P 64, O 64.
// V rows past a request's last key are zeroed in shared memory before the PV
// MMA (0 * NaN would poison whole rows); score columns past a row's causal
// limit are masked by index.  Items are ordered heaviest first (latest query
// rows see the most keys) and dealt round-robin to the CTAs.

#include "kernels.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>

namespace sa {
namespace {

constexpr int kBM = 128;                       // query rows per tile
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kStages = 4;
constexpr int kTileBytes = kBN * kHeadDim * 2;    // 16 KB
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192, kSlotCols = 256;
constexpr float kRescaleLog2 = 8.f;     // lazy O rescale threshold (P < 256)
constexpr int kFlagRing = 4;            // per-item "skipped page" flags in flight

constexpr int kOffQ = 0;                                    // Q_A, Q_B
constexpr int kOffStage = 2 * kTileBytes;                   // K then V per stage
constexpr int kOffBars = kOffStage + kStages * 2 * kTileBytes;
constexpr int kSmemBytes = kOffBars + 256 + 1024;           // barriers + alignment slack

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int bad[kFlagRing];  // an out-of-range page id was skipped for this item
  int abort_all;       // a wait timed out: every role stops
};
static_assert(sizeof(Bars) <= 256, "barrier block");

constexpr uint32_t kIdescQK = umma_idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = umma_idesc_bf16(128, 64, false, true);

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// P = 2^(s * sl2 - mu) for 32 scores, packed as bf16 pairs into r[0..15];
// the pair sums accumulate in `acc` (fp32x2).
template <int E = 0>
__device__ __forceinline__ void pack_chunk(uint32_t (&r)[32], uint64_t scale2, uint64_t negmu2,
                                           uint64_t &acc) {
  if constexpr (E < 16) {
    float x0, x1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * E]), __uint_as_float(r[2 * E + 1])), scale2,
                     negmu2),
              x0, x1);
    const float p0 = ex2(x0);
    const float p1 = ex2(x1);
    acc = f2_add(acc, f2_pack(p0, p1));
    r[E] = pack_bf16(p0, p1);
    pack_chunk<E + 1>(r, scale2, negmu2, acc);
  }
}

// Geometry of one work item, computed identically by every role.
struct Item {
  int seq, head, kvh, pair;
  int q_start, q_len, kv_len, k_start;
  int i0;              // first query row (within the request) of tile A
  int rows[2];         // valid rows of tile A / B (<= 0: tile absent)
  int ntiles[2];       // KV tiles tile A / B needs
  int n;               // KV tiles loaded for the item
  bool bad;            // arguments out of range
  bool empty;          // nothing to compute (bad, or pair past the request's end)
};

template <bool kPaged>
__device__ __forceinline__ Item make_item(const PrefillParams &p, int idx) {
  Item it;
  const int per_pair = p.num_seqs * p.num_qo_heads;
  it.pair = p.num_q_tiles - 1 - idx / per_pair;       // num_q_tiles counts 256-row pairs
  const int rem = idx % per_pair;
  it.head = rem % p.num_qo_heads;
  it.seq = rem / p.num_qo_heads;
  it.kvh = it.head / p.group;
  it.q_start = p.cu_seqlens_q[it.seq];
  const int q_end = p.cu_seqlens_q[it.seq + 1];
  it.q_len = q_end - it.q_start;
  it.k_start = 0;
  if constexpr (kPaged) {
    it.kv_len = p.kv_lens[it.seq];
  } else {
    it.k_start = p.cu_seqlens_k[it.seq];
    it.kv_len = p.cu_seqlens_k[it.seq + 1] - it.k_start;
  }
  bool bad = it.q_start < 0 || it.q_len < 0 || q_end > p.total_q || it.q_len > p.max_q_len ||
             it.kv_len < it.q_len || it.kv_len > p.max_kv_len;
  if constexpr (kPaged) {
    bad = bad || cdiv(it.kv_len, kPageSize) > p.max_pages_per_seq;
  } else {
    bad = bad || it.k_start < 0 || it.k_start + it.kv_len > p.total_k;
  }
  it.bad = bad;
  it.i0 = it.pair * 2 * kBM;
  it.empty = bad || it.i0 >= it.q_len;
  it.rows[0] = it.rows[1] = 0;
  it.ntiles[0] = it.ntiles[1] = 0;
  it.n = 0;
  if (!it.empty) {
    const int shift = it.kv_len - it.q_len;
    for (int t = 0; t < 2; ++t) {
      const int first = it.i0 + t * kBM;
      it.rows[t] = min(kBM, it.q_len - first);
      it.ntiles[t] = it.rows[t] > 0 ? cdiv(shift + first + it.rows[t], kBN) : 0;
    }
    it.n = max(it.ntiles[0], it.ntiles[1]);
  }
  return it;
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_items = p.num_q_tiles * p.num_seqs * p.num_qo_heads;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  Bars &bar = *reinterpret_cast<Bars *>(smem + kOffBars);
  auto sQ = [&](int t) { return smem + kOffQ + t * kTileBytes; };
  auto sK = [&](int s) { return smem + kOffStage + s * 2 * kTileBytes; };
  auto sV = [&](int s) { return smem + kOffStage + s * 2 * kTileBytes + kTileBytes; };

  if (warp == kMmaWarp) {
    tmem_alloc(&bar.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == kProducerWarp * 32) {
    mbar_init(&bar.q_full, 1);
    mbar_init(&bar.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar.kv_full[s], 1);
      mbar_init(&bar.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar.s_full[t], 1);
      mbar_init(&bar.p_full[t], kBM);
      mbar_init(&bar.o_full[t], 1);
      mbar_init(&bar.o_empty[t], kBM);
    }
    mbar_init(&bar.drain, 1);
    for (int f = 0; f < kFlagRing; ++f) bar.bad[f] = 0;
    bar.abort_all = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;
  volatile int *abort_flag = &bar.abort_all;
  auto fail = [&]() { atomicOr(&bar.abort_all, 1); };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    uint32_t kv_iter = 0, items_done = 0;
    for (int idx = blockIdx.x; idx < num_items && !*abort_flag; idx += gridDim.x) {
      const Item it = make_item<kPaged>(p, idx);
      if (it.empty) continue;
      if (items_done > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar.q_empty, (items_done - 1) & 1))) {
        fail();
        break;
      }
      // The flag slot's previous user is kFlagRing items back; the softmax
      // warps have read it long before this item's Q can be loaded.
      int *bad_flag = &bar.bad[items_done % kFlagRing];
      if (lane == 0) {
        *bad_flag = 0;
        mbar_arrive_expect_tx(&bar.q_full, 2 * kTileBytes);
        tma_load_3d(sQ(0), &qmap, &bar.q_full, 0, it.head, it.q_start + it.i0);
        tma_load_3d(sQ(1), &qmap, &bar.q_full, 0, it.head, it.q_start + it.i0 + kBM);
      }
      __syncwarp();
      const int32_t *table =
          kPaged ? p.page_table + static_cast<size_t>(it.seq) * p.max_pages_per_seq : nullptr;
      const int npages = cdiv(it.kv_len, kPageSize);
      bool ok = true;
      for (int j = 0; j < it.n; ++j, ++kv_iter) {
        const int s = kv_iter % kStages;
        if (kv_iter >= kStages &&
            !__all_sync(0xffffffffu, mbar_wait(&bar.kv_empty[s], ((kv_iter / kStages) + 1) & 1))) {
          ok = false;
          break;
        }
        if constexpr (kPaged) {
          // lanes 0..7 each own one 16-token page of the 128-key tile
          const int pg = j * (kBN / kPageSize) + lane;
          int pid = -1;
          if (lane < kBN / kPageSize && pg < npages) pid = table[pg];
          const bool good = pid >= 0 && pid < p.num_pages;
          if (lane < kBN / kPageSize && pg < npages && !good) atomicOr(bad_flag, 1);
          const unsigned mask = __ballot_sync(0xffffffffu, good);
          if (lane == 0)
            mbar_arrive_expect_tx(&bar.kv_full[s], __popc(mask) * 2 * kPageSize * kHeadDim * 2);
          __syncwarp();
          if (good) {
            const int off = lane * kPageSize * kHeadDim * 2;
            tma_load_3d(sK(s) + off, &kmap, &bar.kv_full[s], 0, it.kvh * kPageSize, pid);
            tma_load_3d(sV(s) + off, &vmap, &bar.kv_full[s], 0, it.kvh * kPageSize, pid);
          }
        } else {
          if (lane == 0) {
            mbar_arrive_expect_tx(&bar.kv_full[s], 2 * kTileBytes);
            tma_load_3d(sK(s), &kmap, &bar.kv_full[s], 0, it.kvh, it.k_start + j * kBN);
            tma_load_3d(sV(s), &vmap, &bar.kv_full[s], 0, it.kvh, it.k_start + j * kBN);
          }
        }
        __syncwarp();
      }
      if (!ok) {
        fail();
        break;
      }
      ++items_done;
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------------- MMA
    uint32_t kv_iter = 0, items_done = 0;
    uint32_t s_cnt[2] = {0, 0}, o_cnt[2] = {0, 0};
    const uint64_t dq[2] = {umma_desc_sw128(smem_u32(sQ(0)), 16, 1024),
                            umma_desc_sw128(smem_u32(sQ(1)), 16, 1024)};
    bool ok = true;
    auto wait = [&](uint64_t *b, uint32_t parity) {
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(b, parity));
    };
    for (int idx = blockIdx.x; ok && idx < num_items && !*abort_flag; idx += gridDim.x) {
      const Item it = make_item<kPaged>(p, idx);
      if (it.empty) continue;
      wait(&bar.q_full, items_done & 1);
      tc_fence_after();
      const uint32_t base_iter = kv_iter;
      int waited = -1;                          // last KV tile whose kv_full was awaited
      int zeroed = -1;                          // last KV tile whose V tail was cleared
      auto issue_qk = [&](int t, int j) {
        if (j > waited) {
          wait(&bar.kv_full[(base_iter + j) % kStages], ((base_iter + j) / kStages) & 1);
          tc_fence_after();
          waited = j;
        }
        if (!ok) return;
        if (lane == 0) {
          const uint64_t dk = umma_desc_sw128(smem_u32(sK((base_iter + j) % kStages)), 16, 1024);
          const uint32_t tS = tmem + t * kSlotCols + kColS;
#pragma unroll
          for (int kk = 0; kk < kHeadDim / 16; ++kk)
            umma_ss(tS, dq[t] + 2 * kk, dk + 2 * kk, kIdescQK, kk > 0);   // +32 bytes per k-step
          umma_commit(&bar.s_full[t]);
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int j) {
        wait(&bar.p_full[t], s_cnt[t] & 1);
        ++s_cnt[t];
        if (j == 0 && o_cnt[t] > 0) wait(&bar.o_empty[t], (o_cnt[t] - 1) & 1);
        tc_fence_after();
        if (!ok) return;
        const int s = (base_iter + j) % kStages;
        const int valid = it.kv_len - j * kBN;     // keys of this tile inside the request
        if (valid < kBN && zeroed < j) {
          // zero V rows [valid, 128): whole 128-byte rows, so the swizzle is irrelevant
          uint4 *v = reinterpret_cast<uint4 *>(sV(s));
          for (int i = max(valid, 0) * 8 + lane; i < kBN * 8; i += 32) v[i] = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();
          zeroed = j;
        }
        __syncwarp();
        if (lane == 0) {
          const uint64_t dv = umma_desc_sw128(smem_u32(sV(s)), kTileBytes, 1024);
          const uint32_t tP = tmem + t * kSlotCols + kColP, tO = tmem + t * kSlotCols + kColO;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            umma_ts(tO, tP + 8 * kk, dv + (2048 >> 4) * kk, kIdescPV, (j > 0) || (kk > 0));
          if (j == it.ntiles[t] - 1) umma_commit(&bar.o_full[t]);
        }
        __syncwarp();
        if (j == it.ntiles[t] - 1) ++o_cnt[t];
      };
      for (int t = 0; t < 2; ++t)
        if (it.ntiles[t] > 0) issue_qk(t, 0);
      for (int j = 0; ok && j < it.n; ++j) {
        for (int t = 0; t < 2; ++t) {
          if (j < it.ntiles[t]) issue_pv(t, j);
          if (t == 1) {
            // every MMA reading this stage has been issued
            if (lane == 0 && ok) umma_commit(&bar.kv_empty[(base_iter + j) % kStages]);
            __syncwarp();
          }
          if (j + 1 < it.ntiles[t]) issue_qk(t, j + 1);
        }
      }
      if (lane == 0 && ok) umma_commit(&bar.q_empty);   // all QK of the item issued
      __syncwarp();
      kv_iter = base_iter + it.n;
      ++items_done;
    }
    if (!ok) fail();
  } else {
    // ------------------------------------------------------------- softmax
    const int t = warp >> 2;                            // tile A (0) or B (1)
    const int r = threadIdx.x & (kBM - 1);              // row = TMEM lane
    const uint32_t trow = tmem + t * kSlotCols + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.f;
    // Masked scores are replaced (by index, so NaN keys cannot leak) with the
    // raw value whose scaled logit is -inf.
    const uint32_t masked_raw = pos_scale ? 0xff800000u : 0x7f800000u;
    uint32_t s_cnt = 0, o_cnt = 0, items_done = 0;
    uint32_t x[3][32];
    for (int idx = blockIdx.x; idx < num_items; idx += gridDim.x) {
      const Item it = make_item<kPaged>(p, idx);
      if (it.bad) {
        // Poison every row of the request inside the buffers (pair 0 only).
        if (it.pair == 0 && t == 0 && it.q_start >= 0 && it.q_start < p.total_q) {
          const int stop = min(max(it.q_start + it.q_len, it.q_start), p.total_q);
          for (int row = it.q_start + r; row < stop; row += kBM) {
            const uint4 nan4 = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
            uint4 *dst = reinterpret_cast<uint4 *>(
                p.out + (static_cast<size_t>(row) * p.num_qo_heads + it.head) * kHeadDim);
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = nan4;
            if (p.lse) p.lse[static_cast<size_t>(row) * p.num_qo_heads + it.head] = NAN;
          }
        }
        continue;
      }
      if (it.empty) continue;
      const int *bad_flag = &bar.bad[items_done % kFlagRing];
      ++items_done;
      const int ntiles = it.ntiles[t];
      if (ntiles == 0) continue;                        // tile B past the request's end
      const int i = it.i0 + t * kBM + r;                // query row within the request
      const int limit = min(it.kv_len - it.q_len + i + 1, it.kv_len);   // keys [0, limit)
      // m is the reference max (base 2) that P and the tensor-memory O are
      // relative to.  It starts at the sink (so the sink's term in d is 1)
      // and only moves when a row max exceeds it by more than kRescaleLog2,
      // at which point O and d are rescaled; out = O/d and lse = m + log2(d)
      // are exact for any reference, and P stays below 2^kRescaleLog2.
      float m = p.sinks[it.head] * kLog2e;
      float d = 1.f;
      bool ok = true;
      for (int j = 0; j < ntiles; ++j) {
        // warp-uniform: the tcgen05.ld/st below are .sync.aligned
        if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_full[t], s_cnt & 1))) { ok = false; break; }
        ++s_cnt;
        tc_fence_after();
        // Scores for keys 32c..32c+31 of the tile are chunk c.  Registers hold
        // three chunks: A = c0, B = c1, C = c2 then c3 for the row max; in the
        // exp pass C (= c3) goes first, then c2 is reloaded into C.
        const int k0 = j * kBN;
        const bool edge = __any_sync(0xffffffffu, k0 + kBN > limit);  // causal-edge tile
        auto mask = [&](uint32_t (&v)[32], int c) {
          if (edge) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (k0 + 32 * c + e >= limit) v[e] = masked_raw;
          }
        };
        auto chunk_max = [&](const uint32_t (&v)[32], float acc) {
          if (pos_scale) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) acc = fmax3(acc, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) acc = fmaxf(acc, __uint_as_float(v[e]) * sl2);
          }
          return acc;
        };
        tmem_ld32(trow + kColS, x[0]);
        tmem_ld32(trow + kColS + 32, x[1]);
        tmem_ld32(trow + kColS + 64, x[2]);
        tmem_ld_wait32(x[0]);
        reg_tie32(x[1]);
        reg_tie32(x[2]);
        mask(x[0], 0);
        mask(x[1], 1);
        mask(x[2], 2);
        float mx0 = chunk_max(x[0], -INFINITY), mx1 = chunk_max(x[1], -INFINITY);
        float mx2 = chunk_max(x[2], -INFINITY);
        tmem_ld32(trow + kColS + 96, x[2]);
        tmem_ld_wait32(x[2]);
        mask(x[2], 3);
        mx2 = chunk_max(x[2], mx2);
        float mx = fmax3(mx0, mx1, mx2);
        if (pos_scale) mx *= sl2;
        const float m_new = fmaxf(m, mx);
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {                        // O holds nothing of this item: re-base d
          if (m_new != -INFINITY) {
            d *= ex2(m - m_new);
            m = m_new;
          }
        } else if (m_new > m + kRescaleLog2) {
          alpha = ex2(m - m_new);
          d *= alpha;
          m = m_new;
          rescale = true;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        const uint64_t scale2 = f2_pack(sl2, sl2), negmu2 = f2_pack(-mu, -mu);
        uint64_t acc = 0, acc2 = 0;                       // (+0.f, +0.f)
        pack_chunk(x[2], scale2, negmu2, acc);            // chunk 3, pairs packed in place
        tmem_st16(trow + kColP + 48, *reinterpret_cast<uint32_t(*)[16]>(&x[2][0]));
        tmem_st_wait();                                   // before x[2] is overwritten
        tmem_ld32(trow + kColS + 64, x[2]);               // chunk 2 again
        pack_chunk(x[0], scale2, negmu2, acc2);
        tmem_st16(trow + kColP, *reinterpret_cast<uint32_t(*)[16]>(&x[0][0]));
        pack_chunk(x[1], scale2, negmu2, acc);
        tmem_st16(trow + kColP + 16, *reinterpret_cast<uint32_t(*)[16]>(&x[1][0]));
        tmem_ld_wait32(x[2]);
        mask(x[2], 2);
        pack_chunk(x[2], scale2, negmu2, acc2);
        tmem_st16(trow + kColP + 32, *reinterpret_cast<uint32_t(*)[16]>(&x[2][0]));
        float s0, s1;
        f2_unpack(f2_add(acc, acc2), s0, s1);
        d += s0 + s1;
        tmem_st_wait();
        if (__any_sync(0xffffffffu, rescale)) {
          // rare: scale this row's O (finished by the previous PV; the next
          // PV is issued only after p_full below)
#pragma unroll
          for (int h = 0; h < 2; ++h) tmem_ld32(trow + kColO + 32 * h, x[h]);
          tmem_ld_wait32(x[0]);
          reg_tie32(x[1]);
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 32; ++e) x[h][e] = __float_as_uint(__uint_as_float(x[h][e]) * alpha);
          tmem_st16(trow + kColO, *reinterpret_cast<uint32_t(*)[16]>(&x[0][0]));
          tmem_st16(trow + kColO + 16, *reinterpret_cast<uint32_t(*)[16]>(&x[0][16]));
          tmem_st16(trow + kColO + 32, *reinterpret_cast<uint32_t(*)[16]>(&x[1][0]));
          tmem_st16(trow + kColO + 48, *reinterpret_cast<uint32_t(*)[16]>(&x[1][16]));
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&bar.p_full[t]);
      }
      bool failed = false;
      if (ok && __all_sync(0xffffffffu, mbar_wait(&bar.o_full[t], o_cnt & 1))) {
        tc_fence_after();
        tmem_ld32(trow + kColO, x[0]);
        tmem_ld32(trow + kColO + 32, x[1]);
        tmem_ld_wait32(x[0]);
        reg_tie32(x[1]);
        // this item's skipped-page flag is final once its last PV completed
        // (o_full), and is read before o_empty lets the producer move on
        failed = *static_cast<const volatile int *>(bad_flag) != 0;
        tc_fence_before();
        mbar_arrive(&bar.o_empty[t]);                 // the next item may overwrite O
      } else {
        ok = false;
      }
      ++o_cnt;
      if (!ok) {
        fail();
        break;
      }
      const int rows = it.rows[t];
      if (r < rows) {
        const size_t row = static_cast<size_t>(it.q_start + i) * p.num_qo_heads + it.head;
        const float inv = d > 0.f ? 1.f / d : 0.f;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kHeadDim);
#pragma unroll
        for (int c = 0; c < kHeadDim / 8; ++c) {
          uint4 w;
          if (failed) {
            w = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);
          } else {
            auto o = [&](int e) {
              return __uint_as_float(x[(8 * c + e) >> 5][(8 * c + e) & 31]) * inv;
            };
            w.x = pack_bf16(o(0), o(1));
            w.y = pack_bf16(o(2), o(3));
            w.z = pack_bf16(o(4), o(5));
            w.w = pack_bf16(o(6), o(7));
          }
          dst[c] = w;
        }
        if (p.lse) p.lse[row] = failed ? NAN : (d > 0.f ? (m + lg2(d)) * kLn2 : -INFINITY);
      }
    }
  }
  // teardown: every role is done with tensor memory.  After a timed-out wait,
  // let whatever tensor-core work is still queued drain (bounded) first.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    if (*abort_flag) {
      if (lane == 0) umma_commit(&bar.drain);
      __syncwarp();
      mbar_wait(&bar.drain, 0);
    }
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p, cudaStream_t stream) {
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  const unsigned long long items =
      static_cast<unsigned long long>(p.num_q_tiles) * p.num_seqs * p.num_qo_heads;
  if (items == 0) return cudaSuccess;
  if (items > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const unsigned grid = static_cast<unsigned>(std::min<unsigned long long>(items, sms));
  if (p.paged) {
    err = cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (err != cudaSuccess) return err;
    prefill_kernel<true><<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
  } else {
    err = cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemBytes);
    if (err != cudaSuccess) return err;
    prefill_kernel<false><<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
  }
  return cudaGetLastError();
}

}  // namespace sa
