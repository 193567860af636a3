// Causal prefill (ragged, or appended to a paged KV prefix) with learned
// sinks on the 5th-generation tensor cores (tcgen05 + tensor memory).
//
// Operation: "GPT-OSS on day 0" (Perplexity blog), section "Kernels for
// GPT-OSS / Sink Attention" -- each head's running max starts at its sink and
// its running sum at 1, so the sink joins the softmax denominator without a
// value row.  Query i of a request with kv_len keys and q_len new queries
// sees keys j <= kv_len - q_len + i (for plain prefill kv_len = q_len).
//
// One CTA = one 128-row query tile of one query head (6 warps):
//   warp 4      loads Q once and K tiles of 128 keys into a 3-stage ring
//               (contiguous: one 16 KB box per tile; paged: eight 2 KB page
//               boxes), 128-byte swizzle; one thread issues S = Q K^T
//               (tcgen05.mma, A and B from shared memory, M=128 N=128 K=16
//               x4) into tensor memory as soon as the softmax has read the
//               previous S, so S of tile j+1 is computed during the softmax
//               of tile j.
//   warp 5      loads V tiles into a 2-stage ring; one thread issues
//               O += P V (A = P from tensor memory, B = V from shared memory
//               in MN-major layout, M=128 N=64 K=16 x8), which runs during
//               the softmax of the next tile.  An issuing thread stalls while
//               the tensor pipe is busy, so QK^T and P V have a thread each
//               and S never waits behind P V.
//   warps 0..3  softmax, one thread per query row (= tensor-memory lane):
//               S from tensor memory (read once per tile), online softmax in
//               base 2 started at the sink, P (bf16) back into tensor memory
//               once the previous P V has finished reading it; O
//               accumulates in tensor memory across KV tiles and is rescaled
//               only when a row max grows by more than 2^8.
// Tensor memory per CTA: S 128 columns, P 64, O 64 = 256, so two CTAs share
// an SM and their MMA and softmax phases interleave.  Heavier query tiles
// (later ones, which see more keys) are launched first.
// V rows past a request's last key are zeroed in shared memory before the PV
// MMA (0 * NaN would poison whole rows); score columns past a row's causal
// limit are masked by index.
//
// Verification (kVerify; "Accelerating Sonar through speculation", sections
// "Target-Draft", "MTP" and "EAGLE"): the query rows of one KV head of one
// request -- its q_len newest tokens x the group's heads, ordered (token,
// head) -- form the 128-row tile (Q by one 3-D box {64, group, 128/group}).
// Each softmax thread takes its row's token for the causal limit (or its
// tree bits for the draft keys) and its head for the sink; warps without
// rows stay out of the barrier counts.  Requests go heaviest first (ranked
// from kv_lens by every warp), and under a programmatic launch the ranking,
// the page-table reads and the shared / tensor memory set-up run before the
// wait for the previous kernel on the stream.

#include "kernels.cuh"
#include "ptx.cuh"

#include <cmath>

namespace sa {
namespace {

constexpr int kBM = 128;                       // query rows per CTA
constexpr int kBN = 128;                       // keys per KV tile
constexpr int kKStages = 3, kVStages = 2;   // K is needed a softmax earlier than V
constexpr int kTileBytes = kBN * kHeadDim * 2;    // 16 KB
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColO = 192;
constexpr float kRescaleLog2 = 8.f;     // lazy O rescale threshold (P < 256)

constexpr int kOffQ = 0;
constexpr int kOffK = kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBars = kOffV + kVStages * kTileBytes;
constexpr int kSmemBytes = kOffBars + 256 + 1024;           // barriers + alignment slack

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKStages];
  uint64_t k_empty[kKStages];
  uint64_t v_full[kVStages];
  uint64_t v_empty[kVStages];
  uint64_t s_full;     // S of the current tile is in tensor memory
  uint64_t s_free;     // the softmax has read S (the next QK^T may overwrite it)
  uint64_t p_full;     // P of the current tile is in tensor memory
  uint64_t pv_done;    // the P V of the previous tile has finished (P may be rewritten)
  uint64_t o_final;
  uint32_t tmem_base;
  int bad;
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

// Request of dispatch slot `slot` with the requests heaviest first: 8 size
// classes of ceil(kv_len / 16) pages (largest first), request order within a
// class.  Every warp derives the same order from kv_lens on its own (no block
// barrier; the class by one float multiply, the class counts of 32 requests
// at a time by two warp reductions of packed 6-bit fields, the request by one
// ballot), so the last wave holds the short requests.  Returns -1 past the
// last request.
__device__ int request_by_size(const PrefillParams &p, int slot) {
  constexpr int kClasses = 8, kLow = 4;         // classes 0..3 in the first word, 4..7 in the second
  constexpr int kHeld = 8;                      // groups of 32 classes kept in registers
  const int lane = threadIdx.x & 31;
  const int groups = cdiv(p.num_seqs, 32);
  const float per_page =
      static_cast<float>(kClasses) / static_cast<float>(max(1, cdiv(p.max_kv_len, kPageSize)) + 1);
  auto class_of = [&](int b) {
    if (b >= p.num_seqs) return -1;
    const int pages = cdiv(max(__ldg(p.kv_lens + b), 0), kPageSize);
    return min(kClasses - 1, __float2int_rz(static_cast<float>(pages) * per_page));
  };
  int held[kHeld];
  int total[kClasses];
#pragma unroll
  for (int k = 0; k < kClasses; ++k) total[k] = 0;
  for (int u = 0; u < groups; ++u) {
    const int c = class_of(u * 32 + lane);
#pragma unroll
    for (int v = 0; v < kHeld; ++v)
      if (v == u) held[v] = c;
    const unsigned lo = __reduce_add_sync(0xffffffffu, c >= 0 && c < kLow ? 1u << (6 * c) : 0u);
    const unsigned hi = __reduce_add_sync(0xffffffffu, c >= kLow ? 1u << (6 * (c - kLow)) : 0u);
#pragma unroll
    for (int k = 0; k < kClasses; ++k)
      total[k] += static_cast<int>(((k < kLow ? lo : hi) >> (6 * (k % kLow))) & 63u);
  }
  int rank = slot, cls = -1;
#pragma unroll
  for (int k = kClasses - 1; k >= 0; --k) {
    if (cls < 0) {
      if (rank < total[k]) cls = k;
      else rank -= total[k];
    }
  }
  if (cls < 0) return -1;
  for (int u = 0; u < groups; ++u) {
    int c = -1;
#pragma unroll
    for (int v = 0; v < kHeld; ++v)
      if (v == u) c = held[v];
    if (u >= kHeld) c = class_of(u * 32 + lane);
    const unsigned hit = __ballot_sync(0xffffffffu, c == cls);
    const int n = __popc(hit);
    if (rank < n) return u * 32 + static_cast<int>(__fns(hit, 0, rank + 1));
    rank -= n;
  }
  return -1;                                    // not reached: the classes cover every request
}

// One 128-key tile of the online softmax for this thread's query row (one
// row per thread = its tensor-memory lane): NC chunks of 32 scores from S
// column c0 on (the whole tile: NC = 4, c0 = 0; a key half: NC = 2, c0 = 0 or
// 64), masks, the reference max m (moved only by more than kRescaleLog2),
// P = 2^(s scale - m) in bf16 into tensor memory once the previous P V has
// read it, d updated, O rescaled when m moved.  Returns false when a wait
// timed out.
template <int NC>
__device__ __forceinline__ bool softmax_tile(Bars &bar, uint32_t trow, int j, int c0, int limit,
                                             bool tree, int draft0, uint64_t vis, float sl2,
                                             bool pos_scale, uint32_t masked_raw, float &m,
                                             float &d, uint32_t (&x)[4][32]) {
    // warp-uniform: the tcgen05.ld/st below are .sync.aligned
    if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_full, j & 1))) return false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < NC; ++c) tmem_ld32(trow + kColS + c0 + 32 * c, x[c]);
    tmem_ld_wait32(x[0]);
#pragma unroll
    for (int c = 1; c < NC; ++c) reg_tie32(x[c]);
    tc_fence_before();
    mbar_arrive(&bar.s_free);
    const int k0 = j * kBN + c0;                 // first key of this thread's columns
    if (__any_sync(0xffffffffu, k0 + 32 * NC > limit)) {   // only tiles on the causal edge
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (k0 + 32 * c + e >= limit) x[c][e] = masked_raw;
    }
    if (tree && __any_sync(0xffffffffu, k0 + 32 * NC > draft0)) {   // tiles holding draft keys
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int u = k0 + 32 * c + e - draft0;
          if (u >= 0 && u < 64 && !((vis >> u) & 1)) x[c][e] = masked_raw;
        }
    }
    float mx;
    if (pos_scale) {
      float mc[4];                          // independent chains
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        mc[c] = __uint_as_float(x[c][0]);
#pragma unroll
        for (int e = 1; e < 31; e += 2)
          mc[c] = fmax3(mc[c], __uint_as_float(x[c][e]), __uint_as_float(x[c][e + 1]));
        mc[c] = fmaxf(mc[c], __uint_as_float(x[c][31]));
      }
      mx = (NC == 4 ? fmax3(mc[0], mc[1], fmaxf(mc[2], mc[3])) : fmaxf(mc[0], mc[1])) * sl2;
    } else {
      mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(x[c][e]) * sl2);
    }
    const float m_new = fmaxf(m, mx);
    float alpha = 1.f;
    bool rescale = false;
    if (j == 0) {                        // O holds nothing yet: just re-base d
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
    uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      acc[c] = 0;                                   // (+0.f, +0.f)
      pack_chunk(x[c], scale2, negmu2, acc[c]);     // pairs packed in place
    }
    float s0, s1;
    f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), s0, s1);
    d += s0 + s1;
    // the previous tile's P V reads P and accumulates O: wait for it
    if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(&bar.pv_done, (j - 1) & 1))) return false;
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < NC; ++c)
      tmem_st16(trow + kColP + c0 / 2 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&x[c][0]));
    if (NC == 2 && j == 0) {
      // a half-tile row: the other half's P columns hold zeros for good
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      tmem_st16(trow + kColP + (32 - c0 / 2), z);
      tmem_st16(trow + kColP + (32 - c0 / 2) + 16, z);
    }
    tmem_st_wait();
    if (__any_sync(0xffffffffu, rescale)) {
      // rare: scale this row's O (the previous P V has finished, the next
      // one is issued only after p_full below)
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
    mbar_arrive(&bar.p_full);
  return true;
}

template <bool kPaged, bool kVerify, bool kHalf = false>
__global__ void __launch_bounds__(kThreads, 2)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  static_assert(kPaged || !kVerify, "verification reads the paged cache");
  static_assert(kVerify || !kHalf, "key halves are a verification tile");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4 nan4 = make_uint4(0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u, 0x7fc07fc0u);

  // ---- work item and request geometry (uniform over the CTA).  Prefill: a
  // 128-row query tile of one head.  Verification: the query rows of one KV
  // head of one request, ordered (token, head in group), 128 / group tokens
  // per tile; every request has q_len tokens, the last q_len of its keys.
  int seq, kvh, head = 0, qt, q_start, q_len, kv_len, k_start = 0;
  if constexpr (kVerify) {
    // blockIdx: request slot (heaviest first), then KV head, then query tile
    const int per_req = p.num_kv_heads * p.num_q_tiles;
    const int rem = static_cast<int>(blockIdx.x % per_req);
    qt = rem % p.num_q_tiles;
    kvh = rem / p.num_q_tiles;
    seq = request_by_size(p, static_cast<int>(blockIdx.x / per_req));
    if (seq < 0) return;
    q_len = p.max_q_len;
    q_start = seq * q_len;
    kv_len = p.kv_lens[seq];
  } else {
    const int per_tile = p.num_seqs * p.num_qo_heads;
    qt = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x / per_tile);
    const int rem = static_cast<int>(blockIdx.x % per_tile);
    head = rem % p.num_qo_heads;
    seq = rem / p.num_qo_heads;
    kvh = head / p.group;
    q_start = p.cu_seqlens_q[seq];
    q_len = p.cu_seqlens_q[seq + 1] - q_start;
    if constexpr (kPaged) {
      kv_len = p.kv_lens[seq];
    } else {
      k_start = p.cu_seqlens_k[seq];
      kv_len = p.cu_seqlens_k[seq + 1] - k_start;
    }
  }
  const int q_end = q_start + q_len;
  bool bad = q_start < 0 || q_len < 0 || q_end > p.total_q || q_len > p.max_q_len ||
             kv_len < q_len || kv_len > p.max_kv_len;
  if constexpr (kPaged) {
    bad = bad || cdiv(kv_len, kPageSize) > p.max_pages_per_seq;
  } else {
    bad = bad || k_start < 0 || k_start + kv_len > p.total_k;
  }
  if (bad) {
    // Poison every row this request owns that lies inside the buffers (once:
    // by the CTA of its first query tile).
    if (qt != 0 || q_start < 0 || q_start >= p.total_q) return;
    if constexpr (kVerify) grid_dependency_wait();
    const int stop = min(max(q_end, q_start), p.total_q);
    const int heads_here = kVerify ? p.group : 1;
    for (int idx = threadIdx.x; idx < (stop - q_start) * heads_here; idx += kThreads) {
      const int t = q_start + idx / heads_here;
      const int h = kVerify ? kvh * p.group + idx % heads_here : head;
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + (static_cast<size_t>(t) * p.num_qo_heads + h) * kHeadDim);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = nan4;
      if (p.lse) p.lse[static_cast<size_t>(t) * p.num_qo_heads + h] = NAN;
    }
    return;
  }
  // first query row (token) of the tile, rows (tokens) in it, query rows used
  const int tok_per_tile = kVerify ? kBM / p.group : kBM;
  const int i0 = qt * tok_per_tile;
  if (i0 >= q_len) return;
  const int rows_tok = min(tok_per_tile, q_len - i0);
  const int rows = kVerify ? rows_tok * p.group : rows_tok;
  const int shift = kv_len - q_len;                        // bottom-right causal offset
  const int key_end = shift + i0 + rows_tok;               // keys needed, exclusive (<= kv_len)
  const int n_tiles = cdiv(key_end, kBN);
  const int npages = cdiv(kv_len, kPageSize);
  // Verification with up to 64 query rows (kHalf) splits every key tile in two:
  // the rows are replicated into the next tensor-memory lanes (half_rows
  // further on), the warps on the original rows take keys 0..63 of each
  // tile and those on the replica keys 64..127, each half with its own
  // online softmax (the sink counted in the first half only); the halves
  // merge by log-sum-exp at the end.  Each softmax warp then does half the
  // exponentials of a tile (8-node draft tree, 64 rows: 4797 -> 5140 GB/s;
  // 4 draft tokens, 32 rows: 5604 -> 5670 GB/s).
  const int half_rows = 32 * cdiv(rows, 32);
  constexpr bool half_keys = kHalf;           // chosen by the host from q_len * group
  // softmax threads with a query row (verification tiles may be partly empty)
  const int live_threads =
      kVerify ? (half_keys ? 2 * half_rows : min(kBM, 32 * cdiv(rows, 32))) : kBM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  Bars &bar = *reinterpret_cast<Bars *>(smem + kOffBars);
  uint8_t *sQ = smem + kOffQ;
  auto sK = [&](int s) { return smem + kOffK + s * kTileBytes; };
  auto sV = [&](int s) { return smem + kOffV + s * kTileBytes; };

  if (warp == kMmaWarp) {
    tmem_alloc(&bar.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  // Up to here only the metadata was read (cu_seqlens, kv_lens; the page
  // table below); q, the caches and the outputs may belong to the previous
  // kernel on the stream (verification launches programmatically).
  if (kVerify && warp != kProducerWarp) {
    grid_dependency_wait();
    launch_dependents();
  }
  const int32_t *table = kPaged ? p.page_table + static_cast<size_t>(seq) * p.max_pages_per_seq : nullptr;
  // paged: the page id of this lane's 16 keys of tile j (lanes 0..7), else -1
  auto page_of = [&](int j) -> int {
    const int pg = j * (kBN / kPageSize) + lane;
    return kPaged && lane < kBN / kPageSize && pg < npages ? table[pg] : -1;
  };
  // K (t = 0) or V (t = 1) of tile j into its ring slot, once the slot is
  // free; paged tiles use the page ids `pid` (from page_of, read ahead of time
  // by the issuing warps so the table's latency stays off their loop)
  auto load_with = [&](int j, int t, int pid) -> bool {
    const int ns = t == 0 ? kKStages : kVStages;
    const int s = j % ns;
    uint64_t *full = t == 0 ? &bar.k_full[s] : &bar.v_full[s];
    uint64_t *empty = t == 0 ? &bar.k_empty[s] : &bar.v_empty[s];
    uint8_t *dst = t == 0 ? sK(s) : sV(s);
    const CUtensorMap *map = t == 0 ? &kmap : &vmap;
    if (j >= ns && !__all_sync(0xffffffffu, mbar_wait(empty, ((j / ns) + 1) & 1)))
      return false;
    if constexpr (kPaged) {
      // lanes 0..7 each own one 16-token page of the 128-key tile
      const int pg = j * (kBN / kPageSize) + lane;
      const bool ok = pid >= 0 && pid < p.num_pages;
      if (t == 0 && lane < kBN / kPageSize && pg < npages && !ok) atomicOr(&bar.bad, 1);
      const unsigned mask = __ballot_sync(0xffffffffu, ok);
      if (lane == 0) mbar_arrive_expect_tx(full, __popc(mask) * kPageSize * kHeadDim * 2);
      __syncwarp();
      if (ok) {
        if (kVerify && p.num_q_tiles == 1)    // the only reader of these pages
          tma_load_3d_hint(dst + lane * kPageSize * kHeadDim * 2, map, full, 0, kvh * kPageSize,
                           pid, l2_policy_evict_first());
        else
          tma_load_3d(dst + lane * kPageSize * kHeadDim * 2, map, full, 0, kvh * kPageSize, pid);
      }
    } else {
      if (lane == 0) {
        mbar_arrive_expect_tx(full, kTileBytes);
        tma_load_3d(dst, map, full, 0, kvh, k_start + j * kBN);
      }
    }
    __syncwarp();
    return true;
  };
  auto load = [&](int j, int t) -> bool { return load_with(j, t, page_of(j)); };

  if (warp == kProducerWarp) {
    // barriers, then the loads the first S needs (Q and the first K tiles),
    // before the CTA-wide barrier: their latency runs under the tensor-memory
    // allocation and the barrier
    if (lane == 0) {
      mbar_init(&bar.q_full, 1);
      for (int s = 0; s < kKStages; ++s) {
        mbar_init(&bar.k_full[s], 1);
        mbar_init(&bar.k_empty[s], 1);
      }
      for (int s = 0; s < kVStages; ++s) {
        mbar_init(&bar.v_full[s], 1);
        mbar_init(&bar.v_empty[s], 1);
      }
      mbar_init(&bar.s_full, 1);
      mbar_init(&bar.s_free, live_threads);
      mbar_init(&bar.p_full, live_threads);
      mbar_init(&bar.pv_done, 1);
      mbar_init(&bar.o_final, 1);
      bar.bad = 0;
      fence_mbar_init();
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    // verification: the first K tiles' page ids before waiting for the
    // previous kernel (prefill is launched plainly and reads them on demand)
    int first_ids[kKStages];
#pragma unroll
    for (int j = 0; j < kKStages; ++j) first_ids[j] = kVerify ? page_of(j) : 0;
    if constexpr (kVerify) {
      grid_dependency_wait();
      launch_dependents();
    }
    if (lane == 0) {
      mbar_arrive_expect_tx(&bar.q_full, kBM * kHeadDim * 2);
      if constexpr (kVerify)   // box {64, group, 128 / group}: rows (token, head)
        tma_load_3d(smem + kOffQ, &qmap, &bar.q_full, 0, kvh * p.group, q_start + i0);
      else
        tma_load_3d(smem + kOffQ, &qmap, &bar.q_full, 0, head, q_start + i0);
    }
    __syncwarp();
    for (int j = 0; j < min(n_tiles, kKStages); ++j) {              // fresh slots: no waits
      int pid = 0;
      if constexpr (kVerify) {
#pragma unroll
        for (int u = 0; u < kKStages; ++u)
          if (u == j) pid = first_ids[u];
      } else {
        pid = page_of(j);
      }
      load_with(j, 0, pid);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar.tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------- loads and QK^T (one thread)
    const uint32_t tS = tmem + kColS;
    const uint64_t dq = umma_desc_sw128(smem_u32(sQ), 16, 1024);
    auto issue_qk = [&](int j) -> bool {
      const int s = j % kKStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.k_full[s], (j / kKStages) & 1))) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t dk = umma_desc_sw128(smem_u32(sK(s)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          umma_ss(tS, dq + 2 * kk, dk + 2 * kk, kIdescQK, kk > 0);   // +32 bytes per k-step
        umma_commit(&bar.s_full);
        umma_commit(&bar.k_empty[s]);
      }
      __syncwarp();
      return true;
    };
    bool ok = true;                 // Q and the first K tiles are on their way
    int pk = page_of(kKStages);     // ids of the next K tile to load
    ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar.q_full, 0));
    if (ok && half_keys) {
      // replica of the query rows at half_rows (a multiple of 8 rows, so the
      // 128-byte swizzle pattern of every row is unchanged)
      const uint4 *src = reinterpret_cast<const uint4 *>(sQ);
      uint4 *dst = reinterpret_cast<uint4 *>(sQ + half_rows * kHeadDim * 2);
      for (int e = lane; e < half_rows * (kHeadDim * 2 / 16); e += 32) dst[e] = src[e];
      fence_proxy_async_smem();
      __syncwarp();
    }
    ok = ok && issue_qk(0);
    for (int j = 0; ok && j + 1 < n_tiles; ++j) {
      // S of tile j has been read: compute S of tile j+1 during this softmax
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.s_free, j & 1))) { ok = false; break; }
      tc_fence_after();
      ok = issue_qk(j + 1);
      if (ok && j + kKStages < n_tiles) {             // K slot freed by QK^T of tile j
        ok = load_with(j + kKStages, 0, pk);
        pk = page_of(j + kKStages + 1);
      }
    }
    if (!ok && lane == 0) atomicOr(&bar.bad, 1);
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------- P V (one thread)
    const uint32_t tP = tmem + kColP, tO = tmem + kColO;
    bool ok = true;
    for (int j = 0; ok && j < min(n_tiles, kVStages); ++j) ok = load(j, 1);
    int pv_ids = page_of(kVStages);    // ids of the next V tile to load
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int s = j % kVStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&bar.p_full, j & 1)) ||
          !__all_sync(0xffffffffu, mbar_wait(&bar.v_full[s], (j / kVStages) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int valid = kv_len - j * kBN;        // keys of this tile inside the request
      if (valid < kBN) {
        // zero V rows [valid, 128): whole 128-byte rows, so the swizzle is irrelevant
        uint4 *v = reinterpret_cast<uint4 *>(sV(s));
        for (int idx = max(valid, 0) * 8 + lane; idx < kBN * 8; idx += 32) v[idx] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) {
        const uint64_t dv = umma_desc_sw128(smem_u32(sV(s)), kTileBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          umma_ts(tO, tP + 8 * kk, dv + (2048 >> 4) * kk, kIdescPV, (j > 0) || (kk > 0));  // 16 keys = 2 KB
        umma_commit(&bar.v_empty[s]);
        umma_commit(&bar.pv_done);
      }
      __syncwarp();
      // V of tile j+2 into the slot this P V reads, once it has finished
      if (j + kVStages < n_tiles) {
        if (!load_with(j + kVStages, 1, pv_ids)) { ok = false; break; }
        pv_ids = page_of(j + kVStages + 1);
      }
    }
    if (!ok && lane == 0) atomicOr(&bar.bad, 1);
    if (lane == 0) umma_commit(&bar.o_final);
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;                          // row = TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    // the query row this thread computes (a replica lane: the same row as
    // lane r - half_rows) and the first S column of its keys
    const int lr = half_keys ? r % half_rows : r;
    const int c0 = half_keys && r >= half_rows && r < 2 * half_rows ? kBN / 2 : 0;
    // token (within the request) and head of this thread's query row
    const int i = kVerify ? i0 + lr / p.group : i0 + lr;
    const int row_head = kVerify ? kvh * p.group + lr % p.group : head;
    const bool tree = kVerify && p.tree_mask != nullptr;
    // keys [0, limit) are candidates (causal); with a draft tree, key
    // draft0 + u is visible only if bit u of the row's mask is set
    const int limit = tree ? kv_len : min(shift + i + 1, kv_len);
    const int draft0 = shift;
    uint64_t vis = 0;
    if constexpr (kVerify) {
      if (tree && lr < rows) vis = p.tree_mask[static_cast<size_t>(seq) * q_len + i];
    }
    const float sl2 = p.scale_log2;
    const bool pos_scale = sl2 >= 0.f;
    // Masked scores are replaced (by index, so NaN keys cannot leak) with the
    // raw value whose scaled logit is -inf.
    const uint32_t masked_raw = pos_scale ? 0xff800000u : 0x7f800000u;
    // m is the reference max (base 2) that P and the tensor-memory O are
    // relative to.  It starts at the sink (so the sink's term in d is 1) and
    // only moves when a row max exceeds it by more than kRescaleLog2, at which
    // point O and d are rescaled; out = O/d and lse = m + log2(d) are exact
    // for any reference, and P stays below 2^kRescaleLog2.
    float m = c0 == 0 ? p.sinks[row_head] * kLog2e : -INFINITY;   // the sink: first half only
    float d = c0 == 0 ? 1.f : 0.f;
    bool ok = true;
    uint32_t x[4][32];

    const bool live = warp * 32 < live_threads;         // warp-uniform
    for (int j = 0; live && j < n_tiles; ++j) {
      const bool step = softmax_tile<kHalf ? 2 : 4>(bar, trow, j, c0, limit, tree, draft0, vis, sl2,
                                                    pos_scale, masked_raw, m, d, x);
      if (!step) {
        ok = false;
        break;
      }
    }
    if (!live) {
      // no query rows in this warp: nothing to read
    } else if (__all_sync(0xffffffffu, mbar_wait(&bar.o_final, 0))) {
      tc_fence_after();
      if (ok && n_tiles > 0) {
        tmem_ld32(trow + kColO, x[0]);
        tmem_ld32(trow + kColO + 32, x[1]);
        tmem_ld_wait32(x[0]);
        reg_tie32(x[1]);
      }
    } else {
      ok = false;
    }
    if (!ok) atomicOr(&bar.bad, 1);
    // second key half: (O, m, d) to shared memory for the first half's
    // thread (the K ring is idle: every QK^T has completed)
    float *half2 = reinterpret_cast<float *>(smem + kOffK);
    constexpr int kHalfStride = kHeadDim + 4;
    if (half_keys && c0 != 0 && r < 2 * half_rows && lr < rows) {   // replica lanes only
      float *h2 = half2 + lr * kHalfStride;
#pragma unroll
      for (int c = 0; c < kHeadDim; ++c) h2[c] = __uint_as_float(x[c >> 5][c & 31]);
      h2[kHeadDim] = m;
      h2[kHeadDim + 1] = d;
    }

    // Outputs are written after the CTA-wide barrier below.  Tensor memory is
    // read no more: the P V warp frees it meanwhile.
    tc_fence_before();
    __syncthreads();
    const bool failed = bar.bad != 0;
    if (half_keys && c0 == 0 && r < rows) {
      // merge the two key halves by log-sum-exp (either may have seen no key)
      const float *h2 = half2 + r * kHalfStride;
      const float m2 = h2[kHeadDim], d2 = h2[kHeadDim + 1];
      const float mm = fmaxf(m, m2);
      const float w1 = m == -INFINITY ? 0.f : ex2(m - mm);
      const float w2 = m2 == -INFINITY ? 0.f : ex2(m2 - mm);
#pragma unroll
      for (int c = 0; c < kHeadDim; ++c)
        x[c >> 5][c & 31] = __float_as_uint(__uint_as_float(x[c >> 5][c & 31]) * w1 + h2[c] * w2);
      d = d * w1 + d2 * w2;
      m = mm;
    }
    const float inv = d > 0.f ? 1.f / d : 0.f;
    auto packed = [&](int c) {           // 16-byte chunk c of this row (8 outputs)
      uint4 w;
      if (failed) return nan4;
      auto o = [&](int e) { return __uint_as_float(x[e >> 5][e & 31]) * inv; };
      w.x = pack_bf16(o(8 * c + 0), o(8 * c + 1));
      w.y = pack_bf16(o(8 * c + 2), o(8 * c + 3));
      w.z = pack_bf16(o(8 * c + 4), o(8 * c + 5));
      w.w = pack_bf16(o(8 * c + 6), o(8 * c + 7));
      return w;
    };
    const size_t row = static_cast<size_t>(q_start + i) * p.num_qo_heads + row_head;
    if (!kVerify && r - lane + 32 <= rows && !failed) {
      // Full 32-row slices of prefill / extend: each warp puts its rows in the
      // query buffer (free since the last QK^T completed) and reads them back
      // so that 8 lanes cover one row's 128 contiguous bytes: every store
      // writes 4 whole rows instead of a 16-byte piece of 32 rows 8 KB apart.
      uint4 *sw = reinterpret_cast<uint4 *>(sQ) + (r - lane) * 8;     // this warp's 32 rows
#pragma unroll
      for (int c = 0; c < kHeadDim / 8; ++c) sw[lane * 8 + (c ^ (lane & 7))] = packed(c);
      __syncwarp();
      const int cc = lane & 7;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int rr = 4 * k + (lane >> 3);                  // row within the warp's slice
        const size_t grow = static_cast<size_t>(q_start + i0 + (r - lane) + rr) * p.num_qo_heads + head;
        reinterpret_cast<uint4 *>(p.out + grow * kHeadDim)[cc] = sw[rr * 8 + (cc ^ (rr & 7))];
      }
    } else if (r < rows) {
      uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kHeadDim);
#pragma unroll
      for (int c = 0; c < kHeadDim / 8; ++c) dst[c] = packed(c);
    }
    if (r < rows && p.lse) p.lse[row] = failed ? NAN : (d > 0.f ? (m + lg2(d)) * kLn2 : -INFINITY);
    return;
  }
  tc_fence_before();
  __syncthreads();          // the softmax warps have read O: tensor memory is free
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

template <bool kPaged, bool kVerify, bool kHalf = false>
static cudaError_t launch_prefill_variant(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p, unsigned ctas,
                           cudaStream_t stream, bool programmatic) {
  cudaError_t err = set_smem_once<prefill_kernel<kPaged, kVerify, kHalf>>(kSmemBytes);
  if (err != cudaSuccess) return err;
  // verification follows the caller's launch mode; prefill launches plainly
  return launch_kernel(prefill_kernel<kPaged, kVerify, kHalf>, ctas, kThreads, kSmemBytes, stream,
                       kVerify && programmatic, qmap, kmap, vmap, p);
}

#ifndef SA_VERIFY_HALF_KEYS
#define SA_VERIFY_HALF_KEYS 1
#endif

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p, cudaStream_t stream,
                           bool programmatic) {
  static_assert(kSmemBytes <= 113 * 1024, "two CTAs per SM");
  const unsigned long long ctas = static_cast<unsigned long long>(p.num_q_tiles) * p.num_seqs *
                                  (p.verify ? p.num_kv_heads : p.num_qo_heads);
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  if (p.verify) {
    // one query tile per KV head when verifying (q_len * group <= 128 rows)
    const int rows = p.max_q_len * p.group;
    if (SA_VERIFY_HALF_KEYS && rows <= 64)
      return launch_prefill_variant<true, true, true>(qmap, kmap, vmap, p, static_cast<unsigned>(ctas), stream, programmatic);
    return launch_prefill_variant<true, true>(qmap, kmap, vmap, p, static_cast<unsigned>(ctas), stream, programmatic);
  }
  if (p.paged) return launch_prefill_variant<true, false>(qmap, kmap, vmap, p, static_cast<unsigned>(ctas), stream, false);
  return launch_prefill_variant<false, false>(qmap, kmap, vmap, p, static_cast<unsigned>(ctas), stream, false);
}

}  // namespace sa
