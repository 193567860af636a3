// Paged-KV decode with learned sinks: split-KV with an in-kernel log-sum-exp
// merge of the KV chunks.
//
// Operation: "GPT-OSS on day 0" (Perplexity blog), section "Kernels for
// GPT-OSS / Sink Attention" -- online softmax with the running max started at
// the head's sink (scale d = 1) in the first KV block only, other blocks
// started at -inf, blocks merged by log-sum-exp.
//
// Design (GB300, HBM-bound):
//  * One CTA = one (request, KV head, block of 8 or 16 query heads, KV
//    chunk): a GQA group above 8 takes two 8-head column blocks per CTA, so
//    every page is read once per 16 heads.  When
//    the plan has one chunk per request the requests are dispatched heaviest
//    first (by size class, computed from kv_lens in every CTA) so that the
//    last wave holds the short ones.  Its
//    NW warps take the chunk's 16-token pages round-robin, each warp running
//    its own STAGES-deep TMA pipeline: lane 0 issues two 3-D bulk tensor
//    copies per page (K and V tile, 2 KB each, 128-byte swizzle) onto the
//    stage's mbarrier.  No register staging, so many pages stay in flight.
//    Pages that only this CTA reads carry an evict-first L2 policy, so the
//    small tensors every launch re-reads (kv_lens, page table, q) and the
//    outputs stay in L2.
//  * The GQA group shares every K/V tile: S^T[16 tok x 8 heads] = K . Q^T and
//    O^T[64 x 8] += V^T . P^T, each 4 mma.sync.m16n8k16 (bf16 in, fp32 acc).
//    P^T goes from the score accumulator layout to the B-operand layout with
//    movmatrix.trans; K and V^T come from shared memory by ldmatrix(.trans),
//    bank-conflict free thanks to the swizzle.
//  * Online softmax in base 2: scores scaled by scale*log2(e), sink by log2(e).
//    Row max is reduced with 3 xor-shuffles per page; the running sum stays
//    per lane and is reduced once at the end.
//  * Warps of a CTA merge through shared memory.  A request with one chunk is
//    finished in place; otherwise each chunk CTA writes (o/d, lse) to the
//    workspace and bumps the (request, KV head)'s counter, and the last one
//    to arrive merges the chunks by log-sum-exp -- no second launch.
// There is no tensor-memory (tcgen05) path here: 8 query heads per KV head
// would fill 8 rows of a 128-row tcgen05 tile, or (keys as the rows) need
// 128-key tiles at the tensor pipe's ~46 cycles per instruction, while the
// work is bound by HBM and mma.sync keeps pace with it.

#include "kernels.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>

namespace sa {
namespace {

#ifndef SA_DECODE_NW
#define SA_DECODE_NW 8          // warps per CTA
#endif
#ifndef SA_DECODE_STAGES
#define SA_DECODE_STAGES 3      // pages in flight per warp
#endif
constexpr int kNW = SA_DECODE_NW;
constexpr int kStages = SA_DECODE_STAGES;
constexpr int kTileBytes = kPageSize * kHeadDim * 2;   // 2048
constexpr int kStageBytes = 2 * kTileBytes;            // K + V
constexpr int kHeadsPerTile = 8;

template <int NB>
struct __align__(16) MergeSmem {
  float o[kNW][kHeadsPerTile * NB][kHeadDim];
  float m[kNW][kHeadsPerTile * NB];
  float d[kNW][kHeadsPerTile * NB];
};

constexpr int kPipeBytes = kNW * kStages * kStageBytes;
constexpr int kBarOffset = kPipeBytes;
constexpr int kSmemBytes = kBarOffset + kNW * kStages * 8 + 1024;  // + alignment slack
static_assert(sizeof(MergeSmem<2>) <= kPipeBytes, "merge scratch aliases the stages");

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Chunk count of one request under the plan; 0 marks a request whose
// arguments are out of range (its outputs become NaN).
__device__ __forceinline__ int request_chunks(int kv_len, int min_len, int max_pages_per_seq,
                                              int num_splits, int pages_per_chunk) {
  if (kv_len < min_len) return 0;
  const int npages = ceil_div(kv_len, kPageSize);
  if (npages > max_pages_per_seq || npages > num_splits * pages_per_chunk) return 0;
  return npages == 0 ? 1 : ceil_div(npages, pages_per_chunk);
}

// Query row r of KV head kvh -> index of its [.., Hq] row in q/out/lse
// (-1 past the last row) and its head.  Plain decode has one token per
// request, so row r is head kvh * group + r.
template <bool kVerify>
__device__ __forceinline__ long long row_index(const DecodeParams &p, int b, int kvh, int r,
                                               int &head) {
  if constexpr (!kVerify) {
    head = kvh * p.group + r;
    return r < p.group ? static_cast<long long>(b) * p.num_qo_heads + head : -1;
  } else {
    const int tq = r / p.group;
    head = kvh * p.group + (r - tq * p.group);
    if (r >= p.rows) return -1;
    return (static_cast<long long>(b) * p.q_len + tq) * p.num_qo_heads + head;
  }
}

constexpr int kBuckets = 8;   // size classes of shorter requests in the dispatch order

// Size class of a request in plans with one chunk per request (no division:
// `per_page` = kBuckets / pages_per_chunk): requests as long as the chunk
// limit in the top class kBuckets, shorter ones in classes 0..kBuckets-1 by
// page count; empty and out-of-range requests in class 0.  Every CTA
// evaluates the same instructions on the same lengths, so all agree.
template <bool kVerify>
__device__ __forceinline__ int size_class(const DecodeParams &p, int kv_len, float per_page) {
  const int pages = ceil_div(kv_len, kPageSize);
  if (kv_len < (kVerify ? p.q_len : 0) || pages > p.max_pages_per_seq ||
      pages > p.pages_per_chunk)
    return 0;
  if (pages == p.pages_per_chunk) return kBuckets;
  return min(kBuckets - 1, __float2int_rz(static_cast<float>(pages) * per_page));
}

// The request of dispatch slot `item` for plans with one chunk per request,
// heaviest first so that the last wave holds the short requests: size class
// descending, request order within a class.  Every warp derives the same
// order from kv_lens on its own (no block barrier): class counts of each
// group of 32 requests come from two warp reductions of 6-bit fields, the
// request from one ballot per group.  Returns -1 past the last request;
// `kv_len` gets the request's length.
template <bool kVerify>
__device__ int request_by_size(const DecodeParams &p, int item, int &kv_len) {
  constexpr int kClasses = kBuckets + 1;
  constexpr int kLow = 5;                       // classes 0..4 in the first word, 5..8 in the second
  static_assert(kClasses <= 2 * kLow, "two words of 6-bit counters");
  constexpr int kHeld = 8;                      // groups of 32 requests kept in registers
  const int lane = threadIdx.x & 31;
  const int groups = ceil_div(p.batch, 32);
  const float per_page = static_cast<float>(kBuckets) / static_cast<float>(p.pages_per_chunk);
  int len[kHeld], cls_of[kHeld];
#pragma unroll
  for (int u = 0; u < kHeld; ++u) {
    const int b = u * 32 + lane;
    len[u] = u < groups && b < p.batch ? __ldg(p.kv_lens + b) : 0;
  }
  auto group_class = [&](int u, int &l) {
    const int b = u * 32 + lane;
    l = 0;
    int c = -1;
#pragma unroll
    for (int v = 0; v < kHeld; ++v)
      if (v == u) {
        l = len[v];
        c = cls_of[v];
      }
    if (u >= kHeld) {
      l = b < p.batch ? __ldg(p.kv_lens + b) : 0;
      c = b < p.batch ? size_class<kVerify>(p, l, per_page) : -1;
    }
    return c;
  };
  int total[kClasses];
#pragma unroll
  for (int k = 0; k < kClasses; ++k) total[k] = 0;
  for (int u = 0; u < groups; ++u) {
    const int b = u * 32 + lane;
    int l = 0;
#pragma unroll
    for (int v = 0; v < kHeld; ++v)
      if (v == u) l = len[v];
    if (u >= kHeld) l = b < p.batch ? __ldg(p.kv_lens + b) : 0;
    const int c = b < p.batch ? size_class<kVerify>(p, l, per_page) : -1;
#pragma unroll
    for (int v = 0; v < kHeld; ++v)
      if (v == u) cls_of[v] = c;
    // class counts of the group, 6 bits per class (a group adds at most 32)
    const unsigned lo = __reduce_add_sync(0xffffffffu, c >= 0 && c < kLow ? 1u << (6 * c) : 0u);
    const unsigned hi = __reduce_add_sync(0xffffffffu, c >= kLow ? 1u << (6 * (c - kLow)) : 0u);
#pragma unroll
    for (int k = 0; k < kClasses; ++k)
      total[k] += static_cast<int>(((k < kLow ? lo : hi) >> (6 * (k < kLow ? k : k - kLow))) & 63u);
  }
  int rank = item, cls = -1;
#pragma unroll
  for (int k = kClasses - 1; k >= 0; --k) {
    if (cls < 0) {
      if (rank < total[k]) cls = k;
      else rank -= total[k];
    }
  }
  if (cls < 0) return -1;
  for (int u = 0; u < groups; ++u) {
    int l;
    const int c = group_class(u, l);
    const unsigned hit = __ballot_sync(0xffffffffu, c == cls);
    const int n = __popc(hit);
    if (rank < n) {
      const int src = static_cast<int>(__fns(hit, 0, rank + 1));
      kv_len = __shfl_sync(0xffffffffu, l, src);
      return u * 32 + src;
    }
    rank -= n;
  }
  return -1;                                    // not reached: the classes cover the batch
}

template <int NB, bool kVerify>
__global__ void __launch_bounds__(kNW * 32, 2)
decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const DecodeParams p) {
  // CTA blockIdx.x: (KV head, head block) unit blockIdx.x % U of (request,
  // chunk) slot blockIdx.x / U.  Plans with one chunk per request and at
  // most a few waves of CTAs take the requests heaviest first; other plans
  // take them in order, chunk fastest (their many short CTAs would pay more
  // for the ordering than it saves).
  const int units = p.num_kv_heads * p.head_blocks;
  const int unit_y = static_cast<int>(blockIdx.x % units);
  const int hb = unit_y % p.head_blocks;
  const int kvh = unit_y / p.head_blocks;
  const int slot = static_cast<int>(blockIdx.x / units);
  int b = slot / p.num_splits, chunk = slot % p.num_splits;
  int kv_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.sorted_dispatch) {                 // one chunk per request
    b = request_by_size<kVerify>(p, slot, kv_len);
    chunk = 0;
    if (b < 0) return;
  } else {
    kv_len = p.kv_lens[b];
  }
  const int g = lane >> 2, t = lane & 3;
  constexpr int kCols = kHeadsPerTile * NB;       // query rows of this CTA

  // verification needs its q_len tokens among the keys; plain decode allows kv_len = 0
  const int nchunks = request_chunks(kv_len, kVerify ? p.q_len : 0, p.max_pages_per_seq,
                                     p.num_splits, p.pages_per_chunk);
  bool bad = nchunks == 0;
  if (!bad && chunk >= nchunks) return;        // uniform over the CTA
  if (bad && chunk != 0) return;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kBarOffset) + warp * kStages;
  uint8_t *stages = smem + warp * kStages * kStageBytes;

  const int row0 = hb * kCols;                  // first query row of this CTA
  const int npages = bad ? 0 : ceil_div(kv_len, kPageSize);
  const int p_begin = chunk * p.pages_per_chunk;
  const int p_end = min(npages, p_begin + p.pages_per_chunk);
  const int first = p_begin + warp;
  const int n_my = p_end > first ? ceil_div(p_end - first, kNW) : 0;
  const int32_t *table = p.page_table + static_cast<size_t>(b) * p.max_pages_per_seq;
  // keys [0, kv_len - q_len) are visible to every row; key kv_len - q_len + u
  // (draft token u) to the rows whose visibility mask has bit u
  const int draft0 = kv_len - p.q_len;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (warp == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
  }
  __syncwarp();

  // Page ids of this warp's pages, 32 at a time (lane j holds page j of the batch).
  auto load_ids = [&](int base) -> int {
    const int j = base + lane;
    return j < n_my ? table[first + j * kNW] : -1;
  };
  int ids_cur = load_ids(0), ids_next = load_ids(32);
  // page ids of this warp's first kStages pages, uniform over the warp
  int first_ids[kStages];
#pragma unroll
  for (int j = 0; j < kStages; ++j) first_ids[j] = __shfl_sync(0xffffffffu, ids_cur, j);
  // This warp's first pages into L2 while the previous kernel on the stream
  // may still be draining (a programmatic launch); the copies below then
  // find them there.
  {
    int pf = -1;
#pragma unroll
    for (int j = 0; j < kStages; ++j)
      if (lane == j && j < n_my) pf = first_ids[j];
    if (pf >= 0 && pf < p.num_pages) {
      tma_prefetch_l2_3d(&kmap, 0, kvh * kPageSize, pf);
      tma_prefetch_l2_3d(&vmap, 0, kvh * kPageSize, pf);
    }
  }

  // Up to here only kv_lens and page_table were read; everything below may
  // depend on the previous kernel on the stream (q, the caches, sinks, masks,
  // the outputs and the workspace).
  grid_dependency_wait();
  launch_dependents();

  // Q^T as the B operand: lane (g, t) holds row g of each column block, dims
  // 16ks+2t.. and 16ks+8+2t..
  uint32_t qb[NB][4][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    int head;
    const long long ri = row_index<kVerify>(p, b, kvh, row0 + nb * kHeadsPerTile + g, head);
    const bool live = ri >= 0;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + (live ? ri : 0) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      qb[nb][ks][0] = live ? __ldg(qrow + 8 * ks + t) : 0u;
      qb[nb][ks][1] = live ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  }

  // Softmax state of columns 2t and 2t+1 of each block (identical across the
  // 8 g-lanes); vis: draft-token visibility of those columns.
  float m[NB][2], d[NB][2];
  uint64_t vis[NB][2];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      int head;
      const int r = row0 + nb * kHeadsPerTile + 2 * t + e;
      const long long ri = row_index<kVerify>(p, b, kvh, r, head);
      m[nb][e] = -INFINITY;
      d[nb][e] = 0.f;
      vis[nb][e] = 0;
      if (chunk == 0 && warp == 0 && ri >= 0) {
        m[nb][e] = p.sinks[head] * kLog2e;
        if (g == 0) d[nb][e] = 1.f;          // the sink's e^(sink - m) = 1 counted once
      }
      if constexpr (kVerify) {
        if (ri >= 0) {
          const int tq = r / p.group;
          const uint64_t causal = tq >= 63 ? ~0ull : ((2ull << tq) - 1);
          vis[nb][e] = p.tree_mask ? p.tree_mask[static_cast<size_t>(b) * p.q_len + tq] : causal;
        }
      }
    }
  float o[NB][4][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[nb][i][0] = o[nb][i][1] = o[nb][i][2] = o[nb][i][3] = 0.f;

  bool lane_bad = false;     // meaningful on lane 0
  // With one CTA per (request, KV head, chunk) every page is read once: its
  // lines go first when L2 needs room, so the small tensors every launch
  // re-reads (kv_lens, page table, q) and the outputs stay.  Wider GQA groups
  // split into head blocks read each page twice, the second time from L2.
  const bool read_once = p.head_blocks == 1;
  const uint64_t evict_first = l2_policy_evict_first();

  auto issue = [&](int j) {  // all lanes call; lane 0 issues
    if ((j & 31) == 0 && j > 0) {
      ids_cur = ids_next;
      ids_next = load_ids(j + 32);
    }
    int pid;
    if (j < kStages) {                     // the first pages: ids known already
      pid = first_ids[0];
#pragma unroll
      for (int u = 1; u < kStages; ++u)
        if (j == u) pid = first_ids[u];
    } else {
      pid = __shfl_sync(0xffffffffu, ids_cur, j & 31);
    }
    if (lane == 0) {
      uint64_t *bar = &bars[j % kStages];
      uint8_t *dst = stages + (j % kStages) * kStageBytes;
      if (pid >= 0 && pid < p.num_pages) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, kStageBytes);
        if (read_once) {
          tma_load_3d_hint(dst, &kmap, bar, 0, kvh * kPageSize, pid, evict_first);
          tma_load_3d_hint(dst + kTileBytes, &vmap, bar, 0, kvh * kPageSize, pid, evict_first);
        } else {
          tma_load_3d(dst, &kmap, bar, 0, kvh * kPageSize, pid);
          tma_load_3d(dst + kTileBytes, &vmap, bar, 0, kvh * kPageSize, pid);
        }
      } else {
        lane_bad = true;     // skip the copy; the phase still completes
        mbar_arrive(bar);
      }
    }
  };

  const int n_pro = min(kStages, n_my);
  for (int j = 0; j < n_pro; ++j) issue(j);

  // ldmatrix lane roles (see header comment): K tiles non-transposed, V transposed.
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;

  for (int i = 0; i < n_my; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&bars[st], (i / kStages) & 1)) {
      // A copy never landed: report, then drain (bounded) whatever else this
      // warp still has in flight before the stages are reused below.
      lane_bad = true;
      bad = true;
      for (int j = i + 1; j < min(n_my, i + kStages); ++j)
        mbar_wait(&bars[j % kStages], (j / kStages) & 1);
      break;
    }
    const uint32_t kbase = smem_u32(stages + st * kStageBytes);
    const uint32_t vbase = kbase + kTileBytes;

    float s[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t a[4];
      const int c = 2 * ks + k_hi;
      ldsm_x4(kbase + k_row * 128 + ((c ^ (k_row & 7)) << 4), a);
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(s[nb], a, qb[nb][ks][0], qb[nb][ks][1]);
    }

    const int tok0 = (first + i * kNW) * kPageSize;
    const bool partial = tok0 + kPageSize > kv_len;
    // s[.][0]: token g / column 2t, [1]: token g / column 2t+1, [2], [3]: token g+8.
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int r = 0; r < 4; ++r) s[nb][r] *= p.scale_log2;
    if (partial) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        if (tok0 + g >= kv_len) s[nb][0] = s[nb][1] = -INFINITY;
        if (tok0 + g + 8 >= kv_len) s[nb][2] = s[nb][3] = -INFINITY;
      }
    }
    if constexpr (kVerify) {
      if (tok0 + kPageSize > draft0) {             // the page holds draft tokens
#pragma unroll
        for (int h8 = 0; h8 < 2; ++h8) {
          const int u = tok0 + g + 8 * h8 - draft0;
          if (u >= 0 && u < 64) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              if (!((vis[nb][0] >> u) & 1)) s[nb][2 * h8] = -INFINITY;
              if (!((vis[nb][1] >> u) & 1)) s[nb][2 * h8 + 1] = -INFINITY;
            }
          }
        }
      }
    }
    uint32_t pb[NB][2];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float x0 = fmaxf(s[nb][0], s[nb][2]), x1 = fmaxf(s[nb][1], s[nb][3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m[nb][0], x0), n1 = fmaxf(m[nb][1], x1);
      const float u0 = n0 == -INFINITY ? 0.f : n0;
      const float u1 = n1 == -INFINITY ? 0.f : n1;
      const float p0 = ex2(s[nb][0] - u0), p1 = ex2(s[nb][1] - u1);
      const float p2 = ex2(s[nb][2] - u0), p3 = ex2(s[nb][3] - u1);
      // o and d only need rescaling when a running max grew; otherwise the
      // factor is exactly 1 and the warp skips the multiplies
      if (__any_sync(0xffffffffu, n0 > m[nb][0] || n1 > m[nb][1])) {
        const float a0 = ex2(m[nb][0] - u0), a1 = ex2(m[nb][1] - u1);
        d[nb][0] *= a0;
        d[nb][1] *= a1;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
          o[nb][mt][0] *= a0;
          o[nb][mt][1] *= a1;
          o[nb][mt][2] *= a0;
          o[nb][mt][3] *= a1;
        }
      }
      d[nb][0] += p0 + p2;
      d[nb][1] += p1 + p3;
      m[nb][0] = n0;
      m[nb][1] = n1;
      pb[nb][0] = movmatrix_trans(pack_bf16(p0, p1));   // tokens 0..7
      pb[nb][1] = movmatrix_trans(pack_bf16(p2, p3));   // tokens 8..15
    }

    uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
    if (partial) {
      keep01 = (tok0 + 2 * t < kv_len ? 0x0000ffffu : 0u) |
               (tok0 + 2 * t + 1 < kv_len ? 0xffff0000u : 0u);
      keep23 = (tok0 + 2 * t + 8 < kv_len ? 0x0000ffffu : 0u) |
               (tok0 + 2 * t + 9 < kv_len ? 0xffff0000u : 0u);
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      uint32_t a[4];
      const int c = 2 * mt + v_hi;
      ldsm_x4_trans(vbase + v_row * 128 + ((c ^ (v_row & 7)) << 4), a);
      a[0] &= keep01;       // padded slots may hold anything (even NaN)
      a[1] &= keep01;
      a[2] &= keep23;
      a[3] &= keep23;
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) mma_bf16_16816(o[nb][mt], a, pb[nb][0], pb[nb][1]);
    }
    __syncwarp();
    const int j = i + kStages;
    if (j < n_my) issue(j);
  }

  // Full per-column sums.
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      d[nb][0] += __shfl_xor_sync(0xffffffffu, d[nb][0], off);
      d[nb][1] += __shfl_xor_sync(0xffffffffu, d[nb][1], off);
    }
  bad = bad || (__shfl_sync(0xffffffffu, lane_bad ? 1 : 0, 0) != 0);

  __syncthreads();   // every warp is done with its stages: alias them
  MergeSmem<NB> &ms = *reinterpret_cast<MergeSmem<NB> *>(smem);
  __shared__ int cta_bad;
  if (threadIdx.x == 0) cta_bad = 0;
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int c0 = nb * kHeadsPerTile + 2 * t;
    if (g == 0) {
      ms.m[warp][c0] = m[nb][0];
      ms.m[warp][c0 + 1] = m[nb][1];
      ms.d[warp][c0] = d[nb][0];
      ms.d[warp][c0 + 1] = d[nb][1];
    }
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      ms.o[warp][c0][16 * mt + g] = o[nb][mt][0];
      ms.o[warp][c0 + 1][16 * mt + g] = o[nb][mt][1];
      ms.o[warp][c0][16 * mt + 8 + g] = o[nb][mt][2];
      ms.o[warp][c0 + 1][16 * mt + 8 + g] = o[nb][mt][3];
    }
  }
  __syncthreads();
  if (bad) atomicOr(&cta_bad, 1);
  __syncthreads();
  const bool failed = cta_bad != 0;

  const size_t stride = static_cast<size_t>(p.batch) * p.q_len * p.num_qo_heads;
  for (int item = threadIdx.x; item < kCols * (kHeadDim / 4); item += kNW * 32) {
    const int hh = item / (kHeadDim / 4);
    const int dq = (item % (kHeadDim / 4)) * 4;
    int head;
    const long long ri = row_index<kVerify>(p, b, kvh, row0 + hh, head);
    if (ri < 0) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) mx = fmaxf(mx, ms.m[w][hh]);
    float den = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      const float mw = ms.m[w][hh];
      const float wt = mw == -INFINITY ? 0.f : ex2(mw - mx);
      den += wt * ms.d[w][hh];
      const float4 ov = *reinterpret_cast<const float4 *>(&ms.o[w][hh][dq]);
      acc[0] += wt * ov.x;
      acc[1] += wt * ov.y;
      acc[2] += wt * ov.z;
      acc[3] += wt * ov.w;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float lse2 = den > 0.f ? mx + lg2(den) : -INFINITY;
    if (failed) {
      acc[0] = acc[1] = acc[2] = acc[3] = NAN;
      lse2 = NAN;
    }
    const size_t row = static_cast<size_t>(ri);
    if (nchunks <= 1) {
      uint2 packed;
      packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2 *>(p.out + row * kHeadDim + dq) = packed;
      if (dq == 0 && p.lse) p.lse[row] = lse2 * kLn2;
    } else {
      const size_t wrow = static_cast<size_t>(chunk) * stride + row;
      *reinterpret_cast<float4 *>(p.ws_o + wrow * kHeadDim + dq) =
          make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
      if (dq == 0) p.ws_lse[wrow] = lse2;
    }
  }
  if (nchunks <= 1) return;

  // Split request: the last of its chunk CTAs to get here merges the chunk
  // results by log-sum-exp (and leaves the counter at zero for the next call).
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  const size_t unit = static_cast<size_t>(b) * (p.num_kv_heads * p.head_blocks) + unit_y;
  if (threadIdx.x == 0) is_last = atomicAdd(&p.counters[unit], 1) == nchunks - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int item = threadIdx.x; item < kCols * (kHeadDim / 4); item += kNW * 32) {
    const int hh = item / (kHeadDim / 4);
    const int dq = (item % (kHeadDim / 4)) * 4;
    int head;
    const long long ri = row_index<kVerify>(p, b, kvh, row0 + hh, head);
    if (ri < 0) continue;
    const size_t row = static_cast<size_t>(ri);
    float mx = -INFINITY, den = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool poisoned = false;       // a chunk reported NaN (bad page or failed wait)
    for (int c = 0; c < nchunks; ++c) {
      const float lc = __ldcg(p.ws_lse + c * stride + row);
      if (lc != lc) {
        poisoned = true;
        continue;
      }
      if (lc == -INFINITY) continue;
      const float4 ov = __ldcg(reinterpret_cast<const float4 *>(p.ws_o + (c * stride + row) * kHeadDim + dq));
      const float nm = fmaxf(mx, lc);
      const float a = mx == -INFINITY ? 0.f : ex2(mx - nm);
      const float wt = ex2(lc - nm);
      den = den * a + wt;
      acc[0] = acc[0] * a + wt * ov.x;
      acc[1] = acc[1] * a + wt * ov.y;
      acc[2] = acc[2] * a + wt * ov.z;
      acc[3] = acc[3] * a + wt * ov.w;
      mx = nm;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    uint2 packed;
    if (poisoned) {
      packed = make_uint2(0x7fc07fc0u, 0x7fc07fc0u);
    } else {
      packed.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      packed.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    }
    *reinterpret_cast<uint2 *>(p.out + row * kHeadDim + dq) = packed;
    if (dq == 0 && p.lse)
      p.lse[row] = poisoned ? NAN : (den > 0.f ? (mx + lg2(den)) * kLn2 : -INFINITY);
  }
  if (threadIdx.x == 0) p.counters[unit] = 0;
}

template <int NB, bool kVerify>
cudaError_t launch_variant(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                           cudaStream_t stream, bool programmatic) {
  cudaError_t err = set_smem_once<decode_kernel<NB, kVerify>>(kSmemBytes);
  if (err != cudaSuccess) return err;
  const unsigned long long ctas =
      static_cast<unsigned long long>(p.num_splits) * p.batch * p.num_kv_heads * p.head_blocks;
  if (ctas > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  return launch_kernel(decode_kernel<NB, kVerify>, static_cast<unsigned>(ctas), kNW * 32,
                       kSmemBytes, stream, programmatic, kmap, vmap, p);
}

}  // namespace

int decode_ctas_per_sm() {
  // shared memory bounds residency: 228 KB per SM, 1 KB of it reserved per CTA
  return std::max(1, std::min(228 * 1024 / (kSmemBytes + 1024), 2048 / (kNW * 32)));
}

int decode_max_splits() { return 1024; }

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                          cudaStream_t stream, bool programmatic) {
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  const bool verify = p.q_len > 1 || p.tree_mask != nullptr;
  if (!verify) {
    return p.col_blocks == 1 ? launch_variant<1, false>(kmap, vmap, p, stream, programmatic)
                             : launch_variant<2, false>(kmap, vmap, p, stream, programmatic);
  }
  if (p.col_blocks == 1) return launch_variant<1, true>(kmap, vmap, p, stream, programmatic);
  return launch_variant<2, true>(kmap, vmap, p, stream, programmatic);
}

}  // namespace sa
