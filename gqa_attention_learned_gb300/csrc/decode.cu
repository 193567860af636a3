// Paged-KV decode with learned sinks: page-balanced split-KV with an
// in-kernel log-sum-exp merge.
//
// Operation: "GPT-OSS on day 0" (Perplexity blog), section "Kernels for
// GPT-OSS / Sink Attention" -- online softmax with the running max started at
// the head's sink (scale d = 1) in the first KV block only, other blocks
// started at -inf, blocks merged by log-sum-exp.
//
// Work decomposition (GB300, HBM-bound):
//  * A unit is one (request, KV head, block of <= 8 query heads); its pages
//    are laid end to end, unit after unit, into one global page sequence of
//    W pages.  Worker warp w of Wn takes pages [w W / Wn, (w+1) W / Wn): every
//    worker streams the same number of pages whatever the mix of request
//    lengths, so no long request is left running alone at the end.
//  * A worker's range covers several units.  A unit seen whole is finished in
//    place; a unit cut between workers becomes KV chunks: each worker writes
//    its chunk's (o / d, lse) to the workspace and bumps the unit's counter,
//    and the last one to arrive merges the chunks by log-sum-exp and resets
//    the counter.  Only the chunk holding the unit's first page starts its
//    online softmax at the sink.
//  * Each warp runs its own STAGES-deep TMA pipeline: lane 0 issues 3-D bulk
//    tensor copies of the page's K and V tiles (2 KB each, 128-byte swizzle)
//    onto the stage's mbarrier; 3 CTAs x 4 warps x 4 stages keep 48 pages
//    (192 KB) in flight per SM, which is what HBM latency asks for.  The next
//    unit's Q is loaded into registers one chunk ahead.
//  * The GQA group shares every K/V tile: S^T[16 tok x 8 heads] = K . Q^T and
//    O^T[64 x 8] += V^T . P^T, each 4 mma.sync.m16n8k16 (bf16 in, fp32 acc).
//    P^T goes from the score accumulator layout to the B-operand layout with
//    movmatrix.trans; K and V^T come from shared memory by ldmatrix,
//    bank-conflict free thanks to the swizzle.  Row maxima take 3 xor-shuffles
//    per page; running sums stay per lane until the chunk ends.
// There is no tensor-memory (tcgen05) path here: n = 8 query heads per KV
// head is far below tcgen05's minimum tile, and the work is bound by HBM.

#include "kernels.cuh"
#include "ptx.cuh"

#include <cmath>

namespace sa {
namespace {

constexpr int kNW = 4;                 // worker warps per CTA
constexpr int kStages = 4;             // pages in flight per warp
constexpr int kTileBytes = kPageSize * kHeadDim * 2;   // 2048
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kHeadsPerTile = 8;
constexpr int kMaxBatch = 4096;        // requests per launch (per-CTA tables)

constexpr int kOffStages = 0;
constexpr int kOffBars = kNW * kStages * kStageBytes;
constexpr int kOffTables = kOffBars + kNW * kStages * 8;
constexpr int kSmemFixed = kOffTables + 1024;                       // + alignment slack

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Pages of a request under the arguments' bounds; -1 marks a request whose
// arguments are out of range (its outputs become NaN).
__device__ __forceinline__ int request_pages(int kv_len, int max_pages_per_seq) {
  if (kv_len < 0) return -1;
  const int n = ceil_div(kv_len, kPageSize);
  return n > max_pages_per_seq ? -1 : n;
}

// Where global page x lives: request b (by the prefix table), unit-in-request
// uh, page within the unit pg.
struct PageRef {
  int b, uh, pg;
};

__device__ __forceinline__ PageRef locate(long long x, const long long *prefix, const int *npages,
                                          int batch, int units_per_req) {
  int lo = 0, hi = batch - 1;            // last b with prefix[b] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  PageRef r;
  r.b = lo;
  const long long off = x - prefix[lo];
  const int np = npages[lo];
  r.uh = static_cast<int>(off / np);
  r.pg = static_cast<int>(off % np);
  return r;
}

__global__ void __launch_bounds__(kNW * 32, 3)
decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const DecodeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int units_per_req = p.num_kv_heads * p.head_blocks;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *stages = smem + kOffStages + warp * kStages * kStageBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBars) + warp * kStages;
  long long *prefix = reinterpret_cast<long long *>(smem + kOffTables);   // [batch + 1]
  int *npages = reinterpret_cast<int *>(prefix + p.batch + 1);           // [batch], -1 = bad
  int *kvl = npages + p.batch;                                           // [batch]
  float *sinks2 = reinterpret_cast<float *>(kvl + p.batch);              // [Hq], log2 units

  // ---- per-CTA tables: pages per request and their running sum over units
  for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
    kvl[b] = p.kv_lens[b];
    npages[b] = request_pages(kvl[b], p.max_pages_per_seq);
  }
  for (int h = threadIdx.x; h < p.num_qo_heads; h += blockDim.x) sinks2[h] = p.sinks[h] * kLog2e;
  __syncthreads();
  if (warp == 0) {
    long long run = 0;
    for (int base = 0; base < p.batch; base += 32) {
      const int b = base + lane;
      const long long v = b < p.batch ? static_cast<long long>(max(npages[b], 0)) * units_per_req : 0;
      long long incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (b < p.batch) prefix[b] = run + incl - v;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[p.batch] = run;
  }
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (warp == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
  }
  __syncthreads();

  const long long total = prefix[p.batch];
  const long long workers = min(static_cast<long long>(p.num_workers), max(total, 1ll));
  const long long w = static_cast<long long>(blockIdx.x) * kNW + warp;

  // ---- requests without pages (kv_len 0, or arguments out of range)
  for (long long b = w; b < p.batch; b += static_cast<long long>(gridDim.x) * kNW) {
    if (npages[b] > 0) continue;
    const bool bad = npages[b] < 0;
    for (int i = lane; i < p.num_qo_heads * kHeadDim / 4; i += 32) {
      const size_t off = static_cast<size_t>(b) * p.num_qo_heads * kHeadDim + 4 * i;
      const uint32_t v = bad ? 0x7fc07fc0u : 0u;
      *reinterpret_cast<uint2 *>(p.out + off) = make_uint2(v, v);
    }
    if (p.lse)
      for (int h = lane; h < p.num_qo_heads; h += 32)
        p.lse[static_cast<size_t>(b) * p.num_qo_heads + h] = bad ? NAN : sinks2[h] * kLn2;
  }
  if (w >= workers) return;

  const long long r0 = w * total / workers, r1 = (w + 1) * total / workers;
  const int n_my = static_cast<int>(r1 - r0);

  // Page references of this warp's pages, 32 at a time: lane j holds page
  // base + j as (request, unit-in-request, page-in-unit) and its page id.
  struct Batch {
    int b, uh, pg, pid;
  };
  auto load_batch = [&](int base) {
    Batch bt{0, 0, 0, -1};
    const int j = base + lane;
    if (j < n_my) {
      const PageRef ref = locate(r0 + j, prefix, npages, p.batch, units_per_req);
      bt.b = ref.b;
      bt.uh = ref.uh;
      bt.pg = ref.pg;
      bt.pid = p.page_table[static_cast<size_t>(ref.b) * p.max_pages_per_seq + ref.pg];
    }
    return bt;
  };
  Batch iss = load_batch(0), iss_next = load_batch(32);
  Batch cmp = iss;
  uint32_t stage_bad = 0;    // lane 0: bit s = the page now in stage s had a bad id

  auto issue = [&](int j) {  // all lanes call; lane 0 issues
    if ((j & 31) == 0 && j > 0) {
      iss = iss_next;
      iss_next = load_batch(j + 32);
    }
    const int src = j & 31;
    const int uh = __shfl_sync(0xffffffffu, iss.uh, src);
    const int pid = __shfl_sync(0xffffffffu, iss.pid, src);
    if (lane == 0) {
      uint64_t *bar = &bars[j % kStages];
      uint8_t *dst = stages + (j % kStages) * kStageBytes;
      const int kvh = uh / p.head_blocks;
      fence_proxy_async_smem();
      if (pid >= 0 && pid < p.num_pages) {
        mbar_arrive_expect_tx(bar, 2 * kTileBytes);
        tma_load_3d(dst, &kmap, bar, 0, kvh * kPageSize, pid);
        tma_load_3d(dst + kTileBytes, &vmap, bar, 0, kvh * kPageSize, pid);
      } else {
        stage_bad |= 1u << (j % kStages);   // skip the copy; the phase still completes
        mbar_arrive(bar);
      }
    }
  };

  const int n_pro = min(kStages, n_my);
  for (int j = 0; j < n_pro; ++j) issue(j);

  // ldmatrix lane roles: K and Q tiles non-transposed, V transposed.
  const int k_row = (lane & 7) + 8 * ((lane >> 3) & 1);
  const int k_hi = lane >> 4;
  const int v_row = (lane & 7) + 8 * (lane >> 4);
  const int v_hi = (lane >> 3) & 1;

  // chunk state (heads 2t, 2t+1 of the current unit)
  float m0 = -INFINITY, m1 = -INFINITY, d0 = 0.f, d1 = 0.f;
  float o[4][4];
  uint32_t qb[4][2], qn[4][2];             // Q^T B fragments: current / next unit
  int cur_b = -1, cur_uh = 0, chunk_first_pg = 0, cur_pg = 0;
  bool failed = false, chunk_bad = false;

  // Q^T as the B operand for unit (b, uh): lane (g, t) holds query head g of
  // the unit's 8-head block, dims 16ks+2t.. and 16ks+8+2t..; heads past the
  // GQA group are zero.  Loaded one unit ahead so the latency stays hidden.
  auto load_q = [&](int b, int uh, uint32_t (&dst)[4][2]) {
    const int kvh = uh / p.head_blocks, hb = uh % p.head_blocks;
    const int nheads = min(kHeadsPerTile, p.group - hb * kHeadsPerTile);
    const bool live = b >= 0 && b < p.batch && g < nheads;
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
        p.q + (static_cast<size_t>(live ? b : 0) * p.num_qo_heads + kvh * p.group +
               hb * kHeadsPerTile + (live ? g : 0)) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      dst[ks][0] = live ? __ldg(qrow + 8 * ks + t) : 0u;
      dst[ks][1] = live ? __ldg(qrow + 8 * ks + 4 + t) : 0u;
    }
  };
  auto next_unit = [&](int b, int uh, int &nb, int &nuh) {
    nb = b;
    nuh = uh + 1;
    if (nuh == units_per_req) {
      nuh = 0;
      do { ++nb; } while (nb < p.batch && npages[nb] <= 0);
    }
  };

  // Output element (head, dim) of this lane's fragment value v = o[mt][k].
  auto frag_head = [&](int k) { return 2 * t + (k & 1); };
  auto frag_dim = [&](int mt, int k) { return 16 * mt + g + 8 * (k >> 1); };

  // Finish the current chunk: whole unit -> output; else chunk + merge.
  auto finish_chunk = [&]() {
    float e0 = d0, e1 = d1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      e0 += __shfl_xor_sync(0xffffffffu, e0, off);
      e1 += __shfl_xor_sync(0xffffffffu, e1, off);
    }
    const bool bad = failed || chunk_bad || npages[cur_b] < 0;
    const int np = npages[cur_b];
    const bool whole = chunk_first_pg == 0 && cur_pg == np - 1;
    const int kvh = cur_uh / p.head_blocks, hb = cur_uh % p.head_blocks;
    const int head0 = kvh * p.group + hb * kHeadsPerTile;
    const int nheads = min(kHeadsPerTile, p.group - hb * kHeadsPerTile);
    const float i0 = e0 > 0.f ? 1.f / e0 : 0.f, i1 = e1 > 0.f ? 1.f / e1 : 0.f;
    // base-2 lse of heads 2t, 2t+1
    const float l0 = bad ? NAN : (e0 > 0.f ? m0 + lg2(e0) : -INFINITY);
    const float l1 = bad ? NAN : (e1 > 0.f ? m1 + lg2(e1) : -INFINITY);
    const size_t orow0 = static_cast<size_t>(cur_b) * p.num_qo_heads + head0;
    if (whole) {
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int hh = frag_head(k);
          if (hh < nheads) {
            const float v = bad ? NAN : o[mt][k] * ((k & 1) ? i1 : i0);
            reinterpret_cast<__nv_bfloat16 *>(p.out)[(orow0 + hh) * kHeadDim + frag_dim(mt, k)] =
                __float2bfloat16_rn(v);
          }
        }
      if (p.lse && g == 0) {
        if (2 * t < nheads) p.lse[orow0 + 2 * t] = l0 * kLn2;
        if (2 * t + 1 < nheads) p.lse[orow0 + 2 * t + 1] = l1 * kLn2;
      }
    } else {
      // chunk result in fragment order -> slot (worker, first-or-last chunk)
      const long long unit_start = prefix[cur_b] + static_cast<long long>(cur_uh) * np;
      const bool first_of_range = unit_start + chunk_first_pg == r0;
      const long long slot = 2 * w + (first_of_range ? 0 : 1);
      float4 *dst = reinterpret_cast<float4 *>(p.ws_o + slot * kHeadsPerTile * kHeadDim + lane * 16);
      const float nanv = NAN;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
        dst[mt] = bad ? make_float4(nanv, nanv, nanv, nanv)
                      : make_float4(o[mt][0] * i0, o[mt][1] * i1, o[mt][2] * i0, o[mt][3] * i1);
      if (g == 0) {
        p.ws_lse[slot * kHeadsPerTile + 2 * t] = l0;
        p.ws_lse[slot * kHeadsPerTile + 2 * t + 1] = l1;
      }
      __syncwarp();
      // contributors: workers whose ranges meet the unit
      const long long unit_end = unit_start + np;                 // exclusive
      const long long wf = ((unit_start + 1) * workers - 1) / total;
      const long long wl = (unit_end * workers - 1) / total;
      const int unit_id = cur_b * units_per_req + cur_uh;
      int last = 0;
      if (lane == 0) last = atomic_add_acq_rel(&p.counters[unit_id], 1) == static_cast<int>(wl - wf);
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        // online log-sum-exp over the chunks, per lane: heads 2t, 2t+1
        float mx[2] = {-INFINITY, -INFINITY}, den[2] = {0.f, 0.f};
        bool poisoned = false;     // a chunk reported NaN (bad page, failed wait)
        float acc[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        for (long long c = wf; c <= wl; ++c) {
          const long long cs = 2 * c + ((c * total / workers) >= unit_start ? 0 : 1);
          const float lc[2] = {__ldcg(p.ws_lse + cs * kHeadsPerTile + 2 * t),
                               __ldcg(p.ws_lse + cs * kHeadsPerTile + 2 * t + 1)};
          const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + cs * kHeadsPerTile * kHeadDim + lane * 16);
          float a[2], wgt[2];
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            if (lc[h2] != lc[h2]) poisoned = true;
            if (lc[h2] != lc[h2] || lc[h2] == -INFINITY) {
              a[h2] = 1.f;
              wgt[h2] = 0.f;
              continue;
            }
            const float nm = fmaxf(mx[h2], lc[h2]);
            a[h2] = mx[h2] == -INFINITY ? 0.f : ex2(mx[h2] - nm);
            wgt[h2] = ex2(lc[h2] - nm);
            den[h2] = den[h2] * a[h2] + wgt[h2];
            mx[h2] = nm;
          }
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            const float4 q4 = __ldcg(src + mt);
            acc[mt][0] = wgt[0] == 0.f ? acc[mt][0] : acc[mt][0] * a[0] + wgt[0] * q4.x;
            acc[mt][1] = wgt[1] == 0.f ? acc[mt][1] : acc[mt][1] * a[1] + wgt[1] * q4.y;
            acc[mt][2] = wgt[0] == 0.f ? acc[mt][2] : acc[mt][2] * a[0] + wgt[0] * q4.z;
            acc[mt][3] = wgt[1] == 0.f ? acc[mt][3] : acc[mt][3] * a[1] + wgt[1] * q4.w;
          }
        }
        const float inv[2] = {den[0] > 0.f ? 1.f / den[0] : 0.f, den[1] > 0.f ? 1.f / den[1] : 0.f};
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int hh = frag_head(k);
            if (hh < nheads) {
              const float v = poisoned ? NAN : acc[mt][k] * inv[k & 1];
              reinterpret_cast<__nv_bfloat16 *>(p.out)[(orow0 + hh) * kHeadDim + frag_dim(mt, k)] =
                  __float2bfloat16_rn(v);
            }
          }
        if (p.lse && g == 0) {
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
            if (2 * t + h2 < nheads)
              p.lse[orow0 + 2 * t + h2] =
                  poisoned ? NAN : (den[h2] > 0.f ? (mx[h2] + lg2(den[h2])) * kLn2 : -INFINITY);
        }
        if (lane == 0) p.counters[unit_id] = 0;      // ready for the next call
      }
    }
    __syncwarp();
  };

  for (int i = 0; i < n_my; ++i) {
    // the issue side switched to this batch kStages pages ago
    if ((i & 31) == 0 && i > 0) cmp = iss;
    const int src = i & 31;
    const int b = __shfl_sync(0xffffffffu, cmp.b, src);
    const int uh = __shfl_sync(0xffffffffu, cmp.uh, src);
    const int pg = __shfl_sync(0xffffffffu, cmp.pg, src);
    const int st = i % kStages;
    const bool chunk_start = pg == 0 || i == 0;
    if (chunk_start && i > 0) finish_chunk();

    bool landed = !failed && mbar_wait(&bars[st], (i / kStages) & 1);
    landed = __all_sync(0xffffffffu, landed);
    if (!landed && !failed) {
      // A copy never landed: drain (bounded) what else is in flight, then
      // walk the rest of the range producing NaN chunks so every unit's
      // counter still completes.
      for (int j = i + 1; j < min(n_my, i + kStages); ++j) mbar_wait(&bars[j % kStages], (j / kStages) & 1);
      failed = true;
    }
    const uint32_t sbase = smem_u32(stages + st * kStageBytes);
    const uint32_t kbase = sbase, vbase = sbase + kTileBytes;
    const int kvh = uh / p.head_blocks, hb = uh % p.head_blocks;
    const int nheads = min(kHeadsPerTile, p.group - hb * kHeadsPerTile);
    if (chunk_start) {
      cur_b = b;
      cur_uh = uh;
      chunk_first_pg = pg;
      chunk_bad = false;
      // sink only in the chunk that holds the unit's first page
      const int head0 = kvh * p.group + hb * kHeadsPerTile;
      if (pg == 0) {
        m0 = 2 * t < nheads ? sinks2[head0 + 2 * t] : -INFINITY;
        m1 = 2 * t + 1 < nheads ? sinks2[head0 + 2 * t + 1] : -INFINITY;
        d0 = d1 = (g == 0) ? 1.f : 0.f;      // the sink's e^0 counted once
      } else {
        m0 = m1 = -INFINITY;
        d0 = d1 = 0.f;
      }
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      // this unit's Q (prefetched at the previous chunk start, except for
      // the first chunk), then prefetch the next unit's
      if (i == 0) load_q(b, uh, qb);
      else {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          qb[ks][0] = qn[ks][0];
          qb[ks][1] = qn[ks][1];
        }
      }
      int nb, nuh;
      next_unit(b, uh, nb, nuh);
      load_q(nb, nuh, qn);
    }
    cur_pg = pg;
    if (__shfl_sync(0xffffffffu, (stage_bad >> st) & 1u, 0)) chunk_bad = true;
    if (lane == 0) stage_bad &= ~(1u << st);

    if (!failed) {
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4];
        const int c = 2 * ks + k_hi;
        ldsm_x4(kbase + k_row * 128 + ((c ^ (k_row & 7)) << 4), a);
        mma_bf16_16816(s, a, qb[ks][0], qb[ks][1]);
      }
      const int kv_len = kvl[b];
      const int tok0 = pg * kPageSize;
      const bool partial = tok0 + kPageSize > kv_len;
      // s[0]: token g / head 2t, s[1]: token g / head 2t+1, s[2], s[3]: token g+8.
#pragma unroll
      for (int r = 0; r < 4; ++r) s[r] *= p.scale_log2;
      if (partial) {
        if (tok0 + g >= kv_len) s[0] = s[1] = -INFINITY;
        if (tok0 + g + 8 >= kv_len) s[2] = s[3] = -INFINITY;
      }
      float x0 = fmaxf(s[0], s[2]), x1 = fmaxf(s[1], s[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
      }
      const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
      const float u0 = n0 == -INFINITY ? 0.f : n0;
      const float u1 = n1 == -INFINITY ? 0.f : n1;
      const float a0 = ex2(m0 - u0), a1 = ex2(m1 - u1);
      const float p0 = ex2(s[0] - u0), p1 = ex2(s[1] - u1);
      const float p2 = ex2(s[2] - u0), p3 = ex2(s[3] - u1);
      d0 = d0 * a0 + p0 + p2;
      d1 = d1 * a1 + p1 + p3;
      m0 = n0;
      m1 = n1;
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        o[mt][0] *= a0;
        o[mt][1] *= a1;
        o[mt][2] *= a0;
        o[mt][3] *= a1;
      }
      const uint32_t pb0 = movmatrix_trans(pack_bf16(p0, p1));   // tokens 0..7
      const uint32_t pb1 = movmatrix_trans(pack_bf16(p2, p3));   // tokens 8..15
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
        mma_bf16_16816(o[mt], a, pb0, pb1);
      }
    }
    __syncwarp();
    const int j = i + kStages;
    if (j < n_my && !failed) issue(j);
    if (j < n_my && failed) {
      // keep the issue-side page references in step without issuing
      if ((j & 31) == 0) {
        iss = iss_next;
        iss_next = load_batch(j + 32);
      }
    }
  }
  if (n_my > 0) finish_chunk();
}

}  // namespace

int decode_ctas_per_sm() { return 3; }

int decode_max_batch() { return kMaxBatch; }

size_t decode_smem_bytes(int batch, int num_qo_heads) {
  return kSmemFixed + (batch + 1) * sizeof(long long) + 2 * batch * sizeof(int) +
         num_qo_heads * sizeof(float);
}

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                          int grid, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(p.batch, p.num_qo_heads);
  cudaError_t err = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  decode_kernel<<<grid, kNW * 32, smem, stream>>>(kmap, vmap, p);
  return cudaGetLastError();
}

int decode_warps_per_cta() { return kNW; }

}  // namespace sa
