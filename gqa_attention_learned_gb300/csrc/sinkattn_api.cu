// C ABI of libsinkattn: argument checks, split planning, TMA descriptor
// encoding and kernel launches.  The operations are specified in
// include/sinkattn.h.  Nothing here allocates device memory or synchronises.

#include "sinkattn.h"
#include "kernels.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <atomic>
#include <cmath>
#include <mutex>

namespace {

using sa::kHeadDim;
using sa::kPageSize;

constexpr int kMaxDevices = 64;
constexpr int kMinPagesPerChunk = 16;   // keeps merge traffic under ~3% of KV
constexpr int kWavesTarget = 4;
constexpr int kVerifyWavesTarget = 2;
constexpr int kMaxChunkPages = 512;     // one-chunk plans only up to 8192 tokens
constexpr int kSortedWaves = 4;         // heaviest-first dispatch up to this many waves

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

thread_local char g_last_error[256] = "";

// Record the CUDA error behind a SINKATTN_CUDA_ERROR for sinkattn_last_error.
int cuda_status(cudaError_t err, const char *where) {
  if (err == cudaSuccess) return SINKATTN_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(err),
           static_cast<int>(err));
  return SINKATTN_CUDA_ERROR;
}

int fail_msg(const char *what) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", what);
  return SINKATTN_CUDA_ERROR;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// bf16 tensor viewed as [outer][rows][64] with 128-byte rows; box = box_rows
// rows of one outer index, 128-byte swizzle.
bool encode_rows_map(CUtensorMap *map, const void *base, unsigned long long rows_per_outer,
                     unsigned long long outer, unsigned box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), rows_per_outer, outer};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                           static_cast<cuuint64_t>(rows_per_outer * kHeadDim * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 tensor viewed as [d2][d1][64] (128-byte rows), box {64, b1, b2},
// 128-byte swizzle.
bool encode_map(CUtensorMap *map, const void *base, unsigned long long d1, unsigned long long d2,
                unsigned b1, unsigned b2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), d1, d2};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2),
                           static_cast<cuuint64_t>(d1 * kHeadDim * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), b1, b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr int kPrefillTile = 128;     // query rows per prefill CTA
constexpr int kPrefillKvTile = 128;   // keys per prefill K/V tile

struct DecodePlan {
  int num_splits = 1;
  int pages_per_chunk = 1;
  size_t counters_bytes = 0;  // merge counters (zeroed once, reset by every call)
  size_t workspace_bytes = 0;
  int sorted_dispatch = 0;    // one chunk per request, <= kSortedWaves waves of CTAs
  int tensor_cores = 0;       // verification on the tcgen05 kernel (no KV split)
  int col_blocks = 1;         // 8-row column blocks per CTA
  int head_blocks = 1;        // CTAs per (request, KV head, chunk)
};

// Verification of q_len tokens runs on the tensor-core (tcgen05) kernel when
// the query rows of a KV head fill a good part of its 128-row tile (at least
// 3 blocks of 8), the group divides 128, no request is longer than one
// chunk's limit, and the launch has a wave of CTAs without splitting the KV.
bool verify_on_tensor_cores(int batch, int q_len, int num_qo_heads, int num_kv_heads,
                            int max_pages, int num_sms) {
  const int group = num_qo_heads / num_kv_heads;
  if (q_len < 2 || 128 % group || q_len * group < 24 || max_pages > kMaxChunkPages) return false;
  const long long tiles = ceil_div(q_len, 128 / group);
  return tiles * batch * num_kv_heads >= 2ll * std::max(num_sms, 1);
}

// CTA column blocks and head blocks of q_len tokens per request: more than 8
// query rows per KV head (a draft of several tokens, or a GQA group above 8)
// take two 8-row column blocks per CTA, so the CTA reads each page once for
// 16 rows.  Plain decode does so only when those wider CTAs still fill the
// GPU (at least one wave of (request, KV head, 16-head block) units):
// otherwise 8-row CTAs, twice as many, keep more pages in flight (measured:
// 64 q / 4 KV heads, 64 requests: 4788 GB/s with 8-row CTAs, 4027 with 16-row
// CTAs and split chunks; 128 requests: 4807 and 6130).
void decode_blocks(int q_len, int group, int *col_blocks, int *head_blocks) {
  const int rows = q_len * group;
  *col_blocks = sa::decode_col_blocks(rows);
  *head_blocks = ceil_div(rows, 8 * *col_blocks);
}

void decode_blocks_for(int batch, int q_len, int group, int num_kv_heads, int num_sms,
                       int *col_blocks, int *head_blocks) {
  decode_blocks(q_len, group, col_blocks, head_blocks);
  const long long slots = static_cast<long long>(std::max(num_sms, 1)) * sa::decode_ctas_per_sm();
  if (q_len == 1 && *col_blocks == 2 &&
      static_cast<long long>(batch) * num_kv_heads * *head_blocks < slots) {
    *col_blocks = 1;
    *head_blocks = ceil_div(group, 8);
  }
}

// Split count: by default enough (request, KV head, chunk) CTAs for a few
// waves of the GPU, chunks of at least kMinPagesPerChunk pages; an explicit
// count is honoured up to one page per chunk.
DecodePlan plan_decode(int batch, int q_len, int num_qo_heads, int num_kv_heads, int max_kv_len,
                       int num_sms, int requested) {
  DecodePlan plan;
  const int group = num_qo_heads / num_kv_heads;
  int col_blocks, head_blocks;
  decode_blocks_for(batch, q_len, group, num_kv_heads, num_sms, &col_blocks, &head_blocks);
  plan.col_blocks = col_blocks;
  plan.head_blocks = head_blocks;
  const int max_pages = std::max(1, ceil_div(max_kv_len, kPageSize));
  if (requested == 0 &&
      verify_on_tensor_cores(batch, q_len, num_qo_heads, num_kv_heads, max_pages, num_sms)) {
    plan.tensor_cores = 1;
    plan.pages_per_chunk = max_pages;
    return plan;
  }
  int s;
  if (requested > 0) {
    s = requested;
  } else {
    const long long units = static_cast<long long>(batch) * num_kv_heads * head_blocks;
    const long long slots = static_cast<long long>(std::max(num_sms, 1)) * sa::decode_ctas_per_sm();
    if ((col_blocks == 1 || q_len == 1) && units >= slots) {
      // at least a wave of (request, KV head) CTAs: whole requests, which the
      // kernel dispatches heaviest first, unless a request is very long
      s = std::max(1, ceil_div(max_pages, kMaxChunkPages));
    } else if (col_blocks == 1) {
      s = static_cast<int>(std::min<long long>((kWavesTarget * slots + units - 1) / std::max(units, 1ll),
                                               1 << 20));
    } else {
      // a CTA with two column blocks does twice the work per page, which
      // makes the kernel throughput-bound: fewer, longer chunks (measured)
      s = static_cast<int>(std::min<long long>(kVerifyWavesTarget * slots / std::max(units, 1ll),
                                               1 << 20));
      s = std::max(s, ceil_div(max_pages, kMaxChunkPages));
    }
    s = std::min(s, std::max(1, max_pages / kMinPagesPerChunk));
  }
  s = std::max(1, std::min({s, sa::decode_max_splits(), max_pages}));
  plan.pages_per_chunk = ceil_div(max_pages, s);
  plan.num_splits = ceil_div(max_pages, plan.pages_per_chunk);
  {
    const long long units = static_cast<long long>(batch) * num_kv_heads * head_blocks;
    const long long slots = static_cast<long long>(std::max(num_sms, 1)) * sa::decode_ctas_per_sm();
    plan.sorted_dispatch = plan.num_splits == 1 && units <= kSortedWaves * slots;
  }
  if (plan.num_splits > 1) {
    const size_t units = static_cast<size_t>(batch) * num_kv_heads * head_blocks;
    plan.counters_bytes = (units * sizeof(int) + 255) & ~size_t(255);
    const size_t rows = static_cast<size_t>(plan.num_splits) * batch * q_len * num_qo_heads;
    plan.workspace_bytes = plan.counters_bytes + rows * kHeadDim * sizeof(float) +
                           ((rows * sizeof(float) + 255) & ~size_t(255));
  }
  return plan;
}

}  // namespace

namespace sa {
std::atomic<int> g_programmatic{0};

// Launch mode of one call: its own flag, else the process-wide default.
bool programmatic_for(int launch_flags) {
  if (launch_flags == SINKATTN_LAUNCH_PROGRAMMATIC) return true;
  if (launch_flags == SINKATTN_LAUNCH_PLAIN) return false;
  return g_programmatic.load(std::memory_order_relaxed) != 0;
}

}  // namespace sa

extern "C" {

const char *sinkattn_status_string(int status) {
  switch (status) {
    case SINKATTN_OK: return "ok";
    case SINKATTN_INVALID_ARGUMENT: return "invalid argument";
    case SINKATTN_UNSUPPORTED: return "unsupported configuration";
    case SINKATTN_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SINKATTN_CUDA_ERROR: return "CUDA error";
    default: return "unknown status";
  }
}

int sinkattn_version(void) { return 400; }   // 0.4.0: launch mode per call

int sinkattn_set_programmatic_launch(int enable) {
  return sa::g_programmatic.exchange(enable != 0 ? 1 : 0);
}

size_t sinkattn_decode_workspace_bytes(int batch, int num_qo_heads, int head_dim, int num_splits) {
  if (batch <= 0 || num_qo_heads <= 0 || head_dim != kHeadDim || num_splits <= 1) return 0;
  // counters: one int per (request, KV head, 8-head block) <= one per
  // (request, query head), whatever the KV head count; then the chunk slots
  const size_t counters = (static_cast<size_t>(batch) * num_qo_heads * sizeof(int) + 255) &
                          ~size_t(255);
  const size_t rows = static_cast<size_t>(num_splits) * batch * num_qo_heads;
  return counters + rows * kHeadDim * sizeof(float) + ((rows * sizeof(float) + 255) & ~size_t(255));
}

const char *sinkattn_last_error(void) { return g_last_error; }

int sinkattn_decode_plan(int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                         int max_kv_len, int num_sms, int *num_splits, size_t *workspace_bytes) {
  if (!num_splits || !workspace_bytes) return SINKATTN_INVALID_ARGUMENT;
  if (head_dim != kHeadDim || page_size != kPageSize) return SINKATTN_UNSUPPORTED;
  if (batch < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || max_kv_len < 0 || *num_splits < 0 ||
      num_sms < 0 || num_qo_heads % num_kv_heads)
    return SINKATTN_INVALID_ARGUMENT;
  if (num_sms == 0) {
    num_sms = device_sm_count();
    if (num_sms == 0) return fail_msg("no CUDA device to plan for");
  }
  const DecodePlan plan = plan_decode(batch, 1, num_qo_heads, num_kv_heads, max_kv_len, num_sms, *num_splits);
  *num_splits = plan.num_splits;
  *workspace_bytes = plan.workspace_bytes;
  return SINKATTN_OK;
}

int sinkattn_verify_plan(int batch, int q_len, int num_qo_heads, int num_kv_heads, int head_dim,
                         int page_size, int max_kv_len, int num_sms, int *num_splits,
                         size_t *workspace_bytes) {
  if (!num_splits || !workspace_bytes) return SINKATTN_INVALID_ARGUMENT;
  if (head_dim != kHeadDim || page_size != kPageSize) return SINKATTN_UNSUPPORTED;
  if (batch < 0 || q_len < 1 || q_len > SINKATTN_MAX_VERIFY_TOKENS || num_qo_heads <= 0 ||
      num_kv_heads <= 0 || max_kv_len < 0 || *num_splits < 0 || num_sms < 0 ||
      num_qo_heads % num_kv_heads)
    return SINKATTN_INVALID_ARGUMENT;
  if (num_sms == 0) {
    num_sms = device_sm_count();
    if (num_sms == 0) return fail_msg("no CUDA device to plan for");
  }
  const DecodePlan plan = plan_decode(batch, q_len, num_qo_heads, num_kv_heads, max_kv_len, num_sms,
                                      *num_splits);
  *num_splits = plan.num_splits;
  *workspace_bytes = plan.workspace_bytes;
  return SINKATTN_OK;
}

}  // extern "C"

namespace sa {

// Decode of q_len tokens per request; q_len = 1 with no mask is plain decode.
int decode_entry(const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                 const uint64_t *tree_mask, const float *sinks, float scale, void *out, float *lse,
                 int batch, int q_len, int num_qo_heads, int num_kv_heads, int head_dim,
                 int page_size, int num_pages, int max_kv_len, int num_splits, void *workspace,
                 size_t workspace_bytes, int launch_flags, bool zero_counters, void *stream) {
  if (launch_flags != SINKATTN_LAUNCH_DEFAULT && launch_flags != SINKATTN_LAUNCH_PLAIN &&
      launch_flags != SINKATTN_LAUNCH_PROGRAMMATIC)
    return SINKATTN_INVALID_ARGUMENT;
  if (head_dim != kHeadDim || page_size != kPageSize) return SINKATTN_UNSUPPORTED;
  if (batch < 0 || q_len < 1 || q_len > SINKATTN_MAX_VERIFY_TOKENS || num_qo_heads <= 0 ||
      num_kv_heads <= 0 || num_qo_heads % num_kv_heads || max_kv_len < 0 || num_splits < 0 ||
      num_pages <= 0 || max_pages_per_seq <= 0 || !std::isfinite(scale))
    return SINKATTN_INVALID_ARGUMENT;
  if (batch == 0) return SINKATTN_OK;
  if (!q || !k_cache || !v_cache || !page_table || !kv_lens || !sinks || !out)
    return SINKATTN_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(kv_lens, 4) || !aligned(sinks, 4) ||
      (lse && !aligned(lse, 4)) || (tree_mask && !aligned(tree_mask, 8)))
    return SINKATTN_INVALID_ARGUMENT;
  const int group = num_qo_heads / num_kv_heads;
  {
    // the plan falls back to 8-row CTAs only when the 16-row ones number
    // fewer than the GPU's CTA slots, far below this limit
    int col_blocks, head_blocks;
    decode_blocks(q_len, group, &col_blocks, &head_blocks);
    if (batch > 65535 || static_cast<long long>(num_kv_heads) * head_blocks > 65535)
      return SINKATTN_UNSUPPORTED;
  }

  const int sms = device_sm_count();
  if (sms == 0) return fail_msg("no CUDA device (SM count query failed)");
  const DecodePlan plan = plan_decode(batch, q_len, num_qo_heads, num_kv_heads, max_kv_len, sms,
                                      num_splits);
  const int col_blocks = plan.col_blocks, head_blocks = plan.head_blocks;
  if (plan.num_splits > 1) {
    if (!workspace || workspace_bytes < plan.workspace_bytes) return SINKATTN_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 256)) return SINKATTN_INVALID_ARGUMENT;
  }
  const bool programmatic = programmatic_for(launch_flags);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (plan.tensor_cores) {
    // query rows (token, head) of a KV head: box {64, group, 128 / group}
    CUtensorMap qmap, kmap, vmap;
    const unsigned long long rows = static_cast<unsigned long long>(num_kv_heads) * kPageSize;
    if (!encode_map(&qmap, q, num_qo_heads, static_cast<unsigned long long>(batch) * q_len, group,
                    kPrefillTile / group) ||
        !encode_map(&kmap, k_cache, rows, num_pages, kPageSize, 1) ||
        !encode_map(&vmap, v_cache, rows, num_pages, kPageSize, 1))
      return fail_msg("cuTensorMapEncodeTiled failed");
    sa::PrefillParams pp{};
    pp.q = static_cast<const uint16_t *>(q);
    pp.page_table = page_table;
    pp.kv_lens = kv_lens;
    pp.sinks = sinks;
    pp.out = static_cast<uint16_t *>(out);
    pp.lse = lse;
    pp.scale_log2 = scale * sa::kLog2e;
    pp.num_seqs = batch;
    pp.total_q = batch * q_len;
    pp.max_q_len = q_len;
    pp.max_kv_len = max_kv_len;
    pp.num_qo_heads = num_qo_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.group = group;
    pp.max_pages_per_seq = max_pages_per_seq;
    pp.num_pages = num_pages;
    pp.paged = 1;
    pp.num_q_tiles = ceil_div(q_len, kPrefillTile / group);
    pp.verify = 1;
    pp.tree_mask = tree_mask;
    return cuda_status(launch_prefill(qmap, kmap, vmap, pp, st, programmatic),
                       "verification launch");
  }

  CUtensorMap kmap, vmap;
  const unsigned long long rows = static_cast<unsigned long long>(num_kv_heads) * kPageSize;
  if (!encode_rows_map(&kmap, k_cache, rows, num_pages, kPageSize) ||
      !encode_rows_map(&vmap, v_cache, rows, num_pages, kPageSize))
    return fail_msg("cuTensorMapEncodeTiled failed");

  sa::DecodeParams p{};
  p.q = static_cast<const uint16_t *>(q);
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.tree_mask = tree_mask;
  p.sinks = sinks;
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  if (plan.num_splits > 1) {
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    p.counters = reinterpret_cast<int *>(ws);
    p.ws_o = reinterpret_cast<float *>(ws + plan.counters_bytes);
    p.ws_lse = p.ws_o + static_cast<size_t>(plan.num_splits) * batch * q_len * num_qo_heads * kHeadDim;
  }
  p.scale_log2 = scale * sa::kLog2e;
  p.max_pages_per_seq = max_pages_per_seq;
  p.batch = batch;
  p.q_len = q_len;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.rows = q_len * group;
  p.col_blocks = col_blocks;
  p.head_blocks = head_blocks;
  p.num_pages = num_pages;
  p.num_splits = plan.num_splits;
  p.pages_per_chunk = plan.pages_per_chunk;
  p.sorted_dispatch = plan.sorted_dispatch;
  if (zero_counters && plan.num_splits > 1) {
    // the counters are the workspace's first plan.counters_bytes bytes, all
    // within workspace_bytes (checked above)
    const cudaError_t e = cudaMemsetAsync(workspace, 0, plan.counters_bytes, st);
    if (e != cudaSuccess) return cuda_status(e, "merge counter clear");
  }
  return cuda_status(launch_decode(kmap, vmap, p, st, programmatic), "decode launch");
}

}  // namespace sa

extern "C" {

int sinkattn_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                    const float *sinks, float scale, void *out, float *lse, int batch,
                    int num_qo_heads, int num_kv_heads, int head_dim, int page_size, int num_pages,
                    int max_kv_len, int num_splits, void *workspace, size_t workspace_bytes,
                    void *stream) {
  return sa::decode_entry(q, k_cache, v_cache, page_table, max_pages_per_seq, kv_lens, nullptr,
                         sinks, scale, out, lse, batch, 1, num_qo_heads, num_kv_heads, head_dim,
                         page_size, num_pages, max_kv_len, num_splits, workspace, workspace_bytes,
                         SINKATTN_LAUNCH_DEFAULT, false, stream);
}

int sinkattn_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                       const float *sinks, float scale, void *out, float *lse, int batch,
                       int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                       int num_pages, int max_kv_len, int num_splits, void *workspace,
                       size_t workspace_bytes, int launch_flags, void *stream) {
  return sa::decode_entry(q, k_cache, v_cache, page_table, max_pages_per_seq, kv_lens, nullptr,
                         sinks, scale, out, lse, batch, 1, num_qo_heads, num_kv_heads, head_dim,
                         page_size, num_pages, max_kv_len, num_splits, workspace, workspace_bytes,
                         launch_flags, false, stream);
}

int sinkattn_verify(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                    const uint64_t *tree_mask, const float *sinks, float scale, void *out,
                    float *lse, int batch, int q_len, int num_qo_heads, int num_kv_heads,
                    int head_dim, int page_size, int num_pages, int max_kv_len, int num_splits,
                    void *workspace, size_t workspace_bytes, void *stream) {
  return sa::decode_entry(q, k_cache, v_cache, page_table, max_pages_per_seq, kv_lens, tree_mask,
                         sinks, scale, out, lse, batch, q_len, num_qo_heads, num_kv_heads,
                         head_dim, page_size, num_pages, max_kv_len, num_splits, workspace,
                         workspace_bytes, SINKATTN_LAUNCH_DEFAULT, false, stream);
}

int sinkattn_verify_ex(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                       const uint64_t *tree_mask, const float *sinks, float scale, void *out,
                       float *lse, int batch, int q_len, int num_qo_heads, int num_kv_heads,
                       int head_dim, int page_size, int num_pages, int max_kv_len, int num_splits,
                       void *workspace, size_t workspace_bytes, int launch_flags, void *stream) {
  return sa::decode_entry(q, k_cache, v_cache, page_table, max_pages_per_seq, kv_lens, tree_mask,
                         sinks, scale, out, lse, batch, q_len, num_qo_heads, num_kv_heads,
                         head_dim, page_size, num_pages, max_kv_len, num_splits, workspace,
                         workspace_bytes, launch_flags, false, stream);
}

int sinkattn_prefill(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                     int num_seqs, int total_tokens, int max_seqlen, const float *sinks,
                     float scale, void *out, float *lse, int num_qo_heads, int num_kv_heads,
                     int head_dim, void *stream) {
  if (head_dim != kHeadDim) return SINKATTN_UNSUPPORTED;
  if (num_seqs < 0 || total_tokens < 0 || max_seqlen < 0 || num_qo_heads <= 0 ||
      num_kv_heads <= 0 || num_qo_heads % num_kv_heads || !std::isfinite(scale))
    return SINKATTN_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return SINKATTN_OK;
  if (!q || !k || !v || !cu_seqlens || !sinks || !out) return SINKATTN_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens, 4) || !aligned(sinks, 4) || (lse && !aligned(lse, 4)))
    return SINKATTN_INVALID_ARGUMENT;
  CUtensorMap qmap, kmap, vmap;
  if (!encode_map(&qmap, q, num_qo_heads, total_tokens, 1, kPrefillTile) ||
      !encode_map(&kmap, k, num_kv_heads, total_tokens, 1, kPrefillKvTile) ||
      !encode_map(&vmap, v, num_kv_heads, total_tokens, 1, kPrefillKvTile))
    return fail_msg("cuTensorMapEncodeTiled failed");
  sa::PrefillParams p{};
  p.q = static_cast<const uint16_t *>(q);
  p.cu_seqlens_q = cu_seqlens;
  p.cu_seqlens_k = cu_seqlens;
  p.sinks = sinks;
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.scale_log2 = scale * sa::kLog2e;
  p.num_seqs = num_seqs;
  p.total_q = total_tokens;
  p.total_k = total_tokens;
  p.max_q_len = max_seqlen;
  p.max_kv_len = max_seqlen;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_qo_heads / num_kv_heads;
  p.paged = 0;
  p.num_q_tiles = ceil_div(max_seqlen, kPrefillTile);
  return cuda_status(sa::launch_prefill(qmap, kmap, vmap, p, static_cast<cudaStream_t>(stream),
                                        false),
                     "prefill launch");
}

int sinkattn_prefill_paged(const void *q, const int32_t *cu_seqlens_q, int num_seqs, int total_q,
                           int max_q_len, const void *k_cache, const void *v_cache,
                           const int32_t *page_table, int max_pages_per_seq,
                           const int32_t *kv_lens, int num_pages, int max_kv_len,
                           const float *sinks, float scale, void *out, float *lse,
                           int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
                           void *stream) {
  if (head_dim != kHeadDim || page_size != kPageSize) return SINKATTN_UNSUPPORTED;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || max_kv_len < 0 || num_qo_heads <= 0 ||
      num_kv_heads <= 0 || num_qo_heads % num_kv_heads || num_pages <= 0 ||
      max_pages_per_seq <= 0 || !std::isfinite(scale))
    return SINKATTN_INVALID_ARGUMENT;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return SINKATTN_OK;
  if (!q || !cu_seqlens_q || !k_cache || !v_cache || !page_table || !kv_lens || !sinks || !out)
    return SINKATTN_INVALID_ARGUMENT;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(cu_seqlens_q, 4) || !aligned(page_table, 4) || !aligned(kv_lens, 4) ||
      !aligned(sinks, 4) || (lse && !aligned(lse, 4)))
    return SINKATTN_INVALID_ARGUMENT;
  CUtensorMap qmap, kmap, vmap;
  const unsigned long long rows = static_cast<unsigned long long>(num_kv_heads) * kPageSize;
  if (!encode_map(&qmap, q, num_qo_heads, total_q, 1, kPrefillTile) ||
      !encode_map(&kmap, k_cache, rows, num_pages, kPageSize, 1) ||
      !encode_map(&vmap, v_cache, rows, num_pages, kPageSize, 1))
    return fail_msg("cuTensorMapEncodeTiled failed");
  sa::PrefillParams p{};
  p.q = static_cast<const uint16_t *>(q);
  p.cu_seqlens_q = cu_seqlens_q;
  p.page_table = page_table;
  p.kv_lens = kv_lens;
  p.sinks = sinks;
  p.out = static_cast<uint16_t *>(out);
  p.lse = lse;
  p.scale_log2 = scale * sa::kLog2e;
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.max_q_len = max_q_len;
  p.max_kv_len = max_kv_len;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_qo_heads / num_kv_heads;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages;
  p.paged = 1;
  p.num_q_tiles = ceil_div(max_q_len, kPrefillTile);
  return cuda_status(sa::launch_prefill(qmap, kmap, vmap, p, static_cast<cudaStream_t>(stream),
                                        false),
                     "prefill launch");
}

int sinkattn_yarn_table(int head_dim, double base, double factor, double original_context,
                        double beta_fast, double beta_slow, float *inv_freq, float *mscale) {
  if (!inv_freq || !mscale || head_dim <= 0 || head_dim % 2 || !(base > 1.0) ||
      !(factor >= 1.0) || !(original_context > 0.0) || !(beta_fast > beta_slow) ||
      !std::isfinite(base) || !std::isfinite(factor) || !std::isfinite(original_context))
    return SINKATTN_INVALID_ARGUMENT;
  const double two_pi = 6.283185307179586476925286766559;
  for (int d = 0; d < head_dim / 2; ++d) {
    const double theta = std::pow(base, -2.0 * d / head_dim);
    const double turns = original_context * theta / two_pi;   // rotations over the original context
    double ramp = (turns - beta_slow) / (beta_fast - beta_slow);
    ramp = std::min(1.0, std::max(0.0, ramp));
    inv_freq[d] = static_cast<float>(theta * ramp + theta / factor * (1.0 - ramp));
  }
  *mscale = static_cast<float>(0.1 * std::log(factor) + 1.0);
  return SINKATTN_OK;
}

int sinkattn_qkv_prologue(const void *qkv, const void *bias, const int32_t *positions,
                          const int32_t *slot_mapping, const float *inv_freq, float mscale,
                          int rope_style, void *q_out, void *k_cache, void *v_cache,
                          int num_tokens, int num_qo_heads, int num_kv_heads, int head_dim,
                          int page_size, int num_pages, void *stream) {
  if (head_dim != kHeadDim || page_size != kPageSize) return SINKATTN_UNSUPPORTED;
  if (num_tokens < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || num_pages <= 0 ||
      (rope_style != SINKATTN_ROPE_HALF && rope_style != SINKATTN_ROPE_INTERLEAVED) ||
      !std::isfinite(mscale))
    return SINKATTN_INVALID_ARGUMENT;
  if (num_tokens == 0) return SINKATTN_OK;
  if (!qkv || !positions || !slot_mapping || !inv_freq || !q_out || !k_cache || !v_cache)
    return SINKATTN_INVALID_ARGUMENT;
  if (!aligned(qkv, 16) || (bias && !aligned(bias, 16)) || !aligned(q_out, 16) ||
      !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(positions, 4) ||
      !aligned(slot_mapping, 4))
    return SINKATTN_INVALID_ARGUMENT;
  if (static_cast<long long>(num_tokens) * (num_qo_heads + 2 * num_kv_heads) * 4 > 0x7fffffffll)
    return SINKATTN_UNSUPPORTED;
  sa::PrologueParams p{};
  p.qkv = static_cast<const uint16_t *>(qkv);
  p.bias = static_cast<const uint16_t *>(bias);
  p.positions = positions;
  p.slot_mapping = slot_mapping;
  p.q_out = static_cast<uint16_t *>(q_out);
  p.k_cache = static_cast<uint16_t *>(k_cache);
  p.v_cache = static_cast<uint16_t *>(v_cache);
  for (int i = 0; i < kHeadDim / 2; ++i) {
    if (!std::isfinite(inv_freq[i])) return SINKATTN_INVALID_ARGUMENT;
    p.inv_freq[i] = inv_freq[i];
  }
  p.mscale = mscale;
  p.num_tokens = num_tokens;
  p.num_qo_heads = num_qo_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_pages = num_pages;
  p.interleaved = rope_style == SINKATTN_ROPE_INTERLEAVED;
  return cuda_status(sa::launch_prologue(p, static_cast<cudaStream_t>(stream)), "prologue launch");
}

}  // extern "C"
