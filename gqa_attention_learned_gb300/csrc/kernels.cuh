// Internal interface between the C ABI layer (sinkattn_api.cu) and the
// kernel translation units.  Not installed; no torch types anywhere.
#pragma once

#include <atomic>
#include <utility>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

constexpr int kHeadDim = 64;

// Sets a kernel's dynamic shared memory limit once per device (the attribute
// belongs to the function on the current device); later calls are free.  One
// flag set per kernel: the kernel itself is the template argument.
template <auto kernel>
inline cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}
// Launches `kernel` on `stream`; with `programmatic` the launch may start while
// the previous kernel on the stream is still running (the kernel orders its
// dependent reads and writes after grid_dependency_wait).
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(Params...), unsigned grid, unsigned block,
                                 int smem, cudaStream_t stream, bool programmatic,
                                 Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kPageSize = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ----------------------------------------------------------------- decode
// Decode of q_len new tokens per request (q_len = 1: plain decode; q_len > 1:
// speculative verification, bottom-right causal or a tree mask over the
// request's last q_len keys).  The query rows of one KV head are ordered
// (token, head in group): row r -> token r / group, head kvh*group + r % group.
struct DecodeParams {
  const uint16_t *q;            // bf16 [B][q_len][Hq][64]
  const int32_t *page_table;    // [B][max_pages_per_seq]
  const int32_t *kv_lens;       // [B]
  const uint64_t *tree_mask;    // [B][q_len] or null (causal)
  const float *sinks;           // [Hq]
  uint16_t *out;                // bf16 [B][q_len][Hq][64]
  float *lse;                   // [B][q_len][Hq] or null
  int *counters;                // [B][Hkv * head_blocks], zero between calls (splits > 1)
  float *ws_o;                  // fp32 [splits][B][q_len][Hq][64] (splits > 1)
  float *ws_lse;                // fp32 [splits][B][q_len][Hq]     (base-2 lse)
  float scale_log2;             // scale * log2(e)
  int max_pages_per_seq;
  int batch, q_len, num_qo_heads, num_kv_heads, group;
  int rows;                     // q_len * group query rows per KV head
  int col_blocks;               // 8-row column blocks per CTA (1 or 2)
  int head_blocks;              // CTAs per (request, KV head, chunk) = ceil(rows / (8 col_blocks))
  int num_pages, num_splits, pages_per_chunk;
  int sorted_dispatch;          // one chunk per request: requests heaviest first
};

// Column blocks per CTA for q_len * group query rows per KV head.
inline int decode_col_blocks(int rows) { return rows > 8 ? 2 : 1; }

// Number of CTAs the decode kernel may keep resident per SM (for planning).
int decode_ctas_per_sm();
// Largest split count.
int decode_max_splits();

// `programmatic`: launch with the programmatic-serialization attribute (the
// kernel waits for the previous kernel on the stream before touching anything
// but kv_lens and the page table).
cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap,
                          const DecodeParams &p, cudaStream_t stream, bool programmatic);

// ---------------------------------------------------------------- prefill
struct PrefillParams {
  const uint16_t *q;             // bf16 [Tq][Hq][64]
  const int32_t *cu_seqlens_q;   // [n+1]
  const int32_t *cu_seqlens_k;   // [n+1] (contiguous K/V) or null (paged)
  const int32_t *page_table;     // paged K/V: [n][max_pages_per_seq]
  const int32_t *kv_lens;        // paged K/V: [n]
  const float *sinks;            // [Hq]
  uint16_t *out;                 // bf16 [Tq][Hq][64]
  float *lse;                    // [Tq][Hq] or null
  float scale_log2;
  int num_seqs, total_q, total_k, max_q_len, max_kv_len;
  int num_qo_heads, num_kv_heads, group;
  int max_pages_per_seq, num_pages;
  int paged;                     // 0: k/v [Tk][Hkv][64], 1: paged cache
  int num_q_tiles;               // query tiles per (request, head) -- per (request, KV head) when verifying
  // Verification (paged): every request has max_q_len tokens, the last of
  // its keys; the query rows of a KV head are its (token, head) pairs, q is
  // [num_seqs * max_q_len][Hq][64]; tree_mask [num_seqs][max_q_len] or null.
  int verify;
  const uint64_t *tree_mask;
};

// `programmatic` applies to verification launches only; prefill and extend
// always launch plainly.
cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p,
                           cudaStream_t stream, bool programmatic);

// --------------------------------------------------------------- prologue
struct PrologueParams {
  const uint16_t *qkv;           // bf16 [T][(Hq + 2 Hkv) * 64], q heads, then k, then v
  const uint16_t *bias;          // bf16 [(Hq + 2 Hkv) * 64] or null
  const int32_t *positions;      // [T]
  const int32_t *slot_mapping;   // [T]: page * 16 + slot; < 0 or past the pool: no write
  uint16_t *q_out;               // bf16 [T][Hq][64]
  uint16_t *k_cache, *v_cache;   // bf16 [num_pages][Hkv][16][64]
  float inv_freq[kHeadDim / 2];  // rotary angular frequencies
  float mscale;                  // magnitude factor on cos and sin
  int num_tokens, num_qo_heads, num_kv_heads, num_pages;
  int interleaved;               // 0: pairs (i, i + 32); 1: pairs (2i, 2i + 1)
};

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream);

// ------------------------------------------------------------ C ABI layer
// Decode / verification of q_len tokens per request, shared by
// sinkattn_decode[_ex], sinkattn_verify[_ex] and
// sinkattn_decode_static_scratch: every argument check, the split plan, then
// the launch.  launch_flags is one of SINKATTN_LAUNCH_*.  With zero_counters,
// a plan of more than one split first clears the workspace's merge counters
// on the stream (cudaMemsetAsync, queued only after every check has passed);
// a single-split plan touches no workspace at all.
int decode_entry(const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *page_table, int max_pages_per_seq, const int32_t *kv_lens,
                 const uint64_t *tree_mask, const float *sinks, float scale, void *out, float *lse,
                 int batch, int q_len, int num_qo_heads, int num_kv_heads, int head_dim,
                 int page_size, int num_pages, int max_kv_len, int num_splits, void *workspace,
                 size_t workspace_bytes, int launch_flags, bool zero_counters, void *stream);

}  // namespace sa
