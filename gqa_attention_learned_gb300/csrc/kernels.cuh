// Internal interface between the C ABI layer (sinkattn_api.cu) and the
// kernel translation units.  Not installed; no torch types anywhere.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sa {

constexpr int kHeadDim = 64;
constexpr int kPageSize = 16;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ----------------------------------------------------------------- decode
struct DecodeParams {
  const uint16_t *q;            // bf16 [B][Hq][64]
  const int32_t *page_table;    // [B][max_pages_per_seq]
  const int32_t *kv_lens;       // [B]
  const float *sinks;           // [Hq]
  uint16_t *out;                // bf16 [B][Hq][64]
  float *lse;                   // [B][Hq] or null
  int *counters;                // [B * Hkv * head_blocks], zero between calls
  float *ws_o;                  // fp32 [2 * num_workers][8][64] chunk outputs
  float *ws_lse;                // fp32 [2 * num_workers][8] chunk lse (base 2)
  float scale_log2;             // scale * log2(e)
  int max_pages_per_seq;
  int batch, num_qo_heads, num_kv_heads, group, head_blocks;
  int num_pages, num_workers;
};

// Resident decode CTAs per SM, warps per CTA, requests per launch.
int decode_ctas_per_sm();
int decode_warps_per_cta();
int decode_max_batch();
size_t decode_smem_bytes(int batch, int num_qo_heads);
// Bytes at the start of the decode workspace that must be zero before a call.
size_t decode_counter_bytes(int batch, int num_qo_heads, int num_kv_heads);

cudaError_t launch_decode(const CUtensorMap &kmap, const CUtensorMap &vmap, const DecodeParams &p,
                          int grid, cudaStream_t stream);

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
  int num_q_tiles;               // ceil(max_q_len / tile)
};

cudaError_t launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p,
                           cudaStream_t stream);

}  // namespace sa
