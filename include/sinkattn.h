/*
 * sinkattn.h -- C ABI of libsinkattn: GQA attention with a learned sink logit
 * per query head, for NVIDIA GB300 (sm_103a).
 *
 * The operation ("GPT-OSS on day 0", Perplexity blog, section "Kernels for
 * GPT-OSS / Sink Attention"; the page's displayed formulas were lost, this is
 * the plainest reading of the surviving text): for query head h with KV head
 * g(h) = h / (num_qo_heads / num_kv_heads) and the keys j it may see,
 *
 *     s_j   = scale * dot(q_h, k_{g(h),j})           (the sink is not scaled)
 *     M     = max(sink_h, max_j s_j)
 *     Z     = exp(sink_h - M) + sum_j exp(s_j - M)
 *     out_h = sum_j exp(s_j - M) * v_{g(h),j} / Z     (the sink has no value row)
 *     lse_h = M + ln Z                                (natural log, sink included)
 *
 * A row that sees no key gets out = 0, lse = sink.  sink = -inf is ordinary
 * softmax attention; sink = +inf or NaN is undefined (the output is NaN).
 * Work is split along the KV length the way the same section describes: the
 * online softmax of the first KV block starts at max = sink, scale = 1; the
 * other blocks start at max = -inf; blocks are merged by log-sum-exp.
 *
 * Conventions shared by every entry point
 *   - bf16 = IEEE bfloat16 stored as uint16; all tensors are dense, row-major,
 *     in device memory, 16-byte aligned, and owned by the caller.
 *   - head_dim must be 64 and page_size 16 (else SINKATTN_UNSUPPORTED).
 *   - num_qo_heads % num_kv_heads == 0; the GQA group is contiguous.
 *   - Paged KV cache ("Accelerating Sonar through speculation", Perplexity
 *     blog, section "Inference with speculative decoding": KV pages are
 *     reserved per request and addressed through per-request page lists):
 *       k_cache, v_cache : bf16 [num_pages][num_kv_heads][page_size][head_dim]
 *       page_table       : int32 [batch][max_pages_per_seq]; token t of
 *                          request b is slot t % page_size of page
 *                          page_table[b][t / page_size].
 *     Only the first ceil(kv_len / page_size) entries of a row are read.  A
 *     page id outside [0, num_pages), kv_len < 0, or a kv_len that does not fit
 *     the row or the declared maximum makes that request's outputs NaN; no
 *     memory outside the given buffers is touched.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream), never synchronises, allocates nothing, and keeps no
 *     state beyond per-device caches (the SM count, kernel attributes set
 *     once) and the process-wide default launch mode of
 *     sinkattn_set_programmatic_launch, which the _ex entry points override
 *     per call.  Calls are thread-safe.
 *   - Return value: a sinkattn_status.  Argument checks happen on the host
 *     before any launch; SINKATTN_CUDA_ERROR reports a launch failure.
 */
#ifndef SINKATTN_H
#define SINKATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SINKATTN_API __attribute__((visibility("default")))
#else
#define SINKATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sinkattn_status {
  SINKATTN_OK = 0,
  SINKATTN_INVALID_ARGUMENT = 1,   /* null/misaligned pointer, bad size */
  SINKATTN_UNSUPPORTED = 2,        /* head_dim != 64, page_size != 16, ... */
  SINKATTN_WORKSPACE_TOO_SMALL = 3,
  SINKATTN_CUDA_ERROR = 4
} sinkattn_status;

/* Static description of a status code. */
SINKATTN_API const char *sinkattn_status_string(int status);

/* Detail of the last SINKATTN_CUDA_ERROR returned on the calling thread
 * (the CUDA error name and where it happened); "" if none. */
SINKATTN_API const char *sinkattn_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
SINKATTN_API int sinkattn_version(void);

/*
 * Launch modes of the decode and verification kernels, chosen per call by
 * the launch_flags argument of sinkattn_decode_ex and sinkattn_verify_ex:
 *   SINKATTN_LAUNCH_DEFAULT       the process-wide default below
 *   SINKATTN_LAUNCH_PLAIN         an ordinary launch: the kernel starts after
 *                                 everything before it on the stream
 *   SINKATTN_LAUNCH_PROGRAMMATIC  programmatic dependent launch (below)
 * Any other value returns SINKATTN_INVALID_ARGUMENT without launching.
 */
#define SINKATTN_LAUNCH_DEFAULT 0
#define SINKATTN_LAUNCH_PLAIN 1
#define SINKATTN_LAUNCH_PROGRAMMATIC 2

/*
 * Programmatic dependent launch of the decode and verification kernels
 * (sinkattn_decode, sinkattn_decode_static_scratch, both routes of
 * sinkattn_verify, and the _ex entry points given SINKATTN_LAUNCH_DEFAULT;
 * prefill is unaffected).  This sets the process-wide DEFAULT, off at load;
 * returns the previous setting.  A caller that shares the process with other
 * users of the library should pass its mode per call (the _ex entry points)
 * instead of changing the default.  In programmatic mode a kernel may be scheduled
 * while the kernel launched before it on the same stream is still running:
 * its CTAs rank the requests (kv_lens), read their first page ids
 * (page_table) and set up shared and tensor memory, then wait for the
 * earlier kernel to finish before they read q, the caches, sinks or
 * tree_mask and before they write out, lse or the workspace; they let the
 * next kernel on the stream be scheduled only after that wait.  The
 * prologue kernel (sinkattn_qkv_prologue) lets such a kernel be scheduled
 * as soon as all of its own CTAs have started.
 * Caller's contract while it is on: kv_lens and page_table of a call are not
 * written by the kernel launched immediately before the call on its stream
 * (they may come from host copies, memsets or any earlier kernel).  A
 * violation is not detected: the kernel may read the old kv_lens or page
 * table.  Launches inside CUDA graph capture keep the same ordering.
 */
SINKATTN_API int sinkattn_set_programmatic_launch(int enable);

/*
 * Split plan for sinkattn_decode (host only, no launch).
 *   num_sms          : SMs to plan for; 0 = ask the current CUDA device.
 *   num_splits       : in = requested number of KV chunks per (request, KV
 *                      head) (0 = choose), out = the count sinkattn_decode
 *                      will use (at most one page per chunk).
 *   workspace_bytes  : out = bytes of workspace that decode needs (0 when the
 *                      plan has a single split).
 * Same inputs give the same plan, so the plan can be made once and reused
 * (e.g. under CUDA graph capture); max_kv_len is a host-side bound, so no
 * device-to-host read is needed.
 */
SINKATTN_API int sinkattn_decode_plan(int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                         int page_size, int max_kv_len, int num_sms,
                         int *num_splits, size_t *workspace_bytes);

/*
 * Upper bound on the workspace sinkattn_decode needs with an explicit split
 * count num_splits, for any num_kv_heads that divides num_qo_heads and any
 * kv lengths (host only).  The merge counters take at most one int per
 * (request, query head), 256-byte rounded; each split then holds an fp32 row
 * of head_dim and an fp32 lse per (request, query head), the lse block
 * 256-byte rounded.  Returns 0 for num_splits <= 1 (no workspace), for
 * batch <= 0 or num_qo_heads <= 0, and for head_dim != 64.  The plan may use
 * fewer splits than requested (at most one page per chunk), never more, so
 * the bound always suffices; sinkattn_decode_plan gives the exact figure,
 * including the split count that num_splits = 0 (choose) leads to.
 */
SINKATTN_API size_t sinkattn_decode_workspace_bytes(int batch, int num_qo_heads, int head_dim,
                                        int num_splits);

/*
 * Decode: one new query token per request against its paged KV.
 *   q          : bf16 [batch][num_qo_heads][head_dim]
 *   k_cache,
 *   v_cache    : bf16 paged cache (see conventions), num_pages pages
 *   page_table : int32 [batch][max_pages_per_seq]
 *   kv_lens    : int32 [batch], keys per request (0 allowed)
 *   sinks      : fp32 [num_qo_heads], in natural-log logit units
 *   scale      : softmax scale applied to q.k
 *   out        : bf16 [batch][num_qo_heads][head_dim]
 *   lse        : fp32 [batch][num_qo_heads] (natural log, sink included);
 *                may be NULL
 *   max_kv_len : host-side upper bound on kv_lens (drives the split plan)
 *   num_splits : 0 = choose (see sinkattn_decode_plan), else the number of
 *                KV chunks per (request, KV head)
 *   workspace  : device scratch of workspace_bytes (>= the plan's figure),
 *                256-byte aligned; may be NULL when the plan has a single
 *                split.  It must be ZERO-FILLED BEFORE ITS FIRST USE; every
 *                call leaves it ready for the next (its merge counters return
 *                to zero), so it is zeroed once, not per call.  Calls sharing
 *                a workspace must not overlap on the GPU.
 * Long contexts run as num_splits KV chunks per (request, KV head), the sink
 * entering chunk 0 only; the last chunk to finish merges them by
 * log-sum-exp inside the same kernel.
 * Query heads of a KV head go to CTAs 8 at a time, or 16 at a time when a
 * KV head has more than 8 (a GQA group above 8), so each CTA reads each page
 * once for all of its heads.
 * Limits: batch <= 65535, and num_kv_heads times the CTAs per KV head
 * (ceil(group / 16) for groups above 8, else 1) <= 65535; larger calls return
 * SINKATTN_UNSUPPORTED without launching.
 */
SINKATTN_API int sinkattn_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq,
                    const int32_t *kv_lens, const float *sinks, float scale,
                    void *out, float *lse,
                    int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                    int page_size, int num_pages, int max_kv_len, int num_splits,
                    void *workspace, size_t workspace_bytes, void *stream);

/* sinkattn_decode with the launch mode chosen by this call (launch_flags =
 * SINKATTN_LAUNCH_*), whatever the process-wide default. */
SINKATTN_API int sinkattn_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq,
                    const int32_t *kv_lens, const float *sinks, float scale,
                    void *out, float *lse,
                    int batch, int num_qo_heads, int num_kv_heads, int head_dim,
                    int page_size, int num_pages, int max_kv_len, int num_splits,
                    void *workspace, size_t workspace_bytes, int launch_flags,
                    void *stream);

/*
 * Verification of draft tokens ("Accelerating Sonar through speculation",
 * Perplexity blog: sections "Target-Draft" and "MTP" run the target model
 * over the q_len = k + 1 newest tokens of every request in one pass --
 * single-token MTP verifies 2 per request -- and section "EAGLE" verifies a
 * tree of drafts, which needs a custom attention mask).  Every request has
 * exactly q_len new tokens, already written as the LAST q_len keys of its
 * paged KV.  Query token i (0-based) of request b sees
 *   - every key j < kv_len - q_len (the accepted prefix), and
 *   - draft key kv_len - q_len + u for u in [0, q_len) when
 *       tree_mask == NULL : u <= i                 (causal, aligned at the end)
 *       tree_mask != NULL : bit u of tree_mask[b][i] is set
 *     (a token sees itself only if its own bit is set).
 * The mask covers the draft tokens only, so the prefix costs no mask work.
 *   q          : bf16 [batch][q_len][num_qo_heads][head_dim]
 *   tree_mask  : uint64 [batch][q_len], 8-byte aligned, or NULL
 *   out        : bf16 [batch][q_len][num_qo_heads][head_dim]
 *   lse        : fp32 [batch][q_len][num_qo_heads]; may be NULL
 *   q_len      : 1 .. SINKATTN_MAX_VERIFY_TOKENS
 *   other arguments, the split plan (sinkattn_verify_plan) and the workspace
 *   rules: as for sinkattn_decode.  kv_len < q_len makes the request's rows
 *   NaN.  q_len = 1 with tree_mask = NULL computes what sinkattn_decode does.
 * Kernel choice (host-side sizes only, so a plan can be reused): with
 * num_splits = 0, at least 24 query rows per KV head (q_len times the group
 * size, which must divide 128), max_kv_len <= 8192 and enough (request, KV
 * head) pairs to fill the GPU once, the rows of a KV head run on the tensor
 * cores (tcgen05) in one pass over its keys; the plan then reports one split
 * and no workspace.  Otherwise the split-KV kernel of sinkattn_decode runs.
 */
#define SINKATTN_MAX_VERIFY_TOKENS 64

SINKATTN_API int sinkattn_verify_plan(int batch, int q_len, int num_qo_heads, int num_kv_heads,
                         int head_dim, int page_size, int max_kv_len, int num_sms,
                         int *num_splits, size_t *workspace_bytes);

SINKATTN_API int sinkattn_verify(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq,
                    const int32_t *kv_lens, const uint64_t *tree_mask,
                    const float *sinks, float scale, void *out, float *lse,
                    int batch, int q_len, int num_qo_heads, int num_kv_heads,
                    int head_dim, int page_size, int num_pages, int max_kv_len,
                    int num_splits, void *workspace, size_t workspace_bytes,
                    void *stream);

/* sinkattn_verify with the launch mode chosen by this call (launch_flags =
 * SINKATTN_LAUNCH_*), whatever the process-wide default. */
SINKATTN_API int sinkattn_verify_ex(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *page_table, int max_pages_per_seq,
                    const int32_t *kv_lens, const uint64_t *tree_mask,
                    const float *sinks, float scale, void *out, float *lse,
                    int batch, int q_len, int num_qo_heads, int num_kv_heads,
                    int head_dim, int page_size, int num_pages, int max_kv_len,
                    int num_splits, void *workspace, size_t workspace_bytes,
                    int launch_flags, void *stream);

/*
 * Causal prefill over ragged sequences packed along the token axis.
 *   q          : bf16 [total_tokens][num_qo_heads][head_dim]
 *   k, v       : bf16 [total_tokens][num_kv_heads][head_dim]
 *   cu_seqlens : int32 [num_seqs + 1], prefix sums of sequence lengths,
 *                cu_seqlens[num_seqs] == total_tokens
 *   max_seqlen : host-side upper bound on any sequence length
 *   out        : bf16 [total_tokens][num_qo_heads][head_dim]
 *   lse        : fp32 [total_tokens][num_qo_heads]; may be NULL
 * Query i of a sequence sees keys 0..i of the same sequence.  A sequence
 * longer than max_seqlen, or cu_seqlens that are not non-decreasing within
 * [0, total_tokens], gives NaN rows for the offending sequence.
 */
SINKATTN_API int sinkattn_prefill(const void *q, const void *k, const void *v,
                     const int32_t *cu_seqlens, int num_seqs, int total_tokens,
                     int max_seqlen, const float *sinks, float scale,
                     void *out, float *lse,
                     int num_qo_heads, int num_kv_heads, int head_dim, void *stream);

/*
 * Chunked prefill ("extend"): new query tokens appended to a paged KV prefix.
 * Request r owns queries cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1 and kv_lens[r]
 * keys in the paged cache; its last q_len keys are its own new tokens (already
 * written to the cache).  Query i (0-based within the request) sees keys
 * j <= kv_len - q_len + i (causal, aligned at the end).
 *   q          : bf16 [total_q][num_qo_heads][head_dim]
 *   out, lse   : as for prefill, [total_q]-major
 *   max_q_len, max_kv_len : host-side bounds
 * q_len > kv_len, or any bound exceeded, gives NaN rows for that request.
 */
SINKATTN_API int sinkattn_prefill_paged(const void *q, const int32_t *cu_seqlens_q, int num_seqs,
                           int total_q, int max_q_len,
                           const void *k_cache, const void *v_cache,
                           const int32_t *page_table, int max_pages_per_seq,
                           const int32_t *kv_lens, int num_pages, int max_kv_len,
                           const float *sinks, float scale, void *out, float *lse,
                           int num_qo_heads, int num_kv_heads, int head_dim,
                           int page_size, void *stream);

/*
 * Attention prologue ("GPT-OSS on day 0", Perplexity blog, model summary
 * before section "Attention: GQA with attention sinks": YaRN position
 * encoding as in DeepSeek-V3, QKV projections with biases as in Qwen 2).
 *
 * sinkattn_yarn_table (host only): rotary angular frequencies of the
 * head_dim / 2 pairs and the magnitude factor, after the YaRN paper (Peng et
 * al., 2023, "NTK-by-parts" and the attention temperature): pair d has
 * theta_d = base^(-2d / head_dim) and r_d = original_context * theta_d / (2 pi)
 * rotations over the original context; with ramp g = clamp((r_d - beta_slow)
 * / (beta_fast - beta_slow), 0, 1) its frequency is
 * g * theta_d + (1 - g) * theta_d / factor; mscale = 0.1 ln(factor) + 1.
 * factor = 1 gives plain rotary frequencies and mscale = 1.  The pages give
 * no parameter values.
 *   inv_freq : host float [head_dim / 2] (out);  mscale : host float (out)
 */
SINKATTN_API int sinkattn_yarn_table(int head_dim, double base, double factor,
                        double original_context, double beta_fast, double beta_slow,
                        float *inv_freq, float *mscale);

/*
 * sinkattn_qkv_prologue: one pass over the QKV projection output of
 * num_tokens tokens:
 *   x = qkv[t] + bias (fp32), split into num_qo_heads q rows, num_kv_heads k
 *   rows, num_kv_heads v rows of head_dim;
 *   q and k rows rotated: pair (x1, x2) of pair index i at position p becomes
 *   (x1 cos(p f_i) - x2 sin(p f_i), x2 cos(p f_i) + x1 sin(p f_i)) * mscale;
 *   q_out[t] = bf16(rotated q); k and v written (bf16, round to nearest
 *   even, once) to page slot_mapping[t] / page_size, slot
 *   slot_mapping[t] % page_size of k_cache / v_cache.
 *   qkv          : bf16 [num_tokens][(num_qo_heads + 2 num_kv_heads) * head_dim]
 *   bias         : bf16 [(num_qo_heads + 2 num_kv_heads) * head_dim] or NULL
 *   positions    : int32 [num_tokens] (exact below 2^24)
 *   slot_mapping : int32 [num_tokens]; an entry < 0 or at or past
 *                  num_pages * page_size writes no k/v for that token
 *   inv_freq     : HOST float [head_dim / 2] (copied into the launch, so the
 *                  call can be captured in a CUDA graph); mscale as above
 *   rope_style   : SINKATTN_ROPE_HALF (pairs (i, i + head_dim/2)) or
 *                  SINKATTN_ROPE_INTERLEAVED (pairs (2i, 2i + 1))
 *   q_out        : bf16 [num_tokens][num_qo_heads][head_dim]
 *   k_cache, v_cache : the paged cache (see conventions), num_pages pages
 * Two tokens mapped to the same slot race (one of them wins).
 * Launch: always programmatic, whatever the default above.  The kernel reads
 * and writes nothing before the kernel launched before it on the stream has
 * finished (so it puts no contract on the caller); only its launch and set-up
 * overlap that kernel's last CTAs.  It lets a programmatically launched decode
 * or verification after it be scheduled at once.
 */
#define SINKATTN_ROPE_HALF 0
#define SINKATTN_ROPE_INTERLEAVED 1

SINKATTN_API int sinkattn_qkv_prologue(const void *qkv, const void *bias,
                          const int32_t *positions, const int32_t *slot_mapping,
                          const float *inv_freq, float mscale, int rope_style,
                          void *q_out, void *k_cache, void *v_cache,
                          int num_tokens, int num_qo_heads, int num_kv_heads,
                          int head_dim, int page_size, int num_pages, void *stream);

/*
 * Decode for callers that cannot allocate device memory.
 *
 * Some callers of this library cannot call cudaMalloc at the point where they
 * run decode: code running inside another allocator's critical section,
 * plug-ins hosted by a runtime that owns all device memory, or tools that
 * must not change the process's memory footprint.  For them this entry point
 * takes the same arguments as sinkattn_decode minus the workspace: the split
 * scratch lives in one fixed array of SINKATTN_STATIC_SCRATCH_BYTES (16 MiB)
 * of device memory that is part of the library itself, so every GPU that
 * loads the library holds that array until the process exits.  The pages
 * this library follows have no counterpart to this call; it only changes
 * where the scratch memory comes from.
 *
 *   - Allocates nothing: no cudaMalloc/cudaFree, no allocating library call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture on the device.
 *   - Every argument check of sinkattn_decode runs first; a refused call
 *     queues no work on the stream.  Returns SINKATTN_WORKSPACE_TOO_SMALL,
 *     launching nothing, when the plan for these sizes (see
 *     sinkattn_decode_plan) needs more scratch than the array holds.
 *   - A plan with one split (num_splits = 1, or a chosen plan that keeps
 *     whole requests) neither reads nor writes the array.
 *   - All calls share the one array, and it keeps the last call's contents.
 *     A call whose plan has more than one split first clears the part that
 *     must start at zero (the merge counters, with cudaMemsetAsync on
 *     `stream`); two such calls that overlap on the GPU (different streams,
 *     or different host threads, without ordering between them) race on the
 *     array and may return wrong results.
 *   - The launch mode is the process-wide default
 *     (sinkattn_set_programmatic_launch).
 */
#define SINKATTN_STATIC_SCRATCH_BYTES (16u << 20)

SINKATTN_API int sinkattn_decode_static_scratch(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *page_table,
    int max_pages_per_seq, const int32_t *kv_lens, const float *sinks, float scale, void *out,
    float *lse, int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
    int num_pages, int max_kv_len, int num_splits, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H */
