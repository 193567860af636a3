// Attention prologue: QKV bias, YaRN rotary position encoding of q and k,
// and the write of k and v into the paged KV cache, in one pass.
//
// Operation: "GPT-OSS on day 0" (Perplexity blog), model summary before the
// section "Attention: GQA with attention sinks" -- positions are encoded with
// YaRN (as in DeepSeek-V3) and the QKV projections have biases (as in
// Qwen 2).  The rotary frequencies arrive as a table (sinkattn_yarn_table
// builds it from the YaRN paper's NTK-by-parts rule); pair (x1, x2) of a head
// at position p with frequency f becomes
//     (x1 cos(pf) - x2 sin(pf), x2 cos(pf) + x1 sin(pf)) * mscale,
// pairs being (i, i + 32) (half layout) or (2i, 2i + 1) (interleaved).
//
// Design (GB300, HBM-bound, no contraction): a CTA takes 4 tokens (1 for
// batches of up to 4096 tokens, so that small batches spread over the SMs).  Its
// first threads compute cos/sin of the token's 32 angles once into shared
// memory: the angle p*f is carried as an exact two-float product (hi + lo,
// the low part from an FMA), sincosf of hi corrected to first order by lo, so
// large positions keep their phase to ~1e-7.  Then every thread takes one
// (token, head row, dims 8c..8c+7 and 8c+32..8c+39) item: two coalesced
// 16-byte loads, the bias added in fp32, the rotation in fp32, one rounding
// to bf16, and 16-byte stores to q_out or to the token's cache slot.
// Launched programmatically: it waits for the previous kernel on the stream
// before any memory access and lets the next one (the decode of the layer)
// start ranking its requests at once.

#include "kernels.cuh"
#include "ptx.cuh"

namespace sa {
namespace {

constexpr int kThreads = 256;
constexpr int kPairs = kHeadDim / 2;

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]), pack_bf16(f[4], f[5]),
                    pack_bf16(f[6], f[7]));
}

template <int kTok>                // tokens per CTA
__global__ void __launch_bounds__(kThreads)
prologue_kernel(const __grid_constant__ PrologueParams p) {
  __shared__ float2 cs[kTok][kPairs];          // (cos, sin) * mscale
  // A decode launched programmatically after this kernel may start its
  // request ranking now; it waits for this grid to finish before reading q
  // or the caches.
  launch_dependents();
  // This kernel is itself launched programmatically: it reads and writes
  // nothing before the previous kernel on the stream has finished, so only
  // its launch and set-up overlap that kernel's last CTAs.
  grid_dependency_wait();
  const int tok0 = blockIdx.x * kTok;
  for (int j = threadIdx.x; j < kTok * kPairs; j += kThreads) {
    const int tt = j / kPairs, i = j % kPairs;
    const int t = tok0 + tt;
    if (t >= p.num_tokens) continue;
    const float pos = static_cast<float>(p.positions[t]);
    const float f = p.inv_freq[i];
    const float hi = pos * f;
    const float lo = fmaf(pos, f, -hi);        // pos * f = hi + lo exactly
    float s, c;
    sincosf(hi, &s, &c);
    cs[tt][i] = make_float2((c - lo * s) * p.mscale, (s + lo * c) * p.mscale);
  }
  __syncthreads();

  const int rows = p.num_qo_heads + 2 * p.num_kv_heads;
  const int per_tok = rows * 4;
  const int row_elems = rows * kHeadDim;
  for (int item = threadIdx.x; item < kTok * per_tok; item += kThreads) {
    const int tt = item / per_tok;
    const int t = tok0 + tt;
    if (t >= p.num_tokens) break;              // items are ordered by token
    const int r = item % per_tok;
    const int h = r >> 2, c = r & 3;
    const size_t base = static_cast<size_t>(t) * row_elems + h * kHeadDim;
    float a[8], b[8];                          // dims 8c.. and 8c+32..
    unpack8(__ldg(reinterpret_cast<const uint4 *>(p.qkv + base + 8 * c)), a);
    unpack8(__ldg(reinterpret_cast<const uint4 *>(p.qkv + base + 8 * c + 32)), b);
    if (p.bias) {
      float ba[8], bb[8];
      unpack8(__ldg(reinterpret_cast<const uint4 *>(p.bias + h * kHeadDim + 8 * c)), ba);
      unpack8(__ldg(reinterpret_cast<const uint4 *>(p.bias + h * kHeadDim + 8 * c + 32)), bb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        a[e] += ba[e];
        b[e] += bb[e];
      }
    }
    const bool is_v = h >= p.num_qo_heads + p.num_kv_heads;
    if (!is_v) {
      if (!p.interleaved) {
        // pair 8c+e is (a[e], b[e])
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 w = cs[tt][8 * c + e];
          const float x1 = a[e], x2 = b[e];
          a[e] = x1 * w.x - x2 * w.y;
          b[e] = x2 * w.x + x1 * w.y;
        }
      } else {
        // pairs 4c+u are (a[2u], a[2u+1]); pairs 16+4c+u are (b[2u], b[2u+1])
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 wa = cs[tt][4 * c + u], wb = cs[tt][16 + 4 * c + u];
          const float a1 = a[2 * u], a2 = a[2 * u + 1];
          a[2 * u] = a1 * wa.x - a2 * wa.y;
          a[2 * u + 1] = a2 * wa.x + a1 * wa.y;
          const float b1 = b[2 * u], b2 = b[2 * u + 1];
          b[2 * u] = b1 * wb.x - b2 * wb.y;
          b[2 * u + 1] = b2 * wb.x + b1 * wb.y;
        }
      }
    }
    uint16_t *dst;
    if (h < p.num_qo_heads) {
      dst = p.q_out + (static_cast<size_t>(t) * p.num_qo_heads + h) * kHeadDim;
    } else {
      const int slot = p.slot_mapping[t];
      if (slot < 0 || slot / kPageSize >= p.num_pages) continue;   // no write
      const int kvh = is_v ? h - p.num_qo_heads - p.num_kv_heads : h - p.num_qo_heads;
      uint16_t *cache = is_v ? p.v_cache : p.k_cache;
      dst = cache + ((static_cast<size_t>(slot / kPageSize) * p.num_kv_heads + kvh) * kPageSize +
                     slot % kPageSize) * kHeadDim;
    }
    *reinterpret_cast<uint4 *>(dst + 8 * c) = pack8(a);
    *reinterpret_cast<uint4 *>(dst + 8 * c + 32) = pack8(b);
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams &p, cudaStream_t stream) {
  if (p.num_tokens <= 0) return cudaSuccess;
  if (p.num_tokens <= 4096)          // small batches: one token per CTA, more SMs busy
    return launch_kernel(prologue_kernel<1>, static_cast<unsigned>(p.num_tokens), kThreads, 0,
                         stream, true, p);
  return launch_kernel(prologue_kernel<4>, static_cast<unsigned>((p.num_tokens + 3) / 4), kThreads,
                       0, stream, true, p);
}

}  // namespace sa
