"""Float64 CPU oracle for the attention prologue: QKV bias, YaRN rotary
position encoding of q and k, and the write of k and v into the paged cache.

TEST INFRASTRUCTURE ONLY (like the rest of this package): used by the test
suite and bench.py's CPU legs, never by the product path; it shares no code
with the CUDA path.

Sources
-------
"GPT-OSS on day 0" (Perplexity blog), section "Attention: GQA with attention
sinks" and the model summary before it: positions are encoded with YaRN
(as in DeepSeek-V3) and the QKV projections carry biases (as in Qwen 2).
The page gives no YaRN parameters and no pairing layout, so:
  * the frequency table follows the YaRN paper (Peng, Quesnelle, Fan,
    Shippole, "YaRN: Efficient Context Window Extension of Large Language
    Models", 2023), section "NTK-by-parts": pair d of a head of size D has
    the base angular frequency theta_d = base**(-2d/D), wavelength
    lambda_d = 2*pi / theta_d and r_d = L / lambda_d rotations over the
    original context L; with ramp gamma(r) = 0 for r < alpha, 1 for r > beta,
    (r - alpha) / (beta - alpha) between, the scaled frequency is
    (1 - gamma) * theta_d / s + gamma * theta_d for context factor s;
    section "Dynamic Scaling / YaRN": the attention temperature enters as a
    factor sqrt(1/t) = 0.1 ln(s) + 1 on both q and k;
  * a pair (x1, x2) at position p with frequency f becomes
    (x1 cos(p f) - x2 sin(p f), x2 cos(p f) + x1 sin(p f)), times that factor;
    pairs are (i, i + D/2) ("half" layout, the default) or (2i, 2i + 1)
    ("interleaved");
  * the bias is added before the rotation; v gets the bias and no rotation.
"""

import math

import numpy as np


def yarn_inv_freq(head_dim, base, factor, original_context, beta_fast, beta_slow):
    """YaRN-scaled angular frequencies [head_dim / 2] and the magnitude
    factor (float64).  factor = 1 gives the plain rotary frequencies and 1."""
    if head_dim % 2 or head_dim <= 0 or base <= 1 or factor < 1 or original_context <= 0:
        raise ValueError("bad rotary parameters")
    if not beta_fast > beta_slow:
        raise ValueError("beta_fast must exceed beta_slow")
    half = head_dim // 2
    freqs = np.empty(half)
    for d in range(half):
        theta = base ** (-2.0 * d / head_dim)
        rotations = original_context * theta / (2.0 * math.pi)     # L / lambda_d
        if rotations < beta_slow:
            gamma = 0.0
        elif rotations > beta_fast:
            gamma = 1.0
        else:
            gamma = (rotations - beta_slow) / (beta_fast - beta_slow)
        freqs[d] = (1.0 - gamma) * theta / factor + gamma * theta
    return freqs, 0.1 * math.log(factor) + 1.0


def pair_index(head_dim, style):
    """(first, second) element indices of the rotated pairs of one head."""
    half = head_dim // 2
    if style == "half":
        return np.arange(half), np.arange(half) + half
    if style == "interleaved":
        return 2 * np.arange(half), 2 * np.arange(half) + 1
    raise ValueError(style)


def rotate(x, positions, inv_freq, mscale, style="half"):
    """Rotary encoding of x [T, H, D] at positions [T] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    t, h, d = x.shape
    a, b = pair_index(d, style)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * np.asarray(inv_freq, np.float64)[None, :]
    c = (np.cos(ang) * mscale)[:, None, :]
    s = (np.sin(ang) * mscale)[:, None, :]
    out = np.empty_like(x)
    out[..., a] = x[..., a] * c - x[..., b] * s
    out[..., b] = x[..., b] * c + x[..., a] * s
    return out


def qkv_prologue(qkv, bias, positions, inv_freq, mscale, num_qo_heads, num_kv_heads,
                 style="half"):
    """Split the projection output qkv [T, (Hq + 2 Hkv) * D] into q, k, v,
    add the bias (same layout, or None), rotate q and k.
    Returns q [T, Hq, D], k [T, Hkv, D], v [T, Hkv, D] (float64)."""
    qkv = np.asarray(qkv, dtype=np.float64)
    t = qkv.shape[0]
    heads = num_qo_heads + 2 * num_kv_heads
    d = qkv.shape[1] // heads
    x = qkv.reshape(t, heads, d)
    if bias is not None:
        x = x + np.asarray(bias, dtype=np.float64).reshape(1, heads, d)
    q = rotate(x[:, :num_qo_heads], positions, inv_freq, mscale, style)
    k = rotate(x[:, num_qo_heads:num_qo_heads + num_kv_heads], positions, inv_freq, mscale, style)
    v = x[:, num_qo_heads + num_kv_heads:]
    return q, k, v


def scatter_to_cache(cache, values, slot_mapping, page_size):
    """Write values [T, Hkv, D] into a copy of cache [pages, Hkv, P, D]: token
    t goes to page slot_mapping[t] // P, slot slot_mapping[t] % P; a negative
    entry writes nothing."""
    out = np.array(cache, copy=True)
    for t, s in enumerate(np.asarray(slot_mapping)):
        if s < 0:
            continue
        out[s // page_size, :, s % page_size] = values[t]
    return out
