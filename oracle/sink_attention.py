"""Float64 CPU oracle for GQA attention with a learned sink logit per query head.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only the test suite, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` use it.  It shares no code with the CUDA path and is slow on
purpose: every function is the plainest statement of what it computes.

Sources
-------
"GPT-OSS on day 0" (Perplexity blog, 2025-08-08):
  * section "Attention: GQA with attention sinks" -- every attention head has
    a pretrained sink parameter that enters the softmax;
  * section "Kernels for GPT-OSS / Sink Attention" -- the sink is an extra
    logit next to the Q.K products; the softmax is computed online with a
    running max m (normally started at -inf) and a running scale d (started at
    1); starting m at the head's sink makes the sink count in the softmax; when
    the KV sequence is cut into several blocks the sink goes into the first
    block only.
The extracted pages lost the two displayed formulas of that section.  The
reading taken here (the plainest one every surviving sentence supports):

    s_j   = scale * <q_h, k_{g(h), j}>          (sink is NOT scaled)
    M     = max(sink_h, max_j s_j)
    Z     = exp(sink_h - M) + sum_j exp(s_j - M)
    out_h = sum_j exp(s_j - M) * v_{g(h), j} / Z   (the sink has no value row)
    lse_h = M + ln Z                             (natural log, sink included)

with g(h) = floor(h / (Hq / Hkv)) (contiguous GQA groups).  Splits along the
KV length are combined by log-sum-exp; only the first split carries the sink.
"Accelerating Sonar through speculation" (Perplexity blog), section
"Inference with speculative decoding": KV lives in pages reserved per batch,
addressed through per-request page information.

Conventions (readings where the pages are silent):
  * a row with no visible key: out = 0, lse = sink (so lse = -inf if the sink
    is -inf);
  * sink = +inf is undefined and rejected; sink = -inf is plain attention;
  * causal alignment is bottom-right: query i of a request holding kv_len keys
    of which the last q_len are its own queries sees keys j <= kv_len - q_len + i.

Every function takes float64-convertible NumPy arrays and returns float64.
"""

import math

import numpy as np

NEG_INF = -math.inf


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _check_sinks(sinks):
    sinks = _f64(sinks)
    if np.any(np.isposinf(sinks)) or np.any(np.isnan(sinks)):
        raise ValueError("a sink of +inf or NaN has no defined attention output")
    return sinks


def kv_head_of(h, num_qo_heads, num_kv_heads):
    """GQA head map: query head h reads KV head floor(h / G), G = Hq / Hkv."""
    if num_qo_heads % num_kv_heads:
        raise ValueError("num_qo_heads must be a multiple of num_kv_heads")
    return h // (num_qo_heads // num_kv_heads)


def sink_attention(q, k, v, sink, scale, n_visible):
    """The definition, for one query head.

    q: [n, D] query rows; k, v: [L, D] keys/values of that head's KV head;
    sink: scalar logit; n_visible: [n] ints, row i sees keys 0 .. n_visible[i]-1.
    Returns (out [n, D], lse [n]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    sink = float(_check_sinks(sink))
    n_visible = np.asarray(n_visible, dtype=np.int64)
    n, d = q.shape
    length = k.shape[0]
    if np.any(n_visible < 0) or np.any(n_visible > length):
        raise ValueError("n_visible out of range")
    s = scale * (q @ k.T)                                     # [n, L]
    visible = np.arange(length)[None, :] < n_visible[:, None]
    s = np.where(visible, s, NEG_INF)
    row_max = s.max(axis=1) if length else np.full(n, NEG_INF)
    m = np.maximum(sink, row_max)                             # M per row
    out = np.zeros((n, d))
    lse = np.full(n, sink)
    live = np.isfinite(m)                                     # rows with any mass
    if np.any(live):
        ml = m[live]
        w = np.exp(s[live] - ml[:, None])                     # masked -> exp(-inf) = 0
        z = np.exp(sink - ml) + w.sum(axis=1)
        out[live] = (w @ v) / z[:, None]
        lse[live] = ml + np.log(z)
    return out, lse


def gather_paged_kv(cache, page_table, kv_len, kv_head, page_size):
    """Rows 0..kv_len-1 of one request's K (or V) for one KV head.

    cache: [num_pages, Hkv, page_size, D], anything indexable that returns
    values convertible to float64; token t lives in page
    page_table[t // page_size], slot t % page_size.
    """
    t = np.arange(kv_len)
    pages = np.asarray(page_table)[t // page_size]
    return _f64(cache[pages, kv_head, t % page_size])


def decode(q, k_cache, v_cache, page_table, kv_lens, sinks, scale):
    """One new query token per request against its paged KV.

    q: [B, Hq, D]; k_cache, v_cache: [num_pages, Hkv, P, D];
    page_table: [B, max_pages]; kv_lens: [B]; sinks: [Hq].
    Returns out [B, Hq, D], lse [B, Hq].
    """
    q = _f64(q)
    sinks = _check_sinks(sinks)
    batch, hq, d = q.shape
    hkv, page_size = k_cache.shape[1], k_cache.shape[2]
    out = np.zeros((batch, hq, d))
    lse = np.zeros((batch, hq))
    for b in range(batch):
        n = int(kv_lens[b])
        for kvh in range(hkv):
            k = gather_paged_kv(k_cache, page_table[b], n, kvh, page_size)
            v = gather_paged_kv(v_cache, page_table[b], n, kvh, page_size)
            for h in range(hq):
                if kv_head_of(h, hq, hkv) != kvh:
                    continue
                o, l = sink_attention(q[b, h][None], k, v, sinks[h], scale, [n])
                out[b, h], lse[b, h] = o[0], l[0]
    return out, lse


def prefill(q, k, v, cu_seqlens, sinks, scale, rows=None, q_block=128):
    """Causal self-attention over ragged sequences packed along the token axis.

    q: [T, Hq, D]; k, v: [T, Hkv, D]; cu_seqlens: [n+1] prefix sums.
    rows: optional iterable of global token indices to compute (others stay 0);
    used to sample outputs of very large cases.  Query blocks only bound the
    memory of the score matrix; they do not change what is computed.
    Returns out [T, Hq, D], lse [T, Hq].
    """
    q, sinks = _f64(q), _check_sinks(sinks)
    total, hq, d = q.shape
    hkv = k.shape[1]
    out = np.zeros((total, hq, d))
    lse = np.zeros((total, hq))
    wanted = None if rows is None else np.zeros(total, dtype=bool)
    if wanted is not None:
        wanted[np.asarray(list(rows), dtype=np.int64)] = True
    cu = [int(x) for x in cu_seqlens]
    for i in range(len(cu) - 1):
        start, end = cu[i], cu[i + 1]
        local = np.arange(end - start)
        if wanted is not None:
            local = local[wanted[start:end]]
        for kvh in range(hkv):
            ks = _f64(k[start:end, kvh])
            vs = _f64(v[start:end, kvh])
            for h in range(hq):
                if kv_head_of(h, hq, hkv) != kvh:
                    continue
                for j in range(0, len(local), q_block):
                    r = local[j:j + q_block]
                    o, l = sink_attention(q[start + r, h], ks[: r.max() + 1],
                                          vs[: r.max() + 1], sinks[h], scale, r + 1)
                    out[start + r, h], lse[start + r, h] = o, l
    return out, lse


def prefill_paged(q, cu_seqlens_q, k_cache, v_cache, page_table, kv_lens, sinks,
                  scale, rows=None, q_block=128):
    """New query tokens appended to a paged KV prefix (chunked prefill / extend).

    Request r owns queries cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1 and kv_lens[r]
    keys in the cache; its last q_len keys are the new tokens themselves.
    Query i (0-based within the request) sees keys j <= kv_len - q_len + i.
    Returns out [Tq, Hq, D], lse [Tq, Hq].
    """
    q, sinks = _f64(q), _check_sinks(sinks)
    total, hq, d = q.shape
    hkv, page_size = k_cache.shape[1], k_cache.shape[2]
    out = np.zeros((total, hq, d))
    lse = np.zeros((total, hq))
    wanted = None if rows is None else np.zeros(total, dtype=bool)
    if wanted is not None:
        wanted[np.asarray(list(rows), dtype=np.int64)] = True
    cu = [int(x) for x in cu_seqlens_q]
    for r in range(len(cu) - 1):
        start, end = cu[r], cu[r + 1]
        q_len, kv_len = end - start, int(kv_lens[r])
        if q_len > kv_len:
            raise ValueError("a request cannot have more new queries than keys")
        local = np.arange(q_len)
        if wanted is not None:
            local = local[wanted[start:end]]
        if len(local) == 0:
            continue
        for kvh in range(hkv):
            ks = gather_paged_kv(k_cache, page_table[r], kv_len, kvh, page_size)
            vs = gather_paged_kv(v_cache, page_table[r], kv_len, kvh, page_size)
            for h in range(hq):
                if kv_head_of(h, hq, hkv) != kvh:
                    continue
                for j in range(0, len(local), q_block):
                    i = local[j:j + q_block]
                    o, l = sink_attention(q[start + i, h], ks, vs, sinks[h], scale,
                                          kv_len - q_len + i + 1)
                    out[start + i, h], lse[start + i, h] = o, l
    return out, lse


def verify(q, k_cache, v_cache, page_table, kv_lens, sinks, scale, tree_mask=None):
    """Verification of draft tokens: the q_len newest tokens of every request.

    "Accelerating Sonar through speculation" (Perplexity blog): sections
    "Target-Draft" and "MTP" run the target over the k + 1 newest tokens of a
    request at once (bottom-right causal); section "EAGLE" verifies a tree of
    drafts, which needs a custom mask.  Here the mask covers the draft tokens
    only: query i of request b sees every key j < kv_len - q_len, and draft key
    kv_len - q_len + u when u <= i (tree_mask None) or when bit u of
    tree_mask[b][i] is set.

    Written as a gather: each row's visible keys are collected explicitly and
    handed to the definition above.
    q: [B, q_len, Hq, D]; tree_mask: None or [B, q_len] integers (uint64 bit
    patterns; negative int64 values are read modulo 2**64).
    Returns out [B, q_len, Hq, D], lse [B, q_len, Hq].
    """
    q, sinks = _f64(q), _check_sinks(sinks)
    batch, q_len, hq, d = q.shape
    hkv, page_size = k_cache.shape[1], k_cache.shape[2]
    out = np.zeros((batch, q_len, hq, d))
    lse = np.zeros((batch, q_len, hq))
    for b in range(batch):
        kv_len = int(kv_lens[b])
        prefix = kv_len - q_len
        if prefix < 0:
            raise ValueError("a request cannot have more new queries than keys")
        for kvh in range(hkv):
            k_all = gather_paged_kv(k_cache, page_table[b], kv_len, kvh, page_size)
            v_all = gather_paged_kv(v_cache, page_table[b], kv_len, kvh, page_size)
            for i in range(q_len):
                if tree_mask is None:
                    seen = [u for u in range(q_len) if u <= i]
                else:
                    bits = int(tree_mask[b][i]) % (1 << 64)
                    seen = [u for u in range(q_len) if (bits >> u) & 1]
                keys = np.concatenate([np.arange(prefix), prefix + np.array(seen, dtype=np.int64)])
                k, v = k_all[keys], v_all[keys]
                for h in range(hq):
                    if kv_head_of(h, hq, hkv) != kvh:
                        continue
                    o, l = sink_attention(q[b, i, h][None], k, v, sinks[h], scale, [len(keys)])
                    out[b, i, h], lse[b, i, h] = o[0], l[0]
    return out, lse


# --------------------------------------------------------------------------
# The pages' own algorithm: the online softmax, one key at a time, over KV
# blocks, with the sink only in the first block, then a log-sum-exp merge.
# --------------------------------------------------------------------------

def online_block(q, k, v, scale, sink_or_none):
    """Online softmax over one block of keys, in the order the pages give.

    State (m, d, o) starts at m = sink (first block) or -inf (other blocks),
    d = 1, o = 0.  For each key: m' = max(m, s); d <- d*e^(m-m') + e^(s-m');
    o <- o*e^(m-m') + e^(s-m') v; m <- m'.  The block's normalised result is
    (o / d, m + ln d).  e^(m-m') is taken as 0 while m is still -inf.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    m = NEG_INF if sink_or_none is None else float(sink_or_none)
    d = 1.0
    o = np.zeros(q.shape[0])
    for j in range(k.shape[0]):
        s = scale * float(q @ k[j])
        m_new = max(m, s)
        a = 0.0 if m == NEG_INF else math.exp(m - m_new)
        e = math.exp(s - m_new)
        d = d * a + e
        o = o * a + e * v[j]
        m = m_new
    if m == NEG_INF:          # nothing entered this block
        return np.zeros_like(o), NEG_INF
    return o / d, m + math.log(d)


def merge_blocks(parts):
    """Log-sum-exp merge of normalised block results [(out_c, lse_c), ...]."""
    lses = [l for _, l in parts]
    top = max(lses)
    if top == NEG_INF:
        return np.zeros_like(parts[0][0]), NEG_INF
    total = sum(math.exp(l - top) for l in lses if l != NEG_INF)
    lse = top + math.log(total)
    out = sum(math.exp(l - lse) * o for o, l in parts if l != NEG_INF)
    return out, lse


def split_sink_attention(q, k, v, sink, scale, bounds, sink_in_every_block=False):
    """One query row over keys cut at `bounds` (0 = b_0 < ... < b_C = L).

    The sink enters block 0 only, unless sink_in_every_block is set (a wrong
    variant kept for negative tests).  Returns (out [D], lse).
    """
    parts = []
    for c in range(len(bounds) - 1):
        lo, hi = bounds[c], bounds[c + 1]
        s = sink if (c == 0 or sink_in_every_block) else None
        if s is not None and s == NEG_INF:
            s = None
        parts.append(online_block(q, k[lo:hi], v[lo:hi], scale, s))
    return merge_blocks(parts)
