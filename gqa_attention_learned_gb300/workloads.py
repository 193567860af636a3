"""Seeded synthetic inputs shaped like gpt-oss attention layers.

This module only draws random numbers and lays them out (contiguous ragged
tensors, a shuffled paged KV pool); it holds none of the attention arithmetic,
so both the CUDA path and the float64 oracle can be fed from it.

Every array is drawn in float32 with NumPy's PCG64 generator (stable across
NumPy versions), then rounded once to bfloat16 (round to nearest even) where
the kernel takes bfloat16.  All tensors are CPU tensors; callers move them.

Paged KV layout: ``[num_pages, num_kv_heads, page_size, head_dim]`` -- each
(page, KV head) is one contiguous page_size x head_dim tile.  The pool holds
25% spare pages; spare pages and the unused tail slots of every request's last
page are filled with NaN so that a kernel reading a key it must not see shows
up as NaN.  Unused page-table entries point at a spare (NaN) page.
"""

import math

import numpy as np
import torch

HEAD_DIM = 64
PAGE_SIZE = 16


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def gpt_oss_sinks(rng, num_qo_heads, std=2.0, special=True):
    """Sinks ~ N(0, std); with `special`, heads h = 0 (mod 16) get -inf and
    heads h = 1 (mod 16) get +8 (a sink that dominates the softmax)."""
    s = _normal(rng, (num_qo_heads,), std)
    if special:
        s[0::16] = -np.inf
        s[1::16] = 8.0
    return torch.from_numpy(s.astype(np.float32))


def paged_pool(rng, kv_lens, num_kv_heads, head_dim=HEAD_DIM, page_size=PAGE_SIZE,
               spare_frac=0.25, contents=None):
    """Build a shuffled paged K/V pool holding kv_lens[b] tokens per request.

    contents: optional list of (k [L_b, Hkv, D], v [L_b, Hkv, D]) float32
    arrays to place instead of fresh N(0,1) draws.
    Returns dict(k_cache, v_cache, page_table, kv_lens, num_pages).
    """
    kv_lens = [int(x) for x in kv_lens]
    pages_per = [math.ceil(n / page_size) for n in kv_lens]
    used = sum(pages_per)
    num_pages = used + max(1, math.ceil(spare_frac * used))
    perm = rng.permutation(num_pages)
    spare = int(perm[-1])                      # never assigned to a request
    max_pages = max(1, max(pages_per) if pages_per else 1)
    table = np.full((len(kv_lens), max_pages), spare, dtype=np.int32)
    k_cache = torch.full((num_pages, num_kv_heads, page_size, head_dim), float("nan"),
                         dtype=torch.bfloat16)
    v_cache = torch.full_like(k_cache, float("nan"))
    cursor = 0
    for b, n in enumerate(kv_lens):
        p = pages_per[b]
        ids = perm[cursor:cursor + p]
        cursor += p
        table[b, :p] = ids
        if n == 0:
            continue
        if contents is None:
            kb = _normal(rng, (n, num_kv_heads, head_dim))
            vb = _normal(rng, (n, num_kv_heads, head_dim))
        else:
            kb, vb = contents[b]
        for src, cache in ((kb, k_cache), (vb, v_cache)):
            padded = np.full((p * page_size, num_kv_heads, head_dim), np.nan, np.float32)
            padded[:n] = src
            tiles = padded.reshape(p, page_size, num_kv_heads, head_dim).transpose(0, 2, 1, 3)
            cache[torch.from_numpy(ids.astype(np.int64))] = _bf16(tiles)
    return dict(k_cache=k_cache, v_cache=v_cache, page_table=torch.from_numpy(table),
                kv_lens=torch.tensor(kv_lens, dtype=torch.int32), num_pages=num_pages)


def tiny(seed=0):
    """Batch 1, 4 query heads over 1 KV head, head_dim 64, 37 tokens.

    Causal prefill over the 37 tokens plus one decode step whose query is the
    last token's query against the same 37 keys held in 3 shuffled pages."""
    rng = np.random.default_rng(seed)
    hq, hkv, length = 4, 1, 37
    q = _normal(rng, (length, hq, HEAD_DIM))
    k = _normal(rng, (length, hkv, HEAD_DIM))
    v = _normal(rng, (length, hkv, HEAD_DIM))
    sinks = torch.from_numpy(_normal(rng, (hq,)))
    pool = paged_pool(rng, [length], hkv, contents=[(k, v)])
    return dict(
        name="tiny", num_qo_heads=hq, num_kv_heads=hkv, head_dim=HEAD_DIM, scale=0.125,
        q=_bf16(q), k=_bf16(k), v=_bf16(v), sinks=sinks,
        cu_seqlens=torch.tensor([0, length], dtype=torch.int32),
        q_decode=_bf16(q[-1:]), **pool)


def decode_batch(seed=1, batch=64, num_qo_heads=64, num_kv_heads=8, min_len=1,
                 max_len=4096, sink_std=2.0, special_sinks=True):
    """gpt-oss-20b-shaped decode: one query per request, kv_len ~ U{min..max}."""
    rng = np.random.default_rng(seed)
    kv_lens = rng.integers(min_len, max_len + 1, size=batch)
    q = _bf16(_normal(rng, (batch, num_qo_heads, HEAD_DIM)))
    sinks = gpt_oss_sinks(rng, num_qo_heads, sink_std, special_sinks)
    pool = paged_pool(rng, kv_lens, num_kv_heads)
    return dict(name="decode", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, scale=0.125, q=q, sinks=sinks,
                max_kv_len=int(max(kv_lens)), **pool)


def long_decode(seed=2, batch=8, min_len=32768, max_len=131072):
    """Long-context decode that needs the split-KV path."""
    w = decode_batch(seed=seed, batch=batch, min_len=min_len, max_len=max_len,
                     special_sinks=False)
    w["name"] = "long_decode"
    return w


def ragged_prefill(seed=3, num_seqs=4, min_len=2048, max_len=8192, target=20000,
                   tolerance=0.10, num_qo_heads=64, num_kv_heads=8):
    """Causal prefill over ragged sequences whose total is target +- tolerance."""
    rng = np.random.default_rng(seed)
    while True:
        lens = rng.integers(min_len, max_len + 1, size=num_seqs)
        if abs(int(lens.sum()) - target) <= tolerance * target:
            break
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    q = _bf16(_normal(rng, (total, num_qo_heads, HEAD_DIM)))
    k = _bf16(_normal(rng, (total, num_kv_heads, HEAD_DIM)))
    v = _bf16(_normal(rng, (total, num_kv_heads, HEAD_DIM)))
    sinks = gpt_oss_sinks(rng, num_qo_heads, 2.0, special=False)
    return dict(name="prefill", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, scale=0.125, q=q, k=k, v=v, sinks=sinks,
                cu_seqlens=torch.from_numpy(cu), max_seqlen=int(lens.max()))


def custom_prefill(seqlens, seed=5, num_qo_heads=64, num_kv_heads=8, sink_std=2.0,
                   special_sinks=False):
    """Ragged causal prefill with the given sequence lengths (parity cases)."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
    total = int(cu[-1])
    q = _bf16(_normal(rng, (total, num_qo_heads, HEAD_DIM)))
    k = _bf16(_normal(rng, (total, num_kv_heads, HEAD_DIM)))
    v = _bf16(_normal(rng, (total, num_kv_heads, HEAD_DIM)))
    sinks = gpt_oss_sinks(rng, num_qo_heads, sink_std, special_sinks)
    return dict(name="prefill", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, scale=0.125, q=q, k=k, v=v, sinks=sinks,
                cu_seqlens=torch.from_numpy(cu), max_seqlen=int(max(seqlens) if len(seqlens) else 0))


def extend_batch(q_lens, prefix_lens, seed=6, num_qo_heads=64, num_kv_heads=8,
                 special_sinks=False):
    """Chunked prefill: request r appends q_lens[r] new tokens (already written
    to the paged cache) after prefix_lens[r] cached tokens."""
    rng = np.random.default_rng(seed)
    kv_lens = [int(a) + int(b) for a, b in zip(q_lens, prefix_lens)]
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _bf16(_normal(rng, (int(cu[-1]), num_qo_heads, HEAD_DIM)))
    sinks = gpt_oss_sinks(rng, num_qo_heads, 2.0, special_sinks)
    pool = paged_pool(rng, kv_lens, num_kv_heads)
    return dict(name="extend", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, scale=0.125, q=q, sinks=sinks,
                cu_seqlens_q=torch.from_numpy(cu), max_q_len=int(max(q_lens)),
                max_kv_len=int(max(kv_lens)), **pool)


def mixed_batch(seed=4, num_decode=32, num_extend=4, extend_len=2048,
                decode_range=(512, 16384), prefix_range=(0, 14336)):
    """Serving step: decode requests and chunked-prefill requests sharing one
    shuffled page pool.  Requests 0..num_decode-1 decode, the rest extend."""
    rng = np.random.default_rng(seed)
    hq, hkv = 64, 8
    dec_lens = rng.integers(decode_range[0], decode_range[1] + 1, size=num_decode)
    prefixes = rng.integers(prefix_range[0], prefix_range[1] + 1, size=num_extend)
    ext_lens = prefixes + extend_len
    sinks = gpt_oss_sinks(rng, hq, 2.0, special=False)
    pool = paged_pool(rng, list(dec_lens) + list(ext_lens), hkv)
    table = pool["page_table"]
    kv = pool["kv_lens"]
    q_dec = _bf16(_normal(rng, (num_decode, hq, HEAD_DIM)))
    q_ext = _bf16(_normal(rng, (num_extend * extend_len, hq, HEAD_DIM)))
    cu = torch.arange(0, num_extend + 1, dtype=torch.int32) * extend_len
    return dict(
        name="mixed", num_qo_heads=hq, num_kv_heads=hkv, head_dim=HEAD_DIM, scale=0.125,
        sinks=sinks, k_cache=pool["k_cache"], v_cache=pool["v_cache"],
        num_pages=pool["num_pages"],
        decode=dict(q=q_dec, page_table=table[:num_decode].contiguous(),
                    kv_lens=kv[:num_decode].contiguous(), max_kv_len=int(dec_lens.max())),
        extend=dict(q=q_ext, cu_seqlens_q=cu, page_table=table[num_decode:].contiguous(),
                    kv_lens=kv[num_decode:].contiguous(), max_q_len=extend_len,
                    max_kv_len=int(ext_lens.max())))


def random_tree_masks(rng, batch, q_len):
    """Draft trees for verification: node u > 0 hangs off a uniformly drawn
    earlier node or directly off the accepted prefix; node 0 hangs off the
    prefix.  Row i of a request holds the bits of i and of its ancestors
    (int64 [batch, q_len], bit patterns of uint64)."""
    masks = np.zeros((batch, q_len), dtype=np.uint64)
    for b in range(batch):
        parent = [-1] + [int(rng.integers(-1, u)) for u in range(1, q_len)]
        for u in range(q_len):
            bits, a = 0, u
            while a >= 0:
                bits |= 1 << a
                a = parent[a]
            masks[b, u] = bits
    return torch.from_numpy(masks.view(np.int64))


def verify_batch(seed=5, batch=64, q_len=4, num_qo_heads=64, num_kv_heads=8, min_len=1,
                 max_len=4096, tree=False, special_sinks=True, kv_lens_first=()):
    """Verification of q_len draft tokens per request (speculative decoding):
    the drafts are the last q_len keys of each request's paged KV, whose
    length is ~ U{max(min_len, q_len)..max_len}; with `tree`, each request
    carries a random draft tree's masks, else verification is causal.
    kv_lens_first: lengths that replace the drawn ones of the first requests
    (the pool is built for the final lengths)."""
    rng = np.random.default_rng(seed)
    kv_lens = rng.integers(max(min_len, q_len), max_len + 1, size=batch)
    for i, n in enumerate(kv_lens_first):
        kv_lens[i] = int(n)
    q = _bf16(_normal(rng, (batch, q_len, num_qo_heads, HEAD_DIM)))
    sinks = gpt_oss_sinks(rng, num_qo_heads, 2.0, special_sinks)
    masks = random_tree_masks(rng, batch, q_len) if tree else None
    pool = paged_pool(rng, kv_lens, num_kv_heads)
    return dict(name="verify", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, scale=0.125, q=q, q_len=q_len, sinks=sinks, tree_mask=masks,
                max_kv_len=int(max(kv_lens)), **pool)


def prologue_batch(seq_lens, start_positions, seed=6, num_qo_heads=64, num_kv_heads=8,
                   bias=True):
    """Projection outputs of new tokens for the attention prologue: request r
    appends seq_lens[r] tokens at positions start_positions[r] .. + len - 1
    to a shuffled paged pool that already holds its first start_positions[r]
    tokens.  qkv ~ N(0,1), bias ~ N(0, 0.5) (bf16); slot_mapping gives each
    new token's page * 16 + offset."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in seq_lens]
    starts = [int(x) for x in start_positions]
    heads = num_qo_heads + 2 * num_kv_heads
    total = sum(lens)
    qkv = _bf16(_normal(rng, (total, heads * HEAD_DIM)))
    b = _bf16(_normal(rng, (heads * HEAD_DIM,), 0.5)) if bias else None
    pool = paged_pool(rng, [s + n for s, n in zip(starts, lens)], num_kv_heads)
    table = pool["page_table"].numpy()
    positions, slots = [], []
    for r, (s, n) in enumerate(zip(starts, lens)):
        for p in range(s, s + n):
            positions.append(p)
            slots.append(int(table[r, p // PAGE_SIZE]) * PAGE_SIZE + p % PAGE_SIZE)
    return dict(name="prologue", num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                head_dim=HEAD_DIM, qkv=qkv, bias=b,
                positions=torch.tensor(positions, dtype=torch.int32),
                slot_mapping=torch.tensor(slots, dtype=torch.int32), **pool)
