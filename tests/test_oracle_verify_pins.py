"""Pins of the oracle's draft-token verification (CPU only).

"Accelerating Sonar through speculation" (Perplexity blog): sections
"Target-Draft" and "MTP" verify the k + 1 newest tokens of a request in one
pass (bottom-right causal); section "EAGLE" verifies a tree of drafts with a
custom mask.  ``oracle.verify`` restricts the mask to the draft tokens.

* a hand-worked tree and chain example (tests/golden/hand_examples.json);
* causal verification equals the matching rows of the (pinned) paged extend
  and of a full causal prefill; one token equals decode;
* with sink = -inf a tree mask equals torch's scaled_dot_product_attention
  with the dense boolean mask; with finite sinks the exact sink identity
  out = out_plain * sigmoid(lse_plain - sink) holds against torch;
* a chain-shaped tree mask equals the causal default.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from test_oracle_pins import GOLDEN, _arr, _num, _scatter_pages  # noqa: F401


def _golden():
    import json
    with open(GOLDEN) as f:
        return json.load(f)["verify_tree"]


def test_hand_example_tree_and_chain():
    c = _golden()
    args = (_arr(c["q"]), _arr(c["k_pages"]), _arr(c["v_pages"]), np.array(c["page_table"]),
            c["kv_lens"], _arr(c["sinks"]), c["scale"])
    out, lse = oracle.verify(*args, tree_mask=np.array(c["tree_mask"]))
    np.testing.assert_allclose(out, _arr(c["tree_out"]), atol=1e-14)
    np.testing.assert_allclose(lse, _arr(c["tree_lse"]), atol=1e-14)
    out, lse = oracle.verify(*args)
    np.testing.assert_allclose(out, _arr(c["causal_out"]), atol=1e-14)
    np.testing.assert_allclose(lse, _arr(c["causal_lse"]), atol=1e-14)


def _request_set(rng, prefixes, q_len, hq, hkv, d=8, page=4):
    full = [p + q_len for p in prefixes]
    ks = [rng.standard_normal((n, hkv, d)) for n in full]
    vs = [rng.standard_normal((n, hkv, d)) for n in full]
    qs = [rng.standard_normal((n, hq, d)) for n in full]
    kc, vc, table = _scatter_pages(rng, ks, vs, page, hkv, d)
    return full, ks, vs, qs, kc, vc, table


def _random_tree(rng, q_len):
    """Ancestor-or-self masks of a random tree whose roots hang off the prefix."""
    parent = [-1] + [int(rng.integers(-1, u)) for u in range(1, q_len)]
    masks = []
    for u in range(q_len):
        bits, a = 0, u
        while a >= 0:
            bits |= 1 << a
            a = parent[a]
        masks.append(bits)
    return masks


@pytest.mark.parametrize("q_len", [2, 4])
def test_causal_verify_equals_extend_and_prefill(q_len):
    rng = np.random.default_rng(40 + q_len)
    hq, hkv = 4, 2
    prefixes = [0, 3, 9]
    full, ks, vs, qs, kc, vc, table = _request_set(rng, prefixes, q_len, hq, hkv)
    sinks = rng.normal(0, 2, hq)
    sinks[1] = -math.inf
    q_new = np.stack([x[p:] for x, p in zip(qs, prefixes)])          # [B, q_len, Hq, D]
    out, lse = oracle.verify(q_new, kc, vc, table, full, sinks, 0.2)
    cu_q = np.arange(len(prefixes) + 1) * q_len
    eo, el = oracle.prefill_paged(q_new.reshape(-1, hq, 8), cu_q, kc, vc, table, full, sinks, 0.2)
    np.testing.assert_allclose(out.reshape(-1, hq, 8), eo, atol=1e-13)
    np.testing.assert_allclose(lse.reshape(-1, hq), el, atol=1e-13)
    for r, p in enumerate(prefixes):
        po, pl = oracle.prefill(qs[r], ks[r], vs[r], [0, full[r]], sinks, 0.2)
        np.testing.assert_allclose(out[r], po[p:], atol=1e-13)
        np.testing.assert_allclose(lse[r], pl[p:], atol=1e-13)


def test_one_token_equals_decode():
    rng = np.random.default_rng(47)
    hq, hkv = 8, 2
    full, ks, vs, qs, kc, vc, table = _request_set(rng, [0, 5, 12], 1, hq, hkv)
    sinks = rng.normal(0, 2, hq)
    q1 = np.stack([x[-1:] for x in qs])                                # [B, 1, Hq, D]
    do, dl = oracle.decode(q1[:, 0], kc, vc, table, full, sinks, 0.3)
    for mask in (None, np.ones((3, 1), dtype=np.int64)):
        out, lse = oracle.verify(q1, kc, vc, table, full, sinks, 0.3, tree_mask=mask)
        np.testing.assert_array_equal(out[:, 0], do)
        np.testing.assert_array_equal(lse[:, 0], dl)


def _torch_masked(q, k, v, allowed, scale, hq, hkv):
    """Plain attention of one request with a dense boolean mask, from torch:
    q [n, Hq, D], k/v [L, Hkv, D], allowed [n, L] -> (out [n, Hq, D], lse [n, Hq])."""
    g = hq // hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, 0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, 0)
    m = torch.from_numpy(allowed)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, scale=scale)
    s = (scale * (tq @ tk.transpose(1, 2))).masked_fill(~m, -math.inf)
    return out.permute(1, 0, 2).numpy(), torch.logsumexp(s, dim=-1).T.numpy()


@pytest.mark.parametrize("q_len", [3, 7, 12])
def test_tree_mask_against_torch(q_len):
    rng = np.random.default_rng(50 + q_len)
    hq, hkv, d = 4, 2, 8
    prefixes = [0, 6, 13]
    full, ks, vs, qs, kc, vc, table = _request_set(rng, prefixes, q_len, hq, hkv, d)
    masks = np.array([_random_tree(rng, q_len) for _ in prefixes], dtype=np.int64)
    sinks = rng.normal(0, 2, hq)
    q_new = np.stack([x[p:] for x, p in zip(qs, prefixes)])
    plain_o, plain_l = oracle.verify(q_new, kc, vc, table, full, np.full(hq, -np.inf), 0.25,
                                     tree_mask=masks)
    out, lse = oracle.verify(q_new, kc, vc, table, full, sinks, 0.25, tree_mask=masks)
    for r, p in enumerate(prefixes):
        allowed = np.zeros((q_len, full[r]), dtype=bool)
        allowed[:, :p] = True
        for i in range(q_len):
            for u in range(q_len):
                allowed[i, p + u] = bool((int(masks[r, i]) >> u) & 1)
        to, tl = _torch_masked(q_new[r], ks[r], vs[r], allowed, 0.25, hq, hkv)
        np.testing.assert_allclose(plain_o[r], to, atol=1e-12)
        np.testing.assert_allclose(plain_l[r], tl, atol=1e-12)
        sig = 1.0 / (1.0 + np.exp(sinks[None, :] - tl))
        np.testing.assert_allclose(out[r], to * sig[..., None], atol=1e-12)
        np.testing.assert_allclose(lse[r], np.logaddexp(tl, sinks[None, :]), atol=1e-12)


def test_chain_mask_equals_causal_and_high_bits():
    rng = np.random.default_rng(61)
    hq, hkv, q_len = 4, 1, 5
    full, ks, vs, qs, kc, vc, table = _request_set(rng, [2, 7], q_len, hq, hkv)
    sinks = rng.normal(0, 1, hq)
    q_new = np.stack([x[p:] for x, p in zip(qs, [2, 7])])
    chain = np.array([[(2 << i) - 1 for i in range(q_len)]] * 2, dtype=np.int64)
    a = oracle.verify(q_new, kc, vc, table, full, sinks, 0.2)
    b = oracle.verify(q_new, kc, vc, table, full, sinks, 0.2, tree_mask=chain)
    # bits at or above q_len name no draft token and change nothing; bit 63
    # arrives as a negative int64
    c = oracle.verify(q_new, kc, vc, table, full, sinks, 0.2,
                      tree_mask=chain | np.int64(-(1 << 63)) | np.int64(1 << 40))
    for x, y in ((a, b), (a, c)):
        np.testing.assert_array_equal(x[0], y[0])
        np.testing.assert_array_equal(x[1], y[1])
