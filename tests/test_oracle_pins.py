"""Pins of the float64 oracle to things other than itself (CPU only).

* hand-worked examples (tests/golden/hand_examples.json);
* sink = -inf reduces to standard softmax attention: torch's
  scaled_dot_product_attention in float64, with KV heads repeated for GQA;
* the exact sink identity: out = out_plain * sigmoid(lse_plain - sink) and
  lse = logaddexp(lse_plain, sink), with out_plain/lse_plain from torch;
* the single-key closed form out = v * sigmoid(s - sink);
* sink -> +inf drives the output to 0;
* the pages' blockwise online softmax (sink in the first block only) plus a
  log-sum-exp merge equals the definition, brute-forced over split points;
  putting the sink in every block must NOT;
* probability mass sums to one; decode equals the last prefill row; a
  chunked-prefill request equals the matching rows of a full causal prefill.

Source: "GPT-OSS on day 0" (Perplexity blog), section "Kernels for GPT-OSS /
Sink Attention".
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _num(x):
    if isinstance(x, (int, float)):
        return float(x)
    table = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5),
             "ln6": math.log(6), "ln8": math.log(8), "-inf": -math.inf, "0": 0.0, "1": 1.0}
    if x in table:
        return table[x]
    num, den = x.split("/")
    return float(num) / float(den)


def _arr(x):
    if isinstance(x, list):
        return np.array([_arr(e) for e in x], dtype=np.float64)
    return _num(x)


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_hand_examples_attend(golden):
    for case in golden["attend"]:
        out, lse = oracle.sink_attention(_arr(case["q"]), _arr(case["k"]), _arr(case["v"]),
                                         _num(case["sink"]), case["scale"], case["n_visible"])
        np.testing.assert_allclose(out, _arr(case["out"]), rtol=0, atol=1e-14, err_msg=case["name"])
        np.testing.assert_allclose(lse, _arr(case["lse"]), rtol=0, atol=1e-14, err_msg=case["name"])


def test_hand_example_gqa_map(golden):
    c = golden["gqa"]
    q = _arr(c["q"])                          # [T=1, Hq, D]
    k = np.transpose(_arr(c["k"]), (1, 0, 2))  # given per KV head -> [T, Hkv, D]
    v = np.transpose(_arr(c["v"]), (1, 0, 2))
    # two key tokens, one query: treat as the last row of a 2-token causal prefill
    qq = np.concatenate([np.zeros_like(q), q])
    out, lse = oracle.prefill(qq, k, v, [0, 2], _arr(c["sinks"]), c["scale"])
    np.testing.assert_allclose(out[1:], _arr(c["out"]), atol=1e-14)
    np.testing.assert_allclose(lse[1:], _arr(c["lse"]), atol=1e-14)


def test_hand_example_paged_decode(golden):
    c = golden["paged_decode"]
    out, lse = oracle.decode(_arr(c["q"]), _arr(c["k_pages"]), _arr(c["v_pages"]),
                             np.array(c["page_table"]), c["kv_lens"], _arr(c["sinks"]), c["scale"])
    np.testing.assert_allclose(out, _arr(c["out"]), atol=1e-14)
    np.testing.assert_allclose(lse, _arr(c["lse"]), atol=1e-14)


def test_hand_example_split(golden):
    c = golden["split"]
    q, k, v = _arr(c["q"]), _arr(c["k"]), _arr(c["v"])
    b = c["bounds"]
    for i, blk in enumerate(c["blocks"]):
        o, l = oracle.online_block(q, k[b[i]:b[i + 1]], v[b[i]:b[i + 1]], c["scale"],
                                   _num(c["sink"]) if i == 0 else None)
        np.testing.assert_allclose(o, _arr(blk["out"]), atol=1e-14)
        assert abs(l - _num(blk["lse"])) < 1e-14
    out, lse = oracle.split_sink_attention(q, k, v, _num(c["sink"]), c["scale"], b)
    np.testing.assert_allclose(out, _arr(c["out"]), atol=1e-14)
    assert abs(lse - _num(c["lse"])) < 1e-14


# ---------------------------------------------------------------- torch pins

def _rand_prefill(rng, seqlens, hq, hkv, d=8):
    total = sum(seqlens)
    q = rng.standard_normal((total, hq, d))
    k = rng.standard_normal((total, hkv, d))
    v = rng.standard_normal((total, hkv, d))
    cu = np.concatenate([[0], np.cumsum(seqlens)])
    return q, k, v, cu


def _torch_plain(q, k, v, scale, hq, hkv, causal=True):
    """Standard attention for one sequence from torch: (out [L,Hq,D], lse [L,Hq])."""
    g = hq // hkv
    tq = torch.from_numpy(q).permute(1, 0, 2)                       # [Hq, L, D]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, 0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, 0)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    s = scale * (tq @ tk.transpose(1, 2))
    if causal:
        n = s.shape[-1]
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.T.numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 1), (8, 2), (6, 3), (4, 4)])
def test_no_sink_is_standard_attention(hq, hkv):
    rng = np.random.default_rng(10 + hq + hkv)
    seqlens = [5, 1, 17]
    q, k, v, cu = _rand_prefill(rng, seqlens, hq, hkv)
    scale = 0.3
    out, lse = oracle.prefill(q, k, v, cu, np.full(hq, -np.inf), scale)
    for i in range(len(seqlens)):
        a, b = cu[i], cu[i + 1]
        ref_o, ref_l = _torch_plain(q[a:b], k[a:b], v[a:b], scale, hq, hkv)
        np.testing.assert_allclose(out[a:b], ref_o, atol=1e-12)
        np.testing.assert_allclose(lse[a:b], ref_l, atol=1e-12)


def test_sink_identity_against_torch():
    hq, hkv = 8, 2
    rng = np.random.default_rng(21)
    q, k, v, cu = _rand_prefill(rng, [19], hq, hkv)
    sinks = rng.normal(0, 2, size=hq)
    sinks[3] = 8.0
    scale = 0.125
    out, lse = oracle.prefill(q, k, v, cu, sinks, scale)
    po, pl = _torch_plain(q, k, v, scale, hq, hkv)
    sig = 1.0 / (1.0 + np.exp(sinks[None, :] - pl))
    np.testing.assert_allclose(out, po * sig[..., None], atol=1e-12)
    np.testing.assert_allclose(lse, np.logaddexp(pl, sinks[None, :]), atol=1e-12)


def test_single_key_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(20):
        d = 16
        q, k, v = rng.standard_normal(d), rng.standard_normal(d), rng.standard_normal(d)
        sink, scale = rng.normal(0, 2), rng.uniform(0.05, 1)
        s = scale * sum(q[i] * k[i] for i in range(d))
        out, lse = oracle.sink_attention(q[None], k[None], v[None], sink, scale, [1])
        np.testing.assert_allclose(out[0], v / (1 + math.exp(sink - s)), atol=1e-13)
        assert abs(lse[0] - np.logaddexp(s, sink)) < 1e-13


def test_large_sink_drives_output_to_zero():
    rng = np.random.default_rng(4)
    q, k, v = rng.standard_normal((3, 8)), rng.standard_normal((9, 8)), rng.standard_normal((9, 8))
    out, lse = oracle.sink_attention(q, k, v, 1e3, 0.125, [9, 4, 1])
    assert np.all(np.abs(out) < 1e-300)
    np.testing.assert_allclose(lse, 1e3, rtol=0, atol=1e-12)


def test_plus_inf_sink_rejected():
    with pytest.raises(ValueError):
        oracle.sink_attention(np.zeros((1, 2)), np.zeros((1, 2)), np.zeros((1, 2)), math.inf, 1.0, [1])


def test_no_visible_keys():
    out, lse = oracle.sink_attention(np.ones((2, 4)), np.ones((3, 4)), np.ones((3, 4)), 0.7, 1.0, [0, 0])
    assert np.all(out == 0) and np.all(lse == 0.7)
    out, lse = oracle.sink_attention(np.ones((1, 4)), np.ones((3, 4)), np.ones((3, 4)), -math.inf, 1.0, [0])
    assert np.all(out == 0) and lse[0] == -math.inf


def test_probability_mass_is_one():
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((4, 8)), rng.standard_normal((30, 8)), rng.standard_normal((30, 8))
    sink, scale = 1.3, 0.4
    n_vis = [30, 11, 1, 7]
    _, lse = oracle.sink_attention(q, k, v, sink, scale, n_vis)
    for i in range(4):
        s = [scale * float(q[i] @ k[j]) for j in range(n_vis[i])]
        mass = math.exp(sink - lse[i]) + sum(math.exp(x - lse[i]) for x in s)
        assert abs(mass - 1.0) < 1e-13


# ------------------------------------------------------------ split / merge

def _all_bounds(n, max_cuts):
    for c in range(0, max_cuts + 1):
        for cuts in itertools.combinations(range(0, n + 1), c):
            yield [0, *cuts, n]


def test_split_merge_invariance_bruteforce():
    rng = np.random.default_rng(6)
    d, scale = 4, 0.5
    for n in (0, 1, 2, 5, 9):
        q, k, v = rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d))
        for sink in (-math.inf, -1.5, 0.0, 2.5, 8.0):
            ref_o, ref_l = oracle.sink_attention(q[None], k, v, sink, scale, [n])
            for bounds in _all_bounds(n, 2):      # every split into at most 3 blocks
                o, l = oracle.split_sink_attention(q, k, v, sink, scale, bounds)
                np.testing.assert_allclose(o, ref_o[0], atol=1e-12)
                if ref_l[0] == -math.inf:
                    assert l == -math.inf
                else:
                    assert abs(l - ref_l[0]) < 1e-12


def test_split_merge_invariance_random_up_to_8_blocks():
    rng = np.random.default_rng(7)
    d, scale = 8, 0.125
    for _ in range(40):
        n = int(rng.integers(1, 41))
        q, k, v = rng.standard_normal(d), rng.standard_normal((n, d)), rng.standard_normal((n, d))
        sink = float(rng.normal(0, 2))
        c = int(rng.integers(1, 9))
        cuts = sorted(rng.integers(0, n + 1, size=c - 1).tolist())
        bounds = [0, *cuts, n]
        ref_o, ref_l = oracle.sink_attention(q[None], k, v, sink, scale, [n])
        o, l = oracle.split_sink_attention(q, k, v, sink, scale, bounds)
        np.testing.assert_allclose(o, ref_o[0], atol=1e-12)
        assert abs(l - ref_l[0]) < 1e-12


def test_sink_in_every_block_is_wrong():
    rng = np.random.default_rng(8)
    q, k, v = rng.standard_normal(8), rng.standard_normal((12, 8)), rng.standard_normal((12, 8))
    ref_o, ref_l = oracle.sink_attention(q[None], k, v, 1.0, 0.5, [12])
    o, l = oracle.split_sink_attention(q, k, v, 1.0, 0.5, [0, 4, 8, 12], sink_in_every_block=True)
    assert np.max(np.abs(o - ref_o[0])) > 1e-3 or abs(l - ref_l[0]) > 1e-3


# ------------------------------------------------------- decode / extend

def _scatter_pages(rng, ks, vs, page_size, hkv, d):
    """Lay out per-request contiguous K/V [L, Hkv, D] into a shuffled pool."""
    pages_per = [math.ceil(len(x) / page_size) for x in ks]
    num_pages = sum(pages_per) + 3
    perm = rng.permutation(num_pages)
    kc = np.full((num_pages, hkv, page_size, d), np.nan)
    vc = np.full_like(kc, np.nan)
    table = np.full((len(ks), max(pages_per)), perm[-1])
    cur = 0
    for b, (kb, vb) in enumerate(zip(ks, vs)):
        for t in range(len(kb)):
            p = perm[cur + t // page_size]
            kc[p, :, t % page_size] = kb[t]
            vc[p, :, t % page_size] = vb[t]
        table[b, :pages_per[b]] = perm[cur:cur + pages_per[b]]
        cur += pages_per[b]
    return kc, vc, table


def test_decode_equals_last_prefill_row_and_torch():
    rng = np.random.default_rng(9)
    hq, hkv, d, page = 8, 2, 8, 4
    lens = [1, 4, 5, 13]
    ks = [rng.standard_normal((n, hkv, d)) for n in lens]
    vs = [rng.standard_normal((n, hkv, d)) for n in lens]
    qs = [rng.standard_normal((n, hq, d)) for n in lens]
    sinks = rng.normal(0, 2, hq)
    sinks[0] = -math.inf
    kc, vc, table = _scatter_pages(rng, ks, vs, page, hkv, d)
    q_dec = np.stack([x[-1] for x in qs])
    out, lse = oracle.decode(q_dec, kc, vc, table, lens, sinks, 0.125)
    for b, n in enumerate(lens):
        po, pl = oracle.prefill(qs[b], ks[b], vs[b], [0, n], sinks, 0.125)
        np.testing.assert_allclose(out[b], po[-1], atol=1e-13)
        np.testing.assert_allclose(lse[b], pl[-1], atol=1e-13)
        to, tl = _torch_plain(qs[b], ks[b], vs[b], 0.125, hq, hkv)
        sig = 1.0 / (1.0 + np.exp(sinks - tl[-1]))
        np.testing.assert_allclose(out[b], to[-1] * sig[:, None], atol=1e-12)


def test_extend_equals_rows_of_full_prefill():
    rng = np.random.default_rng(11)
    hq, hkv, d, page = 4, 2, 8, 4
    prefix, qlen = [0, 3, 9], [5, 4, 1]
    full = [p + n for p, n in zip(prefix, qlen)]
    ks = [rng.standard_normal((n, hkv, d)) for n in full]
    vs = [rng.standard_normal((n, hkv, d)) for n in full]
    qs = [rng.standard_normal((n, hq, d)) for n in full]
    sinks = rng.normal(0, 2, hq)
    kc, vc, table = _scatter_pages(rng, ks, vs, page, hkv, d)
    q_new = np.concatenate([x[p:] for x, p in zip(qs, prefix)])
    cu_q = np.concatenate([[0], np.cumsum(qlen)])
    out, lse = oracle.prefill_paged(q_new, cu_q, kc, vc, table, full, sinks, 0.2)
    for r in range(3):
        po, pl = oracle.prefill(qs[r], ks[r], vs[r], [0, full[r]], sinks, 0.2)
        np.testing.assert_allclose(out[cu_q[r]:cu_q[r + 1]], po[prefix[r]:], atol=1e-13)
        np.testing.assert_allclose(lse[cu_q[r]:cu_q[r + 1]], pl[prefix[r]:], atol=1e-13)


def test_page_permutation_invariance():
    rng = np.random.default_rng(12)
    hq, hkv, d, page = 4, 1, 8, 4
    ks = [rng.standard_normal((11, hkv, d))]
    vs = [rng.standard_normal((11, hkv, d))]
    q = rng.standard_normal((1, hq, d))
    sinks = rng.normal(0, 1, hq)
    a = oracle.decode(q, *_scatter_pages(np.random.default_rng(1), ks, vs, page, hkv, d), [11], sinks, 0.3)
    b = oracle.decode(q, *_scatter_pages(np.random.default_rng(2), ks, vs, page, hkv, d), [11], sinks, 0.3)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_sampled_rows_match_full():
    rng = np.random.default_rng(13)
    q, k, v, cu = _rand_prefill(rng, [40, 7], 4, 2)
    sinks = rng.normal(0, 2, 4)
    full_o, full_l = oracle.prefill(q, k, v, cu, sinks, 0.125, q_block=16)
    rows = [0, 5, 39, 40, 46]
    o, l = oracle.prefill(q, k, v, cu, sinks, 0.125, rows=rows)
    np.testing.assert_array_equal(o[rows], full_o[rows])
    np.testing.assert_array_equal(l[rows], full_l[rows])
