"""GPU parity of sinkattn_verify (draft-token verification) against the
float64 oracle, through the C ABI.

"Accelerating Sonar through speculation" (Perplexity blog): sections
"Target-Draft" and "MTP" verify the k + 1 newest tokens of every request in
one pass; section "EAGLE" verifies a draft tree with a custom mask.

Cases: causal verification with 1..16 tokens for GQA groups 1..16, against
the oracle and (for one token) bitwise against sinkattn_decode; random draft
trees of 3..64 nodes; forced chunking (splits 1, 3, 1000); the gpt-oss-20b
batch with 4 tokens per request (sampled requests); rows that see no key;
requests with fewer keys than new tokens.
"""

import numpy as np
import pytest
import torch

import gqa_attention_learned_gb300 as sa
import oracle
from gqa_attention_learned_gb300 import workloads
from tolerances import Bf16Pool, assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_verify(w, **kw):
    q, kc, vc, table, lens, sinks = [w[n].to(DEV) for n in
                                     ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]
    mask = w.get("tree_mask")
    out, lse = sa.verify(q, kc, vc, table, lens, sinks, w["scale"], w["max_kv_len"],
                         tree_mask=None if mask is None else mask.to(DEV), **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def ref_verify(w, requests=None):
    reqs = slice(None) if requests is None else list(requests)
    mask = w.get("tree_mask")
    return oracle.verify(to_np(w["q"][reqs]), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                         w["page_table"].numpy()[reqs], w["kv_lens"].numpy()[reqs],
                         w["sinks"].numpy().astype(np.float64), w["scale"],
                         tree_mask=None if mask is None else mask.numpy()[reqs])


@pytest.mark.parametrize("q_len", [1, 2, 3, 4, 7, 16])
@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 1), (16, 1)])
def test_causal_verify_small(q_len, hq, hkv):
    w = workloads.verify_batch(seed=100 + q_len, batch=6, q_len=q_len, num_qo_heads=hq,
                               num_kv_heads=hkv, max_len=300)
    out, lse = run_verify(w)
    ro, rl = ref_verify(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("q_len", [3, 8, 16, 64])
def test_tree_verify(q_len):
    w = workloads.verify_batch(seed=200 + q_len, batch=5, q_len=q_len, num_qo_heads=16,
                               num_kv_heads=2, max_len=400, tree=True)
    out, lse = run_verify(w)
    ro, rl = ref_verify(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("splits", [1, 3, 1000])
def test_verify_split_counts(splits):
    w = workloads.verify_batch(seed=7, batch=4, q_len=5, num_qo_heads=8, num_kv_heads=1,
                               min_len=100, max_len=2000, tree=True)
    out, lse = run_verify(w, num_splits=splits)
    ro, rl = ref_verify(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_one_token_is_bitwise_decode():
    w = workloads.verify_batch(seed=9, batch=16, q_len=1, max_len=3000)
    d = dict(w, q=w["q"][:, 0].contiguous())
    args = [d[n].to(DEV) for n in ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]
    do, dl = sa.decode(*args, d["scale"], d["max_kv_len"])
    vo, vl = run_verify(w)
    mo, ml = run_verify(dict(w, tree_mask=torch.ones(16, 1, dtype=torch.int64)))
    torch.cuda.synchronize()
    for o, l in ((vo, vl), (mo, ml)):
        assert torch.equal(o[:, 0], do.cpu())
        assert torch.equal(l[:, 0], dl.cpu())


def test_gpt_oss_20b_batch_four_tokens_sampled():
    w = workloads.verify_batch(q_len=4)
    out, lse = run_verify(w)
    reqs = [0, 1, 17, 33, 62, 63]
    ro, rl = ref_verify(w, reqs)
    assert_out_close(out[reqs], ro)
    assert_lse_close(lse[reqs], rl)
    assert torch.isfinite(out.float()).all() and not torch.isnan(lse).any()


def test_rows_that_see_no_key_and_short_requests():
    w = workloads.verify_batch(seed=11, batch=4, q_len=3, num_qo_heads=8, num_kv_heads=2,
                               max_len=50, tree=True)
    lens = w["kv_lens"].clone()
    lens[0] = 3                       # no prefix: the drafts are the whole request
    lens[2] = 2                       # fewer keys than new tokens: NaN rows
    mask = w["tree_mask"].clone()
    mask[0, 1] = 0                    # sees nothing: out = 0, lse = sink
    w = dict(w, kv_lens=lens, tree_mask=mask)
    out, lse = run_verify(w)
    assert torch.isnan(out[2].float()).all() and torch.isnan(lse[2]).all()
    ok = [0, 1, 3]
    ro, rl = ref_verify(w, ok)
    assert_out_close(out[ok], ro)
    assert_lse_close(lse[ok], rl)
    assert torch.equal(out[0, 1].float(), torch.zeros(8, 64))
    sinks = w["sinks"]
    assert torch.equal(torch.isinf(lse[0, 1]), torch.isinf(sinks))


# ---------------------------------------------------- tensor-core (tcgen05) route
# With at least a wave of (request, KV head) CTAs and >= 24 query rows per KV
# head, sinkattn_verify runs the tcgen05 kernel (rows = (token, head) pairs of
# a KV head in one 128-row tile, no KV split); the plan reports one split and
# no workspace for it.

def _tc_batch(q_len, hq, hkv):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = -(-q_len // (128 // (hq // hkv)))
    return -(-2 * sms // (hkv * tiles)) + 2


@pytest.mark.parametrize("q_len,hq,hkv,tree", [(4, 64, 8, False), (8, 64, 8, True),
                                               (16, 64, 8, True), (32, 64, 8, True),
                                               (6, 32, 8, False), (2, 32, 2, True),
                                               (32, 8, 8, True), (2, 128, 1, False),
                                               (64, 64, 8, True)])
def test_tensor_core_route(q_len, hq, hkv, tree):
    b = _tc_batch(q_len, hq, hkv)
    w = workloads.verify_batch(seed=300 + q_len + hq, batch=b, q_len=q_len, num_qo_heads=hq,
                               num_kv_heads=hkv, max_len=180, tree=tree)
    assert sa.verify_plan(b, q_len, hq, hkv, w["max_kv_len"]) == (1, 0)
    out, lse = run_verify(w)
    ro, rl = ref_verify(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("q_len,hq,hkv,tree", [(5, 64, 8, False), (6, 64, 8, True),
                                               (7, 64, 8, False), (3, 32, 2, False),
                                               (4, 32, 2, True), (8, 64, 8, False)])
def test_tensor_core_route_key_halves(q_len, hq, hkv, tree):
    """33 to 64 query rows per KV head: the rows are replicated into the next
    tensor-memory lanes and each copy takes one half of every key tile, the
    halves merged at the end; rows past q_len x group in either half are
    idle.  Lengths from 0 past the drafts (the second half then sees no key
    in the first tile) up to several tiles."""
    b = _tc_batch(q_len, hq, hkv)
    w = workloads.verify_batch(seed=400 + q_len + hq, batch=b, q_len=q_len, num_qo_heads=hq,
                               num_kv_heads=hkv, max_len=700, tree=tree,
                               kv_lens_first=(q_len, q_len + 1, 63, 64, 65, 128, 129))
    assert 32 < q_len * (hq // hkv) <= 64
    assert sa.verify_plan(b, q_len, hq, hkv, w["max_kv_len"]) == (1, 0)
    out, lse = run_verify(w)
    ro, rl = ref_verify(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_tensor_core_route_matches_split_kernel_and_poisons_short_requests():
    q_len, hq, hkv = 8, 64, 8
    b = _tc_batch(q_len, hq, hkv)
    w = workloads.verify_batch(seed=17, batch=b, q_len=q_len, max_len=700, tree=True)
    lens = w["kv_lens"].clone()
    lens[3] = q_len - 1                      # fewer keys than new tokens
    w["kv_lens"] = lens
    tc_out, tc_lse = run_verify(w)                    # tensor-core route
    mma_out, mma_lse = run_verify(w, num_splits=1)    # split-KV route
    assert torch.isnan(tc_out[3].float()).all() and torch.isnan(tc_lse[3]).all()
    assert torch.isnan(mma_out[3].float()).all()
    ok = [i for i in range(b) if i != 3]
    reqs = ok[:6] + ok[-4:]
    ro, rl = ref_verify(w, reqs)
    for o, l in ((tc_out, tc_lse), (mma_out, mma_lse)):
        assert_out_close(o[reqs], ro)
        assert_lse_close(l[reqs], rl)


def test_tensor_core_route_large_batch():
    """400 requests over one KV head on the tensor-core route: the CTAs rank
    the requests by size with several requests per thread."""
    w = workloads.verify_batch(seed=19, batch=400, q_len=4, num_qo_heads=8, num_kv_heads=1,
                               max_len=300, tree=True)
    assert sa.verify_plan(400, 4, 8, 1, w["max_kv_len"]) == (1, 0)
    out, lse = run_verify(w)
    reqs = list(range(0, 400, 7))
    ro, rl = ref_verify(w, reqs)
    assert_out_close(out[reqs], ro)
    assert_lse_close(lse[reqs], rl)


@pytest.mark.parametrize("programmatic", [False, True])
def test_tensor_core_route_long_requests_back_to_back(programmatic):
    """4 tokens x 8 heads = 32 rows per KV head on the tensor-core route with
    long requests (up to 32 key tiles) and many launches back to back, in
    both launch modes: every output finite (no wait gave up), sampled
    requests equal the oracle, every launch equal to the first."""
    w = workloads.verify_batch(seed=71, batch=64, q_len=4, min_len=2000, max_len=4096)
    assert sa.verify_plan(64, 4, 64, 8, w["max_kv_len"]) == (1, 0)
    q, kc, vc, table, lens, sinks = [w[n].to(DEV) for n in
                                     ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]
    prev = sa.set_programmatic_launch(programmatic)
    try:
        outs = [sa.verify(q, kc, vc, table, lens, sinks, w["scale"], w["max_kv_len"])
                for _ in range(12)]
        torch.cuda.synchronize()
    finally:
        sa.set_programmatic_launch(prev)
    first_out, first_lse = outs[0]
    assert torch.isfinite(first_out.float()).all() and torch.isfinite(first_lse).all()
    for out, lse in outs[1:]:
        assert torch.equal(out.view(torch.int16), first_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), first_lse.view(torch.int32))
    reqs = [0, 17, 40, 63]
    ro, rl = ref_verify(w, reqs)
    assert_out_close(first_out.cpu()[reqs], ro)
    assert_lse_close(first_lse.cpu()[reqs], rl)
