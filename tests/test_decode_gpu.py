"""GPU parity of sinkattn_decode against the float64 oracle (through the C ABI).

Cases: the tiny 4-head check, the gpt-oss-20b decode batch (64 requests,
kv_len 1..4096, sinks with -inf and +8 heads, shuffled pages with NaN-filled
spares), the long-context split-KV batch (kv_len 32k..131k, 8 and auto
splits), ragged edges (kv_len 0, 1, 15, 16, 17, ...), GQA groups 1..16,
forced one-page chunks, out-of-range page ids and too-small workspaces.
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


def _dev(w, *names):
    return [w[n].to(DEV) for n in names]


def run_decode(w, q=None, **kw):
    q = w["q"] if q is None else q
    qd, kc, vc, table, lens, sinks = [x.to(DEV) for x in
                                      (q, w["k_cache"], w["v_cache"], w["page_table"],
                                       w["kv_lens"], w["sinks"])]
    max_kv = int(w["kv_lens"].max()) if "max_kv_len" not in w else w["max_kv_len"]
    out, lse = sa.decode(qd, kc, vc, table, lens, sinks, w["scale"], kw.pop("max_kv_len", max_kv),
                         **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def ref_decode(w, q=None):
    q = w["q"] if q is None else q
    return oracle.decode(to_np(q), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                         w["page_table"].numpy(), w["kv_lens"].numpy(),
                         w["sinks"].numpy().astype(np.float64), w["scale"])


def test_tiny_decode_matches_oracle_and_prefill_row():
    tiny = workloads.tiny()
    w = dict(tiny, q=tiny["q_decode"], max_kv_len=37)
    out, lse = run_decode(w)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    # same as the last row of the causal prefill over the 37 tokens
    po, pl = oracle.prefill(to_np(tiny["q"]), to_np(tiny["k"]), to_np(tiny["v"]), [0, 37],
                            tiny["sinks"].numpy().astype(np.float64), tiny["scale"])
    np.testing.assert_allclose(ro[0], po[36], atol=1e-12)
    assert_out_close(out[0], po[36])


@pytest.mark.parametrize("splits", [0, 1, 16])
def test_gpt_oss_20b_decode(splits):
    w = workloads.decode_batch()
    out, lse = run_decode(w, num_splits=splits)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("splits", [0, 8])
def test_long_context_split_decode(splits):
    w = workloads.long_decode()
    if splits:
        assert sa.decode_plan(8, 64, 8, w["max_kv_len"], splits)[0] == 8
    else:
        s, _ = sa.decode_plan(8, 64, 8, w["max_kv_len"])
        assert 8 <= s <= 1024
    out, lse = run_decode(w, num_splits=splits)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_mixed_batch_decode_part():
    """The mixed serving batch's decode half: 32 requests with kv_len in
    [512, 16384] in the page pool they share with the four extend requests
    (shuffled pages, NaN-filled spares), the planner's own split choice (fewer
    (request, KV head) units than one wave, so chunked split-KV with the
    in-kernel merge), all 32 requests x 64 heads against the oracle."""
    m = workloads.mixed_batch()
    d = m["decode"]
    splits, ws = sa.decode_plan(32, 64, 8, d["max_kv_len"])
    assert splits > 1 and ws > 0                  # the split path with its merge
    w = dict(q=d["q"], k_cache=m["k_cache"], v_cache=m["v_cache"], page_table=d["page_table"],
             kv_lens=d["kv_lens"], sinks=m["sinks"], scale=m["scale"],
             max_kv_len=d["max_kv_len"])
    ro, rl = ref_decode(w)
    for _ in range(2):                            # the counters reset: a second call agrees
        out, lse = run_decode(w)
        assert_out_close(out, ro, "mixed decode out")
        assert_lse_close(lse, rl, "mixed decode lse")


@pytest.mark.parametrize("hq,hkv,batch", [(32, 2, 160), (48, 4, 80), (64, 2, 80), (128, 8, 40)])
@pytest.mark.parametrize("splits", [0, 3])
def test_wide_gqa_groups(hq, hkv, batch, splits):
    """GQA groups above 8 (12, 16, 32) with enough requests that the plan
    takes 16-head CTAs (each page read once for 16 heads): whole requests
    heaviest first, and an explicit 3-way split with its merge; kv_len 0..900
    with a few empty requests."""
    w = workloads.decode_batch(seed=hq + hkv + batch + splits, batch=batch, num_qo_heads=hq,
                               num_kv_heads=hkv, min_len=0, max_len=900)
    assert int(w["kv_lens"].min()) >= 0
    out, lse = run_decode(w, num_splits=splits)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


EDGE_LENS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 255, 256, 257, 1000]


@pytest.mark.parametrize("hq,hkv", [(8, 8), (4, 1), (16, 2), (64, 8), (32, 2), (12, 1)])
@pytest.mark.parametrize("splits", [0, 1, 1000])
def test_decode_edges(hq, hkv, splits):
    rng = np.random.default_rng(hq * 7 + hkv + splits)
    lens = EDGE_LENS
    w = workloads.decode_batch(seed=int(rng.integers(1 << 30)), batch=len(lens), num_qo_heads=hq,
                               num_kv_heads=hkv, min_len=1, max_len=2)
    pool = workloads.paged_pool(rng, lens, hkv)
    w.update(pool)
    w["max_kv_len"] = max(lens)
    out, lse = run_decode(w, num_splits=splits)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
    # kv_len = 0: out = 0, lse = sink
    assert torch.all(out[0] == 0)


def test_page_permutation_is_bitwise_invariant():
    w = workloads.decode_batch(batch=16, max_len=700)
    out_a, lse_a = run_decode(w, num_splits=3)
    # rebuild the pool with the same contents in a different page order
    rng = np.random.default_rng(99)
    num_pages = w["num_pages"]
    perm = torch.from_numpy(rng.permutation(num_pages).astype(np.int64))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(num_pages)
    w2 = dict(w)
    w2["k_cache"] = w["k_cache"][perm].contiguous()      # new page i = old page perm[i]
    w2["v_cache"] = w["v_cache"][perm].contiguous()
    w2["page_table"] = inv[w["page_table"].long()].to(torch.int32)
    out_b, lse_b = run_decode(w2, num_splits=3)
    assert torch.equal(out_a, out_b)
    assert torch.equal(lse_a, lse_b)


def test_identical_queries_give_identical_heads():
    w = workloads.decode_batch(batch=4, max_len=300, special_sinks=False)
    q = w["q"].clone()
    q[:, :, :] = q[:, :1, :]                   # every head the same query
    w["sinks"] = torch.zeros_like(w["sinks"])  # and the same sink
    out, lse = run_decode(w, q=q)
    for kvh in range(8):
        blk = out[:, kvh * 8:(kvh + 1) * 8]
        assert torch.equal(blk, blk[:, :1].expand_as(blk))


def test_bad_page_id_poisons_only_its_request():
    w = workloads.decode_batch(batch=6, max_len=200, special_sinks=False)
    table = w["page_table"].clone()
    table[2, 0] = w["num_pages"] + 5              # out of range: never dereferenced
    table[4, 0] = -3
    w["page_table"] = table
    out, lse = run_decode(w)
    assert torch.isnan(out[2].float()).all() and torch.isnan(lse[2]).all()
    assert torch.isnan(out[4].float()).all()
    good = [0, 1, 3, 5]
    sub = dict(w)
    sub["q"] = w["q"][good]
    sub["page_table"] = table[good]
    sub["kv_lens"] = w["kv_lens"][good]
    ro, rl = ref_decode(sub)
    assert_out_close(out[good], ro)
    assert_lse_close(lse[good], rl)


def test_kv_len_beyond_declared_bounds_is_nan():
    w = workloads.decode_batch(batch=3, max_len=100, special_sinks=False)
    lens = w["kv_lens"].clone()
    w["max_kv_len"] = int(lens.max())
    lens[1] = w["page_table"].shape[1] * 16 + 1      # does not fit the table row
    w["kv_lens"] = lens
    out, lse = run_decode(w)
    assert torch.isnan(out[1].float()).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(out[2].float()).all()


def test_workspace_too_small_is_reported():
    w = workloads.decode_batch(batch=4, max_len=4096, min_len=4000)
    args = [x.to(DEV) for x in (w["q"], w["k_cache"], w["v_cache"], w["page_table"], w["kv_lens"],
                                w["sinks"])]
    splits, need = sa.decode_plan(4, 64, 8, 4096, 8)
    assert splits == 8 and need > 0
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode(*args, w["scale"], 4096, num_splits=8, workspace=ws)
    assert e.value.status == sa.WORKSPACE_TOO_SMALL


def test_decode_on_side_stream_and_no_lse():
    w = workloads.decode_batch(batch=8, max_len=1000)
    s = torch.cuda.Stream()
    args = [x.to(DEV) for x in (w["q"], w["k_cache"], w["v_cache"], w["page_table"], w["kv_lens"],
                                w["sinks"])]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, lse = sa.decode(*args, w["scale"], 1000, want_lse=False)
    s.synchronize()
    assert lse is None
    ro, _ = ref_decode(w)
    assert_out_close(out.cpu(), ro)


def test_large_batch_heaviest_first_dispatch():
    """600 requests over one KV head: the plan keeps whole requests and the
    CTAs rank them by size (more groups of 32 lengths than a warp keeps in
    registers, empty requests among them)."""
    w = workloads.decode_batch(seed=77, batch=600, num_qo_heads=8, num_kv_heads=1, min_len=0,
                               max_len=700)
    assert sa.decode_plan(600, 8, 1, w["max_kv_len"]) == (1, 0)
    out, lse = run_decode(w)
    ro, rl = ref_decode(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)
