"""GPU parity of sinkattn_prefill / sinkattn_prefill_paged (tcgen05 kernels)
against the float64 oracle, through the C ABI.

Cases: the tiny 4-head check; ragged sequences around the 128-row tile edges
(1, 2, 127, 128, 129, 300, 513 tokens) for GQA groups 1..8; the causal
ragged prefill workload (4 sequences, ~20k tokens, 64/8 heads) on sampled
rows; sinks at -inf and +8; NaN tokens past the last sequence (they must not
leak through 0 * NaN); chunked prefill on shuffled paged prefixes of 0..1000
tokens; and requests whose arguments are out of range.
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


def run_prefill(w, **kw):
    args = [w[n].to(DEV) for n in ("q", "k", "v", "cu_seqlens", "sinks")]
    out, lse = sa.prefill(*args, w["scale"], w["max_seqlen"], **kw)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def ref_prefill(w, rows=None):
    return oracle.prefill(to_np(w["q"]), to_np(w["k"]), to_np(w["v"]), w["cu_seqlens"].numpy(),
                          w["sinks"].numpy().astype(np.float64), w["scale"], rows=rows)


def test_tiny_prefill():
    w = workloads.tiny()
    w["max_seqlen"] = 37
    out, lse = run_prefill(w)
    ro, rl = ref_prefill(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 1), (8, 8), (16, 2)])
def test_ragged_tile_edges(hq, hkv):
    lens = [1, 2, 127, 128, 129, 300, 513]
    w = workloads.custom_prefill(lens, seed=hq + 10 * hkv, num_qo_heads=hq, num_kv_heads=hkv,
                                 special_sinks=True)
    out, lse = run_prefill(w)
    ro, rl = ref_prefill(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_special_sinks_gpt_oss_heads():
    w = workloads.custom_prefill([700, 260], seed=4, num_qo_heads=64, num_kv_heads=8,
                                 special_sinks=True)
    out, lse = run_prefill(w)
    ro, rl = ref_prefill(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_causal_ragged_prefill_workload_sampled():
    w = workloads.ragged_prefill()
    out, lse = run_prefill(w)
    cu = w["cu_seqlens"].numpy()
    rng = np.random.default_rng(0)
    rows = set(rng.integers(0, int(cu[-1]), size=96).tolist())
    for s in range(len(cu) - 1):          # sequence edges and tile edges
        a, b = int(cu[s]), int(cu[s + 1])
        rows.update([a, a + 1, a + 127, a + 128, b - 129, b - 128, b - 1])
    rows = sorted(r for r in rows if 0 <= r < int(cu[-1]))
    ro, rl = ref_prefill(w, rows=rows)
    assert_out_close(out[rows], ro[rows])
    assert_lse_close(lse[rows], rl[rows])
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


def test_nan_tokens_past_the_last_sequence_do_not_leak():
    lens = [200, 77]
    w = workloads.custom_prefill(lens, seed=9, num_qo_heads=8, num_kv_heads=1)
    pad = 100                              # trailing tokens owned by no sequence
    for n in ("q", "k", "v"):
        t = w[n]
        w[n] = torch.cat([t, torch.full((pad,) + tuple(t.shape[1:]), float("nan"), dtype=t.dtype)])
    out, lse = run_prefill(w)
    ro, rl = ref_prefill(dict(w, q=w["q"][:277], k=w["k"][:277], v=w["v"][:277]))
    assert_out_close(out[:277], ro)
    assert_lse_close(lse[:277], rl)


def test_bad_sequence_bounds_give_nan_rows():
    w = workloads.custom_prefill([50, 60], seed=2, num_qo_heads=8, num_kv_heads=2)
    w["max_seqlen"] = 55                  # the second sequence exceeds the declared bound
    out, lse = run_prefill(w)
    ro, rl = ref_prefill(w)
    assert_out_close(out[:50], ro[:50])
    assert torch.isnan(out[50:].float()).all() and torch.isnan(lse[50:]).all()


# ----------------------------------------------------------------- extend

def run_extend(w):
    args = [w[n].to(DEV) for n in ("q", "cu_seqlens_q", "k_cache", "v_cache", "page_table",
                                   "kv_lens", "sinks")]
    out, lse = sa.prefill_paged(*args, w["scale"], w["max_q_len"], w["max_kv_len"])
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def ref_extend(w, rows=None):
    return oracle.prefill_paged(to_np(w["q"]), w["cu_seqlens_q"].numpy(), Bf16Pool(w["k_cache"]),
                                Bf16Pool(w["v_cache"]), w["page_table"].numpy(),
                                w["kv_lens"].numpy(), w["sinks"].numpy().astype(np.float64),
                                w["scale"], rows=rows)


@pytest.mark.parametrize("hq,hkv", [(8, 2), (64, 8)])
def test_extend_small(hq, hkv):
    q_lens = [1, 7, 128, 129, 300, 16]
    prefixes = [0, 5, 16, 100, 1000, 0]
    w = workloads.extend_batch(q_lens, prefixes, seed=hq, num_qo_heads=hq, num_kv_heads=hkv,
                               special_sinks=True)
    out, lse = run_extend(w)
    ro, rl = ref_extend(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_extend_equals_prefill_on_empty_prefix():
    lens = [129, 64, 300]
    w = workloads.extend_batch(lens, [0, 0, 0], seed=3, num_qo_heads=8, num_kv_heads=2)
    out, lse = run_extend(w)
    ro, rl = ref_extend(w)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def test_mixed_batch_extend_part_sampled():
    m = workloads.mixed_batch()
    e = m["extend"]
    w = dict(q=e["q"], cu_seqlens_q=e["cu_seqlens_q"], k_cache=m["k_cache"],
             v_cache=m["v_cache"], page_table=e["page_table"], kv_lens=e["kv_lens"],
             sinks=m["sinks"], scale=m["scale"], max_q_len=e["max_q_len"],
             max_kv_len=e["max_kv_len"])
    out, lse = run_extend(w)
    rng = np.random.default_rng(1)
    total = int(e["cu_seqlens_q"][-1])
    rows = sorted(set(rng.integers(0, total, size=48).tolist()) |
                  {0, 127, 128, 2047, 2048, total - 1})
    ro, rl = ref_extend(w, rows=rows)
    assert_out_close(out[rows], ro[rows])
    assert_lse_close(lse[rows], rl[rows])


def test_extend_bad_requests():
    w = workloads.extend_batch([10, 20, 30], [5, 5, 5], seed=8, num_qo_heads=8, num_kv_heads=2)
    lens = w["kv_lens"].clone()
    lens[1] = 10                                    # fewer keys than new queries
    w["kv_lens"] = lens
    table = w["page_table"].clone()
    table[2, 0] = w["num_pages"] + 3                # page id out of range
    w["page_table"] = table
    out, lse = run_extend(w)
    assert torch.isnan(out[10:30].float()).all()    # request 1
    assert torch.isnan(out[30:].float()).all()      # request 2
    sub = dict(w, q=w["q"][:10], cu_seqlens_q=w["cu_seqlens_q"][:2],
               page_table=w["page_table"][:1], kv_lens=w["kv_lens"][:1])
    ro, rl = ref_extend(sub)
    assert_out_close(out[:10], ro)
    assert_lse_close(lse[:10], rl)


def test_long_sequence_sampled_rows():
    """One 20,000-token sequence (157 query tiles, up to 157 KV tiles per
    CTA): sampled rows, including the last ones, against the oracle."""
    w = workloads.custom_prefill([20000], seed=31, num_qo_heads=8, num_kv_heads=1,
                                 special_sinks=True)
    out, lse = run_prefill(w)
    rows = [0, 1, 127, 128, 5000, 12345, 19871, 19872, 19998, 19999]
    ro, rl = ref_prefill(w, rows=rows)
    assert_out_close(out[rows], ro[rows])
    assert_lse_close(lse[rows], rl[rows])


def test_extend_on_long_prefix_sampled_rows():
    """Chunked prefill of 256 tokens after a 30,000-token paged prefix."""
    w = workloads.extend_batch([256, 40], [30000, 12000], seed=12, num_qo_heads=8,
                               num_kv_heads=2)
    out, lse = run_extend(w)
    rows = [0, 1, 127, 128, 255, 256, 295]
    ro, rl = ref_extend(w, rows=rows)
    assert_out_close(out[rows], ro[rows])
    assert_lse_close(lse[rows], rl[rows])
