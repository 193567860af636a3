"""Seeded random sweep of the GPU paths against the float64 oracle: decode,
verification (both routes), prefill, paged extend -- random GQA groups,
lengths, split counts and sink values, small enough for the oracle.

Every case is drawn from a fixed seed, so a failure names a reproducible
configuration.
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
GROUPS = [(1, 1), (2, 1), (4, 1), (8, 1), (8, 2), (16, 2), (12, 4), (32, 8), (64, 8)]


def _gqa(rng):
    return GROUPS[int(rng.integers(len(GROUPS)))]


class _launch_mode:
    """Programmatic dependent launch on or off for the calls inside."""

    def __init__(self, on):
        self.on = on

    def __enter__(self):
        self.prev = sa.set_programmatic_launch(self.on)

    def __exit__(self, *exc):
        sa.set_programmatic_launch(self.prev)


def _twice(call):
    """Two calls back to back (the second may overlap the first when launched
    programmatically); both results must agree bit for bit."""
    a = call()
    b = call()
    torch.cuda.synchronize()
    def bits(t):                        # NaN rows compare by their bits
        return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)

    for x, y in zip(a, b):
        if x is not None:
            assert torch.equal(bits(x), bits(y))
    return b


@pytest.mark.parametrize("programmatic", [False, True])
@pytest.mark.parametrize("case", range(12))
def test_random_decode(case, programmatic):
    rng = np.random.default_rng(1000 + case)
    hq, hkv = _gqa(rng)
    batch = int(rng.integers(1, 24))
    max_len = int(rng.choice([1, 15, 16, 17, 300, 2000]))
    w = workloads.decode_batch(seed=2000 + case, batch=batch, num_qo_heads=hq, num_kv_heads=hkv,
                               min_len=0, max_len=max_len, special_sinks=bool(case % 2))
    splits = int(rng.choice([0, 1, 2, 5, 64]))
    args = [w[n].to(DEV) for n in ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]
    with _launch_mode(programmatic):
        out, lse = _twice(lambda: sa.decode(*args, w["scale"], max(1, w["max_kv_len"]),
                                            num_splits=splits))
    ro, rl = oracle.decode(to_np(w["q"]), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                           w["page_table"].numpy(), w["kv_lens"].numpy(),
                           w["sinks"].numpy().astype(np.float64), w["scale"])
    assert_out_close(out.cpu(), ro, f"out case {case}")
    assert_lse_close(lse.cpu(), rl, f"lse case {case}")


@pytest.mark.parametrize("programmatic", [False, True])
@pytest.mark.parametrize("case", range(12))
def test_random_verify(case, programmatic):
    rng = np.random.default_rng(3000 + case)
    hq, hkv = _gqa(rng)
    q_len = int(rng.integers(1, 20))
    tree = bool(rng.integers(2))
    # some cases get a wave of (request, KV head) CTAs: the tensor-core route
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    big = case % 3 == 0
    batch = (-(-2 * sms // hkv) + 1) if big else int(rng.integers(1, 10))
    w = workloads.verify_batch(seed=4000 + case, batch=batch, q_len=q_len, num_qo_heads=hq,
                               num_kv_heads=hkv, max_len=int(rng.choice([q_len, 64, 400])),
                               tree=tree)
    splits = 0 if big else int(rng.choice([0, 1, 3]))
    args = [w[n].to(DEV) for n in ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]
    mask = None if w["tree_mask"] is None else w["tree_mask"].to(DEV)
    with _launch_mode(programmatic):
        out, lse = _twice(lambda: sa.verify(*args, w["scale"], w["max_kv_len"], tree_mask=mask,
                                            num_splits=splits))
    reqs = list(range(batch)) if batch <= 12 else sorted(set(rng.integers(0, batch, 10).tolist()))
    ro, rl = oracle.verify(to_np(w["q"][reqs]), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                           w["page_table"].numpy()[reqs], w["kv_lens"].numpy()[reqs],
                           w["sinks"].numpy().astype(np.float64), w["scale"],
                           tree_mask=None if mask is None else w["tree_mask"].numpy()[reqs])
    assert_out_close(out.cpu()[reqs], ro, f"out case {case}")
    assert_lse_close(lse.cpu()[reqs], rl, f"lse case {case}")


@pytest.mark.parametrize("case", range(10))
def test_random_prefill_and_extend(case):
    rng = np.random.default_rng(5000 + case)
    hq, hkv = _gqa(rng)
    n = int(rng.integers(1, 6))
    lens = [int(x) for x in rng.integers(1, 400, size=n)]
    if case % 2 == 0:
        w = workloads.custom_prefill(lens, seed=6000 + case, num_qo_heads=hq, num_kv_heads=hkv,
                                     special_sinks=True)
        args = [w[k].to(DEV) for k in ("q", "k", "v", "cu_seqlens", "sinks")]
        out, lse = sa.prefill(*args, w["scale"], w["max_seqlen"])
        torch.cuda.synchronize()
        ro, rl = oracle.prefill(to_np(w["q"]), to_np(w["k"]), to_np(w["v"]), w["cu_seqlens"].numpy(),
                                w["sinks"].numpy().astype(np.float64), w["scale"])
    else:
        prefixes = [int(x) for x in rng.integers(0, 700, size=n)]
        w = workloads.extend_batch(lens, prefixes, seed=6000 + case, num_qo_heads=hq,
                                   num_kv_heads=hkv, special_sinks=True)
        args = [w[k].to(DEV) for k in ("q", "cu_seqlens_q", "k_cache", "v_cache", "page_table",
                                       "kv_lens", "sinks")]
        out, lse = sa.prefill_paged(*args, w["scale"], w["max_q_len"], w["max_kv_len"])
        torch.cuda.synchronize()
        ro, rl = oracle.prefill_paged(to_np(w["q"]), w["cu_seqlens_q"].numpy(), Bf16Pool(w["k_cache"]),
                                      Bf16Pool(w["v_cache"]), w["page_table"].numpy(),
                                      w["kv_lens"].numpy(), w["sinks"].numpy().astype(np.float64),
                                      w["scale"])
    assert_out_close(out.cpu(), ro, f"out case {case}")
    assert_lse_close(lse.cpu(), rl, f"lse case {case}")
