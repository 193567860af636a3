"""Programmatic dependent launch of the decode and verification kernels.

With the switch on, a decode or verification may be scheduled while the
kernel before it on the stream still runs: it ranks its requests and reads its
first page ids (kv_lens, page_table), then waits for that kernel before
touching q, the caches or its outputs.  These tests chain kernels whose
outputs feed the next call (decode -> decode and verify -> verify through q,
prologue -> decode through q and the cache) and check that every result
equals the one of the same calls made one at a time with the switch off, bit
for bit, and the float64 oracle.
"""

import numpy as np
import pytest
import torch

import gqa_attention_learned_gb300 as sa
import oracle
from gqa_attention_learned_gb300 import workloads
from oracle import prologue as pro
from tolerances import Bf16Pool, assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


class programmatic:
    def __init__(self, on):
        self.on = on

    def __enter__(self):
        self.prev = sa.set_programmatic_launch(self.on)

    def __exit__(self, *exc):
        sa.set_programmatic_launch(self.prev)


def _dev(w):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in w.items()}


def _chain(d, steps, sync_each):
    """q -> decode -> out used as the next decode's q, `steps` times; every
    output buffer starts as NaN so an early read of it shows."""
    outs, lses = [], []
    q = d["q"]
    for _ in range(steps):
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
        sa.decode(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                  d["scale"], d["max_kv_len"], out=out, lse=lse)
        if sync_each:
            torch.cuda.synchronize()
        outs.append(out)
        lses.append(lse)
        q = out
    torch.cuda.synchronize()
    return outs, lses


def test_switch_returns_previous_setting():
    prev = sa.set_programmatic_launch(True)
    try:
        assert sa.set_programmatic_launch(True) is True
        assert sa.set_programmatic_launch(False) is True
        assert sa.set_programmatic_launch(False) is False
    finally:
        sa.set_programmatic_launch(prev)


@pytest.mark.parametrize("batch,max_len", [(24, 1500), (64, 4096)])
def test_decode_chain_through_q(batch, max_len):
    """Each decode reads the previous one's output as its q.  Batch 24 leaves
    most SMs free, so the next decode's CTAs run their ranking while the
    previous decode is still in flight."""
    w = workloads.decode_batch(seed=batch, batch=batch, max_len=max_len)
    d = _dev(w)
    with programmatic(True):
        fast, fast_lse = _chain(d, 6, sync_each=False)
    with programmatic(False):
        slow, slow_lse = _chain(d, 6, sync_each=True)
    for a, b, la, lb in zip(fast, slow, fast_lse, slow_lse):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(la, lb)
    # the first two links against the oracle (q of the second: the oracle's
    # first output rounded to bf16, as stored)
    pool_k, pool_v = Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"])
    args = (pool_k, pool_v, w["page_table"].numpy(), w["kv_lens"].numpy(),
            w["sinks"].numpy().astype(np.float64), w["scale"])
    ro, rl = oracle.decode(to_np(w["q"]), *args)
    assert_out_close(fast[0].cpu(), ro)
    assert_lse_close(fast_lse[0].cpu(), rl)
    q2 = to_np(torch.from_numpy(ro).to(torch.bfloat16))
    ro2, rl2 = oracle.decode(q2, *args)
    assert_out_close(fast[1].cpu(), ro2)
    assert_lse_close(fast_lse[1].cpu(), rl2)


def test_split_plan_chain_with_workspace():
    """Long contexts: split plan with the in-kernel merge; the workspace
    counters are touched only after the wait."""
    w = workloads.decode_batch(seed=5, batch=4, min_len=20000, max_len=30000)
    d = _dev(w)
    splits, ws_bytes = sa.decode_plan(4, 64, 8, w["max_kv_len"])
    assert splits > 1
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)

    def run(sync_each):
        q, outs = d["q"], []
        for _ in range(4):
            out = torch.full_like(q, float("nan"))
            sa.decode(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                      d["scale"], d["max_kv_len"], out=out, workspace=ws)
            if sync_each:
                torch.cuda.synchronize()
            outs.append(out)
            q = out
        torch.cuda.synchronize()
        return outs

    with programmatic(True):
        fast = run(False)
    with programmatic(False):
        slow = run(True)
    for a, b in zip(fast, slow):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def _prologue_case(seed):
    """Eight long requests' tokens first, then one new token for each of 12
    decode requests, so the decode's q rows and cache slots are written by
    the prologue's last CTAs."""
    rng = np.random.default_rng(seed)
    starts = [int(x) for x in rng.integers(0, 900, size=12)]
    w = workloads.prologue_batch([1024] * 8 + [1] * 12, [0] * 8 + starts, seed=seed)
    kv_lens = torch.tensor([s + 1 for s in starts], dtype=torch.int32)
    sinks = workloads.gpt_oss_sinks(rng, 64)
    return w, starts, kv_lens, sinks


def _prologue_then_decode(w, kv_lens, sinks, inv, ms, sync_between):
    kc, vc = w["k_cache"].to(DEV), w["v_cache"].to(DEV)
    qkv, bias = w["qkv"].to(DEV), w["bias"].to(DEV)
    pos, slots = w["positions"].to(DEV), w["slot_mapping"].to(DEV)
    table = w["page_table"][8:].contiguous().to(DEV)
    lens, sk = kv_lens.to(DEV), sinks.to(DEV)
    torch.cuda.synchronize()
    q_all = torch.full((qkv.shape[0], 64, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    sa.qkv_prologue(qkv, bias, pos, slots, inv, ms, kc, vc, 64, 8, q_out=q_all)
    if sync_between:
        torch.cuda.synchronize()
    out = torch.full((12, 64, 64), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((12, 64), float("nan"), dtype=torch.float32, device=DEV)
    sa.decode(q_all[-12:], kc, vc, table, lens, sk, 0.125, int(kv_lens.max()), out=out, lse=lse)
    torch.cuda.synchronize()
    return out.cpu(), lse.cpu()


def test_prologue_then_programmatic_decode():
    """The prologue lets dependents start early; the decode must still see
    its q rows and the new tokens' k/v."""
    inv, ms = sa.yarn_table()
    for seed in (3, 4):
        w, starts, kv_lens, sinks = _prologue_case(seed)
        with programmatic(True):
            out, lse = _prologue_then_decode(w, kv_lens, sinks, inv, ms, sync_between=False)
        with programmatic(False):
            out0, lse0 = _prologue_then_decode(w, kv_lens, sinks, inv, ms, sync_between=True)
        assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
        assert torch.equal(lse, lse0)
        # oracle: prologue of the 12 decode tokens, written into the pool, decode
        n = w["qkv"].shape[0]
        rows = np.arange(n - 12, n)
        rq, rk, rv = pro.qkv_prologue(to_np(w["qkv"])[rows], to_np(w["bias"]),
                                      w["positions"].numpy()[rows],
                                      np.asarray(inv, dtype=np.float64), ms, 64, 8)
        rq, rk, rv = (to_np(torch.from_numpy(x).to(torch.bfloat16)) for x in (rq, rk, rv))
        slots = w["slot_mapping"].numpy()[rows]
        k64 = pro.scatter_to_cache(to_np(w["k_cache"]), rk, slots, 16)
        v64 = pro.scatter_to_cache(to_np(w["v_cache"]), rv, slots, 16)
        ro, rl = oracle.decode(rq, k64, v64, w["page_table"].numpy()[8:], kv_lens.numpy(),
                               sinks.numpy().astype(np.float64), 0.125)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)


def test_programmatic_chain_in_a_cuda_graph():
    """decode -> decode captured with the switch on and replayed with new
    inputs: equal to eager calls made one at a time."""
    w = workloads.decode_batch(seed=12, batch=32, max_len=2000)
    d = _dev(w)
    q = d["q"].clone()
    out1 = torch.empty_like(q)
    out2 = torch.empty_like(q)

    def step():
        sa.decode(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                  d["scale"], d["max_kv_len"], out=out1, want_lse=False)
        sa.decode(out1, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                  d["scale"], d["max_kv_len"], out=out2, want_lse=False)

    with programmatic(True):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()                                  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
    rng = np.random.default_rng(13)
    for _ in range(3):
        new_q = torch.from_numpy(rng.standard_normal(tuple(q.shape)).astype(np.float32))
        q.copy_(new_q.to(torch.bfloat16).to(DEV))
        out2.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        with programmatic(False):
            e1, _ = sa.decode(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"],
                              d["sinks"], d["scale"], d["max_kv_len"], want_lse=False)
            torch.cuda.synchronize()
            e2, _ = sa.decode(e1, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"],
                              d["sinks"], d["scale"], d["max_kv_len"], want_lse=False)
            torch.cuda.synchronize()
        assert torch.equal(out2.view(torch.int16), e2.view(torch.int16))


@pytest.mark.parametrize("q_len,tree", [(2, False), (4, False), (8, True)])
def test_verify_chain_through_q(q_len, tree):
    """Verification outputs feed the next verification's q ([B, q_len, Hq,
    64] both).  2 tokens (16 rows per KV head) take the split-KV kernel, 4
    and 8 the tensor-core kernel; both launch programmatically."""
    w = workloads.verify_batch(seed=40 + q_len, batch=64, q_len=q_len, max_len=1200, tree=tree)
    d = _dev(w)
    mask = d.get("tree_mask")

    def run(sync_each):
        q, outs, lses = d["q"], [], []
        for _ in range(5):
            out = torch.full_like(q, float("nan"))
            lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=DEV)
            sa.verify(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                      d["scale"], d["max_kv_len"], tree_mask=mask, out=out, lse=lse)
            if sync_each:
                torch.cuda.synchronize()
            outs.append(out)
            lses.append(lse)
            q = out
        torch.cuda.synchronize()
        return outs, lses

    with programmatic(True):
        fast, fast_lse = run(False)
    with programmatic(False):
        slow, slow_lse = run(True)
    for a, b, la, lb in zip(fast, slow, fast_lse, slow_lse):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(la, lb)
    m = w.get("tree_mask")
    ro, rl = oracle.verify(to_np(w["q"]), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                           w["page_table"].numpy(), w["kv_lens"].numpy(),
                           w["sinks"].numpy().astype(np.float64), w["scale"],
                           tree_mask=None if m is None else m.numpy())
    assert_out_close(fast[0].cpu(), ro)
    assert_lse_close(fast_lse[0].cpu(), rl)


def test_tensor_core_verify_chain_with_invalid_requests():
    """Tensor-core verification chained through q under programmatic launch,
    with requests that have fewer keys than new tokens: their CTAs write NaN
    rows after the dependency wait and leave without running the tile loop;
    the other requests must equal the calls made one at a time."""
    q_len = 4
    w = workloads.verify_batch(seed=61, batch=64, q_len=q_len, max_len=900)
    lens = w["kv_lens"].clone()
    lens[5] = q_len - 1
    lens[40] = 0
    w["kv_lens"] = lens
    d = _dev(w)
    assert sa.verify_plan(64, q_len, 64, 8, w["max_kv_len"]) == (1, 0)

    def run(sync_each):
        q, outs = d["q"], []
        for _ in range(4):
            out = torch.full_like(q, float("nan"))
            lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device=DEV)
            sa.verify(q, d["k_cache"], d["v_cache"], d["page_table"], d["kv_lens"], d["sinks"],
                      d["scale"], d["max_kv_len"], out=out, lse=lse)
            if sync_each:
                torch.cuda.synchronize()
            outs.append((out, lse))
            q = out
        torch.cuda.synchronize()
        return outs

    with programmatic(True):
        fast = run(False)
    with programmatic(False):
        slow = run(True)
    for (a, la), (b, lb) in zip(fast, slow):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(la.view(torch.int32), lb.view(torch.int32))
    out0, lse0 = fast[0]
    for bad in (5, 40):
        assert torch.isnan(out0[bad].float()).all() and torch.isnan(lse0[bad]).all()
    reqs = [0, 6, 39, 63]
    ro, rl = oracle.verify(to_np(w["q"][reqs]), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                           w["page_table"].numpy()[reqs], w["kv_lens"].numpy()[reqs],
                           w["sinks"].numpy().astype(np.float64), w["scale"])
    assert_out_close(out0.cpu()[reqs], ro)
    assert_lse_close(lse0.cpu()[reqs], rl)
