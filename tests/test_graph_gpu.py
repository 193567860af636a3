"""Decode, verification and prefill captured in a CUDA graph and replayed
with new inputs ("GPT-OSS on day 0", Perplexity blog, the inference engine
runs decode under CUDA graphs).

The split plan depends only on host-side sizes (batch, heads, max_kv_len), and
every request's chunk count is derived on the device from kv_lens, so one
captured launch serves any kv_lens <= max_kv_len and any page table: replays
with fresh q / kv_lens / page tables must match the oracle and eager calls.
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


def _oracle_decode(q, kc, vc, table, lens, sinks, scale):
    return oracle.decode(to_np(q), Bf16Pool(kc), Bf16Pool(vc), table.cpu().numpy(),
                         lens.cpu().numpy(), sinks.cpu().numpy().astype(np.float64), scale)


def test_decode_graph_replays_with_new_lengths_and_tables():
    batch, hq, hkv, max_kv = 16, 64, 8, 3000
    w0 = workloads.decode_batch(seed=31, batch=batch, max_len=max_kv)
    kc, vc = w0["k_cache"].to(DEV), w0["v_cache"].to(DEV)
    q = w0["q"].to(DEV)
    table = w0["page_table"].to(DEV)
    lens = w0["kv_lens"].to(DEV)
    sinks = w0["sinks"].to(DEV)
    splits, ws_bytes = sa.decode_plan(batch, hq, hkv, max_kv)
    assert splits > 1                                   # the merge path is captured too
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(q)
    lse = torch.empty(batch, hq, dtype=torch.float32, device=DEV)

    def call():
        sa.decode(q, kc, vc, table, lens, sinks, w0["scale"], max_kv, out=out, lse=lse,
                  workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()                                          # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()

    # pages whose 16 slots all hold real (finite) tokens; the pool's spare
    # pages and the tails of last pages are NaN
    full = (torch.isfinite(w0["k_cache"].float()).flatten(1).all(1) &
            torch.isfinite(w0["v_cache"].float()).flatten(1).all(1)).nonzero().flatten()
    rng = np.random.default_rng(5)
    for rep in range(3):
        # new lengths (within max_kv), new page assignments, new queries
        new_lens = torch.from_numpy(rng.integers(0, max_kv // 2, size=batch).astype(np.int32))
        new_lens[0] = min(max_kv, 16 * w0["page_table"].shape[1])    # the longest a row allows
        new_lens[1] = 0
        pages_needed = [(int(n) + 15) // 16 for n in new_lens]
        assert sum(pages_needed) <= len(full)
        perm = full[torch.from_numpy(rng.permutation(len(full)))].to(torch.int32)
        new_table = torch.zeros_like(w0["page_table"])
        used = 0
        for b, n in enumerate(pages_needed):
            new_table[b, :n] = perm[used:used + n]
            used += n
        new_q = torch.from_numpy(rng.standard_normal((batch, hq, 64)).astype(np.float32)).to(torch.bfloat16)
        q.copy_(new_q)
        table.copy_(new_table)
        lens.copy_(new_lens)
        g.replay()
        torch.cuda.synchronize()
        ro, rl = _oracle_decode(new_q, w0["k_cache"], w0["v_cache"], new_table, new_lens,
                                w0["sinks"], w0["scale"])
        assert_out_close(out.cpu(), ro)
        assert_lse_close(lse.cpu(), rl)
        # an eager call on the same inputs gives bitwise the same result
        eo, el = sa.decode(q, kc, vc, table, lens, sinks, w0["scale"], max_kv,
                           workspace=torch.zeros_like(ws))
        torch.cuda.synchronize()
        assert torch.equal(eo.cpu(), out.cpu())
        assert torch.equal(el.cpu(), lse.cpu())


def test_verify_and_prefill_graphs_replay():
    wv = workloads.verify_batch(seed=41, batch=8, q_len=4, max_len=900, tree=True)
    args = {n: wv[n].to(DEV) for n in ("q", "k_cache", "v_cache", "page_table", "kv_lens",
                                       "sinks", "tree_mask")}
    out = torch.empty_like(args["q"])
    lse = torch.empty(args["q"].shape[:3], dtype=torch.float32, device=DEV)
    s, wsb = sa.verify_plan(8, 4, 64, 8, wv["max_kv_len"], 3)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=DEV)

    def vcall():
        sa.verify(args["q"], args["k_cache"], args["v_cache"], args["page_table"],
                  args["kv_lens"], args["sinks"], wv["scale"], wv["max_kv_len"],
                  tree_mask=args["tree_mask"], out=out, lse=lse, num_splits=3, workspace=ws)

    wp = workloads.custom_prefill([300, 129, 64], seed=42, num_qo_heads=16, num_kv_heads=2)
    pa = {n: wp[n].to(DEV) for n in ("q", "k", "v", "cu_seqlens", "sinks")}
    pout = torch.empty_like(pa["q"])
    plse = torch.empty(pa["q"].shape[:2], dtype=torch.float32, device=DEV)

    def pcall():
        sa.prefill(pa["q"], pa["k"], pa["v"], pa["cu_seqlens"], pa["sinks"], wp["scale"], 300,
                   out=pout, lse=plse)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        vcall()
        pcall()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        vcall()
        pcall()

    rng = np.random.default_rng(3)
    for rep in range(2):
        new_q = torch.from_numpy(rng.standard_normal(tuple(wv["q"].shape)).astype(np.float32))
        args["q"].copy_(new_q.to(torch.bfloat16))
        new_cu = torch.tensor([0, 100 + 50 * rep, 400, 493], dtype=torch.int32)
        pa["cu_seqlens"].copy_(new_cu)                  # same total, new boundaries
        g.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.verify(to_np(new_q.to(torch.bfloat16)), Bf16Pool(wv["k_cache"]),
                               Bf16Pool(wv["v_cache"]), wv["page_table"].numpy(),
                               wv["kv_lens"].numpy(), wv["sinks"].numpy().astype(np.float64),
                               wv["scale"], tree_mask=wv["tree_mask"].numpy())
        assert_out_close(out.cpu(), ro)
        assert_lse_close(lse.cpu(), rl)
        po, pl = oracle.prefill(to_np(wp["q"]), to_np(wp["k"]), to_np(wp["v"]), new_cu.numpy(),
                                wp["sinks"].numpy().astype(np.float64), wp["scale"])
        assert_out_close(pout.cpu(), po)
        assert_lse_close(plse.cpu(), pl)
