"""GPU parity of sinkattn_qkv_prologue (QKV bias + YaRN rotary encoding +
paged cache write) against the float64 oracle, through the C ABI; and the
prologue feeding decode.

"GPT-OSS on day 0" (Perplexity blog): YaRN position encoding (as in
DeepSeek-V3) and QKV biases (as in Qwen 2).

Bar: every bf16 output within one bf16 ulp of the float64 reference plus
1e-5 absolute (fp32 cancellation in x1 cos - x2 sin); cache slots that no
token maps to stay bitwise unchanged.
"""

import numpy as np
import pytest
import torch

import gqa_attention_learned_gb300 as sa
import oracle
from gqa_attention_learned_gb300 import workloads
from oracle import prologue as pro
from tolerances import Bf16Pool, assert_lse_close, assert_out_close, bf16_ulp, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
STYLES = {"half": sa.ROPE_HALF, "interleaved": sa.ROPE_INTERLEAVED}


def assert_bf16_close(gpu, ref, what):
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape
    err = np.abs(g - r)
    allowed = bf16_ulp(r) + 1e-5
    bad = err > allowed
    assert not bad.any(), (what, int(bad.sum()), float((err - allowed).max()))


def run(w, style="half", yarn=None):
    inv, ms = sa.yarn_table(**(yarn or {}))
    kc, vc = w["k_cache"].to(DEV), w["v_cache"].to(DEV)
    q = sa.qkv_prologue(w["qkv"].to(DEV), None if w["bias"] is None else w["bias"].to(DEV),
                        w["positions"].to(DEV), w["slot_mapping"].to(DEV), inv, ms, kc, vc,
                        w["num_qo_heads"], w["num_kv_heads"], rope_style=STYLES[style])
    torch.cuda.synchronize()
    return q.cpu(), kc.cpu(), vc.cpu(), inv, ms


def check(w, style="half", yarn=None):
    q, kc, vc, inv, ms = run(w, style, yarn)
    rq, rk, rv = pro.qkv_prologue(to_np(w["qkv"]), None if w["bias"] is None else to_np(w["bias"]),
                                  w["positions"].numpy(), np.asarray(inv, dtype=np.float64), ms,
                                  w["num_qo_heads"], w["num_kv_heads"], style)
    assert_bf16_close(q, rq, "q")
    slots = w["slot_mapping"].numpy()
    pages = w["k_cache"].shape[0]
    live = (slots >= 0) & (slots // 16 < pages)
    sl = slots[live]
    assert_bf16_close(kc[sl // 16, :, sl % 16], rk[live], "k")
    assert_bf16_close(vc[sl // 16, :, sl % 16], rv[live], "v")
    # every other slot is bitwise unchanged (NaN patterns included)
    written = torch.zeros(pages, 16, dtype=torch.bool)
    written[torch.from_numpy(sl // 16), torch.from_numpy(sl % 16)] = True
    keep = ~written
    for new, old in ((kc, w["k_cache"]), (vc, w["v_cache"])):
        a = new.view(torch.int16).permute(0, 2, 1, 3)[keep]
        b = old.view(torch.int16).permute(0, 2, 1, 3)[keep]
        assert torch.equal(a, b)


@pytest.mark.parametrize("style", ["half", "interleaved"])
@pytest.mark.parametrize("bias", [True, False])
def test_small_batches(style, bias):
    w = workloads.prologue_batch([37, 1, 16, 5], [0, 5, 1000, 77], seed=3, num_qo_heads=8,
                                 num_kv_heads=2, bias=bias)
    check(w, style)


@pytest.mark.parametrize("style", ["half", "interleaved"])
def test_gpt_oss_shapes_large_positions(style):
    # decode-like: one token per request at positions up to 2^20
    rng = np.random.default_rng(4)
    starts = list(rng.integers(0, 131072, size=30)) + [131071, (1 << 20) - 1]
    w = workloads.prologue_batch([1] * 32, starts, seed=5)
    check(w, style)


def test_plain_rotary_and_other_yarn_parameters():
    w = workloads.prologue_batch([70, 3], [0, 4093], seed=6, num_qo_heads=16, num_kv_heads=2)
    check(w, "half", dict(factor=1.0, base=10000.0))
    check(w, "half", dict(factor=8.0, base=500000.0, original_context=8192, beta_fast=16.0,
                          beta_slow=2.0))


def test_unmapped_tokens_write_nothing():
    w = workloads.prologue_batch([20, 20], [0, 30], seed=7, num_qo_heads=8, num_kv_heads=1)
    slots = w["slot_mapping"].clone()
    slots[::3] = -1
    slots[1] = w["k_cache"].shape[0] * 16          # past the pool
    w["slot_mapping"] = slots
    check(w)


def test_prologue_then_decode():
    """The prologue writes each request's newest token; decode then attends
    over the cache including it -- against oracle prologue + oracle decode."""
    hq, hkv = 64, 8
    rng = np.random.default_rng(8)
    starts = [int(x) for x in rng.integers(0, 900, size=12)]
    w = workloads.prologue_batch([1] * 12, starts, seed=9)
    q, kc, vc, inv, ms = run(w)
    kv_lens = torch.tensor([s + 1 for s in starts], dtype=torch.int32)
    sinks = workloads.gpt_oss_sinks(rng, hq)
    out, lse = sa.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), w["page_table"].to(DEV),
                         kv_lens.to(DEV), sinks.to(DEV), 0.125, int(kv_lens.max()))
    torch.cuda.synchronize()
    # oracle: rotate in float64, write into a float64 copy of the pool, decode
    rq, rk, rv = pro.qkv_prologue(to_np(w["qkv"]), to_np(w["bias"]), w["positions"].numpy(),
                                  np.asarray(inv, dtype=np.float64), ms, hq, hkv)
    # q, k, v cross the interface as bf16: round the oracle's once, as stored
    rq, rk, rv = (to_np(torch.from_numpy(x).to(torch.bfloat16)) for x in (rq, rk, rv))
    slots = w["slot_mapping"].numpy()
    k64 = pro.scatter_to_cache(to_np(w["k_cache"]), rk, slots, 16)
    v64 = pro.scatter_to_cache(to_np(w["v_cache"]), rv, slots, 16)
    ro, rl = oracle.decode(rq, k64, v64, w["page_table"].numpy(), kv_lens.numpy(),
                           sinks.numpy().astype(np.float64), 0.125)
    assert_out_close(out.cpu(), ro)
    assert_lse_close(lse.cpu(), rl)


def test_prologue_waits_for_the_decode_before_it():
    """decode -> prologue -> decode on one stream, all launched
    programmatically, the prologue writing its q into the buffer the first
    decode reads and its k / v into the pages both decodes read.  600
    requests give the first decode several waves of CTAs, so a prologue that
    wrote before that decode finished would change its later CTAs' q."""
    hq, hkv = 64, 8
    rng = np.random.default_rng(21)
    starts = [int(x) for x in rng.integers(1, 900, size=600)]
    w = workloads.prologue_batch([1] * len(starts), starts, seed=22)
    sinks = workloads.gpt_oss_sinks(rng, hq)
    q1 = torch.from_numpy(rng.standard_normal((len(starts), hq, 64)).astype(np.float32)).to(torch.bfloat16)
    inv, ms = sa.yarn_table()
    kc, vc = w["k_cache"].to(DEV), w["v_cache"].to(DEV)
    table, sk = w["page_table"].to(DEV), sinks.to(DEV)
    lens1 = torch.tensor(starts, dtype=torch.int32)
    lens2 = lens1 + 1
    qbuf = q1.to(DEV)
    out1, lse1 = sa.decode(qbuf, kc, vc, table, lens1.to(DEV), sk, 0.125, int(lens2.max()),
                           programmatic=True)
    sa.qkv_prologue(w["qkv"].to(DEV), w["bias"].to(DEV), w["positions"].to(DEV),
                    w["slot_mapping"].to(DEV), inv, ms, kc, vc, hq, hkv, q_out=qbuf)
    out2, lse2 = sa.decode(qbuf, kc, vc, table, lens2.to(DEV), sk, 0.125, int(lens2.max()),
                           programmatic=True)
    torch.cuda.synchronize()
    s64 = sinks.numpy().astype(np.float64)
    ro1, rl1 = oracle.decode(to_np(q1), Bf16Pool(w["k_cache"]), Bf16Pool(w["v_cache"]),
                             w["page_table"].numpy(), lens1.numpy(), s64, 0.125)
    assert_out_close(out1.cpu(), ro1)
    assert_lse_close(lse1.cpu(), rl1)
    # the prologue's own outputs at its bar (one bf16 ulp of the float64 reference) ...
    q2, k2, v2 = qbuf.cpu(), kc.cpu(), vc.cpu()
    rq, rk, rv = pro.qkv_prologue(to_np(w["qkv"]), to_np(w["bias"]), w["positions"].numpy(),
                                  np.asarray(inv, dtype=np.float64), ms, hq, hkv)
    slots = torch.from_numpy(w["slot_mapping"].numpy().astype(np.int64))
    assert_bf16_close(q2, rq, "q")
    assert_bf16_close(k2[slots // 16, :, slots % 16], rk, "k")
    assert_bf16_close(v2[slots // 16, :, slots % 16], rv, "v")
    # ... and the second decode against the oracle on exactly what it wrote
    ro2, rl2 = oracle.decode(to_np(q2), Bf16Pool(k2), Bf16Pool(v2), w["page_table"].numpy(),
                             lens2.numpy(), s64, 0.125)
    assert_out_close(out2.cpu(), ro2)
    assert_lse_close(lse2.cpu(), rl2)
