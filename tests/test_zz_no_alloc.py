"""The decode entry point for callers that cannot allocate device memory.

sinkattn_decode_static_scratch keeps its split scratch in a fixed device array
inside the library instead of a caller-provided workspace.  These tests call
it through the C ABI and compare it with sinkattn_decode (caller workspace) on
the same inputs, within the parity bars used for the oracle comparisons, on
two calls in a row (the array keeps the first call's contents).  This file is
collected last so that a failure here never hides the other tests.
"""

import ctypes

import pytest
import torch

import gqa_attention_learned_gb300 as sa
from gqa_attention_learned_gb300 import workloads
from tolerances import assert_lse_close, assert_out_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _inputs(w):
    return [w[n].to(DEV) for n in ("q", "k_cache", "v_cache", "page_table", "kv_lens", "sinks")]


def test_static_scratch_matches_workspace_decode_twice():
    w = workloads.decode_batch(seed=17, batch=24, min_len=1500, max_len=6000)
    args = _inputs(w)
    max_kv = w["max_kv_len"]
    splits, need = sa.decode_plan(24, 64, 8, max_kv, 0)
    assert splits > 1 and 0 < need <= sa.STATIC_SCRATCH_BYTES    # the scratch is really used
    ref_out, ref_lse = sa.decode(*args, w["scale"], max_kv)
    torch.cuda.synchronize()
    for _ in range(2):
        out, lse = sa.decode_static_scratch(*args, w["scale"], max_kv)
        torch.cuda.synchronize()
        assert_out_close(out.cpu(), to_np(ref_out), "static-scratch out")
        assert_lse_close(lse.cpu(), to_np(ref_lse), "static-scratch lse")


def test_static_scratch_with_other_inputs_after_first_call():
    # a second, differently sized problem right after: stale scratch contents
    # from the previous call must not leak into this one
    w = workloads.long_decode(seed=23, batch=2, min_len=20000, max_len=40000)
    args = _inputs(w)
    for splits in (0, 12):
        ref_out, ref_lse = sa.decode(*args, w["scale"], w["max_kv_len"], num_splits=splits)
        out, lse = sa.decode_static_scratch(*args, w["scale"], w["max_kv_len"], num_splits=splits)
        torch.cuda.synchronize()
        assert_out_close(out.cpu(), to_np(ref_out), "static-scratch out")
        assert_lse_close(lse.cpu(), to_np(ref_lse), "static-scratch lse")


def test_static_scratch_rejects_plans_beyond_its_size():
    # 1024 requests x 64 heads x 8 splits need ~136 MB of chunk slots: refused
    # on the host, nothing launched
    q = torch.zeros(1024, 64, 64, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(16, 8, 16, 64, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(1024, 1, dtype=torch.int32, device=DEV)
    lens = torch.ones(1024, dtype=torch.int32, device=DEV)
    sinks = torch.zeros(64, dtype=torch.float32, device=DEV)
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode_static_scratch(q, kc, kc, table, lens, sinks, 0.125, 4096, num_splits=8)
    assert e.value.status == sa.WORKSPACE_TOO_SMALL


def test_static_scratch_chained_under_programmatic_launch():
    # decode_static_scratch calls back to back with programmatic launch on,
    # each reading the previous call's output as its q: the scratch clear
    # (a memset on the stream) and the previous decode both precede the
    # kernel, which reads q only after its dependency wait
    w = workloads.decode_batch(seed=19, batch=24, min_len=1500, max_len=6000)
    args = _inputs(w)
    max_kv = w["max_kv_len"]

    def chain():
        q, outs = args[0], []
        for _ in range(4):
            out, lse = sa.decode_static_scratch(q, *args[1:], w["scale"], max_kv)
            outs.append((out, lse))
            q = out
        torch.cuda.synchronize()
        return outs

    prev = sa.set_programmatic_launch(True)
    try:
        fast = chain()
    finally:
        sa.set_programmatic_launch(False)
    try:
        q, slow = args[0], []
        for _ in range(4):
            out, lse = sa.decode(q, *args[1:], w["scale"], max_kv)
            torch.cuda.synchronize()
            slow.append((out, lse))
            q = out
    finally:
        sa.set_programmatic_launch(prev)
    for (a, la), (b, lb) in zip(fast, slow):
        assert_out_close(a.cpu(), to_np(b), "chained static-scratch out")
        assert_lse_close(la.cpu(), to_np(lb), "chained static-scratch lse")


def test_static_scratch_single_split_plans_match():
    # plans with one split use no scratch: an explicit num_splits = 1, and a
    # chosen plan that keeps whole requests (a wave of short requests)
    w = workloads.decode_batch(seed=29, batch=48, min_len=1, max_len=700)
    args = _inputs(w)
    assert sa.decode_plan(48, 64, 8, w["max_kv_len"], 0)[0] == 1
    for splits in (1, 0):
        ref_out, ref_lse = sa.decode(*args, w["scale"], w["max_kv_len"], num_splits=splits)
        for _ in range(2):
            out, lse = sa.decode_static_scratch(*args, w["scale"], w["max_kv_len"],
                                                num_splits=splits)
            torch.cuda.synchronize()
            assert_out_close(out.cpu(), to_np(ref_out), "single-split static-scratch out")
            assert_lse_close(lse.cpu(), to_np(ref_lse), "single-split static-scratch lse")


def _cudart():
    for name in ("libcudart.so.13", "libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("no shared CUDA runtime to inspect a captured graph with")


def _captured_nodes(fn):
    """Number of graph nodes that fn() enqueues on a fresh stream, seen by
    capturing the stream (relaxed mode) into a graph that is never run."""
    rt = _cudart()
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    rt.cudaStreamBeginCapture.argtypes = [vp, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [vp, ctypes.POINTER(vp)]
    rt.cudaGraphGetNodes.argtypes = [vp, vp, ctypes.POINTER(sz)]
    rt.cudaGraphDestroy.argtypes = [vp]
    s = torch.cuda.Stream()
    handle = vp(s.cuda_stream)
    assert rt.cudaStreamBeginCapture(handle, 2) == 0        # cudaStreamCaptureModeRelaxed
    try:
        fn(s.cuda_stream)
    finally:
        graph = vp()
        assert rt.cudaStreamEndCapture(handle, ctypes.byref(graph)) == 0
    n = sz(0)
    try:
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    finally:
        rt.cudaGraphDestroy(graph)
    return n.value


def test_static_scratch_refused_calls_queue_nothing():
    # every check runs before the merge-counter clear: a refused call leaves
    # no memset (and no launch) behind on its stream
    lib = sa.load()
    w = workloads.decode_batch(seed=31, batch=4, min_len=3000, max_len=4000)
    q, kc, vc, table, lens, sinks = _inputs(w)
    out = torch.empty_like(q)
    lse = torch.empty(4, 64, dtype=torch.float32, device=DEV)
    sa.decode_static_scratch(q, kc, vc, table, lens, sinks, w["scale"], w["max_kv_len"],
                             num_splits=8)                  # first call: address lookup
    torch.cuda.synchronize()
    P = lambda t: None if t is None else t.data_ptr()        # noqa: E731

    def call(stream, qp=q, hq=64, hkv=8, splits=8, scale=w["scale"]):
        return lib.sinkattn_decode_static_scratch(
            P(qp), P(kc), P(vc), P(table), table.shape[1], P(lens), P(sinks), scale, P(out),
            P(lse), 4, hq, hkv, 64, 16, kc.shape[0], w["max_kv_len"], splits, stream)

    statuses = []
    refused = [dict(qp=None),                               # null q
               dict(scale=float("inf")),                    # non-finite scale
               dict(hq=70000, hkv=70000),                   # KV heads x head blocks > 65535
               dict(splits=-1)]
    for kw in refused:
        assert _captured_nodes(lambda st, kw=kw: statuses.append(call(st, **kw))) == 0
    assert statuses == [sa.INVALID_ARGUMENT, sa.INVALID_ARGUMENT, sa.UNSUPPORTED,
                        sa.INVALID_ARGUMENT]
    # the same capture sees the clear and the launch of an accepted split call,
    # and only the launch of a single-split one
    assert _captured_nodes(lambda st: statuses.append(call(st))) == 2
    assert _captured_nodes(lambda st: statuses.append(call(st, splits=1))) == 1
    assert statuses[-2:] == [sa.OK, sa.OK]
