"""Concurrent host threads: the C ABI promises thread-safe calls (its only
state is per-device caches and the default launch mode).  Four threads, each
on its own stream, run decode (a split plan with its own workspace) and
tensor-core verification back to back; every result must equal the same call
made alone, bit for bit, in both launch modes.  Threads that pick different
launch modes per call do not affect one another."""

import threading

import pytest
import torch

import gqa_attention_learned_gb300 as sa
from gqa_attention_learned_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _dev(w):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in w.items()}


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("programmatic", [False, True])
def test_concurrent_threads_match_single_calls(programmatic):
    dw = _dev(workloads.decode_batch(seed=21, batch=16, min_len=2000, max_len=6000))
    vw = _dev(workloads.verify_batch(seed=22, batch=64, q_len=4, max_len=1500))
    splits, _ = sa.decode_plan(16, 64, 8, dw["max_kv_len"])
    assert splits > 1                               # the workspace path runs concurrently too
    assert sa.verify_plan(64, 4, 64, 8, vw["max_kv_len"]) == (1, 0)

    def decode(stream=None):
        return sa.decode(dw["q"], dw["k_cache"], dw["v_cache"], dw["page_table"], dw["kv_lens"],
                         dw["sinks"], dw["scale"], dw["max_kv_len"], stream=stream)

    def verify(stream=None):
        return sa.verify(vw["q"], vw["k_cache"], vw["v_cache"], vw["page_table"], vw["kv_lens"],
                         vw["sinks"], vw["scale"], vw["max_kv_len"], stream=stream)

    prev = sa.set_programmatic_launch(programmatic)
    try:
        ref = decode() + verify()
        torch.cuda.synchronize()
        results, errors = [None] * 4, []

        def worker(i):
            try:
                torch.cuda.set_device(0)
                s = torch.cuda.Stream()
                with torch.cuda.stream(s):
                    for _ in range(10):
                        got = decode(s) + verify(s)
                s.synchronize()
                results[i] = got
            except Exception as exc:                # reported on the main thread
                errors.append(exc)

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        for got in results:
            for a, b in zip(got, ref):
                assert torch.equal(_bits(a), _bits(b))
    finally:
        sa.set_programmatic_launch(prev)


def test_threads_with_their_own_launch_modes():
    # one thread launches programmatically, the other plainly, each chaining
    # decode -> decode (q = the previous output) and a tensor-core
    # verification on its own stream, while the process-wide default stays
    # off; both must equal the same chain made one call at a time
    dw = _dev(workloads.decode_batch(seed=23, batch=16, min_len=2000, max_len=6000))
    vw = _dev(workloads.verify_batch(seed=24, batch=64, q_len=4, max_len=1500))
    assert sa.decode_plan(16, 64, 8, dw["max_kv_len"])[0] > 1

    def chain(mode, stream=None):
        q, got = dw["q"], []
        for _ in range(6):
            out, lse = sa.decode(q, dw["k_cache"], dw["v_cache"], dw["page_table"],
                                 dw["kv_lens"], dw["sinks"], dw["scale"], dw["max_kv_len"],
                                 stream=stream, programmatic=mode)
            got += [out, lse]
            q = out
        got += list(sa.verify(vw["q"], vw["k_cache"], vw["v_cache"], vw["page_table"],
                              vw["kv_lens"], vw["sinks"], vw["scale"], vw["max_kv_len"],
                              stream=stream, programmatic=mode))
        return got

    prev = sa.set_programmatic_launch(False)
    try:
        ref = chain(False)
        torch.cuda.synchronize()
        results, errors = {}, []

        def worker(mode):
            try:
                torch.cuda.set_device(0)
                s = torch.cuda.Stream()
                with torch.cuda.stream(s):
                    for _ in range(5):
                        got = chain(mode, s)
                s.synchronize()
                results[mode] = got
            except Exception as exc:                # reported on the main thread
                errors.append(exc)

        threads = [threading.Thread(target=worker, args=(m,)) for m in (True, False)]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        assert sa.set_programmatic_launch(False) is False    # the default never changed
        for mode in (True, False):
            for a, b in zip(results[mode], ref):
                assert torch.equal(_bits(a), _bits(b)), mode
    finally:
        sa.set_programmatic_launch(prev)
