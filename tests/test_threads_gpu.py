"""Concurrent host threads: the C ABI promises thread-safe calls (its only
state is per-device caches and the launch-mode switch).  Four threads, each
on its own stream, run decode (a split plan with its own workspace) and
tensor-core verification back to back; every result must equal the same call
made alone, bit for bit, in both launch modes."""

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
