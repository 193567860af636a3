"""The C ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before touching a GPU (no compute calls here)."""

import ctypes
import os
import re

import pytest

import gqa_attention_learned_gb300 as sa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sinkattn.h")


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"SINKATTN_API\s+[^;(]*?\b(sinkattn_\w+)\s*\(", text)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(sa.LIB_PATH):
        from gqa_attention_learned_gb300 import build
        build.build()
    return sa.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 6
    for name in names:
        assert hasattr(lib, name), name
        assert name in sa.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    assert sa.status_string(0) == "ok"
    assert "workspace" in sa.status_string(3)
    assert sa.status_string(99) == "unknown status"
    assert lib.sinkattn_version() >= 100


def test_plan_is_host_only_and_deterministic(lib):
    a = sa.decode_plan(64, 64, 8, 4096, num_sms=152)
    b = sa.decode_plan(64, 64, 8, 4096, num_sms=152)
    assert a == b
    splits, ws = a
    assert splits >= 1
    assert (ws == 0) == (splits == 1)
    # explicit split counts are honoured up to the page count; the workspace
    # holds the merge counters (one per request and KV head, 256-byte
    # rounded) and one (o, lse) slot per chunk and query head
    s, ws = sa.decode_plan(8, 64, 8, 131072, num_splits=8, num_sms=152)
    assert s == 8 and ws == 256 + 8 * 8 * 64 * 64 * 4 + 8 * 8 * 64 * 4
    s, _ = sa.decode_plan(1, 4, 1, 37, num_splits=64, num_sms=152)
    assert s == 3      # 37 tokens = 3 pages: at most one page per split
    s, ws = sa.decode_plan(4, 4, 1, 0, num_sms=152)
    assert s == 1 and ws == 0


def test_plan_long_context_splits(lib):
    s, _ = sa.decode_plan(8, 64, 8, 131072, num_sms=152)
    assert 8 <= s <= 1024


def test_plan_rejects_bad_arguments(lib):
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode_plan(1, 64, 8, 100, head_dim=128, num_sms=1)
    assert e.value.status == sa.UNSUPPORTED
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode_plan(1, 64, 8, 100, page_size=32, num_sms=1)
    assert e.value.status == sa.UNSUPPORTED
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode_plan(1, 60, 8, 100, num_sms=1)
    assert e.value.status == sa.INVALID_ARGUMENT
    with pytest.raises(sa.SinkAttnError) as e:
        sa.decode_plan(-1, 64, 8, 100, num_sms=1)
    assert e.value.status == sa.INVALID_ARGUMENT


def _raw_decode(lib, **kw):
    args = dict(q=None, k=None, v=None, table=None, maxp=1, lens=None, sinks=None, scale=0.125,
                out=None, lse=None, batch=1, hq=8, hkv=1, d=64, page=16, pages=1, maxkv=16,
                splits=0, ws=None, wsb=0, stream=None)
    args.update(kw)
    return lib.sinkattn_decode(*args.values())


def test_decode_rejects_on_host(lib):
    fake = ctypes.c_void_p(0x1000)
    assert _raw_decode(lib, d=128) == sa.UNSUPPORTED
    assert _raw_decode(lib, page=8) == sa.UNSUPPORTED
    assert _raw_decode(lib, hq=6, hkv=4) == sa.INVALID_ARGUMENT
    assert _raw_decode(lib, pages=0) == sa.INVALID_ARGUMENT
    assert _raw_decode(lib, scale=float("nan")) == sa.INVALID_ARGUMENT
    assert _raw_decode(lib) == sa.INVALID_ARGUMENT                       # null pointers
    odd = ctypes.c_void_p(0x1008)
    assert _raw_decode(lib, q=odd, k=fake, v=fake, table=fake, lens=fake, sinks=fake,
                       out=fake) == sa.INVALID_ARGUMENT                  # misaligned q
    assert _raw_decode(lib, batch=0) == sa.OK                            # nothing to do
    ok = dict(q=fake, k=fake, v=fake, table=fake, lens=fake, sinks=fake, out=fake)
    assert _raw_decode(lib, batch=65536, **ok) == sa.UNSUPPORTED          # documented limit
    assert _raw_decode(lib, batch=1, hq=65536 * 8, hkv=65536, **ok) == sa.UNSUPPORTED


def test_decode_ex_rejects_unknown_launch_flags_on_host(lib):
    # the flags are checked before anything else, so no device is needed
    args = [None, None, None, None, 1, None, None, 0.125, None, None, 1, 8, 1, 64, 16, 1, 16, 0,
            None, 0]
    for flags in (-1, 3, 7):
        assert lib.sinkattn_decode_ex(*args, flags, None) == sa.INVALID_ARGUMENT
    vargs = [None, None, None, None, 1, None, None, None, 0.125, None, None, 1, 2, 8, 1, 64, 16,
             1, 16, 0, None, 0]
    assert lib.sinkattn_verify_ex(*vargs, 3, None) == sa.INVALID_ARGUMENT
    # a valid mode goes on to the ordinary checks (null pointers here)
    for flags in (sa.LAUNCH_DEFAULT, sa.LAUNCH_PLAIN, sa.LAUNCH_PROGRAMMATIC):
        assert lib.sinkattn_decode_ex(*args, flags, None) == sa.INVALID_ARGUMENT
        assert lib.sinkattn_decode_ex(*args[:13], 128, *args[14:], flags,
                                      None) == sa.UNSUPPORTED


@pytest.mark.parametrize("batch,hq", [(1, 1), (8, 64), (64, 64), (3, 40), (1000, 128)])
def test_decode_workspace_bytes_bounds_every_plan(lib, batch, hq):
    assert sa.decode_workspace_bytes(batch, hq, 0) == 0
    assert sa.decode_workspace_bytes(batch, hq, 1) == 0
    assert sa.decode_workspace_bytes(batch, hq, 4, head_dim=128) == 0
    for splits in (2, 3, 8, 64, 1024):
        bound = sa.decode_workspace_bytes(batch, hq, splits)
        assert bound > 0 and bound % 256 == 0
        for hkv in [h for h in (1, 2, 4, 8, 16, 40, 64, 128) if h <= hq and hq % h == 0]:
            for max_kv in (16, 700, 4096, 131072):
                s, ws = sa.decode_plan(batch, hq, hkv, max_kv, num_splits=splits, num_sms=152)
                assert s <= splits and ws <= bound, (splits, hkv, max_kv, s, ws, bound)
    # with group 1 the counters take one int per (request, head): the bound is exact
    s, ws = sa.decode_plan(batch, hq, hq, 1 << 20, num_splits=8, num_sms=152)
    assert s == 8 and ws == sa.decode_workspace_bytes(batch, hq, 8)


def _counter_bytes(units):
    return (units * 4 + 255) // 256 * 256


def _split_workspace(batch, hq, splits, counters_units):
    rows = splits * batch * hq
    return _counter_bytes(counters_units) + rows * 64 * 4 + (rows * 4 + 255) // 256 * 256


def test_plan_takes_16_head_ctas_when_they_fill_a_wave(lib):
    # 2 CTAs per SM x 152 SMs = 304 slots.  GQA group 16 (32 q / 2 KV heads):
    # 160 requests give 320 (request, KV head) units of 16 heads, a full
    # wave, so one merge counter per unit; 100 requests give 200, so the plan
    # keeps 8-head CTAs (two per unit, two counters)
    s, ws = sa.decode_plan(160, 32, 2, 4096, num_splits=2, num_sms=152)
    assert s == 2 and ws == _split_workspace(160, 32, 2, 160 * 2)
    s, ws = sa.decode_plan(100, 32, 2, 4096, num_splits=2, num_sms=152)
    assert s == 2 and ws == _split_workspace(100, 32, 2, 100 * 2 * 2)
    # group 32: two 16-head CTAs per KV head when wide, four 8-head ones when not
    s, ws = sa.decode_plan(80, 64, 2, 4096, num_splits=2, num_sms=152)
    assert ws == _split_workspace(80, 64, 2, 80 * 2 * 2)
    s, ws = sa.decode_plan(40, 64, 2, 4096, num_splits=2, num_sms=152)
    assert ws == _split_workspace(40, 64, 2, 40 * 2 * 4)
    # groups of 8 or less always use 8-head CTAs
    s, ws = sa.decode_plan(400, 64, 8, 4096, num_splits=2, num_sms=152)
    assert ws == _split_workspace(400, 64, 2, 400 * 8)


def test_programmatic_launch_switch_is_host_state(lib):
    prev = sa.set_programmatic_launch(True)
    try:
        assert lib.sinkattn_set_programmatic_launch(0) == 1
        assert lib.sinkattn_set_programmatic_launch(5) == 0              # any non-zero = on
        assert sa.set_programmatic_launch(False) is True
    finally:
        sa.set_programmatic_launch(prev)


def test_prefill_rejects_on_host(lib):
    assert lib.sinkattn_prefill(None, None, None, None, 1, 16, 16, None, 0.125, None, None,
                                8, 1, 128, None) == sa.UNSUPPORTED
    assert lib.sinkattn_prefill(None, None, None, None, 1, 16, 16, None, 0.125, None, None,
                                8, 1, 64, None) == sa.INVALID_ARGUMENT
    assert lib.sinkattn_prefill_paged(None, None, 1, 16, 16, None, None, None, 1, None, 1, 16,
                                      None, 0.125, None, None, 8, 1, 64, 32,
                                      None) == sa.UNSUPPORTED


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(sa, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(sa, "_lib", None)
    with pytest.raises(RuntimeError):
        sa.load()


def test_verify_plan(lib):
    # q_len = 1 plans exactly like decode
    assert sa.verify_plan(64, 1, 64, 8, 4096, num_sms=152) == sa.decode_plan(64, 64, 8, 4096,
                                                                             num_sms=152)
    # 4 tokens x 8 heads = 32 rows per KV head = 2 CTAs of 16 rows; the
    # workspace holds one counter per (request, KV head, CTA) and one
    # (o, lse) slot per chunk and query row
    s, ws = sa.verify_plan(8, 4, 64, 8, 131072, num_splits=8, num_sms=152)
    counters = 8 * 8 * 2 * 4               # batch x Hkv x CTAs per KV head, int32
    rows = 8 * 8 * 4 * 64                  # chunks x batch x q_len x Hq
    assert s == 8
    assert ws == counters + rows * 64 * 4 + rows * 4
    with pytest.raises(sa.SinkAttnError) as e:
        sa.verify_plan(1, sa.MAX_VERIFY_TOKENS + 1, 64, 8, 4096, num_sms=152)
    assert e.value.status == sa.INVALID_ARGUMENT
    with pytest.raises(sa.SinkAttnError) as e:
        sa.verify_plan(1, 0, 64, 8, 4096, num_sms=152)
    assert e.value.status == sa.INVALID_ARGUMENT


def test_verify_rejects_on_host(lib):
    fake = ctypes.c_void_p(0x1000)

    def call(**kw):
        a = dict(q=fake, k=fake, v=fake, table=fake, maxp=1, lens=fake, mask=None, sinks=fake,
                 scale=0.125, out=fake, lse=None, batch=1, q_len=2, hq=8, hkv=1, d=64, page=16,
                 pages=1, maxkv=16, splits=1, ws=None, wsb=0, stream=None)
        a.update(kw)
        return lib.sinkattn_verify(*a.values())

    assert call(d=128) == sa.UNSUPPORTED
    assert call(q_len=0) == sa.INVALID_ARGUMENT
    assert call(q_len=sa.MAX_VERIFY_TOKENS + 1) == sa.INVALID_ARGUMENT
    assert call(mask=ctypes.c_void_p(0x1004)) == sa.INVALID_ARGUMENT     # misaligned mask
    assert call(q=None) == sa.INVALID_ARGUMENT
    assert call(batch=0) == sa.OK


def test_yarn_table_matches_oracle(lib):
    from oracle import prologue as pro
    for args in ((64, 150000.0, 32.0, 4096, 32.0, 1.0), (64, 10000.0, 1.0, 2048, 32.0, 1.0),
                 (64, 500000.0, 8.0, 8192, 16.0, 2.0)):
        f, m = sa.yarn_table(*args)
        fo, mo = pro.yarn_inv_freq(*args)
        assert len(f) == 32
        np_f = [float(x) for x in f]
        for a, b in zip(np_f, fo):
            assert abs(a - b) <= 2 ** -23 * abs(b)          # one float rounding
        assert abs(m - mo) <= 2 ** -23 * mo
    with pytest.raises(sa.SinkAttnError):
        sa.yarn_table(factor=0.5)
    with pytest.raises(sa.SinkAttnError):
        sa.yarn_table(beta_fast=1.0, beta_slow=1.0)


def test_prologue_rejects_on_host(lib):
    fake = ctypes.c_void_p(0x1000)
    freq = (ctypes.c_float * 32)(*([0.5] * 32))

    def call(**kw):
        a = dict(qkv=fake, bias=None, pos=fake, slots=fake, freq=freq, ms=1.0, style=0, q=fake,
                 k=fake, v=fake, t=4, hq=8, hkv=1, d=64, page=16, pages=1, stream=None)
        a.update(kw)
        return lib.sinkattn_qkv_prologue(*a.values())

    assert call(d=128) == sa.UNSUPPORTED
    assert call(page=32) == sa.UNSUPPORTED
    assert call(style=2) == sa.INVALID_ARGUMENT
    assert call(qkv=ctypes.c_void_p(0x1008)) == sa.INVALID_ARGUMENT
    assert call(bias=ctypes.c_void_p(0x1004)) == sa.INVALID_ARGUMENT
    assert call(freq=(ctypes.c_float * 32)(*([float("nan")] * 32))) == sa.INVALID_ARGUMENT
    assert call(t=0) == sa.OK
