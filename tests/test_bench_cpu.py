"""Host-side pieces of bench.py (CPU): the algorithmic byte and FLOP counts
the roofline divides by, the pool copies that keep earlier steps' pages out
of L2, and the traffic figure that lapses when a kernel source changes."""

import math

import torch

import bench


def test_decode_bytes_by_hand():
    # 2 requests of 16 and 1 keys, 2 query heads on 1 KV head, D = 64:
    # K and V rows 17 * 1 * 64 * 2 B * 2 = 4352; q and out 2 * 2 * 64 * 2 B * 2 = 1024;
    # lse 2 * 2 * 4 = 16; sinks 2 * 4 = 8; kv_lens 2 * 4 = 8; one page each: 2 * 4 = 8
    assert bench.decode_bytes([16, 1], 2, 1) == 4352 + 1024 + 16 + 8 + 8 + 8


def test_decode_bytes_scale_with_keys_and_heads():
    one = bench.decode_bytes([4096], 64, 8)
    two = bench.decode_bytes([4096, 4096], 64, 8)
    kv = 4096 * 8 * 64 * 2 * 2
    assert two - one == kv + 2 * 64 * 64 * 2 + 64 * 4 + 4 + 256 * 4


def test_prefill_flops_by_hand():
    # QK^T and P V over the causal pairs: 4 D Hq L (L + 1) / 2
    assert bench.prefill_flops([3], 1) == 4 * 64 * 6
    assert bench.prefill_flops([3, 1], 2) == 4 * 64 * 2 * (6 + 1)


def test_extend_flops_reduce_to_prefill_without_prefix():
    assert bench.extend_flops([5], [5], 4) == bench.prefill_flops([5], 4)
    # a prefix of P keys adds Lq * P pairs
    assert bench.extend_flops([5], [12], 4) == bench.prefill_flops([5], 4) + 4 * 64 * 4 * 5 * 7


def test_pool_copies_cover_the_reuse_distance(monkeypatch):
    k = torch.zeros(8, 2, 16, 64, dtype=torch.bfloat16)
    v = torch.ones_like(k)
    pool_bytes = 2 * k.numel() * k.element_size()
    monkeypatch.setattr(bench, "REUSE_BYTES", 5 * pool_bytes)
    pools = bench.kv_pools(torch, k, v, "cpu")
    assert len(pools) == math.ceil(bench.REUSE_BYTES / pool_bytes) + 1 == 6
    # a page comes back only after REUSE_BYTES of other copies
    assert (len(pools) - 1) * pool_bytes >= bench.REUSE_BYTES
    ptrs = {t.data_ptr() for kc, vc in pools for t in (kc, vc)}
    assert len(ptrs) == 2 * len(pools)                     # distinct storage
    assert all(torch.equal(kc, k) and torch.equal(vc, v) for kc, vc in pools)
    assert "6 KV pool copies" in bench.pools_label(pools)


def test_pool_copies_bounds(monkeypatch):
    k = torch.zeros(4, 1, 16, 64, dtype=torch.bfloat16)
    monkeypatch.setattr(bench, "REUSE_BYTES", 1.0)
    assert len(bench.kv_pools(torch, k, k, "cpu")) == 2      # at least two
    monkeypatch.setattr(bench, "REUSE_BYTES", 1e15)
    assert len(bench.kv_pools(torch, k, k, "cpu")) == 32     # at most 32


def test_traffic_lapses_when_a_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// version 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.sources_hash(["kernel.cu"])
    monkeypatch.setitem(bench.TRAFFIC, "probe", {"sources": ("kernel.cu",), "sha256_16": h,
                                                 "bytes": 1234})
    assert bench.kernel_traffic("probe") == 1234
    src.write_text("// version 2\n")
    assert bench.kernel_traffic("probe") is None
    src.unlink()
    assert bench.kernel_traffic("probe") is None
