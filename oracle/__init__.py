"""Float64 CPU oracle for sink attention.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
CPU-baseline legs of bench.py, never by the product path.
"""
from .sink_attention import (NEG_INF, decode, gather_paged_kv, kv_head_of,
                             merge_blocks, online_block, prefill, prefill_paged,
                             sink_attention, split_sink_attention, verify)

__all__ = ["NEG_INF", "decode", "gather_paged_kv", "kv_head_of", "merge_blocks",
           "online_block", "prefill", "prefill_paged", "sink_attention",
           "split_sink_attention", "verify"]
