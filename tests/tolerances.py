"""Parity bars for comparing the CUDA path with the float64 oracle.

Outputs are bf16 with the stated max-abs bar of 1e-2.  Where |ref| >= 4 half
a bf16 ulp (1/64 there) already exceeds 1e-2, so even a correctly rounded
result can miss the bare bar; only there, an element beyond 1e-2 still passes
when it lies within one bf16 ulp of the reference rounded to bf16.  This only
happens for rows that see about one key with |v| > 4.  LSE is fp32 with a
max-abs bar of 1e-3; infinities must match exactly.

Every comparison is recorded per test (elements compared, max error, how
many references had |ref| >= 4, how many elements needed the one-ulp rule);
with SINKATTN_PARITY_REPORT=<path> set, the session writes the record there
as JSON (see conftest.py).
"""

import os

import numpy as np
import torch

OUT_ATOL = 1e-2
LSE_ATOL = 1e-3
WIDE_ABOVE = 4.0          # |ref| from which half a bf16 ulp exceeds OUT_ATOL

# test node id -> {"out": {...}, "lse": {...}}
RECORD = {}


def _record(kind, **stats):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    slot = RECORD.setdefault(test, {}).setdefault(kind, {"calls": 0, "elements": 0,
                                                          "max_err": 0.0})
    slot["calls"] += 1
    slot["elements"] += stats.pop("elements")
    slot["max_err"] = max(slot["max_err"], stats.pop("max_err"))
    for k, v in stats.items():
        slot[k] = slot.get(k, 0) + v


def bf16_ulp(ref):
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def round_bf16(ref):
    """float64 -> nearest bf16 (ties to even, via fp32), as float64."""
    t = torch.from_numpy(np.asarray(ref, dtype=np.float64).astype(np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def out_errors(gpu, ref):
    """(|gpu - ref|, pass mask): the 1e-2 bar, and for |ref| >= 4 also one
    bf16 ulp around the reference rounded to bf16."""
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    ok = err <= OUT_ATOL
    wide = np.abs(r) >= WIDE_ABOVE
    if np.any(wide & ~ok):
        near = np.abs(g - round_bf16(r)) <= bf16_ulp(r)
        ok = ok | (wide & near)
    return err, ok


def assert_out_close(gpu, ref, what="out"):
    g = to_np(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values in the GPU result"
    err, ok = out_errors(g, r)
    big = np.abs(r) >= WIDE_ABOVE
    _record("out", elements=int(err.size), max_err=float(err.max()) if err.size else 0.0,
            ref_ge_4=int(big.sum()), widened=int((ok & (err > OUT_ATOL)).sum()))
    if not np.all(ok):
        bad = ~ok
        i = np.unravel_index(np.argmax(np.where(bad, err, -1.0)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the bar; worst at {i}: "
                             f"gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3g} (bar {OUT_ATOL}, "
                             f"|ref| >= {WIDE_ABOVE}: one bf16 ulp)")
    return float(err.max()) if err.size else 0.0


def assert_lse_close(gpu, ref, what="lse"):
    g = to_np(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    inf_r = np.isinf(r)
    assert np.array_equal(np.isinf(g), inf_r) and np.array_equal(g[inf_r], r[inf_r]), \
        f"{what}: infinities differ"
    assert not np.any(np.isnan(g)), f"{what}: NaN in the GPU result"
    fin = ~inf_r
    err = np.abs(g[fin] - r[fin])
    _record("lse", elements=int(r.size), max_err=float(err.max()) if err.size else 0.0,
            infinite=int(inf_r.sum()))
    if err.size and err.max() > LSE_ATOL:
        raise AssertionError(f"{what}: max abs error {err.max():.3g} > {LSE_ATOL}")
    return float(err.max()) if err.size else 0.0


class Bf16Pool:
    """Read-only float64 view of a bf16 torch tensor, converted on indexing.

    Lets the oracle gather rows of a multi-GB paged pool without converting
    the whole pool to float64 up front."""

    def __init__(self, t):
        self.t = t.cpu()
        self.shape = tuple(t.shape)

    def __getitem__(self, idx):
        if not isinstance(idx, tuple):
            idx = (idx,)
        idx = tuple(torch.as_tensor(i) if isinstance(i, np.ndarray) else i for i in idx)
        return self.t[idx].float().numpy().astype(np.float64)
