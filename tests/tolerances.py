"""Parity bars for comparing the CUDA path with the float64 oracle.

Outputs are bf16: the bar is max-abs 1e-2, widened to one bf16 ulp of the
reference where |ref| >= 4 (there half an ulp already exceeds 1e-2, so even a
correctly rounded result can miss a bare 1e-2; this only happens when a row
sees about one key and |v| > 4).  LSE is fp32 with a max-abs bar of 1e-3;
infinities must match exactly.
"""

import math

import numpy as np
import torch

OUT_ATOL = 1e-2
LSE_ATOL = 1e-3


def bf16_ulp(ref):
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


def out_errors(gpu, ref):
    g, r = to_np(gpu), np.asarray(ref, dtype=np.float64)
    err = np.abs(g - r)
    allowed = np.maximum(OUT_ATOL, bf16_ulp(r))
    return err, allowed


def assert_out_close(gpu, ref, what="out"):
    g = to_np(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values in the GPU result"
    err, allowed = out_errors(g, r)
    bad = err > allowed
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - allowed), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the bar; worst at {i}: "
                             f"gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3g} allowed={allowed[i]:.3g}")
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
