"""Python binding of libsinkattn (GQA attention with learned per-head sinks).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/sinkattn.h``.  PyTorch supplies
device memory and the current stream.  There is no fallback: if the shared
library is missing or fails to load, every call raises.
"""

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsinkattn.so")

OK, INVALID_ARGUMENT, UNSUPPORTED, WORKSPACE_TOO_SMALL, CUDA_ERROR = range(5)

_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes), in the order of include/sinkattn.h
SIGNATURES = {
    "sinkattn_status_string": (ctypes.c_char_p, [_c_int]),
    "sinkattn_version": (_c_int, []),
    "sinkattn_last_error": (ctypes.c_char_p, []),
    "sinkattn_set_programmatic_launch": (_c_int, [_c_int]),
    "sinkattn_decode_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                      ctypes.POINTER(_c_int), ctypes.POINTER(_c_size)]),
    "sinkattn_decode_workspace_bytes": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "sinkattn_decode": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_float, _vp, _vp,
                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _vp, _c_size, _vp]),
    "sinkattn_decode_ex": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_float, _vp, _vp,
                                    _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _vp, _c_size, _c_int, _vp]),
    "sinkattn_verify_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                      _c_int, ctypes.POINTER(_c_int), ctypes.POINTER(_c_size)]),
    "sinkattn_verify": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _vp, _c_float, _vp, _vp,
                                 _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                 _c_int, _vp, _c_size, _vp]),
    "sinkattn_verify_ex": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _vp, _c_float, _vp,
                                    _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _vp, _c_size, _c_int, _vp]),
    "sinkattn_prefill": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _vp, _c_float, _vp,
                                  _vp, _c_int, _c_int, _c_int, _vp]),
    "sinkattn_prefill_paged": (_c_int, [_vp, _vp, _c_int, _c_int, _c_int, _vp, _vp, _vp, _c_int,
                                        _vp, _c_int, _c_int, _vp, _c_float, _vp, _vp, _c_int,
                                        _c_int, _c_int, _c_int, _vp]),
    "sinkattn_yarn_table": (_c_int, [_c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                     ctypes.c_double, ctypes.c_double,
                                     ctypes.POINTER(_c_float), ctypes.POINTER(_c_float)]),
    "sinkattn_qkv_prologue": (_c_int, [_vp, _vp, _vp, _vp, ctypes.POINTER(_c_float), _c_float,
                                       _c_int, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _vp]),
    "sinkattn_decode_static_scratch": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_float,
                                                _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                                                _c_int, _c_int, _c_int, _vp]),
}

STATIC_SCRATCH_BYTES = 16 << 20
LAUNCH_DEFAULT, LAUNCH_PLAIN, LAUNCH_PROGRAMMATIC = 0, 1, 2
ROPE_HALF, ROPE_INTERLEAVED = 0, 1
MAX_VERIFY_TOKENS = 64

_lib = None


class SinkAttnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        detail = ""
        if status == CUDA_ERROR:
            detail = ": " + load().sinkattn_last_error().decode()
        super().__init__(f"{fn} failed: {status_string(status)} ({status}){detail}")


def load():
    """Load libsinkattn.so (built by ``build.build()``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsinkattn.so not built ({LIB_PATH}); run "
                               "`python -m gqa_attention_learned_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def status_string(status):
    return load().sinkattn_status_string(int(status)).decode()


def set_programmatic_launch(enable):
    """Process-wide DEFAULT launch mode of the decode and verification
    kernels (decode, decode_static_scratch, verify called without
    `programmatic=`); returns the previous setting.  In programmatic mode,
    kv_lens and page_table of a call must not be written by the kernel
    launched just before it on the stream."""
    return bool(load().sinkattn_set_programmatic_launch(1 if enable else 0))


def _launch_flags(programmatic):
    """None: the process-wide default; True / False: this call's own mode."""
    if programmatic is None:
        return LAUNCH_DEFAULT
    return LAUNCH_PROGRAMMATIC if programmatic else LAUNCH_PLAIN


def _check(fn, status):
    if status != OK:
        raise SinkAttnError(fn, status)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _on(dev):
    """Makes `dev` the current device for a call (no-op when it already is)."""
    if dev.index is None or dev.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(dev)


_plans = {}
_PLANS_KEPT = 4096


def _plan(fn, *args):
    """fn(*args) for the current device, memoised: plans depend only on
    host-side sizes and the device's SM count (at most _PLANS_KEPT kept)."""
    key = (fn.__name__, torch.cuda.current_device()) + args
    hit = _plans.get(key)
    if hit is None:
        if len(_plans) >= _PLANS_KEPT:
            _plans.clear()
        hit = _plans[key] = fn(*args)
    return hit


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _want(t, name, dtype, dims=None, device=None):
    if (isinstance(t, torch.Tensor) and t.dtype == dtype and (dims is None or t.dim() == dims)
            and t.is_cuda and (device is None or t.device == device) and t.is_contiguous()):
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def decode_plan(batch, num_qo_heads, num_kv_heads, max_kv_len, num_splits=0, num_sms=0,
                head_dim=64, page_size=16):
    """(split count, workspace bytes) that `decode` will use (host only).  A
    workspace must be zero-filled before its first use (torch.zeros)."""
    s = _c_int(num_splits)
    w = _c_size(0)
    _check("sinkattn_decode_plan",
           load().sinkattn_decode_plan(batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                                       max_kv_len, num_sms, ctypes.byref(s), ctypes.byref(w)))
    return s.value, w.value


def decode_workspace_bytes(batch, num_qo_heads, num_splits, head_dim=64):
    """Upper bound on decode's workspace for an explicit split count, valid
    for any KV head count (host only; 0 for one split)."""
    return int(load().sinkattn_decode_workspace_bytes(batch, num_qo_heads, head_dim, num_splits))


def decode(q, k_cache, v_cache, page_table, kv_lens, sinks, scale, max_kv_len, *, out=None,
           lse=None, num_splits=0, workspace=None, stream=None, want_lse=True, programmatic=None):
    """Paged decode.  q [B, Hq, 64] bf16; caches [pages, Hkv, 16, 64] bf16;
    page_table [B, max_pages] int32; kv_lens [B] int32; sinks [Hq] fp32.
    programmatic: None = the process-wide default launch mode, True / False =
    this call's own.  Returns (out [B, Hq, 64] bf16, lse [B, Hq] fp32 or None)."""
    dev = q.device
    _want(q, "q", torch.bfloat16, 3)
    _want(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _want(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _want(page_table, "page_table", torch.int32, 2, dev)
    _want(kv_lens, "kv_lens", torch.int32, 1, dev)
    _want(sinks, "sinks", torch.float32, 1, dev)
    batch, hq, d = q.shape
    num_pages, hkv, page, d2 = k_cache.shape
    if v_cache.shape != k_cache.shape or d2 != d:
        raise ValueError("k_cache/v_cache shapes disagree with q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(batch, hq, dtype=torch.float32, device=dev)
    with _on(dev):
        splits, ws_bytes = _plan(decode_plan, batch, hq, hkv, int(max_kv_len), int(num_splits),
                                 0, d, page) if batch else (1, 0)
        if workspace is None and ws_bytes:
            # zero-filled once; decode leaves it ready for the next call
            workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check("sinkattn_decode_ex", load().sinkattn_decode_ex(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1],
            _ptr(kv_lens), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), batch, hq, hkv, d,
            page, num_pages, int(max_kv_len), int(num_splits), _ptr(workspace), ws_len,
            _launch_flags(programmatic), _stream(stream)))
    return out, lse


def verify_plan(batch, q_len, num_qo_heads, num_kv_heads, max_kv_len, num_splits=0, num_sms=0,
                head_dim=64, page_size=16):
    """(split count, workspace bytes) that `verify` will use (host only)."""
    s = _c_int(num_splits)
    w = _c_size(0)
    _check("sinkattn_verify_plan",
           load().sinkattn_verify_plan(batch, q_len, num_qo_heads, num_kv_heads, head_dim,
                                       page_size, max_kv_len, num_sms, ctypes.byref(s),
                                       ctypes.byref(w)))
    return s.value, w.value


def verify(q, k_cache, v_cache, page_table, kv_lens, sinks, scale, max_kv_len, *, tree_mask=None,
           out=None, lse=None, num_splits=0, workspace=None, stream=None, want_lse=True,
           programmatic=None):
    """Verification of the q_len newest tokens of every request (speculative
    decoding).  q [B, q_len, Hq, 64] bf16; the tokens are the last q_len keys
    of each request's paged KV.  tree_mask: None (causal) or int64
    [B, q_len] holding the uint64 bit masks (bit u of row i: token i sees
    draft token u).  programmatic: as for decode.  Returns
    (out [B, q_len, Hq, 64], lse [B, q_len, Hq])."""
    dev = q.device
    _want(q, "q", torch.bfloat16, 4)
    _want(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _want(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _want(page_table, "page_table", torch.int32, 2, dev)
    _want(kv_lens, "kv_lens", torch.int32, 1, dev)
    _want(sinks, "sinks", torch.float32, 1, dev)
    batch, q_len, hq, d = q.shape
    if tree_mask is not None:
        _want(tree_mask, "tree_mask", torch.int64, 2, dev)
        if tuple(tree_mask.shape) != (batch, q_len):
            raise ValueError("tree_mask must be [batch, q_len]")
    num_pages, hkv, page, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(batch, q_len, hq, dtype=torch.float32, device=dev)
    with _on(dev):
        splits, ws_bytes = _plan(verify_plan, batch, q_len, hq, hkv, int(max_kv_len),
                                 int(num_splits), 0, d, page) if batch else (1, 0)
        if workspace is None and ws_bytes:
            workspace = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
        _check("sinkattn_verify_ex", load().sinkattn_verify_ex(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1],
            _ptr(kv_lens), _ptr(tree_mask), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), batch,
            q_len, hq, hkv, d, page, num_pages, int(max_kv_len), int(num_splits), _ptr(workspace),
            ws_len, _launch_flags(programmatic), _stream(stream)))
    return out, lse


def prefill(q, k, v, cu_seqlens, sinks, scale, max_seqlen, *, out=None, lse=None, stream=None,
            want_lse=True):
    """Ragged causal prefill.  q [T, Hq, 64], k/v [T, Hkv, 64] bf16;
    cu_seqlens [n+1] int32.  Returns (out [T, Hq, 64], lse [T, Hq] or None)."""
    dev = q.device
    _want(q, "q", torch.bfloat16, 3)
    _want(k, "k", torch.bfloat16, 3, dev)
    _want(v, "v", torch.bfloat16, 3, dev)
    _want(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
    _want(sinks, "sinks", torch.float32, 1, dev)
    total, hq, d = q.shape
    hkv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != total or k.shape[2] != d:
        raise ValueError("q/k/v shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(total, hq, dtype=torch.float32, device=dev)
    with _on(dev):
        _check("sinkattn_prefill", load().sinkattn_prefill(
            _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), cu_seqlens.numel() - 1, total,
            int(max_seqlen), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), hq, hkv, d,
            _stream(stream)))
    return out, lse


def prefill_paged(q, cu_seqlens_q, k_cache, v_cache, page_table, kv_lens, sinks, scale,
                  max_q_len, max_kv_len, *, out=None, lse=None, stream=None, want_lse=True):
    """Chunked prefill against a paged KV prefix (bottom-right causal)."""
    dev = q.device
    _want(q, "q", torch.bfloat16, 3)
    _want(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, dev)
    _want(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _want(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _want(page_table, "page_table", torch.int32, 2, dev)
    _want(kv_lens, "kv_lens", torch.int32, 1, dev)
    _want(sinks, "sinks", torch.float32, 1, dev)
    total, hq, d = q.shape
    num_pages, hkv, page, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(total, hq, dtype=torch.float32, device=dev)
    with _on(dev):
        _check("sinkattn_prefill_paged", load().sinkattn_prefill_paged(
            _ptr(q), _ptr(cu_seqlens_q), cu_seqlens_q.numel() - 1, total, int(max_q_len),
            _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1], _ptr(kv_lens),
            num_pages, int(max_kv_len), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), hq, hkv,
            d, page, _stream(stream)))
    return out, lse


def decode_static_scratch(q, k_cache, v_cache, page_table, kv_lens, sinks, scale, max_kv_len, *,
                          out=None, lse=None, num_splits=0, stream=None, want_lse=True):
    """Decode for callers that cannot allocate device memory: the split
    scratch is the library's own fixed 16 MiB device array instead of a
    caller-provided workspace.  Raises SinkAttnError (WORKSPACE_TOO_SMALL)
    when the sizes need more scratch than that.  Calls that overlap on the GPU
    share the array and race; order them on one stream."""
    dev = q.device
    _want(q, "q", torch.bfloat16, 3)
    _want(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _want(v_cache, "v_cache", torch.bfloat16, 4, dev)
    _want(page_table, "page_table", torch.int32, 2, dev)
    _want(kv_lens, "kv_lens", torch.int32, 1, dev)
    _want(sinks, "sinks", torch.float32, 1, dev)
    batch, hq, d = q.shape
    num_pages, hkv, page, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(batch, hq, dtype=torch.float32, device=dev)
    with _on(dev):
        _check("sinkattn_decode_static_scratch", load().sinkattn_decode_static_scratch(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(page_table), page_table.shape[1],
            _ptr(kv_lens), _ptr(sinks), float(scale), _ptr(out), _ptr(lse), batch, hq, hkv, d,
            page, num_pages, int(max_kv_len), int(num_splits), _stream(stream)))
    return out, lse


def yarn_table(head_dim=64, base=150000.0, factor=32.0, original_context=4096, beta_fast=32.0,
               beta_slow=1.0):
    """(inv_freq list of head_dim/2 floats, mscale): YaRN-scaled rotary
    frequencies and magnitude factor (host only)."""
    freq = (_c_float * (head_dim // 2))()
    ms = _c_float(0)
    _check("sinkattn_yarn_table",
           load().sinkattn_yarn_table(head_dim, float(base), float(factor), float(original_context),
                                      float(beta_fast), float(beta_slow), freq, ctypes.byref(ms)))
    return list(freq), ms.value


def qkv_prologue(qkv, bias, positions, slot_mapping, inv_freq, mscale, k_cache, v_cache,
                 num_qo_heads, num_kv_heads, *, rope_style=ROPE_HALF, q_out=None, stream=None):
    """QKV bias + rotary encoding of q and k + k/v written into the paged
    cache, one launch.  qkv [T, (Hq + 2 Hkv) * 64] bf16; bias same width or
    None; positions, slot_mapping [T] int32 (slot = page * 16 + offset, < 0:
    no write); inv_freq: sequence of 32 floats (host).  Returns q_out
    [T, Hq, 64] bf16; k_cache / v_cache are written in place."""
    dev = qkv.device
    _want(qkv, "qkv", torch.bfloat16, 2)
    if bias is not None:
        _want(bias, "bias", torch.bfloat16, 1, dev)
    _want(positions, "positions", torch.int32, 1, dev)
    _want(slot_mapping, "slot_mapping", torch.int32, 1, dev)
    _want(k_cache, "k_cache", torch.bfloat16, 4, dev)
    _want(v_cache, "v_cache", torch.bfloat16, 4, dev)
    tokens = qkv.shape[0]
    num_pages, hkv, page, d = k_cache.shape
    if hkv != num_kv_heads or qkv.shape[1] != (num_qo_heads + 2 * num_kv_heads) * d:
        raise ValueError("qkv width / cache heads disagree with the head counts")
    freq = (_c_float * (d // 2))(*[float(x) for x in inv_freq])
    if q_out is None:
        q_out = torch.empty(tokens, num_qo_heads, d, dtype=torch.bfloat16, device=dev)
    with _on(dev):
        _check("sinkattn_qkv_prologue", load().sinkattn_qkv_prologue(
            _ptr(qkv), _ptr(bias), _ptr(positions), _ptr(slot_mapping), freq, float(mscale),
            int(rope_style), _ptr(q_out), _ptr(k_cache), _ptr(v_cache), tokens, num_qo_heads,
            num_kv_heads, d, page, num_pages, _stream(stream)))
    return q_out
