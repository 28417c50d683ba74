"""ctypes binding of libspec_verify.so (argument marshalling only).

Every step of the verification runs in the library's CUDA kernels; this module
checks tensor shapes/dtypes, allocates outputs and the workspace with torch on
the caller's device, passes raw device pointers and the current stream, and
raises on a non-zero return code.  There is no CPU fallback: if the library
cannot be loaded the call fails.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspec_verify.so")

F32, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_WORKSPACE, ERR_CUDA, ERR_UNSUPPORTED = 0, 1, 2, 3, 4
ST_NONFINITE, ST_BAD_TOKEN, ST_BAD_GAMMA, ST_ZERO_RESIDUAL = 1, 2, 4, 8
ST_GUARDED, ST_TIMEOUT, ST_BAD_TEMPERATURE, ST_BAD_UNIFORM = 16, 32, 64, 128

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (built by ``build.build()``) and set signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FileNotFoundError(
                f"{p} is missing: build it with `python -m speculative_decoding_verification_26_gb300.build`")
        L = ctypes.CDLL(p)
        P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L.spec_workspace_bytes.argtypes = [I, I, I]
        L.spec_workspace_bytes.restype = SZ
        L.spec_status_string.argtypes = [I]
        L.spec_status_string.restype = ctypes.c_char_p
        L.spec_request_status_string.argtypes = [I]
        L.spec_request_status_string.restype = ctypes.c_char_p
        L.spec_launch_count.argtypes = []
        L.spec_launch_count.restype = ctypes.c_uint64
        L.spec_profile_next_call.argtypes = [P, P]
        L.spec_profile_next_call.restype = I
        L.spec_set_wait_limit.argtypes = [ctypes.c_longlong]
        L.spec_set_wait_limit.restype = I
        L.spec_verify_greedy.argtypes = [P, I, I, I, I, P, P, P, P, P, P, SZ, P]
        L.spec_verify_greedy.restype = I
        L.spec_verify_sample.argtypes = [P, P, I, I, I, I, P, P, P, P, P, P, P, P, P, P, SZ, P]
        L.spec_verify_sample.restype = I
        L.spec_verify_onehot.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P, P, P, SZ, P]
        L.spec_verify_onehot.restype = I
        L.spec_draft_signals.argtypes = [P, I, I, I, I, P, P, P, P, P, P, SZ, P]
        L.spec_divergence_stats.argtypes = [P, P, I, I, I, I, P, P, P, P, P]
        L.spec_divergence_stats.restype = I
        L.spec_gamma_select.argtypes = [P, P, P, I, P, P, P]
        L.spec_filter_top_k_top_p.argtypes = [P, I, I, I, P, P, P, P, P]
        L.spec_filter_top_k_top_p.restype = I
        L.spec_gamma_select.restype = I
        L.spec_draft_signals.restype = I
        if path is None:
            _lib = L
        return L


def status_string(code: int) -> str:
    return lib().spec_status_string(int(code)).decode()


def request_status_string(bit: int) -> str:
    return lib().spec_request_status_string(int(bit)).decode()


def workspace_bytes(B: int, G: int, V: int) -> int:
    return int(lib().spec_workspace_bytes(int(B), int(G), int(V)))


def launch_count() -> int:
    return int(lib().spec_launch_count())


def set_wait_limit(cycles: int) -> None:
    """Testing aid: internal waits of later calls give up after `cycles` SM
    cycles (<= 0 restores the default); see spec_set_wait_limit."""
    rc = lib().spec_set_wait_limit(int(cycles))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_set_wait_limit")


def profile_next_call(begin, end) -> None:
    """Record torch.cuda.Event `begin`/`end` around the verify kernel of
    the next call made by this thread (see spec_profile_next_call)."""
    rc = lib().spec_profile_next_call(ctypes.c_void_p(begin.cuda_event), ctypes.c_void_p(end.cuda_event))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_profile_next_call")


# ----------------------------------------------------------------------------
# torch-facing wrappers

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _check(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


_ws_cache: dict = {}


def workspace(B, G, V, device):
    """A cached workspace tensor for these sizes on `device` (reused by calls
    on the same stream; calls sharing it must not overlap on the device)."""
    torch = _torch()
    n = workspace_bytes(B, G, V)
    if n == 0:
        raise ValueError("sizes outside the library limits")
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < n:
        ws = torch.empty(n, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _out(o, key, make):
    t = o.get(key)
    return make() if t is None else t


def _stream(device):
    return ctypes.c_void_p(_torch().cuda.current_stream(device).cuda_stream)


def verify_greedy(target, draft_tokens, gamma=None, *, ws=None, out=None):
    """Greedy verification.  target [B, G+1, V] bf16/f32; draft_tokens [B, G] int32."""
    torch = _torch()
    B, Gp1, V = target.shape
    G = Gp1 - 1
    dev = target.device
    _check(target, "target", device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(gamma, "gamma", torch.int32, (B,), dev)
    o = out or {}
    acc = _out(o, "accept_len", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    tok = _out(o, "tokens", lambda: torch.empty(B, G + 1, dtype=torch.int32, device=dev))
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    ws = ws if ws is not None else workspace(B, G, V, dev)
    rc = lib().spec_verify_greedy(_ptr(target), _dtype_code(target), B, G, V, _ptr(draft_tokens), _ptr(gamma),
                                  _ptr(acc), _ptr(tok), _ptr(st), _ptr(ws), ws.numel(), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify_greedy")
    return {"accept_len": acc, "tokens": tok, "status": st}


def verify_sample(target, draft, draft_tokens, gamma, temperature, uniforms, *, signals=True,
                  accept_prob=False, ws=None, out=None):
    """Full-q stochastic verification (+ optional draft signals / accept_prob)."""
    torch = _torch()
    B, Gp1, V = target.shape
    G = Gp1 - 1
    dev = target.device
    _check(target, "target", device=dev)
    _check(draft, "draft", target.dtype, (B, G, V), dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(gamma, "gamma", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 1), dev)
    o = out or {}
    acc = _out(o, "accept_len", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    tok = _out(o, "tokens", lambda: torch.empty(B, G + 1, dtype=torch.int32, device=dev))
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    sig = (_out(o, "signals", lambda: torch.empty(B, 4, dtype=torch.float32, device=dev))) if signals else None
    ap = (_out(o, "accept_prob", lambda: torch.empty(B, G, dtype=torch.float32, device=dev))) if accept_prob else None
    ws = ws if ws is not None else workspace(B, G, V, dev)
    rc = lib().spec_verify_sample(_ptr(target), _ptr(draft), _dtype_code(target), B, G, V, _ptr(draft_tokens),
                                  _ptr(gamma), _ptr(temperature), _ptr(uniforms), _ptr(acc), _ptr(tok), _ptr(sig),
                                  _ptr(ap), _ptr(st), _ptr(ws), ws.numel(), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify_sample")
    r = {"accept_len": acc, "tokens": tok, "status": st}
    if sig is not None:
        r["signals"] = sig
    if ap is not None:
        r["accept_prob"] = ap
    return r


def verify_onehot(target, draft_tokens, gamma, temperature, uniforms, *, accept_prob=False, ws=None, out=None):
    """One-hot-q stochastic verification."""
    torch = _torch()
    B, Gp1, V = target.shape
    G = Gp1 - 1
    dev = target.device
    _check(target, "target", device=dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(gamma, "gamma", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 1), dev)
    o = out or {}
    acc = _out(o, "accept_len", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    tok = _out(o, "tokens", lambda: torch.empty(B, G + 1, dtype=torch.int32, device=dev))
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    ap = (_out(o, "accept_prob", lambda: torch.empty(B, G, dtype=torch.float32, device=dev))) if accept_prob else None
    ws = ws if ws is not None else workspace(B, G, V, dev)
    rc = lib().spec_verify_onehot(_ptr(target), _dtype_code(target), B, G, V, _ptr(draft_tokens), _ptr(gamma),
                                  _ptr(temperature), _ptr(uniforms), _ptr(acc), _ptr(tok), _ptr(ap), _ptr(st),
                                  _ptr(ws), ws.numel(), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify_onehot")
    r = {"accept_len": acc, "tokens": tok, "status": st}
    if ap is not None:
        r["accept_prob"] = ap
    return r


def divergence_stats(target, draft, gamma, temperature, *, out=None):
    """Per-position divergence statistics.  target [B, G+1, V], draft [B, G, V];
    returns {"stats": [B, G, 5] (A, L1, KL(p||q), KL(q||p), H(p), bits),
    "status": [B]}."""
    torch = _torch()
    B, G, V = draft.shape
    dev = draft.device
    _check(target, "target", shape=(B, G + 1, V), device=dev)
    _check(draft, "draft", device=dev)
    if target.dtype != draft.dtype:
        raise TypeError("target and draft dtypes differ")
    _check(gamma, "gamma", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    o = out or {}
    stats = _out(o, "stats", lambda: torch.empty(B, G, 5, dtype=torch.float32, device=dev))
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    rc = lib().spec_divergence_stats(_ptr(target), _ptr(draft), _dtype_code(draft), B, G, V, _ptr(gamma),
                                     _ptr(temperature), _ptr(stats), _ptr(st), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_divergence_stats")
    return {"stats": stats, "status": st}


def filter_top_k_top_p(logits, top_k=None, top_p=None, temperature=None, *, status=None):
    """Top-k / top-p filtering of the rows of `logits` ([..., V], contiguous,
    fp32 or bf16) in place; top_k [n] int32, top_p [n] fp32, temperature [n]
    fp32, each optional (n = rows).  Returns the per-row status tensor."""
    torch = _torch()
    V = logits.shape[-1]
    n = logits.numel() // V
    dev = logits.device
    _check(logits, "logits", device=dev)
    _check(top_k, "top_k", torch.int32, (n,), dev)
    _check(top_p, "top_p", torch.float32, (n,), dev)
    _check(temperature, "temperature", torch.float32, (n,), dev)
    st = status if status is not None else torch.empty(n, dtype=torch.int32, device=dev)
    rc = lib().spec_filter_top_k_top_p(_ptr(logits), _dtype_code(logits), n, V, _ptr(top_k), _ptr(top_p),
                                       _ptr(temperature), _ptr(st), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_filter_top_k_top_p")
    return st


GAMMA_MODEL_FLOATS = 141


def gamma_select(signals, model, comp=None, *, out=None):
    """SpecKV gamma selection.  signals [B, 4] fp32 (mean H, max H, mean c,
    min c), model [141] fp32, comp [B] fp32 or None; returns {"gamma": [B]
    int32 (2, 4, 6, 8; -1 for non-finite features), "expected": [B, 4]}."""
    torch = _torch()
    B = signals.shape[0]
    dev = signals.device
    _check(signals, "signals", torch.float32, (B, 4), dev)
    _check(model, "model", torch.float32, (GAMMA_MODEL_FLOATS,), dev)
    _check(comp, "comp", torch.float32, (B,), dev)
    o = out or {}
    g = _out(o, "gamma", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    e = _out(o, "expected", lambda: torch.empty(B, 4, dtype=torch.float32, device=dev))
    rc = lib().spec_gamma_select(_ptr(signals), _ptr(comp), _ptr(model), B, _ptr(g), _ptr(e), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_gamma_select")
    return {"gamma": g, "expected": e}


def draft_signals(draft, gamma, temperature, *, row_signals=False, ws=None, out=None):
    """SpecKV draft signals only.  draft [B, G, V]."""
    torch = _torch()
    B, G, V = draft.shape
    dev = draft.device
    _check(draft, "draft", device=dev)
    _check(gamma, "gamma", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    o = out or {}
    sig = _out(o, "signals", lambda: torch.empty(B, 4, dtype=torch.float32, device=dev))
    rs = (_out(o, "row_signals", lambda: torch.empty(B, G, 2, dtype=torch.float32, device=dev))) if row_signals else None
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    ws = ws if ws is not None else workspace(B, G, V, dev)
    rc = lib().spec_draft_signals(_ptr(draft), _dtype_code(draft), B, G, V, _ptr(gamma), _ptr(temperature),
                                  _ptr(sig), _ptr(rs), _ptr(st), _ptr(ws), ws.numel(), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_draft_signals")
    r = {"signals": sig, "status": st}
    if rs is not None:
        r["row_signals"] = rs
    return r


STATIC_WORKSPACE_BYTES = 8 << 20


def verify_sample_static(target, draft, draft_tokens, gamma, temperature, uniforms, *, signals=True,
                         accept_prob=False, out=None):
    """verify_sample on the library's own static scratch (spec_verify_sample_static).

    The C call allocates nothing; this wrapper allocates outputs only when
    `out` does not supply them.  Calls on one device must not overlap."""
    torch = _torch()
    L = lib()
    f = L.spec_verify_sample_static
    if f.argtypes is None:
        P, I = ctypes.c_void_p, ctypes.c_int
        f.argtypes = [P, P, I, I, I, I, P, P, P, P, P, P, P, P, P, P]
        f.restype = I
    B, Gp1, V = target.shape
    G = Gp1 - 1
    dev = target.device
    _check(target, "target", device=dev)
    _check(draft, "draft", target.dtype, (B, G, V), dev)
    _check(draft_tokens, "draft_tokens", torch.int32, (B, G), dev)
    _check(gamma, "gamma", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(uniforms, "uniforms", torch.float32, (B, G + 1), dev)
    o = out or {}
    acc = _out(o, "accept_len", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    tok = _out(o, "tokens", lambda: torch.empty(B, G + 1, dtype=torch.int32, device=dev))
    st = _out(o, "status", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    sig = (_out(o, "signals", lambda: torch.empty(B, 4, dtype=torch.float32, device=dev))) if signals else None
    ap = (_out(o, "accept_prob", lambda: torch.empty(B, G, dtype=torch.float32, device=dev))) if accept_prob else None
    rc = f(_ptr(target), _ptr(draft), _dtype_code(target), B, G, V, _ptr(draft_tokens), _ptr(gamma),
           _ptr(temperature), _ptr(uniforms), _ptr(acc), _ptr(tok), _ptr(sig), _ptr(ap), _ptr(st), _stream(dev))
    if rc != OK:
        raise SpecVerifyError(rc, "spec_verify_sample_static")
    r = {"accept_len": acc, "tokens": tok, "status": st}
    if sig is not None:
        r["signals"] = sig
    if ap is not None:
        r["accept_prob"] = ap
    return r
