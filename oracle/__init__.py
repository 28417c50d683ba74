"""fp64 CPU oracle for batched speculative-sampling verification.

TEST INFRASTRUCTURE ONLY: tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` use it; the product package never imports it.
The arithmetic lives in ``spec_oracle.c`` (plain C, fp64, libm), which cites
the passages of the tutorial page "5.1 投机解码核心原理" and of the SpecKV
page that each step restates.  This module only compiles that file with gcc
and marshals numpy arrays into it.

Logit arrays are numpy ``float32``, ``float64`` or ``uint16`` (raw bf16 bits).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

GREEDY, SAMPLE, ONEHOT, SIGNALS = 0, 1, 2, 3

# per-request status bits (this oracle's own definitions)
ST_NONFINITE = 1
ST_BAD_TOKEN = 2
ST_BAD_GAMMA = 4
ST_ZERO_RESIDUAL = 8
ST_BAD_TEMPERATURE = 64
ST_BAD_UNIFORM = 128

# planted-mistake ids understood by spec_oracle.c (test-only builds)
PLANTS = {
    "resample_from_p": 1,
    "ratio_inverted": 2,
    "residual_sign": 3,
    "bonus_row": 4,
    "no_temperature": 5,
    "greedy_tie_high": 6,
    "entropy_nats": 7,
    "signal_mean_over_G": 8,
    "draw_nonstrict": 9,
    "onehot_keep_y": 10,
    "no_stop": 11,
    "accept_nonstrict": 12,
    "probe_next_bucket": 13,
    "margin_one_sided": 14,
    "accept_margin_unnormalised": 15,
    "divergence_nats": 16,
    "divergence_kl_swapped": 17,
    "divergence_l1_half": 18,
    "divergence_a_max": 19,
    "divergence_entropy_of_q": 20,
    "gamma_select_no_relu": 21,
    "gamma_select_no_gamma_factor": 22,
    "gamma_select_tie_high": 23,
    "gamma_select_feature_order": 24,
    "filter_topk_strict": 25,
    "filter_topp_exclusive": 26,
    "filter_topp_before_topk": 27,
    "filter_no_temperature": 28,
}

_lock = threading.Lock()
_cache: dict[int, "Oracle"] = {}


def build(plant: int = 0, out_dir: str | None = None) -> str:
    """Compile spec_oracle.c with gcc (-O2, no fast-math) and return the .so path."""
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "libspec_oracle.so" if plant == 0 else f"libspec_oracle_plant{plant}.so"
    out = os.path.join(out_dir, name)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-ffp-contract=off", f"-DORACLE_PLANT={plant}",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 2
    raise TypeError(f"logits must be float32, float64 or uint16 (bf16 bits), got {a.dtype}")


def _ptr(a, ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """Loaded oracle library (one per planted-mistake id)."""

    def __init__(self, path: str):
        self.lib = ctypes.CDLL(path)
        f = self.lib.oracle_run
        P = ctypes.c_void_p
        f.argtypes = [ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      P, P, P, P, P, P, P, P, P, P, P, P, P, P, ctypes.c_int]
        f.restype = ctypes.c_int
        self.lib.oracle_plant_id.restype = ctypes.c_int
        self.plant = self.lib.oracle_plant_id()
        fl = self.lib.oracle_filter
        fl.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, P, P, ctypes.c_int]
        fl.restype = ctypes.c_int
        h = self.lib.oracle_gamma_select
        h.argtypes = [P, P, P, ctypes.c_int, P, P]
        h.restype = ctypes.c_int
        g = self.lib.oracle_divergence
        g.argtypes = [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P, P, P, ctypes.c_int]
        g.restype = ctypes.c_int

    def run(self, mode, target=None, draft=None, draft_tokens=None, gamma=None,
            temperature=None, uniforms=None, *, B=None, G=None, V=None,
            want_signals=False, want_row_signals=False, probe_token=None,
            nthreads=None):
        """Run one mode over a batch; returns a dict of numpy outputs."""
        ref = target if target is not None else draft
        if ref is None:
            raise ValueError("need target or draft logits")
        dt = _dtype_code(ref)
        if target is not None:
            B_, Gp1, V_ = target.shape
            G_ = Gp1 - 1
        else:
            B_, G_, V_ = draft.shape
        B = B_ if B is None else B
        G = G_ if G is None else G
        V = V_ if V is None else V
        c = lambda a, t: None if a is None else np.ascontiguousarray(a, dtype=t)
        target = None if target is None else np.ascontiguousarray(target)
        draft = None if draft is None else np.ascontiguousarray(draft)
        if draft is not None and _dtype_code(draft) != dt:
            raise TypeError("target and draft dtypes differ")
        draft_tokens = c(draft_tokens, np.int32)
        gamma = c(gamma, np.int32)
        temperature = c(temperature, np.float32)
        uniforms = c(uniforms, np.float32)
        probe_token = c(probe_token, np.int32)
        out = {
            "accept_len": np.zeros(B, np.int32),
            "tokens": np.zeros((B, G + 1), np.int32),
            "status": np.zeros(B, np.int32),
            "accept_prob": np.zeros((B, G), np.float64),
            "accept_margin": np.zeros((B, G), np.float64),
            "draw_margin": np.zeros(B, np.float64),
        }
        if want_signals:
            out["signals"] = np.zeros((B, 4), np.float64)
        if want_row_signals:
            out["row_signals"] = np.zeros((B, G, 2), np.float64)
        if probe_token is not None:
            out["probe_distance"] = np.zeros(B, np.float64)
        nthreads = nthreads or os.cpu_count() or 1
        rc = self.lib.oracle_run(
            mode, _ptr(target, ctypes.c_char), _ptr(draft, ctypes.c_char), dt, B, G, V,
            _ptr(draft_tokens, ctypes.c_int32), _ptr(gamma, ctypes.c_int32),
            _ptr(temperature, ctypes.c_float), _ptr(uniforms, ctypes.c_float),
            _ptr(out["accept_len"], ctypes.c_int32), _ptr(out["tokens"], ctypes.c_int32),
            _ptr(out["status"], ctypes.c_int32), _ptr(out.get("signals"), ctypes.c_double),
            _ptr(out.get("row_signals"), ctypes.c_double), _ptr(out["accept_prob"], ctypes.c_double),
            _ptr(out["accept_margin"], ctypes.c_double), _ptr(out["draw_margin"], ctypes.c_double),
            _ptr(probe_token, ctypes.c_int32), _ptr(out.get("probe_distance"), ctypes.c_double),
            int(nthreads))
        if rc != 0:
            raise ValueError("oracle_run rejected its arguments")
        return out

    # convenience wrappers named after the four library calls
    def verify_greedy(self, target, draft_tokens, gamma=None, **kw):
        return self.run(GREEDY, target=target, draft_tokens=draft_tokens, gamma=gamma, **kw)

    def verify_sample(self, target, draft, draft_tokens, gamma, temperature, uniforms, **kw):
        return self.run(SAMPLE, target=target, draft=draft, draft_tokens=draft_tokens, gamma=gamma,
                        temperature=temperature, uniforms=uniforms, **kw)

    def verify_onehot(self, target, draft_tokens, gamma, temperature, uniforms, **kw):
        return self.run(ONEHOT, target=target, draft_tokens=draft_tokens, gamma=gamma,
                        temperature=temperature, uniforms=uniforms, **kw)

    def draft_signals(self, draft, gamma, temperature, **kw):
        kw.setdefault("want_signals", True)
        return self.run(SIGNALS, draft=draft, gamma=gamma, temperature=temperature, **kw)

    def filter_logits(self, logits, top_k=None, top_p=None, temperature=None, *, nthreads=None):
        """Top-k / top-p filtering of rows [n, V] (f32, bf16 bits or f64);
        returns {"logits": [n, V] fp64 filtered, "status": [n], "margin": [n]}."""
        logits = np.ascontiguousarray(logits)
        n, V = logits.shape
        dt = _dtype_code(logits)
        top_k = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32)
        top_p = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32)
        temperature = None if temperature is None else np.ascontiguousarray(temperature, dtype=np.float32)
        out = np.zeros((n, V), np.float64)
        st = np.zeros(n, np.int32)
        mg = np.zeros(n, np.float64)
        nthreads = nthreads or os.cpu_count() or 1
        rc = self.lib.oracle_filter(_ptr(logits, ctypes.c_char), dt, n, V, _ptr(top_k, ctypes.c_int32),
                                    _ptr(top_p, ctypes.c_float), _ptr(temperature, ctypes.c_float),
                                    _ptr(out, ctypes.c_double), _ptr(st, ctypes.c_int32), _ptr(mg, ctypes.c_double),
                                    int(nthreads))
        if rc != 0:
            raise ValueError("oracle_filter rejected its arguments")
        return {"logits": out, "status": st, "margin": mg}

    def gamma_select(self, signals, comp, model):
        """SpecKV gamma selection: signals [B, 4] (mean H, max H, mean c, min c),
        comp [B] or None, model [141] (mu, sd, W1 [16, 6], b1, w2, b2); returns
        {"gamma": [B] int32 (-1: non-finite features), "expected": [B, 4]}."""
        signals = np.ascontiguousarray(signals, dtype=np.float64)
        B = signals.shape[0]
        comp = None if comp is None else np.ascontiguousarray(comp, dtype=np.float64)
        model = np.ascontiguousarray(model, dtype=np.float64)
        if model.shape != (141,):
            raise ValueError("model must hold 141 values")
        gam = np.zeros(B, np.int32)
        exp_ = np.zeros((B, 4), np.float64)
        rc = self.lib.oracle_gamma_select(_ptr(signals, ctypes.c_double), _ptr(comp, ctypes.c_double),
                                          _ptr(model, ctypes.c_double), B, _ptr(gam, ctypes.c_int32),
                                          _ptr(exp_, ctypes.c_double))
        if rc != 0:
            raise ValueError("oracle_gamma_select rejected its arguments")
        return {"gamma": gam, "expected": exp_}

    def divergence_stats(self, target, draft, gamma, temperature, *, nthreads=None):
        """Per-position divergence statistics: target [B, G+1, V] (rows 0..G-1
        are used), draft [B, G, V]; returns {"stats": [B, G, 5] (A, L1,
        KL(p||q), KL(q||p), H(p), bits), "status": [B]}."""
        target = np.ascontiguousarray(target)
        draft = np.ascontiguousarray(draft)
        B, G, V = draft.shape
        if target.shape != (B, G + 1, V):
            raise ValueError("target must be [B, G+1, V] for draft [B, G, V]")
        dt = _dtype_code(target)
        if _dtype_code(draft) != dt:
            raise TypeError("target and draft dtypes differ")
        gamma = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.int32)
        temperature = np.ascontiguousarray(temperature, dtype=np.float32)
        stats = np.zeros((B, G, 5), np.float64)
        status = np.zeros(B, np.int32)
        nthreads = nthreads or os.cpu_count() or 1
        rc = self.lib.oracle_divergence(_ptr(target, ctypes.c_char), _ptr(draft, ctypes.c_char), dt, B, G, V,
                                        _ptr(gamma, ctypes.c_int32), _ptr(temperature, ctypes.c_float),
                                        _ptr(stats, ctypes.c_double), _ptr(status, ctypes.c_int32), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_divergence rejected its arguments")
        return {"stats": stats, "status": status}


def load(plant: int = 0, out_dir: str | None = None) -> Oracle:
    """Build (if needed) and load the oracle; cached per planted-mistake id."""
    with _lock:
        if out_dir is None and plant in _cache:
            return _cache[plant]
        o = Oracle(build(plant, out_dir))
        if out_dir is None:
            _cache[plant] = o
        return o
