"""Seeded synthetic workloads for speculative-sampling verification.

This module only makes random inputs; it holds none of the verification
arithmetic (no softmax, no acceptance test, no draw).  The same generator
feeds the GPU library, the fp64 oracle and the benchmark.

The public suites the pages measure on (GSM8K, SWE-Bench, LiveCodeBench,
MATH500, ...) and the models' weights are not available, so the logits are
synthetic stand-ins with the pages' shapes: draft lengths gamma 2-8 with K = 7
draft positions (DLite page), concurrency 1-64 and beyond, Qwen-family
(V = 151936) and Llama-family (V = 128256) vocabularies, temperatures 0.6-1.0.

Recipe (all numpy PCG64, platform independent; every logit row's normals come
from its own child seed, SeedSequence.spawn, and are drawn on a thread pool, so
the values do not depend on the number of threads):
  * Zipf-like per-token bias shared by every row of a workload:
    b[v] = -1.1 * ln(1 + pi(v)) with pi a seeded random permutation of 0..V-1,
    so frequent tokens are scattered over the vocabulary;
  * target logits = bf16_rne(N(0, sigma_t^2) + b + shift)   (fp32 configs: no
    rounding; shift = 0 unless a test asks for an offset, which softmax
    ignores but fp32 exponent arithmetic does not);
  * draft logits  = bf16_rne(float(target) + N(0, sigma_d^2));
  * uniforms [B, G+1] float32 in [0, 1): u = (bits >> 40) * 2^-24;
  * draft tokens come from a stand-in drafter (see ``resolve_draft_tokens``):
      - "sample_q":      y_i ~ q_i, the draft model's own sampling law
                         softmax(x / T), drawn by the Gumbel-max trick:
                         y = argmax_v (x_v / T + g_v), g_v = -ln(-ln U_v) with
                         U_v uniform from the row's own seed (an exact draw;
                         only noise and an argmax, in fp64);
      - "argmax_replace": y_i = argmax of target row i, replaced with
                         probability 0.3 by a uniform random token;
      - "noisy_argmax":  y_i = argmax of (target row i + N(0, 2^2));
    the two argmax kinds take a caller-supplied argmax (lowest index on
    ties), so that this module computes nothing a verification call does.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F32, BF16 = "f32", "bf16"

# Workload shapes.  "m" is the B=64, gamma=7, V=151936 bf16 full-q + signals
# point on which throughput is quoted; c1..c5 are the parity cases.
CONFIGS = {
    "c1": dict(B=4, G=4, V=1024, dtype=F32, sigma_t=2.0, zipf=False, sigma_d=1.0, T=1.0,
               draft="sample_q", modes=("greedy", "sample"), signals=True),
    "c2": dict(B=64, G=7, V=151936, dtype=BF16, sigma_t=3.0, zipf=True, T=1.0,
               draft="argmax_replace", replace_p=0.3, modes=("greedy",), signals=False),
    "c3": dict(B=32, G=4, V=128256, dtype=BF16, sigma_t=3.0, zipf=True, sigma_d=1.5, T=0.7,
               draft="sample_q", modes=("sample",), signals=True),
    "c4": dict(B=64, G=8, V=151936, dtype=BF16, sigma_t=3.0, zipf=True, T=1.0,
               draft="noisy_argmax", noise=2.0, modes=("onehot",), signals=False),
    "c5": dict(B=256, G=8, V=151936, dtype=BF16, sigma_t=3.0, zipf=True, sigma_d=1.0, T=0.6,
               gammas=(2, 4, 6, 8), draft="sample_q", modes=("sample",), signals=True),
    "m": dict(B=64, G=7, V=151936, dtype=BF16, sigma_t=3.0, zipf=True, sigma_d=1.5, T=0.7,
              draft="sample_q", modes=("sample",), signals=True),
}
_CONFIG_ID = {name: i + 1 for i, name in enumerate(CONFIGS)}


def _rows_parallel(n: int, fn) -> None:
    """fn(lo, hi) over row blocks of [0, n) on a thread pool (numpy releases
    the GIL in its loops; every row is computed the same way whatever the
    block)."""
    nt = max(1, min(32, os.cpu_count() or 1, n))
    step = (n + nt - 1) // nt
    if nt == 1:
        fn(0, n)
        return
    with ThreadPoolExecutor(nt) as ex:
        list(ex.map(lambda lo: fn(lo, min(n, lo + step)), range(0, n, step)))


def bf16_rne_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    src = x.reshape(-1, x.shape[-1]) if x.ndim > 1 else x.reshape(1, -1)
    out = np.empty(src.shape, np.uint16)

    def blk(lo, hi):
        b = src[lo:hi].view(np.uint32)
        r = (b >> np.uint32(16)) & np.uint32(1)
        r += np.uint32(0x7FFF)
        r += b
        r >>= np.uint32(16)
        out[lo:hi] = r

    _rows_parallel(src.shape[0], blk)
    return out.reshape(x.shape)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniforms01(rng: np.random.Generator, shape) -> np.ndarray:
    """float32 uniforms in [0, 1) with 24 random bits: (bits >> 40) * 2^-24."""
    bits = rng.integers(0, 2**64, size=shape, dtype=np.uint64, endpoint=False)
    return ((bits >> np.uint64(40)).astype(np.float64) * 2.0**-24).astype(np.float32)


def zipf_bias(V: int, rng: np.random.Generator, s: float = 1.1) -> np.ndarray:
    perm = rng.permutation(V)
    return (-s * np.log1p(perm.astype(np.float64))).astype(np.float32)


def normal_rows(ss: np.random.SeedSequence, shape, scale: float) -> np.ndarray:
    """float32 N(0, scale^2) of `shape`; row j (over the last axis) is drawn
    from child seed j of `ss`, rows in parallel (numpy releases the GIL)."""
    V = shape[-1]
    n = int(np.prod(shape[:-1]))
    out = np.empty((n, V), np.float32)
    kids = ss.spawn(n)

    def fill(lo, hi):
        for j in range(lo, hi):
            np.random.default_rng(kids[j]).standard_normal(V, dtype=np.float32, out=out[j])
            out[j] *= np.float32(scale)

    _rows_parallel(n, fill)
    return out.reshape(shape)


@dataclass
class Workload:
    name: str
    B: int
    G: int
    V: int
    dtype: str                     # "bf16" (uint16 bit arrays) or "f32"
    target: np.ndarray             # [B, G+1, V]
    draft: np.ndarray | None       # [B, G, V] or None (greedy / one-hot)
    gamma: np.ndarray              # [B] int32
    temperature: np.ndarray        # [B] float32
    uniforms: np.ndarray           # [B, G+1] float32
    draft_kind: str
    draft_aux: dict = field(default_factory=dict)
    draft_tokens: np.ndarray | None = None   # [B, G] int32, after resolve_draft_tokens

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


def make(name: str, round_idx: int = 0, *, B: int | None = None, G: int | None = None,
         V: int | None = None, overrides: dict | None = None) -> Workload:
    """Build the seeded workload `name` for one verification round."""
    cfg = dict(CONFIGS[name])
    if overrides:
        cfg.update(overrides)
    B = B or cfg["B"]
    G = cfg["G"] if G is None else G
    V = V or cfg["V"]
    cid = _CONFIG_ID.get(name, 99)
    ss = np.random.SeedSequence([1000 * cid + round_idx, 7])
    k_bias, k_t, k_d, k_u, k_y, k_g = ss.spawn(6)
    # the Zipf permutation is fixed per config (shared by all rounds)
    bias = zipf_bias(V, np.random.default_rng([cid, 11])) if cfg.get("zipf") else np.float32(0)
    t32 = normal_rows(k_t, (B, G + 1, V), cfg["sigma_t"])
    t32 += bias
    if cfg.get("shift"):
        t32 += np.float32(cfg["shift"])
    if cfg["dtype"] == BF16:
        target = bf16_rne_bits(t32)
        tf = bf16_bits_to_f32(target)
    else:
        target = t32
        tf = t32
    draft = None
    if "sigma_d" in cfg and G > 0:
        d32 = normal_rows(k_d, (B, G, V), cfg["sigma_d"])
        d32 += tf[:, :G, :]
        draft = bf16_rne_bits(d32) if cfg["dtype"] == BF16 else d32
    if "gammas" in cfg:
        gamma = np.random.default_rng(k_g).choice(np.asarray(cfg["gammas"], np.int32), size=B)
    else:
        gamma = np.full(B, G, np.int32)
    temperature = np.full(B, cfg.get("T", 1.0), np.float32)
    uniforms = uniforms01(np.random.default_rng(k_u), (B, G + 1))
    ry = np.random.default_rng(k_y)
    aux = {}
    kind = cfg["draft"]
    if kind == "sample_q":
        aux["gumbel_key"] = [1000 * cid + round_idx, 17]
    elif kind == "argmax_replace":
        aux["replace"] = ry.random((B, G)) < cfg.get("replace_p", 0.3)
        aux["random_tokens"] = ry.integers(0, V, size=(B, G), dtype=np.int32)
    elif kind == "noisy_argmax":
        noise = normal_rows(np.random.SeedSequence([1000 * cid + round_idx, 13]), (B, G, V), cfg.get("noise", 2.0))
        noise += tf[:, :G, :]
        aux["proxy"] = noise                       # float32 [B, G, V]
    return Workload(name, B, G, V, cfg["dtype"], target, draft, gamma.astype(np.int32),
                    temperature, uniforms, kind, aux)


def gumbel_max_tokens(key, rows: np.ndarray, temps: np.ndarray) -> np.ndarray:
    """One draw per row from softmax(row / T) by the Gumbel-max trick:
    argmax_v (x_v / T - ln(-ln U_v)); row j's uniforms come from child seed j
    of SeedSequence(key).  rows: [n, V] float32, float64 or bf16 bits."""
    n, V = rows.shape
    kids = np.random.SeedSequence(key).spawn(n)
    out = np.empty(n, np.int32)

    def blk(lo, hi):
        with np.errstate(divide="ignore"):
            for j in range(lo, hi):
                x = bf16_bits_to_f32(rows[j]) if rows.dtype == np.uint16 else rows[j]
                u = np.random.default_rng(kids[j]).random(V)
                out[j] = int(np.argmax(x.astype(np.float64) / np.float64(temps[j]) - np.log(-np.log(u))))

    _rows_parallel(n, blk)
    return out


def resolve_draft_tokens(wl: Workload, argmax_rows=None) -> np.ndarray:
    """Fill ``wl.draft_tokens`` from the workload's stand-in drafter (drawn
    from the current draft rows, so a test that replaces them redraws).

    argmax_rows(logits [n, V]) -> tokens [n] (lowest index on ties) serves
    the two argmax drafters."""
    B, G, V = wl.B, wl.G, wl.V
    if G == 0:
        wl.draft_tokens = np.zeros((B, 0), np.int32)
        return wl.draft_tokens
    if wl.draft_kind == "sample_q":
        y = gumbel_max_tokens(wl.draft_aux["gumbel_key"], wl.draft.reshape(B * G, V), np.repeat(wl.temperature, G))
    elif wl.draft_kind == "argmax_replace":
        rows = wl.target[:, :G, :].reshape(B * G, V)
        y = np.asarray(argmax_rows(rows), np.int32)
        rep = wl.draft_aux["replace"].reshape(-1)
        y = np.where(rep, wl.draft_aux["random_tokens"].reshape(-1), y).astype(np.int32)
    elif wl.draft_kind == "noisy_argmax":
        y = np.asarray(argmax_rows(wl.draft_aux["proxy"].reshape(B * G, V)), np.int32)
    else:
        raise ValueError(wl.draft_kind)
    y = y.reshape(B, G)
    # positions beyond a request's gamma are padding and never read
    pad = np.arange(G)[None, :] >= wl.gamma[:, None]
    y[pad] = 0
    wl.draft_tokens = np.ascontiguousarray(y, np.int32)
    return wl.draft_tokens
