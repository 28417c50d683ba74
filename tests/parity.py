"""Helpers shared by the GPU parity tests: inputs to torch, oracle-drawn draft
tokens, and the element-by-element comparison with the oracle.

Comparison rule (fp32 GPU vs fp64 oracle on identical input bytes):
  * status bits (SPEC_ST_GUARDED masked), accept lengths and tokens must be
    equal, except where the oracle itself flags the decision as a near tie:
    an acceptance test with |u - a| < FLAG or a draw whose t lies within
    FLAG * W of a bucket edge.  A flagged acceptance test may go either way;
    a flagged draw may only land in a bucket that the oracle confirms lies
    within FLAG * W of t;
  * accept_prob within REL relative (fp32 result of an fp64-exact formula);
  * signals within REL relative with an absolute floor of 1e-6 (bits / prob).
"""
from __future__ import annotations

import numpy as np

import oracle as O
from speculative_decoding_verification_26_gb300 import workloads as W

FLAG = 1e-5
REL = 1e-5
GUARDED = 16


def oracle_samplers(o):
    def sample_rows(rows, T, u):
        return o.run(O.SAMPLE, target=np.ascontiguousarray(rows)[:, None, :], temperature=T,
                     uniforms=np.ascontiguousarray(u)[:, None], G=0)["tokens"][:, 0]

    def argmax_rows(rows):
        return o.run(O.GREEDY, target=np.ascontiguousarray(rows)[:, None, :], G=0)["tokens"][:, 0]

    return sample_rows, argmax_rows


def make_workload(o, name, round_idx=0, **kw):
    wl = W.make(name, round_idx, **kw)
    W.resolve_draft_tokens(wl, *oracle_samplers(o))
    return wl


def to_dev(a, dev, bf16=False):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    if bf16:
        t = t.view(torch.bfloat16)
    return t


def logits_dev(wl, which, dev):
    a = wl.target if which == "target" else wl.draft
    if a is None:
        return None
    if wl.dtype == W.BF16:
        return to_dev(a.view(np.int16), dev, bf16=True)
    return to_dev(a, dev)


def run_gpu(mode, wl, dev, *, signals=True, accept_prob=True, gamma=True):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    T = logits_dev(wl, "target", dev)
    g = to_dev(wl.gamma, dev) if gamma else None
    if mode == "greedy":
        r = sv.verify_greedy(T, to_dev(wl.draft_tokens, dev), g)
    elif mode == "sample":
        r = sv.verify_sample(T, logits_dev(wl, "draft", dev), to_dev(wl.draft_tokens, dev), g,
                             to_dev(wl.temperature, dev), to_dev(wl.uniforms, dev), signals=signals,
                             accept_prob=accept_prob)
    elif mode == "onehot":
        r = sv.verify_onehot(T, to_dev(wl.draft_tokens, dev), g, to_dev(wl.temperature, dev),
                             to_dev(wl.uniforms, dev), accept_prob=accept_prob)
    else:
        raise ValueError(mode)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in r.items()}


def run_oracle(o, mode, wl, *, signals=True, gamma=True, probe=None):
    g = wl.gamma if gamma else None
    if mode == "greedy":
        return o.verify_greedy(wl.target, wl.draft_tokens, g, probe_token=probe)
    if mode == "sample":
        return o.verify_sample(wl.target, wl.draft, wl.draft_tokens, g, wl.temperature, wl.uniforms,
                               want_signals=signals, probe_token=probe)
    return o.verify_onehot(wl.target, wl.draft_tokens, g, wl.temperature, wl.uniforms, probe_token=probe)


class Tally:
    def __init__(self):
        self.decisions = 0
        self.flagged = 0
        self.disagree = 0
        self.notes = []

    def __repr__(self):
        return (f"decisions={self.decisions} flagged={self.flagged} disagreements={self.disagree}"
                + (f" {self.notes[:3]}" if self.notes else ""))


def compare(o, mode, wl, g, ref, tally: Tally, *, check_signals=True, gamma=True):
    """Compare GPU outputs g with oracle outputs ref; raises AssertionError on
    any difference the comparison rule does not allow."""
    B, G = wl.B, wl.G
    st_g = g["status"] & ~GUARDED
    np.testing.assert_array_equal(st_g, ref["status"], err_msg="status")
    alt_probe = np.full(B, -1, np.int32)
    need_probe = []
    for b in range(B):
        ko, kg = int(ref["accept_len"][b]), int(g["accept_len"][b])
        if ref["status"][b] & ~8:
            assert kg == 0 and np.all(g["tokens"][b] == -1), f"void request {b} committed tokens"
            continue
        n_tests = ko + (1 if ko < (wl.gamma[b] if gamma else G) else 0)
        tally.decisions += n_tests + 1
        if mode != "greedy":
            am = ref["accept_margin"][b]
            tally.flagged += int(np.sum(am[:n_tests] < FLAG)) + int(ref["draw_margin"][b] < FLAG)
        if ko != kg:
            j = min(ko, kg)
            if mode != "greedy" and ref["accept_margin"][b][j] < FLAG:
                tally.disagree += 1
                tally.notes.append(("accept", b, j, float(ref["accept_margin"][b][j])))
                continue
            raise AssertionError(f"request {b}: accept_len gpu {kg} != oracle {ko}")
        np.testing.assert_array_equal(g["tokens"][b, :ko], ref["tokens"][b, :ko])
        assert np.all(g["tokens"][b, ko + 1:] == -1)
        if g["tokens"][b, ko] != ref["tokens"][b, ko]:
            if mode == "greedy" or not (ref["draw_margin"][b] < FLAG):
                raise AssertionError(f"request {b}: token gpu {g['tokens'][b, ko]} != oracle "
                                     f"{ref['tokens'][b, ko]} (draw margin {ref['draw_margin'][b]:.3g})")
            alt_probe[b] = g["tokens"][b, ko]
            need_probe.append(b)
        if mode != "greedy" and "accept_prob" in g:
            a_o = ref["accept_prob"][b, :n_tests]
            a_g = g["accept_prob"][b, :n_tests].astype(np.float64)
            np.testing.assert_allclose(a_g, a_o, rtol=REL, atol=1e-30, err_msg=f"accept_prob b={b}")
            assert np.all(np.isnan(g["accept_prob"][b, n_tests:])), f"accept_prob after k, b={b}"
    if need_probe:
        pr = run_oracle(o, mode, wl, signals=False, gamma=gamma, probe=alt_probe)
        for b in need_probe:
            d = pr["probe_distance"][b]
            assert d < FLAG, f"request {b}: gpu token's bucket is {d:.3g} W from t"
            tally.disagree += 1
            tally.notes.append(("draw", b, float(ref["draw_margin"][b])))
    if check_signals and "signals" in g and "signals" in ref:
        so, sg = ref["signals"], g["signals"].astype(np.float64)
        both_nan = np.isnan(so) & np.isnan(sg)
        ok = both_nan | (np.abs(sg - so) <= REL * np.abs(so) + 1e-6)
        assert ok.all(), f"signals differ: {np.argwhere(~ok)[:5]}, {sg[~ok][:5]} vs {so[~ok][:5]}"
    return tally
