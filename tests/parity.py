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
  * signals within REL relative; entropies also within H_ATOL = 1e-6 bits
    absolute.  A near-one-hot draft row has s = 1 + r with r small, and the
    fp32 s carries a relative rounding error of ~1e-7 however small H is: an
    absolute error of ~1.4e-7 bits in log2 s, which is 1e-5 of H only once
    H > 0.014 bits.  Confidences get no absolute term (1/s keeps its
    relative accuracy).
The disagreement budget: decisions that differ from the oracle (each one a
flagged near tie, by the rule above) must stay under BUDGET of all decisions
(acceptance tests plus final draws) over a large sample of rounds.
"""
from __future__ import annotations

import numpy as np

import oracle as O
from speculative_decoding_verification_26_gb300 import workloads as W

FLAG = 1e-5
REL = 1e-5
SIG_ATOL = 1e-12
H_ATOL = 1e-6
BUDGET = 1e-4
GUARDED = 16


def oracle_argmax(o):
    """argmax_rows for the argmax drafters: the oracle's greedy argmax."""
    def argmax_rows(rows):
        return o.run(O.GREEDY, target=np.ascontiguousarray(rows)[:, None, :], G=0)["tokens"][:, 0]
    return argmax_rows


def make_workload(o, name, round_idx=0, **kw):
    wl = W.make(name, round_idx, **kw)
    W.resolve_draft_tokens(wl, oracle_argmax(o))
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


def run_gpu(mode, wl, dev, *, signals=True, accept_prob=True, gamma=True, logits=None, ws=None):
    """One library call through the C ABI on wl's inputs; `logits` may hold
    the (target, draft) device tensors already uploaded."""
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    if logits is None:
        logits = (logits_dev(wl, "target", dev), logits_dev(wl, "draft", dev) if mode != "greedy" else None)
    T, D = logits
    g = to_dev(wl.gamma, dev) if gamma else None
    if mode == "greedy":
        r = sv.verify_greedy(T, to_dev(wl.draft_tokens, dev), g, ws=ws)
    elif mode == "sample":
        r = sv.verify_sample(T, D, to_dev(wl.draft_tokens, dev), g,
                             to_dev(wl.temperature, dev), to_dev(wl.uniforms, dev), signals=signals,
                             accept_prob=accept_prob, ws=ws)
    elif mode == "onehot":
        r = sv.verify_onehot(T, to_dev(wl.draft_tokens, dev), g, to_dev(wl.temperature, dev),
                             to_dev(wl.uniforms, dev), accept_prob=accept_prob, ws=ws)
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
        self.guarded = 0           # draws taken again in extended precision (GPU status bit)
        self.notes = []

    def __repr__(self):
        n = max(self.decisions, 1)
        return (f"decisions={self.decisions} flagged={self.flagged} ({self.flagged / n:.3%}) "
                f"disagreements={self.disagree} ({self.disagree / n:.4%}, budget {BUDGET:.2%}) "
                f"guarded={self.guarded}"
                + (f" {self.notes[:3]}" if self.notes else ""))

    def within_budget(self):
        return self.disagree <= BUDGET * self.decisions


def compare(o, mode, wl, g, ref, tally: Tally, *, check_signals=True, gamma=True):
    """Compare GPU outputs g with oracle outputs ref; raises AssertionError on
    any difference the comparison rule does not allow."""
    B, G = wl.B, wl.G
    tally.guarded += int(np.count_nonzero(g["status"] & GUARDED))
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
        compare_signals(g["signals"], ref["signals"])
    return tally


def compare_signals(sg, so, what="signals"):
    """fp32 signals against fp64 ones (NaN where the oracle has NaN): REL
    relative, plus H_ATOL bits on the entropy columns.  signals [B, 4] hold
    (mean H, max H, mean c, min c); row_signals [B, G, 2] hold (H_i, c_i)."""
    sg = np.asarray(sg, np.float64)
    so = np.asarray(so, np.float64)
    atol = np.full(so.shape[-1], SIG_ATOL)
    atol[:2 if so.shape[-1] == 4 else 1] = H_ATOL
    both_nan = np.isnan(so) & np.isnan(sg)
    ok = both_nan | (np.abs(sg - so) <= REL * np.abs(so) + atol)
    assert ok.all(), f"{what} differ: {np.argwhere(~ok)[:5]}, {sg[~ok][:5]} vs {so[~ok][:5]}"


# ----------------------------------------------------------------------------
# large samples: many rounds of fresh draft tokens and uniforms per logit set

def draft_token_rounds(wl, rounds, seed):
    """[rounds, B, G] draft tokens from wl's stand-in drafter, fresh per round.

    sample_q: y ~ q_i, the draft row's softmax at the request's T in fp64
    (numpy), picked as the smallest index whose cumulative weight exceeds
    u * total with an independent uniform stream (input generation only);
    argmax_replace: the target argmax (lowest index), replaced with
    probability 0.3 by a uniform token, redrawn per round; noisy_argmax: the
    workload's own tokens every round (only the uniforms change)."""
    B, G, V = wl.B, wl.G, wl.V
    rng = np.random.default_rng(seed)
    out = np.zeros((rounds, B, G), np.int32)
    if G == 0:
        return out
    if wl.draft_kind == "sample_q":
        rows = wl.draft.reshape(B * G, V)
        u = rng.random((B * G, rounds))
        for j in range(B * G):
            x = (W.bf16_bits_to_f32(rows[j]) if wl.dtype == W.BF16 else rows[j]).astype(np.float64)
            w = np.exp((x - x.max()) / np.float64(wl.temperature[j // G]))
            c = np.cumsum(w)
            out[:, j // G, j % G] = np.minimum(np.searchsorted(c, u[j] * c[-1], side="right"), V - 1)
    elif wl.draft_kind == "argmax_replace":
        t = wl.target[:, :G, :]
        am = np.argmax(W.bf16_bits_to_f32(t) if wl.dtype == W.BF16 else t, axis=2).astype(np.int32)
        for r in range(rounds):
            rep = rng.random((B, G)) < 0.3
            out[r] = np.where(rep, rng.integers(0, V, (B, G), dtype=np.int32), am)
    else:
        W.resolve_draft_tokens(wl, lambda rows: np.argmax(rows, axis=1))
        out[:] = wl.draft_tokens[None]
    pad = np.arange(G)[None, :] >= wl.gamma[:, None]
    out[:, pad] = 0
    return out


def large_sample(o, dev, name, mode, n_sets, rounds, *, signals=True, seed0=500):
    """n_sets logit sets of workload `name`, `rounds` rounds of fresh draft
    tokens and uniforms on each; every round's GPU outputs are compared with
    the oracle's; signals (which depend on the draft rows only) are compared
    with the oracle once per set and must repeat bit for bit."""
    import torch
    tally = Tally()
    for s_idx in range(n_sets):
        wl = W.make(name, seed0 + s_idx)
        B, G = wl.B, wl.G
        ys = draft_token_rounds(wl, rounds, [seed0, s_idx, 3])
        rng_u = np.random.default_rng([seed0, s_idx, 5])
        logits = (logits_dev(wl, "target", dev), logits_dev(wl, "draft", dev) if mode == "sample" else None)
        sig_ref, sig_first = None, None
        if mode == "sample" and signals:
            sig_ref = o.draft_signals(wl.draft, wl.gamma, wl.temperature)["signals"]
        for r in range(rounds):
            wl.draft_tokens = np.ascontiguousarray(ys[r])
            wl.uniforms = W.uniforms01(rng_u, (B, G + 1))
            g = run_gpu(mode, wl, dev, signals=signals, logits=logits)
            ref = run_oracle(o, mode, wl, signals=False)
            compare(o, mode, wl, g, ref, tally, check_signals=False)
            if sig_ref is not None:
                if sig_first is None:
                    live = ref["status"] == 0
                    compare_signals(g["signals"][live], sig_ref[live])
                    sig_first = g["signals"]
                else:
                    live = (ref["status"] == 0) & (g["status"] == 0)
                    assert np.array_equal(g["signals"][live], sig_first[live]), "signals changed between rounds"
        del logits
        torch.cuda.empty_cache()
    return tally
