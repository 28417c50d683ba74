"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each ``pin_*`` function takes a loaded oracle and raises AssertionError when the
oracle disagrees with the fact it checks.  ``test_oracle_pins.py`` runs them on
the real oracle; ``test_oracle_mutants.py`` runs them on builds of the oracle
with one planted mistake each and requires that some pin fails.

Sources: the tutorial page "5.1 投机解码核心原理" (sections 3.1-3.3, 4.1-4.3,
5.1-5.2, 7) and the SpecKV page (draft signal extraction).  Probabilities are
integrated exactly over the uniforms with a midpoint grid of N points whose
breakpoints all fall on multiples of 1/N, so grid fractions are exact
rationals; distributional facts at general p, q use chi-square tests.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy import special, stats

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
N_GRID = 4200  # multiples of 1/4200: 0.1, 0.3, 1/3, 0.6, 6/7, 0.9 ...


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _grid(n=N_GRID):
    return ((np.arange(n, dtype=np.float64) + 0.5) / n).astype(np.float32)


def _f64_logits(rows):
    """[n_rows, V] probabilities -> fp64 logits ln p (-inf for 0)."""
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(rows, np.float64))


def _hist(tokens, V):
    return np.bincount(tokens, minlength=V).astype(np.float64) / len(tokens)


# ----------------------------------------------------------------------------
# exact integrals over the uniforms for the worked example (gamma = 1, V = 3)

def worked_example_paths(o, p, q, bonus, mode=O.SAMPLE, onehot_y=1):
    """Return (accept_path, reject_path, bonus_dist) integrated exactly.

    accept_path[x] = P(x proposed and accepted); reject_path[x] = P(rejected
    and residual gives x); bonus_dist = law of the extra token after an accept.
    """
    V = len(p)
    u = _grid()
    n = len(u)
    ys = [onehot_y] if mode == O.ONEHOT else list(range(V))
    qy = {y: (1.0 if mode == O.ONEHOT else q[y]) for y in ys}
    tgt1 = np.stack([_f64_logits(p), _f64_logits(bonus)])           # rows 0, 1
    dr1 = _f64_logits(q)[None, :] if q is not None else None
    # (a) acceptance probability of each proposal y: grid over u_0
    B = n * len(ys)
    target = np.broadcast_to(tgt1, (B, 2, V)).copy()
    draft = np.broadcast_to(dr1, (B, 1, V)).copy() if mode == O.SAMPLE else None
    y = np.repeat(np.asarray(ys, np.int32), n)[:, None]
    uni = np.stack([np.tile(u, len(ys)), np.full(B, 0.5, np.float32)], axis=1)
    T = np.ones(B, np.float32)
    r = o.run(mode, target=target, draft=draft, draft_tokens=y, gamma=None,
              temperature=T, uniforms=uni)
    acc = r["accept_len"].reshape(len(ys), n)
    p_acc = {yy: float(np.mean(acc[j] == 1)) for j, yy in enumerate(ys)}
    # (b) residual law after a reject of y (u_0 just below 1 rejects any a < 1)
    rej = {}
    for yy in ys:
        if p_acc[yy] >= 1.0:
            continue
        uni2 = np.stack([np.full(n, np.float32(1.0 - 2**-24)), u], axis=1)
        r2 = o.run(mode, target=np.broadcast_to(tgt1, (n, 2, V)).copy(),
                   draft=None if draft is None else np.broadcast_to(dr1, (n, 1, V)).copy(),
                   draft_tokens=np.full((n, 1), yy, np.int32), temperature=np.ones(n, np.float32),
                   uniforms=uni2)
        assert np.all(r2["accept_len"] == 0), "u_0 = 1 - 2^-24 must reject when a < 1"
        rej[yy] = _hist(r2["tokens"][:, 0], V)
    # (c) the bonus token after an accept: draw grid on u_G with u_0 = 0 (accepts a > 0)
    yb = max(ys, key=lambda yy: p_acc[yy])
    uni3 = np.stack([np.zeros(n, np.float32), u], axis=1)
    r3 = o.run(mode, target=np.broadcast_to(tgt1, (n, 2, V)).copy(),
               draft=None if draft is None else np.broadcast_to(dr1, (n, 1, V)).copy(),
               draft_tokens=np.full((n, 1), yb, np.int32), temperature=np.ones(n, np.float32),
               uniforms=uni3)
    assert np.all(r3["accept_len"] == 1)
    bonus_dist = _hist(r3["tokens"][:, 1], V)
    accept_path = np.zeros(V)
    reject_path = np.zeros(V)
    for yy in ys:
        accept_path[yy] += qy[yy] * p_acc[yy]
        if yy in rej:
            reject_path += qy[yy] * (1.0 - p_acc[yy]) * rej[yy]
    return accept_path, reject_path, bonus_dist


def pin_worked_example(o):
    """Section 4.2 / 7: accept path [0.2,0.3,0.1], 0.4 to token 0, final = p."""
    g = golden("worked_example.json")
    bonus = [0.1, 0.2, 0.7]   # a different row 1, so the bonus row is identified
    acc, rej, bon = worked_example_paths(o, g["p"], g["q"], bonus)
    np.testing.assert_allclose(acc, g["accept_path"], atol=1e-12)
    np.testing.assert_allclose(rej, g["reject_path"], atol=1e-12)
    assert abs(rej.sum() - g["reject_mass"]) < 1e-12
    np.testing.assert_allclose(acc + rej, g["final"], atol=1e-12)
    np.testing.assert_allclose(bon, bonus, atol=1e-12)


def wrong_rule_final(o):
    g = golden("worked_example.json")
    acc, rej, _ = worked_example_paths(o, g["p"], g["q"], g["p"])
    return acc + rej


def pin_worked_example_onehot(o):
    """Section 3.3 / 7: q = one-hot on token 1 -> acceptance 0.3, final = p."""
    g = golden("worked_example.json")
    y = int(np.argmax(g["onehot_q"]))
    acc, rej, _ = worked_example_paths(o, g["p"], None, g["p"], mode=O.ONEHOT, onehot_y=y)
    assert abs(acc.sum() - g["onehot_acceptance"]) < 1e-12
    np.testing.assert_allclose(acc + rej, g["onehot_final"], atol=1e-12)


# ----------------------------------------------------------------------------

def pin_acceptance_is_one_minus_tv(o):
    """Section 4.1 / 4.3: sum_y q(y) a(y) = sum min(p,q) = 1 - TV(p,q) = 1 - sum [p-q]_+."""
    rng = np.random.default_rng(5)
    for V, T in [(5, 1.0), (17, 0.7), (64, 1.3)]:
        T = float(np.float32(T))        # the oracle receives temperature as fp32
        xt = rng.normal(0, 2, V)
        xd = xt + rng.normal(0, 1, V)
        p = special.softmax(xt / T)
        q = special.softmax(xd / T)
        B = V
        r = o.run(O.SAMPLE, target=np.broadcast_to(np.stack([xt, xt]), (B, 2, V)).copy(),
                  draft=np.broadcast_to(xd[None], (B, 1, V)).copy(),
                  draft_tokens=np.arange(V, dtype=np.int32)[:, None], temperature=np.full(B, T, np.float32),
                  uniforms=np.zeros((B, 2), np.float32))
        a = r["accept_prob"][:, 0]
        A = float(np.dot(q, a))
        tv = 0.5 * np.abs(p - q).sum()
        assert abs(A - (1 - tv)) < 1e-12, (A, 1 - tv)
        assert abs(A - np.minimum(p, q).sum()) < 1e-12
        assert abs((1 - A) - np.maximum(p - q, 0).sum()) < 1e-12


def _chi2_ok(counts, probs, min_p=1e-3):
    probs = np.asarray(probs, np.float64)
    n = counts.sum()
    keep = probs > 0
    assert counts[~keep].sum() == 0, "a zero-probability token was produced"
    res = stats.chisquare(counts[keep], probs[keep] / probs[keep].sum() * n)
    return res.pvalue > min_p, res.pvalue


def pin_chi2_final_is_p(o, trials=1_000_000):
    """Section 4.2 / 5: accept + correct together give exactly p; accepted-only
    tokens follow min(p,q)/A (section 4.2 warning); the bonus follows p_{gamma+1}."""
    rng = np.random.default_rng(42)
    V, T = 8, float(np.float32(0.8))
    xt = rng.normal(0, 1.5, (2, V))
    xd = xt[0] + rng.normal(0, 1.0, V)
    p0 = special.softmax(xt[0] / T)
    p1 = special.softmax(xt[1] / T)
    q = special.softmax(xd / T)
    y = rng.choice(V, size=trials, p=q).astype(np.int32)
    uni = rng.random((trials, 2)).astype(np.float32)
    r = o.run(O.SAMPLE, target=np.broadcast_to(xt.astype(np.float32), (trials, 2, V)).copy(),
              draft=np.broadcast_to(xd.astype(np.float32)[None], (trials, 1, V)).copy(),
              draft_tokens=y[:, None], temperature=np.full(trials, T, np.float32), uniforms=uni)
    # the oracle reads fp32 logits: recompute p, q from the same fp32 values
    p0 = special.softmax(xt[0].astype(np.float32).astype(np.float64) / T)
    p1 = special.softmax(xt[1].astype(np.float32).astype(np.float64) / T)
    q = special.softmax(xd.astype(np.float32).astype(np.float64) / T)
    tok0 = r["tokens"][:, 0]
    ok, pv = _chi2_ok(np.bincount(tok0, minlength=V), p0)
    assert ok, f"final token law != p (p-value {pv:.3g})"
    accd = r["accept_len"] == 1
    mn = np.minimum(p0, q)
    ok, pv = _chi2_ok(np.bincount(tok0[accd], minlength=V), mn / mn.sum())
    assert ok, f"accepted-only law != min(p,q)/A (p-value {pv:.3g})"
    assert abs(accd.mean() - mn.sum()) < 5 * math.sqrt(mn.sum() * (1 - mn.sum()) / trials)
    ok, pv = _chi2_ok(np.bincount(r["tokens"][accd, 1], minlength=V), p1)
    assert ok, f"bonus law != p_(gamma+1) (p-value {pv:.3g})"


def pin_chi2_onehot(o, trials=1_000_000):
    """Section 3.3: one-hot q stays lossless: final token law = p."""
    rng = np.random.default_rng(43)
    V, T = 8, 1.0
    xt = rng.normal(0, 1.5, (2, V)).astype(np.float32)
    p0 = special.softmax(xt[0].astype(np.float64) / T)
    r_prop = special.softmax(rng.normal(0, 1.5, V))        # any proposal law is lossless
    y = rng.choice(V, size=trials, p=r_prop).astype(np.int32)
    uni = rng.random((trials, 2)).astype(np.float32)
    r = o.run(O.ONEHOT, target=np.broadcast_to(xt, (trials, 2, V)).copy(), draft_tokens=y[:, None],
              temperature=np.full(trials, T, np.float32), uniforms=uni)
    ok, pv = _chi2_ok(np.bincount(r["tokens"][:, 0], minlength=V), p0)
    assert ok, f"one-hot final law != p (p-value {pv:.3g})"
    # acceptance of proposal y is p(y)
    for yy in range(V):
        sel = y == yy
        a = r["accept_len"][sel].mean()
        assert abs(a - p0[yy]) < 6 * math.sqrt(p0[yy] * (1 - p0[yy]) / sel.sum()) + 1e-9


def pin_chi2_gamma0(o, trials=400_000):
    """gamma = 0: one draw from p_0, i.e. plain categorical sampling."""
    rng = np.random.default_rng(44)
    V, T = 8, float(np.float32(0.6))
    xt = rng.normal(0, 1.0, (1, V)).astype(np.float32)
    p0 = special.softmax(xt[0].astype(np.float64) / T)
    uni = rng.random((trials, 1)).astype(np.float32)
    r = o.run(O.SAMPLE, target=np.broadcast_to(xt, (trials, 1, V)).copy(), draft=None,
              draft_tokens=None, temperature=np.full(trials, T, np.float32), uniforms=uni)
    assert np.all(r["accept_len"] == 0)
    ok, pv = _chi2_ok(np.bincount(r["tokens"][:, 0], minlength=V), p0)
    assert ok, f"gamma=0 draw law != p (p-value {pv:.3g})"


def pin_chain_mean_accept_len(o, trials=200_000):
    """Sections 4.3 and 5.1: with independent positions, E[k] = sum_{i=1}^{gamma}
    prod_{j<i} A_j where A_j = sum min(p_j, q_j) = 1 - TV."""
    rng = np.random.default_rng(45)
    V, G, T = 16, 4, float(np.float32(0.9))
    xt = rng.normal(0, 2, (G + 1, V)).astype(np.float32)
    xd = (xt[:G] + rng.normal(0, 1.2, (G, V))).astype(np.float32)
    P = special.softmax(xt.astype(np.float64) / T, axis=1)
    Q = special.softmax(xd.astype(np.float64) / T, axis=1)
    A = 1.0 - 0.5 * np.abs(P[:G] - Q).sum(axis=1)
    Ek = sum(np.prod(A[:i]) for i in range(1, G + 1))
    y = np.stack([rng.choice(V, size=trials, p=Q[i]) for i in range(G)], axis=1).astype(np.int32)
    uni = rng.random((trials, G + 1)).astype(np.float32)
    r = o.run(O.SAMPLE, target=np.broadcast_to(xt, (trials, G + 1, V)).copy(),
              draft=np.broadcast_to(xd, (trials, G, V)).copy(), draft_tokens=y,
              temperature=np.full(trials, T, np.float32), uniforms=uni)
    k = r["accept_len"].astype(np.float64)
    se = k.std() / math.sqrt(trials)
    assert abs(k.mean() - Ek) < 5 * se, (k.mean(), Ek, se)
    # each round commits between 1 and gamma+1 tokens (section 5.2)
    n_commit = (r["tokens"] >= 0).sum(axis=1)
    assert np.all(n_commit == k + 1)


def pin_first_reject_stops(o):
    """Section 5.1: candidates after the first reject are void."""
    V = 4
    xt = np.log(np.array([[0.4, 0.3, 0.2, 0.1]] * 4))
    xd = np.log(np.array([[0.1, 0.2, 0.3, 0.4]] * 3))
    y = np.array([[3, 3, 0]], np.int32)            # a = 0.25 at positions 0 and 1, 1 at 2
    uni = np.array([[0.9, 0.9, 0.1, 0.5]], np.float32)
    r = o.run(O.SAMPLE, target=xt[None], draft=xd[None], draft_tokens=y,
              temperature=np.ones(1, np.float32), uniforms=uni)
    assert r["accept_len"][0] == 0
    assert r["tokens"][0, 0] in (0, 1)               # residual [p-q]_+ lives on tokens 0, 1
    assert np.all(r["tokens"][0, 1:] == -1)
    assert np.isnan(r["accept_prob"][0, 1]) and np.isnan(r["accept_prob"][0, 2])


def pin_accept_is_strict(o):
    """Section 3.2: accept iff u < a; at u == a exactly the proposal is rejected."""
    V = 4
    xt = np.zeros((1, 2, V))                       # p uniform: p(0) = 0.25 exactly
    xd = np.array([[[0.0, 0.0, -np.inf, -np.inf]]])  # q = [0.5, 0.5, 0, 0] exactly
    uni = np.array([[0.5, 0.5]], np.float32)       # u = a = 0.5
    r = o.run(O.SAMPLE, target=xt, draft=xd, draft_tokens=np.zeros((1, 1), np.int32),
              temperature=np.full(1, 0.7, np.float32), uniforms=uni)
    assert r["accept_prob"][0, 0] == 0.5
    assert r["accept_len"][0] == 0
    uni[0, 0] = np.nextafter(np.float32(0.5), np.float32(0))
    r = o.run(O.SAMPLE, target=xt, draft=xd, draft_tokens=np.zeros((1, 1), np.int32),
              temperature=np.full(1, 0.7, np.float32), uniforms=uni)
    assert r["accept_len"][0] == 1


def pin_draw_convention(o):
    """Inverse-CDF convention: smallest x with C(x) > u W (the page's experiment
    draws with Python's weighted choice, which bisects to the right); tokens of
    weight 0 are never drawn, even when u W lands exactly on a boundary."""
    xt = np.array([[[0.0, -np.inf, 0.0, -np.inf]]])   # p = [0.5, 0, 0.5, 0] exactly
    for u, want in [(0.0, 0), (0.25, 0), (0.5, 2), (0.75, 2), (1 - 2**-24, 2)]:
        r = o.run(O.SAMPLE, target=xt, draft=None, draft_tokens=None,
                  temperature=np.ones(1, np.float32), uniforms=np.array([[u]], np.float32))
        assert r["tokens"][0, 0] == want, (u, r["tokens"][0, 0], want)


def pin_p_equals_q(o):
    """Section 4.2: p = q gives beta = 0, so nothing is ever rejected."""
    rng = np.random.default_rng(46)
    B, G, V = 64, 5, 50
    xt = rng.normal(0, 3, (B, G + 1, V)).astype(np.float32)
    xd = xt[:, :G, :].copy()
    Q = special.softmax(xd.astype(np.float64), axis=2)
    y = np.array([[rng.choice(V, p=Q[b, i]) for i in range(G)] for b in range(B)], np.int32)
    uni = rng.random((B, G + 1)).astype(np.float32)
    r = o.run(O.SAMPLE, target=xt, draft=xd, draft_tokens=y, temperature=np.ones(B, np.float32),
              uniforms=uni)
    assert np.all(r["accept_len"] == G)
    assert np.all(r["tokens"][:, :G] == y)


def pin_greedy_is_target_argmax(o):
    """Section 3.1: the committed tokens are the target's own greedy decoding:
    the accepted prefix equals argmax at each position and the emitted token is
    the argmax at the first mismatch (or the bonus argmax); ties -> lowest index."""
    rng = np.random.default_rng(47)
    B, G, V = 200, 6, 12
    xt = rng.integers(-3, 3, (B, G + 1, V)).astype(np.float32)   # many ties
    am = np.argmax(xt, axis=2)                                   # numpy: first maximum
    y = am[:, :G].copy()
    flip = rng.random((B, G)) < 0.25
    y[flip] = rng.integers(0, V, flip.sum())
    r = o.run(O.GREEDY, target=xt, draft_tokens=y.astype(np.int32))
    for b in range(B):
        k = r["accept_len"][b]
        mism = np.nonzero(y[b] != am[b, :G])[0]
        assert k == (mism[0] if len(mism) else G)
        assert np.all(r["tokens"][b, :k + 1] == am[b, :k + 1])
        assert np.all(r["tokens"][b, k + 1:] == -1)
    # a draft that always proposes the argmax is accepted to the end
    r = o.run(O.GREEDY, target=xt, draft_tokens=am[:, :G].astype(np.int32))
    assert np.all(r["accept_len"] == G)


def pin_signals_closed_forms(o):
    """SpecKV signals: H = -sum q log2 q, c = max q, with per-request mean/max
    entropy and mean/min confidence over the gamma_b draft rows."""
    V, G = 64, 4
    rows = np.full((1, G, V), -1e4)
    rows[0, 0, :] = 0.0                         # uniform: H = log2 V, c = 1/V
    rows[0, 1, :2] = 0.0                        # two-way tie: H = 1, c = 1/2
    rows[0, 2, 5] = 0.0                         # one token: H = 0, c = 1
    rows[0, 3, :] = 0.0                         # padding row, beyond gamma_b = 3
    r = o.draft_signals(rows, gamma=np.array([3], np.int32), temperature=np.ones(1, np.float32),
                        want_row_signals=True)
    H = np.array([math.log2(V), 1.0, 0.0])
    c = np.array([1.0 / V, 0.5, 1.0])
    np.testing.assert_allclose(r["row_signals"][0, :3, 0], H, atol=1e-12)
    np.testing.assert_allclose(r["row_signals"][0, :3, 1], c, atol=1e-12)
    assert np.all(np.isnan(r["row_signals"][0, 3]))
    np.testing.assert_allclose(r["signals"][0], [H.mean(), H.max(), c.mean(), c.min()], atol=1e-12)
    # temperature: logits [ln 3 * T, 0] at T give q = [3/4, 1/4]
    T = float(np.float32(0.6))
    x = np.full((1, 1, 5), -1e4)
    x[0, 0, 0] = math.log(3.0) * T
    x[0, 0, 1] = 0.0
    r = o.draft_signals(x, gamma=np.array([1], np.int32), temperature=np.full(1, T, np.float32))
    Hq = -(0.75 * math.log2(0.75) + 0.25 * math.log2(0.25))
    assert abs(r["signals"][0, 0] - Hq) < 1e-6 and abs(r["signals"][0, 2] - 0.75) < 1e-6
    # random rows against scipy's entropy (base 2)
    rng = np.random.default_rng(48)
    x = rng.normal(0, 2, (3, 6, 300))
    g = np.array([6, 2, 5], np.int32)
    Tb = np.array([1.0, 0.7, 1.4], np.float32)
    r = o.draft_signals(x, gamma=g, temperature=Tb)
    for b in range(3):
        qs = special.softmax(x[b, :g[b]] / np.float64(Tb[b]), axis=1)
        Hs = stats.entropy(qs, base=2, axis=1)
        cs = qs.max(axis=1)
        np.testing.assert_allclose(r["signals"][b], [Hs.mean(), Hs.max(), cs.mean(), cs.min()],
                                   rtol=1e-10)


def pin_bf16_inputs(o):
    """bf16 logits widen exactly: a bf16 row and the same values in fp32 give
    identical results; known bit patterns decode to their values."""
    pats = np.array([0x3F80, 0xC040, 0x4000, 0x0000, 0xBF80, 0x4040], np.uint16)  # 1,-3,2,0,-1,3
    r = o.run(O.GREEDY, target=pats[None, None, :], draft_tokens=np.zeros((1, 0), np.int32),
              G=0)
    assert r["tokens"][0, 0] == 5
    vals = np.array([1.0, -3.0, 2.0, 0.0, -1.0, 3.0], np.float32)
    x = np.stack([pats, pats[::-1].copy()])[None]                 # [1, 2, 6]
    xf = np.stack([vals, vals[::-1].copy()])[None]
    d = pats[None, None, :].copy()
    df = vals[None, None, :].copy()
    kw = dict(draft_tokens=np.array([[2]], np.int32), temperature=np.full(1, 0.9, np.float32),
              uniforms=np.array([[0.3, 0.6]], np.float32), want_signals=True)
    a = o.run(O.SAMPLE, target=x, draft=d, **kw)
    b = o.run(O.SAMPLE, target=xf, draft=df, **kw)
    for key in ("accept_len", "tokens", "accept_prob", "signals"):
        np.testing.assert_array_equal(a[key], b[key])


def pin_status_semantics(o):
    """Readings on bad inputs: errors void the request; rows, tokens and
    uniforms after the first reject are never looked at."""
    V, G = 6, 3
    base_t = np.zeros((1, G + 1, V))
    base_t[0, :, 0] = 2.0
    base_d = np.zeros((1, G, V))
    base_d[0, :, 1] = 3.0                       # q prefers token 1, p token 0
    y = np.array([[1, 0, 0]], np.int32)
    T = np.ones(1, np.float32)
    u = np.array([[0.99, 0.1, 0.1, 0.5]], np.float32)   # position 0 rejects

    def run(mode=O.SAMPLE, **kw):
        args = dict(target=base_t, draft=base_d, draft_tokens=y, temperature=T, uniforms=u)
        args.update(kw)
        if mode != O.SAMPLE:
            args.pop("draft")
        if mode == O.GREEDY:
            args.pop("temperature"); args.pop("uniforms")
        return o.run(mode, **args)

    r = run()
    assert r["status"][0] == 0 and r["accept_len"][0] == 0
    t = base_t.copy(); t[0, 2, 3] = np.nan                   # after the reject: not read
    assert run(target=t)["status"][0] == 0
    t = base_t.copy(); t[0, 0, 3] = np.nan
    r = run(target=t)
    assert r["status"][0] == O.ST_NONFINITE and np.all(r["tokens"] == -1)
    t = base_t.copy(); t[0, 0, 3] = np.inf
    assert run(target=t)["status"][0] == O.ST_NONFINITE
    t = base_t.copy(); t[0, 0, 3] = -np.inf                  # a masked token is fine
    assert run(target=t)["status"][0] == 0
    t = base_t.copy(); t[0, 0, :] = -np.inf                  # no finite maximum
    assert run(target=t)["status"][0] == O.ST_NONFINITE
    assert run(draft_tokens=np.array([[V, 0, 0]], np.int32))["status"][0] == O.ST_BAD_TOKEN
    assert run(draft_tokens=np.array([[1, -1, 0]], np.int32))["status"][0] == 0
    assert run(gamma=np.array([4], np.int32))["status"][0] == O.ST_BAD_GAMMA
    assert run(gamma=np.array([-1], np.int32))["status"][0] == O.ST_BAD_GAMMA
    assert run(temperature=np.zeros(1, np.float32))["status"][0] == O.ST_BAD_TEMPERATURE
    assert run(temperature=np.full(1, np.nan, np.float32))["status"][0] == O.ST_BAD_TEMPERATURE
    assert run(uniforms=np.array([[1.0, 0.1, 0.1, 0.5]], np.float32))["status"][0] == O.ST_BAD_UNIFORM
    assert run(uniforms=np.array([[0.99, 0.1, 0.1, -0.5]], np.float32))["status"][0] == O.ST_BAD_UNIFORM
    assert run(uniforms=np.array([[0.99, 2.0, 0.1, 0.5]], np.float32))["status"][0] == 0
    # greedy: mismatch at position 0 stops; a NaN later is not read
    t = base_t.copy(); t[0, 1, 2] = np.nan
    r = run(O.GREEDY, target=t)
    assert r["status"][0] == 0 and r["accept_len"][0] == 0 and r["tokens"][0, 0] == 0
    # one-hot: proposal 1 has p(1) ~ 0.08, so u = 0.99 rejects it
    r = run(O.ONEHOT)
    assert r["status"][0] == 0


def pin_decision_margins(o):
    """The near-tie diagnostics the parity comparison relies on, on rows whose
    probabilities are exact binary fractions (values computed by hand):
      accept_margin  = |u - a|, a = min(1, p(y)/q(y))   (tutorial section 3.2);
      draw_margin    = min(t - C(z-1), C(z) - t) / W with t = u W, z the drawn
                       token and C the ascending cumulative weight;
      probe_distance = the distance from t to the bucket [C(v-1), C(v)) of a
                       given token v, over W (0 when t lies inside it)."""
    one = np.ones(1, np.float32)
    # draw from p = [1/2, 0, 1/2, 0] (gamma = 0, W = 1): buckets [0, .5), -, [.5, 1), -
    xt = np.array([[[0.0, -np.inf, 0.0, -np.inf]]])
    for u, z, margin in [(0.5 - 2**-24, 0, 2**-24), (0.25, 0, 0.25), (0.125, 0, 0.125),
                         (0.625, 2, 0.125), (0.75, 2, 0.25), (0.5, 2, 0.0)]:
        r = o.run(O.SAMPLE, target=xt, draft=None, draft_tokens=None, temperature=one,
                  uniforms=np.array([[u]], np.float32))
        assert r["tokens"][0, 0] == z, (u, r["tokens"][0, 0])
        assert r["draw_margin"][0] == margin, (u, r["draw_margin"][0], margin)
    # probe distances on p = [1/2, 1/4, 1/4] (logits ln 2, 0, 0): buckets
    # [0, .5), [.5, .75), [.75, 1)
    xt = np.array([[[math.log(2.0), 0.0, 0.0]]])
    for u, probe, dist in [(0.125, 1, 0.375), (0.125, 2, 0.625), (0.125, 0, 0.0),
                           (0.875, 0, 0.375), (0.875, 1, 0.125), (0.625, 1, 0.0),
                           (0.625, 2, 0.125), (0.5, 0, 0.0), (0.5, 1, 0.0)]:
        r = o.run(O.SAMPLE, target=xt, draft=None, draft_tokens=None, temperature=one,
                  uniforms=np.array([[u]], np.float32), probe_token=np.array([probe], np.int32))
        assert abs(r["probe_distance"][0] - dist) < 1e-15, (u, probe, r["probe_distance"][0], dist)
    # on a residual: p = [1/2, 1/4, 1/4], q = [1/4, 1/2, 1/4] -> [p - q]_+ = [1/4, 0, 0];
    # W = 1/4, so t = u / 4 and the margin is measured over W
    xd = np.array([[[0.0, math.log(2.0), 0.0]]])
    tgt = np.concatenate([xt, xt], axis=1)
    for u_draw, margin in [(0.5, 0.5), (0.125, 0.125), (0.875, 0.125)]:
        r = o.run(O.SAMPLE, target=tgt, draft=xd, draft_tokens=np.array([[1]], np.int32), temperature=one,
                  uniforms=np.array([[1 - 2**-24, u_draw]], np.float32))
        assert r["accept_len"][0] == 0 and r["tokens"][0, 0] == 0
        assert abs(r["draw_margin"][0] - margin) < 1e-15, (u_draw, r["draw_margin"][0])
    # acceptance margins: worked example p = [.6, .3, .1], q = [.2, .5, .3]
    # a(0) = 1, a(1) = 0.6, a(2) = 1/3
    g = golden("worked_example.json")
    tg = np.stack([_f64_logits(g["p"]), _f64_logits(g["p"])])[None]
    dr = _f64_logits(g["q"])[None, None]
    for y, u, margin in [(1, 0.5, 0.1), (1, 0.75, 0.15), (2, 0.25, 1.0 / 12), (0, 0.875, 0.125),
                         (2, 0.5, 1.0 / 6)]:
        r = o.run(O.SAMPLE, target=tg, draft=dr, draft_tokens=np.array([[y]], np.int32), temperature=one,
                  uniforms=np.array([[u, 0.5]], np.float32))
        assert abs(r["accept_margin"][0, 0] - margin) < 1e-12, (y, u, r["accept_margin"][0, 0], margin)
    # one-hot: the margin is |u - p(y)|
    r = o.run(O.ONEHOT, target=tg, draft_tokens=np.array([[1]], np.int32), temperature=one,
              uniforms=np.array([[0.5, 0.5]], np.float32))
    assert abs(r["accept_margin"][0, 0] - 0.2) < 1e-12


def pin_divergence(o):
    """Per-position divergence statistics (A = sum min(p, q) = 1 - TV(p, q):
    tutorial section 4.3; L1 and forward KL: the DLite page's distillation
    losses; bidirectional KL and entropies: the DDTE page's selector inputs),
    in bits, against facts that do not restate the oracle's sums:
      - the worked example of section 7: A = 0.6 and L1 = 0.8 by hand, KL both
        ways and H(p) by scipy's (relative) entropy;
      - random rows at T = 0.7: KL both ways and H(p) by scipy, A + L1 / 2 = 1
        (TV = L1 / 2), and A equal to the expected acceptance of the verify
        path, sum_y q(y) min(1, p(y)/q(y)), from the oracle's accept_prob for
        every draft token y (a different code path: the acceptance test);
      - p = q: A = 1, L1 = 0, KL = 0; a uniform target row: H = log2 V;
      - a draft row with a -inf logit where p > 0: KL(p||q) = +inf, KL(q||p)
        finite; positions past gamma and bad gamma / temperature: NaN."""
    g = golden("worked_example.json")
    pw, qw = np.array(g["p"]), np.array(g["q"])
    tg = _f64_logits(np.stack([pw, pw]))[None]
    dr = _f64_logits(qw[None])[None]
    r = o.divergence_stats(tg, dr, None, np.ones(1, np.float32))
    st = r["stats"][0, 0]
    assert abs(st[0] - 0.6) < 1e-12 and abs(st[1] - 0.8) < 1e-12, st
    assert abs(st[2] - stats.entropy(pw, qw, base=2)) < 1e-12, st
    assert abs(st[3] - stats.entropy(qw, pw, base=2)) < 1e-12, st
    assert abs(st[4] - stats.entropy(pw, base=2)) < 1e-12, st
    # random rows at T = 0.7
    rng = np.random.default_rng(11)
    V, T = 40, float(np.float32(0.7))          # the oracle takes T as float32
    xt = rng.normal(0.0, 2.0, V)
    xd = xt + rng.normal(0.0, 1.0, V)
    p = special.softmax(xt / T)
    q = special.softmax(xd / T)
    r = o.divergence_stats(np.stack([xt, xt])[None], xd[None, None], None, np.full(1, T, np.float32))
    st = r["stats"][0, 0]
    assert abs(st[2] - stats.entropy(p, q, base=2)) < 1e-12, (st[2], stats.entropy(p, q, base=2))
    assert abs(st[3] - stats.entropy(q, p, base=2)) < 1e-12
    assert abs(st[4] - stats.entropy(p, base=2)) < 1e-12
    assert abs(st[0] + st[1] / 2 - 1.0) < 1e-12, st
    # A against the acceptance test: one request per draft token y
    ys = np.arange(V, dtype=np.int32)[:, None]
    acc = o.run(O.SAMPLE, target=np.broadcast_to(np.stack([xt, xt])[None], (V, 2, V)),
                draft=np.broadcast_to(xd[None, None], (V, 1, V)), draft_tokens=ys,
                temperature=np.full(V, T, np.float32), uniforms=np.full((V, 2), 0.5, np.float32))["accept_prob"][:, 0]
    assert abs(st[0] - float(np.dot(q, acc))) < 1e-12, (st[0], float(np.dot(q, acc)))
    # p = q and a uniform target row
    r = o.divergence_stats(np.stack([xd, xd])[None], xd[None, None], None, np.full(1, T, np.float32))
    st = r["stats"][0, 0]
    assert abs(st[0] - 1.0) < 1e-12 and abs(st[1]) < 1e-12 and abs(st[2]) < 1e-12 and abs(st[3]) < 1e-12, st
    z = np.zeros(V)
    st = o.divergence_stats(np.stack([z, z])[None], xd[None, None], None, np.ones(1, np.float32))["stats"][0, 0]
    assert abs(st[4] - math.log2(V)) < 1e-12, st
    # a draft zero under target mass
    xd2 = xd.copy()
    xd2[3] = -np.inf
    st = o.divergence_stats(np.stack([xt, xt])[None], xd2[None, None], None, np.ones(1, np.float32))["stats"][0, 0]
    assert st[2] == np.inf and np.isfinite(st[3]), st
    # gamma and temperature handling
    tg3 = np.broadcast_to(np.stack([xt, xt, xt])[None], (3, 3, V))
    dr3 = np.broadcast_to(np.stack([xd, xd])[None], (3, 2, V))
    r = o.divergence_stats(tg3, dr3, np.array([1, 3, 2], np.int32), np.array([1.0, 1.0, -1.0], np.float32))
    s3 = r["stats"]
    assert np.isfinite(s3[0, 0]).all() and np.isnan(s3[0, 1]).all(), s3[0]
    assert np.isnan(s3[1]).all() and r["status"][1] == 4, r["status"]
    assert np.isnan(s3[2]).all() and r["status"][2] == 64, r["status"]
    assert r["status"][0] == 0
    # a row with no finite maximum voids its own position only
    tg4 = np.stack([xt, xt, xt])[None].copy()
    tg4[0, 0, :] = -np.inf
    r = o.divergence_stats(tg4, np.stack([xd, xd])[None], None, np.ones(1, np.float32))
    assert r["status"][0] == 1 and np.isnan(r["stats"][0, 0]).all() and np.isfinite(r["stats"][0, 1]).all(), r


def pin_gamma_select(o):
    """The SpecKV gamma selector (SpecKV page, acceptance prediction and gamma
    selection): E[tokens] = f(x, gamma) gamma + 1 with x = [mean H, mean c,
    max H, min c, comp], gamma* = argmax over {2, 4, 6, 8}; f an MLP with 16
    hidden units on the standardised inputs [x, gamma].
      - f against scikit-learn's MLPRegressor (ReLU hidden layer, identity
        output) fitted on random data, its scaler and weights copied into the
        141-value model;
      - a hand-built selector f = a - b gamma, whose expected tokens
        a gamma - b gamma^2 + 1 peak at gamma = a / (2b): an exact tie between
        4 and 6 (a = 1.25, b = 1/8: the smaller is taken), and a peak at 7.1
        (8 is taken);
      - a non-finite feature gives -1."""
    pytest_sklearn = __import__("importlib").util.find_spec("sklearn")
    rng = np.random.default_rng(21)
    sig = np.column_stack([rng.uniform(0.5, 6, 50), rng.uniform(2, 12, 50),        # mean H, max H
                           rng.uniform(0.2, 0.9, 50), rng.uniform(0.05, 0.5, 50)])  # mean c, min c
    comp = rng.integers(0, 3, 50).astype(np.float64)
    if pytest_sklearn is not None:
        from sklearn.neural_network import MLPRegressor
        from sklearn.preprocessing import StandardScaler
        X = np.column_stack([rng.uniform(0.5, 6, 400), rng.uniform(0.2, 0.9, 400), rng.uniform(2, 12, 400),
                             rng.uniform(0.05, 0.5, 400), rng.integers(0, 3, 400), rng.choice([2, 4, 6, 8], 400)])
        y = rng.uniform(0, 1, 400)
        sc = StandardScaler().fit(X)
        mlp = MLPRegressor(hidden_layer_sizes=(16,), activation="relu", max_iter=300, random_state=0).fit(
            sc.transform(X), y)
        model = np.concatenate([sc.mean_, sc.scale_, mlp.coefs_[0].T.ravel(), mlp.intercepts_[0],
                                mlp.coefs_[1][:, 0], mlp.intercepts_[1]])
        r = o.gamma_select(sig, comp, model)
        for j, g in enumerate((2, 4, 6, 8)):
            xin = np.column_stack([sig[:, 0], sig[:, 2], sig[:, 1], sig[:, 3], comp, np.full(50, g)])
            want = mlp.predict(sc.transform(xin)) * g + 1.0
            assert np.allclose(r["expected"][:, j], want, rtol=1e-12, atol=1e-12), (g, r["expected"][:5, j], want[:5])
        assert np.array_equal(r["gamma"], np.array((2, 4, 6, 8))[np.argmax(r["expected"], axis=1)])
    # f = a - b gamma: one hidden unit passes gamma (mu 0, sd 1), a second
    # one is off (ReLU of -gamma) unless the hidden layer were linear
    def selector(a, b):
        m = np.zeros(141)
        m[6:12] = 1.0                      # sd
        W1 = np.zeros((16, 6))
        W1[0, 5] = 1.0
        W1[1, 5] = -1.0
        m[12:108] = W1.ravel()
        w2 = np.zeros(16)
        w2[0] = -b
        w2[1] = 0.3
        m[124:140] = w2
        m[140] = a
        return m
    one = np.array([[1.0, 2.0, 0.6, 0.3]])
    r = o.gamma_select(one, None, selector(1.25, 0.125))
    assert r["gamma"][0] == 4, r               # E(4) = E(6) = 4 exactly: the smaller gamma
    assert np.array_equal(r["expected"][0], [3.0, 4.0, 4.0, 3.0]), r["expected"]
    r = o.gamma_select(one, None, selector(1.0, 0.07))
    assert r["gamma"][0] == 8, r               # peak at 7.1: E(6) = 4.48 < E(8) = 4.52
    bad = np.array([[np.nan, 2.0, 0.6, 0.3]])
    r = o.gamma_select(bad, None, selector(1.25, 0.125))
    assert r["gamma"][0] == -1 and np.isnan(r["expected"][0]).all()


def pin_filter(o):
    """Top-k / top-p filtering before verification (tutorial page, section
    2.1: p and q already include temperature / top-k / top-p when used),
    read by value: top-k keeps x >= the k-th largest logit; top-p, on the
    distribution left by top-k at temperature T, keeps x >= t*, the largest
    value whose upper mass {x >= t*} reaches top_p.  Checked on rows of exact
    binary fractions by hand, against a brute-force search over every
    candidate threshold on small random rows with ties, and on rows of 200 to
    4000 logits against the same definition computed by sorting in numpy."""
    one = np.ones(1, np.float32)
    x = np.log(np.array([[0.5, 0.25, 0.125, 0.0625, 0.0625]]))

    def kept(k, p, T=1.0, row=x):
        r = o.filter_logits(row, None if k is None else np.array([k]), None if p is None else np.array([p]),
                            np.array([T], np.float32))
        return np.isfinite(r["logits"][0]).astype(int).tolist()
    assert kept(None, 0.7) == [1, 1, 0, 0, 0]      # 0.5, 0.75 >= 0.7
    assert kept(None, 0.75) == [1, 1, 0, 0, 0]     # the crossing value is kept (mass >= top_p)
    assert kept(None, 0.76) == [1, 1, 1, 0, 0]
    assert kept(None, 0.95) == [1, 1, 1, 1, 1]     # the tie group {1/16, 1/16} together
    assert kept(3, None) == [1, 1, 1, 0, 0]
    assert kept(4, None) == [1, 1, 1, 1, 1]        # the 4th largest is tied with the 5th
    assert kept(3, 0.8) == [1, 1, 0, 0, 0]         # after top-k: 4/7, 6/7 >= 0.8
    assert kept(0, 1.0) == [1, 1, 1, 1, 1] and kept(5, None) == [1, 1, 1, 1, 1]
    # T = 2 flattens p to [0.354, 0.25, 0.177, 0.125, 0.125] / 1.030: 0.5 takes 2 tokens
    assert kept(None, 0.5, T=2.0) == [1, 1, 0, 0, 0] and kept(None, 0.5) == [1, 0, 0, 0, 0]
    # brute force: every candidate threshold of the row, in fp64
    rng = np.random.default_rng(31)
    for trial in range(300):
        V = int(rng.integers(2, 12))
        row = np.round(rng.normal(0, 2, V), 1)           # rounding makes ties
        k = int(rng.integers(0, V + 1))
        p = float(np.float32(rng.uniform(0.05, 1.0)))
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        got = np.isfinite(o.filter_logits(row[None], np.array([k]), np.array([p]), np.array([T]))["logits"][0])
        cand = np.sort(np.unique(row))[::-1]
        keep = row >= np.sort(row)[::-1][k - 1] if 1 <= k < V else np.ones(V, bool)
        if p < 1.0:
            w = special.softmax(row[keep] / T)
            vals = row[keep]
            tstar = None
            for v in cand:                                  # descending candidate thresholds
                if (vals >= v).any() and w[vals >= v].sum() >= p:
                    tstar = v
                    break
            keep = keep & (row >= tstar)
        assert np.array_equal(got, keep), (row, k, p, T, got, keep)
    # larger rows: the same definition by sorting (value groups, cumulative fp64
    # softmax mass from the top); rows whose crossing is within 1e-9 of top_p are
    # left out, as summation order may decide them
    checked = 0
    for trial in range(60):
        V = int(rng.choice([200, 1000, 4000]))
        row = np.round(rng.normal(0, 2, V), 2)
        k = int(rng.choice([0, 1, 7, 50, V // 3, V - 1, V]))
        p = float(np.float32(rng.choice([1.0, 0.5, 0.9, 0.99, rng.uniform(0.05, 1.0)])))
        T = float(np.float32(rng.uniform(0.3, 2.0)))
        keep = row >= np.sort(row)[::-1][k - 1] if 1 <= k < V else np.ones(V, bool)
        if p < 1.0:
            vals = row[keep]
            w = special.softmax(vals / T)
            groups = np.unique(vals)[::-1]                  # descending value groups
            mass = np.array([w[vals == g].sum() for g in groups])
            cum = np.cumsum(mass)
            j = int(np.argmax(cum >= p))
            if abs(cum[j] - p) < 1e-9 or (j > 0 and abs(cum[j - 1] - p) < 1e-9):
                continue
            keep = keep & (row >= groups[j])
        got = np.isfinite(o.filter_logits(row[None], np.array([k]), np.array([p]), np.array([T]))["logits"][0])
        assert np.array_equal(got, keep), (V, k, p, T, int(got.sum()), int(keep.sum()))
        checked += 1
    assert checked >= 50


ALL_PINS = [
    pin_worked_example,
    pin_worked_example_onehot,
    pin_acceptance_is_one_minus_tv,
    pin_chi2_final_is_p,
    pin_chi2_onehot,
    pin_chi2_gamma0,
    pin_chain_mean_accept_len,
    pin_first_reject_stops,
    pin_accept_is_strict,
    pin_draw_convention,
    pin_p_equals_q,
    pin_greedy_is_target_argmax,
    pin_signals_closed_forms,
    pin_bf16_inputs,
    pin_status_semantics,
    pin_decision_margins,
    pin_divergence,
    pin_gamma_select,
    pin_filter,
]
