"""spec_filter_top_k_top_p against the fp64 oracle (oracle_filter), through
the C ABI.

Kept sets must be the oracle's exactly, and kept logits bit-identical to the
input, except on rows whose top-p decision the oracle flags as within 1e-5
of its threshold (the fp32 weights carry ~1e-6 of mass error): there the
GPU's threshold may be the oracle's or an adjacent value group.  Removed
logits are -inf; statuses must be equal.
"""
import numpy as np
import pytest

import oracle as O
import parity as PT
from speculative_decoding_verification_26_gb300 import workloads as W

pytestmark = pytest.mark.gpu
FLAG = 1e-5


@pytest.fixture(scope="module")
def o():
    return O.load()


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    return torch.device("cuda:0")


def gpu_filter(dev, rows, bf16, k, p, T):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    x = PT.to_dev(rows.view(np.int16) if bf16 else rows, dev, bf16=bf16)
    kt = None if k is None else torch.from_numpy(np.ascontiguousarray(k, np.int32)).to(dev)
    pt = None if p is None else torch.from_numpy(np.ascontiguousarray(p, np.float32)).to(dev)
    Tt = None if T is None else torch.from_numpy(np.ascontiguousarray(T, np.float32)).to(dev)
    st = sv.filter_top_k_top_p(x, kt, pt, Tt)
    torch.cuda.synchronize()
    out = x.float().cpu().numpy().astype(np.float64) if bf16 else x.cpu().numpy().astype(np.float64)
    return out, st.cpu().numpy()


def check(o, dev, rows, bf16, k, p, T, what):
    want = o.filter_logits(rows, k, p, T)
    got, st = gpu_filter(dev, rows, bf16, k, p, T)
    inp = W.bf16_bits_to_f32(rows).astype(np.float64) if bf16 else rows.astype(np.float64)
    assert np.array_equal(st, want["status"]), (what, st, want["status"])
    n_flag = 0
    for r in range(rows.shape[0]):
        g, w = np.isfinite(got[r]), np.isfinite(want["logits"][r])
        if want["status"][r] != 0:
            assert np.array_equal(got[r], inp[r], equal_nan=True), (what, r)
            continue
        # kept logits unchanged, removed ones -inf
        assert np.array_equal(got[r][g], inp[r][g]), (what, r)
        assert (got[r][~g] == -np.inf).all()
        if np.array_equal(g, w):
            continue
        assert want["margin"][r] < FLAG, (what, r, want["margin"][r], g.sum(), w.sum())
        n_flag += 1
        vals = np.unique(inp[r][np.isfinite(inp[r])])[::-1]
        tg, to = inp[r][g].min(), inp[r][w].min()
        ig, io = int(np.nonzero(vals == tg)[0][0]), int(np.nonzero(vals == to)[0][0])
        assert abs(ig - io) <= 1, (what, r, ig, io)
        assert np.array_equal(g, inp[r] >= tg)
    return n_flag


def rows_of(name, n, V=None, dtype=None):
    kw = {"overrides": {"dtype": dtype}} if dtype else {}
    wl = W.make(name, 5, B=max(1, n // 8 + 1), V=V, **kw)
    rows = wl.target.reshape(-1, wl.V)[:n]
    return np.ascontiguousarray(rows), wl.dtype == W.BF16


@pytest.mark.parametrize("name,V,dtype", [("m", None, None), ("c3", None, None), ("c3", 40000, W.F32),
                                          ("c1", None, None), ("c3", 1001, W.BF16), ("c3", 7, W.F32)])
def test_top_k_top_p(o, dev, name, V, dtype):
    rows, bf16 = rows_of(name, 48, V, dtype)
    n, Vr = rows.shape
    rng = np.random.default_rng(Vr)
    k = rng.choice([0, 1, 2, 5, 20, 50, Vr - 1, Vr, Vr + 3], n).astype(np.int32)
    p = rng.choice([1.0, 0.5, 0.9, 0.99, 0.999, 1e-3], n).astype(np.float32)
    T = rng.choice([0.6, 0.7, 1.0, 1.3], n).astype(np.float32)
    flagged = check(o, dev, rows, bf16, k, p, T, f"{name} V={Vr}")
    assert flagged <= 2


def test_top_k_only_and_top_p_only(o, dev):
    rows, bf16 = rows_of("m", 16)
    n = rows.shape[0]
    check(o, dev, rows, bf16, np.full(n, 40, np.int32), None, None, "top-k only")
    check(o, dev, rows, bf16, None, np.full(n, 0.9, np.float32), np.full(n, 0.7, np.float32), "top-p only")


def test_ties_and_special_rows(o, dev):
    rng = np.random.default_rng(3)
    n, V = 8, 2000
    rows = np.round(rng.normal(0, 2, (n, V)), 1).astype(np.float32)   # many ties
    rows[1, :] = 0.0                          # every logit tied
    rows[2, 5] = -np.inf
    rows[3, 7] = np.nan                       # unchanged, NONFINITE
    rows[4, :] = -np.inf                      # no finite logit: unchanged, NONFINITE
    rows[5, 3] = -0.0                         # -0 and +0 are one value
    rows[5, 4] = 0.0
    k = np.array([10, 5, 30, 10, 10, 100, 1, 2], np.int32)
    p = np.array([0.7, 0.5, 0.95, 0.9, 0.9, 0.999, 1.0, 0.3], np.float32)
    T = np.array([1.0, 1.0, 0.8, 1.0, 1.0, 1.0, 1.0, -1.0], np.float32)   # row 7: bad T with top-p
    check(o, dev, rows, False, k, p, T, "ties and special rows")


def test_deterministic(dev):
    rows, bf16 = rows_of("m", 24)
    n = rows.shape[0]
    args = (np.full(n, 100, np.int32), np.full(n, 0.95, np.float32), np.full(n, 0.7, np.float32))
    a, _ = gpu_filter(dev, rows, bf16, *args)
    b, _ = gpu_filter(dev, rows, bf16, *args)
    assert np.array_equal(a, b)


def test_filtered_rows_feed_the_verification(o, dev):
    """Filter the target and draft rows of a round on the GPU (kept sets equal
    to the oracle's on every row the oracle does not flag), then verify the
    filtered round: GPU and oracle must agree on the same filtered logits."""
    wl = W.make("c3", 4, B=8)
    B, G, V = wl.B, wl.G, wl.V
    kt, pt = np.full(B * (G + 1), 200, np.int32), np.full(B * (G + 1), 0.95, np.float32)
    Tt, Td = np.repeat(wl.temperature, G + 1), np.repeat(wl.temperature, G)
    gt, _ = gpu_filter(dev, wl.target.reshape(-1, V).copy(), True, kt, pt, Tt)
    gd, _ = gpu_filter(dev, wl.draft.reshape(-1, V).copy(), True, kt[:B * G], pt[:B * G], Td)
    ot = o.filter_logits(wl.target.reshape(-1, V), kt, pt, Tt)
    od = o.filter_logits(wl.draft.reshape(-1, V), kt[:B * G], pt[:B * G], Td)
    for g, w in ((gt, ot), (gd, od)):
        ok = w["margin"] >= FLAG
        assert np.array_equal(np.isfinite(g)[ok], np.isfinite(w["logits"])[ok])
    wl.target = W.bf16_rne_bits(gt.astype(np.float32)).reshape(B, G + 1, V)
    wl.draft = W.bf16_rne_bits(gd.astype(np.float32)).reshape(B, G, V)
    W.resolve_draft_tokens(wl, PT.oracle_argmax(o))      # the drafter samples the filtered q
    g = PT.run_gpu("sample", wl, dev, signals=True)
    r = PT.run_oracle(o, "sample", wl, signals=True)
    assert np.array_equal(g["accept_len"], r["accept_len"])
    assert np.array_equal(g["tokens"], r["tokens"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_top_ties_overflow_the_candidate_list(o, dev, dtype):
    """Rows whose top value is shared by more logits than the candidate list
    holds (20000 of 30000): the bound from the threads' maxima keeps them all,
    so the kernel falls back to counting the row; ties stay together.  Row 6
    takes the same fallback with top-p alone; row 7 (nearly flat, top-p 0.99
    alone) gives a list that fits but carries too little mass, the other
    fallback of top-p alone."""
    rng = np.random.default_rng(11)
    n, V = 8, 30000
    rows = rng.normal(-4, 1, (n, V)).astype(np.float32)
    for r in range(7):
        rows[r, rng.choice(V, 20000, replace=False)] = 1.0
    rows[5, :] = 1.0                                   # every logit tied
    rows[7] = rng.normal(0, 0.01, V).astype(np.float32)
    k = np.array([1, 5, 300, 512, 20001, 3, 0, 0], np.int32)
    p = np.array([1.0, 0.9, 0.5, 1.0, 0.99, 0.2, 0.9, 0.99], np.float32)
    T = np.full(n, 0.8, np.float32)
    if dtype == "bf16":
        rows = W.bf16_rne_bits(rows)
    check(o, dev, rows, dtype == "bf16", k, p, T, f"top ties {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_top_p_alone_sampled_reference(o, dev, dtype):
    """Top-p alone sums the row's mass on the max of a quarter-row sample (the
    16-byte vectors of every fourth block of 512), rescaled to the row max.
    Elements 4096..8191 lie outside that sample for both dtypes here.  Row 0:
    a spike 200 above the sample (the weights overflow: exact fallback); row 1:
    every sampled logit -inf (no finite reference: the unfused passes); row 2:
    the max outside the sample (the rescale); row 3: an ordinary row."""
    rng = np.random.default_rng(17)
    n, V = 4, 30000
    rows = rng.normal(0, 1, (n, V)).astype(np.float32)
    rows[0, 5000] = 200.0
    rows[1, :4096] = -np.inf
    rows[1, 8192:] = -np.inf
    rows[2, 6000] = 6.0
    p = np.array([0.9, 0.9, 0.8, 0.95], np.float32)
    T = np.full(n, 0.7, np.float32)
    if dtype == "bf16":
        rows = W.bf16_rne_bits(rows)
    check(o, dev, rows, dtype == "bf16", None, p, T, f"sampled reference {dtype}")
