"""spec_divergence_stats against the fp64 oracle (oracle_divergence), element
by element, through the C ABI.

The five statistics of each position (A = sum min(p, q), L1 = sum |p - q|,
KL(p||q), KL(q||p), H(p), bits) must match within 1e-5 relative, with
absolute floors from the fp32 arithmetic: each token's probability carries
~3e-7 relative error (ex2.approx, one product by 1/S), so a sum of
non-negative terms that add to at most 1 (A, L1) is off by at most ~1e-6
absolute however small it is, and the KL and entropy sums, whose terms carry
a log2 factor of at most ~60 bits on these rows, by ~2e-6 bits.  Infinite
values (a draft zero under target mass) must be infinite on both sides, NaN
positions NaN on both sides, and the status words equal.
"""
import numpy as np
import pytest

import oracle as O
import parity as PT
from speculative_decoding_verification_26_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL = 1e-5
FLOOR = np.array([1e-6, 2e-6, 2e-6, 2e-6, 2e-6])   # A, L1, KL(p||q), KL(q||p), H(p)


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def o():
    return O.load()


def gpu_stats(dev, target, draft, gamma, temperature, bf16):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    t = PT.to_dev(target.view(np.int16) if bf16 else target, dev, bf16=bf16)
    d = PT.to_dev(draft.view(np.int16) if bf16 else draft, dev, bf16=bf16)
    g = torch.from_numpy(np.ascontiguousarray(gamma, np.int32)).to(dev)
    T = torch.from_numpy(np.ascontiguousarray(temperature, np.float32)).to(dev)
    r = sv.divergence_stats(t, d, g, T)
    torch.cuda.synchronize()
    return r["stats"].cpu().numpy().astype(np.float64), r["status"].cpu().numpy()


def compare(gs, gst, os_, ost, what):
    assert np.array_equal(gst, ost), (what, gst, ost)
    nan_g, nan_o = np.isnan(gs), np.isnan(os_)
    assert np.array_equal(nan_g, nan_o), (what, np.argwhere(nan_g != nan_o)[:5])
    inf_g, inf_o = np.isinf(gs), np.isinf(os_)
    assert np.array_equal(inf_g, inf_o), (what, np.argwhere(inf_g != inf_o)[:5])
    fin = np.isfinite(os_)
    err = np.where(fin, np.abs(np.where(fin, gs, 0.0) - np.where(fin, os_, 0.0)), 0.0)   # inf - inf unasked
    tol = REL * np.abs(np.where(fin, os_, 0.0)) + FLOOR
    bad = fin & ~(err <= tol)
    assert not bad.any(), (what, np.argwhere(bad)[:5], gs[bad][:5], os_[bad][:5])
    return int(fin.sum())


def run_case(o, dev, wl, what):
    bf16 = wl.dtype == W.BF16
    res = o.divergence_stats(wl.target, wl.draft, wl.gamma, wl.temperature)
    gs, gst = gpu_stats(dev, wl.target, wl.draft, wl.gamma, wl.temperature, bf16)
    return compare(gs, gst, res["stats"], res["status"], what)


@pytest.mark.parametrize("name", ["c1", "c3", "m"])
def test_configs(o, dev, name):
    wl = W.make(name, 0)
    n = run_case(o, dev, wl, name)
    assert n > 0


def test_ragged_gamma_full_size(o, dev):
    wl = W.make("c5", 0, B=48)              # gamma_b in {2, 4, 6, 8}
    assert len(set(wl.gamma.tolist())) > 1
    run_case(o, dev, wl, "c5 ragged")


@pytest.mark.parametrize("V", [2, 7, 1001, 4093, 65537, 151936])
@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_vocab_sizes(o, dev, V, dtype):
    wl = W.make("c3", 1, B=3, G=3, V=V, overrides={"dtype": dtype})
    run_case(o, dev, wl, f"V={V} {dtype}")


def test_special_rows(o, dev):
    rng = np.random.default_rng(5)
    B, G, V = 5, 2, 1000
    tgt = rng.normal(0, 3, (B, G + 1, V)).astype(np.float32)
    drf = (tgt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    drf[0] = tgt[0, :G]                      # p = q: A = 1, L1 = 0, KL = 0
    drf[1, 0, 17] = -np.inf                  # a draft zero under target mass: KL(p||q) = inf
    drf[2, 1, 3] = np.nan                    # a bad row: that position NaN, status NONFINITE
    tgt[3, 0, :] = -np.inf                   # no finite max
    gamma = np.array([2, 2, 2, 2, 3], np.int32)   # request 4: bad gamma
    T = np.array([1.0, 0.7, 1.3, 1.0, 1.0], np.float32)
    res = o.divergence_stats(tgt, drf, gamma, T)
    gs, gst = gpu_stats(dev, tgt, drf, gamma, T, False)
    compare(gs, gst, res["stats"], res["status"], "special rows")
    assert gst[2] == 1 and gst[3] == 1 and gst[4] == 4
    assert np.isinf(gs[1, 0, 2]) and np.isfinite(gs[1, 0, 3])
    assert abs(gs[0, 0, 0] - 1) < 1e-6 and gs[0, 0, 1] == 0 and gs[0, 0, 2] == 0 and gs[0, 0, 3] == 0


def test_bad_temperature_and_gamma_zero(o, dev):
    wl = W.make("c1", 2)
    wl.temperature[1] = 0.0
    wl.gamma[2] = 0
    run_case(o, dev, wl, "T=0, gamma=0")


def test_repeatable(dev):
    wl = W.make("c3", 2, B=8)
    a = gpu_stats(dev, wl.target, wl.draft, wl.gamma, wl.temperature, True)[0]
    b = gpu_stats(dev, wl.target, wl.draft, wl.gamma, wl.temperature, True)[0]
    assert np.array_equal(a, b, equal_nan=True)
