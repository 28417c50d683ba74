"""The GPU's committed tokens are distributed as the target distribution p
(tutorial page "5.1 投机解码核心原理", section 4: the output of speculative
sampling follows p exactly), checked without the oracle: 10^6 trials of one
position (gamma = 1) on V <= 8 rows, a chi-square test of the first committed
token against p computed in fp64 on the host.

Each call verifies B = 4096 requests that share the same target and draft
rows, with independent uniforms and draft tokens y ~ q drawn on the host; the
first committed token is y when position 0 is accepted, else the draw from
the residual.  A rule that resampled from p after a reject, inverted the
acceptance ratio or drew from [q - p]_+ would move the histogram by far more
than the test's power (see the planted mistakes of the oracle pins: the same
rules give [0.44, 0.42, 0.14] instead of p on the tutorial's worked example).
"""
import numpy as np
import pytest
from scipy import stats

pytestmark = pytest.mark.gpu

TRIALS = 1_000_000
B = 4096


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    return torch.device("cuda:0")


def softmax64(x, T):
    z = np.asarray(x, np.float64) / T
    z = np.exp(z - z.max())
    return z / z.sum()


def first_tokens(dev, xt, xd, T, mode, seed):
    """TRIALS first committed tokens of one position (gamma = 1)."""
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    V = len(xt)
    rng = np.random.default_rng(seed)
    q = softmax64(xd, T) if mode == "sample" else None
    tgt = torch.tensor(np.broadcast_to(np.stack([xt, xt]).astype(np.float32), (B, 2, V)).copy(), device=dev)
    drf = torch.tensor(np.broadcast_to(np.asarray(xd, np.float32)[None], (B, 1, V)).copy(), device=dev) \
        if mode == "sample" else None
    gamma = torch.ones(B, dtype=torch.int32, device=dev)
    temp = torch.full((B,), T, dtype=torch.float32, device=dev)
    counts = np.zeros(V, np.int64)
    n = 0
    while n < TRIALS:
        if mode == "sample":
            y = rng.choice(V, size=B, p=q).astype(np.int32)
        else:   # one-hot q: the draft token is any fixed token; use the draft's argmax
            y = np.full(B, int(np.argmax(xd)), np.int32)
        u = (rng.integers(0, 1 << 24, size=(B, 2)) * 2.0 ** -24).astype(np.float32)
        yt = torch.from_numpy(y[:, None]).to(dev)
        ut = torch.from_numpy(u).to(dev)
        if mode == "sample":
            r = sv.verify_sample(tgt, drf, yt, gamma, temp, ut, signals=False)
        else:
            r = sv.verify_onehot(tgt, yt, gamma, temp, ut)
        tok = r["tokens"][:, 0].cpu().numpy()
        assert (r["status"].cpu().numpy() & ~16 & ~8 == 0).all()
        m = min(B, TRIALS - n)
        counts += np.bincount(tok[:m], minlength=V)
        n += m
    return counts


@pytest.mark.parametrize("case", [
    # the tutorial's worked example (section 7), as logits
    dict(p=[0.6, 0.3, 0.1], q=[0.2, 0.5, 0.3], T=1.0, mode="sample"),
    # random rows at V = 8 and a temperature
    dict(seed=3, V=8, T=0.7, mode="sample"),
    # one-hot q (section 3.3): accept with p(y), else p with y removed
    dict(seed=4, V=6, T=1.0, mode="onehot"),
])
def test_first_token_is_distributed_as_p(dev, case):
    if "p" in case:
        xt, xd = np.log(case["p"]), np.log(case["q"])
    else:
        rng = np.random.default_rng(case["seed"])
        xt = rng.normal(0, 1.5, case["V"])
        xd = xt + rng.normal(0, 1.0, case["V"])
    T = case["T"]
    counts = first_tokens(dev, xt, xd, T, case["mode"], seed=1234 + case.get("seed", 0))
    p = softmax64(np.asarray(xt, np.float32), np.float32(T))
    expected = p * counts.sum()
    chi2, pval = stats.chisquare(counts, expected)
    assert pval > 1e-4, (counts, expected, chi2, pval)
