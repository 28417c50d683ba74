"""GPU path against the fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest

import oracle as O
import parity as PT
from speculative_decoding_verification_26_gb300 import workloads as W

pytestmark = pytest.mark.gpu


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


def _run(o, dev, name, mode, rounds=1, tally=None, **kw):
    tally = tally or PT.Tally()
    for r in range(rounds):
        wl = PT.make_workload(o, name, r, **kw)
        g = PT.run_gpu(mode, wl, dev)
        ref = PT.run_oracle(o, mode, wl)
        PT.compare(o, mode, wl, g, ref, tally)
    return tally


# ---- small case (several tiles and a ragged tail are covered below) ----------

@pytest.mark.parametrize("mode", ["greedy", "sample", "onehot"])
def test_c1_small_fp32(o, dev, mode):
    t = _run(o, dev, "c1", mode, rounds=8)
    assert t.disagree == 0, t


@pytest.mark.parametrize("V", [2, 3, 7, 1000, 1001, 4093, 16385, 40000, 65537])
@pytest.mark.parametrize("dtype", [W.BF16, W.F32])
@pytest.mark.parametrize("mode", ["greedy", "sample", "onehot"])
def test_ragged_vocab(o, dev, V, dtype, mode):
    """Vocabularies that are not multiples of the vector width or of a chunk:
    unaligned rows, scalar heads/tails, several chunks plus a ragged one."""
    over = {"dtype": dtype, "zipf": True, "sigma_d": 1.0, "T": 0.8, "draft": "sample_q"}
    t = PT.Tally()
    for r in range(2):
        wl = PT.make_workload(o, "c3", r, B=5, G=3, V=V, overrides=over)
        g = PT.run_gpu(mode, wl, dev)
        ref = PT.run_oracle(o, mode, wl)
        PT.compare(o, mode, wl, g, ref, t)
    assert t.disagree == 0, t


# ---- the workloads at full size (signals compared with the oracle's every
# round; the disagreement budget over 10^5 decisions is in
# test_gpu_parity_large.py) ------------------------------------------------------

def test_c2_greedy_full(o, dev):
    t = _run(o, dev, "c2", "greedy", rounds=2)
    assert t.disagree == 0


@pytest.mark.parametrize("name,mode,rounds", [("c3", "sample", 2), ("c4", "onehot", 2), ("c5", "sample", 1),
                                              ("m", "sample", 2)])
def test_full_size(o, dev, name, mode, rounds):
    t = _run(o, dev, name, mode, rounds=rounds)
    print(name, t)
    assert t.within_budget(), t


# ---- kernel branches and precision regimes ---------------------------------------

@pytest.mark.parametrize("dtype,V,B,G", [(W.F32, 151936, 4, 3), (W.BF16, 300000, 3, 3), (W.BF16, 300001, 3, 2),
                                         (W.BF16, 600000, 2, 2), (W.F32, 300003, 2, 2)])
@pytest.mark.parametrize("mode", ["greedy", "sample", "onehot"])
def test_many_chunks_and_slices(o, dev, dtype, V, B, G, mode):
    """Rows of more than 8 chunks (the owner's one-row merges) and draws over
    more than 32 slices (the two-level slice search); V = 600000 bf16 and
    V = 300003 fp32 exceed 16 chunks (one row per merge in every mode)."""
    over = {"dtype": dtype, "zipf": True, "sigma_d": 1.0, "T": 0.8, "draft": "sample_q"}
    t = PT.Tally()
    for r in range(2):
        wl = PT.make_workload(o, "c3", 30 + r, B=B, G=G, V=V, overrides=over)
        PT.compare(o, mode, wl, PT.run_gpu(mode, wl, dev), PT.run_oracle(o, mode, wl), t)
    assert t.within_budget(), t


@pytest.mark.parametrize("name", ["c3", "m"])
@pytest.mark.parametrize("over", [{"shift": 64.0}, {"T": 0.2}, {"shift": 64.0, "T": 0.2}],
                         ids=["shift64", "T0.2", "shift64_T0.2"])
def test_offset_logits_and_low_temperature(o, dev, name, over):
    """Softmax ignores a constant offset, fp32 exponents do not: every logit
    shifted by +64 (|m c| ~ 160, 550 at T = 0.2), and the lowest temperature
    of the pages' range.  Probabilities, signals and decisions must still
    match the oracle within the contract."""
    t = PT.Tally()
    for r in range(2):
        wl = PT.make_workload(o, name, 40 + r, overrides=over)
        g = PT.run_gpu("sample", wl, dev)
        PT.compare(o, "sample", wl, g, PT.run_oracle(o, "sample", wl), t)
        wl1 = PT.make_workload(o, name, 40 + r, overrides=dict(over, draft="noisy_argmax", noise=2.0))
        PT.compare(o, "onehot", wl1, PT.run_gpu("onehot", wl1, dev), PT.run_oracle(o, "onehot", wl1), t)
    print(name, over, t)
    assert t.within_budget(), t


def test_timeout_path(o, dev):
    """Waits that give up: with the wait limit lowered to one cycle, every
    request comes back either settled exactly as the oracle settles it or
    void with SPEC_ST_TIMEOUT (accept_len 0, tokens -1, signals NaN), and
    the call returns; a normal call on the same workspace right after it
    matches the oracle."""
    import numpy as np
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    wl = PT.make_workload(o, "m", 45)
    wl_g = PT.make_workload(o, "c2", 45, B=64)
    wl_1 = PT.make_workload(o, "c4", 45)
    B, G, V = wl.B, wl.G, wl.V
    ws = torch.empty(max(sv.workspace_bytes(64, 8, V), sv.workspace_bytes(B, G, V)), dtype=torch.uint8, device=dev)
    ref = {"sample": PT.run_oracle(o, "sample", wl), "greedy": PT.run_oracle(o, "greedy", wl_g),
           "onehot": PT.run_oracle(o, "onehot", wl_1)}
    wls = {"sample": wl, "greedy": wl_g, "onehot": wl_1}
    got = {}
    sv.set_wait_limit(1)
    try:
        for mode in ("sample", "greedy", "onehot"):
            got[mode] = PT.run_gpu(mode, wls[mode], dev, ws=ws)
        sig = sv.draft_signals(PT.logits_dev(wl, "draft", dev), PT.to_dev(wl.gamma, dev),
                               PT.to_dev(wl.temperature, dev), ws=ws)
        torch.cuda.synchronize()
    finally:
        sv.set_wait_limit(0)
    n_timeout = 0
    for mode, g in got.items():
        w, r = wls[mode], ref[mode]
        to = (g["status"] & sv._lib.ST_TIMEOUT) != 0
        n_timeout += int(to.sum())
        assert np.all(g["status"][to] == sv._lib.ST_TIMEOUT), mode
        assert np.all(g["accept_len"][to] == 0) and np.all(g["tokens"][to] == -1), mode
        if "signals" in g:
            assert np.all(np.isnan(g["signals"][to])), mode
        ok = ~to
        np.testing.assert_array_equal(g["status"][ok], r["status"][ok], err_msg=mode)
        np.testing.assert_array_equal(g["accept_len"][ok], r["accept_len"][ok], err_msg=mode)
        np.testing.assert_array_equal(g["tokens"][ok], r["tokens"][ok], err_msg=mode)
    s_st = sig["status"].cpu().numpy()
    n_timeout += int(((s_st & sv._lib.ST_TIMEOUT) != 0).sum())
    assert n_timeout > 0, "a one-cycle wait limit timed nothing out"
    # the same workspace, default limit: every call matches the oracle again
    for mode in ("sample", "greedy", "onehot"):
        PT.compare(o, mode, wls[mode], PT.run_gpu(mode, wls[mode], dev, ws=ws), ref[mode], PT.Tally())


# ---- edge cases ---------------------------------------------------------------

def test_gamma_zero_and_mixed(o, dev):
    """gamma_b = 0 (a plain draw from p_0) mixed with full-length requests."""
    wl = PT.make_workload(o, "c3", 3, B=12, G=4, V=3000)
    wl.gamma[:] = np.array([0, 1, 2, 3, 4, 0, 4, 4, 1, 0, 2, 3], np.int32)
    for mode in ["greedy", "sample", "onehot"]:
        g = PT.run_gpu(mode, wl, dev)
        PT.compare(o, mode, wl, g, PT.run_oracle(o, mode, wl), PT.Tally())


def test_G_zero(o, dev):
    wl = PT.make_workload(o, "c3", 4, B=6, G=0, V=5000)
    for mode in ["greedy", "sample", "onehot"]:
        g = PT.run_gpu(mode, wl, dev)
        PT.compare(o, mode, wl, g, PT.run_oracle(o, mode, wl), PT.Tally())


def test_p_equals_q_never_rejects(o, dev):
    wl = PT.make_workload(o, "c3", 5, B=16, G=6, V=20000)
    wl.draft = np.ascontiguousarray(wl.target[:, :6, :])
    W.resolve_draft_tokens(wl, PT.oracle_argmax(o))
    g = PT.run_gpu("sample", wl, dev)
    assert np.all(g["accept_len"] == 6)
    PT.compare(o, "sample", wl, g, PT.run_oracle(o, "sample", wl), PT.Tally())


def test_greedy_ties_lowest_index(o, dev):
    """Integer-valued logits: many equal maxima; the lowest index must win."""
    rng = np.random.default_rng(9)
    wl = PT.make_workload(o, "c1", 0, B=32, G=5, V=3000)
    wl.target = rng.integers(-4, 4, wl.target.shape).astype(np.float32)
    am = o.run(O.GREEDY, target=wl.target.reshape(-1, 1, 3000), G=0)["tokens"][:, 0].reshape(32, 6)
    wl.draft_tokens = np.ascontiguousarray(am[:, :5]).astype(np.int32)
    flip = rng.random((32, 5)) < 0.2
    wl.draft_tokens[flip] = rng.integers(0, 3000, flip.sum())
    g = PT.run_gpu("greedy", wl, dev)
    PT.compare(o, "greedy", wl, g, PT.run_oracle(o, "greedy", wl), PT.Tally())


def test_bad_inputs_are_reported_per_request(o, dev):
    wl = PT.make_workload(o, "c3", 6, B=10, G=3, V=4000, overrides={"dtype": W.F32})
    wl.target = wl.target.copy()
    wl.target[0, 0, 17] = np.nan                      # NaN in a row that is read
    wl.target[1, 0, 5] = np.inf                       # +inf
    wl.target[2, 0, :] = -np.inf                      # no finite max
    wl.target[3, 0, 100:200] = -np.inf                # masked tokens: fine
    wl.draft_tokens = wl.draft_tokens.copy()
    wl.draft_tokens[4, 0] = 4000                      # bad token
    wl.gamma = wl.gamma.copy()
    wl.gamma[5] = 4                                   # bad gamma
    wl.temperature = wl.temperature.copy()
    wl.temperature[6] = 0.0                           # bad temperature
    wl.uniforms = wl.uniforms.copy()
    wl.uniforms[7, 3] = 1.0                           # bad draw uniform
    wl.target[8, 3, 9] = np.nan                       # after gamma: never read
    for mode in ["greedy", "sample", "onehot"]:
        g = PT.run_gpu(mode, wl, dev)
        ref = PT.run_oracle(o, mode, wl)
        PT.compare(o, mode, wl, g, ref, PT.Tally())
        assert ref["status"][0] == O.ST_NONFINITE


def test_repeatable(o, dev):
    wl = PT.make_workload(o, "m", 0, B=16)
    a = PT.run_gpu("sample", wl, dev)
    b = PT.run_gpu("sample", wl, dev)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def test_more_requests_than_ctas(o, dev):
    """B above the grid (2 CTAs per SM on 152 SMs): each owner warp serves
    several requests, one after the other; past 4096 requests the plan
    kernel reads the request checks back from global memory."""
    for B, G, V in [(700, 3, 1500), (4200, 1, 200)]:
        wl = PT.make_workload(o, "c3", 21, B=B, G=G, V=V)
        for mode in ["greedy", "sample", "onehot"]:
            PT.compare(o, mode, wl, PT.run_gpu(mode, wl, dev), PT.run_oracle(o, mode, wl), PT.Tally())


def test_max_gamma_and_long_acceptance(o, dev):
    """G = 31, the largest the boundary allows, with a draft close to the
    target so that most requests accept deep into the block (every lane of
    the owner's per-position values is used)."""
    wl = PT.make_workload(o, "c3", 22, B=12, G=31, V=2500, overrides=dict(sigma_d=0.02))
    # (draft tokens past a request's gamma are never read)
    wl.gamma[:] = np.array([31, 31, 30, 0, 1, 16, 31, 29, 31, 7, 31, 2], np.int32)
    for mode in ["greedy", "sample", "onehot"]:
        t = PT.Tally()
        PT.compare(o, mode, wl, PT.run_gpu(mode, wl, dev), PT.run_oracle(o, mode, wl), t)
    ref = PT.run_oracle(o, "sample", wl)
    assert int(ref["accept_len"].max()) >= 20          # deep positions are exercised


def test_single_request(o, dev):
    wl = PT.make_workload(o, "m", 23, B=1)
    for mode in ["greedy", "sample", "onehot"]:
        PT.compare(o, mode, wl, PT.run_gpu(mode, wl, dev), PT.run_oracle(o, mode, wl), PT.Tally())


def test_stale_words_in_reused_memory(o, dev):
    """Memory a workspace takes over may hold small integers left by earlier
    tensors or calls.  Here every word after the header is overwritten with a
    value whose low half is 8 * (e + 1) (+ 0..7), the unscrambled tag an epoch
    counted per workspace would use on the next call, and a payload of 1 (in range as a
    request, slice, item or chunk index, so a word taken by mistake reads no
    memory out of bounds); the next call must not take any of them for its
    own partials, queue entries or draw words (tags are scrambled and epochs
    unique on the device)."""
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    wl = PT.make_workload(o, "c3", 11, B=24)
    B, G, V = wl.B, wl.G, wl.V
    ws = torch.empty(sv.workspace_bytes(B, G, V), dtype=torch.uint8, device=dev)
    args = (PT.logits_dev(wl, "target", dev), PT.logits_dev(wl, "draft", dev), PT.to_dev(wl.draft_tokens, dev),
            PT.to_dev(wl.gamma, dev), PT.to_dev(wl.temperature, dev), PT.to_dev(wl.uniforms, dev))
    ref = PT.run_oracle(o, "sample", wl)
    for rep in range(3):
        sv.verify_sample(*args, signals=True, accept_prob=True, ws=ws)
        torch.cuda.synchronize()
        # header: 8 counters of 128 bytes; the epoch is word 5 of the last one
        epoch = int(ws[7 * 128 + 4 * 5: 7 * 128 + 4 * 6].view(torch.int32).item())
        words = ws[1024:(ws.numel() // 8) * 8].view(torch.int64)
        idx = torch.arange(words.numel(), device=dev, dtype=torch.int64)
        words.copy_((1 << 32) | (8 * (epoch + 1) + (idx % 8)))
        r = sv.verify_sample(*args, signals=True, accept_prob=True, ws=ws)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in r.items()}
        PT.compare(o, "sample", wl, g, ref, PT.Tally())


def test_draft_signals_standalone(o, dev):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    for name in ["c1", "c5"]:
        wl = PT.make_workload(o, name, 7, B=min(W.CONFIGS[name]["B"], 48))
        r = sv.draft_signals(PT.logits_dev(wl, "draft", dev), PT.to_dev(wl.gamma, dev),
                             PT.to_dev(wl.temperature, dev), row_signals=True)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy().astype(np.float64) for k, v in r.items()}
        ref = o.draft_signals(wl.draft, wl.gamma, wl.temperature, want_row_signals=True)
        for key in ("signals", "row_signals"):
            PT.compare_signals(g[key], ref[key], f"{name} {key}")
        np.testing.assert_array_equal(g["status"], ref["status"])
