"""Cross-call state: 200 bench-workload calls on one workspace, interleaved
with greedy, one-hot and signals-only calls of other sizes on the same
memory.  Every call must give the oracle's result, and repeats of the same
inputs must be bit-identical: a word left by an earlier call (a chunk
partial, a queue entry, a draw word) taken for a current one, or a
half-published multi-word value, would show up as a changed output.
"""
import numpy as np
import pytest

import oracle as O
import parity as PT

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    return torch.device("cuda:0")


def test_interleaved_calls_on_one_workspace(dev):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    o = O.load()
    jobs = [
        ("sample", PT.make_workload(o, "m", 60)),
        ("sample", PT.make_workload(o, "m", 61)),
        ("greedy", PT.make_workload(o, "c2", 62, B=48)),
        ("onehot", PT.make_workload(o, "c4", 63, B=40)),
        ("signals", PT.make_workload(o, "c5", 64, B=96)),
        ("sample", PT.make_workload(o, "c3", 65, B=20, G=3, V=7001)),
    ]
    nbytes = max(sv.workspace_bytes(w.B, w.G, w.V) for _, w in jobs)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dev_logits = [(PT.logits_dev(w, "target", dev), PT.logits_dev(w, "draft", dev)) for _, w in jobs]

    def call(j):
        mode, w = jobs[j]
        if mode == "signals":
            r = sv.draft_signals(dev_logits[j][1], PT.to_dev(w.gamma, dev), PT.to_dev(w.temperature, dev),
                                 row_signals=True, ws=ws)
            torch.cuda.synchronize()
            return {k: v.cpu().numpy() for k, v in r.items()}
        return PT.run_gpu(mode, w, dev, logits=dev_logits[j], ws=ws)

    first = {}
    for j, (mode, w) in enumerate(jobs):        # each call once against the oracle
        g = call(j)
        if mode == "signals":
            ref = o.draft_signals(w.draft, w.gamma, w.temperature, want_row_signals=True)
            for key in ("signals", "row_signals"):
                PT.compare_signals(g[key], ref[key], key)
            np.testing.assert_array_equal(g["status"], ref["status"])
        else:
            t = PT.Tally()
            PT.compare(o, mode, w, g, PT.run_oracle(o, mode, w), t)
            assert t.within_budget(), t
        first[j] = g
    others = [2, 3, 4, 5]
    for n in range(200):                        # 200 bench-workload calls, others in between
        for j in (n % 2, others[n % len(others)]):
            g = call(j)
            for key, v in first[j].items():
                assert np.array_equal(g[key], v, equal_nan=True), (n, jobs[j][0], key)
