"""The disagreement budget on large samples: at least 10^5 decisions per
full-size workload, GPU against the fp64 oracle, through the C ABI.

Each workload runs on several seeded logit sets, with fresh draft tokens
and uniforms every round (see parity.large_sample).  Every decision whose
oracle margin is at least 1e-5 must match exactly; a flagged near tie may
differ only to the neighbouring bucket; and the decisions that differ must
stay under 0.01 % of all decisions (acceptance tests plus final draws).
The tally (decisions, flagged near ties, disagreements) is printed.
"""
import pytest

import oracle as O
import parity as PT

pytestmark = pytest.mark.gpu

MIN_DECISIONS = 100_000


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


# (workload, call kind, logit sets, rounds per set): sized for >= 10^5
# decisions at the acceptance rates of the seeded workloads
CASES = [
    ("c2", "greedy", 8, 56),
    ("c3", "sample", 12, 110),
    ("c4", "onehot", 16, 50),
    ("c5", "sample", 6, 24),
    ("m", "sample", 10, 64),
]


@pytest.mark.parametrize("name,mode,n_sets,rounds", CASES, ids=[c[0] for c in CASES])
def test_disagreement_budget(o, dev, name, mode, n_sets, rounds):
    t = PT.large_sample(o, dev, name, mode, n_sets, rounds)
    print(f"{name} {mode}: {t}")
    assert t.decisions >= MIN_DECISIONS, t
    if mode == "greedy":
        assert t.disagree == 0, t          # integer work: bit-exact
    assert t.within_budget(), t
