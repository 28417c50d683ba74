"""The C-ABI library: it builds, loads, exports every declared entry point and
rejects bad arguments on the host (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verification_26_gb300 import build
    import speculative_decoding_verification_26_gb300 as sv
    build.build()
    return sv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_\w+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ["spec_verify_greedy", "spec_verify_sample", "spec_verify_onehot", "spec_draft_signals",
              "spec_workspace_bytes"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in declared_functions():
        assert hasattr(L, n), f"{n} declared in spec_verify.h but not exported"


def test_workspace_bytes(L):
    assert L.spec_workspace_bytes(0, 7, 151936) == 0
    assert L.spec_workspace_bytes(64, 32, 151936) == 0
    assert L.spec_workspace_bytes(64, 7, 1) == 0
    # sizes whose queue capacities would not fit in 32 bits are refused, not
    # wrapped (their logits could not exist on a device anyway)
    assert L.spec_workspace_bytes(65535, 0, (1 << 28) - 1) == 0
    a = L.spec_workspace_bytes(64, 7, 151936)
    b = L.spec_workspace_bytes(128, 7, 151936)
    assert 0 < a < b
    assert a % 256 == 0


def test_status_strings(L):
    assert L.spec_status_string(0) == b"ok"
    assert b"workspace" in L.spec_status_string(2)
    assert b"uniform" in L.spec_request_status_string(128)


def test_host_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    fake = P(0x7f0000000000)       # never dereferenced: the host checks fail first
    ws = L.spec_workspace_bytes(4, 4, 1024)
    # null target
    assert L.spec_verify_greedy(None, 0, 4, 4, 1024, fake, None, fake, fake, None, fake, ws, None) == 1
    # bad dtype / sizes
    assert L.spec_verify_greedy(fake, 7, 4, 4, 1024, fake, None, fake, fake, None, fake, ws, None) == 1
    assert L.spec_verify_greedy(fake, 0, 0, 4, 1024, fake, None, fake, fake, None, fake, ws, None) == 1
    assert L.spec_verify_greedy(fake, 0, 4, 40, 1024, fake, None, fake, fake, None, fake, ws, None) == 1
    assert L.spec_verify_greedy(fake, 0, 4, 4, 1, fake, None, fake, fake, None, fake, ws, None) == 1
    # workspace missing / too small
    assert L.spec_verify_greedy(fake, 0, 4, 4, 1024, fake, None, fake, fake, None, None, ws, None) == 2
    assert L.spec_verify_greedy(fake, 0, 4, 4, 1024, fake, None, fake, fake, None, fake, ws - 1, None) == 2
    # misaligned logits / workspace
    assert L.spec_verify_greedy(P(0x7f0000000001), 1, 4, 4, 1024, fake, None, fake, fake, None, fake, ws,
                                None) == 1
    assert L.spec_verify_greedy(fake, 0, 4, 4, 1024, fake, None, fake, fake, None, P(0x7f0000000010), ws,
                                None) == 1
    # sample: missing draft, temperature, uniforms
    args = [fake, fake, 1, 4, 4, 1024, fake, None, fake, fake, fake, fake, None, None, None, fake, ws, None]
    for idx in (1, 8, 9):
        a = list(args)
        a[idx] = None
        assert L.spec_verify_sample(*a) == 1
    # one-hot without uniforms, signals without the signals output
    assert L.spec_verify_onehot(fake, 1, 4, 4, 1024, fake, None, fake, None, fake, fake, None, None, fake, ws,
                                None) == 1
    assert L.spec_draft_signals(fake, 1, 4, 4, 1024, None, fake, None, None, None, fake, ws, None) == 1


def test_divergence_stats_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    fake = P(0x7f0000000000)       # never dereferenced: the host checks fail first
    # no temperature, no stats, no draft, bad dtype, bad sizes, misaligned logits
    assert L.spec_divergence_stats(fake, fake, 1, 4, 4, 1024, None, None, fake, None, None) == 1
    assert L.spec_divergence_stats(fake, fake, 1, 4, 4, 1024, None, fake, None, None, None) == 1
    assert L.spec_divergence_stats(fake, None, 1, 4, 4, 1024, None, fake, fake, None, None) == 1
    assert L.spec_divergence_stats(fake, fake, 5, 4, 4, 1024, None, fake, fake, None, None) == 1
    assert L.spec_divergence_stats(fake, fake, 1, 0, 4, 1024, None, fake, fake, None, None) == 1
    assert L.spec_divergence_stats(P(0x7f0000000001), fake, 1, 4, 4, 1024, None, fake, fake, None, None) == 1


def test_gamma_select_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    fake = P(0x7f0000000000)       # never dereferenced: the host checks fail first
    assert L.spec_gamma_select(None, None, fake, 4, fake, None, None) == 1
    assert L.spec_gamma_select(fake, None, None, 4, fake, None, None) == 1
    assert L.spec_gamma_select(fake, None, fake, 4, None, None, None) == 1
    assert L.spec_gamma_select(fake, None, fake, 0, fake, None, None) == 1
    assert L.spec_gamma_select(P(0x7f0000000004), None, fake, 4, fake, None, None) == 1   # signals not 16-byte aligned


def test_filter_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    fake = P(0x7f0000000000)       # never dereferenced: the host checks fail first
    assert L.spec_filter_top_k_top_p(None, 1, 4, 1024, None, None, None, None, None) == 1
    assert L.spec_filter_top_k_top_p(fake, 3, 4, 1024, None, None, None, None, None) == 1
    assert L.spec_filter_top_k_top_p(fake, 1, 0, 1024, None, None, None, None, None) == 1
    assert L.spec_filter_top_k_top_p(fake, 1, 4, 1, None, None, None, None, None) == 1
    assert L.spec_filter_top_k_top_p(P(0x7f0000000001), 1, 4, 1024, None, None, None, None, None) == 1
