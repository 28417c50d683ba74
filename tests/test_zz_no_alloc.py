"""spec_verify_sample_static: the entry point that allocates nothing.

It must give exactly what spec_verify_sample gives with a caller workspace,
on two calls in a row (the second call finds the first call's leftovers in
the library's static scratch).  This file is collected last so that it also
runs after every other GPU test has used the library.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import parity as PT


def _static_fn():
    import speculative_decoding_verification_26_gb300 as sv
    f = sv.lib().spec_verify_sample_static
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, I, I, I, I, P, P, P, P, P, P, P, P, P, P]
    f.restype = I
    return f


def test_static_scratch_rejects_oversize_before_touching_the_device():
    # The size checks come first and return before any CUDA call, so dummy
    # pointers are never dereferenced.
    import speculative_decoding_verification_26_gb300 as sv
    f = _static_fn()
    d = ctypes.c_void_p(256)
    big = (1024, 8, 151936)
    assert sv.workspace_bytes(*big) > sv.STATIC_WORKSPACE_BYTES
    args = lambda B, G, V: (d, d, sv.BF16, B, G, V, d, d, d, d, d, d, d, d, d, None)
    assert f(*args(*big)) == 2          # SPEC_ERR_WORKSPACE
    assert f(*args(0, 7, 151936)) == 1  # SPEC_ERR_INVALID_ARG (B < 1)
    # the largest request count that fits at G = 8, V = 151936 (the header
    # states it); the B = 256 ragged-gamma workload fits
    bmax = max(B for B in range(1, 2048) if sv.workspace_bytes(B, 8, 151936) <= sv.STATIC_WORKSPACE_BYTES)
    assert bmax >= 256
    assert f(*args(bmax + 1, 8, 151936)) == 2


@pytest.fixture(scope="module")
def dev():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    return torch.device("cuda:0")


def _inputs(wl, dev):
    return (PT.logits_dev(wl, "target", dev), PT.logits_dev(wl, "draft", dev), PT.to_dev(wl.draft_tokens, dev),
            PT.to_dev(wl.gamma, dev), PT.to_dev(wl.temperature, dev), PT.to_dev(wl.uniforms, dev))


def _same(a, b, what):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, what
    if a.dtype.kind == "f":
        assert np.array_equal(a, b, equal_nan=True), what
    else:
        assert np.array_equal(a, b), what


@pytest.mark.gpu
def test_static_matches_caller_workspace_on_two_calls_in_a_row(dev):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    o = O.load()
    # two different workloads, the second with a ragged gamma and B = 256
    wls = [PT.make_workload(o, "c3", 0), PT.make_workload(o, "c5", 1)]
    ins = [_inputs(wl, dev) for wl in wls]
    got = []
    for x in ins:                         # two static calls back to back
        got.append(sv.verify_sample_static(*x, signals=True, accept_prob=True))
    torch.cuda.synchronize()
    for x, g in zip(ins, got):
        ref = sv.verify_sample(*x, signals=True, accept_prob=True)
        torch.cuda.synchronize()
        for key in ("accept_len", "tokens", "status", "signals", "accept_prob"):
            _same(g[key].cpu().numpy(), ref[key].cpu().numpy(), key)
        # no request failed (guarded draws and zero residual mass are informational bits)
        assert int((g["status"] & ~(sv._lib.ST_GUARDED | sv._lib.ST_ZERO_RESIDUAL)).abs().sum()) == 0
    # and once more on the first inputs, after the second call used the scratch
    again = sv.verify_sample_static(*ins[0], signals=True, accept_prob=True)
    torch.cuda.synchronize()
    for key in ("accept_len", "tokens", "status", "signals", "accept_prob"):
        _same(again[key].cpu().numpy(), got[0][key].cpu().numpy(), key)


@pytest.mark.gpu
def test_static_calls_allocate_no_device_memory(dev):
    """With outputs preallocated, static calls leave torch's allocator
    counters and the device's free memory exactly as they were (after one
    warm-up call: loading the library's module is its one-time setup)."""
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    o = O.load()
    wl = PT.make_workload(o, "m", 3)
    x = _inputs(wl, dev)
    B, G = wl.B, wl.G
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               tokens=torch.empty(B, G + 1, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev),
               signals=torch.empty(B, 4, dtype=torch.float32, device=dev),
               accept_prob=torch.empty(B, G, dtype=torch.float32, device=dev))
    sv.verify_sample_static(*x, signals=True, accept_prob=True, out=out)
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev), torch.cuda.mem_get_info(dev)[0])
    for _ in range(2):
        sv.verify_sample_static(*x, signals=True, accept_prob=True, out=out)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(dev), torch.cuda.memory_reserved(dev), torch.cuda.mem_get_info(dev)[0])
    assert after == before, (before, after)

