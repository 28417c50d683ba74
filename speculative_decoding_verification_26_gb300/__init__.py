"""GB300 (sm_103a) batched speculative-sampling verification.

The compute path is ``libspec_verify.so`` (hand-written CUDA, C ABI declared
in ``include/spec_verify.h``); this package holds its sources (``csrc/``), the
nvcc build (``build.py``), a ctypes binding with the same names as the C
entry points (``_lib.py``) and the seeded synthetic workloads
(``workloads.py``).  Importing the package loads nothing; the first call
loads the library and fails loudly if it is missing.
"""
from ._lib import (  # noqa: F401
    BF16, F32, GAMMA_MODEL_FLOATS, SpecVerifyError, divergence_stats, draft_signals, filter_top_k_top_p, gamma_select, launch_count, lib, profile_next_call, request_status_string,
    set_wait_limit, status_string,
    verify_greedy, verify_onehot, verify_sample, workspace, workspace_bytes,
)
from ._lib import STATIC_WORKSPACE_BYTES, verify_sample_static  # noqa: F401
