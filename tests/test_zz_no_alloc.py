"""fd_decode_static, the entry point for callers that cannot allocate device memory.

Such callers (a plugin handed only its input/output buffers, or code that must
not call cudaMalloc because it can synchronise the device) get the same result
as fd_decode, with the scratch taken from a fixed device array inside the
library.  This file is collected last so that a failure here stops a run only
after every other test has run.
"""

import ctypes

import numpy as np
import pytest
import torch

import split_kv_decode_fd_gb300 as fd
from split_kv_decode_fd_gb300 import fdecode as fdb
from workloads import CONFIGS, make_case, small_spec

pytestmark = pytest.mark.gpu

TOL = 1e-4  # the parity tolerance used for every floating-point output


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    ninf = np.isneginf(b)
    assert np.array_equal(np.isneginf(a), ninf)
    assert np.all(np.abs(a[~ninf] - b[~ninf]) <= TOL * (1.0 + np.abs(b[~ninf])))


def _abi_call(case, out, lse, n_splits):
    """Call fd_decode_static through the C ABI with caller-owned buffers only."""
    lib = fd.load_library()
    kv = fdb._kv_desc(case.k, case.v, case.block_table)
    spec = case.spec
    return lib.fd_decode_static(case.q.data_ptr(), ctypes.byref(kv), out.data_ptr(), lse.data_ptr(), spec.B,
                                spec.Hq, spec.Hkv,
                                case.seq_lens.data_ptr() if case.seq_lens is not None else None,
                                case.max_seq_len, spec.D, float(spec.scale), n_splits,
                                torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("which", ["ragged", "paged", "gqa128k"])
@pytest.mark.parametrize("n_splits", [0, 3])
def test_static_matches_decode_twice(which, n_splits):
    if which == "ragged":
        case = make_case(CONFIGS[4], "cuda")
    elif which == "paged":
        case = make_case(small_spec("static_paged", 5, 16, 2, 128, 900, layout="paged",
                                    lengths="uniform:0:900", seed=77), "cuda")
    else:
        case = make_case(CONFIGS[3], "cuda")
    ref_out, ref_lse = fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                                 block_table=case.block_table, scale=case.spec.scale, n_splits=n_splits)
    for _ in range(2):  # two calls in a row share the one scratch array
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        assert _abi_call(case, out, lse, n_splits) == fdb.FD_OK
        torch.cuda.synchronize()
        _close(out, ref_out)
        _close(lse, ref_lse)


def test_static_rejects_problems_beyond_its_scratch():
    # explicit splits whose partials alone exceed the fixed scratch: refused before any launch
    spec = small_spec("too_big", 64, 64, 8, 128, 4096, seed=78)
    case = make_case(spec, "cuda")
    out = torch.zeros((spec.B, spec.Hq, spec.D), device="cuda")
    lse = torch.zeros((spec.B, spec.Hq), device="cuda")
    assert _abi_call(case, out, lse, 512) == fdb.FD_ERR_WORKSPACE_TOO_SMALL
    assert torch.all(out == 0)
