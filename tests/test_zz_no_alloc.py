"""fd_decode_static, the entry point for callers that cannot allocate device memory.

Such callers (a plugin handed only its input/output buffers, or code that must
not call cudaMalloc because it can synchronise the device) get the same result
as fd_decode, with the scratch taken from a fixed device array inside the
library.  Both entry points run the same kernel on the same plan, so their
outputs must be identical bit for bit; each output is also checked against the
float64 oracle.  This file is collected last so that a failure here stops a
run only after every other test has run.
"""

import ctypes

import pytest
import torch

import split_kv_decode_fd_gb300 as fd
from split_kv_decode_fd_gb300 import fdecode as fdb
from workloads import CONFIGS, make_case, small_spec

from test_gpu_parity import assert_close, np64, oracle_for

pytestmark = pytest.mark.gpu


def _abi_call(case, out, lse, n_splits):
    """Call fd_decode_static through the C ABI with caller-owned buffers only."""
    lib = fd.load_library()
    kv = fdb._kv_desc(case.k, case.v, case.block_table)
    spec = case.spec
    return lib.fd_decode_static(case.q.data_ptr(), ctypes.byref(kv), out.data_ptr(),
                                lse.data_ptr() if lse is not None else None, spec.B, spec.Hq, spec.Hkv,
                                case.seq_lens.data_ptr() if case.seq_lens is not None else None,
                                case.max_seq_len, spec.D, float(spec.scale), n_splits,
                                torch.cuda.current_stream().cuda_stream)


def _status():
    return fd.load_library().fd_static_status(torch.cuda.current_stream().cuda_stream)


def _case(which):
    if which == "ragged":
        return make_case(CONFIGS[4], "cuda")
    if which == "paged":
        return make_case(small_spec("static_paged", 5, 16, 2, 128, 900, layout="paged",
                                    lengths="uniform:0:900", seed=77), "cuda")
    if which == "f32_gqa8":
        return make_case(small_spec("static_f32", 3, 16, 2, 64, 700, kv_dtype="f32",
                                    lengths="uniform:1:700", seed=79), "cuda")
    return make_case(CONFIGS[3], "cuda")


@pytest.mark.parametrize("which,with_lse", [("ragged", True), ("paged", True), ("gqa128k", True),
                                            ("f32_gqa8", False)])
@pytest.mark.parametrize("n_splits", [0, 3])
def test_static_matches_decode_twice(which, with_lse, n_splits):
    case = _case(which)
    ref_out, ref_lse = fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                                 block_table=case.block_table, scale=case.spec.scale, n_splits=n_splits)
    torch.cuda.synchronize()
    oracle_out, oracle_lse = oracle_for(case)
    for _ in range(2):  # two calls in a row share the one scratch array
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan")) if with_lse else None
        assert _abi_call(case, out, lse, n_splits) == fdb.FD_OK
        torch.cuda.synchronize()
        assert _status() == fdb.FD_OK
        assert torch.equal(out, ref_out), "fd_decode_static and fd_decode differ"
        assert_close(np64(out), oracle_out, f"{which} out")
        if with_lse:
            assert torch.equal(lse, ref_lse)
            assert_close(np64(lse), oracle_lse, f"{which} lse")


def test_static_reports_a_bad_block_table_entry():
    """A block-table entry outside the pool is skipped by the kernel and reported, not faulted."""
    spec = small_spec("static_badpage", 2, 8, 2, 128, 256, layout="paged", lengths="uniform:100:256", seed=81)
    case = make_case(spec, "cuda")
    table = case.block_table.clone()
    table[1, 0] = case.k.shape[0] + 5  # a live position pointing past the pool
    bad = type(case)(case.spec, case.q, case.k, case.v, case.seq_lens, table, case.max_seq_len)
    out = torch.empty((spec.B, spec.Hq, spec.D), device="cuda")
    lse = torch.empty((spec.B, spec.Hq), device="cuda")
    assert _abi_call(bad, out, lse, 0) == fdb.FD_OK
    assert _status() == fdb.FD_ERR_BAD_INDEX
    assert _status() == fdb.FD_OK  # reading the word cleared it
    # the next call on the same array runs clean and matches fd_decode
    assert _abi_call(case, out, lse, 0) == fdb.FD_OK
    assert _status() == fdb.FD_OK
    ref_out, ref_lse = fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                                 block_table=case.block_table, scale=spec.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_static_rejects_problems_beyond_its_scratch():
    # explicit splits whose partials alone exceed the fixed scratch: refused before any launch
    spec = small_spec("too_big", 64, 64, 8, 128, 4096, seed=78)
    case = make_case(spec, "cuda")
    out = torch.zeros((spec.B, spec.Hq, spec.D), device="cuda")
    lse = torch.zeros((spec.B, spec.Hq), device="cuda")
    assert _abi_call(case, out, lse, 512) == fdb.FD_ERR_WORKSPACE_TOO_SMALL
    assert torch.all(out == 0)
    # More (b, KV head) pairs than the fused merge's 65536 counters would take the
    # split + separate-merge path, but one fp32 partial of D = 64 per pair is
    # already more than the 16 MiB array: the smallest such problem is refused,
    # so fd_decode_static never reaches that path.
    spec = small_spec("pairs_over_counters", 65537, 1, 1, 64, 16, seed=80)
    case = make_case(spec, "cuda")
    out = torch.zeros((spec.B, spec.Hq, spec.D), device="cuda")
    assert _abi_call(case, out, None, 1) == fdb.FD_ERR_WORKSPACE_TOO_SMALL
    assert _abi_call(case, out, None, 0) == fdb.FD_ERR_WORKSPACE_TOO_SMALL
    assert torch.all(out == 0)
