"""The split kernel's bounded waits: a wait that runs out is reported, not hung on.

Every mbarrier wait in the split kernel gives up after a time limit, records
FD_ERR_TIMEOUT in the workspace error word, lets its own copies land and exits.
The testing hook ``fd_debug_stall`` makes every CTA's producer skip the copies of
one stage (nothing is issued for it, so nothing is left in flight) and shortens
the limit to 1 ms: the consumers' waits on that stage run out.  The call must report
FD_ERR_TIMEOUT, and the next call on the same workspace must run clean and match
the oracle.
"""

import pytest
import torch

import split_kv_decode_fd_gb300 as fd
from split_kv_decode_fd_gb300 import fdecode as fdb
from workloads import make_case, small_spec

from test_gpu_parity import assert_close, np64, oracle_for, run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_splits,stage", [(0, 0), (2, 0), (2, 5)])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_clean(n_splits, stage):
    spec = small_spec("stall", 2, 8, 2, 128, 2000, lengths="uniform:1500:2000", seed=95)
    case = make_case(spec, "cuda")
    ws = fd.Workspace()
    lib = fd.load_library()
    try:
        lib.fd_debug_stall(stage, 1_000_000)  # skip one stage in every CTA; waits give up after 1 ms
        run(case, n_splits=n_splits, workspace=ws)
        assert fd.workspace_status(ws) == fdb.FD_ERR_TIMEOUT
    finally:
        lib.fd_debug_stall(-1, 0)
    assert fd.workspace_status(ws) == fdb.FD_OK  # reading the word cleared it
    out, lse = run(case, n_splits=n_splits, workspace=ws)
    torch.cuda.synchronize()
    assert fd.workspace_status(ws) == fdb.FD_OK
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out), ref_out, "out after the timed-out call")
    assert_close(np64(lse), ref_lse, "lse after the timed-out call")


@pytest.mark.parametrize("hq,hkv,B,n_q,stage", [(8, 2, 2, 300, 0), (8, 2, 2, 300, 3), (6, 2, 2, 300, 1),
                                                (32, 8, 2, 1280, 3), (12, 4, 2, 1280, 2)],
                         ids=["two_heads_first_copy", "two_heads_fourth_copy", "one_head", "queue",
                              "one_head_queue"])
def test_prefill_wait_that_runs_out_is_reported_and_the_next_call_is_clean(hq, hkv, B, n_q, stage):
    """The prefill kernel's waits are bounded the same way: with one K/V copy
    skipped in every CTA (two heads per CTA, one head, and the persistent
    launch that takes items from a queue), the call reports FD_ERR_TIMEOUT, and
    the next call on the same workspace is clean, oracle-correct, and finds the
    queue counters at zero."""
    from test_gpu_prefill import oracle_rows, run_prefill, window_q

    spec = small_spec("pstall", B, hq, hkv, 128, 1400, lengths="uniform:1300:1400", seed=97)
    case = make_case(spec, "cuda")
    q = window_q(case, n_q, seed=16)
    ws = fd.Workspace()
    lib = fd.load_library()
    try:
        lib.fd_debug_stall(stage, 1_000_000)
        run_prefill(case, q, True, workspace=ws)
        assert fd.workspace_status(ws) == fdb.FD_ERR_TIMEOUT
    finally:
        lib.fd_debug_stall(-1, 0)
    assert fd.workspace_status(ws) == fdb.FD_OK
    assert torch.all(ws.buf[128:136].cpu() == 0), "queue counters left set"
    out, lse = run_prefill(case, q, True, workspace=ws)
    torch.cuda.synchronize()
    assert fd.workspace_status(ws) == fdb.FD_OK
    ref_out, ref_lse = oracle_rows(case, q, True)
    assert_close(np64(out), ref_out, "out after the timed-out call")
    assert_close(np64(lse), ref_lse, "lse after the timed-out call")
