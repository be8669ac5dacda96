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
