"""Host side of the context-parallel decode: shard ranges, and the partial-state exchange over a
real two-rank gloo process group on CPU.

The ranks' partial states here come from the oracle (this file is a test), the
exchange is the library's ``exchange_partials``, and the merged result must equal
the oracle's unsharded decode.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from split_kv_decode_fd_gb300.context_parallel import exchange_partials, local_lengths, shard_range


@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_shard_ranges_partition_each_sequence(world):
    r = np.random.default_rng(world)
    for L in [0, 1, 15, 16, 17, 100, 1000, 4097] + r.integers(0, 20000, 20).tolist():
        spans = [shard_range(L, world, k) for k in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == L
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0 and a0 <= a1
        assert all(lo % 16 == 0 for lo, hi in spans if hi > lo)  # non-empty slices start on 16-key boundaries
        assert sum(local_lengths([L], world, k)[0] for k in range(world)) == L


def test_shard_range_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard_range(10, 0, 0)
    with pytest.raises(ValueError):
        shard_range(10, 2, 2)


def _problem(seed=3):
    r = np.random.default_rng(seed)
    B, Hq, Hkv, D, T = 3, 8, 2, 16, 90
    q = r.standard_normal((B, Hq, D))
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    lens = [90, 17, 0]
    return q, k, v, lens, 0.25


def _rank_main(rank, world, port, errq):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
        q, k, v, lens, scale = _problem()
        B, Hq, D = q.shape
        g = Hq // k.shape[1]
        o = np.zeros((B, Hq, 1, D)); m = np.full((B, Hq, 1), -np.inf); l = np.zeros((B, Hq, 1))
        for b in range(B):
            lo, hi = shard_range(lens[b], world, rank)
            for h in range(Hq):
                kvh = oracle.kv_head_for(h, g)
                o[b, h, 0], m[b, h, 0], l[b, h, 0] = oracle.split_state(q[b, h], k[b, kvh, lo:hi], v[b, kvh, lo:hi],
                                                                        scale)
        oa, ma, la = exchange_partials(torch.from_numpy(o), torch.from_numpy(m), torch.from_numpy(l))
        assert tuple(oa.shape) == (B, Hq, world, D) and tuple(ma.shape) == (B, Hq, world)
        ref_out, ref_lse = oracle.decode(q, k, v, scale, seq_lens=lens)
        for b in range(B):
            for h in range(Hq):
                out, lse = oracle.combine(oa[b, h].numpy(), ma[b, h].numpy(), la[b, h].numpy())
                np.testing.assert_allclose(out, ref_out[b, h], rtol=0, atol=1e-12)
                if np.isfinite(ref_lse[b, h]):
                    assert abs(lse - ref_lse[b, h]) < 1e-12
                else:
                    assert lse == -np.inf
        torch.distributed.destroy_process_group()
    except Exception as e:  # noqa: BLE001 - reported to the parent
        errq.put(f"rank {rank}: {type(e).__name__}: {e}")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_partials_over_gloo(world):
    ctx = mp.get_context("spawn")
    errq = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, errq)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    errors = []
    while not errq.empty():
        errors.append(errq.get())
    assert not errors, errors
    assert all(p.exitcode == 0 for p in procs)
