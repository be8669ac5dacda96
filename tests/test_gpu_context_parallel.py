"""GPU side of the context-parallel decode.

Ranks are emulated one after another on the one GPU (their kernels never wait on
each other): each computes its slice's partial state with ``fd_split_partial``, the
states are concatenated in rank order as ``exchange_partials`` lays them out, and
``fd_combine`` merges them.  A one-rank NCCL group runs the full ``cp_decode`` path,
and two or three processes sharing the one GPU run it over a gloo group: each
process holds its own slice of the cache, runs the kernels on it, exchanges the
partial states through host memory and merges them, so the processes' kernels are
independent and only the host exchange connects them.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import split_kv_decode_fd_gb300 as fd
from split_kv_decode_fd_gb300.context_parallel import shard_range
from workloads import CONFIGS, make_case, small_spec

from test_gpu_parity import assert_close, np64, oracle_for

pytestmark = pytest.mark.gpu


def local_cache(case, world, rank):
    """This rank's slice of every sequence, moved to row 0 of a local contiguous cache."""
    lens = case.lengths
    spans = [shard_range(L, world, rank) for L in lens]
    cap = max(1, max(hi - lo for lo, hi in spans))
    B, Hkv, _, D = case.k.shape
    k = torch.zeros((B, Hkv, cap, D), dtype=case.k.dtype, device="cuda")
    v = torch.zeros_like(k)
    for b, (lo, hi) in enumerate(spans):
        k[b, :, :hi - lo] = case.k[b, :, lo:hi]
        v[b, :, :hi - lo] = case.v[b, :, lo:hi]
    n = torch.tensor([hi - lo for lo, hi in spans], dtype=torch.int32, device="cuda")
    return k, v, n, cap


@pytest.mark.parametrize("spec", [
    small_spec("gqa4_ragged", 4, 16, 4, 128, 900, lengths="uniform:1:900"),
    small_spec("gqa16", 2, 32, 2, 128, 500),
    small_spec("mha_f32_d64", 3, 4, 4, 64, 333, kv_dtype="f32", lengths="uniform:1:333"),
], ids=lambda s: s.name)
@pytest.mark.parametrize("world", [2, 3, 8])
def test_emulated_ranks_match_oracle(spec, world):
    case = make_case(spec, "cuda")
    parts = []
    for rank in range(world):
        k, v, n, cap = local_cache(case, world, rank)
        parts.append(fd.split_partial(case.q, k, v, 1, seq_lens=n, max_seq_len=cap, scale=spec.scale))
    o = torch.cat([p[0] for p in parts], dim=2)
    m = torch.cat([p[1] for p in parts], dim=2)
    l = torch.cat([p[2] for p in parts], dim=2)
    out, lse = fd.combine(o, m, l)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


def test_emulated_ranks_128k():
    """The 128k GQA workload over 8 emulated ranks of 16k keys each."""
    case = make_case(CONFIGS[3], "cuda")
    world = 8
    parts = []
    for rank in range(world):
        lo, hi = shard_range(case.max_seq_len, world, rank)
        k = case.k[:, :, lo:hi].contiguous()
        v = case.v[:, :, lo:hi].contiguous()
        parts.append(fd.split_partial(case.q, k, v, 1, max_seq_len=hi - lo, scale=case.spec.scale))
    out, lse = fd.combine(torch.cat([p[0] for p in parts], 2), torch.cat([p[1] for p in parts], 2),
                          torch.cat([p[2] for p in parts], 2))
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


def _nccl_one_rank(port, errq):
    try:
        from split_kv_decode_fd_gb300.context_parallel import cp_decode
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
        torch.cuda.set_device(0)
        torch.distributed.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
        spec = small_spec("cp_nccl", 3, 16, 4, 128, 600, lengths="uniform:1:600")
        case = make_case(spec, "cuda")
        out, lse = cp_decode(case.q, case.k, case.v, seq_lens_local=case.seq_lens, max_local_len=case.max_seq_len,
                             scale=spec.scale)
        ref_out, ref_lse = oracle_for(case)
        torch.cuda.synchronize()
        assert_close(np64(out), ref_out, "out")
        assert_close(np64(lse), ref_lse, "lse")
        torch.distributed.destroy_process_group()
    except Exception as e:  # noqa: BLE001
        errq.put(f"{type(e).__name__}: {e}")


def test_cp_decode_through_a_one_rank_nccl_group():
    ctx = mp.get_context("spawn")
    errq = ctx.SimpleQueue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    p = ctx.Process(target=_nccl_one_rank, args=(port, errq))
    p.start()
    p.join(300)
    errors = []
    while not errq.empty():
        errors.append(errq.get())
    assert not errors, errors
    assert p.exitcode == 0


def _gloo_rank(rank, world, port, spec, errq):
    try:
        from split_kv_decode_fd_gb300.context_parallel import cp_decode
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
        torch.cuda.set_device(0)
        torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
        case = make_case(spec, "cuda")  # the same seeded inputs in every process
        k, v, n, cap = local_cache(case, world, rank)
        out, lse = cp_decode(case.q, k, v, seq_lens_local=n, max_local_len=cap, scale=spec.scale)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_for(case)
        assert_close(np64(out), ref_out, f"rank {rank} out")
        assert_close(np64(lse), ref_lse, f"rank {rank} lse")
        torch.distributed.destroy_process_group()
    except Exception as e:  # noqa: BLE001
        errq.put(f"rank {rank}: {type(e).__name__}: {e}")


@pytest.mark.parametrize("world", [2, 3])
def test_cp_decode_across_processes_over_gloo(world):
    """cp_decode in `world` processes on the one GPU: kernels per rank, exchange over gloo, merge."""
    spec = small_spec("cp_gloo", 3, 16, 4, 128, 2000, lengths="uniform:1:2000", seed=91)
    ctx = mp.get_context("spawn")
    errq = ctx.SimpleQueue()
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    procs = [ctx.Process(target=_gloo_rank, args=(r, world, port, spec, errq)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
    errors = []
    while not errq.empty():
        errors.append(errq.get())
    assert not errors, errors
    assert all(p.exitcode == 0 for p in procs)
