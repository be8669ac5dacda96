"""GPU parity of ``fd_append_decode`` (fused append-KV + decode) against the oracle.

Checks, per case: ``out``/``lse`` within ``1e-4 * (1 + |ref|)`` of the oracle's
append-then-decode; the caches afterwards equal the oracle's bit for bit (one new
row per (b, KV head), nothing else touched); and the fused call gives the same
bits as writing the row first and calling ``fd_decode`` with ``L_b + 1``.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_fd_gb300 as fd
from workloads import CONFIGS, make_case, small_spec

from test_gpu_parity import assert_close, np64

pytestmark = pytest.mark.gpu


def new_rows(case, seed=5):
    """k_new, v_new [B, Hkv, D] in the cache dtype, from their own seeded generator."""
    s = case.spec
    gen = torch.Generator(device="cuda").manual_seed(seed)
    shape = (s.B, s.Hkv, s.D)
    k_new = torch.randn(shape, generator=gen, device="cuda").to(case.k.dtype)
    v_new = torch.randn(shape, generator=gen, device="cuda").to(case.k.dtype)
    return k_new, v_new


def append_case(spec, lens_before):
    """A case whose cache has room (and pages) for one more token per sequence."""
    case = make_case(spec, "cuda", lengths=[L + 1 for L in lens_before])
    seq = torch.tensor(lens_before, dtype=torch.int32, device="cuda")
    return case, seq


def oracle_append(case, seq, k_new, v_new):
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    return oracle.append_decode(np64(case.q), np64(case.k), np64(case.v), np64(k_new), np64(v_new),
                                case.spec.scale, seq_lens=seq.cpu().tolist(), max_seq_len=case.max_seq_len - 1,
                                block_table=bt, page_size=case.spec.page_size if bt is not None else None)


def run_append(case, seq, k, v, k_new, v_new, n_splits=0, **kw):
    return fd.append_decode(case.q, k, v, k_new, v_new, seq_lens=seq, max_seq_len=case.max_seq_len - 1,
                            block_table=case.block_table, scale=case.spec.scale, n_splits=n_splits, **kw)


def write_row_then_decode(case, seq, k_new, v_new, n_splits=0):
    """The unfused reference: write the rows with torch indexing, then fd_decode over L_b + 1."""
    k, v = case.k.clone(), case.v.clone()
    ps = case.spec.page_size
    for b, L in enumerate(seq.cpu().tolist()):
        if case.block_table is None:
            k[b, :, L] = k_new[b]
            v[b, :, L] = v_new[b]
        else:
            page = int(case.block_table[b, L // ps])
            k[page, :, L % ps] = k_new[b]
            v[page, :, L % ps] = v_new[b]
    out, lse = fd.decode(case.q, k, v, seq_lens=seq + 1, max_seq_len=case.max_seq_len,
                         block_table=case.block_table, scale=case.spec.scale, n_splits=n_splits)
    return out, lse, k, v


SPECS = [
    small_spec("mha_bf16_d128", 6, 4, 4, 128, 700),
    small_spec("gqa4_bf16_d128", 6, 16, 4, 128, 700),
    small_spec("gqa8_bf16_d64", 6, 16, 2, 64, 700),
    small_spec("gqa16_bf16_d128", 6, 32, 2, 128, 700),
    small_spec("gqa2_f32_d128", 6, 8, 4, 128, 700, kv_dtype="f32"),
    small_spec("paged16_gqa4", 6, 16, 4, 128, 700, layout="paged", page_size=16),
    small_spec("paged32_gqa8_d64", 6, 16, 2, 64, 700, layout="paged", page_size=32),
    small_spec("paged16_f32_mha", 6, 4, 4, 64, 700, kv_dtype="f32", layout="paged", page_size=16),
]
# lengths before the append: empty, page/tile boundaries on both sides, ragged
LENS = [0, 15, 16, 127, 128, 513]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
@pytest.mark.parametrize("n_splits", [0, 3])
def test_append_vs_oracle_and_unfused(spec, n_splits):
    case, seq = append_case(spec, LENS)
    k_new, v_new = new_rows(case)
    ref_out, ref_lse, ref_k, ref_v = oracle_append(case, seq, k_new, v_new)
    un_out, un_lse, un_k, un_v = write_row_then_decode(case, seq, k_new, v_new, n_splits)
    k, v = case.k.clone(), case.v.clone()
    out, lse = run_append(case, seq, k, v, k_new, v_new, n_splits)
    torch.cuda.synchronize()
    assert fd.workspace_status() == 0
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")
    assert np.array_equal(np64(k), ref_k) and np.array_equal(np64(v), ref_v), "cache after the append"
    assert torch.equal(k, un_k) and torch.equal(v, un_v)
    assert torch.equal(out, un_out) and torch.equal(lse, un_lse), "fused and unfused bits differ"


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_append_ignores_the_old_row(layout):
    """Whatever the cache held at position L_b (here NaN) never reaches the output."""
    spec = small_spec("nan_row", 4, 16, 4, 128, 400, layout=layout)
    case, seq = append_case(spec, [1, 100, 255, 399])
    k_new, v_new = new_rows(case, seed=9)
    k, v = case.k.clone(), case.v.clone()
    ps = spec.page_size
    for b, L in enumerate(seq.cpu().tolist()):
        if layout == "contiguous":
            k[b, :, L] = float("nan")
            v[b, :, L] = float("nan")
        else:
            page = int(case.block_table[b, L // ps])
            k[page, :, L % ps] = float("nan")
            v[page, :, L % ps] = float("nan")
    out, lse = run_append(case, seq, k, v, k_new, v_new)
    ref_out, ref_lse, _, _ = oracle_append(case, seq, k_new, v_new)
    torch.cuda.synchronize()
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")
    assert torch.isfinite(k).all() and torch.isfinite(v).all()


def test_append_bad_page_is_reported():
    """A block-table entry outside the pool for position L_b: no cache write, error word set, output intact."""
    spec = small_spec("bad_page", 2, 8, 4, 128, 300, layout="paged", page_size=16)
    case, seq = append_case(spec, [32, 100])
    k_new, v_new = new_rows(case, seed=3)
    ref_out, ref_lse, _, _ = oracle_append(case, seq, k_new, v_new)
    table = case.block_table.clone()
    table[0, 32 // 16] = 1 << 30  # the page that would receive sequence 0's new token
    case_bad = dataclasses.replace(case, block_table=table)
    k, v = case.k.clone(), case.v.clone()
    ws = fd.Workspace()
    out, lse = fd.append_decode(case.q, k, v, k_new, v_new, seq_lens=seq, max_seq_len=case.max_seq_len - 1,
                                block_table=case_bad.block_table, scale=spec.scale, workspace=ws)
    torch.cuda.synchronize()
    assert fd.workspace_status(ws) == 4  # FD_ERR_BAD_INDEX
    # sequence 1 is untouched by the bad entry; sequence 0's output still includes the new token
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


def test_append_at_full_size_128k():
    """The 128k GQA workload with its last row appended (L_b = 131071): sampled heads against the oracle."""
    spec = CONFIGS[3]
    case = make_case(spec, "cuda")
    seq = torch.full((1,), spec.T_cap - 1, dtype=torch.int32, device="cuda")
    k_new, v_new = new_rows(case, seed=13)
    k, v = case.k.clone(), case.v.clone()
    out, lse = run_append(case, seq, k, v, k_new, v_new)
    un_out, un_lse, _, _ = write_row_then_decode(case, seq, k_new, v_new)
    torch.cuda.synchronize()
    assert torch.equal(out, un_out) and torch.equal(lse, un_lse)
    assert torch.equal(k[0, :, -1], k_new[0]) and torch.equal(v[0, :, -1], v_new[0])
    assert torch.equal(k[0, :, :-1], case.k[0, :, :-1])
    g = spec.Hq // spec.Hkv
    for h in (0, 13, 31):
        kvh = oracle.kv_head_for(h, g)
        ro, rl = oracle.attend_row(np64(case.q[0, h]), np64(k[0, kvh]), np64(v[0, kvh]), spec.scale)
        assert_close(np64(out[0, h]), ro, f"out[{h}]")
        assert_close(np.array([float(lse[0, h])]), np.array([rl]), f"lse[{h}]")
