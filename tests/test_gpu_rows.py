"""GPU parity of ``fd_decode_rows`` (several query rows per sequence) against the oracle.

Same tolerance as the single-row tests: ``|gpu - ref| <= 1e-4 * (1 + |ref|)``,
``lse = -inf`` exactly where a row sees no key, and NaN-poisoned padding must
not change one output bit.
"""

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_fd_gb300 as fd
from workloads import CONFIGS, make_case, poison_padding, small_spec

from test_gpu_parity import assert_close, np64

pytestmark = pytest.mark.gpu


def rows_q(case, n_q, seed=11):
    """[B, Hq, n_q, D] queries: the case's q as the last row, more rows drawn from a seeded generator."""
    B, Hq, D = case.q.shape
    gen = torch.Generator(device=case.q.device).manual_seed(seed)
    q = torch.randn((B, Hq, n_q, D), generator=gen, device=case.q.device, dtype=torch.float32)
    q = q * case.spec.q_gain
    q[:, :, -1] = case.q
    return q.contiguous()


def oracle_rows(case, q, causal, heads=None):
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    return oracle.decode_rows(np64(q), np64(case.k), np64(case.v), case.spec.scale, causal=causal,
                              seq_lens=case.lengths, max_seq_len=case.max_seq_len, block_table=bt,
                              page_size=case.spec.page_size if bt is not None else None)


def run_rows(case, q, causal, n_splits=0, **kw):
    return fd.decode_rows(q, case.k, case.v, causal=causal, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                          block_table=case.block_table, scale=case.spec.scale, n_splits=n_splits, **kw)


# (spec, n_q): the virtual group g * n_q picks the engine: bf16 with g * n_q >= 4 runs on tensor cores,
# more than 8 on the sixteen-head one
SPECS = [
    (small_spec("mha_bf16_d128", 2, 4, 4, 128, 700, lengths="uniform:1:700"), 2),   # g'=2, CUDA cores
    (small_spec("mha_bf16_d128_q4", 2, 4, 4, 128, 700, lengths="uniform:1:700"), 4),  # g'=4, tensor cores
    (small_spec("gqa4_bf16_d128", 3, 16, 4, 128, 1000, lengths="uniform:1:1000"), 2),  # g'=8
    (small_spec("gqa4_bf16_d64", 2, 8, 2, 64, 400, lengths="uniform:1:400"), 3),    # g'=12 of 16 rows
    (small_spec("gqa8_bf16_d128", 2, 16, 2, 128, 500), 2),                          # g'=16, sixteen-head engine
    (small_spec("mha_f32_d64", 2, 4, 4, 64, 513, kv_dtype="f32"), 3),               # fp32 cache
    (small_spec("paged16_gqa2", 3, 8, 4, 128, 600, layout="paged", page_size=16, lengths="uniform:1:600"), 4),
    (small_spec("paged32_mha_f32", 2, 2, 2, 64, 300, kv_dtype="f32", layout="paged", page_size=32,
                lengths="uniform:1:300"), 2),
    (small_spec("paged16_gqa8", 3, 16, 2, 128, 700, layout="paged", page_size=16, lengths="uniform:1:700"), 2),
    (small_spec("gqa8_rows4", 2, 16, 2, 128, 400, lengths="uniform:1:400"), 4),     # g'=32, two groups of 16
]


@pytest.mark.parametrize("spec,n_q", SPECS, ids=lambda x: getattr(x, "name", str(x)))
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n_splits", [0, 3])
def test_rows_vs_oracle(spec, n_q, causal, n_splits):
    case = make_case(spec, "cuda")
    q = rows_q(case, n_q)
    ref_out, ref_lse = oracle_rows(case, q, causal)
    out, lse = run_rows(case, q, causal, n_splits)
    torch.cuda.synchronize()
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


@pytest.mark.parametrize("hq,n_q", [(4, 4), (8, 2), (16, 2), (16, 3)])
@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("n_splits", [0, 2])
def test_rows_shorter_than_the_window(hq, n_q, layout, n_splits):
    """Sequences of 0..n_q keys: early causal rows see no key (zeros, -inf)."""
    spec = small_spec("short", 8, hq, 4 if hq != 16 else 2, 128, 300, layout=layout)
    lens = [0, 1, 2, 3, 4, 5, 129, 300]
    case = make_case(spec, "cuda", lengths=lens)
    q = rows_q(case, n_q)
    for causal in (True, False):
        ref_out, ref_lse = oracle_rows(case, q, causal)
        out, lse = run_rows(case, q, causal, n_splits)
        torch.cuda.synchronize()
        assert_close(np64(out), ref_out, f"out causal={causal}")
        assert_close(np64(lse), ref_lse, f"lse causal={causal}")
    assert np.isneginf(ref_lse[0]).all()  # the empty sequence


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("hq,n_q", [(4, 2), (8, 4), (8, 8)])
def test_rows_masked_positions_are_bit_exact(layout, hq, n_q):
    spec = small_spec("poison", 3, hq, 4, 128, 400, layout=layout, lengths="uniform:1:400")
    case = make_case(spec, "cuda")
    bad = poison_padding(case)
    q = rows_q(case, n_q)
    for causal in (True, False):
        a_out, a_lse = run_rows(case, q, causal)
        b_out, b_lse = run_rows(bad, q, causal)
        torch.cuda.synchronize()
        assert torch.equal(a_out, b_out) and torch.equal(a_lse, b_lse)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (32, 8)])
def test_one_row_is_decode(hq, hkv):
    """n_q = 1 runs the same plan as fd_decode: identical bits."""
    spec = small_spec("one_row", 2, hq, hkv, 128, 900, lengths="uniform:1:900")
    case = make_case(spec, "cuda")
    out1, lse1 = fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                           scale=case.spec.scale)
    for causal in (True, False):
        out, lse = run_rows(case, case.q.unsqueeze(2).contiguous(), causal)
        torch.cuda.synchronize()
        assert torch.equal(out[:, :, 0], out1) and torch.equal(lse[:, :, 0], lse1)


def test_causal_rows_equal_shorter_decodes():
    """Row i of a causal window is a one-row decode of the first L - (n_q - 1 - i) keys."""
    spec = small_spec("window", 3, 16, 4, 128, 1000, lengths="uniform:8:1000")
    case = make_case(spec, "cuda")
    n_q = 4
    q = rows_q(case, n_q)
    out, lse = run_rows(case, q, True)
    for i in range(n_q):
        lens = (case.seq_lens - (n_q - 1 - i)).clamp(min=0)
        o1, l1 = fd.decode(q[:, :, i].contiguous(), case.k, case.v, seq_lens=lens, max_seq_len=case.max_seq_len,
                           scale=case.spec.scale)
        torch.cuda.synchronize()
        # different virtual-head grouping, so not bit-identical: the oracle's tolerance
        assert_close(np64(out[:, :, i]), np64(o1).astype(np.float64), f"row {i} out")
        assert_close(np64(lse[:, :, i]), np64(l1).astype(np.float64), f"row {i} lse")


def _sampled_rows(case, q, out, lse, causal, sample):
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    k, v = case.k, case.v
    n_q = q.shape[2]
    g = case.spec.Hq // case.spec.Hkv
    for b, h, i in sample:
        L = case.lengths[b]
        lim = oracle.row_key_limit(L, n_q, i, causal)
        kvh = oracle.kv_head_for(h, g)
        if bt is None:
            kr, vr = np64(k[b, kvh, :lim]), np64(v[b, kvh, :lim])
        else:
            ps = case.spec.page_size
            pages = bt[b, :-(-lim // ps)] if lim else bt[b, :0]
            kr = np64(k[pages, kvh].reshape(-1, k.shape[-1])[:lim])
            vr = np64(v[pages, kvh].reshape(-1, v.shape[-1])[:lim])
        ro, rl = oracle.attend_row(np64(q[b, h, i]), kr, vr, case.spec.scale)
        assert_close(np64(out[b, h, i]), ro, f"out[{b},{h},{i}]")
        assert_close(np.array([float(lse[b, h, i])]), np.array([rl]), f"lse[{b},{h},{i}]")


@pytest.mark.parametrize("cfg,n_q", [(3, 4), (5, 2)])
def test_config_rows_sampled(cfg, n_q):
    """Full-size workloads (128k GQA, paged serving) with a verification window, sampled rows."""
    case = make_case(CONFIGS[cfg], "cuda")
    q = rows_q(case, n_q)
    out, lse = run_rows(case, q, True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    r = np.random.default_rng(cfg)
    B, Hq = case.spec.B, case.spec.Hq
    sample = [(int(r.integers(0, B)), int(r.integers(0, Hq)), int(r.integers(0, n_q))) for _ in range(10)]
    sample += [(0, 0, 0), (B - 1, Hq - 1, n_q - 1)]
    _sampled_rows(case, q, out, lse, True, sample)


def test_rows_reject_bad_window():
    case = make_case(small_spec("bad", 1, 4, 4, 64, 64), "cuda")
    q = torch.zeros((1, 4, 65, 64), device="cuda")
    with pytest.raises(RuntimeError):
        fd.decode_rows(q, case.k, case.v)
