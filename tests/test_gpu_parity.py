"""GPU parity: libfdecode (through its C ABI) against the float64 oracle.

Tolerance (the target accuracy of the method on these workloads):
``|gpu - ref| <= 1e-4 * (1 + |ref|)`` element by element, for ``out`` and for
finite ``lse``; ``lse = -inf`` must match exactly.  Index work is bit-exact:
padding and unreferenced pages poisoned with NaN must not change one output bit.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_fd_gb300 as fd
from workloads import CONFIGS, make_case, poison_padding, small_spec

pytestmark = pytest.mark.gpu

TOL = 1e-4


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(gpu, ref, what):
    gpu = np.asarray(gpu, dtype=np.float64)
    ninf_g, ninf_r = np.isneginf(gpu), np.isneginf(ref)
    assert np.array_equal(ninf_g, ninf_r), f"{what}: -inf pattern differs"
    fin = ~ninf_r
    assert np.all(np.isfinite(gpu[fin])), f"{what}: non-finite values"
    err = np.abs(gpu[fin] - ref[fin])
    bound = TOL * (1.0 + np.abs(ref[fin]))
    worst = np.max(err / bound) if err.size else 0.0
    assert worst <= 1.0, f"{what}: max err/bound = {worst:.3f} (max abs err {err.max():.3e})"


def oracle_for(case, heads=None):
    """Oracle on the same rounded inputs; ``heads``=None means every (b, h)."""
    q = np64(case.q)
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    k, v = np64(case.k), np64(case.v)
    return oracle.decode(q, k, v, case.spec.scale, seq_lens=case.lengths, max_seq_len=case.max_seq_len,
                         block_table=bt, page_size=case.spec.page_size if bt is not None else None)


def run(case, n_splits=None, **kw):
    n = case.spec.n_splits if n_splits is None else n_splits
    return fd.decode(case.q, case.k, case.v, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                     block_table=case.block_table, scale=case.spec.scale, n_splits=n, **kw)


SMALL = [
    small_spec("mha_bf16_d128", 2, 4, 4, 128, 700, lengths="uniform:1:700"),
    small_spec("mha_f32_d64", 2, 4, 4, 64, 513, kv_dtype="f32"),
    small_spec("gqa4_bf16_d128", 3, 16, 4, 128, 1000, lengths="uniform:1:1000"),
    small_spec("gqa2_bf16_d64", 2, 8, 4, 64, 300, lengths="uniform:200:300"),
    small_spec("gqa8_f32_d128", 2, 16, 2, 128, 400, kv_dtype="f32", lengths="uniform:1:400"),
    small_spec("gqa3_bf16_d128", 2, 6, 2, 128, 333, lengths="uniform:100:333"),
    small_spec("gqa12_bf16_d64", 1, 24, 2, 64, 290),
    small_spec("gqa16_bf16_d128", 2, 32, 2, 128, 257, lengths="uniform:1:257"),
    small_spec("paged16_gqa4", 4, 16, 4, 128, 600, layout="paged", page_size=16, lengths="uniform:1:600"),
    small_spec("paged32_mha_f32", 3, 2, 2, 64, 500, kv_dtype="f32", layout="paged", page_size=32,
               lengths="uniform:1:500"),
    small_spec("paged64_gqa8", 2, 16, 2, 128, 700, layout="paged", page_size=64, lengths="uniform:1:700"),
    small_spec("peaked_q", 1, 4, 4, 128, 900, q_gain=6.0),
    small_spec("peaked_q_gqa8", 2, 16, 2, 128, 900, q_gain=6.0, lengths="uniform:1:900"),
    small_spec("gqa8_bf16_d64_ragged", 3, 16, 2, 64, 777, lengths="uniform:1:777"),
    small_spec("gqa16_paged16", 3, 32, 2, 128, 650, layout="paged", page_size=16, lengths="uniform:1:650"),
    small_spec("gqa32_bf16_two_subgroups", 2, 64, 2, 128, 300, lengths="uniform:1:300"),
    small_spec("gqa16_f32_two_subgroups", 2, 32, 2, 64, 300, kv_dtype="f32", lengths="uniform:1:300"),
    small_spec("peaked_q_gqa16", 2, 32, 2, 128, 900, q_gain=6.0, lengths="uniform:1:900"),
]


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("n_splits", [0, 1, 3, 7])
def test_small_shapes_vs_oracle(spec, n_splits):
    case = make_case(spec, "cuda")
    ref_out, ref_lse = oracle_for(case)
    out, lse = run(case, n_splits=n_splits)
    torch.cuda.synchronize()
    assert_close(np64(out), ref_out, f"{spec.name} out")
    assert_close(np64(lse), ref_lse, f"{spec.name} lse")
    assert fd.workspace_status() == 0


EDGE_LENGTHS = [0, 1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 255, 256, 257, 1000]


@pytest.mark.parametrize("layout,page", [("contiguous", 16), ("paged", 16), ("paged", 48)])
@pytest.mark.parametrize("n_splits", [0, 2, 5])
@pytest.mark.parametrize("hq", [8, 16, 32, 24])  # groups of 4, 8, 16 (tensor cores) and 12 (16 padded)
def test_edge_lengths(layout, page, n_splits, hq):
    spec = small_spec(f"edges_{layout}{page}", len(EDGE_LENGTHS), hq, 2, 128, 1024, layout=layout, page_size=page,
                      seed=11)
    case = make_case(spec, "cuda", lengths=EDGE_LENGTHS)
    ref_out, ref_lse = oracle_for(case)
    out, lse = run(case, n_splits=n_splits)
    torch.cuda.synchronize()
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")
    assert np.all(np64(out)[0] == 0.0) and np.all(np.isneginf(np64(lse)[0]))


def test_all_sequences_empty():
    spec = small_spec("empty", 3, 4, 2, 64, 64, seed=3)
    case = make_case(spec, "cuda", lengths=[0, 0, 0])
    for n in (0, 1, 4):
        out, lse = run(case, n_splits=n)
        torch.cuda.synchronize()
        assert np.all(np64(out) == 0) and np.all(np.isneginf(np64(lse)))


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_config_full_oracle(cfg):
    """The workloads small enough for the full oracle: every (b, h) is checked."""
    case = make_case(CONFIGS[cfg], "cuda")
    out, lse = run(case)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out), ref_out, f"config {cfg} out")
    assert_close(np64(lse), ref_lse, f"config {cfg} lse")
    assert fd.workspace_status() == 0


def _oracle_one_paged_sequence(q_b, k_pages, v_pages, length, scale, page_size):
    """Oracle of one sequence of a paged batch, from its own pages gathered in logical order."""
    table = np.arange(k_pages.shape[0], dtype=np.int64)[None, :]
    return oracle.decode(q_b, k_pages, v_pages, scale, seq_lens=[length], block_table=table, page_size=page_size)


def test_config5_paged_full_oracle():
    """Paged serving batch at full size (B=64, Hq=64, Hkv=8, page 16): every (b, h) against the oracle.

    Each sequence's pages are gathered on the GPU in block-table order and the
    oracle runs on them with an identity table; the oracle's own paged gather
    is pinned separately (the gather identity among the oracle pins).
    """
    from concurrent.futures import ThreadPoolExecutor

    spec = CONFIGS[5]
    case = make_case(spec, "cuda")
    out, lse = run(case)
    torch.cuda.synchronize()
    o, l = np64(out), np64(lse)
    lens = case.lengths
    ps = spec.page_size
    jobs = []
    for b in range(spec.B):
        npg = -(-lens[b] // ps)
        pages = case.block_table[b, :npg].long()
        jobs.append((b, np64(case.q[b:b + 1]), case.k.index_select(0, pages).cpu(),
                     case.v.index_select(0, pages).cpu(), lens[b]))

    def one(job):
        b, qb, kb, vb, L = job
        return b, _oracle_one_paged_sequence(qb, kb.double().numpy(), vb.double().numpy(), L, spec.scale, ps)

    with ThreadPoolExecutor(max_workers=4) as ex:
        results = dict(ex.map(lambda j: one(j), jobs))
    assert sorted(results) == list(range(spec.B))
    for b in range(spec.B):
        ref_out, ref_lse = results[b]
        assert_close(o[b:b + 1], ref_out, f"config 5 b={b} out")
        assert_close(l[b:b + 1], ref_lse, f"config 5 b={b} lse")
    assert fd.workspace_status() == 0


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
@pytest.mark.parametrize("n_splits", [0, 3])
@pytest.mark.parametrize("hq,d", [(8, 128), (16, 128), (16, 64), (32, 128), (64, 64)])
def test_masked_positions_are_bit_exact(layout, n_splits, hq, d):
    spec = small_spec(f"mask_{layout}", 6, hq, 2, d, 700, layout=layout, lengths="uniform:1:700", seed=21)
    case = make_case(spec, "cuda")
    clean_out, clean_lse = run(case, n_splits=n_splits)
    for value in (float("nan"), float("inf"), -float("inf")):
        bad = poison_padding(case, value)
        if layout == "paged":
            # block-table entries past ceil(L_b / page) must never be read either
            table = bad.block_table.clone()
            for b, L in enumerate(bad.lengths):
                table[b, -(-L // spec.page_size):] = 2 ** 30
            bad = type(bad)(bad.spec, bad.q, bad.k, bad.v, bad.seq_lens, table, bad.max_seq_len)
        out, lse = run(bad, n_splits=n_splits)
        torch.cuda.synchronize()
        assert torch.equal(out, clean_out) and torch.equal(lse, clean_lse), f"poison {value} leaked"
    assert fd.workspace_status() == 0


def test_deterministic_and_split_invariant():
    case = make_case(CONFIGS[4], "cuda")
    a, la = run(case)
    b, lb = run(case)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)
    # different split counts agree within rounding
    for n in (1, 4, 16):
        c, lc = run(case, n_splits=n)
        torch.cuda.synchronize()
        assert_close(np64(c), np64(a).astype(np.float64), f"n_splits={n} vs auto")


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_partial_api_matches_oracle_and_decode(layout):
    spec = small_spec(f"partial_{layout}", 3, 8, 2, 128, 900, layout=layout, lengths="uniform:1:900", seed=5)
    case = make_case(spec, "cuda", lengths=[900, 37, 0])
    n = 5
    o, m, l = fd.split_partial(case.q, case.k, case.v, n, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                               block_table=case.block_table, scale=spec.scale)
    torch.cuda.synchronize()
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    ro, rm, rl = oracle.split_partials(np64(case.q), np64(case.k), np64(case.v), spec.scale, n,
                                       seq_lens=case.lengths, max_seq_len=case.max_seq_len, block_table=bt,
                                       page_size=spec.page_size if bt is not None else None)
    gm, gl, go = np64(m), np64(l), np64(o)
    empty = rl == 0
    assert np.all(np.isneginf(gm[empty])) and np.all(gl[empty] == 0) and np.all(go[empty] == 0)
    live = ~empty
    # m is compared directly; O and l are compared after putting both on the oracle's max
    assert_close(gm[live], rm[live], "m_part")
    shift = np.exp(gm[live] - rm[live])
    assert_close(gl[live] * shift, rl[live], "l_part")
    assert_close(go[live] * shift[:, None], ro[live], "o_part")
    # combine(split_partial) == fd_decode with the same split count, bit for bit
    out_c, lse_c = fd.combine(o, m, l)
    out_d, lse_d = run(case, n_splits=n)
    torch.cuda.synchronize()
    assert torch.equal(out_c, out_d) and torch.equal(lse_c, lse_d)
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out_c), ref_out, "combine out")
    assert_close(np64(lse_c), ref_lse, "combine lse")


def test_decode_host_matches_device():
    case = make_case(CONFIGS[4], "cuda")
    out_d, lse_d = run(case)
    q_host = case.q.cpu().pin_memory()
    lens_host = case.seq_lens.cpu()
    out_h, lse_h = fd.decode_host(q_host, case.k, case.v, seq_lens_host=lens_host, max_seq_len=case.max_seq_len,
                                  scale=case.spec.scale)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())


@pytest.mark.parametrize("pinned_out", [True, False])
@pytest.mark.parametrize("pinned_in", [True, False])
def test_host_decoder_matches_device(pinned_in, pinned_out):
    """HostDecoder (fd_decode_host, arguments marshalled once) over several steps, the
    caller rewriting q between them: pinned q and lengths are read and pinned outputs
    written by the kernels in place, pageable ones go through the workspace by copy."""
    case = make_case(CONFIGS[4], "cuda")
    q2 = case.q.flip(-1).contiguous()  # another step's q, same magnitudes
    case2 = type(case)(case.spec, q2, case.k, case.v, case.seq_lens, case.block_table, case.max_seq_len)
    out_d, lse_d = run(case)
    out_d2, lse_d2 = run(case2)
    torch.cuda.synchronize()
    assert not torch.equal(out_d, out_d2)
    q_host = torch.empty(case.q.shape, dtype=torch.float32, pin_memory=pinned_in)
    lens_host = case.seq_lens.cpu()
    if pinned_in:
        lens_host = lens_host.pin_memory()
    out_h = torch.full((case.spec.B, case.spec.Hq, case.spec.D), float("nan"), pin_memory=pinned_out)
    lse_h = torch.full((case.spec.B, case.spec.Hq), float("nan"), pin_memory=pinned_out)
    dec = fd.HostDecoder(q_host, case.k, case.v, seq_lens_host=lens_host, max_seq_len=case.max_seq_len,
                         scale=case.spec.scale, out_host=out_h, lse_host=lse_h)
    steps = ((case.q, out_d, lse_d), (q2, out_d2, lse_d2), (case.q, out_d, lse_d))
    for step, (q_src, want_out, want_lse) in enumerate(steps):
        q_host.copy_(q_src.cpu())
        out_h.fill_(float("nan"))
        lse_h.fill_(float("nan"))
        o, l = dec()
        assert o is out_h and l is lse_h
        assert torch.equal(out_h, want_out.cpu()) and torch.equal(lse_h, want_lse.cpu()), f"step {step}"
    ref_out, ref_lse = oracle_for(case)
    assert_close(np64(out_h), ref_out, "out")
    assert_close(np64(lse_h), ref_lse, "lse")


def test_host_decoder_without_lse():
    """lse_host omitted: fd_decode_host gets NULL and writes out only, same bits."""
    case = make_case(CONFIGS[4], "cuda")
    out_d, _ = run(case)
    dec = fd.HostDecoder(case.q.cpu().pin_memory(), case.k, case.v, seq_lens_host=case.seq_lens.cpu().pin_memory(),
                         max_seq_len=case.max_seq_len, scale=case.spec.scale)
    out_h, lse_h = dec()
    assert lse_h is None
    assert torch.equal(out_h, out_d.cpu())


def test_decode_host_pinned_but_unaligned_q_is_staged():
    """A pinned q that starts 4 bytes past a 16-byte boundary cannot be read in place by
    the kernels' vector loads: fd_decode_host stages it by copy, same bits."""
    case = make_case(CONFIGS[4], "cuda")
    out_d, lse_d = run(case)
    n = case.q.numel()
    raw = torch.empty(n + 4, dtype=torch.float32, pin_memory=True)
    q_host = raw[1:1 + n].view(case.q.shape)
    assert q_host.data_ptr() % 16 == 4
    q_host.copy_(case.q.cpu())
    out_h = torch.empty((case.spec.B, case.spec.Hq, case.spec.D), pin_memory=True)
    lse_h = torch.empty((case.spec.B, case.spec.Hq), pin_memory=True)
    fd.decode_host(q_host, case.k, case.v, seq_lens_host=case.seq_lens.cpu().pin_memory(),
                   max_seq_len=case.max_seq_len, scale=case.spec.scale, out_host=out_h, lse_host=lse_h)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())


def test_bad_block_table_entry_is_reported_not_faulted():
    spec = small_spec("badpage", 2, 4, 2, 128, 256, layout="paged", lengths="uniform:100:256", seed=9)
    case = make_case(spec, "cuda")
    table = case.block_table.clone()
    table[1, 0] = case.k.shape[0] + 5  # in a live position, outside the pool
    bad = type(case)(case.spec, case.q, case.k, case.v, case.seq_lens, table, case.max_seq_len)
    ws = fd.Workspace()
    run(bad, workspace=ws)
    assert fd.workspace_status(ws) == 4  # FD_ERR_BAD_INDEX
    run(case, workspace=ws)
    assert fd.workspace_status(ws) == 0


def test_workspace_reused_across_shapes():
    """One workspace serving calls of different shapes gives the same bits as fresh ones."""
    a = make_case(small_spec("reuse_a", 6, 8, 2, 128, 700, lengths="uniform:1:700", seed=31), "cuda")
    b = make_case(CONFIGS[4], "cuda")
    c = make_case(small_spec("reuse_c", 2, 4, 4, 64, 300, kv_dtype="f32", seed=32), "cuda")
    fresh = {}
    for name, case in (("a", a), ("b", b), ("c", c)):
        for n in (0, 3):
            fresh[name, n] = run(case, n_splits=n, workspace=fd.Workspace())
    shared = fd.Workspace()
    for name, case in (("a", a), ("b", b), ("c", c), ("b", b), ("a", a), ("c", c)):
        for n in (0, 3, 0):
            out, lse = run(case, n_splits=n, workspace=shared)
            ref_o, ref_l = fresh[name, n]
            assert torch.equal(out, ref_o) and torch.equal(lse, ref_l), (name, n)
    assert fd.workspace_status(shared) == 0


def _sampled_check(case, out, lse, sample):
    spec = case.spec
    o, l = np64(out), np64(lse)
    for b in sample:
        L = case.lengths[b]
        ref_out, ref_lse = oracle.decode(np64(case.q[b:b + 1]), np64(case.k[b:b + 1, :, :max(L, 1)]),
                                         np64(case.v[b:b + 1, :, :max(L, 1)]), spec.scale, seq_lens=[L])
        assert_close(o[b:b + 1], ref_out, f"b={b} out")
        assert_close(l[b:b + 1], ref_lse, f"b={b} lse")


def test_large_batch_takes_fixed_splits():
    """B above the balanced-plan limit: the library picks a split count itself."""
    spec = small_spec("big_batch", 1100, 4, 2, 64, 64, lengths="uniform:0:64", seed=41)
    case = make_case(spec, "cuda")
    out, lse = run(case, n_splits=0)
    torch.cuda.synchronize()
    _sampled_check(case, out, lse, [0, 1, 517, 1023, 1024, 1099])
    assert fd.workspace_status() == 0


def test_many_pairs_take_the_unfused_merge():
    """More (b, kv head) pairs than the fused merge's counters: split, then a separate merge."""
    spec = small_spec("many_pairs", 8300, 8, 8, 64, 32, lengths="uniform:0:32", seed=43)
    case = make_case(spec, "cuda")
    for n in (0, 2):
        out, lse = run(case, n_splits=n)
        torch.cuda.synchronize()
        _sampled_check(case, out, lse, [0, 7, 4000, 8191, 8299])
    o2, m2, l2 = fd.split_partial(case.q, case.k, case.v, 2, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                                  scale=spec.scale)
    out_c, lse_c = fd.combine(o2, m2, l2)
    out_d, lse_d = run(case, n_splits=2)
    torch.cuda.synchronize()
    assert torch.equal(out_c, out_d) and torch.equal(lse_c, lse_d)
