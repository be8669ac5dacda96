"""GPU parity of ``fd_prefill`` (tcgen05 query tiles) and of the ``fd_attend`` phase dispatch.

Same operation and tolerance as ``fd_decode_rows``: ``|gpu - ref| <= 1e-4 * (1 + |ref|)``
against the oracle's ``decode_rows``, ``lse = -inf`` exactly for rows without keys,
and padding poisoned with NaN must not change one output bit.
"""

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import split_kv_decode_fd_gb300 as fd
from workloads import make_case, poison_padding, small_spec

from test_gpu_parity import assert_close, np64

pytestmark = pytest.mark.gpu


def window_q(case, n_q, seed=5):
    s = case.spec
    gen = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((s.B, s.Hq, n_q, s.D), generator=gen, device="cuda") * s.q_gain


def oracle_rows(case, q, causal):
    bt = None if case.block_table is None else case.block_table.cpu().numpy()
    return oracle.decode_rows(np64(q), np64(case.k), np64(case.v), case.spec.scale, causal=causal,
                              seq_lens=case.lengths, max_seq_len=case.max_seq_len, block_table=bt,
                              page_size=case.spec.page_size if bt is not None else None)


def run_prefill(case, q, causal, **kw):
    return fd.prefill(q, case.k, case.v, causal=causal, seq_lens=case.seq_lens, max_seq_len=case.max_seq_len,
                      block_table=case.block_table, scale=case.spec.scale, **kw)


SPECS = [
    (small_spec("mha_L300", 1, 2, 2, 128, 300), 300),
    (small_spec("gqa4_ragged", 2, 8, 2, 128, 700, lengths="uniform:1:700"), 200),   # some L_b < n_q
    (small_spec("gqa8_prefix", 2, 16, 2, 128, 900, lengths="uniform:400:900"), 129),
    (small_spec("peaked", 1, 4, 1, 128, 520, q_gain=6.0), 260),
    (small_spec("paged16_gqa4", 3, 8, 2, 128, 600, layout="paged", page_size=16, lengths="uniform:1:600"), 150),
    (small_spec("paged64_mha", 2, 2, 2, 128, 500, layout="paged", page_size=64, lengths="uniform:200:500"), 64),
    (small_spec("d64_gqa4", 2, 8, 2, 64, 600, lengths="uniform:1:600"), 300),
    (small_spec("d64_paged32_mha", 2, 3, 3, 64, 400, layout="paged", page_size=32, lengths="uniform:100:400"), 150),
    # odd group size: one head per CTA, alternating S buffers; peaked scores force O rescales
    (small_spec("gqa3_ragged", 2, 6, 2, 128, 900, lengths="uniform:1:900", q_gain=4.0), 517),
    (small_spec("mha_d64_long", 1, 2, 2, 64, 1500, q_gain=5.0), 1500),
]


@pytest.mark.parametrize("spec,n_q", SPECS, ids=lambda x: getattr(x, "name", str(x)))
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_vs_oracle(spec, n_q, causal):
    case = make_case(spec, "cuda")
    q = window_q(case, n_q)
    ws = fd.Workspace()
    out, lse = run_prefill(case, q, causal, workspace=ws)
    ref_out, ref_lse = oracle_rows(case, q, causal)
    torch.cuda.synchronize()
    assert fd.workspace_status(ws) == 0
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


@pytest.mark.parametrize("n_q", [1, 7, 64])
@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_prefill_agrees_with_decode_rows(n_q, layout):
    spec = small_spec("agree", 3, 8, 2, 128, 800, layout=layout, lengths="uniform:64:800")
    case = make_case(spec, "cuda")
    q = window_q(case, n_q, seed=8)
    a_out, a_lse = run_prefill(case, q, True)
    b_out, b_lse = fd.decode_rows(q, case.k, case.v, causal=True, seq_lens=case.seq_lens,
                                  max_seq_len=case.max_seq_len, block_table=case.block_table, scale=spec.scale)
    torch.cuda.synchronize()
    assert_close(np64(a_out), np64(b_out).astype(np.float64), "out vs decode_rows")
    assert_close(np64(a_lse), np64(b_lse).astype(np.float64), "lse vs decode_rows")


@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_prefill_padding_is_bit_exact(layout):
    spec = small_spec("poison", 3, 4, 2, 128, 500, layout=layout, lengths="uniform:1:500")
    case = make_case(spec, "cuda")
    q = window_q(case, 180, seed=4)
    bad = poison_padding(case)
    for causal in (True, False):
        a = run_prefill(case, q, causal)
        b = run_prefill(bad, q, causal)
        torch.cuda.synchronize()
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("hkv", [8, 32], ids=["gqa4", "mha"])
def test_prefill_long_prompt_sampled(hkv):
    """A 4096-token causal prompt over a 4096-key cache (B=1, Hq=32; the benchmark's shape, GQA
    and MHA, i.e. both kernel variants): sampled rows."""
    spec = small_spec("prompt4k", 1, 32, hkv, 128, 4096)
    case = make_case(spec, "cuda")
    n_q = 4096
    q = window_q(case, n_q, seed=11)
    out, lse = run_prefill(case, q, True)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    r = np.random.default_rng(0)
    rows = [(int(r.integers(0, 32)), int(r.integers(0, n_q))) for _ in range(12)] + [(0, 0), (31, n_q - 1)]
    g = 32 // hkv
    for h, i in rows:
        lim = oracle.row_key_limit(4096, n_q, i, True)
        kvh = oracle.kv_head_for(h, g)
        ro, rl = oracle.attend_row(np64(q[0, h, i]), np64(case.k[0, kvh, :lim]), np64(case.v[0, kvh, :lim]),
                                   spec.scale)
        assert_close(np64(out[0, h, i]), ro, f"out[{h},{i}]")
        assert_close(np.array([float(lse[0, h, i])]), np.array([rl]), f"lse[{h},{i}]")


def test_prefill_rejects_what_it_does_not_cover():
    for spec in (small_spec("f32", 1, 2, 2, 128, 64, kv_dtype="f32"), small_spec("f32d64", 1, 2, 2, 64, 64,
                                                                                 kv_dtype="f32")):
        case = make_case(spec, "cuda")
        q = window_q(case, 80)
        with pytest.raises(RuntimeError, match="fd_prefill"):
            run_prefill(case, q, True)


@pytest.mark.parametrize("n_q,hq,hkv,dtype,expect", [
    (1, 8, 2, "bf16", "decode"),
    (4, 8, 2, "bf16", "decode_rows"),     # 4 rows x 4 heads = 16 per KV head
    (5, 8, 2, "bf16", "prefill"),
    (300, 8, 2, "bf16", "prefill"),
    (20, 4, 4, "f32", "decode_rows"),     # no prefill kernel for fp32 caches
])
def test_attend_dispatch(n_q, hq, hkv, dtype, expect):
    assert fd.attend_backend(n_q, hq, hkv, 128, dtype).startswith(expect)
    spec = small_spec("attend", 2, hq, hkv, 128, 400, kv_dtype=dtype, lengths="uniform:300:400")
    case = make_case(spec, "cuda")
    q = window_q(case, n_q, seed=2)
    out, lse, name = fd.attend(q, case.k, case.v, causal=True, seq_lens=case.seq_lens,
                               max_seq_len=case.max_seq_len, scale=spec.scale)
    torch.cuda.synchronize()
    assert name.startswith(expect)
    ref_out, ref_lse = oracle_rows(case, q, True)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


def test_prefill_repeats_bit_identically():
    """The same call twenty times gives the same bits (a pipeline race would show up as drift)."""
    spec = small_spec("repeat", 2, 8, 2, 128, 700, lengths="uniform:1:700", q_gain=3.0)
    case = make_case(spec, "cuda")
    q = window_q(case, 200, seed=6)
    first = run_prefill(case, q, True)
    ref_out, ref_lse = oracle_rows(case, q, True)
    torch.cuda.synchronize()
    assert_close(np64(first[0]), ref_out, "out")
    for _ in range(20):
        o, l = run_prefill(case, q, True)
        torch.cuda.synchronize()
        assert torch.equal(o, first[0]) and torch.equal(l, first[1])


@pytest.mark.parametrize("hq,hkv", [(8, 2), (6, 2)], ids=["two_heads_per_cta", "one_head_per_cta"])
@pytest.mark.parametrize("layout", ["contiguous", "paged"])
def test_prefill_sequences_without_keys(hq, hkv, layout):
    """Sequences with L_b = 0 between ones with keys: their items have no key tiles
    (out = 0, lse = -inf), and the CTAs' barrier phases stay in step around them."""
    spec = small_spec("zero_len", 5, hq, hkv, 128, 400, layout=layout, page_size=16)
    case = make_case(spec, "cuda", lengths=[0, 300, 0, 1, 400])
    q = window_q(case, 140, seed=12)
    for causal in (True, False):
        out, lse = run_prefill(case, q, causal)
        ref_out, ref_lse = oracle_rows(case, q, causal)
        torch.cuda.synchronize()
        assert_close(np64(out), ref_out, "out")
        assert_close(np64(lse), ref_lse, "lse")
        assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
        assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))


@pytest.mark.parametrize("hq,hkv,d", [(4, 2, 128), (6, 2, 128), (4, 4, 64)],
                         ids=["two_heads_per_cta", "one_head_per_cta", "d64_mha"])
def test_prefill_writes_only_its_rows(hq, hkv, d):
    """The epilogue stores 128-row tiles through a tensor map per head: the rows of
    the last tile past n_q (here 2 of 128) must not be written, neither into the
    next head's rows nor past the end of the output."""
    spec = small_spec("tail_rows", 2, hq, hkv, d, 300, lengths="uniform:140:300", seed=31)
    case = make_case(spec, "cuda")
    n_q = 130
    q = window_q(case, n_q, seed=13)
    numel = spec.B * hq * n_q * d
    big = torch.full((numel + 4096,), 12345.0, device="cuda")
    out = big[:numel].view(spec.B, hq, n_q, d)
    lse = torch.empty((spec.B, hq, n_q), device="cuda")
    run_prefill(case, q, True, out=out, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(big[numel:] == 12345.0), "the prefill wrote past its output"
    ref_out, ref_lse = oracle_rows(case, q, True)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


@pytest.mark.parametrize("hq,hkv,B,n_q,d,layout,page", [(32, 8, 2, 1280, 128, "contiguous", 16),
                                                       (6, 2, 8, 512, 128, "contiguous", 16),
                                                       (32, 8, 2, 1280, 64, "contiguous", 16),
                                                       (32, 8, 2, 1280, 128, "paged", 16),
                                                       (32, 8, 2, 1280, 128, "paged", 64),
                                                       (6, 2, 8, 512, 64, "paged", 32)],
                         ids=["two_heads_per_cta", "one_head_per_cta", "two_heads_d64", "two_heads_paged16",
                              "two_heads_paged64", "one_head_d64_paged32"])
@pytest.mark.parametrize("causal", [True, False], ids=["causal", "all_keys"])
def test_prefill_more_items_than_sms(hq, hkv, B, n_q, d, layout, page, causal):
    """More 128-row query tiles than SMs: one CTA per SM takes the items from
    the queue, with two heads or one head per CTA; sequences without keys among
    them, contiguous and paged caches, causal windows and rows that see every
    key: every output matches the oracle."""
    spec = small_spec("many_items", B, hq, hkv, d, 1400, layout=layout, page_size=page, seed=33)
    lengths = [0, 800, 650, 700, 720, 0, 790, 800] if B > 2 else [1400, 0]
    case = make_case(spec, "cuda", lengths=lengths)
    q = window_q(case, n_q, seed=14)
    out, lse = run_prefill(case, q, causal)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_rows(case, q, causal)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")


@pytest.mark.parametrize("hq,hkv", [(32, 8), (12, 4)], ids=["two_heads_per_cta", "one_head_per_cta"])
def test_prefill_queue_counters_return_to_zero(hq, hkv):
    """With more query tiles than SMs, CTAs take items from two counters in the
    workspace header (bytes 128-135): the last CTA leaves both at zero, and the
    results do not depend on which CTA took which item (two heads per CTA, and
    one head for an odd group size)."""
    spec = small_spec("queue", 2, hq, hkv, 128, 1300, seed=35)
    case = make_case(spec, "cuda", lengths=[1300, 1290])
    q = window_q(case, 1280, seed=15)
    ws = fd.Workspace()
    first = run_prefill(case, q, True, workspace=ws)
    torch.cuda.synchronize()
    hdr = ws.buf[128:136].cpu()
    assert torch.all(hdr == 0), f"queue counters left at {hdr.tolist()}"
    for _ in range(3):
        again = run_prefill(case, q, True, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(again[0], first[0]) and torch.equal(again[1], first[1])
    assert torch.all(ws.buf[128:136].cpu() == 0)
    assert fd.workspace_status(ws) == 0


@pytest.mark.parametrize("hq,hkv", [(4, 2), (3, 3)], ids=["two_heads_per_cta", "one_head_per_cta"])
@pytest.mark.parametrize("slope", [30.0, 120.0], ids=["rising", "steep"])
def test_prefill_rising_scores_move_the_max_tile_after_tile(hq, hkv, slope):
    """Scores that grow along the sequence: each 128-key tile holds keys above
    the running max, so the softmax keeps taking its max-first path (P made
    again from the new base) and rescales O tile after tile; the outputs still
    match the oracle."""
    T, n_q, D = 1536, 384, 128
    gen = torch.Generator().manual_seed(41)
    u = torch.randn(D, generator=gen)
    u = u / u.norm()
    ramp = torch.linspace(0.0, 1.0, T)[None, None, :, None]
    k = (ramp * slope * u + 0.3 * torch.randn(1, hkv, T, D, generator=gen)).to(torch.bfloat16)
    v = torch.randn(1, hkv, T, D, generator=gen).to(torch.bfloat16)
    q = 4.0 * u + 0.5 * torch.randn(1, hq, n_q, D, generator=gen)
    scale = D ** -0.5
    out, lse = fd.prefill(q.cuda(), k.cuda(), v.cuda(), causal=True, max_seq_len=T, scale=scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.decode_rows(np64(q), np64(k), np64(v), scale, causal=True, max_seq_len=T)
    assert_close(np64(out), ref_out, "out")
    assert_close(np64(lse), ref_lse, "lse")
