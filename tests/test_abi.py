"""Host-side checks of libfdecode through its C ABI: exports, argument errors, the split planner.

None of these calls reaches the GPU: invalid arguments are rejected on the host
before any CUDA call, and the planner inspector is pure host code.
"""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import split_kv_decode_fd_gb300 as fd
from split_kv_decode_fd_gb300 import fdecode as fdb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fdecode.h")
FAKE = 0x7F0000000000  # a 256-byte aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fd.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return fd.load_library()


def header_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FD_API\s+[\w\s\*]+?\b(fd_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ("fd_decode", "fd_split_partial", "fd_combine", "fd_workspace_bytes", "fd_decode_host"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_only_the_abi_is_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", fd.library_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(header_functions())


def test_split_size_matches_oracle_rule(lib):
    for max_len in (1, 15, 16, 17, 100, 1023, 1024, 4097, 131072):
        for n in (1, 2, 3, 4, 7, 64, 1000):
            assert fd.split_size(max_len, n) == oracle.explicit_split_size(max_len, n), (max_len, n)
    assert fd.split_size(0, 4) == 0 and fd.split_size(100, 0) == 0


def _kv(layout=0, dtype=1, k=FAKE, v=FAKE + 4096, capacity=1024, table=None, max_pages=0, page=0, npages=0):
    d = fdb.KvDesc()
    d.layout, d.dtype, d.k, d.v, d.capacity = layout, dtype, k, v, capacity
    d.block_table, d.max_pages_per_seq, d.page_size, d.num_pages = table, max_pages, page, npages
    return d


def _decode(lib, kv, B=1, Hq=4, Hkv=4, D=128, max_len=1024, n_splits=4, q=FAKE, out=FAKE, ws=FAKE,
            ws_bytes=1 << 30):
    return lib.fd_decode(q, ctypes.byref(kv), out, None, B, Hq, Hkv, None, max_len, D, 0.1, n_splits, ws,
                         ws_bytes, None)


@pytest.mark.parametrize("case,expected", [
    (dict(q=0), fdb.FD_ERR_INVALID_ARG),
    (dict(out=0), fdb.FD_ERR_INVALID_ARG),
    (dict(ws=0), fdb.FD_ERR_INVALID_ARG),
    (dict(q=FAKE + 4), fdb.FD_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), fdb.FD_ERR_INVALID_ARG),
    (dict(B=0), fdb.FD_ERR_INVALID_ARG),
    (dict(D=96), fdb.FD_ERR_UNSUPPORTED),
    (dict(D=256), fdb.FD_ERR_UNSUPPORTED),
    (dict(n_splits=-1), fdb.FD_ERR_INVALID_ARG),
    (dict(max_len=2048), fdb.FD_ERR_INVALID_ARG),  # longer than the cache capacity
    (dict(ws_bytes=1024), fdb.FD_ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_rejects_bad_arguments(lib, case, expected):
    assert _decode(lib, _kv(), **case) == expected


@pytest.mark.parametrize("kv,expected", [
    (_kv(k=0), fdb.FD_ERR_INVALID_ARG),
    (_kv(v=FAKE + 8), fdb.FD_ERR_INVALID_ARG),
    (_kv(dtype=7), fdb.FD_ERR_UNSUPPORTED),
    (_kv(layout=3), fdb.FD_ERR_INVALID_ARG),
    (_kv(layout=1, table=None, max_pages=64, page=16, npages=100), fdb.FD_ERR_INVALID_ARG),
    (_kv(layout=1, table=FAKE, max_pages=64, page=8, npages=100), fdb.FD_ERR_INVALID_ARG),
    (_kv(layout=1, table=FAKE, max_pages=64, page=24, npages=100), fdb.FD_ERR_INVALID_ARG),
    (_kv(layout=1, table=FAKE, max_pages=32, page=16, npages=100), fdb.FD_ERR_INVALID_ARG),  # 32*16 < 1024
    (_kv(layout=1, table=FAKE, max_pages=64, page=16, npages=0), fdb.FD_ERR_INVALID_ARG),
])
def test_decode_rejects_bad_kv(lib, kv, expected):
    assert _decode(lib, kv) == expected


def test_partial_and_combine_reject_bad_arguments(lib):
    kv = _kv()
    sp = lambda **a: lib.fd_split_partial(a.get("q", FAKE), ctypes.byref(kv), 1, 4, 4, None, 1024, a.get("D", 128),
                                          0.1, a.get("n", 4), a.get("o", FAKE), FAKE, FAKE, None)
    assert sp(n=0) == fdb.FD_ERR_INVALID_ARG
    assert sp(o=0) == fdb.FD_ERR_INVALID_ARG
    assert sp(D=32) == fdb.FD_ERR_UNSUPPORTED
    cb = lambda **a: lib.fd_combine(FAKE, FAKE, FAKE, a.get("out", FAKE), None, 1, 4, a.get("D", 128),
                                    a.get("n", 4), None)
    assert cb(n=0) == fdb.FD_ERR_INVALID_ARG
    assert cb(out=0) == fdb.FD_ERR_INVALID_ARG
    assert cb(D=80) == fdb.FD_ERR_UNSUPPORTED


def test_workspace_bytes_cover_fallbacks(lib):
    # batches above the balanced-plan limit and huge pair counts still get a workspace size
    assert fd.workspace_bytes(2000, 8, 2, 128, 0, num_sms=152) > 2000 * 8 * (128 + 2) * 4
    assert fd.workspace_bytes(1, 4, 4, 64, 0, num_sms=152) >= 256 + 65536 * 4


def test_workspace_bytes(lib):
    assert lib.fd_workspace_bytes(1, 6, 4, 128, 0, 152) == 0  # Hq % Hkv != 0
    assert lib.fd_workspace_bytes(1, 4, 4, 96, 0, 152) == 0
    a = fd.workspace_bytes(1, 32, 8, 128, 0, num_sms=152)
    b = fd.workspace_bytes(1, 32, 8, 128, 0, num_sms=304)
    assert 0 < a < b
    # explicit splits: partials [B, Hq, n, D] + m + l must fit
    assert fd.workspace_bytes(2, 8, 2, 64, 5, num_sms=1) >= 2 * 8 * 5 * (64 + 2) * 4


def test_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 4, 64)
    k = torch.zeros(1, 4, 32, 64)
    with pytest.raises(ValueError, match="CUDA"):
        fd.decode(q, k, k)


# ------------------------------------------------------------------ planner
def _check_balanced(B, Hq, Hkv, lens, max_len, grid, kv_dtype="bf16"):
    pieces = fd.plan_pieces(B, Hq, Hkv, lens, max_len, 0, grid, kv_dtype=kv_dtype)
    g = Hq // Hkv
    cap = 16 if kv_dtype == "bf16" else 8  # query heads one CTA serves from one K/V read
    gpad = 1
    while gpad < g and gpad < cap:
        gpad *= 2
    nsub = -(-g // gpad)
    hv = Hkv * nsub
    L = [min(max(int(x), 0), max_len) for x in (lens if lens is not None else [max_len] * B)]
    tiles_per_cta = np.zeros(grid, dtype=np.int64)
    cover = {}
    slots = set()
    for cta, b, vkv, lo, hi, slot, npieces in pieces:
        assert 0 <= b < B and 0 <= vkv < hv and 0 <= cta < grid
        assert lo % 128 == 0 and lo < hi <= L[b]
        assert slot == b * hv + vkv + cta
        assert slot not in slots
        slots.add(slot)
        cover.setdefault((b, vkv), []).append((lo, hi, cta, npieces))
        tiles_per_cta[cta] += -(-(hi - lo) // 128)
    for b in range(B):
        for vkv in range(hv):
            runs = sorted(cover.get((b, vkv), []))
            if L[b] == 0:
                assert not runs
                continue
            # the pieces tile [0, L_b) exactly, in CTA order, and each knows how many there are
            assert runs[0][0] == 0 and runs[-1][1] == L[b]
            for (a0, a1, c0, _), (b0, b1, c1, _) in zip(runs, runs[1:]):
                assert a1 == b0 and c1 == c0 + 1
            assert all(r[3] == len(runs) for r in runs)
    assert len(slots) == 0 or max(slots) <= grid + B * hv - 2
    # Balance by cost: pairs are laid end to end on a line of cost units, each costing
    # 5 units (one more piece for a CTA; 0 when no lengths are given, every sequence
    # being as long as the others) then 4 per tile; CTA i of G = min(grid, U // 4)
    # owns the units [floor(i U / G), floor((i + 1) U / G)), so every CTA gets the same cost
    # to a tile.  Each tile must sit in the CTA owning its unit position.
    total = sum(-(-x // 128) for x in L) * hv
    if total:
        assert tiles_per_cta.sum() == total
        units, start = 0, {}
        for b in range(B):
            nt = -(-L[b] // 128)
            for vkv in range(hv):
                start[b, vkv] = units
                units += (5 if lens is not None else 0) + 4 * nt if nt else 0
        G = min(grid, units // 4)
        owner = {}
        for (b, vkv), runs in cover.items():
            for lo, hi, cta, _ in runs:
                for t in range(lo // 128, -(-hi // 128)):
                    owner[b, vkv, t] = cta
        for (b, vkv, t), cta in owner.items():
            u = start[b, vkv] + (5 if lens is not None else 0) + 4 * t
            assert cta == ((u + 1) * G - 1) // units, (b, vkv, t, cta)
        cost = np.zeros(G)
        for i in range(G):
            cost[i] = (i + 1) * units // G - i * units // G
        assert cost.max() - cost.min() <= 1


@pytest.mark.parametrize("seed", range(12))
def test_balanced_plan_random(lib, seed):
    r = np.random.default_rng(seed)
    B = int(r.integers(1, 40))
    Hkv = int(r.choice([1, 2, 4, 8]))
    g = int(r.choice([1, 2, 3, 4, 8, 12, 16]))
    max_len = int(r.integers(1, 5000))
    lens = r.integers(0, max_len + 1, size=B)
    lens[r.integers(0, B)] = 0
    grid = int(r.choice([1, 7, 148, 152, 300]))
    _check_balanced(B, g * Hkv, Hkv, lens.tolist(), max_len, grid, kv_dtype=["bf16", "f32"][seed % 2])


def test_balanced_plan_workloads(lib):
    _check_balanced(1, 32, 8, None, 131072, 152)   # 128k GQA
    _check_balanced(1, 32, 32, None, 32768, 152)   # long MHA
    r = np.random.default_rng(0)
    _check_balanced(16, 32, 8, r.integers(1024, 16385, 16).tolist(), 16384, 152)
    lens = np.clip(np.floor(np.exp(r.uniform(np.log(512), np.log(65536), 64))), 512, 65536).astype(int)
    _check_balanced(64, 64, 8, lens.tolist(), 65536, 152)
    _check_balanced(3, 4, 4, [0, 0, 0], 100, 152)   # nothing to do
    _check_balanced(4, 64, 2, [5000, 1, 300, 129], 5000, 152, kv_dtype="f32")  # g = 32: four sub-groups of 8
    _check_balanced(4, 64, 2, [5000, 1, 300, 129], 5000, 152)                  # ... two of 16 for bf16


def test_group_cap_follows_the_cache_dtype(lib):
    # g = 16: one virtual KV head per KV head for bf16 (tensor-core engine), two for fp32
    bf = fd.plan_pieces(1, 32, 2, None, 256, 1, kv_dtype="bf16")
    f32 = fd.plan_pieces(1, 32, 2, None, 256, 1, kv_dtype="f32")
    assert sorted(set(bf[:, 2].tolist())) == [0, 1]
    assert sorted(set(f32[:, 2].tolist())) == [0, 1, 2, 3]


def test_explicit_plan(lib):
    lens = [0, 1, 17, 300, 1024]
    for n in (1, 3, 4, 9):
        pieces = fd.plan_pieces(5, 8, 2, lens, 1024, n)
        S = fd.split_size(1024, n)
        assert len(pieces) == 5 * 2 * n
        for cta, b, vkv, lo, hi, s, npieces in pieces:
            assert npieces == n
            assert lo == min(s * S, lens[b]) and hi == max(lo, min((s + 1) * S, lens[b]))


@pytest.mark.parametrize("n_q,causal,expected", [
    (0, 1, fdb.FD_ERR_INVALID_ARG),
    (65, 1, fdb.FD_ERR_INVALID_ARG),
    (2, 2, fdb.FD_ERR_INVALID_ARG),
    (2, 1, fdb.FD_ERR_WORKSPACE_TOO_SMALL),  # valid window; the 1 KB workspace is what fails
])
def test_decode_rows_rejects_bad_window(lib, n_q, causal, expected):
    kv = _kv()
    st = lib.fd_decode_rows(FAKE, n_q, causal, ctypes.byref(kv), FAKE, None, 1, 4, 4, None, 1024, 128, 0.1, 4,
                            FAKE, 1024, None)
    assert st == expected


@pytest.mark.parametrize("case,expected", [
    (dict(k_new=0), fdb.FD_ERR_INVALID_ARG),
    (dict(v_new=0), fdb.FD_ERR_INVALID_ARG),
    (dict(k_new=FAKE + 8), fdb.FD_ERR_INVALID_ARG),
    (dict(max_len=1024), fdb.FD_ERR_INVALID_ARG),  # the new token needs row 1024 of a 1024-row cache
    (dict(max_len=-1), fdb.FD_ERR_INVALID_ARG),
    (dict(max_len=1023, ws_bytes=1024), fdb.FD_ERR_WORKSPACE_TOO_SMALL),  # valid; the workspace is too small
])
def test_append_decode_rejects_bad_arguments(lib, case, expected):
    kv = _kv()
    st = lib.fd_append_decode(FAKE, case.get("k_new", FAKE + 8192), case.get("v_new", FAKE + 12288),
                              ctypes.byref(kv), FAKE, None, 1, 4, 4, None, case.get("max_len", 1023), 128, 0.1, 4,
                              FAKE, case.get("ws_bytes", 1 << 30), None)
    assert st == expected


def _prefill(lib, kv, n_q=100, causal=1, D=128, ws=FAKE, ws_bytes=4096, max_len=1024, q=FAKE):
    return lib.fd_prefill(q, n_q, causal, ctypes.byref(kv), FAKE, None, 1, 4, 4, None, max_len, D, 0.1, ws,
                          ws_bytes, None)


@pytest.mark.parametrize("case,expected", [
    (dict(n_q=0), fdb.FD_ERR_INVALID_ARG),
    (dict(causal=3), fdb.FD_ERR_INVALID_ARG),
    (dict(q=0), fdb.FD_ERR_INVALID_ARG),
    (dict(ws=0), fdb.FD_ERR_INVALID_ARG),
    (dict(ws_bytes=16), fdb.FD_ERR_WORKSPACE_TOO_SMALL),
    (dict(D=96), fdb.FD_ERR_UNSUPPORTED),            # the query-tile kernel is built for D = 64 and 128
    (dict(max_len=2048), fdb.FD_ERR_INVALID_ARG),    # longer than the cache
])
def test_prefill_rejects_bad_arguments(lib, case, expected):
    assert _prefill(lib, _kv(), **case) == expected


def test_prefill_needs_a_bf16_cache(lib):
    assert _prefill(lib, _kv(dtype=fdb.FD_F32)) == fdb.FD_ERR_UNSUPPORTED


@pytest.mark.parametrize("n_q,hq,hkv,d,dtype,expect", [
    (1, 32, 8, 128, "bf16", "decode"),
    (4, 32, 8, 128, "bf16", "decode_rows"),   # 4 rows x 4 heads per KV head = 16
    (5, 32, 8, 128, "bf16", "prefill"),
    (16, 4, 4, 128, "bf16", "decode_rows"),   # 16 rows x 1 head
    (17, 4, 4, 128, "bf16", "prefill"),
    (64, 4, 4, 64, "bf16", "prefill"),
    (64, 4, 4, 96, "bf16", "decode_rows"),    # no query-tile kernel for this D: rows up to 64
    (64, 4, 4, 128, "f32", "decode_rows"),
    (65, 4, 4, 128, "f32", "none"),
])
def test_phase_dispatch_choice(lib, n_q, hq, hkv, d, dtype, expect):
    assert fd.attend_backend(n_q, hq, hkv, d, dtype).startswith(expect)


def test_attend_reports_unsupported(lib):
    chosen = ctypes.c_int32(7)
    st = lib.fd_attend(FAKE, 65, 1, ctypes.byref(_kv(dtype=fdb.FD_F32)), FAKE, None, 1, 4, 4, None, 1024, 128, 0.1,
                       0, FAKE, 1 << 20, None, ctypes.byref(chosen))
    assert st == fdb.FD_ERR_UNSUPPORTED and chosen.value == -1
