"""Checks that pin the float64 oracle to facts other than itself.

Each ``check_*`` function raises ``AssertionError`` when the oracle breaks the
fact it tests.  ``test_oracle.py`` runs them against the oracle as written;
``test_oracle_mutants.py`` runs them against deliberately broken copies of the
oracle and requires that some check fails for every planted mistake.

Facts used (none of them is the oracle's own formula retyped):

* closed forms worked by hand (``golden/closed_forms.txt``);
* brute force at 50 significant digits with mpmath, straight from
  ``sum_t e^{s_t} v_t / sum_t e^{s_t}`` (no max subtraction) on tiny inputs;
* the float64 ``scaled_dot_product_attention`` of PyTorch on CPU (a library
  routine), with the KV heads repeated ``g`` times for GQA;
* shift invariance of softmax ("attn-flash-decoding", answer on why the
  log-sum-exp combine is exact): adding ``c`` to every score leaves ``out``
  unchanged and adds ``c`` to ``lse``;
* split independence: any split size, merged, equals the unsplit result;
  the online tile loop, for any tile, equals it too;
* invariants: output inside the per-dimension hull of the valid V rows;
  constant V returns that constant;
* the paged layout equals the contiguous layout after an independent gather.
"""

from __future__ import annotations

import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "closed_forms.txt")


# ---------------------------------------------------------------- golden file
def load_golden(path=GOLDEN):
    cases, cur = [], None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            if not line and cur is not None:
                cases.append(cur)
                cur = None
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            if cur is not None:
                cases.append(cur)
            cur = {"name": rest, "q": [], "k": [], "v": [], "len": {}, "out": [], "lse": []}
        elif key in ("cite", "why"):
            cur[key] = rest
        elif key == "shape":
            cur["shape"] = tuple(int(x) for x in rest.split())
        elif key == "scale":
            cur["scale"] = float(rest)
        elif key == "len":
            b, n = rest.split()
            cur["len"][int(b)] = int(n)
        else:
            toks = rest.split()
            cur[key].append((int(toks[0]), int(toks[1]), [float(x) for x in toks[2:]]))
    if cur is not None:
        cases.append(cur)
    built = []
    for c in cases:
        B, Hq, Hkv, D = c["shape"]
        q = np.zeros((B, Hq, D))
        for b, h, vals in c["q"]:
            q[b, h] = vals
        rows = {}
        for b, kvh, vals in c["k"]:
            rows.setdefault((b, kvh), []).append(vals)
        T = max(len(r) for r in rows.values())
        k = np.zeros((B, Hkv, T, D))
        v = np.zeros((B, Hkv, T, D))
        for (b, kvh), r in rows.items():
            k[b, kvh, :len(r)] = r
        vrows = {}
        for b, kvh, vals in c["v"]:
            vrows.setdefault((b, kvh), []).append(vals)
        for (b, kvh), r in vrows.items():
            v[b, kvh, :len(r)] = r
        lens = [c["len"].get(b, T) for b in range(B)]
        out = np.zeros((B, Hq, D))
        for b, h, vals in c["out"]:
            out[b, h] = vals
        lse = np.zeros((B, Hq))
        for b, h, vals in c["lse"]:
            lse[b, h] = vals[0]
        built.append(dict(name=c["name"], cite=c.get("cite", ""), q=q, k=k, v=v, lens=lens,
                          scale=c["scale"], out=out, lse=lse))
    return built


def check_golden(case):
    out, lse = oracle.decode(case["q"], case["k"], case["v"], case["scale"], seq_lens=case["lens"])
    np.testing.assert_allclose(out, case["out"], rtol=0, atol=1e-13, err_msg=case["name"])
    both_inf = np.isneginf(lse) & np.isneginf(case["lse"])
    assert np.array_equal(np.isneginf(lse), np.isneginf(case["lse"])), case["name"]
    np.testing.assert_allclose(lse[~both_inf], case["lse"][~both_inf], rtol=0, atol=1e-13,
                               err_msg=case["name"])


# ------------------------------------------------------------------ helpers
def _rng(seed):
    return np.random.default_rng(seed)


def random_problem(seed, B=2, Hq=4, Hkv=2, D=8, T=37, lens=None, gain=1.0):
    r = _rng(seed)
    q = r.standard_normal((B, Hq, D)) * gain
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    if lens is None:
        lens = [int(x) for x in r.integers(1, T + 1, size=B)]
    return q, k, v, lens


# ------------------------------------------------------------- closed forms
def check_single_key():
    r = _rng(1)
    q = r.standard_normal((1, 2, 16))
    k = r.standard_normal((1, 1, 1, 16))
    v = r.standard_normal((1, 1, 1, 16))
    out, lse = oracle.decode(q, k, v, 0.25)
    for h in range(2):
        assert np.array_equal(out[0, h], v[0, 0, 0])
        assert abs(lse[0, h] - 0.25 * float(q[0, h] @ k[0, 0, 0])) < 1e-13


def check_identical_keys_mean():
    r = _rng(2)
    q = r.standard_normal((1, 1, 8))
    row = r.standard_normal(8)
    k = np.broadcast_to(row, (1, 1, 50, 8)).copy()
    v = r.standard_normal((1, 1, 50, 8))
    out, lse = oracle.decode(q, k, v, 0.3)
    np.testing.assert_allclose(out[0, 0], v[0, 0].mean(axis=0), rtol=0, atol=1e-14)
    s = 0.3 * float(q[0, 0] @ row)
    assert abs(lse[0, 0] - (s + math.log(50))) < 1e-12


def check_constant_v():
    q, k, v, lens = random_problem(3, T=40)
    v[:] = 2.5
    out, _ = oracle.decode(q, k, v, 0.4, seq_lens=lens)
    np.testing.assert_allclose(out, 2.5, rtol=0, atol=1e-13)


def check_peaked_returns_v0():
    r = _rng(4)
    D = 16
    k = r.standard_normal((1, 1, 30, D))
    q = (k[0, 0, 7] * 400.0)[None, None, :]
    v = r.standard_normal((1, 1, 30, D))
    out, _ = oracle.decode(q, k, v, 1.0)
    np.testing.assert_allclose(out[0, 0], v[0, 0, 7], rtol=0, atol=1e-15)


def check_hull():
    q, k, v, lens = random_problem(5, B=3, T=64, gain=3.0)
    out, _ = oracle.decode(q, k, v, 0.35, seq_lens=lens)
    g = q.shape[1] // k.shape[1]
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            rows = v[b, h // g, :lens[b]]
            assert np.all(out[b, h] <= rows.max(axis=0) + 1e-12)
            assert np.all(out[b, h] >= rows.min(axis=0) - 1e-12)


# ---------------------------------------------------------- shift invariance
def check_shift_invariance():
    q, k, v, lens = random_problem(6, B=2, Hq=2, Hkv=2, T=33)
    scale = 0.37
    out0, lse0 = oracle.decode(q, k, v, scale, seq_lens=lens)
    for c in (-3.0, 0.5, 11.0):
        k2 = k.copy()
        for b in range(2):
            for h in range(2):
                # k_t + u with q.u = c / scale adds exactly c to every scaled score.
                u = (c / scale) * q[b, h] / float(q[b, h] @ q[b, h])
                k2[b, h] += u
        out1, lse1 = oracle.decode(q, k2, v, scale, seq_lens=lens)
        np.testing.assert_allclose(out1, out0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse1, lse0 + c, rtol=0, atol=1e-11)


# ---------------------------------------------------------- split independence
def check_split_independence():
    q, k, v, lens = random_problem(7, B=2, Hq=2, Hkv=1, T=70, gain=2.0)
    lens = [70, 23]
    scale = 0.5
    out_ref, lse_ref = oracle.decode(q, k, v, scale, seq_lens=lens)
    for size in (1, 2, 3, 7, 16, 23, 64, 70, 100):
        for b in range(2):
            for h in range(2):
                L = lens[b]
                parts = [oracle.split_state(q[b, h], k[b, 0, lo:min(lo + size, L)],
                                            v[b, 0, lo:min(lo + size, L)], scale)
                         for lo in range(0, max(L, 1), size)]
                parts.append(oracle.split_state(q[b, h], k[b, 0, :0], v[b, 0, :0], scale))
                o = np.stack([p[0] for p in parts])
                m = np.array([p[1] for p in parts])
                l = np.array([p[2] for p in parts])
                out, lse = oracle.combine(o, m, l)
                np.testing.assert_allclose(out, out_ref[b, h], rtol=0, atol=1e-12)
                assert abs(lse - lse_ref[b, h]) < 1e-12


def check_split_partials_layout():
    q, k, v, lens = random_problem(8, B=3, Hq=4, Hkv=2, T=90)
    lens = [90, 1, 45]
    scale = 0.3
    out_ref, lse_ref = oracle.decode(q, k, v, scale, seq_lens=lens)
    for n_splits in (1, 2, 3, 5, 9):
        o, m, l = oracle.split_partials(q, k, v, scale, n_splits, seq_lens=lens, max_seq_len=90)
        size = oracle.explicit_split_size(90, n_splits)
        assert size % 16 == 0 and size * n_splits >= 90
        # every key is in exactly one split: the split sums of exp(s - M) add up to L
        for b in range(3):
            for h in range(4):
                out, lse = oracle.combine(o[b, h], m[b, h], l[b, h])
                np.testing.assert_allclose(out, out_ref[b, h], rtol=0, atol=1e-12)
                assert abs(lse - lse_ref[b, h]) < 1e-12
                for s in range(n_splits):
                    lo, hi = s * size, min((s + 1) * size, lens[b])
                    count = max(0, hi - lo)
                    if count == 0:
                        assert m[b, h, s] == -math.inf and l[b, h, s] == 0
                    else:
                        assert 1.0 - 1e-12 <= l[b, h, s] <= count + 1e-12


def check_online_softmax_matches():
    q, k, v, lens = random_problem(9, B=1, Hq=1, Hkv=1, T=200, gain=3.0)
    scale = 0.6
    o_ref, m_ref, l_ref = oracle.split_state(q[0, 0], k[0, 0], v[0, 0], scale)
    for tile in (1, 3, 16, 64, 128, 500):
        o, m, l = oracle.online_softmax_state(q[0, 0], k[0, 0], v[0, 0], scale, tile)
        assert m == m_ref
        assert abs(l - l_ref) < 1e-12 * l_ref
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)


def check_empty_splits_and_sequences():
    o = np.zeros((3, 4))
    m = np.full(3, -math.inf)
    l = np.zeros(3)
    out, lse = oracle.combine(o, m, l)
    assert np.array_equal(out, np.zeros(4)) and lse == -math.inf
    q, k, v, _ = random_problem(10, B=2, Hq=2, Hkv=2, T=5)
    out, lse = oracle.decode(q, k, v, 1.0, seq_lens=[0, 5])
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1]))


# ------------------------------------------------------------- brute force
def check_brute_force_mpmath():
    mpmath = __import__("mpmath")
    mpmath.mp.dps = 50
    for seed in range(6):
        r = _rng(100 + seed)
        L = int(r.integers(1, 9))
        D = int(r.integers(1, 5))
        q = r.standard_normal((1, 1, D)) * 2
        k = r.standard_normal((1, 1, L, D))
        v = r.standard_normal((1, 1, L, D))
        scale = float(r.uniform(0.1, 1.5))
        out, lse = oracle.decode(q, k, v, scale)
        e = [mpmath.exp(mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[0, 0, d]) * mpmath.mpf(k[0, 0, t, d])
                                                          for d in range(D))) for t in range(L)]
        den = mpmath.fsum(e)
        for d in range(D):
            num = mpmath.fsum(e[t] * mpmath.mpf(v[0, 0, t, d]) for t in range(L))
            assert abs(float(num / den) - out[0, 0, d]) <= 1e-14 * (1 + abs(out[0, 0, d]))
        assert abs(float(mpmath.log(den)) - lse[0, 0]) <= 1e-13 * (1 + abs(lse[0, 0]))


# ------------------------------------------------------- library cross-check
def check_torch_sdpa():
    import torch
    import torch.nn.functional as F
    for Hq, Hkv in ((4, 4), (8, 2), (6, 3), (8, 1)):
        q, k, v, lens = random_problem(20 + Hq + Hkv, B=2, Hq=Hq, Hkv=Hkv, D=16, T=41)
        scale = 0.25
        out, lse = oracle.decode(q, k, v, scale, seq_lens=lens)
        g = Hq // Hkv
        for b in range(2):
            L = lens[b]
            qt = torch.from_numpy(q[b][None, :, None, :])
            kt = torch.from_numpy(k[b, :, :L][None]).repeat_interleave(g, dim=1)
            vt = torch.from_numpy(v[b, :, :L][None]).repeat_interleave(g, dim=1)
            ref = F.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0, :].numpy()
            np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-13)
            logits = (torch.einsum("hd,htd->ht", qt[0, :, 0], kt[0]) * scale)
            np.testing.assert_allclose(lse[b], torch.logsumexp(logits, dim=-1).numpy(), rtol=0,
                                       atol=1e-12)


# ------------------------------------------------------------ paged identity
def check_paged_matches_gather():
    r = _rng(30)
    B, Hq, Hkv, D, ps = 3, 4, 2, 8, 4
    lens = [13, 4, 1]
    npages = sum(-(-L // ps) for L in lens)
    pool_k = r.standard_normal((npages + 2, Hkv, ps, D))
    pool_v = r.standard_normal((npages + 2, Hkv, ps, D))
    perm = r.permutation(npages + 2)
    table = np.full((B, 5), -1, dtype=np.int64)
    cur = 0
    for b, L in enumerate(lens):
        n = -(-L // ps)
        table[b, :n] = perm[cur:cur + n]
        cur += n
    # independent gather: walk each sequence page by page
    T = max(lens)
    k = np.zeros((B, Hkv, T, D))
    v = np.zeros((B, Hkv, T, D))
    for b, L in enumerate(lens):
        for t in range(L):
            page, row = table[b][t // ps], t % ps
            k[b, :, t] = pool_k[page, :, row]
            v[b, :, t] = pool_v[page, :, row]
    q = r.standard_normal((B, Hq, D))
    out_c, lse_c = oracle.decode(q, k, v, 0.5, seq_lens=lens)
    out_p, lse_p = oracle.decode(q, pool_k, pool_v, 0.5, seq_lens=lens, block_table=table, page_size=ps)
    assert np.array_equal(out_c, out_p) and np.array_equal(lse_c, lse_p)
    # entries past ceil(L / page) are never read: poison them and the pages nobody owns
    table2 = table.copy()
    table2[table2 < 0] = 10 ** 9
    pool_k2, pool_v2 = pool_k.copy(), pool_v.copy()
    unused = sorted(set(range(npages + 2)) - set(table[table >= 0].tolist()))
    pool_k2[unused] = np.nan
    pool_v2[unused] = np.nan
    out_p2, lse_p2 = oracle.decode(q, pool_k2, pool_v2, 0.5, seq_lens=lens, block_table=table2,
                                   page_size=ps)
    assert np.array_equal(out_p2, out_p) and np.array_equal(lse_p2, lse_p)


# ------------------------------------------------------------ several query rows
def check_rows_against_sdpa_with_mask():
    """Multi-row decode equals SDPA (float64) under the explicit per-row key mask."""
    import torch
    import torch.nn.functional as F
    for causal in (True, False):
        for Hq, Hkv, n_q in ((4, 4, 3), (8, 2, 2), (8, 1, 5)):
            r = _rng(40 + Hq + n_q)
            B, D, T = 2, 8, 23
            q = r.standard_normal((B, Hq, n_q, D))
            k = r.standard_normal((B, Hkv, T, D))
            v = r.standard_normal((B, Hkv, T, D))
            lens = [23, 9]
            out, lse = oracle.decode_rows(q, k, v, 0.3, causal=causal, seq_lens=lens)
            g = Hq // Hkv
            for b in range(B):
                L = lens[b]
                kt = torch.from_numpy(k[b, :, :L][None]).repeat_interleave(g, dim=1)
                vt = torch.from_numpy(v[b, :, :L][None]).repeat_interleave(g, dim=1)
                mask = torch.ones(n_q, L, dtype=torch.bool)
                if causal:  # row i sees keys t <= L - n_q + i
                    mask = torch.arange(L)[None, :] <= (L - n_q + torch.arange(n_q))[:, None]
                ref = F.scaled_dot_product_attention(torch.from_numpy(q[b][None]), kt, vt, attn_mask=mask,
                                                     scale=0.3)[0].numpy()
                np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-13)


def check_rows_reduce_to_single_row():
    """One query row (or the last causal row) is plain decode; rows past the keys are empty."""
    q, k, v, lens = random_problem(41, B=2, Hq=4, Hkv=2, D=8, T=30)
    lens = [30, 2]
    o1, l1 = oracle.decode(q, k, v, 0.5, seq_lens=lens)
    o2, l2 = oracle.decode_rows(q[:, :, None, :], k, v, 0.5, seq_lens=lens)
    assert np.array_equal(o1, o2[:, :, 0]) and np.array_equal(l1, l2[:, :, 0])
    q4 = _rng(42).standard_normal((2, 4, 4, 8))
    o4, l4 = oracle.decode_rows(q4, k, v, 0.5, causal=True, seq_lens=lens)
    ol, ll = oracle.decode(q4[:, :, -1], k, v, 0.5, seq_lens=lens)
    assert np.array_equal(o4[:, :, -1], ol) and np.array_equal(l4[:, :, -1], ll)
    # sequence 1 has 2 keys and 4 causal rows: rows 0 and 1 see no key
    assert np.all(o4[1, :, :2] == 0) and np.all(np.isneginf(l4[1, :, :2]))
    assert oracle.row_key_limit(2, 4, 2, True) == 1 and oracle.row_key_limit(2, 4, 0, False) == 2


def _gather_rows(cache, b, kvh, n, table=None, page=None):
    """First n rows of (b, kvh), gathered here with its own indexing (not the oracle's)."""
    cache = np.asarray(cache, dtype=np.float64)
    if table is None:
        return cache[b, kvh, :n]
    return np.stack([cache[int(table[b][t // page]), kvh, t % page] for t in range(n)]) if n else \
        np.zeros((0, cache.shape[-1]))


def check_append_decode_against_sdpa():
    """Fused append + decode equals SDPA (float64) over the old keys followed by the new one."""
    import torch
    import torch.nn.functional as F
    for paged in (False, True):
        r = _rng(77 + paged)
        B, Hq, Hkv, D, page = 3, 6, 2, 8, 4
        lens = [0, 5, 11]
        if paged:
            npg = [-(-(L + 1) // page) for L in lens]
            perm = r.permutation(sum(npg) + 2)
            table = np.full((B, 4), -1)
            c = 0
            for b, n in enumerate(npg):
                table[b, :n] = perm[c:c + n]
                c += n
            k = r.standard_normal((sum(npg) + 2, Hkv, page, D))
            v = r.standard_normal((sum(npg) + 2, Hkv, page, D))
            kw = dict(block_table=table, page_size=page, max_seq_len=max(lens))
        else:
            table = None
            k = r.standard_normal((B, Hkv, 12, D))
            v = r.standard_normal((B, Hkv, 12, D))
            kw = dict(max_seq_len=max(lens))
        q = r.standard_normal((B, Hq, D))
        k_new = r.standard_normal((B, Hkv, D))
        v_new = r.standard_normal((B, Hkv, D))
        out, lse, _, _ = oracle.append_decode(q, k, v, k_new, v_new, 0.4, seq_lens=lens, **kw)
        g = Hq // Hkv
        for b in range(B):
            L = lens[b]
            ks = np.stack([np.concatenate([_gather_rows(k, b, j, L, table, page), k_new[b, j][None]]) for j in range(Hkv)])
            vs = np.stack([np.concatenate([_gather_rows(v, b, j, L, table, page), v_new[b, j][None]]) for j in range(Hkv)])
            kt = torch.from_numpy(ks[None]).repeat_interleave(g, dim=1)
            vt = torch.from_numpy(vs[None]).repeat_interleave(g, dim=1)
            qt = torch.from_numpy(q[b][None, :, None, :])
            ref = F.scaled_dot_product_attention(qt, kt, vt, scale=0.4)[0, :, 0].numpy()
            np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-13)
            s = 0.4 * np.einsum("hd,htd->ht", q[b], kt[0].numpy())
            np.testing.assert_allclose(lse[b], np.log(np.exp(s).sum(-1)), rtol=0, atol=1e-12)
        # the empty sequence sees only the new key: out = v_new, lse = scale * q . k_new
        np.testing.assert_array_equal(out[0], np.repeat(v_new[0], g, axis=0))


def check_append_writes_one_row():
    """The append changes exactly the row at position L_b of every (b, KV head), to the new values."""
    for paged in (False, True):
        r = _rng(91 + paged)
        B, Hkv, D, page = 2, 3, 4, 4
        lens = [3, 8]
        if paged:
            table = np.array([[5, 1, 7], [2, 6, 0]])
            k = r.standard_normal((9, Hkv, page, D))
            v = r.standard_normal((9, Hkv, page, D))
            kw = dict(block_table=table, page_size=page, max_seq_len=8)
            where = {0: (5, 3), 1: (0, 0)}  # L=3: page table[0][0]=5, row 3; L=8: page table[1][2]=0, row 0
        else:
            k = r.standard_normal((B, Hkv, 10, D))
            v = r.standard_normal((B, Hkv, 10, D))
            kw = dict(max_seq_len=8)
        k_new = r.standard_normal((B, Hkv, D))
        v_new = r.standard_normal((B, Hkv, D))
        k2, v2 = oracle.append_kv(k, v, k_new, v_new, seq_lens=lens, **kw)
        changed = np.argwhere(np.any(k2 != k, axis=-1))
        expect = []
        for b in range(B):
            for j in range(Hkv):
                expect.append((where[b][0], j, where[b][1]) if paged else (b, j, lens[b]))
                idx = expect[-1]
                np.testing.assert_array_equal(k2[idx], k_new[b, j])
                np.testing.assert_array_equal(v2[idx], v_new[b, j])
        assert sorted(map(tuple, changed.tolist())) == sorted(expect)
        assert np.count_nonzero(np.any(v2 != v, axis=-1)) == len(expect)


ALL_CHECKS = [
    check_single_key,
    check_identical_keys_mean,
    check_constant_v,
    check_peaked_returns_v0,
    check_hull,
    check_shift_invariance,
    check_split_independence,
    check_split_partials_layout,
    check_online_softmax_matches,
    check_empty_splits_and_sequences,
    check_brute_force_mpmath,
    check_torch_sdpa,
    check_paged_matches_gather,
    check_rows_against_sdpa_with_mask,
    check_rows_reduce_to_single_row,
    check_append_decode_against_sdpa,
    check_append_writes_one_row,
]


def run_golden():
    for case in load_golden():
        check_golden(case)
