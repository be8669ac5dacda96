"""Plant plausible mistakes in the oracle (on the CPU) and require that the pins catch each one.

A pin suite that passes a broken oracle pins nothing.  Every mutant below is a
small edit of one oracle function (a dropped term, a wrong sign or index, a
wrong log base); the test applies it with ``monkeypatch`` and runs every pin.
"""

import math

import numpy as np
import pytest

import oracle
import oracle.fd_oracle as fo
import oracle_pins


def _mut_head_map(h, g):
    return h % g


def _mut_no_scale(q_row, rows, scale):
    return np.asarray(rows, dtype=np.float64) @ np.asarray(q_row, dtype=np.float64)


def _mut_lse_without_max(q_row, k_rows, v_rows, scale):
    v_rows = np.asarray(v_rows, dtype=np.float64)
    if v_rows.shape[0] == 0:
        return np.zeros(v_rows.shape[1]), -math.inf
    s = fo.scores(q_row, k_rows, scale)
    w = np.exp(s - s.max())
    return (w @ v_rows) / w.sum(), math.log(w.sum())


def _mut_lse_log2(q_row, k_rows, v_rows, scale):
    v_rows = np.asarray(v_rows, dtype=np.float64)
    if v_rows.shape[0] == 0:
        return np.zeros(v_rows.shape[1]), -math.inf
    s = fo.scores(q_row, k_rows, scale)
    m = s.max()
    w = np.exp(s - m)
    return (w @ v_rows) / w.sum(), m + math.log2(w.sum())


def _mut_combine_sign(o_parts, m_parts, l_parts):
    o_parts, m_parts, l_parts = (np.asarray(x, dtype=np.float64) for x in (o_parts, m_parts, l_parts))
    keep = l_parts > 0
    if not keep.any():
        return np.zeros(o_parts.shape[-1]), -math.inf
    o_k, m_k, l_k = o_parts[keep], m_parts[keep], l_parts[keep]
    M = m_k.max()
    w = np.exp(M - m_k)  # wrong sign
    L = (w * l_k).sum()
    return (w @ o_k) / L, M + math.log(L)


def _mut_combine_no_skip(o_parts, m_parts, l_parts):
    o_parts, m_parts, l_parts = (np.asarray(x, dtype=np.float64) for x in (o_parts, m_parts, l_parts))
    M = m_parts.max()
    w = np.exp(m_parts - M)
    L = (w * l_parts).sum()
    return (w @ o_parts) / L, M + math.log(L)


def _mut_online_no_alpha_l(q_row, k_rows, v_rows, scale, tile):
    k_rows, v_rows = np.asarray(k_rows, float), np.asarray(v_rows, float)
    o, m, l = np.zeros(v_rows.shape[1]), -math.inf, 0.0
    for j in range(0, k_rows.shape[0], tile):
        s = fo.scores(q_row, k_rows[j:j + tile], scale)
        m_new = max(m, s.max())
        alpha = math.exp(m - m_new)
        p = np.exp(s - m_new)
        l = l + p.sum()  # rescale dropped
        o = alpha * o + p @ v_rows[j:j + tile]
        m = m_new
    return o, m, l


def _mut_online_no_alpha_o(q_row, k_rows, v_rows, scale, tile):
    k_rows, v_rows = np.asarray(k_rows, float), np.asarray(v_rows, float)
    o, m, l = np.zeros(v_rows.shape[1]), -math.inf, 0.0
    for j in range(0, k_rows.shape[0], tile):
        s = fo.scores(q_row, k_rows[j:j + tile], scale)
        m_new = max(m, s.max())
        alpha = math.exp(m - m_new)
        p = np.exp(s - m_new)
        l = alpha * l + p.sum()
        o = o + p @ v_rows[j:j + tile]  # rescale dropped
        m = m_new
    return o, m, l


def _mut_paged_index(cache, b, kvh, length, block_table=None, page_size=None):
    if length == 0:
        return np.zeros((0, np.shape(cache)[-1]))
    if block_table is None:
        return np.asarray(cache[b, kvh, :length, :], dtype=np.float64)
    t = np.arange(length)
    pages = np.asarray(block_table)[b, t % page_size]  # wrong index
    return np.asarray(np.asarray(cache)[pages, kvh, t // page_size, :], dtype=np.float64)


def _mut_reads_past_length(cache, b, kvh, length, block_table=None, page_size=None):
    if block_table is None:
        return np.asarray(cache[b, kvh, :length + 1, :], dtype=np.float64)
    return fo.__dict__["_orig_sequence_rows"](cache, b, kvh, length, block_table, page_size)


def _mut_split_size_unrounded(max_seq_len, n_splits):
    return -(-int(max_seq_len) // int(n_splits))


def _mut_transposed_v(q_row, k_rows, v_rows, scale):
    v_rows = np.asarray(v_rows, dtype=np.float64)
    if v_rows.shape[0] == 0:
        return np.zeros(v_rows.shape[1]), -math.inf
    s = fo.scores(q_row, k_rows, scale)
    m = s.max()
    w = np.exp(s - m)
    # uses the keys in place of the values
    return (w @ np.asarray(k_rows, dtype=np.float64)) / w.sum(), m + math.log(w.sum())


def _mut_row_limit_off_by_one(length, n_q, row, causal):
    lim = length - (n_q - row) if causal else length  # one key short
    return max(0, min(lim, length))


def _mut_append_one_early(k, v, k_new, v_new, seq_lens=None, max_seq_len=None, block_table=None, page_size=None):
    lens = [max(0, int(x) - 1) for x in np.asarray(seq_lens).reshape(-1)]  # writes over the last old key
    return fo.__dict__["_orig_append_kv"](k, v, k_new, v_new, lens, max_seq_len, block_table, page_size)


def _mut_append_page_row_swapped(k, v, k_new, v_new, seq_lens=None, max_seq_len=None, block_table=None,
                                 page_size=None):
    if block_table is None:
        return fo.__dict__["_orig_append_kv"](k, v, k_new, v_new, seq_lens, max_seq_len, block_table, page_size)
    k2, v2 = np.asarray(k, dtype=np.float64).copy(), np.asarray(v, dtype=np.float64).copy()
    for b, t in enumerate(np.asarray(seq_lens).reshape(-1)):
        page = int(block_table[b][t % page_size]) if t % page_size < len(block_table[b]) else 0
        for j in range(k2.shape[1]):
            k2[max(page, 0), j, t // page_size % page_size] = k_new[b, j]
            v2[max(page, 0), j, t // page_size % page_size] = v_new[b, j]
    return k2, v2


def _mut_append_decode_skips_new_key(q, k, v, k_new, v_new, scale, seq_lens=None, max_seq_len=None,
                                     block_table=None, page_size=None):
    lens = [int(x) for x in np.asarray(seq_lens).reshape(-1)]
    k2, v2 = fo.append_kv(k, v, k_new, v_new, lens, max_seq_len, block_table, page_size)
    out, lse = fo.decode(q, k2, v2, scale, seq_lens=lens, max_seq_len=max_seq_len, block_table=block_table,
                         page_size=page_size)
    return out, lse, k2, v2


MUTANTS = {
    "append_one_early": {"append_kv": _mut_append_one_early},
    "append_page_row_swapped": {"append_kv": _mut_append_page_row_swapped},
    "append_decode_skips_new_key": {"append_decode": _mut_append_decode_skips_new_key},
    "row_limit_off_by_one": {"row_key_limit": _mut_row_limit_off_by_one},
    "head_map_modulo": {"kv_head_for": _mut_head_map},
    "scale_dropped": {"scores": _mut_no_scale},
    "lse_without_max": {"attend_row": _mut_lse_without_max},
    "lse_log2": {"attend_row": _mut_lse_log2},
    "keys_used_as_values": {"attend_row": _mut_transposed_v},
    "combine_weight_sign": {"combine": _mut_combine_sign},
    "combine_keeps_empty": {"combine": _mut_combine_no_skip},
    "online_l_not_rescaled": {"online_softmax_state": _mut_online_no_alpha_l},
    "online_o_not_rescaled": {"online_softmax_state": _mut_online_no_alpha_o},
    "paged_index_swapped": {"sequence_rows": _mut_paged_index},
    "reads_past_length": {"sequence_rows": _mut_reads_past_length},
    "split_size_unrounded": {"explicit_split_size": _mut_split_size_unrounded},
}


def _run_all_pins():
    failures = []
    for case in oracle_pins.load_golden():
        try:
            oracle_pins.check_golden(case)
        except Exception as e:  # noqa: BLE001 - any failure counts as caught
            failures.append(f"golden:{case['name']}:{type(e).__name__}")
    for check in oracle_pins.ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check()
        except Exception as e:  # noqa: BLE001
            failures.append(f"{check.__name__}:{type(e).__name__}")
    return failures


def test_unmutated_oracle_passes_every_pin():
    assert _run_all_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    monkeypatch.setitem(fo.__dict__, "_orig_sequence_rows", fo.sequence_rows)
    monkeypatch.setitem(fo.__dict__, "_orig_append_kv", fo.append_kv)
    for attr, fn in MUTANTS[name].items():
        monkeypatch.setattr(fo, attr, fn)
        if hasattr(oracle, attr):
            monkeypatch.setattr(oracle, attr, fn)
    failures = _run_all_pins()
    assert failures, f"mutant {name} passed every pin"
