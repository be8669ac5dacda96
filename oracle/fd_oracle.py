"""Plain float64 CPU oracle for single-query-row decode attention (Flash-Decoding).

TEST INFRASTRUCTURE ONLY. This module is the yardstick the CUDA path is measured
against; it is not part of the product. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it. The
CUDA library never calls it, and it shares no code, table or helper with the
CUDA library: it depends on NumPy alone.

What it computes (per batch ``b`` and query head ``h``)::

    out[b, h, :] = softmax(scale * q[b, h, :] . K_b^T) . V_b      (over t < L_b)
    lse[b, h]    = log(sum_t exp(scale * q[b, h, :] . k_t))          (natural log)

Sources, by page title and section:

* "Kernel visualization: Flash Decoding" (tinyvolt.com), the ``fd_split`` code
  block: per-split online softmax with running max ``m``, running sum ``l`` and
  an *unnormalised* output ``O`` (the text under "Write partial" says nothing is
  divided inside a split).
* the same page, "Combine kernel -- one thread block per (batch, head)": the
  merge ``M = max_s m_s``, ``L = sum_s exp(m_s - M) l_s``,
  ``O = sum_s exp(m_s - M) O_s / L``.
* "attn-flash-decoding" quiz page (zenaique.com), the answer to "Why does the
  log-sum-exp combine give an exact result": softmax is shift invariant, so
  the merged result equals the unsplit softmax exactly.  Because of that, the
  primary oracle here is the plain two-pass definition (max, then sum), and the
  split/online forms are kept beside it so that tests can show all three agree.
* the same quiz page, "What decode looks like": Q is (batch, n_heads, 1, d_head)
  and K, V are (batch, n_kv_heads, T, d_head).
* "FlashDecoding and split-KV" (guide.dupenodi.dev), "Walking through it":
  paged or ragged KV layouts and GQA head grouping are named (not specified).

Readings taken where the pages are silent:

* GQA head map: query head ``h`` reads KV head ``h // g`` with ``g = Hq // Hkv``.
* LSE is the natural log of the softmax denominator of the *scaled* scores.
* ``L_b == 0``: ``out = 0`` and ``lse = -inf``.
* A split with no keys carries ``m = -inf, l = 0, O = 0`` and is skipped by the
  merge (so no ``exp(-inf - (-inf))`` is ever formed).
* Paged pool layout ``[num_pages, Hkv, page_size, D]``; logical token ``t`` of
  sequence ``b`` lives in page ``block_table[b, t // page_size]`` at row
  ``t % page_size``.
* Explicit split size: ``S = 16 * ceil(ceil(max_seq_len / n_splits) / 16)``;
  split ``s`` covers tokens ``[s*S, min((s+1)*S, L_b))``.
* Several query rows per sequence ("FlashDecoding and split-KV", "Walking
  through it", lets decode carry a few query rows): the ``n_q`` new tokens are
  the last ``n_q`` keys of the cache; with causal masking row ``i`` attends keys
  ``t < L_b - (n_q-1-i)``, without it every row attends all ``L_b`` keys.
* Fused append-KV (named on the same page, not specified): the new token's key
  and value (already in the cache's dtype) are written at position ``L_b`` of
  sequence ``b`` -- contiguous row ``L_b``, or row ``L_b % page_size`` of page
  ``block_table[b, L_b // page_size]`` -- and the decode then attends the
  ``L_b + 1`` keys.  The lengths passed in are the lengths before the append.

All arithmetic is float64.  Inputs are widened exactly (bf16 and fp32 values are
exactly representable in float64); ``scale`` is taken as given.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "kv_head_for",
    "sequence_rows",
    "scores",
    "attend_row",
    "split_state",
    "online_softmax_state",
    "combine",
    "decode",
    "explicit_split_size",
    "split_partials",
    "row_key_limit",
    "decode_rows",
    "append_kv",
    "append_decode",
]


def kv_head_for(h: int, g: int) -> int:
    """KV head read by query head ``h`` when ``g`` query heads share one KV head.

    Reading taken for "GQA head grouping" ("FlashDecoding and split-KV", section
    "Walking through it"), which names the grouping without fixing the map:
    consecutive query heads share a KV head.
    """
    return h // g


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def sequence_rows(cache, b: int, kvh: int, length: int, block_table=None, page_size=None) -> np.ndarray:
    """The ``length`` valid K (or V) rows of sequence ``b``, KV head ``kvh``, as float64.

    Contiguous cache: ``cache`` is ``[B, Hkv, T_cap, D]`` and the rows are
    ``cache[b, kvh, :length]`` (layout of K/V on the quiz page, "What decode
    looks like").  Paged cache: ``cache`` is ``[num_pages, Hkv, page_size, D]``
    and token ``t`` is row ``t % page_size`` of page ``block_table[b, t // page_size]``.
    Only the first ``ceil(length / page_size)`` block-table entries are read.
    """
    if length == 0:
        return np.zeros((0, np.shape(cache)[-1]), dtype=np.float64)
    if block_table is None:
        return _f64(cache[b, kvh, :length, :])
    t = np.arange(length)
    pages = np.asarray(block_table)[b, t // page_size]
    return _f64(np.asarray(cache)[pages, kvh, t % page_size, :])


def scores(q_row, rows, scale) -> np.ndarray:
    """``s_t = scale * (q . k_t)`` for every row ``k_t`` (the ``Sij = Qi @ Kj.T`` step, times scale)."""
    return float(scale) * (_f64(rows) @ _f64(q_row))


def attend_row(q_row, k_rows, v_rows, scale):
    """Exact softmax attention of one query row over the given rows, two passes.

    Returns ``(out[D], lse)``.  Pass 1 takes the maximum score ``M``; pass 2
    forms ``w_t = exp(s_t - M)``, ``L = sum w_t`` and ``out = sum w_t v_t / L``;
    ``lse = M + ln L``.  With no rows: ``out = 0`` and ``lse = -inf``.
    """
    v_rows = _f64(v_rows)
    if v_rows.shape[0] == 0:
        return np.zeros(v_rows.shape[1], dtype=np.float64), -math.inf
    s = scores(q_row, k_rows, scale)
    m = s.max()
    w = np.exp(s - m)
    denom = w.sum()
    return (w @ v_rows) / denom, m + math.log(denom)


def split_state(q_row, k_rows, v_rows, scale):
    """Per-split state ``(O, m, l)`` of one split, by definition.

    ``m = max_t s_t``, ``l = sum_t exp(s_t - m)``, ``O = sum_t exp(s_t - m) v_t``
    (unnormalised, as the "Write partial" step of the ``fd_split`` walkthrough
    states).  An empty split is ``(0, -inf, 0)``.
    """
    v_rows = _f64(v_rows)
    if v_rows.shape[0] == 0:
        return np.zeros(v_rows.shape[1], dtype=np.float64), -math.inf, 0.0
    s = scores(q_row, k_rows, scale)
    m = s.max()
    w = np.exp(s - m)
    return w @ v_rows, m, w.sum()


def online_softmax_state(q_row, k_rows, v_rows, scale, tile: int):
    """The same ``(O, m, l)`` reached by the online-softmax tile loop of ``fd_split``.

    Walks the rows in tiles of ``tile`` keys.  Per tile: ``m_new = max(m, max_c S_c)``,
    ``alpha = exp(m - m_new)``, ``l = alpha * l + sum_c exp(S_c - m_new)``,
    ``O = alpha * O + sum_c exp(S_c - m_new) v_c``, then ``m = m_new``; state
    starts at ``m = -inf, l = 0, O = 0`` (the ``fd_split`` walkthrough: its
    initialisation step and its per-tile update step).
    """
    k_rows = _f64(k_rows)
    v_rows = _f64(v_rows)
    d = v_rows.shape[1]
    o = np.zeros(d, dtype=np.float64)
    m = -math.inf
    l = 0.0
    for j in range(0, k_rows.shape[0], tile):
        s_tile = scores(q_row, k_rows[j:j + tile], scale)
        m_new = max(m, s_tile.max())
        alpha = math.exp(m - m_new)  # exp(-inf) == 0 on the first tile
        p = np.exp(s_tile - m_new)
        l = alpha * l + p.sum()
        o = alpha * o + p @ v_rows[j:j + tile]
        m = m_new
    return o, m, l


def combine(o_parts, m_parts, l_parts):
    """Log-sum-exp merge of split states (the ``fd_combine`` walkthrough).

    ``o_parts`` is ``[n, D]``, ``m_parts`` and ``l_parts`` are ``[n]``.  Splits
    with ``l == 0`` (no keys) are skipped.  ``M = max m_s``,
    ``L = sum exp(m_s - M) l_s``, ``out = sum exp(m_s - M) O_s / L``,
    ``lse = M + ln L``.  If every split is empty: ``out = 0``, ``lse = -inf``.
    """
    o_parts = _f64(o_parts)
    m_parts = _f64(m_parts)
    l_parts = _f64(l_parts)
    keep = l_parts > 0
    if not keep.any():
        return np.zeros(o_parts.shape[-1], dtype=np.float64), -math.inf
    o_k, m_k, l_k = o_parts[keep], m_parts[keep], l_parts[keep]
    m_glob = m_k.max()
    w = np.exp(m_k - m_glob)
    l_glob = (w * l_k).sum()
    return (w @ o_k) / l_glob, m_glob + math.log(l_glob)


def _lengths(seq_lens, batch: int, default: int):
    if seq_lens is None:
        return [int(default)] * batch
    return [int(x) for x in np.asarray(seq_lens).reshape(-1)]


def decode(q, k, v, scale, seq_lens=None, max_seq_len=None, block_table=None, page_size=None):
    """Reference decode attention for a whole batch.

    ``q``: ``[B, Hq, D]``.  Contiguous: ``k, v``: ``[B, Hkv, T_cap, D]`` and,
    when ``seq_lens`` is None, every sequence has ``max_seq_len`` (default
    ``T_cap``) keys.  Paged: ``k, v``: ``[num_pages, Hkv, page_size, D]`` with
    ``block_table`` ``[B, max_pages]`` and ``seq_lens`` required.
    Returns ``(out [B, Hq, D], lse [B, Hq])`` in float64.
    """
    q = _f64(q)
    batch, hq, d = q.shape
    hkv = np.shape(k)[1]
    g = hq // hkv
    if block_table is None and max_seq_len is None:
        max_seq_len = np.shape(k)[2]
    lens = _lengths(seq_lens, batch, max_seq_len)
    out = np.zeros((batch, hq, d), dtype=np.float64)
    lse = np.full((batch, hq), -math.inf, dtype=np.float64)
    for b in range(batch):
        for kvh in range(hkv):
            k_rows = sequence_rows(k, b, kvh, lens[b], block_table, page_size)
            v_rows = sequence_rows(v, b, kvh, lens[b], block_table, page_size)
            for h in range(hq):
                if kv_head_for(h, g) != kvh:
                    continue
                out[b, h], lse[b, h] = attend_row(q[b, h], k_rows, v_rows, scale)
    return out, lse


def explicit_split_size(max_seq_len: int, n_splits: int) -> int:
    """Tokens per split when the caller fixes ``n_splits`` (reading of the ``S`` template).

    The ``fd_split`` sketch takes the split size ``S`` as a parameter and sets
    ``n_start = s * S``, ``n_end = min(n_start + S, N)``.  The reading used here
    is ``S = ceil(max_seq_len / n_splits)`` rounded up to a multiple of 16 tokens.
    """
    s = -(-int(max_seq_len) // int(n_splits))
    return max(16, -(-s // 16) * 16)


def split_partials(q, k, v, scale, n_splits, seq_lens=None, max_seq_len=None,
                   block_table=None, page_size=None):
    """Per-split states in the partial layout ``O[B, Hq, n_splits, D]``, ``m, l [B, Hq, n_splits]``.

    Split ``s`` of sequence ``b`` covers tokens ``[s*S, min((s+1)*S, L_b))`` with
    ``S = explicit_split_size(max_seq_len, n_splits)``; ``m`` is in the natural
    units of the scaled scores.  Empty splits hold ``(0, -inf, 0)``.
    """
    q = _f64(q)
    batch, hq, d = q.shape
    hkv = np.shape(k)[1]
    g = hq // hkv
    if block_table is None and max_seq_len is None:
        max_seq_len = np.shape(k)[2]
    lens = _lengths(seq_lens, batch, max_seq_len)
    size = explicit_split_size(max_seq_len, n_splits)
    o_part = np.zeros((batch, hq, n_splits, d), dtype=np.float64)
    m_part = np.full((batch, hq, n_splits), -math.inf, dtype=np.float64)
    l_part = np.zeros((batch, hq, n_splits), dtype=np.float64)
    for b in range(batch):
        for kvh in range(hkv):
            k_rows = sequence_rows(k, b, kvh, lens[b], block_table, page_size)
            v_rows = sequence_rows(v, b, kvh, lens[b], block_table, page_size)
            for h in range(hq):
                if kv_head_for(h, g) != kvh:
                    continue
                for s in range(n_splits):
                    lo, hi = s * size, min((s + 1) * size, lens[b])
                    if lo >= hi:
                        continue
                    o_part[b, h, s], m_part[b, h, s], l_part[b, h, s] = split_state(
                        q[b, h], k_rows[lo:hi], v_rows[lo:hi], scale)
    return o_part, m_part, l_part


def row_key_limit(length: int, n_q: int, row: int, causal: bool) -> int:
    """Number of keys row ``row`` of ``n_q`` query rows attends (never below 0).

    Reading for a small batch of query rows per sequence: the rows are the last
    ``n_q`` tokens, already written to the cache, so under causal masking row
    ``i`` sees keys ``t < L_b - (n_q - 1 - i)``; otherwise all ``L_b`` keys.
    """
    lim = length - (n_q - 1 - row) if causal else length
    return max(0, min(lim, length))


def decode_rows(q, k, v, scale, causal=True, seq_lens=None, max_seq_len=None, block_table=None,
                page_size=None):
    """Decode attention with ``n_q`` query rows per (batch, head).

    ``q``: ``[B, Hq, n_q, D]``; other arguments as in :func:`decode`.  Returns
    ``(out [B, Hq, n_q, D], lse [B, Hq, n_q])``; a row with no keys gives zeros
    and ``-inf``.
    """
    q = _f64(q)
    batch, hq, n_q, d = q.shape
    hkv = np.shape(k)[1]
    g = hq // hkv
    if block_table is None and max_seq_len is None:
        max_seq_len = np.shape(k)[2]
    lens = _lengths(seq_lens, batch, max_seq_len)
    out = np.zeros((batch, hq, n_q, d), dtype=np.float64)
    lse = np.full((batch, hq, n_q), -math.inf, dtype=np.float64)
    for b in range(batch):
        for kvh in range(hkv):
            k_rows = sequence_rows(k, b, kvh, lens[b], block_table, page_size)
            v_rows = sequence_rows(v, b, kvh, lens[b], block_table, page_size)
            for h in range(hq):
                if kv_head_for(h, g) != kvh:
                    continue
                for i in range(n_q):
                    lim = row_key_limit(lens[b], n_q, i, causal)
                    out[b, h, i], lse[b, h, i] = attend_row(q[b, h, i], k_rows[:lim], v_rows[:lim], scale)
    return out, lse


def append_kv(k, v, k_new, v_new, seq_lens=None, max_seq_len=None, block_table=None, page_size=None):
    """Caches after writing one new token per (b, KV head) at position ``L_b``.

    ``k_new``, ``v_new``: ``[B, Hkv, D]``.  Returns float64 copies of ``k`` and
    ``v`` in which only the rows at position ``L_b`` (per sequence and KV head)
    differ from the input.
    """
    k2, v2 = _f64(k).copy(), _f64(v).copy()
    k_new, v_new = _f64(k_new), _f64(v_new)
    batch, hkv = k_new.shape[0], k_new.shape[1]
    if block_table is None and max_seq_len is None:
        max_seq_len = np.shape(k)[2] - 1
    lens = _lengths(seq_lens, batch, max_seq_len)
    for b in range(batch):
        t = lens[b]
        for kvh in range(hkv):
            if block_table is None:
                k2[b, kvh, t] = k_new[b, kvh]
                v2[b, kvh, t] = v_new[b, kvh]
            else:
                page = int(block_table[b][t // page_size])
                k2[page, kvh, t % page_size] = k_new[b, kvh]
                v2[page, kvh, t % page_size] = v_new[b, kvh]
    return k2, v2


def append_decode(q, k, v, k_new, v_new, scale, seq_lens=None, max_seq_len=None, block_table=None,
                  page_size=None):
    """Fused append-KV + decode: :func:`append_kv`, then :func:`decode` over ``L_b + 1`` keys.

    Returns ``(out, lse, k_after, v_after)``.
    """
    batch = np.shape(q)[0]
    if block_table is None and max_seq_len is None:
        max_seq_len = np.shape(k)[2] - 1
    lens = _lengths(seq_lens, batch, max_seq_len)
    k2, v2 = append_kv(k, v, k_new, v_new, lens, max_seq_len, block_table, page_size)
    out, lse = decode(q, k2, v2, scale, seq_lens=[x + 1 for x in lens], max_seq_len=max_seq_len + 1,
                      block_table=block_table, page_size=page_size)
    return out, lse, k2, v2
