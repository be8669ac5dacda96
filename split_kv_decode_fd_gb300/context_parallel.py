"""Split-KV decode with every sequence's cache sharded across GPUs (context parallel).

Flash-Decoding cuts one sequence's keys into splits that run in parallel and
merges their partial states with the log-sum-exp combine ("Kernel
visualization: Flash Decoding", the ``fd_split`` walkthrough and "Combine kernel
-- one thread block per (batch, head)").  Nothing in the combine cares where a
split ran, so the same decomposition spans GPUs: rank ``r`` of ``world`` holds
the contiguous slice ``[lo_r, hi_r)`` of every sequence's K/V, computes that
slice's partial state ``(O, m, l)`` with ``fd_split_partial`` (one split), the
states are all-gathered -- the one exchange step, ``B * Hq * (D + 2)`` floats per
rank -- and every rank merges them, in rank order, with ``fd_combine``.

Slices follow the explicit split rule of the library: ``S = 16 * ceil(ceil(L /
world) / 16)``, rank ``r`` gets ``[min(r*S, L), min((r+1)*S, L))``.  A rank whose
slice is empty contributes ``m = -inf, l = 0, O = 0``, which the combine skips.
"""

from __future__ import annotations

from typing import Optional, Sequence, Tuple

__all__ = ["shard_range", "local_lengths", "exchange_partials", "cp_decode"]

SHARD_ALIGN = 16


def shard_range(length: int, world: int, rank: int, align: int = SHARD_ALIGN) -> Tuple[int, int]:
    """Token range ``[lo, hi)`` of a sequence of ``length`` keys held by ``rank``."""
    if world < 1 or not 0 <= rank < world or align < 1:
        raise ValueError("bad world / rank / align")
    length = max(0, int(length))
    per = -(-length // world) if length else 0
    size = -(-per // align) * align
    lo = min(rank * size, length)
    return lo, min(lo + size, length)


def local_lengths(lengths: Sequence[int], world: int, rank: int, align: int = SHARD_ALIGN):
    """Keys of each sequence held by ``rank`` (``hi - lo`` of :func:`shard_range`)."""
    out = []
    for L in lengths:
        lo, hi = shard_range(int(L), world, rank, align)
        out.append(hi - lo)
    return out


def exchange_partials(o_part, m_part, l_part, group=None):
    """All-gather one split's state per rank; returns ``(o, m, l)`` with the ranks' splits in rank order.

    Inputs: ``o_part [B, Hq, 1, D]``, ``m_part`` and ``l_part [B, Hq, 1]`` (the
    ``fd_split_partial`` layout with one split).  Outputs: ``[B, Hq, world, D]``
    and ``[B, Hq, world]``.  One collective: the three are packed into
    ``[B, Hq, D + 2]`` first.  NCCL gathers the CUDA tensors directly; a gloo
    group gathers host tensors, so CUDA inputs are staged through host memory
    there and the result is moved back to the inputs' device.
    """
    import torch
    import torch.distributed as dist

    if o_part.dim() != 4 or o_part.shape[2] != 1:
        raise ValueError("o_part must be [B, Hq, 1, D]")
    B, Hq, _, D = o_part.shape
    packed = torch.cat([o_part[:, :, 0, :], m_part[:, :, :1], l_part[:, :, :1]], dim=-1).contiguous()
    world = dist.get_world_size(group)
    device = packed.device
    if packed.is_cuda and dist.get_backend(group) == "gloo":
        packed = packed.cpu()
    parts = [torch.empty_like(packed) for _ in range(world)]
    dist.all_gather(parts, packed, group=group)
    allp = torch.stack(parts, dim=2).to(device)  # [B, Hq, world, D + 2]
    return allp[..., :D].contiguous(), allp[..., D].contiguous(), allp[..., D + 1].contiguous()


def cp_decode(q, k_local, v_local, *, seq_lens_local=None, max_local_len: Optional[int] = None,
              block_table=None, scale=None, group=None, stream=None):
    """Decode attention over a cache sharded across the ranks of ``group``.

    ``k_local``/``v_local`` hold this rank's slice of every sequence (contiguous
    ``[B, Hkv, T_local, D]`` or a paged pool with ``block_table``), with
    ``seq_lens_local`` keys each (device int32, or None for ``max_local_len``).
    Every rank gets the same ``(out [B, Hq, D], lse [B, Hq])``.
    """
    from . import fdecode as fd

    o, m, l = fd.split_partial(q, k_local, v_local, 1, seq_lens=seq_lens_local, max_seq_len=max_local_len,
                               block_table=block_table, scale=scale, stream=stream)
    o_all, m_all, l_all = exchange_partials(o, m, l, group)
    return fd.combine(o_all, m_all, l_all, stream=stream)
