"""Seeded synthetic inputs for decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both sides of every parity check (the CUDA library and
the float64 oracle) read the tensors it returns, so a mismatch can only come
from one of the two implementations.

Recipe (every draw comes from ``torch.Generator`` objects seeded with
``seed = 1000 + config_id`` unless a seed is passed):

1. Structure first, on a CPU generator: per-sequence lengths, then (paged) a
   ``torch.randperm`` of the page pool handed out in order to each sequence's
   logical pages; unused block-table slots hold -1.
2. Values second, on a generator living on the target device: ``q`` (fp32,
   N(0,1), times ``q_gain``), then ``K``, then ``V`` (N(0,1) drawn in fp32 and
   rounded once to the cache dtype).
3. The oracle receives exactly these rounded values (widened to float64).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["CaseSpec", "CONFIGS", "Case", "config_spec", "make_case", "small_spec", "poison_padding"]


@dataclasses.dataclass(frozen=True)
class CaseSpec:
    """Shape and structure of one decode-attention workload."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T_cap: int  # contiguous capacity, or the longest allowed sequence when paged
    kv_dtype: str = "bf16"  # "bf16" or "f32"
    layout: str = "contiguous"  # "contiguous" or "paged"
    page_size: int = 16
    lengths: str = "full"  # "full", "uniform:<lo>:<hi>", "loguniform:<lo>:<hi>"
    q_gain: float = 1.0
    n_splits: int = 0  # 0 = let the library plan the splits
    seed: int = 1000

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


# The five workloads: tiny MHA, long peaked MHA, 128k GQA, ragged GQA, paged serving.
CONFIGS = {
    1: CaseSpec("tiny_mha_fp32_T1024", B=1, Hq=4, Hkv=4, D=64, T_cap=1024, kv_dtype="f32",
                n_splits=4, seed=1001),
    2: CaseSpec("long_mha_peaked_T32768", B=1, Hq=32, Hkv=32, D=128, T_cap=32768, q_gain=4.0,
                seed=1002),
    3: CaseSpec("gqa128k_B1_Hq32_Hkv8_T131072", B=1, Hq=32, Hkv=8, D=128, T_cap=131072,
                seed=1003),
    4: CaseSpec("ragged_gqa_B16_T16384", B=16, Hq=32, Hkv=8, D=128, T_cap=16384,
                lengths="uniform:1024:16384", seed=1004),
    5: CaseSpec("paged_B64_Hq64_Hkv8_page16", B=64, Hq=64, Hkv=8, D=128, T_cap=65536,
                layout="paged", page_size=16, lengths="loguniform:512:65536", seed=1005),
}


def config_spec(config_id: int) -> CaseSpec:
    return CONFIGS[config_id]


def small_spec(name: str, B: int, Hq: int, Hkv: int, D: int, T_cap: int, *, kv_dtype="bf16",
               layout="contiguous", page_size=16, lengths="full", q_gain=1.0, n_splits=0,
               seed=7) -> CaseSpec:
    return CaseSpec(name, B, Hq, Hkv, D, T_cap, kv_dtype, layout, page_size, lengths, q_gain,
                    n_splits, seed)


@dataclasses.dataclass
class Case:
    spec: CaseSpec
    q: torch.Tensor  # [B, Hq, D] fp32
    k: torch.Tensor  # contiguous [B, Hkv, T_cap, D]; paged [num_pages, Hkv, page_size, D]
    v: torch.Tensor
    seq_lens: Optional[torch.Tensor]  # [B] int32 (None = every sequence is T_cap long)
    block_table: Optional[torch.Tensor]  # [B, max_pages] int32, paged only
    max_seq_len: int

    @property
    def lengths(self):
        if self.seq_lens is None:
            return [self.max_seq_len] * self.spec.B
        return [int(x) for x in self.seq_lens.cpu().tolist()]

    def kv_bytes(self) -> int:
        """Bytes of K and V over the valid positions only."""
        es = self.k.element_size()
        return sum(self.lengths) * self.spec.Hkv * self.spec.D * 2 * es


def _draw_lengths(spec: CaseSpec, gen: torch.Generator):
    if spec.lengths == "full":
        return None
    kind, lo, hi = spec.lengths.split(":")
    lo, hi = int(lo), int(hi)
    if kind == "uniform":
        return torch.randint(lo, hi + 1, (spec.B,), generator=gen, dtype=torch.int64)
    if kind == "loguniform":
        u = torch.rand(spec.B, generator=gen, dtype=torch.float64)
        lens = torch.floor(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))))
        return lens.clamp(lo, hi).to(torch.int64)
    if kind == "list":
        raise ValueError("use make_case(lengths=...) for explicit lengths")
    raise ValueError(f"unknown length recipe {spec.lengths!r}")


def _cache_dtype(name: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _randn(shape, gen, device, dtype):
    """N(0,1) drawn in fp32 and rounded once to ``dtype``, in slices to bound temporaries."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    step = 1 << 27
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out


def make_case(spec: CaseSpec, device="cpu", lengths=None) -> Case:
    """Draw one workload on ``device`` following the recipe in the module docstring.

    ``lengths`` (a list of ints) overrides the spec's length recipe; explicit
    lengths make edge cases (zeros, one token, page-boundary tails) easy to state.
    """
    device = torch.device(device)
    cpu_gen = torch.Generator().manual_seed(spec.seed)
    lens = torch.tensor(lengths, dtype=torch.int64) if lengths is not None else _draw_lengths(spec, cpu_gen)
    if lens is not None:
        lens = lens.clamp(0, spec.T_cap)
    kv_dtype = _cache_dtype(spec.kv_dtype)

    block_table = None
    if spec.layout == "paged":
        if lens is None:
            lens = torch.full((spec.B,), spec.T_cap, dtype=torch.int64)
        pages_per_seq = [(-(-int(x) // spec.page_size)) for x in lens.tolist()]
        num_pages = max(1, sum(pages_per_seq))
        max_pages = max(1, -(-spec.T_cap // spec.page_size))
        perm = torch.randperm(num_pages, generator=cpu_gen)
        table = torch.full((spec.B, max_pages), -1, dtype=torch.int32)
        cursor = 0
        for b, npg in enumerate(pages_per_seq):
            table[b, :npg] = perm[cursor:cursor + npg].to(torch.int32)
            cursor += npg
        block_table = table.to(device)
        kv_shape = (num_pages, spec.Hkv, spec.page_size, spec.D)
    else:
        kv_shape = (spec.B, spec.Hkv, spec.T_cap, spec.D)

    dev_gen = torch.Generator(device=device).manual_seed(spec.seed)
    q = torch.randn((spec.B, spec.Hq, spec.D), generator=dev_gen, device=device,
                    dtype=torch.float32) * spec.q_gain
    k = _randn(kv_shape, dev_gen, device, kv_dtype)
    v = _randn(kv_shape, dev_gen, device, kv_dtype)
    seq_lens = None if lens is None else lens.to(torch.int32).to(device)
    max_seq_len = spec.T_cap if lens is None else max(1, int(lens.max()))
    if spec.layout == "contiguous" and lens is None:
        max_seq_len = spec.T_cap
    return Case(spec, q, k, v, seq_lens, block_table, max_seq_len)


def poison_padding(case: Case, value=float("nan")) -> Case:
    """Copy of ``case`` whose never-read cache positions hold ``value``.

    Contiguous: every row at or beyond ``L_b``.  Paged: rows beyond ``L_b`` in
    each sequence's last page, plus one extra page appended to the pool that no
    block-table entry points at.  A correct kernel produces bit-identical output
    for the poisoned and the clean case.
    """
    k, v = case.k.clone(), case.v.clone()
    lens = case.lengths
    if case.spec.layout == "contiguous":
        for b, L in enumerate(lens):
            k[b, :, L:, :] = value
            v[b, :, L:, :] = value
        return Case(case.spec, case.q, k, v, case.seq_lens, case.block_table, case.max_seq_len)
    ps = case.spec.page_size
    table = case.block_table.cpu()
    for b, L in enumerate(lens):
        if L % ps:
            page = int(table[b, L // ps])
            k[page, :, L % ps:, :] = value
            v[page, :, L % ps:, :] = value
    extra = torch.full((1,) + tuple(k.shape[1:]), value, dtype=k.dtype, device=k.device)
    k = torch.cat([k, extra])
    v = torch.cat([v, extra])
    return Case(case.spec, case.q, k, v, case.seq_lens, case.block_table, case.max_seq_len)
