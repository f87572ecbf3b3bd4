"""Seeded synthetic workloads for block-sparse attention.

This module is the only code shared by the fp64 oracle and the CUDA path. It
holds workload *definitions* (shapes, block size, pattern parameters) and the
seeded generators that draw Q, K, V as bf16 bytes. It contains none of the
attention arithmetic: no masks are expanded, no scores are formed, nothing is
pooled or selected here.

Workloads (the five shapes of the method's reference configurations):

* ``tiny_window_global``  B=1 H=2 N=1024 D=64, block 64: key blocks i-1..i+1
  plus global block 0, block 0 attends to all blocks, non-causal.
* ``window_16k``          B=1 H=16 N=16384 D=128, block 128: window of 512
  tokens = key blocks i-4..i+4 clipped, causal.
* ``window_global_64k``   B=1 H=32 N=65536 D=128, block 128: key blocks
  i-63..i plus global blocks 0 and 1, global query blocks attend to everything
  up to themselves, causal.
* ``long_window_128k``    B=1 H=32 N=131072 D=128, block 128, values scaled by
  0.5: key blocks i-31..i plus global block 0 (the 8 sink tokens live in it),
  causal.
* ``content_topk``        B=2 H=16 N=32768 D=128, block 64: clustered Q and K,
  top-16 key blocks by pooled block score plus the diagonal, non-causal.

Draw order (torch CPU generator, ``manual_seed(1000 + index)``), float32 draws
rounded to bf16 with round-to-nearest-even by ``Tensor.to(torch.bfloat16)``:

* plain workloads: Q, then K, then V; each tensor drawn as B*H slabs of
  ``randn(N, D)`` in (b, h) order, multiplied by ``value_scale`` before the
  bf16 rounding;
* ``content_topk``: 32 centroids ``randn(32, D)``; centroid ids
  ``randint(0, 32, (B, H, nb))`` for K, then for Q; then per (b, h) slab the
  noise ``randn(N, D)`` for Q, then for K (each slab adds ``2.0 * centroid`` of
  its block before rounding); then V as N(0, 1) slabs.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence, Tuple

import torch

__all__ = ["Workload", "WORKLOADS", "workload", "make_qkv", "small_workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """A synthetic attention workload: shapes, block size and mask recipe."""

    name: str
    B: int
    H: int
    N: int
    D: int
    block: int
    # Pattern mask parameters (unused when ``topk`` > 0).
    window_left: int = 0
    window_right: int = 0
    causal: bool = False
    global_blocks: Tuple[int, ...] = ()
    global_rows_attend_all: bool = False
    # Global query rows take no causal cut (see every block of the sequence).
    global_rows_noncausal: bool = False
    # Content-based selection parameters.
    topk: int = 0
    include_diag: bool = True
    n_centroids: int = 0
    centroid_gain: float = 0.0
    # Value distribution.
    value_scale: float = 1.0
    seed: int = 1000

    @property
    def n_blocks(self) -> int:
        return self.N // self.block

    @property
    def is_topk(self) -> bool:
        return self.topk > 0

    @property
    def scale(self) -> float:
        return 1.0 / float(self.D) ** 0.5

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Tuple[Workload, ...] = (
    Workload("tiny_window_global", 1, 2, 1024, 64, 64, window_left=1, window_right=1,
             causal=False, global_blocks=(0,), global_rows_attend_all=True, seed=1000),
    Workload("window_16k", 1, 16, 16384, 128, 128, window_left=4, window_right=4,
             causal=True, seed=1001),
    Workload("window_global_64k", 1, 32, 65536, 128, 128, window_left=63, window_right=0,
             causal=True, global_blocks=(0, 1), global_rows_attend_all=True, seed=1002),
    Workload("long_window_128k", 1, 32, 131072, 128, 128, window_left=31, window_right=0,
             causal=True, global_blocks=(0,), global_rows_attend_all=True,
             value_scale=0.5, seed=1003),
    Workload("content_topk", 2, 16, 32768, 128, 64, causal=False, topk=16, include_diag=True,
             n_centroids=32, centroid_gain=2.0, seed=1004),
)


def workload(name_or_index) -> Workload:
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    for w in WORKLOADS:
        if w.name == name_or_index:
            return w
    raise KeyError(name_or_index)


def small_workload(base: Workload, *, B: Optional[int] = None, H: Optional[int] = None,
                   N: Optional[int] = None, seed: Optional[int] = None, **kw) -> Workload:
    """A reduced copy of ``base`` (same pattern recipe) for fast parity checks."""
    return base.with_(B=B if B is not None else base.B, H=H if H is not None else base.H,
                      N=N if N is not None else base.N,
                      seed=seed if seed is not None else base.seed, **kw)


def _slabs(gen: torch.Generator, B: int, H: int, N: int, D: int, scale: float) -> torch.Tensor:
    out = torch.empty((B, H, N, D), dtype=torch.bfloat16)
    for b in range(B):
        for h in range(H):
            x = torch.randn((N, D), generator=gen, dtype=torch.float32)
            if scale != 1.0:
                x.mul_(scale)
            out[b, h] = x.to(torch.bfloat16)
    return out


def make_qkv(w: Workload) -> Dict[str, torch.Tensor]:
    """Draw Q, K, V (bf16, CPU, contiguous [B, H, N, D]) for workload ``w``."""
    gen = torch.Generator().manual_seed(int(w.seed))
    B, H, N, D, bs = w.B, w.H, w.N, w.D, w.block
    if w.n_centroids > 0:
        nb = N // bs
        cent = torch.randn((w.n_centroids, D), generator=gen, dtype=torch.float32)
        cid_k = torch.randint(0, w.n_centroids, (B, H, nb), generator=gen)
        cid_q = torch.randint(0, w.n_centroids, (B, H, nb), generator=gen)
        q = torch.empty((B, H, N, D), dtype=torch.bfloat16)
        k = torch.empty((B, H, N, D), dtype=torch.bfloat16)
        for b in range(B):
            for h in range(H):
                for dst, cid in ((q, cid_q), (k, cid_k)):
                    z = torch.randn((N, D), generator=gen, dtype=torch.float32)
                    add = cent[cid[b, h]].mul(w.centroid_gain)            # [nb, D]
                    z.view(nb, bs, D).add_(add.unsqueeze(1))
                    dst[b, h] = z.to(torch.bfloat16)
        v = _slabs(gen, B, H, N, D, 1.0)
        return {"q": q, "k": k, "v": v, "centroid_ids_q": cid_q, "centroid_ids_k": cid_k}
    q = _slabs(gen, B, H, N, D, w.value_scale)
    k = _slabs(gen, B, H, N, D, w.value_scale)
    v = _slabs(gen, B, H, N, D, w.value_scale)
    return {"q": q, "k": k, "v": v}


def make_grad_out(w: Workload, seed_offset: int = 500) -> torch.Tensor:
    """Upstream gradient dO for the backward: N(0, 1) bf16 [B, H, N, D] slabs
    in (b, h) order, from its own generator (seed + seed_offset)."""
    gen = torch.Generator().manual_seed(int(w.seed) + seed_offset)
    return _slabs(gen, w.B, w.H, w.N, w.D, 1.0).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of ``t`` as a numpy uint16 array (no copy of values)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(w: Workload, n_random_blocks: int = 16, seed: int = 7,
                blocks: Optional[Sequence[int]] = None):
    """Query rows to check at full size: every (b, h), query blocks {0, 1, 2, nb-1}
    plus ``n_random_blocks`` seeded random ones drawn separately for each
    (b, h), all rows of each chosen block.  ``blocks`` fixes one list for
    every (b, h) instead.

    Returns an int64 tensor of flat row ids ``bh * N + t``.
    """
    nb = w.n_blocks
    gen = torch.Generator().manual_seed(seed)
    fixed = [0, 1, 2, nb - 1]
    rows = []
    t_in = torch.arange(w.block, dtype=torch.int64)
    for bh in range(w.B * w.H):
        if blocks is None:
            extra = torch.randint(0, nb, (n_random_blocks,), generator=gen).tolist()
            blks = sorted(set(b for b in fixed + extra if 0 <= b < nb))
        else:
            blks = list(blocks)
        for blk in blks:
            rows.append(bh * w.N + blk * w.block + t_in)
    return torch.cat(rows)


def head_rows(w: Workload, bh: int):
    """Every query row of head slab ``bh`` as flat row ids ``bh * N + t``."""
    return torch.arange(bh * w.N, (bh + 1) * w.N, dtype=torch.int64)
