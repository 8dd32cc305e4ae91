"""Seeded synthetic inputs shaped like the source pages' workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so the float64 oracle and the CUDA library can both be
fed from it without sharing any of the method's code.

Recipe (identical for every workload):

* one ``torch.Generator`` seeded with ``seed`` (0 by default), drawing in the
  order q, k, v, then the block index list;
* TRA: ``q, k ~ N(0,1) * D**-0.25`` and ``v ~ N(0,1)``, drawn in float32 and
  cast to the workload dtype with round-to-nearest-even;
* NSA: ``q, k, v ~ N(0,1)`` in float32, cast to bfloat16;
* NSA ``block_idx[b, hkv, i, :]``: slot 0 is the block holding ``i``
  (``c = i // block_size``); slots ``1..min(S-1, c)`` are that many distinct
  earlier blocks drawn uniformly without replacement from ``0..c-1`` (the
  ``min(S-1, c)`` smallest of ``c`` independent U(0,1) keys), in ascending
  order; remaining slots are ``-1``.

Tensors are returned on the CPU, contiguous; callers move them to a device.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class TraWorkload:
    """A threshold rectified attention forward workload."""

    name: str
    B: int
    H: int
    T: int
    D: int
    beta: float
    p: float
    dtype: str  # "f32" or "bf16"

    @property
    def flops(self) -> int:
        """Causal FLOPs: 2 multiply-adds of length D per pair (i, j <= i)."""
        return 4 * self.D * self.B * self.H * (self.T * (self.T + 1) // 2)

    @property
    def io_bytes(self) -> int:
        """q, k, v read once and out written once."""
        el = 4 if self.dtype == "f32" else 2
        return 4 * self.B * self.H * self.T * self.D * el


@dataclass(frozen=True)
class NsaWorkload:
    """An NSA selection-branch forward workload."""

    name: str
    B: int
    Hq: int
    Hkv: int
    T: int
    D: int
    block_size: int
    S: int
    extra: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def pairs_per_group(self) -> int:
        """Valid (query, key) pairs of one kv group under this generator:
        query i sees (i % bs + 1) + bs * min(S - 1, i // bs) keys."""
        bs, T, k = self.block_size, self.T, self.S - 1
        n_blk = T // bs
        # sum over blocks c of  [bs*(bs+1)/2 + bs*bs*min(k, c)]
        return sum(bs * (bs + 1) // 2 + bs * bs * min(k, c) for c in range(n_blk))

    @property
    def flops(self) -> int:
        """4 * D FLOPs per (query head, valid key) pair."""
        return 4 * self.D * self.G * self.B * self.Hkv * self.pairs_per_group

    @property
    def algorithmic_bytes(self) -> int:
        """Gathered valid K and V tokens of every query group, plus q and o
        once, the index list and the lse output."""
        B, Hq, Hkv, T, D, S = self.B, self.Hq, self.Hkv, self.T, self.D, self.S
        kv = B * Hkv * self.pairs_per_group * D * 2 * 2
        qo = 2 * B * Hq * T * D * 2
        idx = B * Hkv * T * S * 4
        lse = B * Hq * T * 4
        return kv + qo + idx + lse

    @property
    def unique_bytes(self) -> int:
        """q, o, and every K/V token once (the HBM floor if K/V stay in L2)."""
        B, Hq, Hkv, T, D, S = self.B, self.Hq, self.Hkv, self.T, self.D, self.S
        return 2 * B * Hq * T * D * 2 + 2 * B * Hkv * T * D * 2 + B * Hkv * T * S * 4 + B * Hq * T * 4


TRA_WORKLOADS = {
    w.name: w
    for w in [
        TraWorkload("tra_f32_B1_H2_T256_D64", 1, 2, 256, 64, 1.0, 2.0, "f32"),
        TraWorkload("tra_bf16_B4_H16_T4096_D128", 4, 16, 4096, 128, 1.0, 2.0, "bf16"),
        TraWorkload("tra_bf16_B2_H32_T8192_D64", 2, 32, 8192, 64, 2.0, 1.5, "bf16"),
    ]
}

NSA_WORKLOADS = {
    w.name: w
    for w in [
        NsaWorkload("nsa_bf16_B2_Hq32_Hkv2_T8192_D128", 2, 32, 2, 8192, 128, 64, 16),
        NsaWorkload("nsa_bf16_B1_Hq64_Hkv4_T32768_D128", 1, 64, 4, 32768, 128, 64, 16),
        # A quarter of the T=8192 workload (half the groups, half the length):
        # small enough for multi-pass profiler captures of the split-K form,
        # whose workspace is 1.1 GB here instead of 4.4 GB.
        NsaWorkload("nsa_bf16_B1_Hq32_Hkv2_T4096_D128", 1, 32, 2, 4096, 128, 64, 16),
        # Smaller head dim and blocks (the general kernel's shapes).
        NsaWorkload("nsa_bf16_B2_Hq32_Hkv2_T8192_D32_bs32", 2, 32, 2, 8192, 32, 32, 16),
    ]
}


def _dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def tra_inputs(B: int, H: int, T: int, D: int, dtype: str = "bf16", seed: int = 0, device: str = "cpu"):
    """``(q, k, v)`` tensors ``[B, H, T, D]`` of the TRA recipe, drawn on
    ``device`` (CPU by default; a CUDA device draws its own seeded stream,
    for inputs too large to draw on the host)."""
    g = torch.Generator(device=device).manual_seed(seed)
    shape = (B, H, T, D)
    sc = float(D) ** -0.25
    q = (torch.randn(shape, generator=g, device=device) * sc).to(_dtype(dtype))
    k = (torch.randn(shape, generator=g, device=device) * sc).to(_dtype(dtype))
    v = torch.randn(shape, generator=g, device=device).to(_dtype(dtype))
    return q.contiguous(), k.contiguous(), v.contiguous()


def selection_indices(B: int, Hkv: int, T: int, block_size: int, S: int,
                      generator: torch.Generator, chunk: int = 4096) -> torch.Tensor:
    """``block_idx [B, Hkv, T, S]`` int32 of the synthetic NSA selection
    (current block, then up to ``S-1`` distinct uniformly drawn earlier blocks
    in ascending order, then ``-1`` padding)."""
    n_blk = T // block_size
    k = S - 1
    out = torch.full((B, Hkv, T, S), -1, dtype=torch.int32)
    blk = torch.arange(n_blk)
    for b in range(B):
        for h in range(Hkv):
            for i0 in range(0, T, chunk):
                i1 = min(T, i0 + chunk)
                c = torch.arange(i0, i1) // block_size  # current block per row
                out[b, h, i0:i1, 0] = c.to(torch.int32)
                if k == 0:
                    continue
                u = torch.rand((i1 - i0, n_blk), generator=generator)
                u[blk[None, :] >= c[:, None]] = 2.0  # only earlier blocks
                kk = min(k, n_blk)
                vals, pick = torch.topk(u, kk, dim=1, largest=False)
                pick = torch.where(vals < 2.0, pick, torch.full_like(pick, n_blk))
                pick, _ = torch.sort(pick, dim=1)
                pick = torch.where(pick == n_blk, torch.full_like(pick, -1), pick)
                out[b, h, i0:i1, 1:1 + kk] = pick.to(torch.int32)
    return out.contiguous()


def nsa_inputs(B: int, Hq: int, Hkv: int, T: int, D: int, block_size: int, S: int,
               seed: int = 0, device: str = "cpu"):
    """``(q, k, v, block_idx)`` of the NSA recipe (bf16 / int32).  q, k, v
    are drawn on ``device`` (CPU by default); block_idx is always drawn on
    the host (with the same generator on CPU, a CPU generator of the same
    seed otherwise)."""
    g = torch.Generator(device=device).manual_seed(seed)
    q = torch.randn((B, Hq, T, D), generator=g, device=device).to(torch.bfloat16).contiguous()
    k = torch.randn((B, Hkv, T, D), generator=g, device=device).to(torch.bfloat16).contiguous()
    v = torch.randn((B, Hkv, T, D), generator=g, device=device).to(torch.bfloat16).contiguous()
    gi = g if torch.device(device).type == "cpu" else torch.Generator().manual_seed(seed)
    idx = selection_indices(B, Hkv, T, block_size, S, gi)
    return q, k, v, idx


def shard_range(units: int, world: int, rank: int) -> tuple[int, int]:
    """The contiguous slice [start, end) of ``units`` independent units (the
    (b, h) heads of TRA, the (b, hkv) groups of NSA) that rank ``rank`` of
    ``world`` takes: sizes differ by at most one, and the slices of all ranks
    cover 0..units-1 exactly once."""
    if world < 1 or not 0 <= rank < world or units < 0:
        raise ValueError("shard_range: need 0 <= rank < world and units >= 0")
    base, extra = divmod(units, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_seed(rank: int, seed: int = 0) -> int:
    """Seed of rank ``rank``'s slice of a batch-sharded problem: rank 0 draws
    exactly the single-GPU inputs, the others their own batches."""
    return seed + rank


def workload_inputs(w, seed: int = 0):
    """Inputs of a named workload (a ``TraWorkload`` or ``NsaWorkload``)."""
    if isinstance(w, TraWorkload):
        return tra_inputs(w.B, w.H, w.T, w.D, w.dtype, seed)
    return nsa_inputs(w.B, w.Hq, w.Hkv, w.T, w.D, w.block_size, w.S, seed)
