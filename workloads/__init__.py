"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers and names workload shapes; it holds none
of the attention arithmetic.  Inputs are drawn in float32 from a
``torch.Generator`` seeded per tensor on the requested device, scaled by
``std`` and rounded once to the working dtype, so that the CUDA path and the
oracle receive bit-identical values (the oracle gets an exact float64 copy).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

__all__ = ["normal", "qkv", "prefix_lengths", "Workload", "WORKLOADS"]


def normal(shape, seed: int, std: float = 1.0, dtype=torch.bfloat16,
           device="cpu") -> torch.Tensor:
    """N(0, std^2) samples of ``shape`` from a generator seeded with ``seed``."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32,
                    device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def qkv(rows: int, heads: int, head_dim: int, seed: int, std: float = 1.0,
        dtype=torch.bfloat16, device="cpu"):
    """Token-major Q, K, V of shape [rows][heads][head_dim].

    Q, K and V use seeds 3*seed, 3*seed+1 and 3*seed+2.
    """
    shape = (rows, heads, head_dim)
    return tuple(normal(shape, 3 * seed + k, std, dtype, device)
                 for k in range(3))


def prefix_lengths(batch: int, lo: int, hi: int, seed: int) -> list:
    """Per-sequence prefix lengths m_b ~ U{lo..hi} (inclusive), seeded."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


@dataclass(frozen=True)
class Workload:
    """One named workload: shapes only."""
    name: str
    batch: int
    heads: int
    head_dim: int
    m: int                 # prefix length (or the maximum, when ragged)
    n: int                 # output window
    T: int                 # output tokens
    dtype: str             # "f32" or "bf16"
    std: float = 1.0
    m_range: tuple = None  # (lo, hi) for ragged prefixes
    layers: int = 1
    T_sweep: tuple = field(default=())


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 64, 16, 8, 64, "f32"),
    "single_page_bf16": Workload("single_page_bf16", 1, 10, 128, 288, 128,
                                 6000, "bf16", std=128 ** -0.5),
    "batched_decode_bf16": Workload("batched_decode_bf16", 64, 10, 128, 2048,
                                    128, 4096, "bf16", m_range=(256, 2048)),
    "multipage_prefill_bf16": Workload("multipage_prefill_bf16", 1, 10, 128,
                                       10272, 128, 22496, "bf16", layers=12),
    "decode_sweep_bf16": Workload("decode_sweep_bf16", 32, 10, 128, 2600, 128,
                                  100000, "bf16",
                                  T_sweep=(256, 512, 1024, 2048, 4096, 8192,
                                           16384, 32768, 65536, 100000)),
}
