"""Seeded synthetic inputs for the attention forward pass.

This module is the one piece shared by the CUDA path's callers and the oracle's
callers: it draws inputs and describes workloads, and holds none of the
attention arithmetic.  Inputs are drawn on the CPU with a seeded
``torch.Generator`` in the order Q, K, V, as fp32 normals scaled by the stated
standard deviation and rounded to bf16 (round-to-nearest-even).

The pages measure on "26 configurations", "182 scenarios" and "production
request shapes" without giving them (article "L'agent a questions depasse
l'agent a outils : 113% contre 50% de la vitesse de FlashAttention-3", sections
"Ce que cela a donne" and the introduction); the workloads below stand in for
them: LLM training prefill, grouped-query causal, chunked prefill against a long
KV cache, and long context.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    causal: int          # 0 none, 1 bottom-right aligned, 2 top-left aligned
    seed: int
    qk_std: float = 1.0  # standard deviation of Q and K entries
    v_std: float = 1.0   # standard deviation of V entries

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D), as the fp32 value the kernel receives."""
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def label(self) -> str:
        mask = {0: "none", 1: "causal-bottom-right", 2: "causal-top-left"}[self.causal]
        return (f"{self.name}: B={self.B} Hq={self.Hq} Hkv={self.Hkv} Sq={self.Sq} "
                f"Sk={self.Sk} D={self.D} {mask}")


# Workloads: shapes, value distributions and seeds.  For Sq == Sk top-left and
# bottom-right causal alignment coincide; every causal workload uses 1.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 128, 128, 64, 0, seed=0),
    "train": Workload("train", 4, 16, 16, 2048, 2048, 128, 1, seed=1),
    "gqa": Workload("gqa", 2, 32, 8, 8192, 8192, 128, 1, seed=2, qk_std=3.0),
    "chunked128": Workload("chunked128", 8, 32, 8, 512, 16384, 128, 1, seed=3),
    "chunked64": Workload("chunked64", 8, 32, 8, 512, 16384, 64, 1, seed=4),
    "long": Workload("long", 1, 32, 8, 65536, 65536, 128, 1, seed=5),
}


def draw(B, Hq, Hkv, Sq, Sk, D, seed, qk_std=1.0, v_std=1.0):
    """Draw (q, k, v) as CPU bf16 tensors [B,Hq,Sq,D], [B,Hkv,Sk,D], [B,Hkv,Sk,D]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = (torch.randn((B, Hq, Sq, D), generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    k = (torch.randn((B, Hkv, Sk, D), generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    v = (torch.randn((B, Hkv, Sk, D), generator=g, dtype=torch.float32) * v_std).to(torch.bfloat16)
    return q, k, v


def draw_workload(w: Workload):
    return draw(w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.seed, w.qk_std, w.v_std)


def draw_on_device(shape, seed, std=1.0, device="cuda"):
    """One bf16 tensor of N(0, std^2) entries drawn on ``device`` with a seeded generator, one slice of the
    second dimension at a time (fp32 normals, scaled, rounded to bf16 nearest-even).  For inputs of several GB,
    which take too long to draw on the CPU; whoever checks the result copies out the rows it needs."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for h in range(shape[1]):
        out[:, h].copy_(torch.randn(out[:, h].shape, generator=g, dtype=torch.float32, device=device) * std)
    return out


def sample_rows(B, Hq, Sq, per_head, seed):
    """Distinct uniformly drawn query rows per (b, h), always including rows 0 and Sq-1.

    Returns flat row ids ``(b*Hq + h)*Sq + i`` (int64, sorted within each head).
    """
    rng = np.random.default_rng(int(seed))
    out = []
    for bh in range(B * Hq):
        n = min(per_head, Sq)
        if n >= Sq:
            rows = np.arange(Sq, dtype=np.int64)
        else:
            inner = rng.choice(np.arange(1, Sq - 1, dtype=np.int64), size=max(n - 2, 0), replace=False)
            rows = np.unique(np.concatenate([[0, Sq - 1], inner]).astype(np.int64))
        out.append(bh * Sq + rows)
    return np.concatenate(out)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a CPU bf16 tensor as a numpy uint16 array (no copy of values)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_values(values, dtype=torch.bfloat16) -> torch.Tensor:
    """A CPU bf16 tensor from (exactly representable, for pins) numeric values."""
    return torch.as_tensor(np.asarray(values, dtype=np.float32)).to(dtype)


def block_mask_blocks(B: int, Hm: int, Sq: int, Sk: int, density: float, seed: int,
                      keep_diagonal: bool = True, block: int = 128, row_group: int = 1) -> np.ndarray:
    """Seeded random block mask: bool ``[B, Hm, ceil(Sq/block), ceil(Sk/block)]``, each block marked with
    probability ``density`` (blocks on the bottom-right-aligned diagonal always marked when ``keep_diagonal``).
    With ``row_group = g`` each run of g consecutive query blocks shares one draw (the same key blocks)."""
    rng = np.random.default_rng(int(seed))
    QB, KB = -(-Sq // block), -(-Sk // block)
    groups = rng.random((B, Hm, -(-QB // row_group), KB)) < density
    blocks = np.repeat(groups, row_group, axis=2)[:, :, :QB]
    if keep_diagonal:
        off = (Sk - Sq) // block
        for qb in range(QB):
            kb = qb + off
            if 0 <= kb < KB:
                blocks[:, :, qb, kb] = True
    return blocks
