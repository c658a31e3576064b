"""Seeded synthetic inputs and the named workloads.

This module holds no attention arithmetic: it only draws random tensors.  It
is the one module that both the CUDA path's callers (tests, bench, smoke) and
the oracle-side checks use, so both see identical input bits.

Recipe: a CPU ``torch.Generator`` seeded with the workload's seed draws q, k,
v and dO, in that order, as float32 ``randn * std``; each is then rounded to
the workload's 16-bit dtype (round to nearest even).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch

_TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    dtype: str = "bf16"
    std: float = 1.0
    causal: bool = True
    seed: int = 1000

    @property
    def scale(self) -> float:
        """1/sqrt(D) rounded to float32 (the value the C ABI receives)."""
        return float(np.float32(1.0 / math.sqrt(self.D)))

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPES[self.dtype]

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The workloads, shaped like the ones the pages measure or describe.  The
# last two are long-cache rectangles (few query rows against a long key
# range; "Add a fused full-attention path for head_dim 256 on NAX devices",
# section "Kernel benchmarks", 1024 x 8192 and 2048 x 8192).
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_gqa_l128_d64", B=1, Hq=2, Hkv=1, Lq=128, Lk=128, D=64, seed=1000),
        Workload("llama_gqa_l2048_d128", B=2, Hq=32, Hkv=8, Lq=2048, Lk=2048, D=128, seed=1001),
        Workload("qwen3_8b_gqa_l8192_d128", B=1, Hq=32, Hkv=8, Lq=8192, Lk=8192, D=128, seed=1002),
        Workload("gqa_l8192_d256", B=1, Hq=16, Hkv=2, Lq=8192, Lk=8192, D=256, seed=1003),
        Workload(
            "ragged_mha_q4064_k4112_d96",
            B=4, Hq=16, Hkv=16, Lq=4064, Lk=4112, D=96, dtype="fp16", std=0.5, seed=1004,
        ),
        Workload("longcache_q1024_k8192_d128", B=1, Hq=32, Hkv=8, Lq=1024, Lk=8192, D=128, seed=1006),
        Workload("longcache_q2048_k8192_d256", B=1, Hq=16, Hkv=2, Lq=2048, Lk=8192, D=256, seed=1007),
        # profiling case: the 8192 workload's heads at half the length (160 MB, above L2)
        Workload("qwen3_8b_gqa_l4096_d128", B=1, Hq=32, Hkv=8, Lq=4096, Lk=4096, D=128, seed=1009),
        # decode-shaped: 8 new query rows per sequence against an 8192-key context
        Workload("decode_b4_q8_k8192_d128", B=4, Hq=32, Hkv=8, Lq=8, Lk=8192, D=128, seed=1008),
    ]
}

# Long-context memory check shape (same heads as the 8192 workload).
MEMORY_CHECK = WORKLOADS["qwen3_8b_gqa_l8192_d128"].with_(
    name="qwen3_8b_gqa_l23040_d128_memcheck", Lq=23040, Lk=23040, seed=1005
)


def make_inputs(w: Workload, device: str | torch.device = "cpu"):
    """q, k, v, dO as contiguous [B, H, L, D] tensors of the workload's dtype."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    shapes = [
        (w.B, w.Hq, w.Lq, w.D),
        (w.B, w.Hkv, w.Lk, w.D),
        (w.B, w.Hkv, w.Lk, w.D),
        (w.B, w.Hq, w.Lq, w.D),
    ]
    out = []
    for s in shapes:
        t = torch.randn(s, generator=gen, dtype=torch.float32) * w.std
        out.append(t.to(w.torch_dtype).to(device).contiguous())
    return tuple(out)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact decode of a 16-bit (or fp32) tensor to a float64 numpy array."""
    return t.detach().to("cpu").to(torch.float64).numpy()


def block_mask(spec: str, Lq: int, Lk: int, seed: int = 0, blk: int = 128):
    """A block-mask pattern of shape [ceil(Lq/blk), ceil(Lk/blk)] (uint8,
    nonzero = the block pair is kept), or None for "none".

    "window:W"  each query block keeps the W key blocks ending at the block
                that holds its bottom-right-aligned diagonal (a sliding
                window of W*blk keys, the pattern the pages name first);
    "random:P"  each block pair kept with probability P (seeded).
    """
    if spec in (None, "", "none"):
        return None
    kind, _, arg = spec.partition(":")
    nqb, nkb = -(-Lq // blk), -(-Lk // blk)
    if kind == "window":
        width = int(arg)
        if width < 1:
            raise ValueError("window width must be at least one block")
        # key block holding the last key that row qb*blk + blk-1 may see
        diag = np.minimum(nkb - 1, (np.minimum(Lq, (np.arange(nqb) + 1) * blk) - 1 + Lk - Lq) // blk)
        kb = np.arange(nkb)[None, :]
        return ((kb <= diag[:, None]) & (kb > diag[:, None] - width)).astype(np.uint8)
    if kind == "random":
        rng = np.random.default_rng(seed)
        return (rng.random((nqb, nkb)) < float(arg)).astype(np.uint8)
    raise ValueError(f"unknown block-mask pattern {spec!r}")


# ---------------------------------------------------------------------------
# Linear cross-entropy inputs ("When the Bottleneck Moved", section 1: the
# output layer of a Qwen3-8B fine-tune, hidden 4096, vocabulary 151936)
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class LceWorkload:
    name: str
    N: int  # tokens
    Dm: int  # hidden size
    V: int  # vocabulary
    dtype: str = "bf16"
    h_std: float = 1.0  # hidden states after the final RMS norm
    w_std: float = 0.02  # output-projection weights
    ignore_frac: float = 0.0  # share of rows whose target is -1 (ignored)
    seed: int = 2000

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPES[self.dtype]

    def with_(self, **kw) -> "LceWorkload":
        return replace(self, **kw)


LCE_WORKLOADS = {
    w.name: w
    for w in [
        LceWorkload("lce_tiny_n200_d128_v1000", N=200, Dm=128, V=1000, seed=2000),
        LceWorkload("lce_qwen3_8b_n8192", N=8192, Dm=4096, V=151936, seed=2001),
        # profiling case: same hidden size, a fifth of the vocabulary (256 MB of weights, above L2)
        LceWorkload("lce_n2048_d4096_v32768", N=2048, Dm=4096, V=32768, seed=2002),
    ]
}


def make_lce_inputs(w: LceWorkload, device: str | torch.device = "cpu"):
    """hidden [N, Dm], weight [V, Dm] (16-bit), targets [N] int32 (-1 =
    ignored) and the upstream gradient dloss [N] float32 (1/N: the gradient
    of the mean loss), drawn in that order from a CPU generator."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    h = (torch.randn((w.N, w.Dm), generator=gen, dtype=torch.float32) * w.h_std).to(w.torch_dtype)
    wt = (torch.randn((w.V, w.Dm), generator=gen, dtype=torch.float32) * w.w_std).to(w.torch_dtype)
    t = torch.randint(0, w.V, (w.N,), generator=gen, dtype=torch.int64)
    if w.ignore_frac > 0:
        drop = torch.rand((w.N,), generator=gen) < w.ignore_frac
        t = torch.where(drop, torch.full_like(t, -1), t)
    t = t.to(torch.int32)
    dloss = torch.full((w.N,), 1.0 / w.N, dtype=torch.float32)
    return tuple(x.to(device).contiguous() for x in (h, wt, t, dloss))
