"""Work accounting for the attention hot path: credited FLOPs for the metric
and algorithmic FLOPs / bytes per kernel launch for the roofline.

Conventions ("Add a fused full-attention path for head_dim 256 on NAX
devices", section Performance, "Kernel benchmarks" table; "feat(attention):
complete Flash Attention VJP implementation", section "Background"):
* forward credit: 4*B*Hq*Lq*Lk*D FLOPs, halved when causal;
* backward credit: 2.5x the forward; forward plus backward: 3.5x.

Algorithmic work per kernel counts the exact visible (query, key) pairs,
2*D FLOPs per pair per matmul:
* fwd: S = Q K^T and O = P V, 2 matmuls;
* dQ kernel: S, dP, dQ, 3 matmuls;
* dK/dV kernel: S^T, dP^T, dV, dK, 4 matmuls;
* both backward kernels together ("bwd"): 7 matmuls;
* delta: reads O and dO once (2 bytes per element each) and writes one
  float32 per row.
"""

from __future__ import annotations


def visible_pairs(Lq: int, Lk: int, causal: bool) -> int:
    """Number of (i, j) with key j visible to query i, per head.

    Bottom-right causal alignment: row i sees keys 0 .. min(Lk-1, i + Lk - Lq).
    """
    if not causal:
        return Lq * Lk
    off = Lk - Lq
    if off >= 0:  # row i sees i + off + 1 keys
        return Lq * (off + 1) + Lq * (Lq - 1) // 2
    # Lq > Lk: rows below -off see nothing, the last Lk rows see 1 .. Lk keys
    return Lk * (Lk + 1) // 2


def visible_pairs_masked(Lq: int, Lk: int, causal: bool, block_mask, blk: int = 128) -> int:
    """Visible (i, j) pairs per head when a block mask (one entry per blk x blk
    block of queries and keys, nonzero = kept) is applied on top of the causal
    rule ("feat(attention): complete Flash Attention VJP implementation",
    section "Sparse Block Masks")."""
    import numpy as np

    bm = np.asarray(block_mask) != 0
    nqb, nkb = -(-Lq // blk), -(-Lk // blk)
    assert bm.shape == (nqb, nkb), (bm.shape, nqb, nkb)
    i = np.arange(Lq)
    # last visible key of each row (Lk - 1 when not causal), -1 if none
    last = np.minimum(Lk - 1, i + (Lk - Lq)) if causal else np.full(Lq, Lk - 1)
    total = 0
    for kb in range(nkb):
        lo, hi = kb * blk, min(Lk, (kb + 1) * blk)  # keys lo .. hi-1
        n = np.clip(np.minimum(last, hi - 1) - lo + 1, 0, hi - lo)
        total += int((n * bm[i // blk, kb]).sum())
    return total


def credited_forward(B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> float:
    f = 4.0 * B * Hq * Lq * Lk * D
    return f / 2.0 if causal else f


def credited_fwd_bwd(B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> float:
    return 3.5 * credited_forward(B, Hq, Lq, Lk, D, causal)


MATMULS = {"fwd": 2, "bwd_dq": 3, "bwd_dkv": 4, "bwd": 7}


def kernel_flops(kernel: str, B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> float:
    """Algorithmic FLOPs of one launch of `kernel` (fwd, bwd_dq or bwd_dkv)."""
    return 2.0 * D * MATMULS[kernel] * B * Hq * visible_pairs(Lq, Lk, causal)


def kernel_flops_pairs(kernel: str, B: int, Hq: int, D: int, pairs: int) -> float:
    """Algorithmic FLOPs of one launch given the visible pairs per head."""
    return 2.0 * D * MATMULS[kernel] * B * Hq * pairs


def delta_bytes(B: int, Hq: int, Lq: int, D: int, elem_bytes: int = 2) -> int:
    rows = B * Hq * Lq
    return 2 * rows * D * elem_bytes + 4 * rows


def decode_bytes(kernel: str, B: int, Hq: int, Hkv: int, Lq: int, Lk: int, D: int, elem_bytes: int = 2) -> int:
    """Compulsory HBM bytes of the decode-shaped calls, which are bound by
    reading the key/value range: fwd reads q, k, v and writes o and lse; bwd
    reads q, k, v, dO, lse, delta and writes dq, dk, dv (the split partials
    stay in L2 and are not counted)."""
    q = B * Hq * Lq * D * elem_bytes
    kv = B * Hkv * Lk * D * elem_bytes
    rows = B * Hq * Lq * 4
    if kernel == "fwd":
        return q + 2 * kv + q + rows
    if kernel == "bwd":
        return 2 * q + 2 * kv + 2 * rows + q + 2 * kv
    raise ValueError(kernel)
