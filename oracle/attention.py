"""fp64 CPU oracle for exact causal grouped-query attention and its gradients.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only the tests, the smoke check and the bench's CPU-baseline leg
use it.  It shares no code with the CUDA kernels.

What it computes, written as the plain definition (no tiling, no online
softmax, no log2 tricks), for every batch b and query head hq:

* Forward (page 3, "When the Bottleneck Moved", section 3 "What the
  FlashAttention schedule changes": S = scale * Q K^T + mask, P = softmax(S),
  O = P V, L = m + log l):
    S_ij  = scale * sum_d Q_id K_jd, with key j visible to query i iff the
            attention is not causal or j <= i + (Lk - Lq)   (bottom-right
            causal alignment, page 2 "Add a fused full-attention path for
            head_dim 256", section "Ragged causal inputs": the offset
            qL_off = kL - qL comes from the true lengths);
    P_ij  = exp(S_ij - m_i) / sum_visible exp(S_ij - m_i), 0 when masked;
    O_i   = sum_j P_ij V_j;
    LSE_i = m_i + ln sum_visible exp(S_ij - m_i)  (natural log), and the
            base-2 value lse2_i = LSE_i * log2(e) that the kernels keep (page
            1, "feat(attention): complete Flash Attention VJP", section
            "Background": P = exp2(S * scale_log2 - LSE)).
* delta (page 1, section "Architecture"/"Two-Kernel Design": delta =
  rowsum(dO * O) in f32, computed once before the two gradient kernels):
    delta_i = sum_d dO_id * O_id, with O the output passed in.
* Backward (page 1, section "Background", backward pass):
    dP_ij = sum_d dO_id V_jd,
    dS_ij = P_ij * (dP_ij - delta_i)         (S here already holds the scale),
    dQ_i  = scale * sum_j dS_ij K_j,
    dK_j  = scale * sum_{g,i} dS_ij Q_i,   dV_j = sum_{g,i} P_ij dO_i,
  where the sums over g run over the G = Hq / Hkv query heads that share KV
  head hk = hq // G (consecutive query heads share one KV head).

* Block-sparse attention (page 1, section "Sparse Block Masks": an optional
  uint8 mask with one entry per (query tile, key tile) pair; a zero entry
  skips the pair): key j is visible to query i only if, in addition,
  block_mask[i // blk, j // blk] != 0.  The kernels fix blk = 128.  A query
  row that then sees no key (the pages are silent on this case) has P = 0,
  O = 0 and LSE = +inf, so its dQ is 0 and it adds nothing to dK and dV.

Layouts: q, o, do, dq are [B, Hq, Lq, D]; k, v, dk, dv are [B, Hkv, Lk, D];
lse and delta are [B, Hq, Lq]; block_mask is [ceil(Lq/blk), ceil(Lk/blk)],
shared by all batches and heads.  All arrays are float64 numpy arrays;
callers decode fp16/bf16 inputs to float64 exactly before calling.
"""

from __future__ import annotations

import numpy as np

LOG2E = 1.0 / np.log(2.0)
MASK_BLOCK = 128  # rows and columns covered by one block-mask entry in the kernels


def visible(Lq: int, Lk: int, causal: bool, block_mask=None, blk: int = MASK_BLOCK) -> np.ndarray:
    """Boolean [Lq, Lk]: True where key j is visible to query i.

    Bottom-right causal alignment: j <= i + (Lk - Lq) (page 2, "Ragged causal
    inputs").  Non-causal attention sees every key.  With a block mask, key j
    is visible only where block_mask[i // blk, j // blk] != 0 (page 1, "Sparse
    Block Masks").
    """
    if not causal:
        vis = np.ones((Lq, Lk), dtype=bool)
    else:
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        vis = j <= i + (Lk - Lq)
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        if bm.shape != (-(-Lq // blk), -(-Lk // blk)):
            raise ValueError("block mask shape must be [ceil(Lq/blk), ceil(Lk/blk)]")
        vis = vis & bm[np.arange(Lq)[:, None] // blk, np.arange(Lk)[None, :] // blk]
    return vis


def _softmax_rows(S: np.ndarray, mask: np.ndarray):
    """Masked softmax of each row: (P, LSE_natural).  A row with no visible
    entry gets P = 0 and LSE = +inf."""
    has = mask.any(axis=1, keepdims=True)
    S = np.where(mask, S, -np.inf)
    m = np.where(has, S.max(axis=1, keepdims=True, initial=-np.inf), 0.0)
    E = np.where(mask, np.exp(np.where(mask, S, 0.0) - m), 0.0)
    l = E.sum(axis=1, keepdims=True)
    P = np.where(has, E / np.where(has, l, 1.0), 0.0)
    lse = np.where(has, m + np.log(np.where(has, l, 1.0)), np.inf)[:, 0]
    return P, lse


def _group(Hq: int, Hkv: int) -> int:
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return Hq // Hkv


def head_forward(qh: np.ndarray, kh: np.ndarray, vh: np.ndarray, scale: float, causal: bool, block_mask=None,
                 blk: int = MASK_BLOCK):
    """One (b, hq) head: returns (P, O, LSE_natural) with P the full [Lq, Lk]
    probability matrix (page 3, section 3: S = scale*QK^T + mask,
    P = softmax(S), O = PV; L = m + log l)."""
    Lq, Lk = qh.shape[0], kh.shape[0]
    mask = visible(Lq, Lk, causal, block_mask, blk)
    S = scale * (qh @ kh.T)
    P, lse = _softmax_rows(S, mask)
    O = P @ vh
    return P, O, lse


def forward(q, k, v, scale: float, causal: bool, block_mask=None, blk: int = MASK_BLOCK):
    """Returns (o, lse2, lse_nat): o [B,Hq,Lq,D]; lse2 = base-2 LSE [B,Hq,Lq]."""
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G = _group(Hq, Hkv)
    o = np.zeros((B, Hq, Lq, D))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        for hq in range(Hq):
            hk = hq // G
            _, o[b, hq], lse[b, hq] = head_forward(q[b, hq], k[b, hk], v[b, hk], scale, causal, block_mask, blk)
    return o, lse * LOG2E, lse


def delta(o, do):
    """delta_i = sum_d dO_id * O_id (page 1, "Two-Kernel Design")."""
    return (o * do).sum(axis=-1)


def head_backward(qh, kh, vh, oh, doh, scale: float, causal: bool, block_mask=None, blk: int = MASK_BLOCK):
    """One (b, hq) head: returns (dq, dk_part, dv_part) where the dk/dv parts
    are this query head's contribution to its KV head (page 1, "Background",
    backward pass: dP = dO V^T, dS = scale * P * (dP - delta), dQ = dS K,
    dK = dS^T Q, dV = P^T dO)."""
    P, _, _ = head_forward(qh, kh, vh, scale, causal, block_mask, blk)
    dP = doh @ vh.T
    dlt = delta(oh, doh)[:, None]
    dS = P * (dP - dlt)
    dq = scale * (dS @ kh)
    dk = scale * (dS.T @ qh)
    dv = P.T @ doh
    return dq, dk, dv


def backward(q, k, v, o, do, scale: float, causal: bool, block_mask=None, blk: int = MASK_BLOCK):
    """Returns (dq, dk, dv) with the GQA group sums folded into dk and dv."""
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    G = _group(Hq, Hkv)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for hq in range(Hq):
            hk = hq // G
            a, bk, bv = head_backward(q[b, hq], k[b, hk], v[b, hk], o[b, hq], do[b, hq], scale, causal, block_mask,
                                      blk)
            dq[b, hq] = a
            dk[b, hk] += bk
            dv[b, hk] += bv
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Helpers for checking large problems on a sample of outputs.  They evaluate
# the same definitions restricted to chosen heads / rows.
# ---------------------------------------------------------------------------


def forward_rows(q, k, v, scale: float, causal: bool, b: int, hq: int, rows):
    """O and base-2 LSE for selected query rows of head (b, hq)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    hk = hq // _group(Hq, Hkv)
    Lq, Lk = q.shape[2], k.shape[2]
    rows = np.asarray(rows)
    qh = q[b, hq, rows]
    S = scale * (qh @ k[b, hk].T)
    mask = visible(Lq, Lk, causal)[rows]
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.where(mask, np.exp(S - m), 0.0)
    l = E.sum(axis=1, keepdims=True)
    O = (E / l) @ v[b, hk]
    return O, (m + np.log(l))[:, 0] * LOG2E


def lse_all_rows(q, k, scale: float, causal: bool, b: int, hq: int, block: int = 1024):
    """Natural-log LSE of every query row of head (b, hq), one row block at a
    time (same definition as head_forward, without holding all of S)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    hk = hq // _group(Hq, Hkv)
    Lq, Lk = q.shape[2], k.shape[2]
    out = np.empty(Lq)
    kh = k[b, hk]
    for r0 in range(0, Lq, block):
        rows = np.arange(r0, min(Lq, r0 + block))
        S = scale * (q[b, hq, rows] @ kh.T)
        mask = visible(Lq, Lk, causal)[rows] if causal else np.ones((len(rows), Lk), dtype=bool)
        S = np.where(mask, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        l = np.where(mask, np.exp(S - m), 0.0).sum(axis=1, keepdims=True)
        out[rows] = (m + np.log(l))[:, 0]
    return out


def backward_query_rows(q, k, v, o, do, scale: float, causal: bool, b: int, hq: int, rows):
    """dQ for selected query rows of head (b, hq): each row needs only its own
    softmax row, dP row and delta (dQ_i = scale * sum_j dS_ij K_j)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    hk = hq // _group(Hq, Hkv)
    Lq, Lk = q.shape[2], k.shape[2]
    rows = np.asarray(rows)
    S = scale * (q[b, hq, rows] @ k[b, hk].T)
    mask = visible(Lq, Lk, causal)[rows]
    S = np.where(mask, S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.where(mask, np.exp(S - m), 0.0)
    P = E / E.sum(axis=1, keepdims=True)
    dP = do[b, hq, rows] @ v[b, hk].T
    dlt = delta(o[b, hq, rows], do[b, hq, rows])[:, None]
    dS = P * (dP - dlt)
    return scale * (dS @ k[b, hk])


def backward_key_rows(q, k, v, o, do, scale: float, causal: bool, b: int, hk: int, keys):
    """dK and dV for selected key rows of KV head (b, hk): column j of P needs
    the LSE of every query row (dK_j = scale * sum_{g,i} dS_ij Q_i,
    dV_j = sum_{g,i} P_ij dO_i)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = _group(Hq, Hkv)
    Lq, Lk = q.shape[2], k.shape[2]
    keys = np.asarray(keys)
    dk = np.zeros((len(keys), k.shape[3]))
    dv = np.zeros((len(keys), v.shape[3]))
    mask = visible(Lq, Lk, causal)[:, keys]  # [Lq, n_keys]
    for g in range(G):
        hq = hk * G + g
        lse = lse_all_rows(q, k, scale, causal, b, hq)
        S = scale * (q[b, hq] @ k[b, hk, keys].T)  # [Lq, n_keys]
        P = np.where(mask, np.exp(np.where(mask, S, 0.0) - lse[:, None]), 0.0)
        dP = do[b, hq] @ v[b, hk, keys].T
        dlt = delta(o[b, hq], do[b, hq])[:, None]
        dS = P * (dP - dlt)
        dk += scale * (dS.T @ q[b, hq])
        dv += P.T @ do[b, hq]
    return dk, dv


def backward_kv_head(q, k, v, o, do, scale: float, causal: bool, b: int, hk: int):
    """dQ for the G query heads of KV head (b, hk), and that head's dK, dV."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = _group(Hq, Hkv)
    dqs = []
    dk = np.zeros_like(k[b, hk])
    dv = np.zeros_like(v[b, hk])
    for g in range(G):
        hq = hk * G + g
        a, bk, bv = head_backward(q[b, hq], k[b, hk], v[b, hk], o[b, hq], do[b, hq], scale, causal)
        dqs.append(a)
        dk += bk
        dv += bv
    return np.stack(dqs), dk, dv


def flops_forward(B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> float:
    """Forward FLOP credit: two matmuls of 2*Lq*Lk*D each per head, halved when
    causal (page 2's benchmark table: 42.8 TF for 8192^2, 16 heads, D=256 at
    12.84 ms is exactly this count over that time)."""
    f = 4.0 * B * Hq * Lq * Lk * D
    return f / 2.0 if causal else f


def flops_fwd_bwd(B: int, Hq: int, Lq: int, Lk: int, D: int, causal: bool) -> float:
    """Forward plus backward credit: the backward counts 2.5x the forward (page
    1, "Background": five matmuls per block pair against two)."""
    return 3.5 * flops_forward(B, Hq, Lq, Lk, D, causal)
