"""fp64 CPU oracle for the linear cross-entropy loss and its gradients.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module: only the tests, the smoke check and the bench's CPU-baseline leg
use it.  It shares no code with the CUDA kernels.

What it computes, written as the plain definition with the (N, V) logits
matrix materialised (page 3, "When the Bottleneck Moved", section 1 "The
first hypothesis: remove logits, train longer": logits = hidden @ W.T and
loss_i = logsumexp(logits_i) - logits_i,target_i; the fused kernel streams
over vocabulary tiles with an online log-sum-exp instead, which reaches the
same value up to rounding):

* Forward, for every row i with target t_i:
    z_iv   = sum_d H_id W_vd                      (logits, v < V)
    lse_i  = m_i + ln sum_v exp(z_iv - m_i),  m_i = max_v z_iv
    loss_i = lse_i - z_i,t_i
* Backward, with an upstream gradient dloss_i per row (the derivative of the
  definition above; the pages give no formula for it):
    p_iv  = exp(z_iv - lse_i)                     (softmax of the row)
    g_iv  = dloss_i * (p_iv - [v == t_i])
    dH    = g W,   dW = g^T H.
* A negative target marks a row that takes no part (a padding token; the
  pages are silent): its loss is 0 and its gradient rows are 0.
"""

from __future__ import annotations

import numpy as np


def logits(h: np.ndarray, w: np.ndarray) -> np.ndarray:
    """z = H W^T, [N, V]."""
    return h @ w.T


def forward(h: np.ndarray, w: np.ndarray, t: np.ndarray):
    """(loss [N], lse [N]) in float64; lse is the natural-log log-sum-exp."""
    z = logits(h, w)
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    rows = np.arange(z.shape[0])
    valid = t >= 0
    zt = np.where(valid, z[rows, np.where(valid, t, 0)], 0.0)
    loss = np.where(valid, lse - zt, 0.0)
    return loss, lse


def grad_logits(h: np.ndarray, w: np.ndarray, t: np.ndarray, lse: np.ndarray, dloss: np.ndarray) -> np.ndarray:
    """g = dloss * (softmax(z) - onehot(t)), [N, V]; zero rows where t < 0."""
    z = logits(h, w)
    g = np.exp(z - lse[:, None])
    valid = t >= 0
    rows = np.arange(z.shape[0])[valid]
    g[rows, t[valid]] -= 1.0
    return g * np.where(valid, dloss, 0.0)[:, None]


def backward(h: np.ndarray, w: np.ndarray, t: np.ndarray, lse: np.ndarray, dloss: np.ndarray):
    """(dH [N, Dm], dW [V, Dm]) in float64."""
    g = grad_logits(h, w, t, lse, dloss)
    return g @ w, g.T @ h


# ---------------------------------------------------------------------------
# Helpers for large problems: the same definitions evaluated on chosen rows or
# vocabulary entries, with the weight matrix decoded one vocabulary chunk at a
# time (w_chunk(v0, v1) returns rows v0..v1-1 of W as float64).
# ---------------------------------------------------------------------------


def logits_rows(h_rows: np.ndarray, w_chunk, V: int, chunk: int = 16384) -> np.ndarray:
    """z for the given rows of H, [n, V]."""
    return np.concatenate([h_rows @ w_chunk(v0, min(V, v0 + chunk)).T for v0 in range(0, V, chunk)], axis=1)


def forward_rows(h_rows: np.ndarray, t_rows: np.ndarray, w_chunk, V: int):
    """(loss, lse) of the given rows."""
    z = logits_rows(h_rows, w_chunk, V)
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    valid = t_rows >= 0
    zt = np.where(valid, z[np.arange(len(t_rows)), np.where(valid, t_rows, 0)], 0.0)
    return np.where(valid, lse - zt, 0.0), lse


def grad_logits_rows(h_rows, t_rows, dloss_rows, w_chunk, V: int, chunk: int = 16384) -> np.ndarray:
    """g = dloss * (softmax - onehot) for the given rows, [n, V]."""
    z = logits_rows(h_rows, w_chunk, V, chunk)
    _, lse = forward_rows(h_rows, t_rows, w_chunk, V)
    g = np.exp(z - lse[:, None])
    valid = t_rows >= 0
    g[np.arange(len(t_rows))[valid], t_rows[valid]] -= 1.0
    g *= np.where(valid, dloss_rows, 0.0)[:, None]
    return g


def dhidden_rows(h_rows, t_rows, dloss_rows, w_chunk, V: int, chunk: int = 16384):
    """dH for the given rows: (dloss * (softmax - onehot)) W."""
    g = grad_logits_rows(h_rows, t_rows, dloss_rows, w_chunk, V, chunk)
    out = np.zeros((h_rows.shape[0], h_rows.shape[1]))
    for v0 in range(0, V, chunk):
        out += g[:, v0:v0 + chunk] @ w_chunk(v0, min(V, v0 + chunk))
    return out


def lse_rows(h: np.ndarray, w_chunk, V: int, block: int = 1024) -> np.ndarray:
    """The natural-log lse of every row of h, a block of rows at a time (each
    row's whole logits row is formed, as in forward_rows)."""
    out = np.empty(h.shape[0])
    for r0 in range(0, h.shape[0], block):
        z = logits_rows(h[r0:r0 + block], w_chunk, V)
        m = z.max(axis=1)
        out[r0:r0 + block] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    return out


def grad_logits_entries(h: np.ndarray, t: np.ndarray, dloss: np.ndarray, w_chunk, V: int, entries) -> np.ndarray:
    """Columns `entries` of g for every row, [N, len(entries)] (needs every
    row's lse)."""
    entries = np.asarray(entries)
    lse = lse_rows(h, w_chunk, V)
    z = h @ np.concatenate([w_chunk(v, v + 1) for v in entries]).T  # [N, len(entries)]
    g = np.exp(z - lse[:, None])
    valid = t >= 0
    g -= (t[:, None] == entries[None, :]) & valid[:, None]
    g *= np.where(valid, dloss, 0.0)[:, None]
    return g


def dweight_entries(h: np.ndarray, t: np.ndarray, dloss: np.ndarray, w_chunk, V: int, entries):
    """dW for the given vocabulary entries: g[:, entries]^T H."""
    return grad_logits_entries(h, t, dloss, w_chunk, V, entries).T @ h
