"""GPU parity of the linear cross-entropy calls (lce_fwd, lce_bwd) against
the fp64 oracle (oracle/linear_ce.py; "When the Bottleneck Moved", section 1).

Tolerances, from the arithmetic.  Logits accumulate exact 16-bit products in
fp32, so loss and lse (fp32) are held to 1e-3 absolute like the attention
LSE.  The gradients: g is rounded to the 16-bit type before the two
products, each element with an error of at most u|g| + eta (u the unit
roundoff, 2^-8 for bf16 and 2^-11 for fp16; eta half the smallest
subnormal, 2^-134 and 2^-25); the products then accumulate in fp32, and the
result is rounded once more to 16 bits.  So element (i, d) of dH = g W obeys
    |gpu - ref| <= u|ref| + eta + sum_v (u|g_iv| + eta) |W_vd|,
and dW = g^T H likewise with H in place of W.  The tests allow twice the sum
(the fp32 accumulation and the fp32 evaluation of g add well under 1% of it)
and compute |g| from the oracle."""

import numpy as np
import pytest
import torch

import oracle.linear_ce as L
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import LCE_WORKLOADS, LceWorkload, make_lce_inputs, to_f64

pytestmark = pytest.mark.gpu

ROUNDING = {"bf16": (2.0 ** -8, 2.0 ** -134), "fp16": (2.0 ** -11, 2.0 ** -25)}
LOSS_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    gbattn.load_library()


def grad_tolerance(ref, g_abs_times_m, ones_times_m, dtype):
    """u|ref| + eta + 2 (u (|g| @ |M|) + eta (1 @ |M|)), M the other operand."""
    u, eta = ROUNDING[dtype]
    return u * np.abs(ref) + eta + 2.0 * (u * g_abs_times_m + eta * ones_times_m)


def assert_grad_close(gpu, ref, tol, what):
    g = to_f64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bad = err > tol
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g} tol {tol[idx]:.3g}")
    return float((err / tol).max())


def run(w: LceWorkload, h, wt, t, dloss):
    ws = gbattn.lce_workspace(h, wt)
    loss = torch.empty(w.N, dtype=torch.float32, device=h.device)
    lse = torch.empty_like(loss)
    gbattn.lce_fwd(h, wt, t, loss, lse, ws)
    dh, dw = torch.empty_like(h), torch.empty_like(wt)
    gbattn.lce_bwd(h, wt, t, lse, dloss, dh, dw, ws)
    torch.cuda.synchronize()
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    return loss, lse, dh, dw


SMALL = [
    LCE_WORKLOADS["lce_tiny_n200_d128_v1000"],
    LceWorkload("lce_fp16_n333_d256_v513_ignore", N=333, Dm=256, V=513, dtype="fp16", ignore_frac=0.2, seed=2100),
    LceWorkload("lce_three_chunks_n64_d64_v40000", N=64, Dm=64, V=40000, seed=2101),
    LceWorkload("lce_one_row_n1_d192_v300", N=1, Dm=192, V=300, seed=2102),
    LceWorkload("lce_n129_d512_v257", N=129, Dm=512, V=257, ignore_frac=0.1, seed=2103),
    # two vocabulary chunks; the dW product has 256 tiles, so CTAs run several
    LceWorkload("lce_two_chunks_n1024_d512_v20000", N=1024, Dm=512, V=20000, seed=2105),
    LceWorkload("lce_fp16_two_chunks_n300_d320_v17000", N=300, Dm=320, V=17000, dtype="fp16", ignore_frac=0.05,
                seed=2106),
]


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_lce_matches_oracle(w):
    h, wt, t, dloss = make_lce_inputs(w, "cuda")
    loss, lse, dh, dw = run(w, h, wt, t, dloss)
    hd, wd = to_f64(h), to_f64(wt)
    tn, dn = t.cpu().numpy().astype(np.int64), dloss.cpu().numpy().astype(np.float64)
    loss_ref, lse_ref = L.forward(hd, wd, tn)
    assert np.abs(to_f64(loss) - loss_ref).max() <= LOSS_ATOL
    assert np.abs(to_f64(lse) - lse_ref).max() <= LOSS_ATOL
    dh_ref, dw_ref = L.backward(hd, wd, tn, lse_ref, dn)
    ga = np.abs(L.grad_logits(hd, wd, tn, lse_ref, dn))
    assert_grad_close(dh, dh_ref, grad_tolerance(dh_ref, ga @ np.abs(wd), np.abs(wd).sum(0), w.dtype), "dH")
    assert_grad_close(dw, dw_ref, grad_tolerance(dw_ref, ga.T @ np.abs(hd), np.abs(hd).sum(0), w.dtype), "dW")
    assert torch.count_nonzero(dh[t < 0]) == 0


def _w_chunk(wt):
    return lambda v0, v1: to_f64(wt[v0:v1])


def test_qwen_shape_sampled_rows():
    """N = 8192, hidden 4096, vocabulary 151936: loss, lse and dH on sampled
    rows; the rows of dW sum to zero (each row of g does) within the output
    rounding."""
    w = LCE_WORKLOADS["lce_qwen3_8b_n8192"]
    h, wt, t, dloss = make_lce_inputs(w, "cuda")
    loss, lse, dh, dw = run(w, h, wt, t, dloss)
    for x in (loss, lse, dh, dw):
        assert torch.isfinite(x).all()
    rows = np.array([0, 1, 127, 128, 4095, 8190, 8191, 3333])
    hd = to_f64(h[rows])
    tn = t[rows].cpu().numpy().astype(np.int64)
    dn = dloss[rows].cpu().numpy().astype(np.float64)
    loss_ref, lse_ref = L.forward_rows(hd, tn, _w_chunk(wt), w.V)
    assert np.abs(to_f64(loss[rows]) - loss_ref).max() <= LOSS_ATOL
    assert np.abs(to_f64(lse[rows]) - lse_ref).max() <= LOSS_ATOL
    dh_ref = L.dhidden_rows(hd, tn, dn, _w_chunk(wt), w.V)
    ga = np.abs(L.grad_logits_rows(hd, tn, dn, _w_chunk(wt), w.V))
    gw, wsum = np.zeros_like(dh_ref), np.zeros(w.Dm)
    for v0 in range(0, w.V, 16384):  # |g| @ |W| and the column sums of |W|, a chunk at a time
        wa = np.abs(to_f64(wt[v0:v0 + 16384]))
        gw += ga[:, v0:v0 + 16384] @ wa
        wsum += wa.sum(0)
    assert_grad_close(dh[rows], dh_ref, grad_tolerance(dh_ref, gw, wsum, w.dtype), "dH rows")
    # sum_v dW[v, :] = sum_i (sum_v g_iv) H_i = 0; the 16-bit rounding of each
    # dW entry (at most 2^-8 of it) bounds what the sum can show
    dwf = dw.float()
    assert (dwf.sum(dim=0).abs() <= 2.0 ** -8 * dwf.abs().sum(dim=0) + 1e-12).all()


@pytest.mark.parametrize("N", [256, 8192])
def test_qwen_vocab_dweight_entries(N):
    """Full vocabulary (151936) and hidden size (4096) with 256 rows and with
    the whole 8192-row batch: dW on sampled vocabulary entries -- both ends
    of every backward chunk boundary crossed, the last entry, and the rows'
    targets -- against the oracle, element by element."""
    base = LCE_WORKLOADS["lce_qwen3_8b_n8192"]
    w = base if N == base.N else base.with_(name=f"lce_qwen_n{N}", N=N, seed=2104)
    h, wt, t, dloss = make_lce_inputs(w, "cuda")
    loss, lse, dh, dw = run(w, h, wt, t, dloss)
    hd = to_f64(h)
    tn, dn = t.cpu().numpy().astype(np.int64), dloss.cpu().numpy().astype(np.float64)
    w32 = wt.float().cpu().numpy()  # exact; decoded to float64 one chunk at a time
    chunk = lambda v0, v1: w32[v0:v1].astype(np.float64)  # noqa: E731
    edges = [e for c in range(16384, w.V, 16384) for e in (c - 1, c)]
    entries = sorted(set([0, 1, 255, 256, w.V - 1] + edges + tn[:6].tolist()))
    g = L.grad_logits_entries(hd, tn, dn, chunk, w.V, entries)
    dw_ref = g.T @ hd
    ha = np.abs(hd)
    tol = grad_tolerance(dw_ref, np.abs(g).T @ ha, ha.sum(0), w.dtype)
    assert_grad_close(dw[entries], dw_ref, tol, f"dW entries (N={N})")
