"""GPU parity of the linear cross-entropy calls (lce_fwd, lce_bwd) against
the fp64 oracle (oracle/linear_ce.py; "When the Bottleneck Moved", section 1).

Tolerances, from the arithmetic: logits accumulate exact 16-bit products in
fp32, so loss and lse (fp32) are held to 1e-3 absolute like the attention
LSE; g is rounded to 16 bits before the two gradient products, whose sums run
over V (dH) or N (dW) terms, so dH and dW are held to
2e-2 |ref| + 1e-2 max|ref| (bf16; halved for fp16) element by element, the
absolute part scaled by the tensor's largest entry because the gradients of
a mean loss are small in absolute terms."""

import numpy as np
import pytest
import torch

import oracle.linear_ce as L
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import LCE_WORKLOADS, LceWorkload, make_lce_inputs, to_f64

pytestmark = pytest.mark.gpu

REL = {"bf16": 2e-2, "fp16": 1e-2}
SCALE = {"bf16": 1e-2, "fp16": 5e-3}
LOSS_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    gbattn.load_library()


def assert_grad_close(gpu, ref, dtype, what):
    g = to_f64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    tol = REL[dtype] * np.abs(ref) + SCALE[dtype] * np.abs(ref).max()
    err = np.abs(g - ref)
    bad = err > tol
    if bad.any():
        idx = np.unravel_index(np.argmax(err - tol), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g} (max|ref| {np.abs(ref).max():.3g})")


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
    assert_grad_close(dh, dh_ref, w.dtype, "dH")
    assert_grad_close(dw, dw_ref, w.dtype, "dW")
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
    assert_grad_close(dh[rows], dh_ref, w.dtype, "dH rows")
    # sum_v dW[v, :] = sum_i (sum_v g_iv) H_i = 0; the 16-bit rounding of each
    # dW entry (at most 2^-9 of it) bounds what the sum can show
    dwf = dw.float()
    assert (dwf.sum(dim=0).abs() <= 2.0 ** -8 * dwf.abs().sum(dim=0) + 1e-12).all()


def test_qwen_vocab_dweight_entries():
    """Full vocabulary and hidden size, 256 rows: dW on sampled vocabulary
    entries (including every row's target) against the oracle."""
    w = LCE_WORKLOADS["lce_qwen3_8b_n8192"].with_(name="lce_qwen_n256", N=256, seed=2104)
    h, wt, t, dloss = make_lce_inputs(w, "cuda")
    loss, lse, dh, dw = run(w, h, wt, t, dloss)
    hd = to_f64(h)
    tn, dn = t.cpu().numpy().astype(np.int64), dloss.cpu().numpy().astype(np.float64)
    entries = sorted(set([0, 1, 255, 256, 16383, 16384, w.V - 1] + tn[:6].tolist()))
    dw_ref = L.dweight_entries(hd, tn, dn, _w_chunk(wt), w.V, entries)
    assert_grad_close(dw[entries], dw_ref, w.dtype, "dW entries")
