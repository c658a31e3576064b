"""GPU parity when the row maximum keeps rising along the keys.

The forward kernels keep a reference maximum per row and rescale the O
accumulator and the running sum only when a key tile raises the row maximum
by more than 8 (log2 units); with N(0,1) inputs that happens almost only on
the first tile.  Here every key row is scaled up with its position, so the
scores of each new key tile exceed the previous maximum by more than that
threshold and the rescaling path runs on nearly every tile (D <= 128: the
two-tile forward; D = 256: the one-tile forward), followed by the backward,
which works from the saved lse.

O and lse are compared with the fp64 oracle on the same 16-bit inputs.  The
gradients are compared with the oracle's backward run on the GPU's own
(16-bit) O, so that both sides form delta = rowsum(dO * O) from the same O,
and within the usual tolerance plus what rounding the 16-bit dS and P the
products read can contribute (derived from the fp64 intermediates below):
with keys scaled up to ~150x, dQ = scale * sum dS K carries the rounding of
dS times |K|, which the flat tolerance alone does not cover.
"""

import numpy as np
import pytest
import torch

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs, to_f64

from test_parity_gpu import LSE_ATOL, TOL, assert_abs, assert_close, run_chain

pytestmark = pytest.mark.gpu

# unit roundoff of the 16-bit dS and P that the gradient products read
ROUNDING = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    gbattn.load_library()


def rising_keys(k, per_tile: float, tile: int = 64):
    """k with key row j scaled by 1 + per_tile * j / tile (16-bit)."""
    L = k.shape[2]
    ramp = 1.0 + per_tile * torch.arange(L, dtype=torch.float32, device=k.device) / tile
    return (k.float() * ramp[None, None, :, None]).to(k.dtype)


def scores(w, qd, kd):
    """scale * Q K^T with K repeated over the query heads of a group, and the
    causal mask (bottom-right aligned) as a boolean of kept entries."""
    kr = np.repeat(kd, w.Hq // w.Hkv, axis=1)
    s = np.einsum("bhqd,bhkd->bhqk", qd, kr) * w.scale
    keep = np.ones((w.Lq, w.Lk), dtype=bool)
    if w.causal:
        keep = np.arange(w.Lk)[None, :] <= np.arange(w.Lq)[:, None] + (w.Lk - w.Lq)
    return s, kr, keep


def row_max_rise_log2(w, qd, kd):
    """Median rise (log2 units) of a row's running score maximum from one
    64-key tile to the next, over the rows and tiles that see keys."""
    s, _, keep = scores(w, qd, kd)
    s = np.where(keep, s * 1.4426950408889634, -np.inf)
    tiles = np.stack([s[..., t:t + 64].max(axis=-1) for t in range(0, w.Lk, 64)], axis=-1)
    run = np.maximum.accumulate(tiles, axis=-1)
    with np.errstate(invalid="ignore"):
        rise = np.diff(run, axis=-1)
    seen = np.isfinite(rise) & np.isfinite(tiles[..., 1:])  # skip tiles the mask empties
    return float(np.median(rise[seen]))


def rounding_bounds(w, qd, kd, vd, dod, od):
    """Per-element bounds on what rounding dS and P to 16 bits can move dQ,
    dK and dV by: u * scale * |dS| |K| (dQ), u * scale * |dS|^T |Q| (dK,
    summed over the group's query heads), u * |P|^T |dO| (dV)."""
    u = ROUNDING[w.dtype]
    G = w.Hq // w.Hkv
    s, kr, keep = scores(w, qd, kd)
    m = np.where(keep, s, -np.inf).max(axis=-1, keepdims=True)
    p = np.where(keep, np.exp(s - m), 0.0)
    p /= p.sum(axis=-1, keepdims=True)
    vr = np.repeat(vd, G, axis=1)
    dp = np.einsum("bhqd,bhkd->bhqk", dod, vr)
    dlt = (dod * od).sum(axis=-1, keepdims=True)
    ds = p * (dp - dlt)
    b_dq = u * w.scale * np.einsum("bhqk,bhkd->bhqd", np.abs(ds), np.abs(kr))
    b_dk = u * w.scale * np.einsum("bhqk,bhqd->bhkd", np.abs(ds), np.abs(qd))
    b_dv = u * np.einsum("bhqk,bhqd->bhkd", np.abs(p), np.abs(dod))

    def fold(t):  # sum over the query heads of each KV group
        return t.reshape(w.B, w.Hkv, G, w.Lk, w.D).sum(axis=2)

    return b_dq, fold(b_dk), fold(b_dv)


def assert_within(gpu, ref, bound, dtype, what):
    atol, rtol = TOL[dtype]
    g = to_f64(gpu)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    lim = atol + rtol * np.abs(ref) + bound
    bad = err > lim
    if bad.any():
        idx = np.unravel_index(np.argmax(err - lim), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g} bound {bound[idx]:.3g}")


CASES = [
    Workload("rise_d64_causal", B=1, Hq=2, Hkv=1, Lq=512, Lk=512, D=64, seed=6100),
    Workload("rise_d128_causal_gqa", B=1, Hq=4, Hkv=2, Lq=640, Lk=640, D=128, seed=6101),
    Workload("rise_d128_dense", B=1, Hq=2, Hkv=1, Lq=384, Lk=640, D=128, causal=False, seed=6102),
    Workload("rise_d96_causal_fp16", B=1, Hq=2, Hkv=1, Lq=576, Lk=576, D=96, dtype="fp16", std=0.5, seed=6103),
    Workload("rise_d256_causal", B=1, Hq=2, Hkv=1, Lq=512, Lk=512, D=256, seed=6104),
    Workload("rise_d256_dense_rect", B=1, Hq=2, Hkv=1, Lq=200, Lk=700, D=256, causal=False, seed=6105),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_rising_row_maximum(w):
    q, k, v, do = make_inputs(w, "cuda")
    k = rising_keys(k, per_tile=4.0 if w.dtype == "bf16" else 16.0)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    med = row_max_rise_log2(w, qd, kd)
    assert med > 8.0, f"the inputs should raise the row maximum past the threshold on most tiles (median {med})"
    o, lse, dlt, dq, dk, dv = run_chain(w, q, k, v, do)
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal)
    assert_close(o, o_ref, w.dtype, "O")
    assert_abs(lse, lse_ref, LSE_ATOL, "LSE")
    og = to_f64(o)
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, og, dod, w.scale, w.causal)
    b_dq, b_dk, b_dv = rounding_bounds(w, qd, kd, vd, dod, og)
    assert_within(dq, dq_ref, b_dq, w.dtype, "dQ")
    assert_within(dk, dk_ref, b_dk, w.dtype, "dK")
    assert_within(dv, dv_ref, b_dv, w.dtype, "dV")
