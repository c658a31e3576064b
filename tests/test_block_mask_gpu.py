"""GPU parity of the block-sparse entry points (attn_fwd_masked,
attn_bwd_masked) against the fp64 oracle with the same block mask
("feat(attention): complete Flash Attention VJP implementation", section
"Sparse Block Masks"; one uint8 entry per 128 x 128 block pair).

Tolerances as in test_parity_gpu.py.  Rows that see no key must come back
with O = 0, lse = +inf and dQ = 0; key blocks no query reaches get dK = dV = 0.
"""

import numpy as np
import pytest
import torch

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "fp16": (1e-2, 1e-2)}
LSE_ATOL = 1e-3
BLK = A.MASK_BLOCK


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    gbattn.load_library()


def assert_close(gpu, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g = to_f64(gpu)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g}")


def assert_lse(gpu, ref, what="LSE"):
    g = to_f64(gpu)
    assert np.array_equal(np.isposinf(g), np.isposinf(ref)), f"{what}: +inf rows differ"
    fin = np.isfinite(ref)
    assert np.isfinite(g[fin]).all(), f"{what}: non-finite values"
    err = np.abs(g[fin] - ref[fin])
    assert err.size == 0 or err.max() <= LSE_ATOL, f"{what}: max abs err {err.max():.3g}"


def masked_chain(w: Workload, q, k, v, do, bm):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device=q.device)
    gbattn.attn_fwd_masked(q, k, v, o, lse, bm, w.scale, w.causal)
    dlt = gbattn.delta(o, do)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    gbattn.attn_bwd_masked(q, k, v, o, do, lse, dlt, bm, dq, dk, dv, w.scale, w.causal)
    torch.cuda.synchronize()
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    return o, lse, dq, dk, dv


def check_masked(w: Workload, bm_np: np.ndarray):
    q, k, v, do = make_inputs(w, "cuda")
    bm = torch.tensor(bm_np, dtype=torch.uint8, device="cuda")
    o, lse, dq, dk, dv = masked_chain(w, q, k, v, do, bm)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal, bm_np, BLK)
    assert_close(o, o_ref, w.dtype, "O")
    assert_lse(lse, lse_ref)
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal, bm_np, BLK)
    assert_close(dq, dq_ref, w.dtype, "dQ")
    assert_close(dk, dk_ref, w.dtype, "dK")
    assert_close(dv, dv_ref, w.dtype, "dV")


def random_mask(nqb, nkb, seed, density=0.5, empty_row=None, empty_col=None):
    rng = np.random.default_rng(seed)
    bm = (rng.random((nqb, nkb)) < density).astype(np.uint8)
    if empty_row is not None:
        bm[empty_row] = 0
    if empty_col is not None:
        bm[:, empty_col] = 0
    return bm


def window_mask(nqb, nkb, width, off_blocks=0):
    """Each query block keeps the `width` key blocks ending at its diagonal."""
    qb = np.arange(nqb)[:, None] + off_blocks
    kb = np.arange(nkb)[None, :]
    return ((kb <= qb) & (kb > qb - width)).astype(np.uint8)


CASES = []
for D in (64, 96, 128):
    CASES.append((Workload(f"mask_d{D}_bf16_causal_l700", B=1, Hq=4, Hkv=2, Lq=700, Lk=700, D=D, seed=5000 + D),
                  "random"))
    CASES.append((Workload(f"mask_d{D}_fp16_dense_l700", B=1, Hq=2, Hkv=2, Lq=700, Lk=700, D=D, dtype="fp16",
                           causal=False, seed=5100 + D), "random"))
CASES += [
    (Workload("mask_d256_bf16_causal_gqa_l700", B=1, Hq=4, Hkv=2, Lq=700, Lk=700, D=256, seed=5256), "random"),
    (Workload("mask_d256_fp16_dense_q300_k520", B=1, Hq=2, Hkv=1, Lq=300, Lk=520, D=256, dtype="fp16",
              causal=False, seed=5257), "random"),
    (Workload("mask_d256_window_l1024_g8", B=1, Hq=8, Hkv=1, Lq=1024, Lk=1024, D=256, seed=5258), "window"),
    (Workload("mask_rect_causal_q300_k900_d128", B=2, Hq=4, Hkv=1, Lq=300, Lk=900, D=128, seed=5201), "window"),
    # With this seed every non-empty row sees only the 4-key tail block, so
    # each dS term is ~30x larger than with a full block and the 16-bit
    # rounding of dS (which the method prescribes before the dK product)
    # reaches 0.9 of the bf16 bound in an fp64 emulation of that rounding
    # alone; fp16 rounds 8x finer.  The bf16 twin keeps a full block beside
    # the tail.
    (Workload("mask_rect_dense_q500_k260_d64_fp16", B=1, Hq=2, Hkv=1, Lq=500, Lk=260, D=64, dtype="fp16",
              causal=False, seed=5202), "random"),
    (Workload("mask_rect_dense_q500_k260_d64", B=1, Hq=2, Hkv=1, Lq=500, Lk=260, D=64, causal=False, seed=5202),
     "tail_plus_full"),
    (Workload("mask_window_l2048_gqa_d128", B=1, Hq=8, Hkv=2, Lq=2048, Lk=2048, D=128, seed=5203), "window"),
    (Workload("mask_ragged_l1031_d96_fp16", B=1, Hq=2, Hkv=1, Lq=1031, Lk=1031, D=96, dtype="fp16", std=0.5,
              seed=5204), "random"),
]


@pytest.mark.parametrize("w,kind", CASES, ids=[c[0].name for c in CASES])
def test_masked_chain_matches_oracle(w, kind):
    nqb, nkb = -(-w.Lq // BLK), -(-w.Lk // BLK)
    if kind == "window":
        bm = window_mask(nqb, nkb, 3, off_blocks=(w.Lk - w.Lq) // BLK)
    elif kind == "tail_plus_full":
        bm = np.array([[0, 1, 1], [0, 0, 0], [0, 1, 1], [1, 1, 0]], dtype=np.uint8)
    else:
        bm = random_mask(nqb, nkb, w.seed, empty_row=1 if nqb > 2 else None, empty_col=0 if nkb > 1 else None)
    check_masked(w, bm)


@pytest.mark.parametrize("D", [128, 256])
def test_all_ones_mask_matches_unmasked(D):
    w = Workload(f"mask_ones_l600_d{D}", B=1, Hq=4, Hkv=2, Lq=600, Lk=600, D=D, seed=5300)
    q, k, v, do = make_inputs(w, "cuda")
    bm = torch.ones((-(-w.Lq // BLK), -(-w.Lk // BLK)), dtype=torch.uint8, device="cuda")
    om, lm, dqm, dkm, dvm = masked_chain(w, q, k, v, do, bm)
    o, lse = gbattn.forward(q, k, v, w.scale, w.causal)
    dlt = gbattn.delta(o, do)
    dq, dk, dv = gbattn.backward(q, k, v, o, do, lse, dlt, w.scale, w.causal)
    torch.cuda.synchronize()
    for a, b, n in ((om, o, "O"), (lm, lse, "LSE"), (dqm, dq, "dQ"), (dkm, dk, "dK"), (dvm, dv, "dV")):
        assert torch.equal(a, b), n


def test_all_zero_mask_gives_zeros():
    w = Workload("mask_zero_l300_d64", B=1, Hq=2, Hkv=1, Lq=300, Lk=300, D=64, causal=False, seed=5301)
    q, k, v, do = make_inputs(w, "cuda")
    bm = torch.zeros((-(-w.Lq // BLK), -(-w.Lk // BLK)), dtype=torch.uint8, device="cuda")
    o, lse, dq, dk, dv = masked_chain(w, q, k, v, do, bm)
    assert torch.count_nonzero(o) == 0 and torch.isposinf(lse).all()
    for t, n in ((dq, "dQ"), (dk, "dK"), (dv, "dV")):
        assert torch.count_nonzero(t) == 0, n


def test_masked_rejects_null_mask():
    w2 = Workload("mask_null", B=1, Hq=1, Hkv=1, Lq=128, Lk=128, D=64, seed=5303)
    q, k, v, do = make_inputs(w2, "cuda")
    o, lse = torch.empty_like(q), torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    assert gbattn.attn_fwd_masked(q, k, v, o, lse, None, w2.scale, True, check=False) == gbattn.ATTN_ERR_INVALID_ARG
