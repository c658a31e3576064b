"""K and V sliced out of a longer cache ("Add a fused full-attention path for
head_dim 256 on NAX devices", section "Ragged causal inputs"; its tests put
large finite stale rows behind the slice so that any read past Lk shows).

attn_fwd_ex / attn_bwd_ex read k and v as the first Lk rows of each head of a
[B, Hkv, capacity, D] buffer.  They must give the same bits as the contiguous
calls on the same values, and the oracle's result, whatever the stale rows
hold (large finite values, or NaN)."""

import numpy as np
import pytest
import torch

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, block_mask, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "fp16": (1e-2, 1e-2)}


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
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, max err {err.max():.3g}"


def cache_slice(t, capacity, stale):
    """t [B, H, L, D] copied into the front of a [B, H, capacity, D] buffer
    whose remaining rows hold `stale`; returns the [:, :, :L] view."""
    B, H, L, D = t.shape
    buf = torch.full((B, H, capacity, D), stale, dtype=t.dtype, device=t.device)
    if stale == stale:  # finite: alternate the sign row by row
        buf[:, :, L::2] = -stale
    buf[:, :, :L].copy_(t)
    return buf[:, :, :L]


def chain(w, q, k, v, do, bm=None, ex=True):
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device=q.device)
    dq = torch.empty_like(q)
    dk = torch.empty((w.B, w.Hkv, w.Lk, w.D), dtype=q.dtype, device=q.device)
    dv = torch.empty_like(dk)
    if ex:
        gbattn.attn_fwd_ex(q, k, v, o, lse, w.scale, w.causal, block_mask=bm)
    elif bm is None:
        gbattn.attn_fwd(q, k, v, o, lse, w.scale, w.causal)
    else:
        gbattn.attn_fwd_masked(q, k, v, o, lse, bm, w.scale, w.causal)
    dlt = gbattn.delta(o, do)
    if ex:
        gbattn.attn_bwd_ex(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, w.causal, block_mask=bm)
    elif bm is None:
        gbattn.attn_bwd(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, w.causal)
    else:
        gbattn.attn_bwd_masked(q, k, v, o, do, lse, dlt, bm, dq, dk, dv, w.scale, w.causal)
    torch.cuda.synchronize()
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    return o, lse, dq, dk, dv


CASES = [
    (Workload("slice_d64_causal_q300_k520", B=2, Hq=4, Hkv=2, Lq=300, Lk=520, D=64, seed=7001), 640, 3.0e4),
    (Workload("slice_d96_fp16_dense_257", B=1, Hq=2, Hkv=2, Lq=257, Lk=257, D=96, dtype="fp16", causal=False,
              seed=7002), 300, float("nan")),
    (Workload("slice_d128_gqa_q700_k1031", B=1, Hq=8, Hkv=2, Lq=700, Lk=1031, D=128, seed=7003), 1280, 3.0e4),
    (Workload("slice_d256_q200_k333_cap3329", B=1, Hq=4, Hkv=2, Lq=200, Lk=333, D=256, seed=7004), 3329,
     float("nan")),
]


@pytest.mark.parametrize("w,cap,stale", CASES, ids=[c[0].name for c in CASES])
def test_slice_matches_contiguous_and_oracle(w, cap, stale):
    q, k, v, do = make_inputs(w, "cuda")
    ks, vs = cache_slice(k, cap, stale), cache_slice(v, cap, stale)
    assert gbattn.kv_row_pitch(ks, vs) == cap
    got = chain(w, q, ks, vs, do)
    ref = chain(w, q, k, v, do, ex=False)
    for a, b, n in zip(got, ref, ("O", "LSE", "dQ", "dK", "dV")):
        assert torch.equal(a, b), n
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, _, _ = A.forward(qd, kd, vd, w.scale, w.causal)
    assert_close(got[0], o_ref, w.dtype, "O")
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal)
    assert_close(got[2], dq_ref, w.dtype, "dQ")
    assert_close(got[3], dk_ref, w.dtype, "dK")
    assert_close(got[4], dv_ref, w.dtype, "dV")


def test_slice_with_block_mask():
    w = Workload("slice_mask_d128_q600_k900", B=1, Hq=4, Hkv=1, Lq=600, Lk=900, D=128, seed=7005)
    q, k, v, do = make_inputs(w, "cuda")
    ks, vs = cache_slice(k, 1024, float("nan")), cache_slice(v, 1024, float("nan"))
    bm = torch.from_numpy(block_mask("window:3", w.Lq, w.Lk)).cuda()
    got = chain(w, q, ks, vs, do, bm)
    ref = chain(w, q, k, v, do, bm, ex=False)
    for a, b, n in zip(got, ref, ("O", "LSE", "dQ", "dK", "dV")):
        assert torch.equal(a, b), n


def test_explicit_pitch_equal_to_lk_is_contiguous():
    w = Workload("pitch_eq_lk", B=1, Hq=2, Hkv=1, Lq=200, Lk=260, D=64, seed=7006)
    q, k, v, do = make_inputs(w, "cuda")
    o1, l1 = torch.empty_like(q), torch.empty((1, 2, 200), dtype=torch.float32, device="cuda")
    o2, l2 = torch.empty_like(q), torch.empty_like(l1)
    gbattn.attn_fwd_ex(q, k, v, o1, l1, w.scale, True, kv_pitch=w.Lk)
    gbattn.attn_fwd(q, k, v, o2, l2, w.scale, True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_pitch_below_lk_is_rejected():
    w = Workload("pitch_small", B=1, Hq=2, Hkv=1, Lq=200, Lk=260, D=64, seed=7007)
    q, k, v, do = make_inputs(w, "cuda")
    o, lse = torch.empty_like(q), torch.empty((1, 2, 200), dtype=torch.float32, device="cuda")
    st = gbattn.attn_fwd_ex(q, k, v, o, lse, w.scale, True, kv_pitch=w.Lk - 1, check=False)
    assert st == gbattn.ATTN_ERR_INVALID_ARG
