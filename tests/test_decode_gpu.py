"""GPU parity of the decode-shaped calls (attn_fwd_decode, attn_bwd_decode)
against the fp64 oracle: short query lengths ("feat(attention): complete
Flash Attention VJP implementation": vector kernels for sequences of at most
8) against key ranges of a few hundred to several thousand, every head
dimension, GQA groups of 1 to 8, causal (bottom-right) and dense.

The key range of each KV head is split over CTAs; with Lk = 1025 the last
split holds a single key that most rows of a causal problem cannot see, so
their partial result is empty and the merge must ignore it."""

import numpy as np
import pytest
import torch

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "fp16": (1e-2, 1e-2)}
LSE_ATOL = 1e-3


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
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g}")


def decode_chain(w: Workload, q, k, v, do):
    ws = gbattn.decode_workspace(q, k)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device=q.device)
    gbattn.attn_fwd_decode(q, k, v, o, lse, ws, w.scale, w.causal)
    dlt = gbattn.delta(o, do)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    gbattn.attn_bwd_decode(q, k, v, o, do, lse, dlt, dq, dk, dv, ws, w.scale, w.causal)
    torch.cuda.synchronize()
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    return o, lse, dq, dk, dv


CASES = []
for D, dtype in ((64, "bf16"), (96, "fp16"), (128, "bf16"), (256, "bf16")):
    CASES.append(Workload(f"dec_d{D}_g4_q8_k1000", B=2, Hq=8, Hkv=2, Lq=8, Lk=1000, D=D, dtype=dtype,
                          seed=8000 + D))
    CASES.append(Workload(f"dec_d{D}_g1_q1_k300_dense", B=1, Hq=3, Hkv=3, Lq=1, Lk=300, D=D, dtype=dtype,
                          causal=False, seed=8100 + D))
CASES += [
    Workload("dec_d128_g8_q3_k4097", B=1, Hq=16, Hkv=2, Lq=3, Lk=4097, D=128, seed=8201),
    Workload("dec_d128_g1_q8_k1025_split_tail", B=1, Hq=1, Hkv=1, Lq=8, Lk=1025, D=128, seed=8202),
    Workload("dec_d64_g16_q8_k777", B=1, Hq=16, Hkv=1, Lq=8, Lk=777, D=64, seed=8203),
    Workload("dec_d256_g8_q2_k2050_fp16", B=1, Hq=8, Hkv=1, Lq=2, Lk=2050, D=256, dtype="fp16", std=0.5,
             seed=8204),
    Workload("dec_d96_q5_eq_k5", B=1, Hq=4, Hkv=2, Lq=5, Lk=5, D=96, seed=8205),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_decode_matches_oracle(w):
    q, k, v, do = make_inputs(w, "cuda")
    o, lse, dq, dk, dv = decode_chain(w, q, k, v, do)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal)
    assert_close(o, o_ref, w.dtype, "O")
    err = np.abs(to_f64(lse) - lse_ref).max()
    assert err <= LSE_ATOL, f"LSE max abs err {err:.3g}"
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal)
    assert_close(dq, dq_ref, w.dtype, "dQ")
    assert_close(dk, dk_ref, w.dtype, "dK")
    assert_close(dv, dv_ref, w.dtype, "dV")


def test_decode_agrees_with_general_path():
    """Same problem through attn_fwd / attn_bwd: dK and dV come from the same
    kernel (identical bits); O, lse and dQ differ only by summation order."""
    w = Workload("dec_vs_general", B=2, Hq=32, Hkv=8, Lq=4, Lk=2048, D=128, seed=8300)
    q, k, v, do = make_inputs(w, "cuda")
    o, lse, dq, dk, dv = decode_chain(w, q, k, v, do)
    o2, lse2 = gbattn.forward(q, k, v, w.scale, w.causal)
    dq2, dk2, dv2 = gbattn.backward(q, k, v, o2, do, lse2, gbattn.delta(o2, do), w.scale, w.causal)
    torch.cuda.synchronize()
    assert (lse - lse2).abs().max().item() <= 1e-4
    assert (o.float() - o2.float()).abs().max().item() <= 2e-2
    assert (dq.float() - dq2.float()).abs().max().item() <= 5e-2
    if torch.equal(o, o2):
        assert torch.equal(dk, dk2) and torch.equal(dv, dv2)


def test_decode_rejects_wide_groups_and_small_workspace():
    w = Workload("dec_reject", B=1, Hq=32, Hkv=1, Lq=8, Lk=256, D=64, seed=8301)  # G * Lq = 256
    assert gbattn.attn_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D) == 0
    q, k, v, do = make_inputs(w, "cuda")
    o, lse = torch.empty_like(q), torch.empty((1, 32, 8), dtype=torch.float32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    st = gbattn.attn_fwd_decode(q, k, v, o, lse, ws, w.scale, True, check=False)
    assert st == gbattn.ATTN_ERR_UNSUPPORTED
    w2 = w.with_(Hq=4)
    q, k, v, do = make_inputs(w2, "cuda")
    o, lse = torch.empty_like(q), torch.empty((1, 4, 8), dtype=torch.float32, device="cuda")
    need = gbattn.attn_decode_workspace_bytes(1, 4, 1, 8, 256, 64)
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    st = gbattn.attn_fwd_decode(q, k, v, o, lse, small, w2.scale, True, check=False)
    assert st == gbattn.ATTN_ERR_INVALID_ARG
