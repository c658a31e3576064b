"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (per element): |gpu - ref| <= 2e-2 + 2e-2 |ref| for bf16 outputs,
1e-2 + 1e-2 |ref| for fp16 outputs, and 1e-3 absolute for the float32 LSE
(base 2) and delta.

The forward/backward chain is compared end to end: the GPU backward consumes
the GPU's own lse and delta (delta from the bf16/fp16 O the forward stored),
the oracle works from its exact O.  delta itself is checked on its own, on a
seeded O that does not come from the forward.
"""

import math

import numpy as np
import pytest
import torch

import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import MEMORY_CHECK, WORKLOADS, Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "fp16": (1e-2, 1e-2)}
LSE_ATOL = 1e-3
DELTA_ATOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    gbattn.load_library()


def assert_close(gpu, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g = gpu if isinstance(gpu, np.ndarray) else to_f64(gpu)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst at {idx}: "
                             f"gpu {g[idx]:.6g} ref {ref[idx]:.6g}")


def assert_abs(gpu, ref, atol, what):
    g = gpu if isinstance(gpu, np.ndarray) else to_f64(gpu)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    if (err > atol).any():
        idx = np.unravel_index(np.argmax(err), err.shape)
        raise AssertionError(f"{what}: max abs err {err.max():.3g} at {idx}: gpu {g[idx]} ref {ref[idx]}")


def nan_like(t, shape=None, dtype=None):
    """An output buffer filled with NaN, so that an element no kernel writes
    stays non-finite and fails the checks."""
    return torch.full(t.shape if shape is None else shape, float("nan"), dtype=t.dtype if dtype is None else dtype,
                      device=t.device)


def run_chain(w: Workload, q, k, v, do):
    """fwd -> delta -> bwd through the C ABI on the current stream, into
    NaN-filled outputs."""
    rows = (w.B, w.Hq, w.Lq)
    o, lse, dlt = nan_like(q), nan_like(q, rows, torch.float32), nan_like(q, rows, torch.float32)
    dq, dk, dv = nan_like(q), nan_like(k), nan_like(v)
    gbattn.attn_fwd(q, k, v, o, lse, w.scale, w.causal)
    gbattn.attn_bwd_delta(o, do, dlt)
    gbattn.attn_bwd(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, w.causal)
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    return o, lse, dlt, dq, dk, dv


def check_full(w: Workload):
    q, k, v, do = make_inputs(w, "cuda")
    o, lse, dlt, dq, dk, dv = run_chain(w, q, k, v, do)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal)
    assert_close(o, o_ref, w.dtype, "O")
    assert_abs(lse, lse_ref, LSE_ATOL, "LSE")
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal)
    assert_close(dq, dq_ref, w.dtype, "dQ")
    assert_close(dk, dk_ref, w.dtype, "dK")
    assert_close(dv, dv_ref, w.dtype, "dV")


# ---------------------------------------------------------------------------
# Element-by-element parity on problems the oracle finishes in seconds
# ---------------------------------------------------------------------------

SMALL = [WORKLOADS["tiny_gqa_l128_d64"]]
for D in (64, 96, 128, 256):
    for dt in ("bf16", "fp16"):
        for causal in (True, False):
            SMALL.append(Workload(f"d{D}_{dt}_{'causal' if causal else 'dense'}_l300", B=1, Hq=4, Hkv=2,
                                  Lq=300, Lk=300, D=D, dtype=dt, causal=causal, seed=2000 + D))
SMALL += [
    Workload("rect_causal_q200_k333_d128", B=1, Hq=2, Hkv=1, Lq=200, Lk=333, D=128, seed=3001),
    Workload("rect_dense_q200_k333_d64_fp16", B=1, Hq=2, Hkv=2, Lq=200, Lk=333, D=64, dtype="fp16",
             causal=False, seed=3002),
    Workload("rect_causal_q77_k700_d96_fp16", B=2, Hq=2, Hkv=1, Lq=77, Lk=700, D=96, dtype="fp16",
             std=0.5, seed=3003),
    Workload("rect_causal_q130_k4100_d256", B=1, Hq=2, Hkv=1, Lq=130, Lk=4100, D=256, seed=3004),
    Workload("single_query_row_k1000", B=1, Hq=4, Hkv=1, Lq=1, Lk=1000, D=128, seed=3005),
    Workload("single_row_single_key", B=1, Hq=1, Hkv=1, Lq=1, Lk=1, D=64, seed=3006),
    Workload("dense_single_key", B=2, Hq=2, Hkv=1, Lq=9, Lk=1, D=128, causal=False, seed=3007),
    Workload("odd_1031_d128", B=1, Hq=2, Hkv=1, Lq=1031, Lk=1031, D=128, seed=3008),
    Workload("odd_2049_d64_fp16", B=1, Hq=2, Hkv=2, Lq=2049, Lk=2049, D=64, dtype="fp16", seed=3009),
]
# the correctness grid of "When the Bottleneck Moved" (section 3): lengths 61,
# 64, 257; head dims 64, 128; batch 1 and 2; GQA 32/8 at length 64
for L in (61, 64, 257):
    for D in (64, 128):
        for B in (1, 2):
            SMALL.append(Workload(f"grid_l{L}_d{D}_b{B}", B=B, Hq=2, Hkv=2, Lq=L, Lk=L, D=D, seed=4000 + L + D + B))
SMALL.append(Workload("grid_gqa32_8_l64_d128", B=1, Hq=32, Hkv=8, Lq=64, Lk=64, D=128, seed=4100))


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_chain_matches_oracle(w):
    check_full(w)


# Problems with more work items than a GB300 has SMs, compared on every output
# element: the persistent forward (items of 256 query rows) and dQ (items of
# 128 query rows) kernels launch one CTA per SM, so only here does a CTA run
# several items -- the next-item prefetch, the item-boundary hand-over and the
# snake order of the work list.  Outputs start as NaN, so an item no CTA
# writes fails.  The first is the B2 Hq32 Hkv8 L2048 D128 workload itself
# (512 forward items, 1024 dQ items).
MULTI_ITEM = [
    WORKLOADS["llama_gqa_l2048_d128"],
    Workload("multi_item_ragged_q1100_k1300_d96_fp16", B=2, Hq=16, Hkv=4, Lq=1100, Lk=1300, D=96, dtype="fp16",
             std=0.5, seed=3101),
    Workload("multi_item_dense_l900_d64", B=3, Hq=16, Hkv=2, Lq=900, Lk=900, D=64, causal=False, seed=3102),
    Workload("multi_key_tile_l1536_d256", B=1, Hq=8, Hkv=2, Lq=1536, Lk=1536, D=256, seed=3103),
]


@pytest.mark.parametrize("w", MULTI_ITEM, ids=[w.name for w in MULTI_ITEM])
def test_multi_item_every_element(w):
    check_full(w)


@pytest.mark.parametrize("D", [64, 96, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_delta_matches_oracle(D, dtype):
    w = Workload("delta", B=2, Hq=3, Hkv=3, Lq=1001, Lk=1001, D=D, dtype=dtype, seed=5000 + D)
    o, _, _, do = make_inputs(w, "cuda")  # O drawn independently of any forward
    d = gbattn.delta(o, do)
    torch.cuda.synchronize()
    assert_abs(d, A.delta(to_f64(o), to_f64(do)), DELTA_ATOL, "delta")


@pytest.mark.parametrize("w", [SMALL[0], SMALL[5], SMALL[-1]], ids=lambda w: w.name)
def test_backward_alone_with_oracle_lse_delta(w):
    """The backward kernels fed the oracle's lse/delta (rounded to fp32)."""
    q, k, v, do = make_inputs(w, "cuda")
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal)
    lse = torch.tensor(lse_ref, dtype=torch.float32, device="cuda")
    dlt = torch.tensor(A.delta(o_ref, dod), dtype=torch.float32, device="cuda")
    o = torch.tensor(o_ref, dtype=w.torch_dtype, device="cuda")
    dq, dk, dv = gbattn.backward(q, k, v, o, do, lse, dlt, w.scale, w.causal)
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal)
    assert_close(dq, dq_ref, w.dtype, "dQ")
    assert_close(dk, dk_ref, w.dtype, "dK")
    assert_close(dv, dv_ref, w.dtype, "dV")


def test_guard_bands_untouched():
    """Outputs written into the middle of NaN-filled buffers: nothing outside
    the output's extent changes (ragged Q and K tails)."""
    w = Workload("guard", B=2, Hq=4, Hkv=2, Lq=190, Lk=250, D=96, dtype="fp16", seed=6000)
    q, k, v, do = make_inputs(w, "cuda")
    pad = 4096

    def guarded(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + 2 * pad,), float("nan"), dtype=dtype, device="cuda")
        return buf, buf[pad:pad + n].view(shape)

    ob, o = guarded(q.shape, q.dtype)
    lb, lse = guarded((2, 4, 190), torch.float32)
    db, dlt = guarded((2, 4, 190), torch.float32)
    dqb, dq = guarded(q.shape, q.dtype)
    dkb, dk = guarded(k.shape, k.dtype)
    dvb, dv = guarded(v.shape, v.dtype)
    gbattn.attn_fwd(q, k, v, o, lse, w.scale, True)
    gbattn.attn_bwd_delta(o, do, dlt)
    gbattn.attn_bwd(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, True)
    torch.cuda.synchronize()
    for buf, name in ((ob, "o"), (lb, "lse"), (db, "delta"), (dqb, "dq"), (dkb, "dk"), (dvb, "dv")):
        assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[-pad:]).all(), f"{name} guard band written"
        assert not torch.isnan(buf[pad:-pad]).any(), f"{name} has unwritten elements"
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, True)
    assert_close(o, o_ref, "fp16", "O")


def test_stale_rows_behind_kv_do_not_leak():
    """K/V live at the front of larger buffers whose tail holds large finite
    stale rows; a read past Lk would show in O and the gradients."""
    w = Workload("stale", B=1, Hq=2, Hkv=1, Lq=100, Lk=180, D=128, seed=6100)
    q, k, v, do = make_inputs(w, "cuda")
    kb = torch.full((1, 1, 512, 128), 3.0e4, dtype=k.dtype, device="cuda")
    vb = torch.full((1, 1, 512, 128), -3.0e4, dtype=v.dtype, device="cuda")
    kb[:, :, :180].copy_(k)
    vb[:, :, :180].copy_(v)
    ks = kb.view(-1)[: k.numel()].view(k.shape)
    vs = vb.view(-1)[: v.numel()].view(v.shape)
    o, lse, dlt, dq, dk, dv = run_chain(w, q, ks, vs, do)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, True)
    assert_close(o, o_ref, "bf16", "O")
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, True)
    assert_close(dq, dq_ref, "bf16", "dQ")
    assert_close(dk, dk_ref, "bf16", "dK")


def test_deterministic():
    """No atomics anywhere: two runs give identical bits."""
    w = WORKLOADS["llama_gqa_l2048_d128"].with_(B=1, Lq=1000, Lk=1000)
    q, k, v, do = make_inputs(w, "cuda")
    a = run_chain(w, q, k, v, do)
    b = run_chain(w, q, k, v, do)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# The named workloads at full size: sampled outputs against the oracle
# ---------------------------------------------------------------------------


def _sample_rows(L, rng):
    base = [0, 1, 63, 64, 127, 128, 129, L // 2, L - 129, L - 128, L - 2, L - 1]
    extra = rng.integers(0, L, size=8).tolist()
    return sorted({r for r in base + extra if 0 <= r < L})


def check_sampled(w: Workload):
    rng = np.random.default_rng(w.seed)
    q, k, v, do = make_inputs(w, "cuda")
    o, lse, dlt, dq, dk, dv = run_chain(w, q, k, v, do)
    for t, name in ((o, "o"), (lse, "lse"), (dlt, "delta"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        assert torch.isfinite(t).all(), f"{name}: elements left unwritten (NaN) or non-finite"
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    G = w.Hq // w.Hkv
    heads = sorted({(0, 0), (w.B - 1, w.Hq - 1), (w.B // 2, w.Hq // 2)})
    rows = _sample_rows(w.Lq, rng)
    o_cpu, lse_cpu, dq_cpu = to_f64(o), to_f64(lse), to_f64(dq)
    o_ref_all = np.zeros_like(dod)  # oracle O, filled only where the checks read it
    for b, hq in heads:
        o_ref, lse_ref = A.forward_rows(qd, kd, vd, w.scale, w.causal, b, hq, rows)
        assert_close(o_cpu[b, hq, rows], o_ref, w.dtype, f"O[{b},{hq}]")
        assert_abs(lse_cpu[b, hq, rows], lse_ref, LSE_ATOL, f"LSE[{b},{hq}]")
        o_ref_all[b, hq, rows] = o_ref
        dq_ref = A.backward_query_rows(qd, kd, vd, o_ref_all, dod, w.scale, w.causal, b, hq, rows)
        assert_close(dq_cpu[b, hq, rows], dq_ref, w.dtype, f"dQ[{b},{hq}]")
    keys = _sample_rows(w.Lk, rng)
    dk_cpu, dv_cpu = to_f64(dk), to_f64(dv)
    for b, hk in sorted({(0, 0), (w.B - 1, w.Hkv - 1)}):
        for g in range(G):
            hq = hk * G + g
            o_ref_all[b, hq] = oracle_head_output(qd, kd, vd, w, b, hq)
        dk_ref, dv_ref = A.backward_key_rows(qd, kd, vd, o_ref_all, dod, w.scale, w.causal, b, hk, keys)
        assert_close(dk_cpu[b, hk, keys], dk_ref, w.dtype, f"dK[{b},{hk}]")
        assert_close(dv_cpu[b, hk, keys], dv_ref, w.dtype, f"dV[{b},{hk}]")


def oracle_head_output(qd, kd, vd, w, b, hq):
    """The oracle's O for every row of head (b, hq), in row blocks."""
    out = np.empty((w.Lq, w.D))
    for r0 in range(0, w.Lq, 1024):
        rows = list(range(r0, min(w.Lq, r0 + 1024)))
        out[rows], _ = A.forward_rows(qd, kd, vd, w.scale, w.causal, b, hq, rows)
    return out


FULL = [WORKLOADS[n] for n in ("llama_gqa_l2048_d128", "qwen3_8b_gqa_l8192_d128", "gqa_l8192_d256",
                               "ragged_mha_q4064_k4112_d96", "longcache_q1024_k8192_d128",
                               "longcache_q2048_k8192_d256")]


@pytest.mark.parametrize("w", FULL, ids=[w.name for w in FULL])
def test_workload_sampled(w):
    check_sampled(w)


def test_long_context_memory_and_sampled_parity():
    """L = 23040: the path allocates nothing beyond the caller's tensors (no
    Lq x Lk buffer), and sampled outputs match the oracle."""
    w = MEMORY_CHECK
    q, k, v, do = make_inputs(w, "cuda")
    rows = (w.B, w.Hq, w.Lq)
    o, lse, dlt = nan_like(q), nan_like(q, rows, torch.float32), nan_like(q, rows, torch.float32)
    dq, dk, dv = nan_like(q), nan_like(k), nan_like(v)
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    free0, _ = torch.cuda.mem_get_info()
    gbattn.attn_fwd(q, k, v, o, lse, w.scale, True)
    gbattn.attn_bwd_delta(o, do, dlt)
    gbattn.attn_bwd(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, True)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.max_memory_allocated() == base
    assert free0 - free1 <= 4 * 2**20, (free0 - free1)
    assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
    for t, name in ((o, "o"), (lse, "lse"), (dlt, "delta"), (dq, "dq"), (dk, "dk"), (dv, "dv")):
        assert torch.isfinite(t).all(), f"{name}: elements left unwritten (NaN) or non-finite"
    rng = np.random.default_rng(1)
    rows = _sample_rows(w.Lq, rng)
    qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
    o_ref, lse_ref = A.forward_rows(qd, kd, vd, w.scale, True, 0, 5, rows)
    assert_close(to_f64(o)[0, 5, rows], o_ref, "bf16", "O")
    assert_abs(to_f64(lse)[0, 5, rows], lse_ref, LSE_ATOL, "LSE")
    o_full = np.zeros_like(dod)
    o_full[0, 5, rows] = o_ref
    dq_ref = A.backward_query_rows(qd, kd, vd, o_full, dod, w.scale, True, 0, 5, rows)
    assert_close(to_f64(dq)[0, 5, rows], dq_ref, "bf16", "dQ")


def test_binding_rejects_bad_layouts():
    """Non-contiguous tensors, a float32 tensor where a 16-bit one belongs and
    mixed 16-bit types are refused by the binding before the C ABI."""
    w = Workload("layout", B=1, Hq=2, Hkv=1, Lq=64, Lk=64, D=64, seed=6200)
    q, k, v, do = make_inputs(w, "cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 2, 64), dtype=torch.float32, device="cuda")
    qt = q.transpose(2, 3).contiguous().transpose(2, 3)  # same shape, D not the fastest axis
    with pytest.raises(ValueError, match="not contiguous"):
        gbattn.attn_fwd(qt, k, v, o, lse, w.scale, True)
    with pytest.raises(TypeError):
        gbattn.attn_fwd(q.float(), k, v, o, lse, w.scale, True)
    with pytest.raises(TypeError):
        gbattn.attn_fwd(q, k.half(), v, o, lse, w.scale, True)
    with pytest.raises(TypeError):
        gbattn.attn_fwd(q, k, v, o, lse.double(), w.scale, True)
