"""The debug build (libgbattn_debug.so: the same kernels compiled with
GBATTN_DEBUG_CHECKS, every plain global load and store checked against its
tensor's extent).

* The check itself: run on an index range outside the extent it records
  kDevBoundsBase + site in the status word, and inside it records nothing
  (libgbattn_checks.so runs the same check on chosen numbers and touches no
  memory at those indices).
* The kernels under the checks: every path of the library (every head
  dimension, masked, sliced K/V, decode-shaped, the no-allocation entry
  point, the linear cross-entropy) runs in the debug build, no check fires
  (attn_last_device_status stays ATTN_OK), and the results match the oracle.
  The library is chosen per process (GBATTN_DEBUG=1), so this runs in a child.
"""

import ctypes
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BOUNDS_BASE = 200  # kDevBoundsBase in kernel_common.cuh


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    build.build(debug=True)


def test_index_check_records_and_skips():
    from bwd_flashattention_fwd_gb300 import build

    lib = ctypes.CDLL(build.CHECKS_LIB)
    u64 = ctypes.c_ulonglong
    lib.gbattn_check_index.argtypes = [ctypes.c_void_p, u64, u64, u64, ctypes.c_int, ctypes.c_void_p]
    lib.gbattn_check_index.restype = ctypes.c_int
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for first, count, extent in ((0, 32, 32), (96, 32, 128), (5, 1, 6)):
        assert lib.gbattn_check_index(status.data_ptr(), first, count, extent, 7, s) == 0
    torch.cuda.synchronize()
    assert status.item() == 0
    assert lib.gbattn_check_index(status.data_ptr(), 100, 32, 128, 9, s) == 0  # runs 4 past the end
    torch.cuda.synchronize()
    assert status.item() == BOUNDS_BASE + 9
    # the first failure is kept
    assert lib.gbattn_check_index(status.data_ptr(), 2**63, 2**63, 10, 3, s) == 0  # wraps around
    torch.cuda.synchronize()
    assert status.item() == BOUNDS_BASE + 9


CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import oracle.attention as A
import oracle.linear_ce as L
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import (LCE_WORKLOADS, Workload, block_mask, make_inputs,
                                                make_lce_inputs, to_f64)

lib = gbattn.load_library()
assert lib._name.endswith("libgbattn_debug.so"), lib._name
torch.cuda.set_device(0)

def close(got, ref, dt, what):
    atol = 2e-2 if dt == "bf16" else 1e-2
    err = np.abs(to_f64(got) - ref)
    assert (err <= atol + atol * np.abs(ref)).all(), (what, float(err.max()))

def check(w, bm=None, pitch=0, decode=False, noalloc=False):
    q, k, v, do = make_inputs(w, "cuda")
    if pitch:
        caches = []
        for t in (k, v):
            c = torch.full((w.B, w.Hkv, pitch, w.D), float("nan"), dtype=t.dtype, device="cuda")
            c[:, :, :w.Lk].copy_(t)
            caches.append(c[:, :, :w.Lk])
        k, v = caches
    bmt = None if bm is None else torch.from_numpy(bm).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty(k.shape, dtype=k.dtype, device="cuda"), torch.empty(v.shape, dtype=v.dtype, device="cuda")
    if decode:
        ws = gbattn.decode_workspace(q, k)
        gbattn.attn_fwd_decode(q, k, v, o, lse, ws, w.scale, w.causal)
        dlt = gbattn.delta(o, do)
        gbattn.attn_bwd_decode(q, k, v, o, do, lse, dlt, dq, dk, dv, ws, w.scale, w.causal)
    else:
        gbattn.attn_fwd_ex(q, k, v, o, lse, w.scale, w.causal, block_mask=bmt)
        dlt = gbattn.delta(o, do)
        if noalloc:
            gbattn.attn_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.scale, w.causal)
        else:
            gbattn.attn_bwd_ex(q, k, v, o, do, lse, dlt, dq, dk, dv, w.scale, w.causal, block_mask=bmt)
    st = gbattn.attn_last_device_status()
    assert st == gbattn.ATTN_OK, (w.name, gbattn.status_string(st))
    qd, kd, vd, dod = (to_f64(t) for t in make_inputs(w, "cpu"))
    o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, w.causal, bm)
    dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, w.causal, bm)
    for name, got, ref in (("O", o, o_ref), ("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)):
        close(got, ref, w.dtype, (w.name, name))

for D in (64, 96, 128, 256):
    check(Workload(f"dbg_d{D}", B=2, Hq=4, Hkv=2, Lq=300, Lk=333, D=D, seed=9000 + D))
check(Workload("dbg_dense_fp16", B=1, Hq=2, Hkv=1, Lq=200, Lk=130, D=64, dtype="fp16", causal=False, seed=9001))
wm = Workload("dbg_mask", B=1, Hq=4, Hkv=2, Lq=700, Lk=700, D=128, seed=9002)
check(wm, bm=block_mask("random:0.5", wm.Lq, wm.Lk, seed=9002))
wm2 = Workload("dbg_mask_256", B=1, Hq=4, Hkv=1, Lq=400, Lk=600, D=256, seed=9003)
check(wm2, bm=block_mask("window:2", wm2.Lq, wm2.Lk))
check(Workload("dbg_slice", B=2, Hq=4, Hkv=2, Lq=150, Lk=260, D=96, dtype="fp16", seed=9004), pitch=400)
check(Workload("dbg_slice_256", B=1, Hq=2, Hkv=1, Lq=150, Lk=260, D=256, seed=9005), pitch=300)
check(Workload("dbg_decode", B=2, Hq=8, Hkv=2, Lq=3, Lk=1000, D=128, seed=9006), decode=True)
check(Workload("dbg_decode_256", B=1, Hq=4, Hkv=1, Lq=2, Lk=700, D=256, seed=9007), decode=True)
check(Workload("dbg_noalloc", B=1, Hq=4, Hkv=2, Lq=300, Lk=300, D=64, seed=9008), noalloc=True)
check(Workload("dbg_multi_item", B=2, Hq=32, Hkv=8, Lq=700, Lk=700, D=128, seed=9009))

lw = LCE_WORKLOADS["lce_tiny_n200_d128_v1000"]
h, wt, t, dloss = make_lce_inputs(lw, "cuda")
ws = gbattn.lce_workspace(h, wt)
loss = torch.empty(lw.N, dtype=torch.float32, device="cuda")
lse = torch.empty_like(loss)
gbattn.lce_fwd(h, wt, t, loss, lse, ws)
dh, dw = torch.empty_like(h), torch.empty_like(wt)
gbattn.lce_bwd(h, wt, t, lse, dloss, dh, dw, ws)
assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
loss_ref, _ = L.forward(to_f64(h), to_f64(wt), t.cpu().numpy().astype(np.int64))
assert np.abs(to_f64(loss) - loss_ref).max() <= 1e-3
print("debug build: no index check fired; results match the oracle")
"""


def test_kernels_pass_their_index_checks():
    env = dict(os.environ, GBATTN_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "no index check fired" in r.stdout
