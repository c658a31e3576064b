"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (its delta and status word live in the library's fixed scratch array).

Its results must equal those of the allocating entry points (attn_bwd_delta
followed by attn_bwd) within the parity tolerances, on two calls in a row --
the second call reuses the scratch the first one left behind.  This file is
collected last, and it also passes when run alone in a fresh process (the
first call on a device is the one that sets the scratch up).
"""

import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bwd_flashattention_fwd_gb300 import build, gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 2e-2), "fp16": (1e-2, 1e-2)}

CASES = [
    Workload("noalloc_gqa_l300_d128", B=1, Hq=4, Hkv=2, Lq=300, Lk=300, D=128, seed=7001),
    Workload("noalloc_ragged_q190_k250_d96_fp16", B=2, Hq=4, Hkv=4, Lq=190, Lk=250, D=96, dtype="fp16",
             std=0.5, seed=7002),
]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    gbattn.load_library()


def _close(got, ref, dtype, what):
    atol, rtol = TOL[dtype]
    g, r = to_f64(got), to_f64(ref)
    assert np.isfinite(g).all(), what
    bad = np.abs(g - r) > atol + rtol * np.abs(r)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements differ"


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_backward_matches_allocating_path(w):
    q, k, v, do = make_inputs(w, "cuda")
    o, lse = gbattn.forward(q, k, v, w.scale, w.causal)
    dlt = gbattn.delta(o, do)
    dq_ref, dk_ref, dv_ref = gbattn.backward(q, k, v, o, do, lse, dlt, w.scale, w.causal)
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        st = gbattn.load_library().attn_bwd_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, ctypes.c_float(w.scale),
            int(w.causal), gbattn._dtype_code(q), torch.cuda.current_stream().cuda_stream)
        assert st == gbattn.ATTN_OK, gbattn.status_string(st)
        torch.cuda.synchronize()
        if call == 1:
            # set-up is done: the call itself takes no device memory
            free1, _ = torch.cuda.mem_get_info()
            assert free1 == free0, (free0, free1)
        assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
        _close(dq, dq_ref, w.dtype, f"dQ call {call}")
        _close(dk, dk_ref, w.dtype, f"dK call {call}")
        _close(dv, dv_ref, w.dtype, f"dV call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    # B*Hq*Lq = 2**20 + 64 query rows: more delta values than the scratch holds
    w = Workload("noalloc_too_big", B=1, Hq=1, Hkv=1, Lq=2**20 + 64, Lk=2**20 + 64, D=64, seed=7003)
    fake = 0x10000  # never dereferenced: the size check comes first
    st = gbattn.load_library().attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake, w.B, w.Hq,
                                                w.Hkv, w.Lq, w.Lk, w.D, ctypes.c_float(w.scale), 1,
                                                gbattn.ATTN_DTYPE_BF16, None)
    assert st == gbattn.ATTN_ERR_UNSUPPORTED


CAPTURE_CHILD = r"""
import ctypes, sys
import torch
sys.path.insert(0, ROOT)
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs

lib = gbattn.load_library()
torch.cuda.set_device(0)
w = Workload("noalloc_capture", B=1, Hq=2, Hkv=1, Lq=200, Lk=200, D=64, seed=7004)
q, k, v, do = make_inputs(w, "cuda")
o, lse = gbattn.forward(q, k, v, w.scale, True)
dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
args = lambda s: (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D,
                  ctypes.c_float(w.scale), 1, gbattn.ATTN_DTYPE_BF16, s)
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.stream(s):
    g.capture_begin()
    st = lib.attn_bwd_noalloc(*args(s.cuda_stream))
    g.capture_end()
assert st == gbattn.ATTN_ERR_INVALID_ARG, gbattn.status_string(st)
st = lib.attn_bwd_noalloc(*args(torch.cuda.current_stream().cuda_stream))
assert st == gbattn.ATTN_OK, gbattn.status_string(st)
assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
print("first call under capture refused; the next call ran")
"""


def test_noalloc_first_call_under_capture_is_refused():
    """Set-up (the scratch address look-up) must not run inside a stream
    capture: a first call made there is refused, and a later call outside
    capture works.  Runs in a fresh process, where no call has set up yet."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", f"ROOT = {root!r}\n" + CAPTURE_CHILD], cwd=root,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "next call ran" in r.stdout
