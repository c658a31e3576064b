"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (its delta and status word live in the library's fixed scratch array).

Its results must equal those of the allocating entry points (attn_bwd_delta
followed by attn_bwd) within the parity tolerances, on two calls in a row --
the second call reuses the scratch the first one left behind.  This file is
collected last, and it also passes when run alone in a fresh process (the
first call on a device is the one that sets the scratch up).
"""

import ctypes

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
        st = gbattn.load_library().attn_bwd_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(), dq.data_ptr(),
            dk.data_ptr(), dv.data_ptr(), w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D, ctypes.c_float(w.scale),
            int(w.causal), gbattn._dtype_code(q), torch.cuda.current_stream().cuda_stream)
        assert st == gbattn.ATTN_OK, gbattn.status_string(st)
        torch.cuda.synchronize()
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
