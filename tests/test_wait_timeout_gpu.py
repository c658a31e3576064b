"""The failure-reporting path on the GPU: a bounded device wait that runs out
is reported as ATTN_ERR_TIMEOUT, the report clears, and the context stays
usable for a normal call afterwards.

The wait that runs out is attn_wait_probe's (a wait on an mbarrier nothing
completes), never a real kernel's: no copy or MMA is in flight when it gives
up.  The limit is set to 50 ms through GBATTN_WAIT_LIMIT_NS, which the
library reads once per process, so the check runs in a child process.
"""

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, time
import numpy as np
import torch
sys.path.insert(0, ROOT)
import oracle.attention as A
from bwd_flashattention_fwd_gb300 import gbattn
from bwd_flashattention_fwd_gb300.inputs import Workload, make_inputs, to_f64

gbattn.load_library()
torch.cuda.set_device(0)
assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
t0 = time.perf_counter()
gbattn.attn_wait_probe()
st = gbattn.attn_last_device_status()
dt = time.perf_counter() - t0
assert st == gbattn.ATTN_ERR_TIMEOUT, gbattn.status_string(st)
assert 0.04 <= dt < 5.0, dt  # the 50 ms limit, not the 2 s default
assert gbattn.attn_last_device_status() == gbattn.ATTN_OK  # the report was cleared

# a normal call afterwards: same context, correct results, no timeout
w = Workload("after_timeout", B=1, Hq=4, Hkv=2, Lq=300, Lk=300, D=128, seed=7100)
q, k, v, do = make_inputs(w, "cuda")
o, lse = gbattn.forward(q, k, v, w.scale, True)
dq, dk, dv = gbattn.backward(q, k, v, o, do, lse, gbattn.delta(o, do), w.scale, True)
assert gbattn.attn_last_device_status() == gbattn.ATTN_OK
qd, kd, vd, dod = (to_f64(t) for t in (q, k, v, do))
o_ref, lse_ref, _ = A.forward(qd, kd, vd, w.scale, True)
dq_ref, dk_ref, dv_ref = A.backward(qd, kd, vd, o_ref, dod, w.scale, True)
for name, got, ref in (("O", o, o_ref), ("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)):
    err = np.abs(to_f64(got) - ref)
    assert (err <= 2e-2 + 2e-2 * np.abs(ref)).all(), (name, err.max())
print("timeout reported, cleared, and a normal call afterwards matched the oracle")
"""


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()


def test_wait_probe_reports_timeout_then_context_is_usable():
    env = dict(os.environ, GBATTN_WAIT_LIMIT_NS="50000000")
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + CHILD], env=env, cwd=ROOT,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]
    assert "matched the oracle" in r.stdout
