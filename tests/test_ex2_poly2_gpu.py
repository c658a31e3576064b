"""ex2_poly2 -- the FMA-pipe 2^x that the dQ and dK/dV kernels use for part
of their exponentials -- against its stated bounds on [-126, 0] (the range
the kernels feed it: P = 2^x <= 1), measured against exact float64 2^x, with
CUDA's exp2f alongside for comparison: relative error at most 7.5e-5 down to
x = -125.9998, and at most 1.45e-4 on the last sliver above the clamp at
-126, where the result is encoded as a subnormal.

The device code is the kernels' own inline function, run by a small kernel in
libgbattn_checks.so."""

import ctypes
import os

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BOUND = 7.5e-5
EDGE = -125.9998    # below this the result's exponent field can be at its minimum
EDGE_BOUND = 1.45e-4
# the final fp32 rounding and the packed fp32 arithmetic add a few units of
# 2^-24 to the polynomial's own error
SLACK = 4 * 2.0 ** -24


@pytest.fixture(scope="module")
def checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bwd_flashattention_fwd_gb300 import build

    build.build()
    lib = ctypes.CDLL(build.CHECKS_LIB)
    lib.gbattn_check_ex2_poly2.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    lib.gbattn_check_ex2_poly2.restype = ctypes.c_int
    return lib


def evaluate(lib, x: np.ndarray) -> np.ndarray:
    xd = torch.from_numpy(x.astype(np.float32)).cuda()
    yd = torch.full_like(xd, float("nan"))
    assert lib.gbattn_check_ex2_poly2(xd.data_ptr(), yd.data_ptr(), xd.numel(),
                                      torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    return yd.cpu().numpy()


def test_ex2_poly2_relative_error_bound(checks):
    rng = np.random.default_rng(11)
    x = np.concatenate([
        np.linspace(-126.0, 0.0, 4_000_001, dtype=np.float32),
        rng.uniform(-126.0, 0.0, 2_000_000).astype(np.float32),
        rng.uniform(-8.0, 0.0, 2_000_000).astype(np.float32),  # where most P values lie
        np.arange(-126, 1, dtype=np.float32),                   # integers: f = 0
        np.arange(-126, 0, dtype=np.float32) + np.float32(0.5),  # the range reduction's ties
        np.nextafter(np.arange(-125, 1, dtype=np.float32) - np.float32(0.5), np.float32(0)),
        np.float32([-0.0, -1e-30, -1e-7]),
    ])
    y = evaluate(checks, x).astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y - exact) / exact
    assert np.isfinite(y).all()
    main = x >= np.float32(EDGE)
    worst = int(np.argmax(np.where(main, rel, 0.0)))
    assert rel[main].max() <= BOUND + SLACK, f"max relative error {rel[main].max():.3g} at x = {x[worst]!r}"
    assert rel.max() <= EDGE_BOUND + SLACK, f"max relative error {rel.max():.3g} near the clamp"
    # exp2f on the same device, for comparison (it is far more accurate)
    ref = torch.exp2(torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    assert (np.abs(ref - exact) / exact).max() < 1e-6


def test_ex2_poly2_clamps_below_range(checks):
    """Inputs below -126 are evaluated at -126, i.e. give 2^-126 within the
    bound (the kernels meet them only for keys whose probability is far below
    the 16-bit types' resolution)."""
    y = evaluate(checks, np.float32([-126.0, -127.0, -200.0, -1e30])).astype(np.float64)
    assert np.all(y == y[0])
    assert abs(y[0] / 2.0 ** -126 - 1.0) <= EDGE_BOUND + SLACK
