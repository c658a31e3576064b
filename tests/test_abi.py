"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/gbattn.h declares, and rejects bad arguments on the host
before touching any device memory."""

import ctypes
import math
import os
import re

import pytest

from bwd_flashattention_fwd_gb300 import build, gbattn

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
HEADERS = [os.path.join(INCLUDE, h) for h in ("gbattn.h", "gblce.h")]
FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


@pytest.fixture(scope="module")
def lib():
    build.build()
    return gbattn.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b((?:attn|lce)_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert set(names) == set(gbattn.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=4, Hkv=2, Lq=64, Lk=64, D=128, scale=0.1,
        causal=1, dtype=1):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Lq, Lk, D, ctypes.c_float(scale), causal, dtype, None)


def bwd(lib, ptrs=None, B=1, Hq=4, Hkv=2, Lq=64, Lk=64, D=128, scale=0.1, causal=1, dtype=1):
    ptrs = ptrs or [FAKE] * 10
    return lib.attn_bwd(*ptrs, B, Hq, Hkv, Lq, Lk, D, ctypes.c_float(scale), causal, dtype, None)


@pytest.mark.parametrize(
    "kw,expected",
    [
        (dict(q=None), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(lse=None), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(q=FAKE + 8), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(B=0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(Lq=0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(Lk=-3, causal=0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(Hkv=3), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(Hkv=0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(Lq=65, Lk=64), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(scale=0.0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(scale=-1.0), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(scale=math.nan), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(scale=math.inf), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(causal=2), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(dtype=5), gbattn.ATTN_ERR_INVALID_ARG),
        (dict(D=80), gbattn.ATTN_ERR_UNSUPPORTED),
        (dict(D=32), gbattn.ATTN_ERR_UNSUPPORTED),
        (dict(D=512), gbattn.ATTN_ERR_UNSUPPORTED),
    ],
)
def test_fwd_rejects_on_host(lib, kw, expected):
    assert fwd(lib, **kw) == expected


def test_bwd_rejects_on_host(lib):
    for i in range(10):
        ptrs = [FAKE] * 10
        ptrs[i] = None
        assert bwd(lib, ptrs) == gbattn.ATTN_ERR_INVALID_ARG
    assert bwd(lib, Lq=100, Lk=99) == gbattn.ATTN_ERR_INVALID_ARG
    assert bwd(lib, D=48) == gbattn.ATTN_ERR_UNSUPPORTED
    assert bwd(lib, Hq=5, Hkv=2) == gbattn.ATTN_ERR_INVALID_ARG


def test_delta_rejects_on_host(lib):
    assert lib.attn_bwd_delta(None, FAKE, FAKE, 1, 2, 3, 64, 1, None) == gbattn.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_delta(FAKE, FAKE, FAKE + 4, 1, 2, 3, 64, 1, None) == gbattn.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_delta(FAKE, FAKE, FAKE, 0, 2, 3, 64, 1, None) == gbattn.ATTN_ERR_INVALID_ARG
    assert lib.attn_bwd_delta(FAKE, FAKE, FAKE, 1, 2, 3, 100, 1, None) == gbattn.ATTN_ERR_UNSUPPORTED


def test_status_strings(lib):
    names = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
             4: "ATTN_ERR_TIMEOUT", 5: "ATTN_ERR_DEVICE_CHECK"}
    for code, name in names.items():
        assert gbattn.status_string(code) == name
    assert gbattn.status_string(99) == "ATTN_ERR_UNKNOWN"


def test_binding_raises_on_error(lib):
    with pytest.raises(gbattn.AttnError):
        gbattn._check(gbattn.ATTN_ERR_UNSUPPORTED, "attn_fwd", True)


def test_binding_rejects_host_tensors_before_the_abi():
    """The wrappers check their tensors before any pointer reaches the
    library: host tensors, wrong dtypes and mixed 16-bit types are refused."""
    import torch

    q = torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16)
    lse = torch.zeros((1, 2, 8), dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gbattn.attn_fwd(q, q, q, q, lse, 0.125, True)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gbattn.attn_bwd_delta(q, q, lse)
    with pytest.raises(ValueError, match="CUDA tensor"):
        gbattn.lce_fwd(q[0, 0], q[0, 0], lse[0, 0].int(), lse[0, 0], lse[0, 0], lse)


def fwd_masked(lib, mask=FAKE, D=128, Lq=300, Lk=300):
    return lib.attn_fwd_masked(FAKE, FAKE, FAKE, FAKE, FAKE, mask, 1, 4, 2, Lq, Lk, D, ctypes.c_float(0.1), 1, 1,
                               None)


def bwd_masked(lib, ptrs=None, D=128, Lq=300, Lk=300):
    ptrs = ptrs or [FAKE] * 11
    return lib.attn_bwd_masked(*ptrs, 1, 4, 2, Lq, Lk, D, ctypes.c_float(0.1), 1, 1, None)


def test_masked_rejects_on_host(lib):
    # the block mask is required (the unmasked calls serve a mask of all ones)
    assert fwd_masked(lib, mask=None) == gbattn.ATTN_ERR_INVALID_ARG
    # the mask is a byte array: any address is accepted for it, but not for the tensors
    assert fwd_masked(lib, D=48) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_masked(lib, D=80) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_masked(lib, Lq=301, Lk=300) == gbattn.ATTN_ERR_INVALID_ARG
    for i in range(11):
        ptrs = [FAKE] * 11
        ptrs[i] = None
        assert bwd_masked(lib, ptrs) == gbattn.ATTN_ERR_INVALID_ARG
    assert bwd_masked(lib, Lq=301, Lk=300) == gbattn.ATTN_ERR_INVALID_ARG


def fwd_ex(lib, mask=None, pitch=0, D=128, Lq=300, Lk=300):
    return lib.attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, mask, pitch, 1, 4, 2, Lq, Lk, D, ctypes.c_float(0.1), 1, 1,
                           None)


def bwd_ex(lib, ptrs=None, mask=None, pitch=0, D=128, Lq=300, Lk=300):
    ptrs = ptrs or [FAKE] * 10
    return lib.attn_bwd_ex(*ptrs[:7], mask, pitch, *ptrs[7:], 1, 4, 2, Lq, Lk, D, ctypes.c_float(0.1), 1, 1, None)


def test_ex_rejects_on_host(lib):
    assert fwd_ex(lib, pitch=-1) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_ex(lib, pitch=299) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_ex(lib, pitch=1 << 40) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_ex(lib, D=80) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_ex(lib, Lq=301) == gbattn.ATTN_ERR_INVALID_ARG
    for i in range(10):
        ptrs = [FAKE] * 10
        ptrs[i] = None
        assert bwd_ex(lib, ptrs) == gbattn.ATTN_ERR_INVALID_ARG
    assert bwd_ex(lib, pitch=100) == gbattn.ATTN_ERR_INVALID_ARG


def test_kv_row_pitch_from_strides():
    import torch

    cache = torch.empty((2, 3, 40, 64), dtype=torch.bfloat16)
    k = cache[:, :, :25]
    assert gbattn.kv_row_pitch(k, cache[:, :, :25]) == 40
    assert gbattn.kv_row_pitch(cache, cache) == 0
    with pytest.raises(ValueError):
        gbattn.kv_row_pitch(cache[:, :, :, :32], cache[:, :, :, :32])
    with pytest.raises(ValueError):
        gbattn.kv_row_pitch(k, cache.transpose(1, 2)[:, :25])


def test_decode_workspace_and_rejects_on_host(lib):
    lib.attn_decode_workspace_bytes.restype = ctypes.c_size_t
    need = lib.attn_decode_workspace_bytes(4, 32, 8, 8, 8192, 128)
    assert need > 0 and need % 16 == 0
    assert lib.attn_decode_workspace_bytes(1, 32, 1, 8, 8192, 128) == 0  # G * Lq = 256 rows
    assert lib.attn_decode_workspace_bytes(1, 32, 8, 8, 8192, 80) == 0

    def fwd_dec(ws=FAKE, nbytes=need, Hq=32, Hkv=8, Lq=8, D=128):
        return lib.attn_fwd_decode(FAKE, FAKE, FAKE, FAKE, FAKE, ws, ctypes.c_size_t(nbytes), 4, Hq, Hkv, Lq, 8192,
                                   D, ctypes.c_float(0.1), 1, 1, None)

    assert fwd_dec(ws=None) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_dec(ws=FAKE + 8) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_dec(nbytes=need - 1) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_dec(Hq=32, Hkv=1) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_dec(D=48) == gbattn.ATTN_ERR_UNSUPPORTED
    ptrs = [FAKE] * 10
    ptrs[3] = None
    assert lib.attn_bwd_decode(*ptrs, FAKE, ctypes.c_size_t(need), 4, 32, 8, 8, 8192, 128, ctypes.c_float(0.1), 1,
                               1, None) == gbattn.ATTN_ERR_INVALID_ARG


def test_lce_rejects_on_host(lib):
    lib.lce_workspace_bytes.restype = ctypes.c_size_t
    need = lib.lce_workspace_bytes(300, 128, 1000)
    assert need > 0 and lib.lce_workspace_bytes(300, 100, 1000) == 0 and lib.lce_workspace_bytes(0, 128, 10) == 0

    def fwd_l(ptrs=None, nbytes=need, N=300, Dm=128, V=1000, dtype=1):
        ptrs = ptrs or [FAKE] * 6
        return lib.lce_fwd(*ptrs, ctypes.c_size_t(nbytes), N, Dm, V, dtype, None)

    for i in range(6):
        ptrs = [FAKE] * 6
        ptrs[i] = None
        assert fwd_l(ptrs) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_l([FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE]) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_l(Dm=100) == gbattn.ATTN_ERR_UNSUPPORTED
    assert fwd_l(N=0) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_l(dtype=7) == gbattn.ATTN_ERR_INVALID_ARG
    assert fwd_l(nbytes=0) == gbattn.ATTN_ERR_INVALID_ARG
    for i in range(8):
        ptrs = [FAKE] * 8
        ptrs[i] = None
        assert lib.lce_bwd(*ptrs, ctypes.c_size_t(need), 300, 128, 1000, 1, None) == gbattn.ATTN_ERR_INVALID_ARG
    assert lib.lce_bwd(*([FAKE] * 8), ctypes.c_size_t(need - 16), 300, 128, 1000, 1, None) == \
        gbattn.ATTN_ERR_INVALID_ARG
