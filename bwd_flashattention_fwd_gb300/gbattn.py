"""Thin Python binding of libgbattn.so (declared in include/gbattn.h).

Argument marshalling only: torch tensors supply device pointers, shapes and
the stream; every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or a call fails, an exception
is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgbattn.so")
# the debug build: the same kernels with index checks (GBATTN_DEBUG_CHECKS)
DEBUG_LIB_PATH = os.path.join(_HERE, "libgbattn_debug.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_DEVICE_CHECK = 5
ATTN_DTYPE_FP16 = 0
ATTN_DTYPE_BF16 = 1

EXPORTED = ("attn_fwd", "attn_bwd_delta", "attn_bwd", "attn_bwd_dq", "attn_bwd_dkv", "attn_bwd_noalloc",
            "attn_fwd_masked", "attn_bwd_masked", "attn_fwd_ex", "attn_bwd_ex", "attn_decode_workspace_bytes",
            "attn_fwd_decode", "attn_bwd_decode", "attn_last_device_status", "attn_wait_probe", "attn_status_string",
            "lce_workspace_bytes", "lce_fwd", "lce_bwd")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} ({status})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libgbattn.so once and declare its C signatures.  With
    GBATTN_DEBUG=1 in the environment the process uses the debug build
    (libgbattn_debug.so) instead."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = DEBUG_LIB_PATH if os.environ.get("GBATTN_DEBUG") == "1" else LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built; run bwd_flashattention_fwd_gb300.build.build() (or __graft_entry__.build())"
        )
    lib = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_fwd.restype = ci
    lib.attn_bwd_delta.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp]
    lib.attn_bwd_delta.restype = ci
    lib.attn_bwd.argtypes = [vp] * 10 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd.restype = ci
    lib.attn_bwd_dq.argtypes = [vp] * 7 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_dq.restype = ci
    lib.attn_bwd_dkv.argtypes = [vp] * 8 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_dkv.restype = ci
    lib.attn_bwd_noalloc.argtypes = [vp] * 9 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_noalloc.restype = ci
    lib.attn_fwd_masked.argtypes = [vp] * 6 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_fwd_masked.restype = ci
    lib.attn_bwd_masked.argtypes = [vp] * 11 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_masked.restype = ci
    i64 = ctypes.c_int64
    lib.attn_fwd_ex.argtypes = [vp] * 6 + [i64, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_fwd_ex.restype = ci
    lib.attn_bwd_ex.argtypes = [vp] * 8 + [i64] + [vp] * 3 + [ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_ex.restype = ci
    sz = ctypes.c_size_t
    lib.attn_decode_workspace_bytes.argtypes = [ci] * 6
    lib.attn_decode_workspace_bytes.restype = sz
    lib.attn_fwd_decode.argtypes = [vp] * 6 + [sz, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_fwd_decode.restype = ci
    lib.attn_bwd_decode.argtypes = [vp] * 11 + [sz, ci, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.attn_bwd_decode.restype = ci
    lib.lce_workspace_bytes.argtypes = [ci, ci, ci]
    lib.lce_workspace_bytes.restype = sz
    lib.lce_fwd.argtypes = [vp] * 6 + [sz, ci, ci, ci, ci, vp]
    lib.lce_fwd.restype = ci
    lib.lce_bwd.argtypes = [vp] * 8 + [sz, ci, ci, ci, ci, vp]
    lib.lce_bwd.restype = ci
    lib.attn_last_device_status.argtypes = [vp]
    lib.attn_last_device_status.restype = ci
    lib.attn_wait_probe.argtypes = [vp]
    lib.attn_wait_probe.restype = ci
    lib.attn_status_string.argtypes = [ci]
    lib.attn_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    if t.dtype == torch.float16:
        return ATTN_DTYPE_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16 or float16")


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _require(call: str, dense=(), sliced=(), f32=(), u8=(), i32=()):
    """Reject tensors the C ABI cannot take before any pointer crosses it.
    dense: 16-bit tensors that must be contiguous (one dtype for all of them
    and for `sliced`); sliced: 16-bit tensors whose layout the caller has
    checked separately (k / v slices of a cache); f32 / u8 / i32: contiguous
    float32 / uint8 / int32 tensors.  Every tensor must be on the current CUDA
    device.  None entries are skipped."""
    half = None
    dev = None
    groups = ((dense, None, True), (sliced, None, False), (f32, torch.float32, True), (u8, torch.uint8, True),
              (i32, torch.int32, True))
    for ts, want, contig in groups:
        for t in ts:
            if t is None:
                continue
            if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
                raise ValueError(f"{call}: every tensor must be a CUDA tensor; got {getattr(t, 'device', type(t))}")
            dev = torch.cuda.current_device() if dev is None else dev
            if t.device.index != dev:
                raise ValueError(f"{call}: every tensor must be on the current CUDA device (cuda:{dev}); got {t.device}")
            if contig and not t.is_contiguous():
                raise ValueError(f"{call}: tensor of shape {tuple(t.shape)} strides {t.stride()} is not contiguous")
            if want is None:
                half = half or t.dtype
                if t.dtype not in (torch.bfloat16, torch.float16) or t.dtype != half:
                    raise TypeError(f"{call}: 16-bit tensors must all be bfloat16 or all float16; got {t.dtype}")
            elif t.dtype != want:
                raise TypeError(f"{call}: expected {want}, got {t.dtype}")


def _check(status: int, call: str, check: bool) -> int:
    if check and status != ATTN_OK:
        raise AttnError(status, call)
    return status


def attn_fwd(q, k, v, o, lse, scale: float, causal: bool, stream=None, check: bool = True) -> int:
    """O and base-2 LSE of causal/non-causal GQA attention (writes o, lse)."""
    _require("attn_fwd", dense=(q, k, v, o), f32=(lse,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lk, D,
                                 float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_fwd", check)


def attn_bwd_delta(o, dO, delta, stream=None, check: bool = True) -> int:
    """delta = rowsum(dO * O) in float32 (writes delta)."""
    _require("attn_bwd_delta", dense=(o, dO), f32=(delta,))
    B, Hq, Lq, D = o.shape
    st = load_library().attn_bwd_delta(_ptr(o), _ptr(dO), _ptr(delta), B, Hq, Lq, D, _dtype_code(o),
                                       _stream_handle(stream))
    return _check(st, "attn_bwd_delta", check)


def attn_bwd(q, k, v, o, dO, lse, delta, dq, dk, dv, scale: float, causal: bool, stream=None,
             check: bool = True) -> int:
    """dQ, dK, dV of the attention (writes dq, dk, dv)."""
    _require("attn_bwd", dense=(q, k, v, o, dO, dq, dk, dv), f32=(lse, delta))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, D, float(scale),
                                 int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd", check)


def attn_bwd_dq(q, k, v, dO, lse, delta, dq, scale: float, causal: bool, stream=None, check: bool = True) -> int:
    """dQ only (the query-row-owning half of attn_bwd)."""
    _require("attn_bwd_dq", dense=(q, k, v, dO, dq), f32=(lse, delta))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(delta), _ptr(dq), B, Hq,
                                    Hkv, Lq, Lk, D, float(scale), int(bool(causal)), _dtype_code(q),
                                    _stream_handle(stream))
    return _check(st, "attn_bwd_dq", check)


def attn_bwd_dkv(q, k, v, dO, lse, delta, dk, dv, scale: float, causal: bool, stream=None,
                 check: bool = True) -> int:
    """dK and dV only (the key-row-owning half of attn_bwd)."""
    _require("attn_bwd_dkv", dense=(q, k, v, dO, dk, dv), f32=(lse, delta))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd_dkv(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(lse), _ptr(delta), _ptr(dk),
                                     _ptr(dv), B, Hq, Hkv, Lq, Lk, D, float(scale), int(bool(causal)),
                                     _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd_dkv", check)


def attn_bwd_noalloc(q, k, v, o, dO, lse, dq, dk, dv, scale: float, causal: bool, stream=None,
                     check: bool = True) -> int:
    """attn_bwd for callers that cannot allocate device memory: delta and the
    status word live in the library's fixed scratch array (B*Hq*Lq <= 2**20)."""
    _require("attn_bwd_noalloc", dense=(q, k, v, o, dO, dq, dk, dv), f32=(lse,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(dq),
                                         _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, D, float(scale),
                                         int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd_noalloc", check)


def attn_fwd_masked(q, k, v, o, lse, block_mask, scale: float, causal: bool, stream=None,
                    check: bool = True) -> int:
    """attn_fwd with a uint8 block mask [ceil(Lq/128), ceil(Lk/128)] on the device."""
    _require("attn_fwd_masked", dense=(q, k, v, o), f32=(lse,), u8=(block_mask,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(block_mask), B, Hq,
                                        Hkv, Lq, Lk, D, float(scale), int(bool(causal)), _dtype_code(q),
                                        _stream_handle(stream))
    return _check(st, "attn_fwd_masked", check)


def attn_bwd_masked(q, k, v, o, dO, lse, delta, block_mask, dq, dk, dv, scale: float, causal: bool, stream=None,
                    check: bool = True) -> int:
    """attn_bwd with the block mask of attn_fwd_masked."""
    _require("attn_bwd_masked", dense=(q, k, v, o, dO, dq, dk, dv), f32=(lse, delta), u8=(block_mask,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta),
                                        _ptr(block_mask), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, D,
                                        float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd_masked", check)


def kv_row_pitch(k, v) -> int:
    """Row pitch of k and v for attn_fwd_ex / attn_bwd_ex: 0 when both are
    contiguous, else the capacity P of a [B, Hkv, P, D] buffer they are the
    first Lk rows of (cache[:, :, :Lk, :]).  Any other layout is rejected."""
    if k.is_contiguous() and v.is_contiguous():
        return 0
    B, Hkv, Lk, D = k.shape
    st = k.stride()
    if st[3] != 1 or st[2] != D or st[1] % D or st[0] != Hkv * st[1] or tuple(v.stride()) != tuple(st):
        raise ValueError(f"k/v strides {tuple(k.stride())}, {tuple(v.stride())} are not a slice of a "
                         f"[B, Hkv, capacity, D] cache")
    return st[1] // D


def attn_fwd_ex(q, k, v, o, lse, scale: float, causal: bool, block_mask=None, kv_pitch=None, stream=None,
                check: bool = True) -> int:
    """attn_fwd with an optional block mask and k / v sliced from a longer
    cache (kv_pitch None: taken from the tensors' strides)."""
    _require("attn_fwd_ex", dense=(q, o), sliced=(k, v), f32=(lse,), u8=(block_mask,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    pitch = kv_row_pitch(k, v) if kv_pitch is None else int(kv_pitch)
    st = load_library().attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(block_mask), pitch, B, Hq,
                                    Hkv, Lq, Lk, D, float(scale), int(bool(causal)), _dtype_code(q),
                                    _stream_handle(stream))
    return _check(st, "attn_fwd_ex", check)


def attn_bwd_ex(q, k, v, o, dO, lse, delta, dq, dk, dv, scale: float, causal: bool, block_mask=None, kv_pitch=None,
                stream=None, check: bool = True) -> int:
    """attn_bwd with the options of attn_fwd_ex (dk, dv contiguous)."""
    _require("attn_bwd_ex", dense=(q, o, dO, dq, dk, dv), sliced=(k, v), f32=(lse, delta), u8=(block_mask,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    pitch = kv_row_pitch(k, v) if kv_pitch is None else int(kv_pitch)
    st = load_library().attn_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta),
                                    _ptr(block_mask), pitch, _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Lq, Lk, D,
                                    float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd_ex", check)


def attn_decode_workspace_bytes(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, D: int) -> int:
    """Bytes of device workspace attn_fwd_decode / attn_bwd_decode need (0: shape not served)."""
    return int(load_library().attn_decode_workspace_bytes(B, Hq, Hkv, Lq, Lk, D))


def decode_workspace(q, k) -> torch.Tensor:
    """A workspace tensor (uint8, on q's device) for the decode calls on q, k."""
    B, Hq, Lq, D = q.shape
    n = attn_decode_workspace_bytes(B, Hq, k.shape[1], Lq, k.shape[2], D)
    if n == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "attn_decode_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def attn_fwd_decode(q, k, v, o, lse, workspace, scale: float, causal: bool, stream=None, check: bool = True) -> int:
    """attn_fwd for short query lengths (G * Lq <= 128), key range split over CTAs."""
    _require("attn_fwd_decode", dense=(q, k, v, o), f32=(lse,), u8=(workspace,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), B, Hq, Hkv, Lq, Lk, D,
                                        float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_fwd_decode", check)


def attn_bwd_decode(q, k, v, o, dO, lse, delta, dq, dk, dv, workspace, scale: float, causal: bool, stream=None,
                    check: bool = True) -> int:
    """attn_bwd for short query lengths (G * Lq <= 128)."""
    _require("attn_bwd_decode", dense=(q, k, v, o, dO, dq, dk, dv), f32=(lse, delta), u8=(workspace,))
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    st = load_library().attn_bwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse), _ptr(delta),
                                        _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), B, Hq, Hkv, Lq, Lk, D,
                                        float(scale), int(bool(causal)), _dtype_code(q), _stream_handle(stream))
    return _check(st, "attn_bwd_decode", check)


def lce_workspace_bytes(N: int, Dm: int, V: int) -> int:
    """Bytes of device workspace lce_fwd / lce_bwd need (0: shape rejected)."""
    return int(load_library().lce_workspace_bytes(N, Dm, V))


def lce_workspace(hidden, weight) -> torch.Tensor:
    N, Dm = hidden.shape
    n = lce_workspace_bytes(N, Dm, weight.shape[0])
    if n == 0:
        raise AttnError(ATTN_ERR_UNSUPPORTED, "lce_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=hidden.device)


def lce_fwd(hidden, weight, targets, loss, lse, workspace, stream=None, check: bool = True) -> int:
    """Per-row linear cross-entropy loss and natural-log lse (writes loss, lse)."""
    _require("lce_fwd", dense=(hidden, weight), f32=(loss, lse), u8=(workspace,), i32=(targets,))
    N, Dm = hidden.shape
    st = load_library().lce_fwd(_ptr(hidden), _ptr(weight), _ptr(targets), _ptr(loss), _ptr(lse), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), N, Dm, weight.shape[0],
                                _dtype_code(hidden), _stream_handle(stream))
    return _check(st, "lce_fwd", check)


def lce_bwd(hidden, weight, targets, lse, dloss, dhidden, dweight, workspace, stream=None, check: bool = True) -> int:
    """dhidden and dweight of sum_i dloss[i] * loss[i] (writes both)."""
    _require("lce_bwd", dense=(hidden, weight, dhidden, dweight), f32=(lse, dloss), u8=(workspace,),
             i32=(targets,))
    N, Dm = hidden.shape
    st = load_library().lce_bwd(_ptr(hidden), _ptr(weight), _ptr(targets), _ptr(lse), _ptr(dloss), _ptr(dhidden),
                                _ptr(dweight), _ptr(workspace), workspace.numel() * workspace.element_size(), N, Dm,
                                weight.shape[0], _dtype_code(hidden), _stream_handle(stream))
    return _check(st, "lce_bwd", check)


def attn_last_device_status(stream=None) -> int:
    return load_library().attn_last_device_status(_stream_handle(stream))


def attn_wait_probe(stream=None, check: bool = True) -> int:
    """Launch the failure-reporting check: one wait that can only run out
    (after GBATTN_WAIT_LIMIT_NS); the next attn_last_device_status reports
    ATTN_ERR_TIMEOUT."""
    return _check(load_library().attn_wait_probe(_stream_handle(stream)), "attn_wait_probe", check)


def attn_status_string(status: int) -> str:
    return status_string(status)


# ---------------------------------------------------------------------------
# Conveniences that allocate the outputs with torch and call the ABI.
# ---------------------------------------------------------------------------


def forward(q, k, v, scale: float, causal: bool = True, stream=None):
    B, Hq, Lq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def delta(o, dO, stream=None):
    B, Hq, Lq, _ = o.shape
    d = torch.empty((B, Hq, Lq), dtype=torch.float32, device=o.device)
    attn_bwd_delta(o, dO, d, stream)
    return d


def backward(q, k, v, o, dO, lse, dlt, scale: float, causal: bool = True, stream=None):
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    attn_bwd(q, k, v, o, dO, lse, dlt, dq, dk, dv, scale, causal, stream)
    return dq, dk, dv
