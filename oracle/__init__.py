"""fp64 CPU oracle for MXFP4 MLA decode attention (ctypes binding of mla_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
bench's CPU-baseline leg, never by the product package.  It shares no code with
the CUDA library; the only thing both sides see is the seeded input generator.

The C source states what is computed and cites the pages it follows.  A second,
separately written pure-Python implementation lives in ``oracle.brute`` and is
used to cross-check this one on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmla_oracle.so")
_lib = None

HEADS, QK, V, PACKED, NSCALE = 16, 576, 512, 288, 18


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags only)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        d, i, u8p, u16p, i32p, dp = (ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p)
        _lib.mxo_e2m1_table.restype = d
        _lib.mxo_e2m1_table.argtypes = [i]
        _lib.mxo_e2m1_fields.restype = d
        _lib.mxo_e2m1_fields.argtypes = [i]
        _lib.mxo_e8m0.restype = d
        _lib.mxo_e8m0.argtypes = [i]
        _lib.mxo_double_to_bf16.restype = ctypes.c_uint16
        _lib.mxo_double_to_bf16.argtypes = [d]
        _lib.mxo_bf16_to_double.restype = d
        _lib.mxo_bf16_to_double.argtypes = [ctypes.c_uint16]
        _lib.mxo_dequant_token.restype = None
        _lib.mxo_dequant_token.argtypes = [u8p, u8p, dp]
        _lib.mxo_attend.restype = i
        _lib.mxo_attend.argtypes = [u16p, u8p, u8p, ctypes.c_int64, ctypes.c_int64, d, dp]
        _lib.mxo_decode.restype = i
        _lib.mxo_decode.argtypes = [u16p, u8p, u8p, i32p, i, d, dp]
        _lib.mxo_decode_split.restype = i
        _lib.mxo_decode_split.argtypes = [u16p, u8p, u8p, i32p, i, d, i, dp]
    return _lib


def _np(t, dtype):
    """torch tensor or array -> contiguous numpy array of `dtype` (bf16 -> uint16 bits)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            t = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(t).view(dtype) if np.asarray(t).dtype.itemsize ==
                                np.dtype(dtype).itemsize else np.asarray(t, dtype=dtype))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def e2m1_table(code: int) -> float:
    return lib().mxo_e2m1_table(code)


def e2m1_fields(code: int) -> float:
    return lib().mxo_e2m1_fields(code)


def e8m0(b: int) -> float:
    return lib().mxo_e8m0(b)


def to_bf16_bits(x: float) -> int:
    return int(lib().mxo_double_to_bf16(float(x)))


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round an fp64 array to bf16 (RNE), returned as uint16 bit patterns."""
    f = np.vectorize(lambda v: lib().mxo_double_to_bf16(float(v)), otypes=[np.uint16])
    return f(np.asarray(a, dtype=np.float64))


def dequant_rows(kv_packed, kv_scale) -> np.ndarray:
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    out = np.empty((p.shape[0], QK), dtype=np.float64)
    for t in range(p.shape[0]):
        lib().mxo_dequant_token(_ptr(p[t]), _ptr(s[t]), _ptr(out[t]))
    return out


def decode(q, kv_packed, kv_scale, kv_indptr, sm_scale: float) -> np.ndarray:
    """Full decode in fp64: returns out [batch,16,512] float64 (not yet rounded)."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    ip = _np(kv_indptr, np.int32)
    B = ip.shape[0] - 1
    out = np.zeros((B, HEADS, V), dtype=np.float64)
    rc = lib().mxo_decode(_ptr(qa), _ptr(p), _ptr(s), _ptr(ip), B, float(sm_scale), _ptr(out))
    if rc:
        raise MemoryError(f"oracle decode failed ({rc})")
    return out


def decode_one(q, kv_packed, kv_scale, kv_indptr, sm_scale: float, b: int) -> np.ndarray:
    """Output of sequence `b` only ([16,512] float64); for sampled checks at full size."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    ip = _np(kv_indptr, np.int64)
    out = np.zeros((HEADS, V), dtype=np.float64)
    qb = np.ascontiguousarray(qa[b])
    rc = lib().mxo_attend(_ptr(qb), _ptr(p), _ptr(s), int(ip[b]), int(ip[b + 1]), float(sm_scale),
                          _ptr(out))
    if rc:
        raise MemoryError("oracle attend failed")
    return out


def decode_split(q, kv_packed, kv_scale, kv_indptr, sm_scale: float, nsplit: int) -> np.ndarray:
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    ip = _np(kv_indptr, np.int32)
    B = ip.shape[0] - 1
    out = np.zeros((B, HEADS, V), dtype=np.float64)
    rc = lib().mxo_decode_split(_ptr(qa), _ptr(p), _ptr(s), _ptr(ip), B, float(sm_scale),
                                int(nsplit), _ptr(out))
    if rc:
        raise RuntimeError(f"oracle split decode failed ({rc})")
    return out
