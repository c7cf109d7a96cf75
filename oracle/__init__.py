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
    """Compile the oracle with the host C compiler (portable flags only; OpenMP for the
    multi-threaded driver when the compiler has it, else a single-threaded build)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        base = ["gcc", "-O2", "-fPIC", "-shared", "-std=gnu99", "-fno-fast-math", "-ffp-contract=off"]
        try:
            subprocess.check_call(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], stderr=subprocess.DEVNULL)
        except subprocess.CalledProcessError:
            subprocess.check_call(base + [_SRC, "-o", tmp, "-lm"])
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
        _lib.mxo_decode_mt.restype = i
        _lib.mxo_decode_mt.argtypes = [u16p, u8p, u8p, i32p, i, d, dp, i]
        _lib.mxo_decode_rows.restype = i
        _lib.mxo_decode_rows.argtypes = [u16p, u8p, u8p, i32p, i32p, i, d, dp]
        _lib.mxo_decode_paged.restype = i
        _lib.mxo_decode_paged.argtypes = [u16p, u8p, u8p, i32p, i32p, i32p, i32p, i, i, d, dp]
        _lib.mxo_e4m3.restype = d
        _lib.mxo_e4m3.argtypes = [i]
        _lib.mxo_decode_fp8.restype = i
        _lib.mxo_decode_fp8.argtypes = [u16p, u8p, d, i32p, i, d, dp]
        _lib.mxo_max_threads.restype = i
        _lib.mxo_max_threads.argtypes = []
        _lib.mxo_online_cpus.restype = i
        _lib.mxo_online_cpus.argtypes = []
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


def max_threads() -> int:
    """Threads the multi-threaded driver uses by default (1 in a build without OpenMP)."""
    return int(lib().mxo_max_threads())


def online_cpus() -> int:
    return int(lib().mxo_online_cpus())


def decode_mt(q, kv_packed, kv_scale, kv_indptr, sm_scale: float, nthreads: int | None = None) -> np.ndarray:
    """decode() with its (sequence, head) pairs on `nthreads` threads (default: all the
    OpenMP runtime offers); every element is computed exactly as decode() computes it."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    ip = _np(kv_indptr, np.int32)
    B = ip.shape[0] - 1
    out = np.zeros((B, HEADS, V), dtype=np.float64)
    n = max_threads() if nthreads is None else int(nthreads)
    rc = lib().mxo_decode_mt(_ptr(qa), _ptr(p), _ptr(s), _ptr(ip), B, float(sm_scale), _ptr(out), n)
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


def decode_rows(q, kv_packed, kv_scale, qo_indptr, kv_indptr, sm_scale: float) -> np.ndarray:
    """Several query rows per sequence: q [total_q,16,576]; rows [qo_indptr[b], qo_indptr[b+1])
    attend to KV rows [kv_indptr[b], kv_indptr[b+1]).  Returns out [total_q,16,512] float64."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    qo = _np(qo_indptr, np.int32)
    ip = _np(kv_indptr, np.int32)
    out = np.zeros((qa.shape[0], HEADS, V), dtype=np.float64)
    rc = lib().mxo_decode_rows(_ptr(qa), _ptr(p), _ptr(s), _ptr(qo), _ptr(ip), ip.shape[0] - 1, float(sm_scale),
                               _ptr(out))
    if rc:
        raise MemoryError("oracle decode_rows failed")
    return out


def decode_paged(q, kv_packed, kv_scale, kv_indptr, kv_indices, kv_last_page_len, page_size: int,
                 sm_scale: float, qo_indptr=None) -> np.ndarray:
    """Paged KV: kv_indptr [B+1] over kv_indices (page ids); kv_packed/kv_scale hold
    num_pages * page_size rows.  One query row per sequence unless qo_indptr is given."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    p = _np(kv_packed, np.uint8).reshape(-1, PACKED)
    s = _np(kv_scale, np.uint8).reshape(-1, NSCALE)
    ip = _np(kv_indptr, np.int32)
    ix = _np(kv_indices, np.int32) if np.asarray(kv_indices).size else np.zeros(1, np.int32)
    last = _np(kv_last_page_len, np.int32) if np.asarray(kv_last_page_len).size else np.zeros(1, np.int32)
    qo = _np(qo_indptr, np.int32) if qo_indptr is not None else None
    out = np.zeros((qa.shape[0], HEADS, V), dtype=np.float64)
    rc = lib().mxo_decode_paged(_ptr(qa), _ptr(p), _ptr(s), _ptr(qo) if qo is not None else None, _ptr(ip),
                                _ptr(ix), _ptr(last), int(page_size), ip.shape[0] - 1, float(sm_scale), _ptr(out))
    if rc:
        raise MemoryError("oracle decode_paged failed")
    return out


def e4m3(byte: int) -> float:
    return lib().mxo_e4m3(int(byte))


def decode_fp8(q, kv_fp8, kv_scale: float, kv_indptr, sm_scale: float) -> np.ndarray:
    """fp8 (e4m3, no infinities) KV with one per-tensor scale: kv_fp8 [rows,576] bytes."""
    qa = _np(q, np.uint16).reshape(-1, HEADS, QK)
    kv = _np(kv_fp8, np.uint8).reshape(-1, QK)
    ip = _np(kv_indptr, np.int32)
    B = ip.shape[0] - 1
    out = np.zeros((B, HEADS, V), dtype=np.float64)
    rc = lib().mxo_decode_fp8(_ptr(qa), _ptr(kv), float(kv_scale), _ptr(ip), B, float(sm_scale), _ptr(out))
    if rc:
        raise MemoryError("oracle decode_fp8 failed")
    return out
