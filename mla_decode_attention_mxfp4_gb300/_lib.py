"""ctypes binding of libmla_mxfp4.so: argument marshalling only.

Every step of the decode runs in the library's CUDA kernels; there is no
Python or CPU fallback.  If the shared library is missing, loading it raises
instead of degrading.
"""
from __future__ import annotations

import ctypes
import os
import re

from .build import INCLUDE, LIB_PATH

_lib = None

# status codes (include/mla_mxfp4.h)
MLA_OK = 0
MLA_ERR_NULL_PTR = 1
MLA_ERR_BAD_BATCH = 2
MLA_ERR_BAD_ALIGN = 3
MLA_ERR_BAD_SCALE = 4
MLA_ERR_WORKSPACE = 5
MLA_ERR_CUDA = 6
MLA_ERR_BAD_LAYOUT = 7
MLA_DEVICE_BAD_INDPTR = 1
MLA_DEVICE_TIMEOUT = 2
# mla_decode_mxfp4_device_status(stream, MLA_STATIC_SCRATCH, ...) reads the no-allocation scratch
MLA_STATIC_SCRATCH = 1


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def declared_functions() -> list[str]:
    """Names of the functions declared in include/*.h."""
    names = []
    for fn in sorted(os.listdir(INCLUDE)):
        if fn.endswith(".h"):
            txt = open(os.path.join(INCLUDE, fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(mla_\w+)\s*\(", txt)
    return names


def lib():
    """Load libmla_mxfp4.so (fails loudly if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m mla_decode_attention_mxfp4_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.mla_decode_mxfp4.restype = i
    L.mla_decode_mxfp4.argtypes = [vp, vp, vp, vp, vp, i, f, vp]
    L.mla_decode_mxfp4_ws.restype = i
    L.mla_decode_mxfp4_ws.argtypes = [vp, vp, vp, vp, vp, i, f, vp, vp, sz]
    L.mla_decode_mxfp4_ws_timed.restype = i
    L.mla_decode_mxfp4_ws_timed.argtypes = [vp, vp, vp, vp, vp, i, f, vp, vp, sz, vp, vp]
    L.mla_decode_mxfp4_paged_ws.restype = i
    L.mla_decode_mxfp4_paged_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, vp, i, i, f, vp, vp, sz]
    L.mla_decode_mxfp4_paged_ws_timed.restype = i
    L.mla_decode_mxfp4_paged_ws_timed.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, vp, i, i, f, vp, vp, sz, vp, vp]
    L.mla_decode_fp8_ws.restype = i
    L.mla_decode_fp8_ws.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, f, vp, vp, sz]
    L.mla_decode_fp8_ws_timed.restype = i
    L.mla_decode_fp8_ws_timed.argtypes = [vp, vp, vp, vp, vp, i, vp, i, i, f, vp, vp, sz, vp, vp]
    L.mla_decode_mxfp4_ws_stalled.restype = i
    L.mla_decode_mxfp4_ws_stalled.argtypes = [vp, vp, vp, vp, vp, i, f, vp, vp, sz, ctypes.c_ulonglong]
    L.mla_decode_mxfp4_workspace_bytes.restype = sz
    L.mla_decode_mxfp4_workspace_bytes.argtypes = [i, i]
    L.mla_decode_mxfp4_device_status.restype = i
    L.mla_decode_mxfp4_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    L.mla_decode_mxfp4_last_device_status.restype = i
    L.mla_decode_mxfp4_last_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    L.mla_decode_mxfp4_release.restype = None
    L.mla_decode_mxfp4_release.argtypes = []
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_status_string.argtypes = [i]
    L.mla_host_device_pointer.restype = i
    L.mla_host_device_pointer.argtypes = [vp, ctypes.POINTER(vp)]
    _lib = L
    return L


def status_string(code: int) -> str:
    return lib().mla_status_string(int(code)).decode()


def host_device_pointer(host_ptr: int) -> tuple[int, int]:
    """(status, device address) of a pointer into mapped page-locked host memory."""
    out = ctypes.c_void_p(0)
    rc = lib().mla_host_device_pointer(host_ptr, ctypes.byref(out))
    return rc, (out.value or 0)


# ---- raw C-ABI calls (integer device pointers) ---------------------------------------

def mla_decode_mxfp4(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream) -> int:
    return lib().mla_decode_mxfp4(q, kv_packed, kv_scale, kv_indptr, out, int(batch), float(sm_scale), stream)


def mla_decode_mxfp4_ws(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace,
                        ws_bytes) -> int:
    return lib().mla_decode_mxfp4_ws(q, kv_packed, kv_scale, kv_indptr, out, int(batch), float(sm_scale),
                                     stream, workspace, int(ws_bytes))


def mla_decode_mxfp4_ws_timed(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace,
                              ws_bytes, ev_split_begin, ev_split_end) -> int:
    return lib().mla_decode_mxfp4_ws_timed(q, kv_packed, kv_scale, kv_indptr, out, int(batch), float(sm_scale),
                                           stream, workspace, int(ws_bytes), ev_split_begin, ev_split_end)


def mla_decode_mxfp4_paged_ws(q, kv_packed, kv_scale, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, page_size,
                              num_pages, out, batch, total_q, sm_scale, stream, workspace, ws_bytes) -> int:
    return lib().mla_decode_mxfp4_paged_ws(q, kv_packed, kv_scale, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                                           int(page_size), int(num_pages), out, int(batch), int(total_q),
                                           float(sm_scale), stream, workspace, int(ws_bytes))


def mla_decode_mxfp4_paged_ws_timed(q, kv_packed, kv_scale, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                                    page_size, num_pages, out, batch, total_q, sm_scale, stream, workspace, ws_bytes,
                                    ev_split_begin, ev_split_end) -> int:
    return lib().mla_decode_mxfp4_paged_ws_timed(q, kv_packed, kv_scale, qo_indptr, kv_indptr, kv_indices,
                                                 kv_last_page_len, int(page_size), int(num_pages), out, int(batch),
                                                 int(total_q), float(sm_scale), stream, workspace, int(ws_bytes),
                                                 ev_split_begin, ev_split_end)


def mla_decode_fp8_ws(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, kv_rows, out, batch, total_q, sm_scale, stream,
                      workspace, ws_bytes) -> int:
    return lib().mla_decode_fp8_ws(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, int(kv_rows), out, int(batch),
                                   int(total_q), float(sm_scale), stream, workspace, int(ws_bytes))


def mla_decode_fp8_ws_timed(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, kv_rows, out, batch, total_q, sm_scale,
                            stream, workspace, ws_bytes, ev_split_begin, ev_split_end) -> int:
    return lib().mla_decode_fp8_ws_timed(q, kv_fp8, kv_scale, qo_indptr, kv_indptr, int(kv_rows), out, int(batch),
                                         int(total_q), float(sm_scale), stream, workspace, int(ws_bytes),
                                         ev_split_begin, ev_split_end)


def mla_decode_mxfp4_ws_stalled(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream, workspace,
                                ws_bytes, timeout_ns) -> int:
    """Test-only: the attention kernel's copy role issues nothing, so its waits run out."""
    return lib().mla_decode_mxfp4_ws_stalled(q, kv_packed, kv_scale, kv_indptr, out, int(batch), float(sm_scale),
                                             stream, workspace, int(ws_bytes), int(timeout_ns))


def mla_decode_mxfp4_noalloc(q, kv_packed, kv_scale, kv_indptr, out, batch, sm_scale, stream) -> int:
    """The entry point that allocates nothing (uses the library's static device scratch)."""
    f = lib().mla_decode_mxfp4_noalloc
    vp = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_float, vp]
    return f(q, kv_packed, kv_scale, kv_indptr, out, int(batch), float(sm_scale), stream)


def mla_decode_mxfp4_workspace_bytes(batch: int, device: int) -> int:
    return int(lib().mla_decode_mxfp4_workspace_bytes(int(batch), int(device)))


def mla_decode_mxfp4_device_status(stream=None, workspace=None) -> int:
    st = ctypes.c_int(0)
    rc = lib().mla_decode_mxfp4_device_status(stream, workspace, ctypes.byref(st))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_mxfp4_device_status")
    return st.value


def mla_decode_mxfp4_last_device_status(stream=None) -> int:
    st = ctypes.c_int(0)
    rc = lib().mla_decode_mxfp4_last_device_status(stream, ctypes.byref(st))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_mxfp4_last_device_status")
    return st.value


def mla_decode_mxfp4_release() -> None:
    lib().mla_decode_mxfp4_release()
