"""GB300-native (sm_103a) MXFP4 MLA decode attention.

Public API:
  decode(q, kv_packed, kv_scale, kv_indptr, sm_scale, out=None, stream=None, workspace=None)
  decode_general(...)  several query rows per sequence and/or paged KV
  decode_fp8(...)      fp8 (e4m3) KV with one per-tensor scale
  alloc_workspace(batch), workspace_bytes(batch), device_status(), HostDecoder
and the raw C ABI mirrored in ``_lib`` (same names as include/mla_mxfp4.h).
"""
from .api import (HostDecoder, alloc_workspace, decode, decode_fp8, decode_general, device_status,  # noqa: F401
                  workspace_bytes)
from .build import LIB_PATH  # noqa: F401
from .build import build as build_library  # noqa: F401

SM_SCALE = 1.0 / 24.0  # 1/sqrt(576)
