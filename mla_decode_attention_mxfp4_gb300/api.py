"""PyTorch-facing wrapper of the C ABI (tensor checks + pointer marshalling).

Tensor contract (kernelindex amd-mixed-mla 608791, "check_mla_inputs"):
  q          bf16  [batch, 16, 576]   CUDA, contiguous
  kv_packed  uint8 [rows, 288]        (or [rows, 1, 288]) CUDA, contiguous
  kv_scale   uint8 [rows, 18]         CUDA, contiguous
  kv_indptr  int32 [batch + 1]        CUDA, contiguous, non-decreasing
returns      bf16  [batch, 16, 512]
"""
from __future__ import annotations

import torch

from . import _lib

NUM_HEADS, QK_DIM, V_DIM, PACKED, NSCALE = 16, 576, 512, 288, 18


def _check(q, kv_packed, kv_scale, kv_indptr):
    for name, t in (("q", q), ("kv_packed", kv_packed), ("kv_scale", kv_scale), ("kv_indptr", kv_indptr)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[1] != NUM_HEADS or q.shape[2] != QK_DIM:
        raise ValueError("q must be bf16 [batch, 16, 576]")
    if kv_packed.dtype != torch.uint8 or kv_packed.shape[-1] != PACKED or kv_packed.numel() % PACKED:
        raise ValueError("kv_packed must be uint8 [rows, 288] (packed fp4x2)")
    if kv_scale.dtype != torch.uint8 or kv_scale.shape[-1] != NSCALE:
        raise ValueError("kv_scale must be uint8 [rows, 18] (E8M0)")
    if kv_scale.numel() // NSCALE != kv_packed.numel() // PACKED:
        raise ValueError("kv_scale row count must match kv_packed")
    if kv_indptr.dtype != torch.int32 or kv_indptr.dim() != 1 or kv_indptr.numel() != q.shape[0] + 1:
        raise ValueError("kv_indptr must be int32 [batch + 1]")
    dev = q.device
    for name, t in (("kv_packed", kv_packed), ("kv_scale", kv_scale), ("kv_indptr", kv_indptr)):
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")


def workspace_bytes(batch: int, device=None) -> int:
    dev = torch.device(device if device is not None else "cuda").index
    if dev is None:
        dev = torch.cuda.current_device()
    return _lib.mla_decode_mxfp4_workspace_bytes(batch, dev)


def alloc_workspace(batch: int, device=None) -> torch.Tensor:
    """A caller-owned workspace for decode(..., workspace=...) (256-byte aligned)."""
    n = workspace_bytes(batch, device)
    if n == 0:
        raise RuntimeError("could not size the workspace")
    return torch.empty(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def decode(q: torch.Tensor, kv_packed: torch.Tensor, kv_scale: torch.Tensor, kv_indptr: torch.Tensor,
           sm_scale: float, out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """MXFP4 MLA decode on the GPU; returns out bf16 [batch, 16, 512]."""
    _check(q, kv_packed, kv_scale, kv_indptr)
    B = q.shape[0]
    if out is None:
        out = torch.empty(B, NUM_HEADS, V_DIM, dtype=torch.bfloat16, device=q.device)
    elif (out.dtype != torch.bfloat16 or tuple(out.shape) != (B, NUM_HEADS, V_DIM) or not out.is_contiguous()
          or out.device != q.device):
        raise ValueError("out must be contiguous bf16 [batch, 16, 512] on q's device")
    with torch.cuda.device(q.device):
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        args = (q.data_ptr(), kv_packed.data_ptr(), kv_scale.data_ptr(), kv_indptr.data_ptr(), out.data_ptr(),
                B, float(sm_scale), s.cuda_stream)
        if workspace is None:
            rc = _lib.mla_decode_mxfp4(*args)
        else:
            if workspace.device != q.device or not workspace.is_contiguous():
                raise ValueError("workspace must be a contiguous tensor on q's device")
            rc = _lib.mla_decode_mxfp4_ws(*args, workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if rc != _lib.MLA_OK:
        raise _lib.MlaError(rc, "mla_decode_mxfp4")
    return out


def decode_general(q: torch.Tensor, kv_packed: torch.Tensor, kv_scale: torch.Tensor, kv_indptr: torch.Tensor,
                   sm_scale: float, qo_indptr: torch.Tensor | None = None, kv_indices: torch.Tensor | None = None,
                   kv_last_page_len: torch.Tensor | None = None, page_size: int = 0, num_pages: int = 0,
                   out: torch.Tensor | None = None, stream: torch.cuda.Stream | None = None,
                   workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Decode with several query rows per sequence (qo_indptr) and/or paged KV (kv_indices,
    kv_last_page_len, page_size, num_pages); see mla_decode_mxfp4_paged_ws.  q is
    [total_q, 16, 576]; returns out [total_q, 16, 512].  kv_indptr has batch + 1 entries."""
    for name, t in (("q", q), ("kv_packed", kv_packed), ("kv_scale", kv_scale), ("kv_indptr", kv_indptr),
                    ("qo_indptr", qo_indptr), ("kv_indices", kv_indices), ("kv_last_page_len", kv_last_page_len)):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous CUDA tensor on q's device")
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[1] != NUM_HEADS or q.shape[2] != QK_DIM:
        raise ValueError("q must be bf16 [total_q, 16, 576]")
    for name, t in (("kv_indptr", kv_indptr), ("qo_indptr", qo_indptr), ("kv_indices", kv_indices),
                    ("kv_last_page_len", kv_last_page_len)):
        if t is not None and t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    batch, total_q = kv_indptr.numel() - 1, q.shape[0]
    if out is None:
        out = torch.empty(total_q, NUM_HEADS, V_DIM, dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(max(batch, total_q, 1), q.device)
    ptr = lambda t: t.data_ptr() if t is not None else None
    with torch.cuda.device(q.device):
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        rc = _lib.mla_decode_mxfp4_paged_ws(q.data_ptr(), kv_packed.data_ptr(), kv_scale.data_ptr(), ptr(qo_indptr),
                                            kv_indptr.data_ptr(), ptr(kv_indices), ptr(kv_last_page_len), page_size,
                                            num_pages, out.data_ptr(), batch, total_q, float(sm_scale), s.cuda_stream,
                                            workspace.data_ptr(), workspace.numel())
    if rc != _lib.MLA_OK:
        raise _lib.MlaError(rc, "mla_decode_mxfp4_paged_ws")
    return out


def decode_fp8(q: torch.Tensor, kv_fp8: torch.Tensor, kv_scale: torch.Tensor, kv_indptr: torch.Tensor,
               sm_scale: float, qo_indptr: torch.Tensor | None = None, out: torch.Tensor | None = None,
               stream: torch.cuda.Stream | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Decode against fp8 (e4m3) KV with one per-tensor scale (see mla_decode_fp8_ws).
    kv_fp8: uint8 (or float8_e4m3fn) [rows, 576]; kv_scale: float32 CUDA tensor holding the
    scale; q [total_q, 16, 576] bf16; returns out [total_q, 16, 512] bf16."""
    if kv_fp8.dtype == torch.float8_e4m3fn:
        kv_fp8 = kv_fp8.view(torch.uint8)
    for name, t in (("q", q), ("kv_fp8", kv_fp8), ("kv_scale", kv_scale), ("kv_indptr", kv_indptr),
                    ("qo_indptr", qo_indptr)):
        if t is None:
            continue
        if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous CUDA tensor on q's device")
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[1] != NUM_HEADS or q.shape[2] != QK_DIM:
        raise ValueError("q must be bf16 [total_q, 16, 576]")
    if kv_fp8.dtype != torch.uint8 or kv_fp8.shape[-1] != QK_DIM:
        raise ValueError("kv_fp8 must be uint8 [rows, 576] (e4m3 bytes)")
    if kv_scale.dtype != torch.float32 or kv_scale.numel() < 1:
        raise ValueError("kv_scale must be a float32 tensor holding the per-tensor scale")
    batch, total_q = kv_indptr.numel() - 1, q.shape[0]
    if out is None:
        out = torch.empty(total_q, NUM_HEADS, V_DIM, dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(max(batch, total_q, 1), q.device)
    with torch.cuda.device(q.device):
        s = stream if stream is not None else torch.cuda.current_stream(q.device)
        rc = _lib.mla_decode_fp8_ws(q.data_ptr(), kv_fp8.data_ptr(), kv_scale.data_ptr(),
                                    qo_indptr.data_ptr() if qo_indptr is not None else None, kv_indptr.data_ptr(),
                                    kv_fp8.numel() // QK_DIM, out.data_ptr(), batch, total_q, float(sm_scale),
                                    s.cuda_stream, workspace.data_ptr(), workspace.numel())
    if rc != _lib.MLA_OK:
        raise _lib.MlaError(rc, "mla_decode_fp8_ws")
    return out


def device_status(stream: torch.cuda.Stream | None = None, workspace: torch.Tensor | None = None) -> int:
    """Synchronise and read the device status bits of the last call (see mla_device_status)."""
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    return _lib.mla_decode_mxfp4_device_status(s, workspace.data_ptr() if workspace is not None else None)


class HostDecoder:
    """End-to-end decode from pinned host buffers, output copied back to a host tensor.

    direct (default): the kernels read q, kv_packed and kv_scale in place from the pinned
    host buffers (mla_host_device_pointer gives their device addresses; each byte crosses
    the host link once, inside the decode); kv_indptr is copied to the device first.
    Otherwise, or when an input is not pinned: H2D copies, decode, D2H of the output.
    Device buffers are allocated once for the largest shape seen.  The batch is cut into
    `chunks` groups of whole sequences with about equal KV rows; the copies of group c+1
    (on a copy stream) overlap the decode of group c (on the compute stream).  kv_indptr
    holds absolute row indices, so every group decodes against the full device KV buffer
    through its own slice of the indptr, with no rebasing.  A kv_indptr that is not a
    non-decreasing sequence within the rows is sent as one group.
    """

    def __init__(self, device="cuda", chunks: int = 4, direct: bool = True):
        self.device = torch.device(device)
        self.stream = torch.cuda.Stream(self.device)
        self.copy_stream = torch.cuda.Stream(self.device)
        self.chunks = max(1, int(chunks))
        self.direct = bool(direct)
        self._bufs = {}
        self._ws = None

    def _buf(self, name, like: torch.Tensor):
        b = self._bufs.get(name)
        if b is None or b.numel() < like.numel() or b.dtype != like.dtype:
            b = torch.empty(like.numel(), dtype=like.dtype, device=self.device)
            self._bufs[name] = b
        return b[: like.numel()].view(like.shape)

    def _groups(self, ip: list, rows: int):
        B = len(ip) - 1
        ok = all(0 <= ip[i] <= ip[i + 1] <= rows for i in range(B))
        if not ok or self.chunks == 1 or B < 2:
            return [(0, B, 0, rows)]
        total = ip[B] - ip[0]
        groups, c0 = [], 0
        for c in range(1, self.chunks + 1):
            target = ip[0] + total * c // self.chunks
            c1 = c0 + 1
            while c1 < B and ip[c1] < target:
                c1 += 1
            if c == self.chunks:
                c1 = B
            if c1 > c0:
                groups.append((c0, c1, ip[c0], ip[c1]))
                c0 = c1
            if c0 >= B:
                break
        return groups

    def _device_address(self, t: torch.Tensor) -> int:
        rc, addr = _lib.host_device_pointer(t.data_ptr())
        if rc != _lib.MLA_OK or not addr:
            raise _lib.MlaError(rc, "mla_host_device_pointer")
        return addr

    def _call_direct(self, q, kv_packed, kv_scale, kv_indptr, sm_scale, out_host):
        B = q.shape[0]
        if (q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[1] != NUM_HEADS or q.shape[2] != QK_DIM
                or kv_packed.dtype != torch.uint8 or kv_packed.shape[-1] != PACKED
                or kv_scale.dtype != torch.uint8 or kv_scale.shape[-1] != NSCALE
                or kv_scale.numel() // NSCALE != kv_packed.numel() // PACKED
                or kv_indptr.dtype != torch.int32 or kv_indptr.numel() != B + 1):
            raise ValueError("host inputs: q bf16 [B,16,576], kv_packed uint8 [rows,288], "
                             "kv_scale uint8 [rows,18], kv_indptr int32 [B+1]")
        aq, akv, asc = (self._device_address(t) for t in (q, kv_packed, kv_scale))
        dip, dout = self._buf("ip", kv_indptr), self._buf("out", out_host)
        if self._ws is None or self._ws_batch < B:
            self._ws, self._ws_batch = alloc_workspace(B, self.device), B
        ms = self.stream
        with torch.cuda.stream(ms):
            dip.copy_(kv_indptr, non_blocking=True)
            rc = _lib.mla_decode_mxfp4_ws(aq, akv, asc, dip.data_ptr(), dout.data_ptr(), B, float(sm_scale),
                                          ms.cuda_stream, self._ws.data_ptr(), self._ws.numel())
            if rc != _lib.MLA_OK:
                raise _lib.MlaError(rc, "mla_decode_mxfp4_ws")
            out_host.copy_(dout, non_blocking=True)
        return out_host

    def __call__(self, q, kv_packed, kv_scale, kv_indptr, sm_scale, out_host: torch.Tensor) -> torch.Tensor:
        if (self.direct and all(t.device.type == "cpu" and t.is_pinned() and t.is_contiguous()
                                for t in (q, kv_packed, kv_scale, kv_indptr))):
            return self._call_direct(q, kv_packed, kv_scale, kv_indptr, sm_scale, out_host)
        dq, dkv, dsc = self._buf("q", q), self._buf("kv", kv_packed), self._buf("sc", kv_scale)
        dip, dout = self._buf("ip", kv_indptr), self._buf("out", out_host)
        ip = kv_indptr.tolist()
        groups = self._groups(ip, kv_packed.shape[0])
        cs, ms = self.copy_stream, self.stream
        cs.wait_stream(ms)  # buffers are reused across calls
        with torch.cuda.stream(cs):
            dip.copy_(kv_indptr, non_blocking=True)
        for c0, c1, r0, r1 in groups:
            with torch.cuda.stream(cs):
                dq[c0:c1].copy_(q[c0:c1], non_blocking=True)
                if r1 > r0:
                    dkv[r0:r1].copy_(kv_packed[r0:r1], non_blocking=True)
                    dsc[r0:r1].copy_(kv_scale[r0:r1], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
            ms.wait_event(ev)
            with torch.cuda.stream(ms):
                decode(dq[c0:c1], dkv, dsc, dip[c0:c1 + 1], sm_scale, out=dout[c0:c1], stream=ms)
                out_host[c0:c1].copy_(dout[c0:c1], non_blocking=True)
        return out_host

    def synchronize(self):
        self.copy_stream.synchronize()
        self.stream.synchronize()
