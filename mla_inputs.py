"""Seeded synthetic inputs for MXFP4 MLA decode (shared by tests and bench).

This module only *constructs* inputs: it draws Q and a latent KV cache from a
seeded CPU ``torch.Generator`` and encodes the KV cache as MXFP4 (OCP MX,
e2m1 elements in blocks of 32 with one E8M0 power-of-two scale per block).
It holds none of the decode method's arithmetic (no dequantisation, no
attention) and is imported by neither the CUDA path nor the oracle.

Tensor contract produced (kernelindex amd-mixed-mla-608791, "check_mla_inputs"):
  q          bf16  [batch, 16, 576]
  kv_packed  uint8 [total_kv, 288]   byte j: element 2j low nibble, 2j+1 high nibble
  kv_scale   uint8 [total_kv, 18]    E8M0, block b covers elements 32b..32b+31
  kv_indptr  int32 [batch + 1]       sequence b owns rows [indptr[b], indptr[b+1])

Recipe (one generator per workload, seeded with the workload's seed), drawn in
this order: per-sequence lengths (ragged workload only) -> Q -> outlier channel
indices (outlier workload only) -> latent KV, chunk by chunk (CHUNK_TOKENS rows
per draw). Each chunk of latent KV (fp32 ~ N(0,1), outlier channels x16) is
quantised before the next chunk is drawn, so memory stays bounded.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

NUM_HEADS = 16
QK_DIM = 576
V_DIM = 512
PACKED_BYTES = QK_DIM // 2   # 288
BLOCK = 32
NUM_SCALES = QK_DIM // BLOCK  # 18
SM_SCALE = 1.0 / math.sqrt(QK_DIM)  # exactly 1/24
CHUNK_TOKENS = 16384

# e2m1 magnitudes in code order 0..7 and the midpoints between neighbours;
# used only to *encode* (round-to-nearest-even onto this grid).
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MIDS = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=torch.float32)


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    kv_len: int | None          # uniform length, or None for ragged
    seed: int
    q_std: float = 1.0
    ragged_max: int = 0         # ragged: lengths ~ U[1, ragged_max] inclusive
    outlier_frac: float = 0.0   # fraction of the 576 channels scaled by outlier_gain
    outlier_gain: float = 16.0
    note: str = field(default="", compare=False)


# The five decode workloads (shapes and distributions of the method's
# benchmark; seeds are the workload index).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 0, note="B=1 kv=256"),
    "small": Workload("small", 4, 1024, 1, note="B=4 kv=1024"),
    "outlier": Workload("outlier", 32, 8192, 2, q_std=0.5, outlier_frac=0.01,
                        note="B=32 kv=8192, Q std 0.5, 6 outlier channels x16"),
    "uniform": Workload("uniform", 128, 4096, 3, note="B=128 kv=4096"),
    "ragged": Workload("ragged", 64, None, 4, ragged_max=32768,
                       note="B=64 kv~U[1,32768]"),
}
WORKLOAD_ORDER = ["tiny", "small", "outlier", "uniform", "ragged"]


@dataclass
class DecodeInputs:
    q: torch.Tensor          # bf16 [B,16,576] (CPU)
    kv_packed: torch.Tensor  # uint8 [N,288]
    kv_scale: torch.Tensor   # uint8 [N,18]
    kv_indptr: torch.Tensor  # int32 [B+1]
    sm_scale: float
    outlier_channels: tuple = ()

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.numel()) - 1

    @property
    def total_kv(self) -> int:
        return int(self.kv_packed.shape[0])

    def algorithmic_bytes(self) -> int:
        """Q + packed KV + scales + bf16 output bytes of one decode call."""
        return (self.q.numel() * 2 + self.kv_packed.numel() + self.kv_scale.numel()
                + self.batch * NUM_HEADS * V_DIM * 2)


def quantize_mxfp4(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
    """Encode fp32 rows [n, 576] as MXFP4: (packed uint8 [n,288], scales uint8 [n,18]).

    Per 32-element block: amax = max|x|; the shared exponent is
    floor(log2 amax) - 2 (the e2m1 largest exponent is 2), stored biased by 127
    and clamped to [0, 254]; an all-zero block stores 127.  Each element is
    x / 2^(scale-127) rounded to nearest-even on the e2m1 grid, saturating at 6.
    Negative values keep the sign bit (so -0 is code 8).
    """
    assert x.dim() == 2 and x.shape[1] == QK_DIM
    n = x.shape[0]
    xb = x.to(torch.float32).reshape(n, NUM_SCALES, BLOCK)
    amax = xb.abs().amax(dim=-1)
    _, ex = torch.frexp(amax)  # amax = m * 2^ex, m in [0.5, 1)
    e = ex.to(torch.int32) - 1 - 2
    sbyte = torch.clamp(e + 127, 0, 254)
    sbyte = torch.where(amax == 0, torch.full_like(sbyte, 127), sbyte)
    # |x| / 2^(s-127): a power-of-two rescale, exact in fp32 for every value that
    # can round to a non-zero code.
    y = torch.ldexp(xb.abs(), -(sbyte - 127).unsqueeze(-1).to(torch.float32))
    idx = torch.bucketize(y, _E2M1_MIDS, right=False)  # exact midpoints go down
    at_mid = y == _E2M1_MIDS[idx.clamp(max=6)]
    idx = idx + (at_mid & (idx % 2 == 1)).to(idx.dtype)  # ...unless that code is odd
    code = idx | torch.where(xb < 0, 8, 0)
    code = code.reshape(n, QK_DIM).to(torch.uint8)
    packed = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.contiguous(), sbyte.to(torch.uint8).contiguous()


def make_inputs(w: Workload | str, batch: int | None = None) -> DecodeInputs:
    """Build the seeded inputs of a workload (optionally only its first `batch` sequences'
    lengths, for reduced-size parity runs that keep the same draws)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator().manual_seed(w.seed)
    B = w.batch
    if w.kv_len is None:
        lens = torch.randint(1, w.ragged_max + 1, (B,), generator=g)
    else:
        lens = torch.full((B,), w.kv_len, dtype=torch.int64)
    q = (torch.randn(B, NUM_HEADS, QK_DIM, generator=g) * w.q_std).to(torch.bfloat16)
    outliers = ()
    if w.outlier_frac > 0:
        k = int(round(w.outlier_frac * QK_DIM))
        outliers = tuple(sorted(torch.randperm(QK_DIM, generator=g)[:k].tolist()))
    if batch is not None and batch < B:
        lens, q = lens[:batch], q[:batch].contiguous()
        B = batch
    indptr = torch.zeros(B + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(lens, 0)
    total = int(indptr[-1])
    packed = torch.empty(total, PACKED_BYTES, dtype=torch.uint8)
    scale = torch.empty(total, NUM_SCALES, dtype=torch.uint8)
    gain = None
    if outliers:
        gain = torch.ones(QK_DIM)
        gain[list(outliers)] = w.outlier_gain
    for s in range(0, total, CHUNK_TOKENS):
        e = min(total, s + CHUNK_TOKENS)
        lat = torch.randn(e - s, QK_DIM, generator=g)
        if gain is not None:
            lat = lat * gain
        packed[s:e], scale[s:e] = quantize_mxfp4(lat)
    return DecodeInputs(q=q, kv_packed=packed, kv_scale=scale,
                        kv_indptr=indptr.to(torch.int32), sm_scale=SM_SCALE,
                        outlier_channels=outliers)


def make_custom(lens, seed: int = 1234, q_std: float = 1.0) -> DecodeInputs:
    """Seeded inputs with explicit per-sequence lengths (edge cases: empty, ragged tails)."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.as_tensor(list(lens), dtype=torch.int64)
    B = lens.numel()
    q = (torch.randn(B, NUM_HEADS, QK_DIM, generator=g) * q_std).to(torch.bfloat16)
    indptr = torch.zeros(B + 1, dtype=torch.int64)
    if B:
        indptr[1:] = torch.cumsum(lens, 0)
    total = int(indptr[-1])
    lat = torch.randn(total, QK_DIM, generator=g)
    packed, scale = quantize_mxfp4(lat) if total else (
        torch.empty(0, PACKED_BYTES, dtype=torch.uint8), torch.empty(0, NUM_SCALES, dtype=torch.uint8))
    return DecodeInputs(q=q, kv_packed=packed, kv_scale=scale,
                        kv_indptr=indptr.to(torch.int32), sm_scale=SM_SCALE)


def scatter_into_pages(d: DecodeInputs, page_size: int, seed: int, spare_pages: int = 3,
                       fill_packed: int = 0x77, fill_scale: int = 200):
    """Place every sequence's KV rows, in order, into randomly chosen pages of a larger buffer
    (the paged layout: page p holds rows [p*page_size, (p+1)*page_size)).  Unused rows hold
    junk.  Returns (kv_packed, kv_scale, kv_indptr over pages, kv_indices, kv_last_page_len,
    num_pages); a sequence without rows has no page (its last-page length is 1, unused)."""
    g = torch.Generator().manual_seed(seed)
    lens = (d.kv_indptr[1:] - d.kv_indptr[:-1]).tolist()
    npages = [(n + page_size - 1) // page_size for n in lens]
    total = sum(npages) + spare_pages
    perm = torch.randperm(total, generator=g).tolist()
    kp = torch.full((total * page_size, PACKED_BYTES), fill_packed, dtype=torch.uint8)
    ks = torch.full((total * page_size, NUM_SCALES), fill_scale, dtype=torch.uint8)
    indptr, indices, last = [0], [], []
    nxt = 0
    for b, n in enumerate(lens):
        r0 = int(d.kv_indptr[b])
        for j in range(npages[b]):
            page = perm[nxt]
            nxt += 1
            indices.append(page)
            rows = min(page_size, n - j * page_size)
            kp[page * page_size: page * page_size + rows] = d.kv_packed[r0 + j * page_size: r0 + j * page_size + rows]
            ks[page * page_size: page * page_size + rows] = d.kv_scale[r0 + j * page_size: r0 + j * page_size + rows]
        indptr.append(len(indices))
        last.append(n - (npages[b] - 1) * page_size if npages[b] else 1)
    return (kp, ks, torch.tensor(indptr, dtype=torch.int32), torch.tensor(indices, dtype=torch.int32),
            torch.tensor(last, dtype=torch.int32), total)


def query_rows(q_per_seq, seed: int, q_std: float = 1.0):
    """Several query rows per sequence: bf16 q [total_q,16,576] and qo_indptr [B+1]."""
    g = torch.Generator().manual_seed(seed)
    qo = torch.zeros(len(q_per_seq) + 1, dtype=torch.int32)
    if len(q_per_seq):
        qo[1:] = torch.cumsum(torch.as_tensor(list(q_per_seq), dtype=torch.int64), 0).to(torch.int32)
    q = (torch.randn(int(qo[-1]), NUM_HEADS, QK_DIM, generator=g) * q_std).to(torch.bfloat16)
    return q, qo


@dataclass
class Fp8Inputs:
    q: torch.Tensor          # bf16 [total_q,16,576]
    kv_fp8: torch.Tensor     # uint8 [rows,576]: e4m3 ("fn") bytes
    kv_scale: float          # the per-tensor scale: K = e4m3(kv_fp8) * kv_scale
    kv_indptr: torch.Tensor  # int32 [B+1]
    sm_scale: float

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.numel()) - 1

    @property
    def total_kv(self) -> int:
        return int(self.kv_fp8.shape[0])

    def algorithmic_bytes(self) -> int:
        """Q + fp8 KV + bf16 output bytes of one decode call."""
        return self.q.numel() * 2 + self.kv_fp8.numel() + self.q.shape[0] * NUM_HEADS * V_DIM * 2


def quantize_fp8(x: torch.Tensor, scale: float) -> torch.Tensor:
    """e4m3 bytes of x / scale (round to nearest even; |x| / scale <= 448 by the choice of scale)."""
    return (x.to(torch.float32) / scale).to(torch.float8_e4m3fn).view(torch.uint8)


def make_fp8_inputs(w: Workload | str, batch: int | None = None) -> Fp8Inputs:
    """A workload's shapes and draws (lengths -> Q -> latent KV, as make_inputs) with the KV
    cache stored as fp8 e4m3 under one per-tensor scale amax / 448 (the largest e4m3 value)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    g = torch.Generator().manual_seed(w.seed)
    B = w.batch
    if w.kv_len is None:
        lens = torch.randint(1, w.ragged_max + 1, (B,), generator=g)
    else:
        lens = torch.full((B,), w.kv_len, dtype=torch.int64)
    q = (torch.randn(B, NUM_HEADS, QK_DIM, generator=g) * w.q_std).to(torch.bfloat16)
    if w.outlier_frac > 0:
        k = int(round(w.outlier_frac * QK_DIM))
        outliers = sorted(torch.randperm(QK_DIM, generator=g)[:k].tolist())
    else:
        outliers = []
    if batch is not None and batch < B:
        lens, q = lens[:batch], q[:batch].contiguous()
        B = batch
    indptr = torch.zeros(B + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(lens, 0)
    total = int(indptr[-1])
    lat = torch.empty(total, QK_DIM, dtype=torch.float32)
    for s0 in range(0, total, CHUNK_TOKENS):
        e = min(total, s0 + CHUNK_TOKENS)
        lat[s0:e] = torch.randn(e - s0, QK_DIM, generator=g)
    if outliers:
        lat[:, outliers] *= w.outlier_gain
    amax = float(lat.abs().max()) if total else 1.0
    scale = amax / 448.0 if amax > 0 else 1.0
    return Fp8Inputs(q=q, kv_fp8=quantize_fp8(lat, scale), kv_scale=scale,
                     kv_indptr=indptr.to(torch.int32), sm_scale=SM_SCALE)


def make_fp8_custom(lens, seed: int = 1234, q_std: float = 1.0) -> Fp8Inputs:
    """fp8 inputs with explicit per-sequence lengths."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.as_tensor(list(lens), dtype=torch.int64)
    B = lens.numel()
    q = (torch.randn(B, NUM_HEADS, QK_DIM, generator=g) * q_std).to(torch.bfloat16)
    indptr = torch.zeros(B + 1, dtype=torch.int64)
    if B:
        indptr[1:] = torch.cumsum(lens, 0)
    total = int(indptr[-1])
    lat = torch.randn(total, QK_DIM, generator=g)
    amax = float(lat.abs().max()) if total else 1.0
    scale = amax / 448.0 if amax > 0 else 1.0
    return Fp8Inputs(q=q, kv_fp8=quantize_fp8(lat, scale) if total else torch.empty(0, QK_DIM, dtype=torch.uint8),
                     kv_scale=scale, kv_indptr=indptr.to(torch.int32), sm_scale=SM_SCALE)
