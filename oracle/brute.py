"""Second, separately written oracle in pure Python (tiny inputs only).

TEST INFRASTRUCTURE ONLY.  It shares nothing with ``oracle/mla_oracle.c``:
e2m1 codes are decoded from their bit fields (kernelindex amd-mixed-mla 717900,
"_nibble_to_f32"), scales with ``math.ldexp`` (608791, "e8m0_to_float"),
sums with ``math.fsum`` and the softmax is written as weights over the
sequence (676098, "_naive_fallback").  Agreement with the C oracle to ~1e-12
is one of the oracle's pins.
"""
from __future__ import annotations

import math
import struct


def _e2m1(code: int) -> float:
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    v = m / 2.0 if e == 0 else (2.0 ** (e - 1)) * (1.0 + m / 2.0)
    return -v if s else v


def _scale(b: int) -> float:
    return float("nan") if b == 255 else math.ldexp(1.0, b - 127)


def _bf16(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (bits & 0xFFFF) << 16))[0]


def token(packed_row, scale_row):
    """One token's 576 values; packed byte j holds element 2j (low) and 2j+1 (high)."""
    vals = []
    for j, byte in enumerate(packed_row):
        for code in (byte & 0xF, byte >> 4):
            d = len(vals)
            vals.append(_e2m1(code) * _scale(scale_row[d // 32]))
    return vals


def decode(q_bits, packed, scale, indptr, sm_scale):
    """q_bits: nested [B][16][576] ints (bf16 bits); packed [N][288]; scale [N][18].
    Returns nested [B][16][512] floats."""
    out = []
    for b in range(len(indptr) - 1):
        rows = [token(packed[t], scale[t]) for t in range(indptr[b], indptr[b + 1])]
        heads = []
        for h in range(16):
            qv = [_bf16(x) for x in q_bits[b][h]]
            if not rows:
                heads.append([0.0] * 512)
                continue
            s = [sm_scale * math.fsum(qv[d] * k[d] for d in range(576)) for k in rows]
            top = max(s)
            w = [math.exp(x - top) for x in s]
            tot = math.fsum(w)
            heads.append([math.fsum(w[i] * rows[i][d] for i in range(len(rows))) / tot
                          for d in range(512)])
        out.append(heads)
    return out
