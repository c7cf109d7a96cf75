"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

Each test is chosen so that a plausible slip in the oracle (a wrong nibble
order, scale block, sign, sm_scale, softmax shift, K/V row mix-up or merge
weight) fails at least one of them.
"""
import math
import struct

import numpy as np
import pytest
import torch

import mla_inputs as MI
import oracle
from oracle import brute
from tests.conftest import read_golden

SM = MI.SM_SCALE


def _bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def _rows(n, fill_scale=127):
    return np.zeros((n, 288), np.uint8), np.full((n, 18), fill_scale, np.uint8)


def _set_code(packed, t, d, code):
    j = d // 2
    if d % 2 == 0:
        packed[t, j] = (packed[t, j] & 0xF0) | code
    else:
        packed[t, j] = (packed[t, j] & 0x0F) | (code << 4)


def _q_bits(B, fill=None):
    q = torch.zeros(B, 16, 576, dtype=torch.bfloat16)
    if fill is not None:
        fill(q)
    return q


# ---- element decode -------------------------------------------------------

def test_e2m1_all_codes_match_page_table_and_fields():
    rows = read_golden("e2m1_codes.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code, val = int(code_s), float(val_s)
        for got in (oracle.e2m1_table(code), oracle.e2m1_fields(code)):
            assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val)
        assert brute._e2m1(code) == val


def test_e8m0_all_bytes():
    special = {int(b): int(bits, 16) for b, bits in read_golden("e8m0_special.txt")}
    for b in range(256):
        v = oracle.e8m0(b)
        if b == 255:
            assert math.isnan(v)
            continue
        assert v == math.ldexp(1.0, b - 127)
        if b in special:  # the page's fp32 bit patterns denote the same values
            assert struct.unpack("<f", struct.pack("<I", special[b]))[0] == v
    assert math.isnan(struct.unpack("<f", struct.pack("<I", special[255]))[0])


def test_nibble_order_and_scale_blocks():
    p, s = _rows(1)
    p[0, 0], p[0, 1], p[0, 2], p[0, 3], p[0, 16] = 0x72, 0x9A, 0x0F, 0x80, 0x35
    s[0, 1] = 129
    k = oracle.dequant_rows(p, s)[0]
    for idx, val in read_golden("nibble_order.txt"):
        i, v = int(idx), float(val)
        assert k[i] == v and math.copysign(1, k[i]) == math.copysign(1, v), (i, k[i], v)
    assert k[34:].tolist() == [0.0] * (576 - 34)


def test_dequant_every_code_in_every_block():
    # each block gets its own scale; every code appears at every position class
    rng = np.random.default_rng(7)
    p = rng.integers(0, 256, (4, 288), dtype=np.uint8)
    s = rng.integers(100, 150, (4, 18), dtype=np.uint8)
    k = oracle.dequant_rows(p, s)
    for t in range(4):
        for d in range(576):
            byte = int(p[t, d // 2])
            code = byte & 15 if d % 2 == 0 else byte >> 4
            assert k[t, d] == brute._e2m1(code) * 2.0 ** (int(s[t, d // 32]) - 127)


def test_bf16_rounding_is_rne():
    one = 1.0
    assert oracle.to_bf16_bits(one + 2 ** -8) == 0x3F80          # tie -> even (down)
    assert oracle.to_bf16_bits(one + 3 * 2 ** -8) == 0x3F82      # tie -> even (up)
    assert oracle.to_bf16_bits(one + 2 ** -8 + 2 ** -30) == 0x3F81
    assert oracle.to_bf16_bits(-2.0) == 0xC000
    assert oracle.to_bf16_bits(float("inf")) == 0x7F80
    assert oracle.to_bf16_bits(3.5e38) == 0x7F80                 # overflow
    assert oracle.to_bf16_bits(2.0 ** -133) == 0x0001            # smallest subnormal
    # against torch's fp32 -> bf16 (RNE) on values exactly representable in fp32
    rng = np.random.default_rng(3)
    xs = (rng.standard_normal(4000) * np.exp(rng.uniform(-30, 30, 4000))).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(xs.astype(np.float64))
    assert np.array_equal(got, ref)


# ---- attention -------------------------------------------------------------

def test_brute_force_agrees_on_tiny_inputs():
    for lens, seed in (([1, 5, 3], 11), ([2, 0, 4], 12), ([5], 13)):
        d = MI.make_custom(lens, seed=seed)
        ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
        qb = d.q.view(torch.int16).numpy().view(np.uint16).tolist()
        got = np.array(brute.decode(qb, d.kv_packed.tolist(), d.kv_scale.tolist(),
                                    d.kv_indptr.tolist(), SM))
        scale = max(1.0, np.abs(ref).max())
        assert np.abs(got - ref).max() <= 1e-12 * scale


def test_kv_len_one_returns_v_exactly():
    d = MI.make_custom([1, 1], seed=21)
    out = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    k = oracle.dequant_rows(d.kv_packed, d.kv_scale)
    for b in range(2):
        for h in range(16):
            assert np.array_equal(out[b, h], k[b, :512])


def test_zero_query_gives_mean_of_v():
    d = MI.make_custom([37], seed=22)
    q = torch.zeros_like(d.q)
    out = oracle.decode(q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    toks = [brute.token(d.kv_packed[t].tolist(), d.kv_scale[t].tolist()) for t in range(37)]
    mean = np.array([math.fsum(r[j] for r in toks) / 37 for j in range(512)])
    for h in range(16):
        assert np.allclose(out[0, h], mean, rtol=1e-13, atol=1e-15)


def test_shared_rope_and_zero_lora_query_gives_mean():
    # q has only RoPE components, and every token has the same RoPE dims, so all
    # scores are equal (but non-zero): the softmax must still be uniform.
    d = MI.make_custom([23], seed=23)
    q = d.q.clone()
    q[:, :, :512] = 0
    p, s = d.kv_packed.clone(), d.kv_scale.clone()
    p[:, 256:] = p[0, 256:]
    s[:, 16:] = s[0, 16:]
    out = oracle.decode(q, p, s, d.kv_indptr, SM)
    k = oracle.dequant_rows(p, s)
    assert abs(float(q[0, 0, 512:].float() @ torch.from_numpy(k[0, 512:]).float())) > 0.1
    mean = k[:, :512].mean(axis=0)
    for h in range(16):
        assert np.allclose(out[0, h], mean, rtol=1e-12, atol=1e-14)


def test_identical_tokens_give_that_token():
    d = MI.make_custom([9], seed=24)
    p = d.kv_packed.clone()
    s = d.kv_scale.clone()
    p[:] = p[4]
    s[:] = s[4]
    out = oracle.decode(d.q, p, s, d.kv_indptr, SM)
    k = oracle.dequant_rows(p[:1], s[:1])[0]
    for h in range(16):
        assert np.allclose(out[0, h], k[:512], rtol=1e-14, atol=0)


def test_two_token_closed_form():
    # Hand-built: token 0 has K[0]=2, K[1]=1, K[570]=6; token 1 has K[0]=-1,
    # K[1]=3, K[570]=-6 (scale 2^0).  Head 0 queries dim 0, head 1 queries dim 1
    # with weight 4, head 2 queries the RoPE dim 570.
    p, s = _rows(2)
    for t, (a, b, r) in enumerate(((4, 2, 7), (10, 5, 15))):  # codes
        _set_code(p, t, 0, a)
        _set_code(p, t, 1, b)
        _set_code(p, t, 570, r)
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    q[0, 1, 1] = 4.0
    q[0, 2, 570] = 1.0
    ip = torch.tensor([0, 2], dtype=torch.int32)
    out = oracle.decode(q, p, s, ip, SM)
    v0, v1 = np.zeros(512), np.zeros(512)
    v0[0], v0[1], v1[0], v1[1] = 2.0, 1.0, -1.0, 3.0
    for h, (s0, s1) in {0: (2 / 24, -1 / 24), 1: (4 / 24, 12 / 24), 2: (6 / 24, -6 / 24)}.items():
        w0, w1 = math.exp(s0), math.exp(s1)
        want = (w0 * v0 + w1 * v1) / (w0 + w1)
        assert np.allclose(out[0, h], want, rtol=1e-14, atol=1e-16), h
    # heads with q = 0 average the two tokens
    assert np.allclose(out[0, 5], (v0 + v1) / 2, rtol=1e-14, atol=1e-16)


def test_token_permutation_invariance():
    d = MI.make_custom([31], seed=25)
    perm = torch.randperm(31, generator=torch.Generator().manual_seed(1))
    a = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    b = oracle.decode(d.q, d.kv_packed[perm], d.kv_scale[perm], d.kv_indptr, SM)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("nsplit", [1, 2, 3, 7, 41])
def test_split_merge_invariance(nsplit):
    d = MI.make_custom([41, 0, 17, 1], seed=26)
    full = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    split = oracle.decode_split(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM, nsplit)
    assert np.allclose(split, full, rtol=1e-12, atol=1e-15)


def test_empty_sequence_is_zero_and_nan_scale_poisons_only_its_sequence():
    d = MI.make_custom([0, 6, 5], seed=27)
    s = d.kv_scale.clone()
    s[8, 3] = 255  # a token of sequence 2
    out = oracle.decode(d.q, d.kv_packed, s, d.kv_indptr, SM)
    assert np.all(out[0] == 0.0)
    assert np.all(np.isfinite(out[1]))
    assert np.all(np.isnan(out[2]))


def test_sharp_softmax_selects_the_aligned_token():
    # With a huge sm_scale the softmax becomes argmax over tokens.
    d = MI.make_custom([12], seed=28)
    out = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, 1e6)
    k = oracle.dequant_rows(d.kv_packed, d.kv_scale)
    qf = d.q[0].float().double().numpy()
    for h in range(16):
        best = int(np.argmax(k @ qf[h]))
        assert np.array_equal(out[0, h], k[best, :512])


@pytest.mark.parametrize("nthreads", [1, 3, 8])
def test_multithreaded_driver_is_bitwise_the_single_threaded_oracle(nthreads):
    """The OpenMP driver (used for full-size parity and the multi-core CPU baseline) runs
    the same per-head arithmetic: identical bits for every element, empty sequences and
    the (sequence, head) task split included."""
    for lens in ([5, 0, 3], [1] * 40, [70, 2, 0, 0, 33]):
        d = MI.make_custom(lens, seed=len(lens))
        a = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
        b = oracle.decode_mt(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM, nthreads)
        assert np.array_equal(a.view(np.int64), b.view(np.int64))
