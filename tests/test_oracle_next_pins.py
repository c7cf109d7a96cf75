"""Pins of the oracle's functions for the further decode forms: several query rows per
sequence, paged KV and fp8 KV with a per-tensor scale.  Each is tied to something other
than itself: the already pinned single-row MXFP4 decode (by reductions that must hold
exactly), a separately written pure-Python computation, or the fp8 format's definition
and torch's independent fp8 conversion."""
import math

import numpy as np
import pytest
import torch

import mla_inputs as MI
import oracle
from tests.conftest import read_golden

SM = MI.SM_SCALE


# ---- several query rows per sequence ----------------------------------------------

def test_one_row_per_sequence_is_the_single_row_decode():
    d = MI.make_custom([5, 0, 17, 3], seed=2)
    qo = torch.arange(d.batch + 1, dtype=torch.int32)
    a = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    b = oracle.decode_rows(d.q, d.kv_packed, d.kv_scale, qo, d.kv_indptr, SM)
    assert np.array_equal(a, b)


def test_every_query_row_attends_to_all_rows_of_its_sequence():
    """Rows of one sequence are independent problems over the same KV rows (no mask): each
    row's output equals a single-row decode of that row against that sequence's rows."""
    d = MI.make_custom([7, 0, 12], seed=3)
    qlens = [3, 2, 4]
    q = (torch.randn(sum(qlens), 16, 576, generator=torch.Generator().manual_seed(9))).to(torch.bfloat16)
    qo = torch.tensor([0, 3, 5, 9], dtype=torch.int32)
    out = oracle.decode_rows(q, d.kv_packed, d.kv_scale, qo, d.kv_indptr, SM)
    for b in range(3):
        for r in range(int(qo[b]), int(qo[b + 1])):
            ip = torch.tensor([int(d.kv_indptr[b]), int(d.kv_indptr[b + 1])], dtype=torch.int32)
            want = oracle.decode(q[r:r + 1], d.kv_packed, d.kv_scale, ip, SM)[0]
            assert np.array_equal(out[r], want), (b, r)
    assert not out[3:5].any()  # sequence 1 has no KV rows


# ---- paged KV -------------------------------------------------------------------

def _scatter_into_pages(d, page_size, seed, spare_pages=3):
    """Place every sequence's rows into randomly chosen pages of a larger buffer."""
    rng = np.random.default_rng(seed)
    lens = (d.kv_indptr[1:] - d.kv_indptr[:-1]).tolist()
    npages = [(n + page_size - 1) // page_size for n in lens]
    total = sum(npages) + spare_pages
    perm = rng.permutation(total)
    kp = np.full((total * page_size, 288), 0x77, np.uint8)   # junk in unused rows
    ks = np.full((total * page_size, 18), 200, np.uint8)
    indptr, indices, last = [0], [], []
    src_p, src_s = d.kv_packed.numpy(), d.kv_scale.numpy()
    nxt = 0
    for b, n in enumerate(lens):
        r0 = int(d.kv_indptr[b])
        for j in range(npages[b]):
            page = int(perm[nxt]); nxt += 1
            indices.append(page)
            rows = min(page_size, n - j * page_size)
            kp[page * page_size: page * page_size + rows] = src_p[r0 + j * page_size: r0 + j * page_size + rows]
            ks[page * page_size: page * page_size + rows] = src_s[r0 + j * page_size: r0 + j * page_size + rows]
        indptr.append(len(indices))
        last.append(n - (npages[b] - 1) * page_size if npages[b] else 1)
    t = lambda a, dt: torch.tensor(a, dtype=dt)
    return (torch.from_numpy(kp), torch.from_numpy(ks), t(indptr, torch.int32), t(indices, torch.int32),
            t(last, torch.int32), total)


@pytest.mark.parametrize("page_size", [1, 8, 16, 64])
def test_paged_decode_is_the_decode_of_the_gathered_rows(page_size):
    d = MI.make_custom([37, 0, 16, 1, 100], seed=4)
    kp, ks, ip, ix, last, _ = _scatter_into_pages(d, page_size, seed=page_size)
    want = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, SM)
    got = oracle.decode_paged(d.q, kp, ks, ip, ix, last, page_size, SM)
    assert np.array_equal(got, want)


def test_paged_decode_with_several_query_rows():
    d = MI.make_custom([20, 9], seed=5)
    q = torch.randn(5, 16, 576, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    qo = torch.tensor([0, 2, 5], dtype=torch.int32)
    kp, ks, ip, ix, last, _ = _scatter_into_pages(d, 8, seed=6)
    want = oracle.decode_rows(q, d.kv_packed, d.kv_scale, qo, d.kv_indptr, SM)
    got = oracle.decode_paged(q, kp, ks, ip, ix, last, 8, SM, qo_indptr=qo)
    assert np.array_equal(got, want)


# ---- fp8 KV -----------------------------------------------------------------------

def test_e4m3_every_byte_matches_the_format_and_torch():
    gold = {int(b, 16): float(v) for b, v in read_golden("e4m3_special.txt")}
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(256):
        got = oracle.e4m3(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b] and math.copysign(1, got) == math.copysign(1, ref[b]), b
        if b in gold:
            g = gold[b]
            assert (math.isnan(got) and math.isnan(g)) or (got == g and math.copysign(1, got) == math.copysign(1, g))


def _fp8_case(lens, seed):
    g = torch.Generator().manual_seed(seed)
    n = sum(lens)
    lat = torch.randn(n, 576, generator=g)
    scale = float(lat.abs().max()) / 448.0
    kv = (lat / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    q = torch.randn(len(lens), 16, 576, generator=g).to(torch.bfloat16)
    ip = torch.zeros(len(lens) + 1, dtype=torch.int32)
    ip[1:] = torch.cumsum(torch.tensor(lens), 0)
    return q, kv, scale, ip


def test_fp8_decode_matches_a_separate_python_computation():
    q, kv, scale, ip = _fp8_case([3, 0, 5], seed=7)
    got = oracle.decode_fp8(q, kv, scale, ip, SM)
    K = kv.view(torch.float8_e4m3fn).to(torch.float64).numpy() * scale
    Q = q.to(torch.float64).numpy()
    for b in range(3):
        r0, r1 = int(ip[b]), int(ip[b + 1])
        for h in range(16):
            if r1 == r0:
                assert not got[b, h].any()
                continue
            s = [SM * math.fsum(Q[b, h] * K[t]) for t in range(r0, r1)]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            L = math.fsum(w)
            want = [math.fsum(w[i] * K[r0 + i, dd] for i in range(r1 - r0)) / L for dd in range(512)]
            assert np.allclose(got[b, h], want, rtol=1e-12, atol=1e-14)


def test_fp8_scale_enters_both_scores_and_values():
    """Doubling the per-tensor scale while halving the query keeps every score, so the
    output doubles exactly; and one KV row returns that row times the scale."""
    q, kv, scale, ip = _fp8_case([6, 1], seed=8)
    a = oracle.decode_fp8(q, kv, scale, ip, SM)
    qh = (q.float() / 2).to(torch.bfloat16)  # exact: halving a bf16 value
    b = oracle.decode_fp8(qh, kv, 2 * scale, ip, SM)
    assert np.allclose(b, 2 * a, rtol=1e-13, atol=0)
    row = kv[6].view(torch.float8_e4m3fn).to(torch.float64).numpy()[:512] * scale
    for h in range(16):
        assert np.allclose(a[1, h], row, rtol=1e-15, atol=0)
