"""GPU parity of the fp8-KV kernel (mla_decode_fp8_ws): e4m3 KV with one per-tensor scale,
against the oracle's fp8 definition, at the stated tolerance."""
import numpy as np
import pytest
import torch

import mla_inputs as MI
import oracle
from tests.test_parity_gpu import as64, check_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    yield


def run_fp8(d, kv_fp8=None, qo_indptr=None, q=None):
    from mla_decode_attention_mxfp4_gb300 import alloc_workspace, decode_fp8, device_status
    dev = torch.device("cuda:0")
    kv = (d.kv_fp8 if kv_fp8 is None else kv_fp8).to(dev)
    qq = (d.q if q is None else q).to(dev)
    sc = torch.tensor([d.kv_scale], dtype=torch.float32, device=dev)
    ws = alloc_workspace(max(d.batch, qq.shape[0], 1))
    torch.cuda.synchronize()
    out = decode_fp8(qq, kv, sc, d.kv_indptr.to(dev), d.sm_scale,
                     qo_indptr=qo_indptr.to(dev) if qo_indptr is not None else None, workspace=ws)
    torch.cuda.synchronize()
    return out, device_status(None, ws)


@pytest.mark.parametrize("lens", [[256], [1024] * 4, [300, 0, 1000, 5, 129, 1], [127, 128, 129, 255, 256, 257],
                                  [50000], [5] * 300])
def test_fp8_small_and_ragged(lens):
    d = MI.make_fp8_custom(lens, seed=len(lens))
    out, st = run_fp8(d)
    assert st == 0
    ref = oracle.decode_fp8(d.q, d.kv_fp8, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, f"fp8 {lens[:6]}")


def test_fp8_rows_past_a_sequence_never_leak():
    """The copies bring whole 128-row boxes, so a sequence's last tile also holds rows past it:
    here the buffer continues with rows of NaN bytes (0x7F).  They must neither reach the
    scores nor the output."""
    d = MI.make_fp8_custom([300, 129, 70], seed=5)
    junk = torch.full((200, 576), 0x7F, dtype=torch.uint8)
    kv = torch.cat([d.kv_fp8, junk]).contiguous()
    out, st = run_fp8(d, kv_fp8=kv)
    assert st == 0
    got = as64(out)
    assert np.isfinite(got).all()
    ref = oracle.decode_fp8(d.q, d.kv_fp8, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(got, ref, "rows past the sequences")


def test_fp8_nan_byte_poisons_its_sequence_only():
    d = MI.make_fp8_custom([40, 300, 9], seed=6)
    kv = d.kv_fp8.clone()
    kv[100, 17] = 0x7F
    out, st = run_fp8(d, kv_fp8=kv)
    got = as64(out)
    assert np.isnan(got[1]).all()
    assert np.isfinite(got[0]).all() and np.isfinite(got[2]).all()


def test_fp8_several_query_rows():
    d = MI.make_fp8_custom([700, 0, 2000, 33], seed=7)
    q, qo = MI.query_rows([3, 1, 2, 4], seed=8)
    out, st = run_fp8(d, qo_indptr=qo, q=q)
    assert st == 0
    ref = np.concatenate([_rows_ref(d, q, qo, b) for b in range(4)])
    check_close(as64(out), ref, "fp8 query rows")


def _rows_ref(d, q, qo, b):
    """Oracle output of sequence b's query rows: each row attends to all of b's KV rows."""
    rows = []
    for r in range(int(qo[b]), int(qo[b + 1])):
        ip = torch.tensor([int(d.kv_indptr[b]), int(d.kv_indptr[b + 1])], dtype=torch.int32)
        rows.append(oracle.decode_fp8(q[r:r + 1], d.kv_fp8, d.kv_scale, ip, d.sm_scale))
    return np.concatenate(rows) if rows else np.zeros((0, 16, 512))


def test_fp8_indptr_past_the_buffer_is_clamped_and_flagged():
    d = MI.make_fp8_custom([100, 60], seed=9)
    d.kv_indptr = torch.tensor([0, 100, 400], dtype=torch.int32)  # claims 240 rows past the buffer
    out, st = run_fp8(d)
    assert st & 1
    ref = oracle.decode_fp8(d.q, d.kv_fp8, d.kv_scale, torch.tensor([0, 100, 160], dtype=torch.int32), d.sm_scale)
    check_close(as64(out), ref, "clamped to the buffer")


@pytest.mark.parametrize("name", ["uniform", "ragged"])
def test_fp8_full_size_every_element(name):
    d = MI.make_fp8_inputs(name)
    out, st = run_fp8(d)
    assert st == 0
    got = as64(out)
    ref = oracle.decode_fp8(d.q, d.kv_fp8, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(got, ref, f"fp8 {name}")
    for b in range(d.batch):
        assert np.linalg.norm(got[b] - ref[b]) <= 1e-2 * np.linalg.norm(ref[b]), b
