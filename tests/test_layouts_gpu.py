"""GPU parity of the general layouts (mla_decode_mxfp4_paged_ws): several query rows per
sequence, paged KV with several page sizes, both together, unaligned scale rows, malformed
page tables, and the full-size ragged workload paged, every element against the oracle."""
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


def run_general(q, kv_packed, kv_scale, kv_indptr, sm_scale, **kw):
    from mla_decode_attention_mxfp4_gb300 import decode_general, device_status
    from mla_decode_attention_mxfp4_gb300 import alloc_workspace
    dev = torch.device("cuda:0")
    to = lambda t: t.to(dev) if isinstance(t, torch.Tensor) else t
    args = {k: to(v) for k, v in kw.items()}
    batch, total_q = kv_indptr.numel() - 1, q.shape[0]
    ws = alloc_workspace(max(batch, total_q, 1))
    torch.cuda.synchronize()
    out = decode_general(to(q), to(kv_packed), to(kv_scale), to(kv_indptr), sm_scale, workspace=ws, **args)
    torch.cuda.synchronize()
    return out, device_status(None, ws)


@pytest.mark.parametrize("lens,qlens", [
    ([300, 0, 1000, 5, 129], [2, 3, 1, 4, 0]),
    ([9000, 20000], [3, 2]),
    ([1, 2, 3], [8, 1, 5]),
])
def test_several_query_rows_per_sequence(lens, qlens):
    d = MI.make_custom(lens, seed=len(lens) + sum(qlens))
    q, qo = MI.query_rows(qlens, seed=sum(lens) % 97)
    out, st = run_general(q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, qo_indptr=qo)
    assert st == 0
    ref = oracle.decode_rows(q, d.kv_packed, d.kv_scale, qo, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, f"query rows {qlens}")


@pytest.mark.parametrize("page_size", [1, 8, 12, 16, 64, 128, 256])
def test_paged_kv(page_size):
    d = MI.make_custom([300, 0, 1000, 5, 129, 4096], seed=page_size)
    kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, page_size, seed=page_size + 1)
    out, st = run_general(d.q, kp, ks, ip, d.sm_scale, kv_indices=ix, kv_last_page_len=last,
                          page_size=page_size, num_pages=npages)
    assert st == 0
    ref = oracle.decode_paged(d.q, kp, ks, ip, ix, last, page_size, d.sm_scale)
    check_close(as64(out), ref, f"paged {page_size}")
    # the same values as the contiguous layout's definition
    assert np.array_equal(ref, oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale))


def test_paged_kv_with_several_query_rows_and_many_sequences():
    """9000 sequences (their sanitised query offsets live in the workspace, not in shared
    memory), pages of 16 rows, 1..3 query rows each."""
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 40, 9000).tolist()
    qlens = rng.integers(1, 4, 9000).tolist()
    d = MI.make_custom(lens, seed=12)
    q, qo = MI.query_rows(qlens, seed=13)
    kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, 16, seed=14)
    out, st = run_general(q, kp, ks, ip, d.sm_scale, qo_indptr=qo, kv_indices=ix, kv_last_page_len=last,
                          page_size=16, num_pages=npages)
    assert st == 0
    ref = oracle.decode_rows(q, d.kv_packed, d.kv_scale, qo, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, "paged + query rows, 9000 sequences")


@pytest.mark.parametrize("offset", [0, 5])
def test_paged_kv_with_scale_rows_off_a_16_byte_boundary(offset):
    """kv_scale starting `offset` bytes past a 16-byte boundary: page chunks are no longer
    congruent modulo 16 (offset 5) and go through plain loads; results are unchanged."""
    d = MI.make_custom([700, 33, 2000], seed=20 + offset)
    kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, 16, seed=21)
    raw = torch.empty(ks.numel() + 32, dtype=torch.uint8)
    shifted = raw[offset:offset + ks.numel()].view(ks.shape)
    shifted.copy_(ks)
    dev = torch.device("cuda:0")
    from mla_decode_attention_mxfp4_gb300 import alloc_workspace, decode_general, device_status
    raw_d = raw.to(dev)
    ks_d = raw_d[offset:offset + ks.numel()].view(ks.shape)
    assert ks_d.data_ptr() % 16 == offset % 16 or offset == 0
    ws = alloc_workspace(3)
    out = decode_general(d.q.to(dev), kp.to(dev), ks_d, ip.to(dev), d.sm_scale, kv_indices=ix.to(dev),
                         kv_last_page_len=last.to(dev), page_size=16, num_pages=npages, workspace=ws)
    torch.cuda.synchronize()
    assert device_status(None, ws) == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, f"paged, scale offset {offset}")


def test_bad_page_ids_are_clamped_and_flagged():
    d = MI.make_custom([100, 50], seed=30)
    kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, 16, seed=31)
    ix = ix.clone()
    ix[1] = npages + 5     # beyond the buffers
    ix[-1] = -3            # negative
    out, st = run_general(d.q, kp, ks, ip, d.sm_scale, kv_indices=ix, kv_last_page_len=last, page_size=16,
                          num_pages=npages)
    assert st & 1
    ixc = ix.clamp(0, npages - 1)
    ref = oracle.decode_paged(d.q, kp, ks, ip, ixc, last, 16, d.sm_scale)
    check_close(as64(out), ref, "clamped pages")


def test_full_size_ragged_workload_paged_every_element():
    """The ragged workload (64 sequences, 1.15 M tokens) in pages of 64 rows scattered over
    the buffer, in the bench's launch configuration: every element against the oracle."""
    d = MI.make_inputs("ragged")
    kp, ks, ip, ix, last, npages = MI.scatter_into_pages(d, 64, seed=40, spare_pages=0)
    out, st = run_general(d.q, kp, ks, ip, d.sm_scale, kv_indices=ix, kv_last_page_len=last, page_size=64,
                          num_pages=npages)
    assert st == 0
    ref = oracle.decode_mt(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, "ragged, paged 64")
