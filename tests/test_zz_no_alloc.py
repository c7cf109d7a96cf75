"""The no-allocation entry point (mla_decode_mxfp4_noalloc).

Some callers cannot call cudaMalloc at all: code that runs inside an allocator or
memory-pool callback (allocating there would re-enter the allocator), or a serving
process whose device memory is reserved up front by its runtime (an allocation
would fail or break the reservation).  For them the library offers one entry point
that works entirely out of a statically defined device scratch array.  These tests
call it through the C ABI and check it against the fp64 oracle and against the
allocating entry point, within the parity tolerance used elsewhere, on two calls in
a row (the second call reuses scratch left behind by the first), and read its
device status word through MLA_STATIC_SCRATCH.  This file is named to be collected
last.
"""
import numpy as np
import pytest
import torch

import mla_inputs as MI
import oracle

pytestmark = pytest.mark.gpu

ATOL, RTOL, REL_L2 = 2e-2, 2e-2, 1e-2


def _close(x: np.ndarray, y: np.ndarray):
    assert np.array_equal(np.isfinite(x), np.isfinite(y))
    fin = np.isfinite(y)
    err = np.abs(x[fin] - y[fin])
    assert (err <= ATOL + RTOL * np.abs(y[fin])).all(), float(err.max())
    ny = np.linalg.norm(y[fin])
    assert (np.linalg.norm(x[fin] - y[fin]) / ny if ny > 0 else np.linalg.norm(x[fin])) <= REL_L2


def _as64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().double().numpy()


def _run(entry, d, dev, stream):
    from mla_decode_attention_mxfp4_gb300 import _lib
    q, kv, sc, ip = (d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev))
    out = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize(dev)
    rc = entry(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), ip.data_ptr(), out.data_ptr(), d.batch, d.sm_scale,
               stream.cuda_stream)
    assert rc == _lib.MLA_OK, _lib.status_string(rc)
    torch.cuda.synchronize(dev)
    return out


def test_noalloc_matches_the_oracle_and_the_allocating_entry_point_twice_in_a_row():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    from mla_decode_attention_mxfp4_gb300 import _lib
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    # two different calls: the second one runs on scratch the first one left behind;
    # both include sequences split across CTAs (partials live in the scratch)
    cases = [MI.make_custom([300, 0, 9000, 1, 4100], seed=91), MI.make_inputs("small")]
    for d in cases:
        got = _run(_lib.mla_decode_mxfp4_noalloc, d, dev, stream)
        assert _lib.mla_decode_mxfp4_device_status(stream.cuda_stream, _lib.MLA_STATIC_SCRATCH) == 0
        ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
        _close(_as64(got), ref)
        want = _run(_lib.mla_decode_mxfp4, d, dev, stream)
        _close(_as64(got), _as64(want))


def test_noalloc_status_word_reports_a_malformed_indptr():
    import __graft_entry__
    __graft_entry__.build()
    from mla_decode_attention_mxfp4_gb300 import _lib
    dev = torch.device("cuda:0")
    stream = torch.cuda.Stream(dev)
    d = MI.make_custom([30, 30], seed=81)
    d.kv_indptr = torch.tensor([0, 50, 20], dtype=torch.int32)  # decreasing: clamped to rows < 20
    got = _run(_lib.mla_decode_mxfp4_noalloc, d, dev, stream)
    st = _lib.mla_decode_mxfp4_device_status(stream.cuda_stream, _lib.MLA_STATIC_SCRATCH)
    assert st & _lib.MLA_DEVICE_BAD_INDPTR
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, torch.tensor([0, 20, 20], dtype=torch.int32), d.sm_scale)
    _close(_as64(got), ref)
    # a well-formed call clears it again
    _run(_lib.mla_decode_mxfp4_noalloc, MI.make_custom([7, 3], seed=82), dev, stream)
    assert _lib.mla_decode_mxfp4_device_status(stream.cuda_stream, _lib.MLA_STATIC_SCRATCH) == 0


def test_noalloc_rejects_batches_beyond_its_static_limit():
    import __graft_entry__
    __graft_entry__.build()
    from mla_decode_attention_mxfp4_gb300 import _lib
    dev = torch.device("cuda:0")
    B = 4097
    q = torch.zeros(B, 16, 576, dtype=torch.bfloat16, device=dev)
    kv = torch.zeros(B, 288, dtype=torch.uint8, device=dev)
    sc = torch.full((B, 18), 127, dtype=torch.uint8, device=dev)
    ip = torch.arange(B + 1, dtype=torch.int32, device=dev)
    out = torch.empty(B, 16, 512, dtype=torch.bfloat16, device=dev)
    rc = _lib.mla_decode_mxfp4_noalloc(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), ip.data_ptr(), out.data_ptr(),
                                       B, 1 / 24, torch.cuda.current_stream(dev).cuda_stream)
    assert rc == _lib.MLA_ERR_WORKSPACE
