"""The C-ABI library: it builds, loads, exports every declared symbol, and its
host-side argument checks return the documented status codes (no GPU needed:
these paths return before any CUDA call)."""
import math

import pytest

from mla_decode_attention_mxfp4_gb300 import _lib


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return _lib.lib()


def test_exports_every_declared_symbol(L):
    names = _lib.declared_functions()
    assert set(names) >= {"mla_decode_mxfp4", "mla_decode_mxfp4_ws", "mla_decode_mxfp4_workspace_bytes",
                          "mla_decode_mxfp4_device_status", "mla_decode_mxfp4_release", "mla_status_string",
                          "mla_decode_mxfp4_ws_timed", "mla_decode_mxfp4_ws_stalled",
                          "mla_decode_mxfp4_noalloc", "mla_decode_mxfp4_last_device_status"}
    for n in names:
        assert hasattr(L, n), n


def test_host_device_pointer_checks_its_arguments(L):
    assert _lib.host_device_pointer(0) == (_lib.MLA_ERR_NULL_PTR, 0)


def test_host_argument_checks(L):
    f = _lib.mla_decode_mxfp4
    ok = dict(q=0x1000, kv=0x2000, sc=0x3001, ip=0x4004, out=0x5000)  # kv_scale: no alignment rule
    assert f(0, 0, 0, 0, 0, 0, 1.0, None) == _lib.MLA_OK            # batch 0: no-op
    assert f(0, 0, 0, 0, 0, -1, 1.0, None) == _lib.MLA_ERR_BAD_BATCH
    assert f(0, ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, 1.0, None) == _lib.MLA_ERR_NULL_PTR
    assert f(ok["q"], ok["kv"], ok["sc"], 0, ok["out"], 2, 1.0, None) == _lib.MLA_ERR_NULL_PTR
    assert f(ok["q"], ok["kv"], ok["sc"], ok["ip"], 0, 2, 1.0, None) == _lib.MLA_ERR_NULL_PTR
    assert f(ok["q"] + 8, ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, 1.0, None) == _lib.MLA_ERR_BAD_ALIGN
    assert f(ok["q"], ok["kv"] + 4, ok["sc"], ok["ip"], ok["out"], 2, 1.0, None) == _lib.MLA_ERR_BAD_ALIGN
    assert f(ok["q"], ok["kv"], ok["sc"], ok["ip"] + 2, ok["out"], 2, 1.0, None) == _lib.MLA_ERR_BAD_ALIGN
    assert f(ok["q"], ok["kv"], ok["sc"], ok["ip"], ok["out"] + 1, 2, 1.0, None) == _lib.MLA_ERR_BAD_ALIGN
    for bad in (math.nan, math.inf, -math.inf):
        assert f(ok["q"], ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, bad, None) == _lib.MLA_ERR_BAD_SCALE
    w = _lib.mla_decode_mxfp4_ws
    assert w(ok["q"], ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, 1.0, None, 0, 1 << 20) == _lib.MLA_ERR_NULL_PTR
    assert w(ok["q"], ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, 1.0, None, 0x10010, 1 << 20) == _lib.MLA_ERR_BAD_ALIGN
    st = _lib.mla_decode_mxfp4_ws_stalled  # the test hook's wait limit must be 1 ns .. 1 s
    for bad in (0, 1_000_000_001):
        assert st(ok["q"], ok["kv"], ok["sc"], ok["ip"], ok["out"], 2, 1.0, None, 0x10000, 1 << 20,
                  bad) == _lib.MLA_ERR_BAD_SCALE


def test_status_strings(L):
    for code in range(7):
        assert _lib.status_string(code).startswith("MLA_")
    assert "unknown" in _lib.status_string(99)


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle, and decode() demands CUDA tensors."""
    import inspect

    import torch

    import mla_decode_attention_mxfp4_gb300 as pkg
    from mla_decode_attention_mxfp4_gb300 import api
    for mod in (pkg, api, _lib):
        assert "import oracle" not in inspect.getsource(mod)
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        api.decode(q, torch.zeros(1, 288, dtype=torch.uint8), torch.zeros(1, 18, dtype=torch.uint8),
                   torch.tensor([0, 1], dtype=torch.int32), 1 / 24)


def test_host_argument_checks_of_the_general_entry(L):
    from mla_decode_attention_mxfp4_gb300 import _lib
    f = _lib.mla_decode_mxfp4_paged_ws
    a = dict(q=0x1000, kv=0x2000, sc=0x3000, ip=0x4000, out=0x5000, ws=0x10000)
    # total_q != batch without query offsets
    assert f(a["q"], a["kv"], a["sc"], None, a["ip"], None, None, 0, 0, a["out"], 2, 3, 1.0, None, a["ws"],
             1 << 24) == _lib.MLA_ERR_BAD_LAYOUT
    # paged without a positive page size or without last-page lengths
    assert f(a["q"], a["kv"], a["sc"], None, a["ip"], 0x6000, 0x7000, 0, 4, a["out"], 2, 2, 1.0, None, a["ws"],
             1 << 24) == _lib.MLA_ERR_BAD_LAYOUT
    assert f(a["q"], a["kv"], a["sc"], None, a["ip"], 0x6000, None, 16, 4, a["out"], 2, 2, 1.0, None, a["ws"],
             1 << 24) == _lib.MLA_ERR_BAD_LAYOUT
    assert f(a["q"], a["kv"], a["sc"], None, a["ip"], None, None, 0, 0, a["out"], -1, -1, 1.0, None, a["ws"],
             1 << 24) == _lib.MLA_ERR_BAD_BATCH
