"""GPU parity: the CUDA path against the fp64 oracle on the same seeded inputs.

Gates (per output element, bf16 output vs fp64 reference):
  |gpu - ref| <= 2e-2 + 2e-2 * |ref|            (the stated tolerance)
  ||gpu - ref||_2 / ||ref||_2 <= 1e-2           (a stricter aggregate gate: the
                                                 per-element bound alone would
                                                 pass an all-zero output on
                                                 small-magnitude workloads)
kv_len = 1 must reproduce V exactly (V is exactly representable in bf16).
"""
import numpy as np
import pytest
import torch

import mla_inputs as MI
import oracle

pytestmark = pytest.mark.gpu

ATOL, RTOL, REL_L2 = 2e-2, 2e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    yield


def gpu_decode(d, stream=None, workspace=None):
    from mla_decode_attention_mxfp4_gb300 import decode, device_status
    dev = torch.device("cuda:0")
    args = (d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev))
    torch.cuda.synchronize()  # inputs were copied on the default stream
    out = decode(*args, d.sm_scale, stream=stream, workspace=workspace)
    torch.cuda.synchronize()
    return out, device_status(stream, workspace)


def as64(out):
    return out.float().cpu().double().numpy()


def check_close(got, ref, what=""):
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: finiteness differs"
    g, r = got[fin], ref[fin]
    err = np.abs(g - r)
    bad = err > ATOL + RTOL * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g)
    assert rel <= REL_L2, f"{what}: rel L2 {rel:.3e}"
    return float(err.max()) if err.size else 0.0, float(rel)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_workload_full(name):
    d = MI.make_inputs(name)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, name)


@pytest.mark.parametrize("name,batch", [("outlier", 3), ("uniform", 6), ("ragged", 3)])
def test_workload_leading_sequences(name, batch):
    d = MI.make_inputs(name, batch=batch)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, name)


@pytest.mark.parametrize("name", ["outlier", "uniform", "ragged"])
def test_workload_full_size_sampled(name):
    """Full-size workload in the bench's launch configuration; the oracle checks
    sampled sequences one by one, and every output must be finite."""
    d = MI.make_inputs(name)
    out, st = gpu_decode(d)
    assert st == 0
    got = as64(out)
    assert np.isfinite(got).all()
    rng = np.random.default_rng(0)
    B = d.batch
    picks = sorted(set([0, B - 1] + rng.integers(0, B, 3).tolist()))
    for b in picks:
        ref = oracle.decode_one(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, b)
        check_close(got[b], ref, f"{name}[{b}]")


def test_kv_len_one_reproduces_v_exactly():
    d = MI.make_custom([1, 1, 1, 1], seed=31)
    out, st = gpu_decode(d)
    assert st == 0
    k = oracle.dequant_rows(d.kv_packed, d.kv_scale)
    # exact value equality (the sign of a zero is not a value: V codes 0 and 8
    # both decode to zero, and an fp32 accumulation of -0 yields +0)
    want = oracle.round_bf16(k[:, :512]).view(np.int16)
    want = torch.from_numpy(want.copy()).view(torch.bfloat16).double().numpy()
    got = as64(out)
    assert (k[:, :512] == want).all()  # V is exactly representable in bf16
    for b in range(4):
        for h in range(16):
            assert np.array_equal(got[b, h], want[b]), (b, h)


@pytest.mark.parametrize("lens", [
    [127, 128, 129, 255, 256, 257],
    [0, 3, 0, 0, 1, 2, 0],
    [50000],
    [9000, 20000, 3000, 0, 12000, 1, 7000],
    [0, 0],
    [5] * 300,
])
def test_ragged_edges(lens):
    d = MI.make_custom(lens, seed=sum(lens) % 1000)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, str(lens[:8]))


def test_many_tiny_sequences():
    rng = np.random.default_rng(9)
    lens = rng.integers(0, 7, 700).tolist()
    d = MI.make_custom(lens, seed=41)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, "tiny seqs")


def test_empty_batch():
    from mla_decode_attention_mxfp4_gb300 import decode
    dev = torch.device("cuda:0")
    q = torch.empty(0, 16, 576, dtype=torch.bfloat16, device=dev)
    kv = torch.empty(0, 288, dtype=torch.uint8, device=dev)
    sc = torch.empty(0, 18, dtype=torch.uint8, device=dev)
    ip = torch.zeros(1, dtype=torch.int32, device=dev)
    out = decode(q, kv, sc, ip, 1 / 24)
    assert out.shape == (0, 16, 512)


def test_scale_extremes_and_query_range():
    d = MI.make_custom([300, 200, 64], seed=51)
    s = d.kv_scale.clone()
    s[:300] = s[:300] + 60            # large exponents (values ~2^60)
    s[300:500] = s[300:500] - 100     # tiny exponents (values ~2^-100)
    s[500:, 3] = 0                    # the 2^-127 byte
    s[520, :] = 1
    q = d.q.clone()
    q[0, 0] *= 1e4
    q[0, 1] *= 1e-4
    q[1, 2, :100] = 0
    d.kv_scale, d.q = s.contiguous(), q.contiguous()
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    got = as64(out)
    for b in range(3):  # relative to each sequence's own magnitude
        scale = np.abs(ref[b]).max()
        check_close(got[b] / scale, ref[b] / scale, f"extreme[{b}]")


def test_running_maxima_move_late_in_a_sequence():
    """A token far into a sequence whose scale bytes are raised: its scores jump by far
    more than the raise threshold and so does its token exponent, so the running maxima
    move in the middle of a segment and the accumulator is rescaled (the full path of the
    softmax statistics); a later block of tokens with raised exponents does the same for
    the token-exponent maximum alone."""
    d = MI.make_custom([1000, 700, 300], seed=71)
    s = d.kv_scale.clone().to(torch.int32)
    s[900] += 6                      # one late token 64x larger than the rest
    s[1000 + 450:1000 + 460] += 9    # a late run of tokens with exponents 9 binades higher
    s[1700 + 290] -= 20              # a tiny token at the end of the third sequence
    d.kv_scale = s.clamp(0, 254).to(torch.uint8).contiguous()
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    got = as64(out)
    for b in range(3):  # relative to each sequence's own magnitude
        scale = np.abs(ref[b]).max()
        check_close(got[b] / scale, ref[b] / scale, f"late maxima[{b}]")


def test_special_cases_zero_query_identical_tokens():
    d = MI.make_custom([77, 40], seed=61)
    q = d.q.clone()
    q[0] = 0
    p = d.kv_packed.clone()
    s = d.kv_scale.clone()
    p[77:] = p[80]
    s[77:] = s[80]
    d.q, d.kv_packed, d.kv_scale = q, p, s
    out, st = gpu_decode(d)
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, "special")


def test_nan_scale_poisons_its_sequence_only():
    d = MI.make_custom([40, 300, 9], seed=71)
    s = d.kv_scale.clone()
    s[100, 5] = 255
    d.kv_scale = s
    out, st = gpu_decode(d)
    got = as64(out)
    assert np.isnan(got[1]).all()
    assert np.isfinite(got[0]).all() and np.isfinite(got[2]).all()


def test_workspace_stream_and_determinism():
    from mla_decode_attention_mxfp4_gb300 import alloc_workspace
    d = MI.make_inputs("small")
    a, _ = gpu_decode(d)
    s = torch.cuda.Stream()
    ws = alloc_workspace(d.batch)
    b, st = gpu_decode(d, stream=s, workspace=ws)
    assert st == 0
    c, _ = gpu_decode(d)
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("offset", [1, 7, 13])
def test_scale_buffer_off_a_16_byte_boundary(offset):
    """kv_scale has no alignment rule: a view starting `offset` bytes past a 16-byte
    boundary gives the same bits as the aligned buffer (the producer loads the bytes
    before the buffer's first boundary and after its last one with plain loads)."""
    from mla_decode_attention_mxfp4_gb300 import decode, device_status
    d = MI.make_custom([300, 129, 0, 1000, 5], seed=90 + offset)
    dev = torch.device("cuda:0")
    q, kv, ip = d.q.to(dev), d.kv_packed.to(dev), d.kv_indptr.to(dev)
    sc = d.kv_scale.to(dev).contiguous()
    raw = torch.empty(sc.numel() + 32, dtype=torch.uint8, device=dev)
    shifted = raw[offset:offset + sc.numel()].view(sc.shape)
    shifted.copy_(sc)
    assert shifted.data_ptr() % 16 == offset
    torch.cuda.synchronize()
    a = decode(q, kv, sc, ip, d.sm_scale)
    b = decode(q, kv, shifted, ip, d.sm_scale)
    torch.cuda.synchronize()
    assert device_status() == 0
    assert torch.equal(a, b)
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(b), ref, f"scale offset {offset}")


def test_malformed_indptr_is_flagged_and_in_bounds():
    d = MI.make_custom([30, 30], seed=81)
    d.kv_indptr = torch.tensor([0, 50, 20], dtype=torch.int32)  # decreasing: clamped to rows < 20
    out, st = gpu_decode(d)
    assert st & 1
    from mla_decode_attention_mxfp4_gb300 import _lib
    assert _lib.mla_decode_mxfp4_last_device_status() & 1  # the library workspace's status word
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, torch.tensor([0, 20, 20], dtype=torch.int32), d.sm_scale)
    check_close(as64(out), ref, "clamped")


def test_host_decoder_chunked_pipeline_matches_device_decode():
    """End-to-end path from pinned host buffers, cut into groups of sequences whose
    copies overlap the previous group's decode: same result as one device decode."""
    from mla_decode_attention_mxfp4_gb300 import HostDecoder
    d = MI.make_custom([700, 0, 1500, 33, 2600, 1, 0, 900, 4100], seed=77)
    dev = torch.device("cuda:0")
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    hq, hkv, hsc, hip = (d.q.pin_memory(), d.kv_packed.pin_memory(), d.kv_scale.pin_memory(),
                         d.kv_indptr.pin_memory())
    for chunks in (1, 3, 8):
        hd = HostDecoder(dev, chunks=chunks)
        hout = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16).pin_memory()
        for _ in range(2):  # the second call reuses the device buffers
            hout.fill_(float("nan"))
            hd(hq, hkv, hsc, hip, d.sm_scale, hout)
            hd.synchronize()
            check_close(as64(hout), ref, f"host decoder, {chunks} groups")
