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
def test_workload_full_size_every_element(name):
    """Full-size workload in the bench's launch configuration (one CTA per SM, every
    sequence split where a range boundary cuts it): every output element of every
    sequence against the oracle (its multi-threaded driver, bitwise the same values)."""
    d = MI.make_inputs(name)
    out, st = gpu_decode(d)
    assert st == 0
    got = as64(out)
    assert np.isfinite(got).all()
    ref = oracle.decode_mt(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(got, ref, name)
    # per sequence too: a bad sequence cannot hide behind the aggregate L2 gate
    for b in range(d.batch):
        nr = np.linalg.norm(ref[b])
        assert np.linalg.norm(got[b] - ref[b]) <= REL_L2 * nr, f"{name}[{b}]"


# ---- within-token scale spreads ------------------------------------------------------
# The K/V operand of a 128-token tile is its codes rebased to the tile's reference exponent
# (its largest scale byte, or up to 4 above it) with 13 binades of headroom (e5m2): every
# block down to 27 binades below the reference is exact, and blocks further below are read
# as zero.  These cases put some blocks of every token far above the others, with values
# left at their natural size (not normalised), so a block read wrongly shows up at the
# per-element tolerance.

BIG_BLOCKS = (0, 7, 17)  # blocks holding each token's largest scale (17: RoPE dims 544..575)


def _spread_case(lens, spreads, seed, lo=126):
    """Seeded inputs whose token t has blocks BIG_BLOCKS at scale byte lo + spread_t, block 3
    at exactly lo and the other blocks in [lo, lo + 2]; the query is zero on BIG_BLOCKS'
    dims, so the scores come from the small blocks, whose values keep the generator's
    natural MXFP4 scale at lo = 126.  The big blocks' codes are made positive, so that
    their dims' outputs (up to ~2^28) are weighted means without cancellation and the
    per-element relative tolerance measures them."""
    d = MI.make_custom(lens, seed=seed)
    rng = np.random.default_rng(seed)
    n = d.total_kv
    s = lo + rng.integers(0, 3, (n, 18))
    s[:, 3] = lo
    sp = np.array([spreads[t % len(spreads)] for t in range(n)], dtype=np.int64)
    for b in BIG_BLOCKS:
        s[:, b] = lo + sp
    assert s.max() <= 254 and s.min() >= 0
    d.kv_scale = torch.from_numpy(s.astype(np.uint8)).contiguous()
    p = d.kv_packed.numpy().copy()
    for b in BIG_BLOCKS:
        p[:, 16 * b:16 * b + 16] &= 0x77
    d.kv_packed = torch.from_numpy(p).contiguous()
    q = d.q.clone()
    for b in BIG_BLOCKS:
        q[:, :, 32 * b:32 * b + 32] = 0
    d.q = q.contiguous()
    return d


def _far_blocks_zeroed(d, limit=27):
    """The same inputs with every block more than `limit` binades below its token's
    largest set to code 0 (what the kernel reads there)."""
    s = d.kv_scale.numpy().astype(np.int64)
    far = s.max(axis=1, keepdims=True) - s > limit
    p = d.kv_packed.numpy().copy()
    for t, b in zip(*np.nonzero(far)):
        p[t, 16 * b:16 * b + 16] = 0
    return torch.from_numpy(p), int(far.sum())


@pytest.mark.parametrize("lo,spreads", [(128, [14, 15, 20, 27]), (10, [14, 27]), (200, [27, 20])])
def test_kv_len_one_is_bit_exact_across_legal_scale_spreads(lo, spreads):
    """One token per sequence: out = bf16(V) bit for bit, for tokens whose blocks span 14,
    15, 20 and 27 binades, at small (2^-117), unit and large (2^73) magnitudes."""
    d = _spread_case([1] * 8, spreads, seed=lo + len(spreads), lo=lo)
    out, st = gpu_decode(d)
    assert st == 0
    k = oracle.dequant_rows(d.kv_packed, d.kv_scale)
    want = torch.from_numpy(oracle.round_bf16(k[:, :512]).view(np.int16).copy()).view(torch.bfloat16)
    want = want.double().numpy()
    assert (k[:, :512] == want).all()  # V is exactly representable in bf16
    got = as64(out)
    for b in range(8):
        for h in range(16):
            assert np.array_equal(got[b, h], want[b]), (b, h)


def test_scale_spreads_up_to_27_binades_match_the_oracle_unnormalised():
    """Multi-tile sequences of tokens with 14-, 15-, 20- and 27-binade spreads: every
    element within the stated tolerance of the definition, at its natural magnitude
    (outputs up to ~2^30 in the large blocks' dims, ~1..10 in the others)."""
    d = _spread_case([200, 37, 129, 1, 300], [14, 15, 20, 27], seed=5)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, "spreads <= 27")


@pytest.mark.parametrize("spreads", [[28, 29, 33, 60], [40]])
def test_blocks_28_or_more_binades_below_are_read_as_zero_one_token(spreads):
    """The other side of the exact range, one token per sequence (each tile's reference is
    that token's largest scale byte): bf16 of V with the blocks 28 or more binades below
    the token's largest zeroed, bit for bit."""
    d = _spread_case([1] * 8, spreads, seed=28)
    p0, nfar = _far_blocks_zeroed(d)
    assert nfar > 0
    out, st = gpu_decode(d)
    assert st == 0
    k = oracle.dequant_rows(p0, d.kv_scale)
    want = torch.from_numpy(oracle.round_bf16(k[:, :512]).view(np.int16).copy()).view(torch.bfloat16)
    want = want.double().numpy()
    got = as64(out)
    for b in range(8):
        for h in range(16):
            assert np.array_equal(got[b, h], want[b]), (b, h)


@pytest.mark.parametrize("spread", [28, 40])
def test_blocks_28_or_more_binades_below_are_read_as_zero_multi_tile(spread):
    """The same for multi-tile sequences whose tokens all share one largest scale byte (so
    the reference of every tile is that byte, whatever the tiling): the output matches the
    oracle run on the zeroed inputs, while the unmodified definition differs there by more
    than the tolerance."""
    d = _spread_case([200, 37, 129], [spread], seed=29)
    p0, nfar = _far_blocks_zeroed(d)
    assert nfar > 0
    out, st = gpu_decode(d)
    assert st == 0
    got = as64(out)
    ref0 = oracle.decode(d.q, p0, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(got, ref0, "far blocks zeroed")
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    assert (np.abs(ref0 - ref) > ATOL + RTOL * np.abs(ref)).any()


@pytest.mark.parametrize("gap_nats", [8.0, 10.0, 12.0])
def test_long_flat_tail_of_small_weights_is_kept(gap_nats):
    """One token per sequence (a "sink") scores `gap_nats` above thousands of others of equal
    score, so a large share of the attention mass sits in weights 2^-11 .. 2^-18 below the
    largest.  Dims 1..31 are 1.0 for every tail token and 0 for the sink, so their outputs
    are exactly the tail's share of the mass (about 0.5 .. 0.02 here): a kernel that drops
    small weights fails them.  The tiles holding the tail carry P in e5m2, whose exponent
    range reaches these weights."""
    d = MI.make_custom([4096, 2048, 700], seed=21)
    p, s = d.kv_packed.clone(), d.kv_scale.clone()
    p[:, 0:16] = 0x22                       # every token: code 1.0 in dims 0..31 ...
    for t0 in (0, 4096 + 1000, 4096 + 2048 + 699):
        p[t0, 0] = 0x07                     # ... the sink: 6.0 in dim 0, 0 in dims 1..31
        p[t0, 1:16] = 0
    s[:, 0] = 127
    d.kv_packed, d.kv_scale = p.contiguous(), s.contiguous()
    q = torch.zeros(3, 16, 576)
    q[:, :, 0] = gap_nats / (5.0 * d.sm_scale)  # score gap = sm_scale * q0 * (6 - 1)
    d.q = q.to(torch.bfloat16)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, f"tail {gap_nats} nats")


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


def _resident_ctas():
    return torch.cuda.get_device_properties(0).multi_processor_count  # one split CTA per SM


@pytest.mark.parametrize("case", ["tiles_below_grid", "tiles_at_grid", "tiles_above_grid",
                                  "one_sequence_over_every_range", "one_sequence_one_tile_more"])
def test_ranges_of_whole_tiles_at_the_grid_size(case):
    # The partition gives each resident CTA floor(gT/G) .. floor((g+1)T/G) of the T tiles:
    # T just below, at and just above G, and a single sequence split over every range (the
    # merge then combines G partials, or G partials with one range holding two tiles).
    G = _resident_ctas()
    lens = {"tiles_below_grid": [128] * (G - 2) + [77],
            "tiles_at_grid": [128] * G,
            "tiles_above_grid": [128] * G + [3],
            "one_sequence_over_every_range": [128 * G],
            "one_sequence_one_tile_more": [128 * G + 5]}[case]
    d = MI.make_custom(lens, seed=len(lens) + 7)
    out, st = gpu_decode(d)
    assert st == 0
    ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
    check_close(as64(out), ref, case)


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
    more than the raise threshold and so does its tile's reference exponent, so the running
    maxima move in the middle of a segment and the accumulator is rescaled (the full path of
    the softmax statistics); a later block of tokens with raised exponents moves the tile
    reference up and back down again."""
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
        hd = HostDecoder(dev, chunks=chunks, direct=False)
        hout = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16).pin_memory()
        for _ in range(2):  # the second call reuses the device buffers
            hout.fill_(float("nan"))
            hd(hq, hkv, hsc, hip, d.sm_scale, hout)
            hd.synchronize()
            check_close(as64(hout), ref, f"host decoder, {chunks} groups")


def test_host_decoder_reading_pinned_inputs_in_place():
    """The direct mode: the kernels read q, kv_packed and kv_scale straight from the pinned
    host buffers (through mla_host_device_pointer); the output is bit-identical to the decode
    of the same inputs copied to the device, and unpinned inputs fall back to the copies."""
    from mla_decode_attention_mxfp4_gb300 import HostDecoder, _lib, decode
    d = MI.make_custom([700, 0, 1500, 33, 2600, 1, 0, 900, 4100], seed=78)
    dev = torch.device("cuda:0")
    hq, hkv, hsc, hip = (d.q.pin_memory(), d.kv_packed.pin_memory(), d.kv_scale.pin_memory(),
                         d.kv_indptr.pin_memory())
    rc, addr = _lib.host_device_pointer(hkv.data_ptr())
    assert rc == _lib.MLA_OK and addr != 0
    rc, addr = _lib.host_device_pointer(d.kv_packed.data_ptr())  # pageable memory: refused
    assert rc == _lib.MLA_ERR_CUDA and addr == 0
    dev_out = decode(d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev), d.sm_scale)
    torch.cuda.synchronize()
    hd = HostDecoder(dev, chunks=1)  # the copy path then decodes the batch in one call, as above
    hout = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16).pin_memory()
    for _ in range(2):
        hout.fill_(float("nan"))
        hd(hq, hkv, hsc, hip, d.sm_scale, hout)
        hd.synchronize()
        assert torch.equal(hout, dev_out.cpu())
    hout.fill_(float("nan"))
    hd(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale, hout)  # not pinned: copies
    hd.synchronize()
    assert torch.equal(hout, dev_out.cpu())


def test_wait_limit_runs_out_cleanly_and_the_context_stays_usable():
    """The failure path of the attention kernel's bounded waits, made to run out on purpose
    without any fault: the test entry point's copy role issues nothing, so the first wait for
    a landed tile gives up after 1 ms.  The call must come back promptly with
    MLA_DEVICE_TIMEOUT in the workspace's status word, and the next normal call on the same
    workspace and stream must be correct with a clear status word."""
    import time

    from mla_decode_attention_mxfp4_gb300 import _lib, alloc_workspace, decode, device_status
    d = MI.make_custom([300, 0, 1000, 5, 129], seed=13)
    dev = torch.device("cuda:0")
    q, kv, sc, ip = d.q.to(dev), d.kv_packed.to(dev), d.kv_scale.to(dev), d.kv_indptr.to(dev)
    out = torch.empty(d.batch, 16, 512, dtype=torch.bfloat16, device=dev)
    ws = alloc_workspace(d.batch)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize()
    for _ in range(2):
        t0 = time.time()
        rc = _lib.mla_decode_mxfp4_ws_stalled(q.data_ptr(), kv.data_ptr(), sc.data_ptr(), ip.data_ptr(),
                                              out.data_ptr(), d.batch, d.sm_scale, stream.cuda_stream,
                                              ws.data_ptr(), ws.numel(), 1_000_000)
        assert rc == _lib.MLA_OK, _lib.status_string(rc)
        st = _lib.mla_decode_mxfp4_device_status(stream.cuda_stream, ws.data_ptr())
        assert st & _lib.MLA_DEVICE_TIMEOUT
        assert time.time() - t0 < 30.0
        good = decode(q, kv, sc, ip, d.sm_scale, workspace=ws)
        assert device_status(None, ws) == 0
        ref = oracle.decode(d.q, d.kv_packed, d.kv_scale, d.kv_indptr, d.sm_scale)
        check_close(as64(good), ref, "after a stalled call")
