"""The seeded MXFP4 input generator: layout, scale rule and rounding."""
import math

import numpy as np
import torch

import mla_inputs as MI
import oracle


def test_on_grid_values_round_trip_exactly():
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    rng = np.random.default_rng(0)
    x = torch.zeros(8, 576)
    for t in range(8):
        for b in range(18):
            e = int(rng.integers(-20, 20))
            vals = rng.choice(grid, 32) * rng.choice([-1.0, 1.0], 32)
            vals[0] = 6.0  # amax 6 -> shared exponent e exactly
            x[t, 32 * b:32 * b + 32] = torch.from_numpy(vals * 2.0 ** e)
    p, s = MI.quantize_mxfp4(x)
    back = oracle.dequant_rows(p, s)
    assert np.array_equal(back, x.double().numpy())


def test_scale_rule_and_ties_to_even():
    x = torch.zeros(1, 576)
    x[0, :12] = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.1, 0.0, 6.0, 4.0])
    x[0, 32:34] = torch.tensor([0.75, -0.375])      # amax 0.75 -> exponent -1-2
    p, s = MI.quantize_mxfp4(x)
    assert s[0, 0] == 127 and s[0, 1] == 124 and s[0, 2] == 127  # zero block -> 127
    k = oracle.dequant_rows(p, s)[0]
    assert k[:12].tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.0, 0.0, 6.0, 4.0]
    assert k[32] == 0.75 and k[33] == -0.375
    assert p[0, 4] & 0xF == 8  # -0.1 rounds to negative zero


def test_workload_shapes_and_ragged_lengths():
    d = MI.make_inputs("tiny")
    assert d.q.shape == (1, 16, 576) and d.q.dtype == torch.bfloat16
    assert d.kv_packed.shape == (256, 288) and d.kv_scale.shape == (256, 18)
    assert d.kv_indptr.tolist() == [0, 256]
    assert d.algorithmic_bytes() == 18432 + 256 * 306 + 16384
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1, 32769, (64,), generator=g)
    assert int(lens.sum()) == 1152539 and int(lens.min()) == 1589 and int(lens.max()) == 32617
    d = MI.make_inputs("ragged", batch=2)
    assert d.kv_indptr.tolist() == [0, int(lens[0]), int(lens[0] + lens[1])]


def test_generator_is_deterministic():
    a, b = MI.make_inputs("small", batch=1), MI.make_inputs("small", batch=1)
    assert torch.equal(a.kv_packed, b.kv_packed) and torch.equal(a.q, b.q)
    assert torch.equal(a.kv_scale, b.kv_scale)
