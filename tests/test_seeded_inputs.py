"""The seeded input generator: deterministic, sliceable, N(0,1), bf16 round-to-nearest-even."""
import numpy as np
import torch

import seeded_inputs as si


def test_deterministic_and_sliceable():
    a = si.normals_f64(42, 1, 0, 5000)
    b = si.normals_f64(42, 1, 0, 5000)
    assert np.array_equal(a, b)
    assert np.array_equal(si.normals_f64(42, 1, 1234, 100), a[1234:1334])
    assert not np.array_equal(si.normals_f64(42, 2, 0, 5000), a)
    assert not np.array_equal(si.normals_f64(43, 1, 0, 5000), a)


def test_standard_normal_moments():
    x = si.normals_f64(42, 1, 0, 1 << 20)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert abs((x > 1.0).mean() - 0.158655) < 2e-3


def test_bf16_rounding_is_round_to_nearest_even():
    x = si.normals_f64(42, 5, 0, 100000) * 7.0
    ours = si.f64_to_bf16_bits(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = si.bf16_bits_to_f64(ours)
    assert np.all(np.abs(back - x.astype(np.float32)) <= np.abs(x) * 2.0 ** -8)


def test_outlier_channels():
    ch = si.outlier_channels(42, si.TENSOR_Q, 32, 128)
    assert len(ch) == 41 and len(set(ch.tolist())) == 41
    assert len(si.outlier_channels(42, si.TENSOR_K, 8, 128)) == 10
    base = si.bshd_bf16(42, si.TENSOR_Q, 1, 4, 32, 128)
    out = si.bshd_bf16(42, si.TENSOR_Q, 1, 4, 32, 128, outlier_fraction=0.01)
    flat_b = si.bf16_bits_to_f64(base).reshape(1, 4, -1)
    flat_o = si.bf16_bits_to_f64(out).reshape(1, 4, -1)
    np.testing.assert_array_equal(flat_o[:, :, ch], 8.0 * flat_b[:, :, ch])
    mask = np.ones(32 * 128, bool)
    mask[ch] = False
    np.testing.assert_array_equal(flat_o[:, :, mask], flat_b[:, :, mask])


def test_sampled_rows_and_heads():
    rows = si.sample_rows(42, 8192, 256)
    assert len(rows) == 256 and rows[0] == 0 and rows[-1] == 8191
    assert {1, 127, 128}.issubset(set(rows.tolist()))
    heads = si.sample_heads(42, 1, 32, 8, 8)
    assert len(heads) == 8 and len({h // 4 for _, h in heads}) == 8
    heads = si.sample_heads(42, 4, 32, 32, 8)
    assert (0, 0) in heads and (3, 31) in heads and len(set(heads)) == 8
