"""Pins of the FP8 block-quantisation oracle (``oracle/fp8.py``; "Lower latency and higher
throughput with multi-node DeepSeek deployment", Quantization: 128 x 128 weight tiles,
1 x 128 activation vectors).  CPU only."""
from fractions import Fraction

import numpy as np
import torch

from oracle import fp8


def test_e4m3_table_matches_the_library_format():
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    ours = fp8.e4m3_values()
    nan = np.isnan(ours)
    assert np.array_equal(nan, np.isnan(codes)) and nan.sum() == 2      # 0x7F, 0xFF
    assert np.array_equal(ours[~nan], codes[~nan])
    assert np.nanmax(ours) == 448.0 and np.nanmin(np.abs(ours[ours != 0])) == 2.0 ** -9


def test_e4m3_rounding_matches_the_library_cast():
    rng = np.random.default_rng(0)
    v = rng.uniform(-448, 448, 20000) * np.exp(rng.uniform(-14, 0, 20000))
    grid = fp8.e4m3_values()
    grid = np.unique(grid[~np.isnan(grid)])
    mids = (grid[1:] + grid[:-1]) / 2                                   # every tie
    v = np.concatenate([v, mids, grid, [0.0, -0.0]]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v).float().to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(fp8.e4m3_round(v), ref)


def test_scale_exponent_worked_values():
    # the smallest k with amax <= 448 * 2^k
    assert fp8.scale_exponent(448.0) == 0
    assert fp8.scale_exponent(449.0) == 1
    assert fp8.scale_exponent(224.0) == -1
    assert fp8.scale_exponent(1.0) == -8          # 448 / 256 = 1.75 >= 1 > 0.875
    assert fp8.scale_exponent(1.75) == -8
    assert fp8.scale_exponent(1.7578125) == -7
    assert fp8.scale_exponent(0.0) == 0
    assert fp8.scale_exponent(2.0 ** -130) == -124                  # clamped: tiny blocks
    assert fp8.scale_exponent(2.0 ** -116) == -124
    assert fp8.scale_exponent(2.0 ** -115) == -123
    rng = np.random.default_rng(1)
    for a in rng.uniform(1e-6, 1e4, 2000):
        k = fp8.scale_exponent(a)
        assert a <= 448.0 * 2.0 ** k and a > 448.0 * 2.0 ** (k - 1)


def test_quantisation_error_bound_and_idempotence():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((6, 384)) * np.exp(rng.uniform(-8, 4, (6, 1)))
    xq = fp8.fake_quant_rows(x)
    for j in range(0, 384, 128):
        blk, bq = x[:, j:j + 128], xq[:, j:j + 128]
        for r in range(6):
            k = fp8.scale_exponent(np.abs(blk[r]).max())
            # half a grid step: 2^(e-4) relative in the normal range, 2^-10 * 2^k below it
            bound = np.maximum(np.abs(blk[r]) * 2.0 ** -4, 2.0 ** (k - 10))
            assert np.all(np.abs(bq[r] - blk[r]) <= bound)
    np.testing.assert_array_equal(fp8.fake_quant_rows(xq), xq)


def test_values_on_the_grid_with_full_range_pass_unchanged():
    grid = fp8.e4m3_values()
    grid = grid[~np.isnan(grid)]
    rng = np.random.default_rng(3)
    x = rng.choice(grid, (4, 256))
    x[:, 0] = 448.0
    x[:, 128] = -448.0                     # amax 448 in every block: scale 2^0
    np.testing.assert_array_equal(fp8.fake_quant_rows(x), x)
    q, k = fp8.quantize_weight(np.tile(x, (32, 1))[:128])
    assert np.all(k == 0)


def test_weight_blocks_are_independent():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((2, 256, 384)) * 0.02
    W[1, 128:, 256:] *= 1000.0             # one block 1000x larger: only its scale moves
    q, k = fp8.quantize_weight(W)
    assert k.shape == (2, 2, 3)
    assert k[1, 1, 2] == fp8.scale_exponent(np.abs(W[1, 128:, 256:]).max())
    assert k[1, 1, 2] >= k[1, 1, 1] + 9
    # quantising a single block on its own gives the same codes and scale
    qb, kb = fp8.quantize_weight(W[1, 128:, 128:256])
    np.testing.assert_array_equal(qb, q[1, 128:, 128:256])
    assert kb[0, 0] == k[1, 1, 1]
    Wd = fp8.dequantize_weight(q, k)
    kk = np.repeat(np.repeat(k, 128, axis=-2), 128, axis=-1)
    err = np.abs(Wd - W)
    assert np.all((err <= np.abs(W) * 2.0 ** -4) | (err <= 2.0 ** (kk - 10)))


def test_round_bf16_is_the_nearest_even_value():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(3000) * np.exp(rng.uniform(-20, 5, 3000))
    r = fp8.round_bf16(x)
    for xi, ri in zip(x[:300], r[:300]):
        # the neighbours of ri on the bf16 grid: one unit in the 8th significant bit
        m, e = np.frexp(ri)
        ulp = 2.0 ** (e - 8)
        d = abs(Fraction(xi) - Fraction(ri))
        assert d <= Fraction(ulp) / 2
    # exactly representable float32 values: the library cast is exact to compare with
    f = x.astype(np.float32)
    np.testing.assert_array_equal(fp8.round_bf16(f.astype(np.float64)),
                                  torch.from_numpy(f).to(torch.bfloat16).double().numpy())


def test_fp8_expert_is_close_to_the_exact_expert():
    # the FP8 expert differs from the exact one by the quantisation noise only
    rng = np.random.default_rng(6)
    H, I = 256, 128
    x = rng.standard_normal((8, H))
    W1, W3 = rng.standard_normal((H, I)) * 0.05, rng.standard_normal((H, I)) * 0.05
    W2 = rng.standard_normal((I, H)) * 0.05
    d = [fp8.dequantize_weight(*fp8.quantize_weight(W)) for W in (W1, W3, W2)]
    y8 = fp8.expert_rows_fp8(x, *d)
    u, v = x @ W1, x @ W3
    y = (u / (1 + np.exp(-u)) * v) @ W2
    rel = np.linalg.norm(y8 - y) / np.linalg.norm(y)
    assert 1e-3 < rel < 0.08
