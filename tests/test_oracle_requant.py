"""Pins of the oracle's 4-bit requantisation (the draft-only LM head of
"MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime"), checked against
what the definition fixes rather than against the oracle's own arithmetic:
exact recovery of weights already on a 4-bit grid, the nearest-level property
by brute force over all 16 levels, the half-step error bound, constant
groups, the nibble layout, and a round trip through the oracle's qmv.
"""
import numpy as np
import pytest

import workloads as wl


def _bits(x):
    return wl.to_bf16_bits(np.asarray(x, np.float32))


def _val(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def _nibbles(wp, K):
    wp = np.asarray(wp, np.uint32)
    q = np.empty((wp.shape[0], K), np.int64)
    for j in range(8):
        q[:, j::8] = (wp >> (4 * j)) & 15
    return q


@pytest.mark.parametrize("s0,b0", [(2.0 ** -7, -8 * 2.0 ** -7), (0.75 * 2.0 ** -6, -4 * 2.0 ** -6),
                                   (3.0, 0.5)])
def test_weights_on_a_grid_are_recovered_exactly(oracle, s0, b0):
    N, K = 6, 320
    g = np.random.default_rng(1)
    q = g.integers(0, 16, size=(N, K))
    q[:, ::64] = 0          # every group spans the whole range
    q[:, 1::64] = 15
    w = (s0 * q + b0).astype(np.float32)
    assert np.array_equal(_val(_bits(w)), w.astype(np.float64)), "grid values must be bf16-exact"
    wp, s, b = oracle.requantize(_bits(w))
    assert (s == _bits(s0)).all() and (b == _bits(b0)).all()
    assert np.array_equal(_nibbles(wp, K), q)


def test_nearest_level_and_error_bound(oracle):
    N, K = 40, 512
    w = _bits(np.random.default_rng(2).normal(0, 0.02, (N, K)))
    wp, s, b = oracle.requantize(w)
    q = _nibbles(wp, K)
    wv = _val(w)
    sv = np.repeat(_val(s), 64, axis=1)
    bv = np.repeat(_val(b), 64, axis=1)
    # the group minimum is the bias; the scale is the range over 15 within bf16
    lo = wv.reshape(N, K // 64, 64).min(axis=2)
    hi = wv.reshape(N, K // 64, 64).max(axis=2)
    assert np.array_equal(_val(b), lo)
    assert (np.abs(_val(s) - (hi - lo) / 15) <= 2.0 ** -8 * (hi - lo) / 15).all()
    # brute force: the code is the nearest of the 16 levels (ties and fp32
    # rounding at a tie excepted), and the error is at most half a step plus
    # the top level's shortfall from bf16 rounding of the scale
    levels = bv[..., None] + sv[..., None] * np.arange(16)
    dist = np.abs(wv[..., None] - levels)
    best = dist.argmin(axis=-1)
    srt = np.sort(dist, axis=-1)
    clear = srt[..., 1] - srt[..., 0] > 1e-6 * sv
    assert np.array_equal(q[clear], best[clear])
    err = np.abs(wv - (bv + sv * q))
    assert (err <= 0.55 * sv).all()
    assert (q >= 0).all() and (q <= 15).all() and (q == 0).any() and (q == 15).any()


def test_constant_groups_and_zero(oracle):
    w = np.zeros((3, 128), np.float32)
    w[1, :64] = 0.375
    w[2, 64:] = -2.5
    wp, s, b = oracle.requantize(_bits(w))
    assert (s == 0).all()
    assert np.array_equal(_val(b), np.array([[0, 0], [0.375, 0], [0, -2.5]]))
    assert (wp == 0).all()


def test_zero_extremes_are_positive_zero(oracle):
    w = np.zeros((2, 64), np.float32)
    w[0, 5] = -0.0
    w[0, 9] = 1.5
    w[1, ::2] = -0.0          # a group of signed zeros only
    wp, s, b = oracle.requantize(_bits(w))
    assert b[0, 0] == 0x0000 and s[0, 0] == _bits(np.float32(1.5) / np.float32(15))
    assert b[1, 0] == 0x0000 and s[1, 0] == 0x0000 and wp[1].max() == 0


def test_nibble_order_is_lsb_first(oracle):
    """inputs 0..63 of one group hold levels 0, 1, ..., 15, 0, 1, ...: the
    first packed word of the row is 0x76543210."""
    K = 64
    w = (np.arange(K) % 16).astype(np.float32)[None, :]
    wp, s, b = oracle.requantize(_bits(w))
    assert _val(s)[0, 0] == 1.0 and _val(b)[0, 0] == 0.0
    assert wp[0, 0] == 0x76543210 and wp[0, 1] == 0xFEDCBA98


def test_round_trip_through_qmv(oracle):
    """the requantised matrix times x is the bf16 matrix times x within the
    quantisation error bound sum_i |x_i| * 0.55 s"""
    N, K, M = 24, 384, 3
    w = _bits(np.random.default_rng(3).normal(0, 0.02, (N, K)))
    x = np.random.default_rng(4).standard_normal((M, K)).astype(np.float32)
    wp, s, b = oracle.requantize(w)
    y = oracle.qmv(wp, s, b, x).astype(np.float64)
    dense = x.astype(np.float64) @ _val(w).T
    sv = np.repeat(_val(s), 64, axis=1)
    bound = np.abs(x.astype(np.float64)) @ (0.55 * sv).T + 1e-5
    assert (np.abs(y - dense) <= bound).all()
