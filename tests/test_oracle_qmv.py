"""Pins for the oracle's quantised mat-vec (CPU only).

The oracle (C, float64) is checked against things other than itself:
  * the nibble order fixture in tests/golden (hand-written words);
  * a dense dequantise-then-matmul path in numpy (library matmul);
  * closed forms: one-hot rows pick single weights, zero scales leave only the
    bias term, constant nibbles reduce to a row sum.
"""
from pathlib import Path

import numpy as np
import pytest

import workloads as wl

GOLDEN = Path(__file__).resolve().parent / "golden"


def _dense(w, s, b):
    """Dense float64 W[N, K] from packed words (vectorised numpy)."""
    N, words = w.shape
    K = words * 8
    shifts = np.arange(8, dtype=np.uint32) * np.uint32(4)
    q = ((w[:, :, None] >> shifts[None, None, :]) & np.uint32(15)).reshape(N, K)
    sf = np.repeat(wl.bf16_bits_to_f32(s).astype(np.float64), 64, axis=1)
    bf = np.repeat(wl.bf16_bits_to_f32(b).astype(np.float64), 64, axis=1)
    return q.astype(np.float64) * sf + bf


def _x64(x):
    return wl.bf16_bits_to_f32(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


def test_nibble_order_golden(oracle):
    rows = []
    for line in (GOLDEN / "qmv_nibble_order.txt").read_text().splitlines():
        if line.strip() and not line.startswith("#"):
            parts = line.split()
            rows.append((int(parts[0], 16), [int(t) for t in parts[1:]]))
    # one output row per word: K = 64 (one group), word in slot 0, rest zero;
    # scale 1, bias 0, x = identity rows -> y[m, n] = q[n, m]
    N, K = len(rows), 64
    w = np.zeros((N, K // 8), np.uint32)
    for n, (word, _) in enumerate(rows):
        w[n, 0] = word
    one = wl.to_bf16_bits(np.ones((N, 1), np.float32))
    zero = wl.to_bf16_bits(np.zeros((N, 1), np.float32))
    x = np.eye(8, K, dtype=np.float32)
    y = oracle.qmv(w, one, zero, x)
    for n, (_, vals) in enumerate(rows):
        assert y[:, n].tolist() == [float(v) for v in vals]


@pytest.mark.parametrize("M,N,K,xdt", [(4, 512, 256, "f32"), (1, 48, 64, "bf16"),
                                       (8, 96, 640, "bf16"), (3, 17, 192, "f32")])
def test_matches_dense_dequant(oracle, M, N, K, xdt):
    w, s, b = wl.qmv_weights(100 + M, N, K)
    x = wl.qmv_activations(100 + M, M, K, xdt)
    y = oracle.qmv(w, s, b, x)
    ref = _x64(x) @ _dense(w, s, b).T
    # the oracle rounds a float64 sum once to fp32
    np.testing.assert_allclose(y, ref.astype(np.float32), rtol=2e-7, atol=1e-30)
    assert np.abs(y.astype(np.float64) - ref).max() <= 6e-8 * np.abs(ref).max()


def test_one_hot_rows_pick_weights(oracle):
    N, K = 32, 256
    w, s, b = wl.qmv_weights(7, N, K)
    W = _dense(w, s, b)
    idx = np.array([0, 1, 63, 64, 130, 255])
    x = np.zeros((len(idx), K), np.float32)
    x[np.arange(len(idx)), idx] = 1.0
    y = oracle.qmv(w, s, b, x)
    np.testing.assert_array_equal(y, W[:, idx].T.astype(np.float32))


def test_zero_scale_leaves_bias_times_group_sum(oracle):
    N, K = 16, 320
    w, _, b = wl.qmv_weights(8, N, K)
    s = np.zeros_like(b)
    x = wl.qmv_activations(8, 5, K, "f32").astype(np.float64)
    y = oracle.qmv(w, s, b, x.astype(np.float32))
    gsum = x.reshape(5, K // 64, 64).sum(axis=2)  # [M, G]
    ref = gsum @ wl.bf16_bits_to_f32(b).astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-6, atol=1e-9)


def test_constant_nibbles_reduce_to_row_sum(oracle):
    N, K = 8, 128
    w = np.full((N, K // 8), 0x33333333, np.uint32)  # every q = 3
    s = wl.to_bf16_bits(np.full((N, K // 64), 0.5, np.float32))
    b = wl.to_bf16_bits(np.full((N, K // 64), -0.25, np.float32))
    x = wl.qmv_activations(9, 2, K, "bf16")
    y = oracle.qmv(w, s, b, x)
    ref = _x64(x).sum(axis=1) * (0.5 * 3 - 0.25)
    np.testing.assert_allclose(y, np.repeat(ref[:, None], N, axis=1), rtol=1e-7)


def test_rejects_bad_group(oracle):
    w = np.zeros((4, 12), np.uint32)  # K = 96, not a multiple of 64
    s = np.zeros((4, 1), np.uint16)
    with pytest.raises(ValueError):
        oracle.qmv(w, s, s, np.zeros((1, 96), np.float32))
