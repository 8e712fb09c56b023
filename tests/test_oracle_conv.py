"""Oracle pins for the short causal convolution windows ("MTP와 DFlash",
section "Qwen3.8-Flash-Next (qwen4_exp) MTP": the rollback replays the
GatedDeltaNet recurrence and two convolution windows over the accepted
tokens).  Reading: depthwise causal convolution of width W whose state is
the W-1 most recent inputs of each channel."""
import numpy as np
import pytest

import workloads as wl


def _stream(window, x):
    """[B, W-1+T, C]: the committed window followed by the verify inputs."""
    return np.concatenate([window, x], axis=1).astype(np.float64)


@pytest.mark.parametrize("W", [2, 3, 4, 6])
def test_capture_equals_numpy_convolution(oracle, W):
    d = wl.conv_inputs(1, 3, 5, 17, W)
    y = oracle.conv_capture(d["window"], d["x"], d["weight"])
    h = _stream(d["window"], d["x"])
    for b in range(3):
        for c in range(17):
            ref = np.convolve(h[b, :, c], d["weight"][::-1, c].astype(np.float64), mode="valid")
            np.testing.assert_allclose(y[b, :, c], ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("W", [2, 4, 8])
def test_replay_equals_token_by_token_shift(oracle, W):
    T = 6
    d = wl.conv_inputs(2, 4, T, 9, W)
    for L in range(T + 1):
        got = oracle.conv_replay(d["window"], d["x"], np.full(4, L, np.int32))
        win = d["window"].astype(np.float64).copy()
        for t in range(L):  # drop the oldest entry, append the token's input
            win = np.concatenate([win[:, 1:], d["x"][:, t:t + 1].astype(np.float64)], axis=1)
        np.testing.assert_array_equal(got, win)


def test_replay_zero_keeps_window_and_full_takes_last_inputs(oracle):
    d = wl.conv_inputs(3, 2, 5, 7, 4)
    np.testing.assert_array_equal(oracle.conv_replay(d["window"], d["x"], np.zeros(2, np.int32)),
                                  d["window"].astype(np.float64))
    np.testing.assert_array_equal(oracle.conv_replay(d["window"], d["x"], np.full(2, 5, np.int32)),
                                  d["x"][:, 2:5].astype(np.float64))


def test_commit_then_next_block_equals_one_long_stream(oracle):
    """capture(block 1) -> commit L tokens -> capture(block 2) gives the same
    outputs as one convolution over window, block 1[:L], block 2"""
    W, C = 4, 11
    d1 = wl.conv_inputs(4, 2, 5, C, W)
    d2 = wl.conv_inputs(5, 2, 5, C, W)
    for L in (0, 2, 5):
        win = oracle.conv_replay(d1["window"], d1["x"], np.full(2, L, np.int32))
        y2 = oracle.conv_capture(win, d2["x"], d1["weight"])
        xs = np.concatenate([d1["x"][:, :L], d2["x"]], axis=1)
        y_all = oracle.conv_capture(d1["window"], xs, d1["weight"])
        np.testing.assert_allclose(y2, y_all[:, L:], rtol=1e-13, atol=1e-13)


def test_one_hot_weights(oracle):
    W = 4
    d = wl.conv_inputs(6, 2, 5, 8, W)
    w_last = np.zeros((W, 8), np.float32)
    w_last[W - 1] = 1.0
    np.testing.assert_array_equal(oracle.conv_capture(d["window"], d["x"], w_last),
                                  d["x"].astype(np.float64))
    w_first = np.zeros((W, 8), np.float32)
    w_first[0] = 1.0
    y = oracle.conv_capture(d["window"], d["x"], w_first)
    h = _stream(d["window"], d["x"])
    np.testing.assert_array_equal(y, h[:, :5])  # y_t = h(t - (W - 1))
