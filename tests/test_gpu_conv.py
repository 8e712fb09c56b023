"""Short causal convolution windows on the GPU against the oracle.

Capture outputs: |y - ref| <= 2e-6 * sum_j |w_j h_j| (an fp32 multiply-add
chain of W <= 8 terms is within W * 2^-24 of that sum).  The commit is a copy:
bit for bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _to(d):
    return {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev()) for k, v in d.items()}


def _bound(d):
    W = d["weight"].shape[0]
    h = np.concatenate([d["window"], d["x"]], axis=1).astype(np.float64)
    T = d["x"].shape[1]
    w = np.abs(d["weight"].astype(np.float64))
    return sum(w[j][None, None, :] * np.abs(h[:, j:j + T]) for j in range(W))


@pytest.mark.parametrize("W", [2, 3, 4, 5, 8])
@pytest.mark.parametrize("B,T,C", [(3, 5, 17), (2, 1, 300), (4, 9, 257)])
def test_capture_matches_oracle(sv, oracle, W, B, T, C):
    d = wl.conv_inputs(10 + W + C, B, T, C, W)
    t = _to(d)
    before = t["window"].clone()
    y = sv.conv_window_capture(t["window"], t["x"], t["weight"])
    torch.cuda.synchronize()
    ref = oracle.conv_capture(d["window"], d["x"], d["weight"])
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert (err <= 2e-6 * _bound(d) + 1e-30).all()
    assert torch.equal(t["window"], before)  # the committed window is read only


@pytest.mark.parametrize("W", [2, 4, 8])
def test_replay_is_exact(sv, oracle, W):
    B, T, C = 6, 5, 300
    d = wl.conv_inputs(20 + W, B, T, C, W)
    d["n_replay"] = np.array([0, 1, 2, 3, 5, 4], np.int32)
    t = _to(d)
    sv.conv_window_replay(t["window"], t["x"], t["n_replay"])
    torch.cuda.synchronize()
    ref = oracle.conv_replay(d["window"], d["x"], d["n_replay"])
    np.testing.assert_array_equal(t["window"].cpu().numpy().astype(np.float64), ref)


def test_replay_bias_shared_count_and_clamp_flags(sv, oracle):
    B, T, C, W = 4, 5, 64, 4
    d = wl.conv_inputs(31, B, T, C, W)
    t = _to(d)
    n = torch.tensor([4], dtype=torch.int32, device=dev())  # one count for all, +1 -> 5
    flags = torch.zeros(B, dtype=torch.int32, device=dev())
    sv.conv_window_replay(t["window"], t["x"], n, n_replay_bias=1, err_flags=flags)
    torch.cuda.synchronize()
    ref = oracle.conv_replay(d["window"], d["x"], np.full(B, 5, np.int32))
    np.testing.assert_array_equal(t["window"].cpu().numpy().astype(np.float64), ref)
    assert (flags.cpu().numpy() == 0).all()
    n2 = torch.tensor([5, -3, 2, 9], dtype=torch.int32, device=dev())  # +1: 6, -2, 3, 10
    t2 = _to(d)
    sv.conv_window_replay(t2["window"], t2["x"], n2, n_replay_bias=1, err_flags=flags)
    torch.cuda.synchronize()
    ref2 = oracle.conv_replay(d["window"], d["x"], np.array([5, 0, 3, 5], np.int32))
    np.testing.assert_array_equal(t2["window"].cpu().numpy().astype(np.float64), ref2)
    assert flags.cpu().numpy().tolist() == [16, 16, 0, 16]


def test_full_size_layer_sampled(sv, oracle):
    """48 heads x (q, k, v) x 128 channels, W = 4, T = 5, batch 16"""
    B, T, C, W = 16, 5, wl.CONV_CHANNELS, wl.CONV_WIDTH
    d = wl.conv_inputs(40, B, T, C, W)
    t = _to(d)
    y = sv.conv_window_capture(t["window"], t["x"], t["weight"]).cpu().numpy()
    cols = np.random.default_rng(1).choice(C, 256, replace=False)
    sub = {k: (v[..., cols] if k != "n_replay" else v) for k, v in d.items()}
    ref = oracle.conv_capture(sub["window"], sub["x"], sub["weight"])
    err = np.abs(y[..., cols].astype(np.float64) - ref)
    assert (err <= 2e-6 * _bound(sub) + 1e-30).all()
    sv.conv_window_replay(t["window"], t["x"], t["n_replay"])
    torch.cuda.synchronize()
    got = t["window"].cpu().numpy()[..., cols].astype(np.float64)
    np.testing.assert_array_equal(got, oracle.conv_replay(sub["window"], sub["x"], d["n_replay"]))
    sv.device_status()
