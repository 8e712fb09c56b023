"""qmv_requantize (the drafter's own 4-bit LM head) on the GPU against the
oracle: packed codes, scales and biases bit for bit (the codes are integers
decided in fp32 on both sides), on random and special weights, ragged
shapes and the full LM head (sampled rows); then the draft step itself,
qmv_smallm at M = 1 on the requantised head, against the oracle's qmv of the
oracle's requantisation.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_qmv_close, dev, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _gpu(sv, w_bits):
    wt = torch.from_numpy(np.ascontiguousarray(w_bits).view(np.int16)).to(dev()).view(torch.bfloat16)
    wp, s, b = sv.qmv_requantize(wt)
    torch.cuda.synchronize()
    return (wp.cpu().numpy().view(np.uint32), s.view(torch.int16).cpu().numpy().view(np.uint16),
            b.view(torch.int16).cpu().numpy().view(np.uint16))


def _check(got, want):
    for g, w, name in zip(got, want, ("w_packed", "scales", "biases")):
        if not np.array_equal(g, w):
            bad = np.argwhere(g != w)
            raise AssertionError(f"{name}: {len(bad)} differ, first at {tuple(bad[0])}: "
                                 f"gpu {g[tuple(bad[0])]:#x} oracle {w[tuple(bad[0])]:#x}")


@pytest.mark.parametrize("N,K", [(1, 64), (7, 192), (300, 1024), (1000, 5120), (33, 17408)])
def test_random_weights_bit_exact(sv, oracle, N, K):
    w = wl.to_bf16_bits(wl.rng(40, N + K).normal(0, 0.02, (N, K)).astype(np.float32))
    _check(_gpu(sv, w), oracle.requantize(w))


def test_special_weights_bit_exact(sv, oracle):
    """constant groups, signed zeros, a group on an exact 4-bit grid, ties at
    half a step, huge and tiny magnitudes, one outlier per group"""
    K = 64
    rows = [np.zeros(K), np.full(K, 0.375), np.where(np.arange(K) % 2, 0.0, -0.0),
            (np.arange(K) % 16) * 0.25 - 1.0, (np.arange(K) % 31) * 0.5,
            np.linspace(-1e30, 1e30, K), np.linspace(-1e-30, 3e-30, K),
            np.r_[np.full(K - 1, 0.01), 40.0], np.r_[-40.0, np.full(K - 1, 0.01)]]
    w = wl.to_bf16_bits(np.stack(rows).astype(np.float32))
    _check(_gpu(sv, w), oracle.requantize(w))


def test_lm_head_full_size_sampled_rows(sv, oracle):
    N, K = wl.VOCAB, wl.HIDDEN
    w = np.empty((N, K), np.uint16)
    step = 8192
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        w[r0:r1] = wl.to_bf16_bits(wl.rng(41, r0).normal(0, 0.02, (r1 - r0, K)).astype(np.float32))
    got = _gpu(sv, w)
    rows = np.unique(np.concatenate([np.random.default_rng(41).choice(N, 256, replace=False),
                                     [0, 1, N - 2, N - 1]]))
    want = oracle.requantize(w[rows])
    _check(tuple(a[rows] for a in got), want)


def test_draft_step_on_the_requantised_head(sv, oracle):
    """drafter logits: qmv_smallm(requantise(W), x) at M = 1, against the
    oracle's qmv of the oracle's requantisation"""
    N, K = 2000, 5120
    w = wl.to_bf16_bits(wl.rng(42, 0).normal(0, 0.02, (N, K)).astype(np.float32))
    x = wl.qmv_activations(42, 1, K, "bf16")
    wt = torch.from_numpy(w.view(np.int16)).to(dev()).view(torch.bfloat16)
    wp, s, b = sv.qmv_requantize(wt)
    xt = torch.from_numpy(x.view(np.int16)).to(dev()).view(torch.bfloat16)
    y = sv.qmv_smallm(wp, s, b, xt)
    torch.cuda.synchronize()
    sv.device_status()
    assert_qmv_close(y.cpu().numpy(), oracle.qmv(*oracle.requantize(w), x))


def test_rejections(sv):
    w = torch.zeros((4, 100), dtype=torch.bfloat16, device=dev())
    with pytest.raises(sv.SvError, match="K"):
        sv.qmv_requantize(w)
    out = sv.qmv_requantize(torch.zeros((0, 128), dtype=torch.bfloat16, device=dev()))
    assert out[0].shape == (0, 16)
