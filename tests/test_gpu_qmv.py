"""qmv_smallm on the GPU against the oracle (element by element).

Tolerance, per output: |y_gpu - y_ref| <= 2e-3 * max(|y_ref|, rms of the
row of y_ref) -- "within 2e-3 relative error in fp32 accumulation" with a
row-RMS floor so that outputs near zero are judged against the row's scale.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_qmv_close, qmv_to_device, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _run(sv, w, s, b, x):
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    y = sv.qmv_smallm(wt, st, bt, xt)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def test_tiny_config_fp32_rows(sv, oracle):
    """one 4-bit linear, out=512 in=256, 4 fp32 rows ~ N(0,1), s/b ~ N(0,0.02)"""
    w, s, b = wl.qmv_weights(0, 512, 256)
    x = wl.qmv_activations(0, 4, 256, "f32")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_every_m_ragged_tiles(sv, oracle, M, xdt):
    N, K = 100, 640  # 4 CTAs, last one 4 rows; 10 groups: one full stage + a partial one
    w, s, b = wl.qmv_weights(10 + M, N, K)
    x = wl.qmv_activations(10 + M, M, K, xdt)
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("N,K", [(1, 64), (16, 64), (17, 192), (31, 128), (33, 576), (48, 1024),
                                 (1000, 64), (7, 1536)])
def test_edge_shapes(sv, oracle, N, K):
    w, s, b = wl.qmv_weights(N + K, N, K)
    x = wl.qmv_activations(N + K, 5, K, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


def _sampled(sv, oracle, N, K, M, stream, xdt="bf16", n_rows=192):
    w, s, b = wl.qmv_weights(stream, N, K)
    x = wl.qmv_activations(stream, M, K, xdt)
    y = _run(sv, w, s, b, x)
    g = np.random.default_rng(stream)
    rows = np.unique(np.concatenate([g.choice(N, n_rows, replace=False), [0, 15, 16, 31, N - 1]]))
    ref = oracle.qmv(w[rows], s[rows], b[rows], x)
    assert_qmv_close(y[:, rows], ref)
    return y


@pytest.mark.parametrize("M", [1, 4, 8])
def test_mlp_gate_up_shape(sv, oracle, M):
    _sampled(sv, oracle, 17408, 5120, M, 100 + M)


@pytest.mark.parametrize("M", [2, 4, 6])
def test_mlp_down_shape(sv, oracle, M):
    _sampled(sv, oracle, 5120, 17408, M, 200 + M)


def test_lm_head_shape(sv, oracle):
    _sampled(sv, oracle, 151936, 5120, 4, 300, n_rows=128)


def test_attention_shape_fp32_rows(sv, oracle):
    _sampled(sv, oracle, 5120, 5120, 3, 400, xdt="f32")


def test_deterministic_and_pdl_invariant(sv):
    w, s, b = wl.qmv_weights(500, 4096, 2048)
    x = wl.qmv_activations(500, 4, 2048, "bf16")
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    sv.set_pdl(False)
    y0 = sv.qmv_smallm(wt, st, bt, xt).clone()
    sv.set_pdl(True)
    try:
        ys = [sv.qmv_smallm(wt, st, bt, xt) for _ in range(8)]
        # a chain: each call's rows come from the previous output
        chain = xt.clone()
        for _ in range(4):
            yy = sv.qmv_smallm(wt, st, bt, chain)
            chain = yy[:, :2048].to(torch.bfloat16).contiguous()
        torch.cuda.synchronize()
    finally:
        sv.set_pdl(False)
    for y in ys:
        assert torch.equal(y, y0)
    ref = xt.clone()
    for _ in range(4):
        yy = sv.qmv_smallm(wt, st, bt, ref)
        ref = yy[:, :2048].to(torch.bfloat16).contiguous()
    torch.cuda.synchronize()
    assert torch.equal(chain, ref)
    sv.device_status()


def test_empty_and_invalid(sv):
    w, s, b = wl.qmv_weights(600, 32, 64)
    wt, st, bt, _ = qmv_to_device(w, s, b, wl.qmv_activations(600, 1, 64, "bf16"))
    x0 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda:0")
    assert sv.qmv_smallm(wt, st, bt, x0).shape == (0, 32)
    x17 = torch.zeros((17, 64), dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(sv.SvError):
        sv.qmv_smallm(wt, st, bt, x17)


# ---- 9..16 rows (a DFlash-width verify block): two 8-row MMA n-tiles ------

@pytest.mark.parametrize("M", [9, 10, 12, 15, 16])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_wide_m_ragged_tiles(sv, oracle, M, xdt):
    N, K = 100, 640  # ragged row tile, K not a multiple of 512 (scale block path)
    w, s, b = wl.qmv_weights(700 + M, N, K)
    x = wl.qmv_activations(700 + M, M, K, xdt)
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("N,K", [(1, 64), (33, 576), (130, 2048), (7, 1536)])
def test_wide_m_edge_shapes(sv, oracle, N, K):
    w, s, b = wl.qmv_weights(800 + N, N, K)
    x = wl.qmv_activations(800 + N, 16, K, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("N,K,M", [(5120, 5120, 16), (17408, 5120, 12), (5120, 17408, 16)])
def test_wide_m_full_shapes(sv, oracle, N, K, M):
    """split-K clusters (5120 rows: 80 tiles) and many tiles (17408 rows)"""
    _sampled(sv, oracle, N, K, M, 900 + M)


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_wide_m_rows_equal_single_rows(sv, xdt):
    """row m of a 16-row product is bitwise the product of row m alone (the
    block-vs-sequential identity holds across the two n-tiles too)"""
    N, K = 5120, 5120
    w, s, b = wl.qmv_weights(950, N, K)
    x = wl.qmv_activations(950, 16, K, xdt)
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    block = sv.qmv_smallm(wt, st, bt, xt)
    rows = [sv.qmv_smallm(wt, st, bt, xt[m:m + 1].contiguous()) for m in (0, 7, 8, 9, 15)]
    torch.cuda.synchronize()
    block = block.cpu().numpy()
    for m, r in zip((0, 7, 8, 9, 15), rows):
        np.testing.assert_array_equal(block[m], r.cpu().numpy()[0], err_msg=f"row {m}")
