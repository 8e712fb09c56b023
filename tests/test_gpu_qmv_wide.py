"""qmv_wide (the tcgen05 product for wide verify blocks) on the GPU against
the oracle, element by element, with the tolerance of the qmv tests:
|y_gpu - y_ref| <= 2e-3 * max(|y_ref|, rms of the row of y_ref).

Shapes span several 128-row tiles with a ragged last tile, more tiles than
SMs (so CTAs take several tiles and both accumulators alternate), K from one
512-input stage upwards, and M from 1 to 128 (the MMA's N rounded up to 16,
the activation tile's missing rows filled with zeros by the tensor copy).
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_qmv_close, dev, qmv_to_device, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _run(sv, w, s, b, x, **kw):
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    y = sv.qmv_wide(wt, st, bt, xt, **kw)
    torch.cuda.synchronize()
    sv.device_status()
    return y.cpu().numpy()


@pytest.mark.parametrize("M", [17, 32, 33, 64, 100, 127, 128])
def test_every_width_ragged_tiles(sv, oracle, M):
    N, K = 300, 1024  # three tiles, the last 44 rows; 16 groups + one bias stage
    w, s, b = wl.qmv_weights(400 + M, N, K)
    x = wl.qmv_activations(400 + M, M, K, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_narrow_blocks(sv, oracle, M):
    w, s, b = wl.qmv_weights(420 + M, 200, 512)
    x = wl.qmv_activations(420 + M, M, 512, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


@pytest.mark.parametrize("N,K", [(1, 512), (128, 512), (129, 512), (255, 1536), (640, 2560),
                                 (130, 8192)])
def test_edge_shapes(sv, oracle, N, K):
    w, s, b = wl.qmv_weights(430 + N + K, N, K)
    x = wl.qmv_activations(430 + N + K, 48, K, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


def test_more_tiles_than_sms(sv, oracle):
    """157+ tiles: every CTA takes two or three tiles, accumulators alternate."""
    N, K, M = 128 * 400 + 77, 512, 96
    w, s, b = wl.qmv_weights(440, N, K)
    x = wl.qmv_activations(440, M, K, "bf16")
    y = _run(sv, w, s, b, x)
    g = np.random.default_rng(440)
    rows = np.unique(np.concatenate([g.choice(N, 512, replace=False),
                                     [0, 127, 128, 151 * 128, 152 * 128, 304 * 128, N - 1]]))
    assert_qmv_close(y[:, rows], oracle.qmv(w[rows], s[rows], b[rows], x))


def test_bias_dominated_groups(sv, oracle):
    """Scales tiny against the biases: the result is mostly sum_g b X_g, the
    path through the split group sums."""
    N, K, M = 256, 2048, 64
    w, _, _ = wl.qmv_weights(450, N, K)
    _, s, b = wl.qmv_weights(451, N, K, scale_std=1e-4)
    _, _, b = wl.qmv_weights(452, N, K, scale_std=0.5)
    x = wl.qmv_activations(450, M, K, "bf16")
    assert_qmv_close(_run(sv, w, s, b, x), oracle.qmv(w, s, b, x))


def test_lm_head_batch_of_32_sequences(sv, oracle):
    """The LM head 5120 -> 151936 at M = 128 (32 sequences x 4 verify rows):
    sampled rows, all 128 columns."""
    N, K, M = 151936, 5120, 128
    w, s, b = wl.qmv_weights(300, N, K)
    x = wl.qmv_activations(460, M, K, "bf16")
    y = _run(sv, w, s, b, x)
    g = np.random.default_rng(460)
    rows = np.unique(np.concatenate([g.choice(N, 160, replace=False), [0, 127, 128, N - 1]]))
    assert_qmv_close(y[:, rows], oracle.qmv(w[rows], s[rows], b[rows], x))


def test_deterministic_pdl_and_graph(sv, oracle):
    """Bit-identical across calls, with programmatic dependent launch, and
    inside a captured CUDA graph with a caller workspace."""
    N, K, M = 1000, 1536, 80
    w, s, b = wl.qmv_weights(470, N, K)
    x = wl.qmv_activations(470, M, K, "bf16")
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    y0 = sv.qmv_wide(wt, st, bt, xt)
    ws = sv.make_wide_workspace(M, K, dev())
    y1 = torch.empty_like(y0)
    sv.set_pdl(True)
    try:
        stream = torch.cuda.Stream(dev())
        with torch.cuda.stream(stream):
            sv.qmv_wide(wt, st, bt, xt, y=y1, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(y0, y1)
        y2 = torch.full_like(y0, float("nan"))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            sv.qmv_wide(wt, st, bt, xt, y=y2, workspace=ws)
        with torch.cuda.stream(stream):
            graph.replay()
            graph.replay()
        torch.cuda.synchronize()
    finally:
        sv.set_pdl(False)
    sv.device_status()
    assert torch.equal(y0, y2)
    assert_qmv_close(y0.cpu().numpy(), oracle.qmv(w, s, b, x))


def test_rejections(sv):
    d = dev()
    w = torch.zeros((256, 512 // 8), dtype=torch.int32, device=d)
    s = torch.zeros((256, 8), dtype=torch.bfloat16, device=d)
    x = torch.zeros((129, 512), dtype=torch.bfloat16, device=d)
    with pytest.raises(sv.SvError, match="M=129"):
        sv.qmv_wide(w, s, s, x)
    ws = torch.zeros(16, dtype=torch.uint8, device=d)
    with pytest.raises(sv.SvError, match="workspace"):
        sv.qmv_wide(w, s, s, x[:64], workspace=ws)
    y = sv.qmv_wide(w, s, s, x[:0])
    assert y.shape == (0, 256)
