"""Block-vs-sequential identity ("MTP와 DFlash", section "MTP 정확성 검사": a
block verify must equal single-token steps byte for byte).

Row m of a verify product over M rows must be bitwise equal to the product
of that row alone (M = 1): the reduction order of each output may not depend
on M.  Checked for qmv_smallm (with and without split-K clusters, ragged
tiles, bf16 and fp32 activations) and for qmv plans.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev, qmv_to_device, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


@pytest.mark.parametrize("N,K", [(5120, 5120), (4352, 5120), (100, 640), (64, 17408)])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_qmv_rows_equal_single_row_calls(sv, N, K, xdt):
    w, s, b = wl.qmv_weights(300 + N % 97, N, K)
    x = wl.qmv_activations(300 + N % 97, 5, K, xdt)
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    block = sv.qmv_smallm(wt, st, bt, xt)
    rows = [sv.qmv_smallm(wt, st, bt, xt[m:m + 1].contiguous()) for m in range(5)]
    torch.cuda.synchronize()
    block = block.cpu().numpy()
    for m, r in enumerate(rows):
        np.testing.assert_array_equal(block[m], r.cpu().numpy()[0], err_msg=f"row {m}")


def test_plan_rows_equal_single_row_plans(sv):
    shapes = [(5120, 5120), (17408 // 4, 5120), (5120 // 2, 17408 // 2)]
    probs = []
    for i, (N, K) in enumerate(shapes):
        w, s, b = wl.qmv_weights(400 + i, N, K)
        x = wl.qmv_activations(400 + i, 4, K, "bf16")
        probs.append(qmv_to_device(w, s, b, x))
    ys = [torch.empty((4, N), device=dev()) for N, _ in shapes]
    plan = sv.QmvPlan([(w, s_, b_, x, y, False) for (w, s_, b_, x), y in zip(probs, ys)])
    plan.run()
    torch.cuda.synchronize()
    for m in range(4):
        y1 = [torch.empty((1, N), device=dev()) for N, _ in shapes]
        plan1 = sv.QmvPlan([(w, s_, b_, x[m:m + 1].contiguous(), y, False)
                            for (w, s_, b_, x), y in zip(probs, y1)])
        plan1.run()
        torch.cuda.synchronize()
        for i, (a, r) in enumerate(zip(ys, y1)):
            np.testing.assert_array_equal(a.cpu().numpy()[m], r.cpu().numpy()[0],
                                          err_msg=f"problem {i} row {m}")


@pytest.mark.parametrize("N,K", [(5120, 5120), (100, 640), (64, 17408), (17408, 5120)])
@pytest.mark.parametrize("M", [2, 4, 8])
@pytest.mark.parametrize("xdt", [torch.bfloat16, torch.float32])
def test_identity_probe_reports_exact(sv, N, K, M, xdt):
    """the start-up probe (three synthetic blocks, compared on the device)
    finds no differing output bit"""
    w, s, b = wl.qmv_weights(500 + N % 89, N, K)
    wt, st, bt, _ = qmv_to_device(w, s, b, np.zeros((1, K), np.float32))
    assert sv.qmv_identity_probe(wt, st, bt, M, xdt) == 0
    sv.device_status()


def test_identity_probe_counts_what_a_host_comparison_counts(sv):
    """the probe's verdict agrees with comparing the same products on the
    host: here both are zero for M = 5 on a ragged shape, and the probe leaves
    the weights untouched"""
    N, K = 1000, 1536
    w, s, b = wl.qmv_weights(601, N, K)
    wt, st, bt, _ = qmv_to_device(w, s, b, np.zeros((1, K), np.float32))
    before = wt.clone()
    assert sv.qmv_identity_probe(wt, st, bt, 5) == 0
    assert torch.equal(wt, before)
    x = wl.qmv_activations(601, 5, K, "bf16")
    _, _, _, xt = qmv_to_device(w, s, b, x)
    block = sv.qmv_smallm(wt, st, bt, xt).cpu().numpy()
    rows = np.concatenate([sv.qmv_smallm(wt, st, bt, xt[m:m + 1].contiguous()).cpu().numpy()
                           for m in range(5)])
    assert int((block.view(np.uint32) != rows.view(np.uint32)).sum()) == 0
