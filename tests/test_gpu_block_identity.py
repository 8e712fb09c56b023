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
