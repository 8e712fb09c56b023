"""qmv plan (one persistent launch over an ordered list of projections) on the
GPU against the oracle, element by element, with the qmv tolerance
|y - ref| <= 2e-3 * max(|ref|, rms of ref's row).

Chained problems (`after`) read an earlier problem's fp32 output as their
activations; the oracle chains its own outputs (rounded to fp32), never the
GPU's.
"""
import time

import numpy as np
import pytest
import torch

from gpu_util import assert_qmv_close, dev, qmv_to_device, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _weights(stream, N, K):
    w, s, b = wl.qmv_weights(stream, N, K)
    wt, st, bt, _ = qmv_to_device(w, s, b, np.zeros((1, K), np.float32))
    return (w, s, b), (wt, st, bt)


def _plan_case(sv, oracle, specs, M, xdt, seed):
    """specs: list of (N, K, src) with src None (fresh activations) or the
    index of the earlier problem whose output is x (then K == that N)."""
    host, probs, refs = [], [], []
    for i, (N, K, src) in enumerate(specs):
        (w, s, b), (wt, st, bt) = _weights(seed * 100 + i, N, K)
        if src is None:
            x = wl.qmv_activations(seed * 100 + i, M, K, xdt)
            _, _, _, xt = qmv_to_device(w, s, b, x)
        else:
            assert specs[src][0] == K and xdt == "f32"
            x = refs[src].astype(np.float32)
            xt = probs[src][4]
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev())
        probs.append((wt, st, bt, xt, y, src is not None))
        refs.append(oracle.qmv(w, s, b, x))
        host.append((w, s, b, x))
    plan = sv.QmvPlan(probs)
    return plan, probs, refs


def _check(probs, refs):
    torch.cuda.synchronize()
    for i, (p, r) in enumerate(zip(probs, refs)):
        assert_qmv_close(p[4].cpu().numpy(), r)


def test_independent_problems_bf16(sv, oracle):
    specs = [(512, 1024, None), (100, 512, None), (1000, 1536, None), (64, 512, None),
             (2048, 512, None)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "bf16", 1)
    plan.run()
    _check(probs, refs)
    sv.device_status()


@pytest.mark.parametrize("M", [1, 3, 4, 8])
def test_chained_problems_f32(sv, oracle, M):
    """every problem after the first reads the previous output: each phase
    waits for the one before it"""
    specs = [(1024, 512, None), (512, 1024, 0), (1536, 512, 1), (512, 1536, 2),
             (2560, 512, 3)]
    plan, probs, refs = _plan_case(sv, oracle, specs, M, "f32", 2 + M)
    plan.run()
    _check(probs, refs)
    sv.device_status()


def test_tiny_phases_fewer_stages_than_ctas(sv, oracle):
    """phases of 1..3 stages (far fewer than CTAs) and ragged row tiles"""
    specs = [(512, 512, None),                    # phase 1: 8 stages
             (40, 512, 0), (512, 512, None),       # phase 2: 1 + 8 stages
             (1, 512, 2), (130, 1024, None)]       # phase 3: 1 + 3 x 2 stages
    plan, probs, refs = _plan_case(sv, oracle, specs, 2, "f32", 9)
    plan.run()
    _check(probs, refs)
    sv.device_status()


def test_repeat_runs_are_identical(sv, oracle):
    """counters are left ready: back-to-back runs give bit-identical results"""
    specs = [(2048, 2048, None), (512, 2048, 0), (4096, 512, 1)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "f32", 11)
    outs = []
    for _ in range(3):
        for p in probs:
            p[4].fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        outs.append([p[4].cpu().numpy().copy() for p in probs])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            np.testing.assert_array_equal(a, b)
    _check(probs, refs)
    sv.device_status()


def test_matches_qmv_smallm(sv, oracle):
    """same problems one call at a time: equal up to fp32 summation order"""
    specs = [(17408 // 8, 5120, None), (5120 // 4, 17408 // 2, None)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "bf16", 12)
    plan.run()
    torch.cuda.synchronize()
    for (wt, st, bt, xt, y, _), r in zip(probs, refs):
        y1 = sv.qmv_smallm(wt, st, bt, xt)
        torch.cuda.synchronize()
        a, b = y.cpu().numpy(), y1.cpu().numpy()
        rms = np.sqrt((r ** 2).mean(axis=1, keepdims=True))
        assert (np.abs(a - b) <= 1e-5 * np.maximum(np.abs(r), rms)).all()
    _check(probs, refs)


def test_graph_capture_and_replay(sv, oracle):
    specs = [(1024, 1024, None), (2048, 1024, 0)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "f32", 13)
    stream = torch.cuda.Stream(dev())
    with torch.cuda.stream(stream):
        plan.run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        plan.run()
    for p in probs:
        p[4].fill_(float("nan"))
    with torch.cuda.stream(stream):
        g.replay()
        g.replay()
    _check(probs, refs)
    sv.device_status()


def test_one_layer_full_size_sampled(sv, oracle):
    """one 27B-class layer (q, k, v, o 5120x5120; gate, up 5120->17408; down
    17408->5120) at M=4 bf16 with the real dependency phases, sampled rows"""
    specs = [(5120, 5120, "q"), (5120, 5120, "k"), (5120, 5120, "v"), (5120, 5120, "o"),
             (17408, 5120, "gate"), (17408, 5120, "up"), (5120, 17408, "down")]
    after = {"o": True, "gate": True, "down": True}
    probs, samples = [], []
    g = np.random.default_rng(5)
    for i, (N, K, name) in enumerate(specs):
        (w, s, b), (wt, st, bt) = _weights(700 + i, N, K)
        x = wl.qmv_activations(700 + i, 4, K, "bf16")
        _, _, _, xt = qmv_to_device(w, s, b, x)
        y = torch.full((4, N), float("nan"), dtype=torch.float32, device=dev())
        probs.append((wt, st, bt, xt, y, after.get(name, False)))
        rows = np.unique(np.concatenate([g.choice(N, 96, replace=False), [0, 63, 64, N - 1]]))
        samples.append((rows, oracle.qmv(w[rows], s[rows], b[rows], x)))
    plan = sv.QmvPlan(probs)
    plan.run()
    torch.cuda.synchronize()
    for p, (rows, ref) in zip(probs, samples):
        y = p[4].cpu().numpy()
        assert not np.isnan(y).any()
        assert_qmv_close(y[:, rows], ref)
    sv.device_status()


def test_plan_rejects(sv):
    _, (wt, st, bt) = _weights(1, 64, 640)
    x = torch.zeros((4, 640), dtype=torch.bfloat16, device=dev())
    y = torch.zeros((4, 64), dtype=torch.float32, device=dev())
    with pytest.raises(sv.SvError) as e:
        sv.QmvPlan([(wt, st, bt, x, y, False)])  # K % 512 != 0
    assert e.value.status == 2
    _, (wt, st, bt) = _weights(2, 64, 512)
    _, (w1, s1, b1) = _weights(3, 512, 512)
    x = torch.zeros((4, 512), dtype=torch.float32, device=dev())
    y0 = torch.zeros((4, 512), dtype=torch.float32, device=dev())
    y = torch.zeros((4, 64), dtype=torch.float32, device=dev())
    with pytest.raises(sv.SvError):  # reads problem 0's output without `after`
        sv.QmvPlan([(w1, s1, b1, x, y0, False), (wt, st, bt, y0, y, False)])
    sv.QmvPlan([(w1, s1, b1, x, y0, False), (wt, st, bt, y0, y, True)]).close()


def test_phase_wait_gives_up_and_reports(sv, oracle):
    """Failure detection without a fault: the finished-tile count of a
    two-phase plan (the last 256 bytes of its buffer hold the counters) is
    preset so that the second phase's wait can never be met.  Every CTA gives
    up after its bounded wait (about a second), sets the device error word
    and finishes; sv_device_status reports it, the plan's last CTA has put
    the count back to zero and the context and the plan work again."""
    specs = [(1024, 512, None), (512, 1024, 0)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "f32", 21)
    end = plan._off + plan._nbytes
    done = plan.buffer[end - 256:end - 252].view(torch.int32)
    done.fill_(-(1 << 30))
    torch.cuda.synchronize()
    t0 = time.time()
    plan.run()
    torch.cuda.synchronize()
    took = time.time() - t0
    with pytest.raises(sv.SvError) as e:
        sv.device_status()
    assert e.value.status == 4
    assert 0.5 < took < 60
    assert int(done.item()) == 0
    for p in probs:
        p[4].fill_(float("nan"))
    plan.run()
    _check(probs, refs)
    sv.device_status()


def test_cooperative_run_equals_run(sv, oracle):
    """qmv_plan_run_cooperative gives the same bits as qmv_plan_run"""
    specs = [(2048, 1024, None), (1024, 2048, 0), (512, 1024, 1)]
    plan, probs, refs = _plan_case(sv, oracle, specs, 4, "f32", 21)
    plan.run()
    torch.cuda.synchronize()
    first = [p[4].cpu().numpy().copy() for p in probs]
    for p in probs:
        p[4].fill_(float("nan"))
    plan.run(cooperative=True)
    torch.cuda.synchronize()
    for a, p in zip(first, probs):
        np.testing.assert_array_equal(p[4].cpu().numpy(), a)
    _check(probs, refs)
    sv.device_status()


def test_two_cooperative_plans_on_two_streams(sv, oracle):
    """Two multi-phase plans launched cooperatively on two streams at once:
    the device keeps each plan's CTAs resident together, so neither plan's
    phase waits run out and both results are right."""
    specs = [(4096, 2048, None), (2048, 4096, 0), (1024, 2048, 1)]
    plan_a, probs_a, refs_a = _plan_case(sv, oracle, specs, 4, "f32", 22)
    plan_b, probs_b, refs_b = _plan_case(sv, oracle, specs, 4, "f32", 23)
    streams = [torch.cuda.Stream(dev()), torch.cuda.Stream(dev())]
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(streams[0]):
            plan_a.run(cooperative=True)
        with torch.cuda.stream(streams[1]):
            plan_b.run(cooperative=True)
    torch.cuda.synchronize()
    sv.device_status()  # raises if a wait gave up
    _check(probs_a, refs_a)
    _check(probs_b, refs_b)
