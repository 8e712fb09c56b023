"""The verify+accept cycle in the launch configuration the benchmark times:
one CUDA graph with programmatic dependent launch; per layer a qmv plan for
q, k, v, the GatedDeltaNet tape capture, qmv_smallm for o, a qmv plan for
gate, up and a qmv plan for down; then the LM-head plan (the full
151936-row vocabulary), spec_accept and one tape replay over all layers.
The LM head either writes the logits (spec_accept reads them) or, fused,
keeps per-CTA top-64 lists that spec_accept_lists merges.

Two layers of the 27B-class shapes, every input replaced in place by the
seeded generators, one graph replay.  Checked against the oracle: sampled
rows of every projection, the LM head (every logit, or every listed logit
and the rows' leading tokens), the GatedDeltaNet outputs and tape, and each
layer's committed state; the accept result must equal a standalone accept
launch on the same logits (lists) and be a valid outcome.
"""
import numpy as np
import pytest
import torch

import bench
from gpu_util import assert_qmv_close, dev, sv_module, wl

pytestmark = pytest.mark.gpu

LAYERS, DEPTH = 2, 3
T, TOP_K, TOP_P = float(np.float32(0.6)), 20, float(np.float32(0.95))


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _set(t, a):
    """Copies host array a into device tensor t in place (the plans keep t's
    address); bf16 tensors take uint16 bit patterns, int32 ones uint32 words."""
    a = np.ascontiguousarray(a)
    if t.dtype == torch.bfloat16:
        src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    elif t.dtype == torch.int32:
        src = torch.from_numpy(a.view(np.int32))
    else:
        src = torch.from_numpy(a.astype(np.float32))
    t.copy_(src.reshape(t.shape))


def _split_tape(tape, B, Tn, H, dk, dv):
    blk = Tn * H * (dv + dk) + (Tn * H + 3) // 4 * 4
    t = tape.reshape(B, blk)
    e = t[:, : Tn * H * dv].reshape(B, Tn, H, dv)
    k = t[:, Tn * H * dv: Tn * H * (dv + dk)].reshape(B, Tn, H, dk)
    a = t[:, Tn * H * (dv + dk): Tn * H * (dv + dk) + Tn * H].reshape(B, Tn, H)
    return e, k, a


@pytest.mark.parametrize("fused_head", [True, False])
def test_cycle_in_the_benchmark_launch_configuration(sv, oracle, fused_head):
    M = DEPTH + 1
    sv.set_pdl(True)
    try:
        cyc = bench.Cycle(sv, torch, dev(), depth=DEPTH, layers=LAYERS, layout="plans",
                          fused_head=fused_head)
        V = cyc.V
        host = []
        for i, (w_t, s_t, b_t, x_t, _) in enumerate(cyc.proj + [cyc.lm]):
            N, Kin = w_t.shape[0], w_t.shape[1] * 8
            w, s, b = wl.qmv_weights(2000 + i, N, Kin)
            x = wl.qmv_activations(2000 + i, M, Kin, "bf16")
            for t, a in ((w_t, w), (s_t, s), (b_t, b), (x_t, x)):
                _set(t, a)
            host.append((w, s, b, x))
        gdn = wl.gdn_inputs(2100, LAYERS, M, cyc.heads, cyc.dim, cyc.dim)
        for l in range(LAYERS):
            for t, n in ((cyc.gq[l], "q"), (cyc.gk[l], "k"), (cyc.gv[l], "v"),
                         (cyc.galpha[l], "alpha"), (cyc.gbeta[l], "beta")):
                _set(t, gdn[n][l:l + 1])
        # the oracle's target logits give the drafts: draft = target + N(0, 0.5),
        # tokens drawn from the filtered draft distributions by inverse CDF
        target_ref = oracle.qmv(*host[-1])                       # [M, V]
        draft = (target_ref[None, :DEPTH] + wl.noise(2200, (1, DEPTH, V), 0.5)).astype(np.float32)
        u = wl.uniforms(2300, DEPTH)
        tokens = np.zeros((1, DEPTH), np.int32)
        for k in range(DEPTH):
            q = oracle.filter_row(draft[0, k], T, TOP_K, TOP_P)[0]
            c = np.cumsum(q)
            tokens[0, k] = min(int(np.searchsorted(c, u[k] * c[-1], side="right")), V - 1)
        ua, us = wl.accept_uniforms(2400, 1, DEPTH)
        for t, a in ((cyc.draft, draft), (cyc.draft_tokens, tokens), (cyc.ua, ua), (cyc.us, us)):
            _set(t, a)

        stream = torch.cuda.Stream(dev())
        graph = bench.capture(torch, cyc.run, stream)  # two eager runs, then the capture
        _set(cyc.state, gdn["state0"])                # start again from the snapshot
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        sv.device_status()
    finally:
        sv.set_pdl(False)

    # every projection of every layer: sampled rows
    g = wl.rng(9, 1)
    for i, (w, s, b, x) in enumerate(host[:-1]):
        N = w.shape[0]
        rows = np.unique(np.concatenate([g.choice(N, 48, replace=False), [0, 63, 64, N - 1]]))
        assert_qmv_close(cyc.proj[i][4].cpu().numpy()[:, rows],
                         oracle.qmv(w[rows], s[rows], b[rows], x))
    if fused_head:
        # every listed logit against the oracle's, and each row's 20 leading
        # tokens (ties within the tolerance excepted)
        G = cyc.head_grid
        raw = cyc.topk.cpu().numpy()
        keys = raw[: G * M * 64 * 8].view(np.uint64).reshape(G, M, 64)
        for m in range(M):
            k = keys[:, m][keys[:, m] != 0]
            hi = (k >> np.uint64(32)).astype(np.uint32)
            ids = (0xFFFFFFFF - (k & np.uint64(0xFFFFFFFF))).astype(np.int64)
            vals = np.where(hi & 0x80000000, hi & 0x7FFFFFFF, ~hi).astype(np.uint32).view(np.float32)
            rms = np.sqrt((target_ref[m].astype(np.float64) ** 2).mean())
            assert (np.abs(vals - target_ref[m, ids]) <= 2e-3 * np.maximum(np.abs(target_ref[m, ids]), rms)).all()
            top = ids[np.argsort(-vals, kind="stable")][:TOP_K]
            ref_sorted = np.sort(target_ref[m])[::-1]
            margin = 4e-3 * max(abs(ref_sorted[0]), rms)
            clear = ref_sorted[:TOP_K - 1] - ref_sorted[1:TOP_K] > margin
            want = np.argsort(-target_ref[m], kind="stable")[:TOP_K]
            for j in range(TOP_K):
                if clear[: j + 1].all():
                    assert top[j] == want[j]
        # accept: the cycle's result equals a standalone launch on the same lists
        tok, nacc, flags = sv.spec_accept_lists(cyc.topk.clone(), G, V, cyc.draft,
                                                cyc.draft_tokens, cyc.ua, cyc.us, T, TOP_K, TOP_P)
    else:
        # the LM head: every row
        assert_qmv_close(cyc.lm[4].cpu().numpy(), target_ref)
        # accept: the cycle's result equals a standalone launch on the same logits
        tok, nacc, flags = sv.spec_accept(cyc.target.clone(), cyc.draft, cyc.draft_tokens,
                                          cyc.ua, cyc.us, T, TOP_K, TOP_P)
    torch.cuda.synchronize()
    assert torch.equal(tok, cyc.out_tokens) and torch.equal(nacc, cyc.n_acc)
    n = int(nacc[0])
    tk = tok.cpu().numpy()[0]
    assert 0 <= n <= DEPTH and int(flags[0]) == 0 and int(cyc.flags[0]) == 0
    assert (tk[:n] == tokens[0, :n]).all() and 0 <= tk[n] < V and (tk[n + 1:] == -1).all()

    # GatedDeltaNet: outputs and tape of every layer, then the committed state
    out_ref, tape_ref = oracle.gdn_capture(gdn["state0"], gdn["q"], gdn["k"], gdn["v"],
                                           gdn["alpha"], gdn["beta"])
    for l in range(LAYERS):
        o = cyc.gout[l].cpu().numpy()[0]
        np.testing.assert_array_less(np.abs(o - out_ref[l]), 1e-5 * np.maximum(1.0, np.abs(out_ref[l])))
    e, k, a = _split_tape(cyc.tape.cpu().numpy(), LAYERS, M, cyc.heads, cyc.dim, cyc.dim)
    np.testing.assert_array_less(np.abs(e - tape_ref["e"]), 1e-5 * np.maximum(1.0, np.abs(tape_ref["e"])))
    np.testing.assert_array_equal(k, gdn["k"])
    np.testing.assert_array_equal(a, gdn["alpha"])
    # the replay commits the accepted drafts plus the emitted token in every
    # layer: the oracle's state after each possible count, the one for n + 1
    # compared
    refs = [oracle.gdn_replay(gdn["state0"], tape_ref, np.full(LAYERS, L, np.int32))
            for L in range(M + 1)]
    assert np.abs(cyc.state.cpu().numpy() - refs[n + 1]).max() <= 1e-5
