"""The fused LM head (a qmv plan problem with the top-64 epilogue) and
spec_accept_lists on the GPU.

Checks:
- every per-CTA list is sorted, holds distinct keys, and each key decodes
  to an index whose logit, written by the same plan without the epilogue, is
  bit-identical;
- the 64 largest keys over all lists of a row are that row's 64 largest
  (logit, lower index first) from the written logits;
- acceptance from the lists equals spec_accept on the written logits
  exactly (tokens, counts, flags) for sampling (top_k 20 and 64), greedy, and
  rows with non-finite logits;
- the sampled result is a valid outcome against the oracle's logits.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev, f32, qmv_to_device, sv_module, wl

pytestmark = pytest.mark.gpu

K_DRAFT = 3
M = K_DRAFT + 1


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _decode(keys):
    keys = np.asarray(keys, np.uint64)
    hi = (keys >> np.uint64(32)).astype(np.uint32)
    lo = (keys & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    bits = np.where(hi & 0x80000000, hi & 0x7FFFFFFF, ~hi).astype(np.uint32)
    return bits.view(np.float32), (0xFFFFFFFF - lo).astype(np.int64)


def _keys_of(y_row):
    """Composite keys of a row of logits (finite values), as the kernels form them."""
    u = y_row.astype(np.float32).view(np.uint32).copy()
    u[(u & 0x7FFFFFFF) == 0] = 0
    k = np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint64)
    idx = np.arange(len(y_row), dtype=np.uint64)
    return (k << np.uint64(32)) | (np.uint64(0xFFFFFFFF) - idx)


def _plans(sv, N, Kin, seed, x_override=None):
    w, s, b = wl.qmv_weights(seed, N, Kin)
    x = wl.qmv_activations(seed, M, Kin, "bf16") if x_override is None else x_override
    wt, st, bt, xt = qmv_to_device(w, s, b, x)
    y = torch.empty((M, N), device=dev())
    lists = sv.make_topk_lists(M, torch.bfloat16, dev())
    p_y = sv.QmvPlan([(wt, st, bt, xt, y, False)])
    p_t = sv.QmvPlan([(wt, st, bt, xt, None, False, lists)])
    assert p_y.grid == p_t.grid
    p_y.run()
    p_t.run()
    torch.cuda.synchronize()
    sv.device_status()
    return (w, s, b, x), y, lists, p_t.grid, (p_y, p_t)


def _split(lists, G):
    raw = lists.cpu().numpy()
    keys = raw[: G * M * 64 * 8].view(np.uint64).reshape(G, M, 64)
    flags = raw[G * M * 64 * 8: G * M * 64 * 8 + G * M * 4].view(np.uint32).reshape(G, M)
    return keys, flags


@pytest.mark.parametrize("N,Kin", [(151936, 512), (20000, 1024), (1000, 512)])
def test_lists_hold_each_rows_top64(sv, N, Kin):
    _, y, lists, G, _ = _plans(sv, N, Kin, 500 + N % 97)
    keys, flags = _split(lists, G)
    yn = y.cpu().numpy()
    assert (flags == 0).all()
    for m in range(M):
        k = keys[:, m, :]
        nz = k[k != 0]
        # each list sorted descending with distinct keys, zeros only at the end
        for g in range(G):
            row = k[g]
            n = int((row != 0).sum())
            assert (row[n:] == 0).all()
            assert (row[:n][:-1] > row[:n][1:]).all()  # strictly descending: sorted, distinct
        vals, ids = _decode(nz)
        assert len(np.unique(ids)) == len(ids)
        assert np.array_equal(vals.view(np.uint32), yn[m, ids].astype(np.float32).view(np.uint32))
        want = np.sort(_keys_of(yn[m]))[::-1][:64]
        got = np.sort(nz)[::-1][:64]
        assert np.array_equal(got, want)


def _drafts(target, seed, T, top_k, top_p):
    """draft logits = target + N(0, 0.5); draft tokens drawn from the draft
    distributions filtered as the acceptance filters them (argmax when
    greedy), on the host, seeded"""
    import oracle

    V = target.shape[-1]
    draft = (target[None, :K_DRAFT] + wl.noise(seed, (1, K_DRAFT, V), 0.5)).astype(np.float32)
    u = wl.uniforms(seed + 1, K_DRAFT)
    tokens = np.zeros((1, K_DRAFT), np.int32)
    for k in range(K_DRAFT):
        if T == 0:
            tokens[0, k] = int(np.argmax(draft[0, k]))
            continue
        q = oracle.filter_row(draft[0, k], f32(T), top_k, f32(top_p))[0]
        c = np.cumsum(q)
        tokens[0, k] = min(int(np.searchsorted(c, u[k] * c[-1], side="right")), V - 1)
    ua, us = wl.accept_uniforms(seed + 2, 1, K_DRAFT)
    return draft, tokens, ua, us


@pytest.mark.parametrize("T,top_k,top_p", [(0.6, 20, 0.95), (0.6, 64, 1.0), (1.0, 1, 1.0),
                                            (0.0, 1, 1.0)])
def test_accept_from_lists_equals_accept_from_logits(sv, oracle, T, top_k, top_p):
    N, Kin = 151936, 512
    host, y, lists, G, _ = _plans(sv, N, Kin, 510)
    xs = host[3]
    target = y.cpu().numpy()
    for seed in (520, 530, 540):
        draft, tokens, ua, us = _drafts(target, seed, T, top_k, top_p)
        d = dev()
        dl = torch.from_numpy(draft).to(d)
        dt = torch.from_numpy(tokens).to(d)
        uat, ust = torch.from_numpy(ua).to(d), torch.from_numpy(us).to(d)
        T32, tp32 = f32(T), f32(top_p)
        a = sv.spec_accept(y.view(1, M, N), None if T == 0 else dl, dt, uat, ust, T32, top_k, tp32)
        b = sv.spec_accept_lists(lists, G, N, None if T == 0 else dl, dt, uat, ust, T32, top_k,
                                 tp32)
        torch.cuda.synchronize()
        for u, v in zip(a, b):
            assert torch.equal(u, v)
        n = int(b[1][0])
        tk = b[0].cpu().numpy()[0]
        assert 0 <= n <= K_DRAFT and int(b[2][0]) == 0
        assert (tk[:n] == tokens[0, :n]).all() and 0 <= tk[n] < N and (tk[n + 1:] == -1).all()
        if T == 0:  # greedy: the emitted token is the argmax of the oracle's logits
            ref = oracle.qmv(*host[:3], xs).astype(np.float64)
            top2 = np.sort(ref[n])[-2:]
            if top2[1] - top2[0] > 1e-3 * abs(top2[1]):
                assert tk[n] == int(np.argmax(ref[n]))


def test_non_finite_logits_are_flagged_alike(sv):
    N, Kin = 30000, 512
    x = wl.qmv_activations(550, M, Kin, "f32")
    x[0, 7] = 3e38            # row 0 (always consulted) overflows to +-inf / NaN
    xs = wl.to_bf16_bits(x)
    _, y, lists, G, _ = _plans(sv, N, Kin, 550, x_override=xs)
    keys, flags = _split(lists, G)
    assert flags[:, 0].any() and not flags[:, 1].any()
    d = dev()
    V = N
    draft = torch.from_numpy(np.nan_to_num(y.cpu().numpy()[:K_DRAFT][None], nan=0.0,
                                           posinf=0.0, neginf=0.0)).to(d)
    dt = torch.zeros((1, K_DRAFT), dtype=torch.int32, device=d)
    ua, us = wl.accept_uniforms(551, 1, K_DRAFT)
    uat, ust = torch.from_numpy(ua).to(d), torch.from_numpy(us).to(d)
    a = sv.spec_accept(y.view(1, M, V), draft, dt, uat, ust, f32(0.6), 20, f32(0.95))
    b = sv.spec_accept_lists(lists, G, V, draft, dt, uat, ust, f32(0.6), 20, f32(0.95))
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert int(b[2][0]) & 4  # nonfinite_logit


def test_rejections(sv):
    d = dev()
    lists = torch.zeros(8 << 20, dtype=torch.uint8, device=d)
    dt = torch.zeros((1, K_DRAFT), dtype=torch.int32, device=d)
    ua = torch.zeros((1, K_DRAFT), device=d)
    us = torch.zeros((1,), device=d)
    with pytest.raises(sv.SvError, match="G=3000"):
        sv.spec_accept_lists(lists, 3000, 1000, None, dt, ua, us, 0.0, 1, 1.0)
    # a small vocabulary takes more chunks than its logits fill: one per 32 lists
    assert sv.lib().spec_accept_lists_workspace_bytes(1, 3, 30000, 304) > \
        sv.lib().spec_accept_workspace_bytes(1, 3, 30000)
    assert sv.lib().spec_accept_lists_workspace_bytes(1, 3, 151936, 304) == \
        sv.lib().spec_accept_workspace_bytes(1, 3, 151936)


def test_topk_problem_after_a_phase(sv):
    """a two-phase plan: a projection, then the LM head with the top-64
    epilogue reading its output; the lists equal those of the same head read
    from the logits the plan writes without the epilogue"""
    d = dev()
    N1, K1 = 1024, 512
    N2, K2 = 20000, 1024
    w1, s1, b1 = wl.qmv_weights(560, N1, K1)
    w2, s2, b2 = wl.qmv_weights(561, N2, N1)
    x = wl.qmv_activations(560, M, K1, "f32")
    p1 = qmv_to_device(w1, s1, b1, x)
    wt2, st2, bt2, _ = qmv_to_device(w2, s2, b2, np.zeros((M, N1), np.float32))
    h = torch.empty((M, N1), device=d)
    y = torch.empty((M, N2), device=d)
    lists = sv.make_topk_lists(M, torch.float32, d)
    p_y = sv.QmvPlan([(*p1, h, False), (wt2, st2, bt2, h, y, True)])
    p_t = sv.QmvPlan([(*p1, h, False), (wt2, st2, bt2, h, None, True, lists)])
    p_y.run()
    p_t.run()
    p_t.run()  # twice: the lists are rebuilt, the plan's counters reset
    torch.cuda.synchronize()
    sv.device_status()
    G = p_t.grid
    keys, flags = _split(lists, G)
    yn = y.cpu().numpy()
    assert (flags == 0).all()
    for m in range(M):
        k = keys[:, m, :]
        nz = k[k != 0]
        vals, ids = _decode(nz)
        assert np.array_equal(vals.view(np.uint32), yn[m, ids].astype(np.float32).view(np.uint32))
        assert np.array_equal(np.sort(nz)[::-1][:64], np.sort(_keys_of(yn[m]))[::-1][:64])


def test_two_sequences_from_stacked_blocks(sv):
    """two sequences, each with its own fused LM-head run; their list blocks
    stacked at spec_accept_lists_block_bytes give the same result as
    spec_accept on the two sequences' logits"""
    N, Kin = 30000, 512
    d = dev()
    runs = [_plans(sv, N, Kin, 570 + i) for i in range(2)]
    G = runs[0][3]
    blk = int(sv.lib().spec_accept_lists_block_bytes(G, K_DRAFT))
    stacked = torch.zeros(2 * blk, dtype=torch.uint8, device=d)
    for i, r in enumerate(runs):
        n = r[2].numel()
        assert n <= blk
        stacked[i * blk:i * blk + n].copy_(r[2])
    y = torch.stack([r[1] for r in runs])                       # [2, M, N]
    draft = (y[:, :K_DRAFT] + torch.from_numpy(wl.noise(580, (2, K_DRAFT, N), 0.5)).to(d)).contiguous()
    tokens = draft.argmax(dim=-1).to(torch.int32)               # the drafts' own top tokens
    ua, us = wl.accept_uniforms(581, 2, K_DRAFT)
    uat, ust = torch.from_numpy(ua).to(d), torch.from_numpy(us).to(d)
    for T, top_k, top_p in ((0.6, 20, 0.95), (0.0, 1, 1.0)):
        a = sv.spec_accept(y, None if T == 0 else draft, tokens, uat, ust, f32(T), top_k, f32(top_p))
        b = sv.spec_accept_lists(stacked, G, N, None if T == 0 else draft, tokens, uat, ust, f32(T),
                                 top_k, f32(top_p))
        torch.cuda.synchronize()
        for u, v in zip(a, b):
            assert torch.equal(u, v)
