"""gdn_tape_capture / gdn_tape_replay on the GPU.

* Against the oracle (float64): replayed state within 1e-5 max abs, outputs
  o_t within 1e-5 * max(1, |o|), tape innovations within 1e-5 * max(1, |e|),
  tape gates and keys exact copies.
* Bit for bit on the GPU: replaying L records of a T-token tape gives exactly
  the state the capture itself reaches after its first L tokens (the capture's
  state_out over the first L tokens), for every L in 0..T.
"""
import numpy as np
import pytest
import torch

from gpu_util import dev, sv_module, wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    return sv_module()


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def _split_tape(tape, B, T, H, dk, dv):
    """Per-sequence blocks: e [T][H][dv], k [T][H][dk], alpha [T][H] (padded)."""
    blk = T * H * (dv + dk) + (T * H + 3) // 4 * 4
    t = tape.reshape(B, blk)
    e = t[:, : T * H * dv].reshape(B, T, H, dv)
    k = t[:, T * H * dv: T * H * (dv + dk)].reshape(B, T, H, dk)
    a = t[:, T * H * (dv + dk): T * H * (dv + dk) + T * H].reshape(B, T, H)
    return e, k, a


def _capture(sv, x, T=None, state_out=True):
    T = x["q"].shape[1] if T is None else T
    args = [_t(x[n][:, :T]) for n in ("q", "k", "v", "alpha", "beta")]
    s0 = _t(x["state0"])
    so = torch.empty_like(s0) if state_out else None
    out, tape = sv.gdn_tape_capture(s0, *args, state_out=so)
    torch.cuda.synchronize()
    return out, tape, so


@pytest.mark.parametrize("B,T,H,dk,dv", [(16, 5, 48, 128, 128), (2, 3, 3, 64, 64),
                                         (3, 7, 2, 32, 96), (1, 1, 1, 128, 4), (2, 16, 1, 8, 128),
                                         (2, 12, 3, 128, 128), (1, 16, 2, 128, 64)])
def test_capture_and_replay_match_the_oracle(sv, oracle, B, T, H, dk, dv):
    x = wl.gdn_inputs(B * 100 + T, B, T, H, dk, dv)
    out_ref, tape_ref = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"],
                                           x["beta"])
    out, tape, _ = _capture(sv, x)
    out = out.cpu().numpy()
    np.testing.assert_array_less(np.abs(out - out_ref), 1e-5 * np.maximum(1.0, np.abs(out_ref)))
    e, k, a = _split_tape(tape.cpu().numpy(), B, T, H, dk, dv)
    np.testing.assert_array_less(np.abs(e - tape_ref["e"]),
                                 1e-5 * np.maximum(1.0, np.abs(tape_ref["e"])))
    np.testing.assert_array_equal(k, x["k"])
    np.testing.assert_array_equal(a, x["alpha"])
    # replay the accepted prefixes
    n = x["n_replay"]
    state = _t(x["state0"])
    sv.gdn_tape_replay(state, tape, _t(n), T)
    torch.cuda.synchronize()
    ref = oracle.gdn_replay(x["state0"], tape_ref, n)
    assert np.abs(state.cpu().numpy() - ref).max() <= 1e-5


def test_replay_is_bit_exact_to_the_capture(sv):
    B, T, H, d = 4, 6, 8, 128
    x = wl.gdn_inputs(7, B, T, H, d, d)
    _, tape, _ = _capture(sv, x, state_out=False)
    for L in range(T + 1):
        st = _t(x["state0"])
        sv.gdn_tape_replay(st, tape, torch.full((B,), L, dtype=torch.int32, device=dev()), T)
        if L == 0:
            ref = _t(x["state0"])
        else:
            _, _, ref = _capture(sv, x, T=L)
        torch.cuda.synchronize()
        assert torch.equal(st.view(torch.int32), ref.view(torch.int32)), L


def test_capture_leaves_the_snapshot(sv):
    x = wl.gdn_inputs(8, 2, 5, 4, 128, 128)
    s0 = _t(x["state0"])
    before = s0.clone()
    sv.gdn_tape_capture(s0, *[_t(x[n]) for n in ("q", "k", "v", "alpha", "beta")])
    torch.cuda.synchronize()
    assert torch.equal(s0.view(torch.int32), before.view(torch.int32))


def test_warm_state_and_bias_and_clamp(sv, oracle):
    """State from 16 warm-up tokens of the oracle recurrence; the replay count
    comes from accepted lengths + 1; out-of-range counts are clamped and
    flagged."""
    B, T, H, d = 5, 5, 6, 128
    warm = wl.gdn_inputs(9, B, 16, H, d, d)
    s_warm, _ = oracle.gdn_sequential(np.zeros((B, H, d, d), np.float32), warm["q"], warm["k"],
                                      warm["v"], warm["alpha"], warm["beta"])
    x = wl.gdn_inputs(10, B, T, H, d, d)
    x["state0"] = s_warm.astype(np.float32)
    _, tape_ref = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    _, tape, _ = _capture(sv, x, state_out=False)
    n_acc = np.array([0, 2, 4, 6, -3], np.int32)          # +1 bias; 6+1 and -3+1 clamp
    flags = torch.zeros(B, dtype=torch.int32, device=dev())
    st = _t(x["state0"])
    sv.gdn_tape_replay(st, tape, _t(n_acc), T, n_replay_bias=1, err_flags=flags)
    torch.cuda.synchronize()
    L = np.clip(n_acc + 1, 0, T).astype(np.int32)
    ref = oracle.gdn_replay(x["state0"], tape_ref, L)
    assert np.abs(st.cpu().numpy() - ref).max() <= 1e-5
    assert flags.cpu().tolist() == [0, 0, 0, 16, 16]


def test_layers_share_one_count_per_sequence(sv, oracle):
    """Three layers' states of the same two sequences stacked as one batch of
    six blocks; one accepted length per sequence commits all layers."""
    layers, Bs, T, H, d = 3, 2, 4, 3, 64
    x = wl.gdn_inputs(11, layers * Bs, T, H, d, d)
    _, tape_ref = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    _, tape, _ = _capture(sv, x, state_out=False)
    n_seq = np.array([2, 3], np.int32)
    st = _t(x["state0"])
    sv.gdn_tape_replay(st, tape, _t(n_seq), T)
    torch.cuda.synchronize()
    ref = oracle.gdn_replay(x["state0"], tape_ref, np.tile(n_seq, layers))
    assert np.abs(st.cpu().numpy() - ref).max() <= 1e-5
