"""Pins for the oracle's GatedDeltaNet recurrence and innovation tape (CPU only).

"MTPLX 2.24x faster TPS", section "Layer 0: MLX Runtime": replaying the tape
is bit-exact to the reference recurrence.  Pinned here by:
  * replay of L records == the sequential recurrence stopped after L tokens,
    bit for bit, for every L in 0..T;
  * the gated delta rule in matrix form, S_t = S_{t-1} alpha (I - beta k k^T)
    + beta v k^T, evaluated with numpy matmuls;
  * closed forms: beta = 0 only decays; alpha = 0 leaves beta v k^T;
    alpha = beta = 1 writes v at key k (S_t k_t = v_t);
  * the capture never writes its snapshot.
"""
import numpy as np
import pytest

import workloads as wl


def _small(stream, B=2, T=5, H=3, d=16, **kw):
    return wl.gdn_inputs(stream, B, T, H, d, d, **kw)


def test_replay_is_bit_exact_to_sequential(oracle):
    x = _small(1)
    B, T = x["q"].shape[:2]
    out, tape = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    for L in range(T + 1):
        n = np.full(B, L, np.int32)
        seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], n)
        rep = oracle.gdn_replay(x["state0"], tape, n)
        assert np.array_equal(seq.view(np.uint64), rep.view(np.uint64)), L
    # ragged prefixes per sequence
    n = np.array([0, T], np.int32)
    seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"], n)
    assert np.array_equal(seq, oracle.gdn_replay(x["state0"], tape, n))


def _matrix_form(S0, q, k, v, alpha, beta):
    """Gated delta rule as matrix products (float64); returns states and outputs."""
    B, T, H, dk = k.shape
    S = S0.astype(np.float64).copy()
    states, outs = [], []
    eye = np.eye(dk)
    for t in range(T):
        for b in range(B):
            for h in range(H):
                kk = k[b, t, h].astype(np.float64)
                a, be = float(alpha[b, t, h]), float(beta[b, t, h])
                S[b, h] = S[b, h] @ (a * (eye - be * np.outer(kk, kk))) + be * np.outer(v[b, t, h], kk)
        states.append(S.copy())
        outs.append(np.einsum("bhij,bhj->bhi", S, q[:, t].astype(np.float64)))
    return states, np.stack(outs, axis=1)


def test_matches_matrix_form(oracle):
    x = _small(2, B=2, T=4, H=2, d=12)
    states, outs = _matrix_form(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    out, _ = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    np.testing.assert_allclose(out, outs, rtol=0, atol=1e-12)
    for L in range(1, 5):
        seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"],
                                       x["beta"], np.full(2, L, np.int32))
        np.testing.assert_allclose(seq, states[L - 1], rtol=0, atol=1e-12)


def test_beta_zero_only_decays(oracle):
    x = _small(3)
    x["beta"][:] = 0.0
    seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    ref = x["state0"].astype(np.float64)
    for t in range(x["q"].shape[1]):
        ref = x["alpha"][:, t, :, None, None].astype(np.float64) * ref
    assert np.array_equal(seq, ref)


def test_alpha_zero_writes_beta_v_k(oracle):
    x = _small(4)
    x["alpha"][:] = 0.0
    T = x["q"].shape[1]
    seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    bv = x["beta"][:, T - 1, :, None].astype(np.float64) * x["v"][:, T - 1].astype(np.float64)
    ref = bv[..., :, None] * x["k"][:, T - 1, :, None, :].astype(np.float64)
    np.testing.assert_array_equal(seq, ref)


def test_unit_gates_write_value_at_key(oracle):
    x = _small(5, T=1)
    x["alpha"][:] = 1.0
    x["beta"][:] = 1.0
    seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    Sk = np.einsum("bhij,bhj->bhi", seq, x["k"][:, 0].astype(np.float64))
    np.testing.assert_allclose(Sk, x["v"][:, 0], rtol=0, atol=1e-6)


def test_capture_outputs_are_state_times_query(oracle):
    x = _small(6)
    out, _ = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    B, T = x["q"].shape[:2]
    for L in range(1, T + 1):
        seq, _ = oracle.gdn_sequential(x["state0"], x["q"], x["k"], x["v"], x["alpha"],
                                       x["beta"], np.full(B, L, np.int32))
        ref = np.einsum("bhij,bhj->bhi", seq, x["q"][:, L - 1].astype(np.float64))
        np.testing.assert_allclose(out[:, L - 1], ref, rtol=0, atol=1e-13)


def test_capture_leaves_snapshot_untouched(oracle):
    x = _small(7)
    before = x["state0"].copy()
    oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    assert np.array_equal(before.view(np.uint32), x["state0"].view(np.uint32))


def test_tape_holds_gate_innovation_key(oracle):
    x = _small(8, T=2)
    _, tape = oracle.gdn_capture(x["state0"], x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    np.testing.assert_array_equal(tape["alpha"], x["alpha"].astype(np.float64))
    np.testing.assert_array_equal(tape["k"], x["k"].astype(np.float64))
    # e_0 = beta_0 (v_0 - alpha_0 S0 k_0)
    S0 = x["state0"].astype(np.float64)
    a0 = x["alpha"][:, 0, :, None, None].astype(np.float64)
    u = np.einsum("bhij,bhj->bhi", a0 * S0, x["k"][:, 0].astype(np.float64))
    e0 = x["beta"][:, 0, :, None] * (x["v"][:, 0] - u)
    np.testing.assert_allclose(tape["e"][:, 0], e0, rtol=0, atol=1e-13)
