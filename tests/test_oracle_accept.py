"""Pins for the oracle's sampling filter and verify-and-accept (CPU only).

What fixes the oracle here, other than itself:
  * losslessness ("MTPLX 2.24x faster TPS", sections "QWEN 3.6 27B @ 63 TPS"
    and "Layer 2: Speculative cycle": exact probability-ratio rejection
    sampling with residual correction keeps the target distribution): the
    analytic law of (accepted length, emitted token) equals p at every
    position to 1e-12, and a large seeded Monte Carlo run through the oracle
    code matches that law within binomial error;
  * the greedy loop of "MTP in llama.cpp", section "lossless": at temperature
    0 the oracle equals a separate accept-until-mismatch loop;
  * closed forms: q == p accepts every draft; disjoint supports accept none;
  * brute force: the top-p set equals the smallest-mass-covering subset found
    by enumerating all subsets of a tiny vocabulary; the kept-set softmax
    equals scipy's softmax.
"""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

import workloads as wl


# ----------------------------------------------------------------------------
# filter
# ----------------------------------------------------------------------------
def test_greedy_filter_is_argmax_lowest_id(oracle):
    z = np.array([1.0, 3.0, -2.0, 3.0, 0.5], np.float32)
    p, flags, _ = oracle.filter_row(z, 0.0, 0, 1.0)
    assert p.tolist() == [0, 1, 0, 0, 0] and flags == 0


def test_top_k_keeps_exactly_k_with_lower_id_ties(oracle):
    z = np.array([5, 1, 4, 4, 4, 0, 4, -3], np.float32)
    p, _, _ = oracle.filter_row(z, 1.0, 3, 1.0)
    assert np.flatnonzero(p).tolist() == [0, 2, 3]
    ref = softmax(z[[0, 2, 3]].astype(np.float64))
    np.testing.assert_allclose(p[[0, 2, 3]], ref, rtol=1e-14)


@pytest.mark.parametrize("T", [0.6, 1.0, 2.5])
def test_kept_softmax_matches_scipy(oracle, T):
    z = wl.accept_logits(11, 1, 0, 300)[0][0, 0]
    p, _, _ = oracle.filter_row(z, T, 20, 1.0)
    kept = np.argsort(-z.astype(np.float64), kind="stable")[:20]
    ref = np.zeros(300)
    ref[kept] = softmax(z[kept].astype(np.float64) / T)
    np.testing.assert_allclose(p, ref, rtol=1e-13, atol=1e-300)


def _brute_top_p(probs: np.ndarray, top_p: float) -> set:
    """Smallest subset with mass >= top_p; among those of that size the one of
    largest mass, then the lexicographically smallest ids (tiny V only)."""
    V = len(probs)
    for size in range(1, V + 1):
        best = None
        for sub in itertools.combinations(range(V), size):
            mass = sum(probs[i] for i in sub)
            if mass >= top_p and (best is None or mass > best[0] + 1e-15):
                best = (mass, sub)
        if best is not None:
            return set(best[1])
    return set(range(V))


@pytest.mark.parametrize("seed", range(40))
def test_top_p_matches_subset_enumeration(oracle, seed):
    g = np.random.default_rng(seed)
    V = 7
    z = (g.standard_normal(V) * 1.5).astype(np.float32)
    top_p = float(g.uniform(0.3, 0.99))
    T = float(g.uniform(0.5, 1.5))
    full, _, _ = oracle.filter_row(z, T, 0, 1.0)      # no truncation
    p, _, margin = oracle.filter_row(z, T, 0, top_p)
    kept = set(np.flatnonzero(p).tolist())
    if margin > 1e-9:
        assert kept == _brute_top_p(full, top_p)
    np.testing.assert_allclose(p[list(kept)], full[list(kept)] / full[list(kept)].sum(), rtol=1e-13)
    assert abs(p.sum() - 1.0) < 1e-14


def test_nonfinite_and_empty_rows(oracle):
    z = np.array([np.nan, -np.inf, 2.0, np.inf], np.float32)
    p, flags, _ = oracle.filter_row(z, 1.0, 5, 1.0)
    assert p.tolist() == [0, 0, 1, 0] and flags == oracle.FLAG_NONFINITE_LOGIT
    p, flags, _ = oracle.filter_row(np.full(4, -np.inf, np.float32), 0.7, 2, 0.9)
    assert p.tolist() == [0, 0, 0, 0] and flags == 0


# ----------------------------------------------------------------------------
# accept: temperature 0
# ----------------------------------------------------------------------------
def _greedy_loop(target_rows, drafts):
    """Accept-until-mismatch with one extra target token (llama.cpp behaviour)."""
    result = []
    for i, d in enumerate(drafts):
        tok = int(np.argmax(target_rows[i]))
        result.append(tok)
        if d != tok:
            break
    else:
        result.append(int(np.argmax(target_rows[len(drafts)])))
    return result


def test_temperature_zero_is_the_greedy_loop(oracle):
    g = np.random.default_rng(5)
    B, K, V = 10000, 4, 6
    tl = g.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32)  # integer logits: ties happen
    am = np.argmax(tl[:, :K], axis=2)
    # drafts agree with the argmax with probability 0.7 per position
    dr = np.where(g.random((B, K)) < 0.7, am, g.integers(0, V, size=(B, K))).astype(np.int32)
    ua, us = wl.accept_uniforms(1, B, K)
    r = oracle.spec_accept(tl, None, dr, ua, us, 0.0, 0, 1.0)
    for b in range(B):
        ref = _greedy_loop(tl[b], dr[b].tolist())
        got = r["out_tokens"][b]
        assert r["n_accepted"][b] == len(ref) - 1
        assert got[: len(ref)].tolist() == ref and (got[len(ref):] == -1).all()
    assert (r["err_flags"] == 0).all()


# ----------------------------------------------------------------------------
# accept: closed forms
# ----------------------------------------------------------------------------
def test_identical_draft_accepts_everything(oracle):
    B, K, V = 200, 3, 50
    tl, _ = wl.accept_logits(21, B, K, V)
    dl = np.ascontiguousarray(tl[:, :K])
    dr = np.zeros((B, K), np.int32)
    us_draw = wl.uniforms(21, (B, K))
    for b in range(B):
        for k in range(K):
            q, _, _ = oracle.filter_row(dl[b, k], 0.6, 20, 0.95)
            dr[b, k] = int(np.searchsorted(np.cumsum(q), us_draw[b, k] * q.sum(), side="right"))
    ua, us = wl.accept_uniforms(21, B, K)
    r = oracle.spec_accept(tl, dl, dr, ua, us, 0.6, 20, 0.95)
    assert (r["n_accepted"] == K).all()
    assert (r["out_tokens"][:, :K] == dr).all()
    for b in range(B):
        p, _, _ = oracle.filter_row(tl[b, K], 0.6, 20, 0.95)
        assert p[r["out_tokens"][b, K]] > 0


def test_disjoint_supports_accept_nothing(oracle):
    B, K, V = 300, 2, 40
    g = np.random.default_rng(3)
    tl = np.full((B, K + 1, V), -np.inf, np.float32)
    dl = np.full((B, K, V), -np.inf, np.float32)
    tl[:, :, :20] = g.standard_normal((B, K + 1, 20))
    dl[:, :, 20:] = g.standard_normal((B, K, 20))
    dr = np.full((B, K), 25, np.int32)
    dl[:, :, 25] = 10.0  # the draft is q's favourite, p gives it nothing
    ua, us = wl.accept_uniforms(4, B, K)
    r = oracle.spec_accept(tl, dl, dr, ua, us, 1.0, 0, 1.0)
    assert (r["n_accepted"] == 0).all()
    assert (r["out_tokens"][:, 0] < 20).all() and (r["out_tokens"][:, 1:] == -1).all()


def test_invalid_drafts_raise_flags(oracle):
    B, K, V = 3, 2, 30
    tl, dl = wl.accept_logits(5, B, K, V)
    dr = np.array([[-1, 0], [V, 0], [0, 0]], np.int32)
    dl[2, 0, :] = -np.inf
    dl[2, 0, 1] = 0.0                                 # q is one-hot on token 1: q(0) = 0
    ua, us = wl.accept_uniforms(5, B, K)
    r = oracle.spec_accept(tl, dl, dr, ua, us, 0.8, 10, 1.0)
    assert (r["n_accepted"] == 0).all()
    assert r["err_flags"].tolist() == [oracle.FLAG_DRAFT_OUT_OF_RANGE] * 2 + [oracle.FLAG_DRAFT_ZERO_Q]
    for b in range(B):
        p, _, _ = oracle.filter_row(tl[b, 0], 0.8, 10, 1.0)
        assert p[r["out_tokens"][b, 0]] > 0


def test_empty_target_row_emits_minus_one(oracle):
    B, K, V = 1, 1, 8
    tl = np.full((B, K + 1, V), -np.inf, np.float32)
    dl = np.zeros((B, K, V), np.float32)
    ua, us = wl.accept_uniforms(6, B, K)
    r = oracle.spec_accept(tl, dl, np.zeros((B, K), np.int32), ua, us, 1.0, 4, 1.0)
    assert r["n_accepted"][0] == 0 and r["out_tokens"][0].tolist() == [-1, -1]
    assert r["err_flags"][0] == oracle.FLAG_EMPTY_DIST


# ----------------------------------------------------------------------------
# accept: losslessness
# ----------------------------------------------------------------------------
def _analytic_law(P, Q):
    """P: [K+1, V] target dists, Q: [K, V] draft dists.  Returns law[j, x] =
    Pr(n_accepted = j and emitted token = x), drafts d_k ~ Q[k] independent."""
    K1, V = P.shape
    K = K1 - 1
    law = np.zeros((K1, V))
    reach = 1.0
    for k in range(K):
        alpha = np.minimum(P[k], Q[k]).sum()                 # Pr(accept at k)
        R = np.maximum(P[k] - Q[k], 0.0)
        Z = R.sum()
        law[k] = reach * (1.0 - alpha) * (R / Z if Z > 0 else P[k])
        reach *= alpha
    law[K] = reach * P[K]
    return law


def _position_marginal(P, Q, law, k):
    """Pr(token emitted at position k = x | position k reached)."""
    K = Q.shape[0]
    reach = np.prod([np.minimum(P[i], Q[i]).sum() for i in range(k)]) if k else 1.0
    if k == K:
        return law[K] / reach
    acc = np.minimum(P[k], Q[k])                             # accepted draft equals x
    return acc + law[k] / reach


@pytest.mark.parametrize("K,T,top_k,top_p", [(2, 1.0, 0, 1.0), (3, 0.6, 4, 0.95),
                                              (3, 1.3, 5, 0.8), (2, 0.7, 3, 1.0)])
def test_emitted_distribution_equals_target(oracle, K, T, top_k, top_p):
    V = 6
    tl, dl = wl.accept_logits(40 + K, 1, K, V, sigma=1.2)
    P = np.stack([oracle.filter_row(tl[0, k], T, top_k, top_p)[0] for k in range(K + 1)])
    Q = np.stack([oracle.filter_row(dl[0, k], T, top_k, top_p)[0] for k in range(K)])
    law = _analytic_law(P, Q)
    assert abs(law.sum() - 1.0) < 1e-12
    for k in range(K + 1):
        np.testing.assert_allclose(_position_marginal(P, Q, law, k), P[k], rtol=0, atol=1e-12)

    # the oracle's own code, run on 400k seeded draws
    B = 400_000
    g = wl.rng(77, K)
    ud = g.random((B, K))
    dr = np.stack([np.minimum(np.searchsorted(np.cumsum(Q[k]), ud[:, k] * Q[k].sum(), side="right"),
                              V - 1) for k in range(K)], axis=1).astype(np.int32)
    ua = g.random((B, K), dtype=np.float32)
    us = g.random(B, dtype=np.float32)
    TL = np.ascontiguousarray(np.broadcast_to(tl, (B, K + 1, V)))
    DL = np.ascontiguousarray(np.broadcast_to(dl, (B, K, V)))
    r = oracle.spec_accept(TL, DL, dr, ua, us, T, top_k, top_p)
    assert (r["err_flags"] == 0).all()
    n = r["n_accepted"]
    emitted = r["out_tokens"][np.arange(B), n]
    for j in range(K):  # accepted prefix is the drafts
        sel = n > j
        assert (r["out_tokens"][sel, j] == dr[sel, j]).all()
    emp = np.zeros_like(law)
    np.add.at(emp, (n, emitted), 1.0)
    emp /= B
    sigma = np.sqrt(law * (1 - law) / B)
    assert (np.abs(emp - law) <= 5 * sigma + 2e-5).all(), np.abs(emp - law).max()


def test_acceptance_rate_is_leviathan_alpha(oracle):
    V, K = 12, 1
    tl, dl = wl.accept_logits(60, 1, K, V, sigma=1.0)
    P = oracle.filter_row(tl[0, 0], 1.0, 0, 1.0)[0]
    Q = oracle.filter_row(dl[0, 0], 1.0, 0, 1.0)[0]
    B = 100_000
    g = wl.rng(61)
    dr = np.minimum(np.searchsorted(np.cumsum(Q), g.random(B) * Q.sum(), side="right"), V - 1)
    r = oracle.spec_accept(np.ascontiguousarray(np.broadcast_to(tl, (B, 2, V))),
                           np.ascontiguousarray(np.broadcast_to(dl, (B, 1, V))),
                           dr.astype(np.int32)[:, None], g.random((B, 1), dtype=np.float32),
                           g.random(B, dtype=np.float32), 1.0, 0, 1.0)
    alpha = np.minimum(P, Q).sum()
    rate = (r["n_accepted"] == 1).mean()
    assert abs(rate - alpha) < 5 * np.sqrt(alpha * (1 - alpha) / B)


def test_margins_report_exact_ties(oracle):
    V, K = 4, 1
    tl = np.zeros((1, 2, V), np.float32)          # p uniform: 0.25 each
    dl = np.log(np.array([[[0.5, 0.25, 0.125, 0.125]]], np.float32))
    dr = np.array([[0]], np.int32)                # ratio p/q = 0.5
    r = oracle.spec_accept(tl, dl, dr, np.array([[0.5]], np.float32),
                           np.array([0.3], np.float32), 1.0, 0, 1.0)
    assert r["diag"][0, 0] < 1e-7                 # u == p/q up to fp32 rounding of q
    assert r["n_accepted"][0] in (0, 1)


def test_sampling_on_a_midpoint_grid(oracle):
    """One uniform axis through the oracle's code: with q == p every draft is
    accepted and the bonus is drawn from p_{K+1}; over the midpoint grid
    u = (j + 1/2)/N the share of each token must equal p within 1/N."""
    V, K, N = 9, 1, 20000
    tl, _ = wl.accept_logits(70, 1, K, V, sigma=1.0)
    p = oracle.filter_row(tl[0, 1], 0.9, 6, 0.97)[0]
    q0 = oracle.filter_row(tl[0, 0], 0.9, 6, 0.97)[0]
    d = int(np.argmax(q0))
    us = ((np.arange(N) + 0.5) / N).astype(np.float32)
    r = oracle.spec_accept(np.ascontiguousarray(np.broadcast_to(tl, (N, K + 1, V))),
                           np.ascontiguousarray(np.broadcast_to(tl[:, :K], (N, K, V))),
                           np.full((N, K), d, np.int32), np.zeros((N, K), np.float32), us,
                           0.9, 6, 0.97)
    assert (r["n_accepted"] == K).all()
    share = np.bincount(r["out_tokens"][:, K], minlength=V) / N
    assert np.abs(share - p).max() <= 1.0 / N + 1e-12
    # tokens come out in ascending id order along the grid (inverse CDF)
    assert (np.diff(r["out_tokens"][:, K]) >= 0).all()


def test_residual_on_a_midpoint_grid(oracle):
    """Same grid on the rejection branch: a draft with p(d) = 0 is always
    rejected and the replacement follows norm((p - q)+)."""
    V, K, N = 8, 1, 20000
    tl, dl = wl.accept_logits(71, 1, K, V, sigma=1.0)
    p = oracle.filter_row(tl[0, 0], 1.0, 5, 1.0)[0]
    q = oracle.filter_row(dl[0, 0], 1.0, 5, 1.0)[0]
    cand = np.flatnonzero((q > 0) & (p == 0))
    assert cand.size, "seed must give a draft outside p's support"
    us = ((np.arange(N) + 0.5) / N).astype(np.float32)
    r = oracle.spec_accept(np.ascontiguousarray(np.broadcast_to(tl, (N, K + 1, V))),
                           np.ascontiguousarray(np.broadcast_to(dl, (N, K, V))),
                           np.full((N, K), cand[0], np.int32), np.zeros((N, K), np.float32), us,
                           1.0, 5, 1.0)
    assert (r["n_accepted"] == 0).all()
    R = np.maximum(p - q, 0.0)
    share = np.bincount(r["out_tokens"][:, 0], minlength=V) / N
    assert np.abs(share - R / R.sum()).max() <= 1.0 / N + 1e-12


def test_zero_residual_falls_back_to_target(oracle):
    """p == q with an out-of-range draft: (p - q)+ has no mass, so the
    replacement is drawn from p itself (and only the range flag is raised)."""
    V, K, N = 10, 1, 4000
    tl, _ = wl.accept_logits(72, 1, K, V, sigma=1.0)
    p = oracle.filter_row(tl[0, 0], 1.0, 0, 1.0)[0]
    us = ((np.arange(N) + 0.5) / N).astype(np.float32)
    r = oracle.spec_accept(np.ascontiguousarray(np.broadcast_to(tl, (N, K + 1, V))),
                           np.ascontiguousarray(np.broadcast_to(tl[:, :K], (N, K, V))),
                           np.full((N, K), V, np.int32), np.zeros((N, K), np.float32), us,
                           1.0, 0, 1.0)
    assert (r["err_flags"] == oracle.FLAG_DRAFT_OUT_OF_RANGE).all()
    share = np.bincount(r["out_tokens"][:, 0], minlength=V) / N
    assert np.abs(share - p).max() <= 1.0 / N + 1e-12


def test_topp_margin_reaches_the_sequence_diagnostics(oracle):
    """A top-p threshold placed on a cumulative sum is reported as a near tie."""
    V, K = 6, 1
    tl, dl = wl.accept_logits(73, 1, K, V, sigma=1.0)
    p_full = oracle.filter_row(tl[0, 0], 1.0, 0, 1.0)[0]
    order = np.argsort(-p_full, kind="stable")
    top_p = float(np.cumsum(p_full[order])[2])          # exactly the 3-token mass
    dr = np.array([[order[0]]], np.int32)
    r = oracle.spec_accept(tl, dl, dr, np.array([[0.5]], np.float32), np.array([0.5], np.float32),
                           1.0, 0, top_p)
    assert r["diag"][0, 1] < 1e-12
    r = oracle.spec_accept(tl, dl, dr, np.array([[0.5]], np.float32), np.array([0.5], np.float32),
                           1.0, 0, top_p - 0.01)
    assert r["diag"][0, 1] > 1e-4
