"""Pins of the oracle's speculative acceptance ("Mixed-precision compression of DeepSeek-V4-Flash", "What
compression does not solve": accept a draft with probability min(1, p/q), on rejection draw from the normalised
max(p - q, 0)).

The pins do not restate the oracle's arithmetic. They check what the rule guarantees and what it reduces to:
  * losslessness: over the draft's randomness (d ~ q, u uniform) the first committed token is distributed as p.
    The law is computed exactly: the decision and the draw are monotone in their uniforms, so bisection over the
    fp32 uniforms finds where they change, and the drafts are summed with weights q;
  * greedy decoding (one-hot p and q): the committed tokens are the target's argmaxes, whatever the uniforms;
  * p = q: every draft is accepted; the extra token is then distributed as the last target row;
  * disjoint supports: no draft is accepted and the residual is p itself;
  * the edge cases of the quotient (q = 0 < p accepts, p = q = 0 rejects) and a draft id outside [0, V).
A plausible mistake -- accepting on u > p/q, the residual as q - p or not clamped at 0, the extra token from q,
an off-by-one in the draw -- fails at least one of them.
"""
import numpy as np
import pytest

import oracle
from moe_inputs import spec_inputs

ONE_BITS = 0x3F800000  # bits of 1.0f: the fp32 values in [0, 1) are the bit patterns 0 .. ONE_BITS - 1, in order


def _f32(bits: int) -> float:
    return float(np.array([bits], np.uint32).view(np.float32)[0])


def _first_true(pred) -> float:
    """The smallest u in [0, 1) (as a real: fp32 values are ordered like their bits) where a monotone predicate
    of the fp32 uniform turns true; 1.0 if it never does."""
    lo, hi = 0, ONE_BITS  # pred(lo - 1) false (or lo = 0), pred(hi) true by convention
    if pred(0.0):
        return 0.0
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if pred(_f32(mid)):
            hi = mid
        else:
            lo = mid
    return 1.0 if hi == ONE_BITS else _f32(hi)


def _accept_prob(p, q, d, accept=oracle.spec_accept):
    """Measure of the acceptance uniforms (u in [0, 1)) that accept draft d (K = 1)."""
    return _first_true(lambda ua: accept(p, q, [d], [ua, 0.5])[0] == 0)


def _draw_law(p, q, draft, ua, accept=oracle.spec_accept):
    """Law of the drawn token over its uniform: the draw is monotone in it, so each token's share is the
    distance between the uniforms where the token first reaches v and v + 1."""
    V = p.shape[1]
    starts = [0.0] + [_first_true(lambda us: accept(p, q, draft, list(ua) + [us])[1] >= v)
                      for v in range(1, V)] + [1.0]
    return np.diff(np.array(starts))


def _first_token_law(p, q, accept=oracle.spec_accept):
    """Law of the first committed token with K = 1 over the draft d ~ q and both uniforms."""
    V = p.shape[1]
    law = np.zeros(V)
    for d in range(V):
        if q[0, d] == 0:
            continue
        pa = _accept_prob(p, q, d, accept)
        law[d] += q[0, d] * pa
        if pa < 1.0:
            law += q[0, d] * (1.0 - pa) * _draw_law(p, q, [d], [0.9999999], accept)
    return law


def test_lossless_first_token_dyadic():
    p = np.array([[6, 5, 3, 2], [1, 1, 1, 13]], np.float32) / 16
    q = np.array([[2, 9, 4, 1]], np.float32) / 16
    np.testing.assert_allclose(_first_token_law(p, q), p[0], atol=1e-6)


def test_lossless_first_token_random():
    for seed in (5, 6, 7):
        p, q, _, _ = spec_inputs(seed, 1, 6, spread=1.0, noise=1.0)
        np.testing.assert_allclose(_first_token_law(p, q), p[0], atol=1e-6)


def test_greedy_is_argmax_chain():
    rng = np.random.default_rng(3)
    V, K = 11, 5
    for trial in range(40):
        a = rng.integers(0, V, size=K + 1)          # target argmax per position
        d = np.where(rng.random(K) < 0.6, a[:K], rng.integers(0, V, size=K)).astype(np.int32)
        p = np.zeros((K + 1, V), np.float32)
        p[np.arange(K + 1), a] = 1
        q = np.zeros((K, V), np.float32)
        q[np.arange(K), d] = 1
        u = rng.random(K + 1).astype(np.float32)
        n, tok = oracle.spec_accept(p, q, d, u)
        m = 0
        while m < K and d[m] == a[m]:
            m += 1
        assert n == m
        assert tok == a[m]


def test_equal_distributions_accept_everything_and_draw_from_last_row():
    p, _, d, _ = spec_inputs(7, 3, 6, spread=1.0)
    q = p[:3].copy()
    for us in (0.0, 0.3, 0.9999999):
        assert oracle.spec_accept(p, q, d, [0.9999999, 0.5, 0.0, us])[0] == 3
    np.testing.assert_allclose(_draw_law(p, q, d, [0.9999999, 0.5, 0.0]), p[3], atol=1e-6)


def test_disjoint_supports_reject_and_draw_from_target():
    p = np.array([[0.5, 0.5, 0, 0], [0.25, 0.25, 0.25, 0.25]], np.float32)
    q = np.array([[0, 0, 0.5, 0.5]], np.float32)
    for us in (0.0, 0.6, 0.9999999):
        assert oracle.spec_accept(p, q, [2], [0.0, us])[0] == 0
    np.testing.assert_allclose(_draw_law(p, q, [2], [0.0]), p[0], atol=1e-6)


def test_quotient_edge_cases_and_bad_ids():
    p = np.array([[0.5, 0.5, 0.0], [1.0, 0.0, 0.0]], np.float32)
    q = np.array([[0.0, 0.5, 0.5]], np.float32)
    assert oracle.spec_accept(p, q, [0], [0.999, 0.3])[0] == 1    # q = 0 < p: accepted
    n, tok = oracle.spec_accept(p, q, [2], [0.0, 0.3])             # p = 0 < q: rejected
    assert n == 0 and tok in (0, 1)
    p2 = np.array([[0.5, 0.5, 0.0], [1.0, 0.0, 0.0]], np.float32)
    q2 = np.array([[0.5, 0.5, 0.0]], np.float32)
    n, tok = oracle.spec_accept(p2, q2, [2], [0.0, 0.7])           # p = q = 0: rejected; no residual mass,
    assert n == 0 and tok == 1                                      # so the draw follows p
    assert oracle.spec_accept(p, q, [3], [0.0, 0.3]) == (-1, -1)
    assert oracle.spec_accept(p, q, [-1], [0.0, 0.3]) == (-1, -1)


def test_no_drafts_draws_from_target():
    p = np.array([[0.125, 0.375, 0.5]], np.float32)
    q = np.zeros((0, 3), np.float32)
    assert oracle.spec_accept(p, q, [], [0.2])[0] == 0
    np.testing.assert_allclose(_draw_law(p, q, [], []), p[0], atol=1e-6)


def test_acceptance_rate_matches_closed_form():
    # P(accept draft d) = min(1, p(d)/q(d)); over d ~ q it is sum_v min(p(v), q(v))
    p, q, _, _ = spec_inputs(11, 1, 6, spread=1.0, noise=1.0)
    rate = sum(q[0, d] * _accept_prob(p, q, d) for d in range(6))
    assert rate == pytest.approx(np.minimum(p[0], q[0]).astype(np.float64).sum(), abs=1e-6)
