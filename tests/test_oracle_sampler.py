"""Pins for the oracle's draft/target rejection sampler (CPU only).

The method: alpha_i = min(1, P(x_i)/Q(x_i)) per draft token, the expected
accepted count E[K] = sum_i prod_{j<=i} alpha_j and the speed-up
eta = (E[K]+1)/(gamma r + 1) ("LOW-LATENCY INFERENCE: SPECULATIVE DECODING &
PAGING", section "Verification Acceptance Probabilities and Speedup Math");
on rejection the position is resampled ("Rejection Recovery (Resample)" in
the same page's architecture diagram) so that the emitted tokens follow the
target distribution exactly ("Speculative Decoding and KV-Cache Compression",
section 2.1-2.2).

Pins that do not restate the oracle:
  * Monte-Carlo: the emitted token at every reached position is distributed as
    P at that position (the exactness theorem), chi-square on 10^6 rows at
    V = 8 and 25,000 rows at V = 1000;
  * the mean accepted length equals the page's E[K] formula for fixed drafts,
    and sum_i prod_j (1 - TV(P_j, Q_j)) for drafts drawn from Q;
  * special cases: P == Q always accepts; a draft one-hot on a token the
    target never emits always rejects; a one-hot bonus row is deterministic;
  * the page's worked example alpha >= 0.85, r ~ 0.08 => eta >= 2.8;
  * the tree sampler on a chain equals the linear sampler; on a real tree its
    first emitted token is distributed as P at the root.
"""
import os

import numpy as np
import pytest
from scipy import stats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def fixed_rows(rng, n_rows, V, spread=1.5):
    logits = rng.normal(0, spread, size=(n_rows, V))
    e = np.exp(logits - logits.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def draw_from(rng, probs, n):
    """n draws from each row of probs [R, V] -> [n, R] (independent, numpy RNG)."""
    cdf = np.cumsum(probs.astype(np.float64), axis=-1)
    cdf /= cdf[:, -1:]
    u = rng.random((n, probs.shape[0]))
    return (u[..., None] >= cdf[None, :, :]).sum(-1).astype(np.int32)


def broadcast_rows(rows, B):
    return np.ascontiguousarray(np.broadcast_to(rows, (B,) + rows.shape))


def chi2_ok(tokens, probs, min_p=1e-4):
    V = probs.shape[0]
    obs = np.bincount(tokens, minlength=V).astype(np.float64)
    exp = probs.astype(np.float64) / probs.sum() * obs.sum()
    keep = exp > 5
    obs_k, exp_k = obs[keep], exp[keep]
    exp_k *= obs_k.sum() / exp_k.sum()
    return stats.chisquare(obs_k, exp_k).pvalue > min_p


def test_output_distribution_equals_target(oracle_mod):
    rng = np.random.default_rng(2024)
    gamma, V, B = 3, 8, 1_000_000
    P = fixed_rows(rng, gamma + 1, V)
    Q = fixed_rows(rng, gamma, V)
    x = draw_from(rng, Q, B)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, out, near, _ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    for i in range(gamma + 1):
        reached = k >= i
        assert reached.sum() > 5000
        assert chi2_ok(out[reached, i], P[i]), f"position {i} is not distributed as P_{i}"
    # positions past the emitted ones are -1; accepted positions carry the drafts
    idx = np.arange(gamma + 1)[None, :]
    assert np.all(out[idx > k[:, None]] == -1)
    assert np.all(out[:, :gamma][idx[:, :gamma] < k[:, None]] == x[idx[:, :gamma] < k[:, None]])
    assert np.all(out[idx == k[:, None]] >= 0)


def test_output_distribution_equals_target_large_vocabulary(oracle_mod):
    # V = 1000 (the tiny workload's vocabulary): every reached position is
    # distributed as P there, bins with fewer than 5 expected draws aside
    rng = np.random.default_rng(77)
    gamma, V, B = 3, 1000, 25_000
    P = fixed_rows(rng, gamma + 1, V, spread=1.0)
    Q = fixed_rows(rng, gamma, V, spread=1.0)
    x = draw_from(rng, Q, B)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, out, near, _ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    for i in range(gamma + 1):
        reached = k >= i
        assert reached.sum() > 2000
        assert chi2_ok(out[reached, i], P[i]), f"position {i} is not distributed as P_{i}"


def test_resampling_from_target_instead_of_residual_would_fail(oracle_mod):
    # sanity of the statistic: tokens drawn from P_0 itself at rejected rows
    # (the p3 skeleton's fallback) are visibly biased and fail the same check
    rng = np.random.default_rng(7)
    gamma, V, B = 1, 8, 200_000
    P = fixed_rows(rng, gamma + 1, V)
    Q = fixed_rows(rng, gamma, V)
    x = draw_from(rng, Q, B)[:, 0]
    u = rng.random(B)
    acc = u * Q[0][x] <= P[0][x]
    wrong = np.where(acc, x, draw_from(rng, P[:1], B)[:, 0])
    assert not chi2_ok(wrong, P[0])


def test_mean_accepted_matches_expected_k_fixed_drafts(oracle_mod):
    rng = np.random.default_rng(99)
    gamma, V, B = 5, 16, 400_000
    P = fixed_rows(rng, gamma + 1, V)
    Q = fixed_rows(rng, gamma, V)
    x1 = np.array([int(np.argmax(Q[i])) for i in range(gamma)], np.int32)
    alpha = [min(1.0, float(P[i][x1[i]]) / float(Q[i][x1[i]])) for i in range(gamma)]
    ek = oracle_mod.expected_accepted(alpha)
    closed = sum(np.prod(alpha[:i + 1]) for i in range(gamma))
    assert abs(ek - closed) < 1e-12
    x = np.ascontiguousarray(np.broadcast_to(x1, (B, gamma)))
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, *_ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    se = k.std() / np.sqrt(B)
    assert abs(k.mean() - ek) < 5 * se + 1e-3


def test_mean_accepted_drafts_from_q(oracle_mod):
    rng = np.random.default_rng(5)
    gamma, V, B = 4, 8, 300_000
    P = fixed_rows(rng, gamma + 1, V)
    Q = fixed_rows(rng, gamma, V)
    beta = [float(np.minimum(P[i].astype(np.float64), Q[i]).sum()) for i in range(gamma)]
    ek = sum(np.prod(beta[:i + 1]) for i in range(gamma))
    x = draw_from(rng, Q, B)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, *_ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    assert abs(k.mean() - ek) < 5 * k.std() / np.sqrt(B) + 1e-3


def test_identical_distributions_always_accept(oracle_mod):
    rng = np.random.default_rng(3)
    gamma, V, B = 4, 10, 100_000
    P = fixed_rows(rng, gamma + 1, V)
    Q = P[:gamma].copy()
    x = draw_from(rng, Q, B)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, out, _, _ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    assert np.all(k == gamma)
    assert np.array_equal(out[:, :gamma], x)
    assert chi2_ok(out[:, gamma], P[gamma])


def test_draft_on_impossible_token_always_rejects(oracle_mod):
    rng = np.random.default_rng(4)
    gamma, V, B = 2, 8, 100_000
    P = fixed_rows(rng, gamma + 1, V)
    P[0, 3] = 0.0
    P[0] /= P[0].sum()
    Q = fixed_rows(rng, gamma, V)
    Q[0] = 0.0
    Q[0, 3] = 1.0
    x = draw_from(rng, Q, B)
    assert np.all(x[:, 0] == 3)
    ua = rng.random((B, gamma), dtype=np.float32)
    ua[ua == 0] = 0.5
    us = rng.random(B, dtype=np.float32)
    k, out, _, _ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    assert np.all(k == 0)
    assert np.all(out[:, 0] != 3) and np.all(out[:, 1:] == -1)
    assert chi2_ok(out[:, 0], P[0])


def test_one_hot_bonus_is_deterministic(oracle_mod):
    rng = np.random.default_rng(6)
    gamma, V, B = 3, 12, 1000
    P = fixed_rows(rng, gamma + 1, V)
    P[gamma] = 0.0
    P[gamma, 7] = 1.0
    Q = P[:gamma].copy()
    x = draw_from(rng, Q, B)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, out, _, _ = oracle_mod.spec_accept(broadcast_rows(P, B), broadcast_rows(Q, B), x, ua, us)
    assert np.all(k == gamma) and np.all(out[:, gamma] == 7)


def test_inverse_cdf_strict_threshold_skips_zero_mass(oracle_mod):
    # the draw is the first token whose running sum exceeds u*S: a token with
    # zero mass is never chosen, even at u = 0
    P = np.zeros((1, 2, 6), np.float32)
    P[0, 1] = [0.0, 0.25, 0.0, 0.25, 0.5, 0.0]
    P[0, 0] = [0, 0, 1, 0, 0, 0]
    Q = P[:, :1].copy()
    x = np.array([[2]], np.int32)
    for u, expect in [(0.0, 1), (0.2499, 1), (0.25, 3), (0.5, 4), (0.9999, 4)]:
        k, out, _, _ = oracle_mod.spec_accept(P, Q, x, np.array([[0.5]], np.float32),
                                              np.array([u], np.float32))
        assert k[0] == 1 and out[0, 1] == expect, (u, out)


def test_accept_comparison_is_fp32_product_le(oracle_mod):
    # accept iff fp32(u*Q) <= P: equality accepts
    P = np.zeros((1, 2, 4), np.float32)
    Q = np.zeros((1, 1, 4), np.float32)
    P[0, 0] = [0.25, 0.25, 0.25, 0.25]
    P[0, 1] = [1, 0, 0, 0]
    Q[0, 0] = [0.5, 0.5, 0.0, 0.0]
    x = np.array([[0]], np.int32)
    k, *_ = oracle_mod.spec_accept(P, Q, x, np.array([[0.5]], np.float32), np.array([0.1], np.float32))
    assert k[0] == 1
    k, *_ = oracle_mod.spec_accept(P, Q, x, np.array([[np.nextafter(np.float32(0.5), np.float32(1))]], np.float32),
                                   np.array([0.1], np.float32))
    assert k[0] == 0


def test_eta_worked_example(oracle_mod):
    rows = [l.split() for l in open(os.path.join(GOLDEN, "eta_worked_example.txt"))
            if l.strip() and not l.startswith("#")]
    alpha, r, gamma, bound = float(rows[0][0]), float(rows[0][1]), int(rows[0][2]), float(rows[0][3])
    ek = oracle_mod.expected_accepted([alpha] * gamma)
    # closed form of the geometric series sum_{i=1}^{g} a^i
    assert abs(ek - alpha * (1 - alpha ** gamma) / (1 - alpha)) < 1e-12
    eta = oracle_mod.speedup(ek, gamma, r)
    assert eta >= bound
    assert abs(eta - (ek + 1) / (gamma * r + 1)) < 1e-15
    # the bound is tight-ish: gamma = 3 would not reach it
    assert oracle_mod.speedup(oracle_mod.expected_accepted([alpha] * 3), 3, r) < bound


def chain_inputs(rng, B, gamma, V):
    P = rng.dirichlet(np.ones(V), size=(B, gamma + 1)).astype(np.float32)
    Q = rng.dirichlet(np.ones(V), size=(B, gamma)).astype(np.float32)
    x = np.stack([draw_from(rng, Q[b], 1)[0] for b in range(B)]).astype(np.int32)
    ua = rng.random((B, gamma), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    return P, Q, x, ua, us


def test_tree_chain_equals_linear(oracle_mod):
    rng = np.random.default_rng(12)
    B, gamma, V = 500, 4, 50
    P, Q, x, ua, us = chain_inputs(rng, B, gamma, V)
    k, out, _, _ = oracle_mod.spec_accept(P, Q, x, ua, us)
    parent = np.array([-1, 0, 1, 2, 3], np.int32)
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    ua_t = np.concatenate([np.zeros((B, 1), np.float32), ua], axis=1)
    kt, path, outt, _ = oracle_mod.spec_accept_tree(parent, P, Q, tok, ua_t, us)
    assert np.array_equal(k, kt)
    assert np.array_equal(out, outt)
    for b in range(B):
        assert list(path[b, :k[b] + 1]) == list(range(k[b] + 1))
        assert np.all(path[b, k[b] + 1:] == -1)


def test_tree_first_token_distribution(oracle_mod):
    rng = np.random.default_rng(31)
    B, V = 200_000, 6
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32)   # branching 3-2
    n = parent.shape[0]
    internal = [0, 1, 2, 3]
    Prow = fixed_rows(rng, n, V, spread=1.2)
    Qrow = fixed_rows(rng, len(internal), V, spread=1.2)
    tok = np.zeros((B, n), np.int32)
    for c in range(1, n):
        tok[:, c] = draw_from(rng, Qrow[internal.index(parent[c])][None], B)[:, 0]
    ua = rng.random((B, n), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    k, path, out, near = oracle_mod.spec_accept_tree(parent, broadcast_rows(Prow, B),
                                                     broadcast_rows(Qrow, B), tok, ua, us)
    assert chi2_ok(out[:, 0], Prow[0])
    # given that node 1 was accepted, the next token follows P at node 1
    sel = path[:, 1] == 1
    assert sel.sum() > 5000 and chi2_ok(out[sel, 1], Prow[1])
    # path consistency: each accepted node is a child of the previous one, and
    # its token is the emitted one
    for b in range(2000):
        for d in range(1, k[b] + 1):
            assert parent[path[b, d]] == path[b, d - 1]
            assert out[b, d - 1] == tok[b, path[b, d]]
    assert near.mean() < 1e-3
