"""Pins for the oracle's draft-tree sampler fed by logits (CPU only).

The target scores every node of a draft tree in one pass ("The Sub-Millisecond
Speculative Decoding Meltdown", tree attention) and each draft token's
acceptance ratio takes softmax(logits)[x] ("Speculative Decoding and KV-Cache
Compression", section 2.3).  At a node the children are tested in index order
against the residual left by the siblings rejected before them.

Pins that do not restate the oracle:
  * examples worked by hand on three tokens with -inf masking, where the
    probabilities are small fractions: a later child is tested as
    u * Q(x) * Z <= R(x) (dropping Z decides the other way), and the draw
    after every child is rejected comes from the twice-reduced residual
    (7/45, 0, 0) -- not from P, not from the once-reduced residual and not
    from a residual reduced by Q instead of Z Q;
  * on a chain the sampler is the linear sampler fed by logits (pinned on its
    own), with separate target and draft temperatures;
  * on a real tree it makes the decisions of the probability-input tree
    sampler (pinned on its own) on the softmax rows wherever neither flags a
    near-boundary case;
  * temperature identity: logits doubled at temperature 2 give every output
    bit for bit;
  * Monte-Carlo at V = 8: the first emitted token follows P at the root, and
    given that node 1 was accepted the next one follows P at node 1;
  * the outcome sets: with a zero band they hold exactly the oracle's own end
    node and token; with a band of 1 every node and every token; with the
    default band they hold the oracle's outcome.
"""
import numpy as np
import pytest
from scipy import stats

NEG = -np.inf


def tree_inputs(rng, parent, B, V, sigma=1.0, sigma_d=0.5, T=1.0, Td=1.0):
    """Logits N(0, sigma) per node, drafts = parent's logits + N(0, sigma_d),
    each child's token drawn from its parent's draft softmax."""
    n = len(parent)
    internal = [i for i in range(n) if i in set(parent[1:])]
    lp = rng.normal(0, sigma, (B, n, V)).astype(np.float32)
    lq = (lp[:, internal, :] + rng.normal(0, sigma_d, (B, len(internal), V))).astype(np.float32)
    q = np.exp(lq.astype(np.float64) / Td - (lq.astype(np.float64) / Td).max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    tok = np.zeros((B, n), np.int32)
    cdf = np.cumsum(q, -1)
    for c in range(1, n):
        r = internal.index(parent[c])
        u = rng.random((B, 1))
        tok[:, c] = np.minimum((u >= cdf[:, r, :]).sum(-1), V - 1)
    ua = rng.random((B, n)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    return lp, lq, tok, ua, us


def run(o, parent, lp, lq, tok, ua, us, **kw):
    f = lambda a, t: np.ascontiguousarray(np.asarray(a, dtype=t))
    return o.spec_accept_tree_logits(f(parent, np.int32), f(lp, np.float32), f(lq, np.float32), f(tok, np.int32),
                                     f(ua, np.float32), f(us, np.float32), **kw)


# root with two leaf children: node 0 -> nodes 1, 2
PARENT2 = [-1, 0, 0]


def test_worked_later_child_uses_scaled_residual(oracle_mod):
    # root P = softmax(0, 0, -inf) = (1/2, 1/2, 0); Q = softmax(0, 0, 0) = (1/3, 1/3, 1/3)
    # child 1 drafts token 2: u Q(2) = u/3 > P(2) = 0: rejected for any u > 0;
    #   R = max(0, P - Q) = (1/6, 1/6, 0), Z = 1/3
    # child 2 drafts token 0: u Q(0) Z = u/9 <= R(0) = 1/6 for every u <= 1:
    #   accepted (without the Z factor, u Q(0) <= R(0) would reject u > 1/2)
    # node 2 is a leaf: the bonus comes from its P = softmax(-inf, 0, -inf): token 1
    lp = np.array([[[0, 0, NEG], [0, NEG, NEG], [NEG, 0, NEG]]])
    lq = np.array([[[0, 0, 0]]])
    for u2 in (0.6, 0.9, 0.999):
        k, path, out, near = run(oracle_mod, PARENT2, lp, lq, [[0, 2, 0]], [[0, 0.5, u2]], [0.5])
        assert k[0] == 1 and path[0].tolist() == [0, 2] and out[0].tolist() == [0, 1] and not near[0]


def test_worked_draw_after_all_children_rejected(oracle_mod):
    # Q = (1/3, 1/3, 1/3) and both children draft token 2, which the target
    # never emits: both are rejected.
    lq = np.array([[[0, 0, 0]]])
    ln2, ln3 = float(np.log(2.0)), float(np.log(3.0))
    # root P = softmax(0, ln 2, -inf) = (1/3, 2/3, 0):
    #   after child 1: R = (0, 1/3, 0), Z = 1/3
    #   after child 2: R = max(0, R - Z Q) = (0, 1/3 - 1/9, 0) = (0, 2/9, 0)
    # every draw is token 1 (a draw from P would give token 0 for u_s < 1/3)
    lp = np.array([[[0, ln2, NEG], [0, 0, 0], [0, 0, 0]]])
    for us in (0.05, 0.3, 0.9):
        k, path, out, near = run(oracle_mod, PARENT2, lp, lq, [[0, 2, 2]], [[0, 0.5, 0.5]], [us])
        assert k[0] == 0 and path[0].tolist() == [0, -1] and out[0].tolist() == [1, -1] and not near[0]
    # root P = softmax(ln 3, ln 2, -inf) = (3/5, 2/5, 0):
    #   after child 1: R = (3/5 - 1/3, 2/5 - 1/3, 0) = (4/15, 1/15, 0), Z = 1/3
    #   after child 2: R = (4/15 - 1/9, 1/15 - 1/9 -> 0, 0) = (7/45, 0, 0)
    # every draw is token 0; at u_s = 0.9 a draw from the once-reduced residual
    # (4/15, 1/15) or from P would give token 1, and so would a residual
    # reduced by Q instead of Z Q (empty after child 2, so P is drawn from)
    lp = np.array([[[ln3, ln2, NEG], [0, 0, 0], [0, 0, 0]]])
    for us in (0.05, 0.5, 0.9):
        k, path, out, near = run(oracle_mod, PARENT2, lp, lq, [[0, 2, 2]], [[0, 0.5, 0.5]], [us])
        assert k[0] == 0 and out[0].tolist() == [0, -1] and not near[0]


def test_worked_first_child_and_bonus(oracle_mod):
    # root P = softmax(ln 2, 0, 0) = (1/2, 1/4, 1/4); Q = softmax(0, ln 2, ln 2) =
    # (1/5, 2/5, 2/5); child 1 drafts token 1, child 2 token 2.
    # u_1 = 0.5: 0.5 * 2/5 = 1/5 <= 1/4: child 1 accepted; it is a leaf whose
    #   P = softmax(-inf, -inf, 0) gives the bonus token 2.
    # u_1 = 1: 2/5 > 1/4: rejected; R = (3/10, 0, 0), Z = 3/10; child 2:
    #   u Q(2) Z = 0.12 > R(2) = 0: rejected; the draw is token 0.
    ln2 = float(np.log(2.0))
    lp = np.array([[[ln2, 0, 0], [NEG, NEG, 0], [0, NEG, NEG]]])
    lq = np.array([[[0, ln2, ln2]]])
    k, path, out, _ = run(oracle_mod, PARENT2, lp, lq, [[0, 1, 2]], [[0, 0.5, 1.0]], [0.7])
    assert k[0] == 1 and path[0].tolist() == [0, 1] and out[0].tolist() == [1, 2]
    k, path, out, _ = run(oracle_mod, PARENT2, lp, lq, [[0, 1, 2]], [[0, 1.0, 1.0]], [0.7])
    assert k[0] == 0 and path[0].tolist() == [0, -1] and out[0].tolist() == [0, -1]


@pytest.mark.parametrize("T,Td", [(1.0, 1.0), (0.8, 1.3)])
def test_chain_equals_linear_logits_sampler(oracle_mod, T, Td):
    rng = np.random.default_rng(41)
    B, gamma, V = 400, 4, 300
    parent = [-1, 0, 1, 2, 3]
    lp, lq, tok, ua, us = tree_inputs(rng, parent, B, V, T=T, Td=Td)
    k, out, _ = oracle_mod.spec_accept_logits(lp, lq, np.ascontiguousarray(tok[:, 1:]),
                                              np.ascontiguousarray(ua[:, 1:]), us, temperature=T,
                                              draft_temperature=Td)
    kt, path, outt, _ = run(oracle_mod, parent, lp, lq, tok, ua, us, temperature=T, draft_temperature=Td)
    assert np.array_equal(k, kt)
    assert np.array_equal(out, outt)
    for b in range(B):
        assert path[b, :k[b] + 1].tolist() == list(range(k[b] + 1))
        assert np.all(path[b, k[b] + 1:] == -1)
    assert 0 < k.mean() < gamma


def test_agrees_with_probability_tree_sampler(oracle_mod):
    rng = np.random.default_rng(42)
    parent = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 5]
    B, V = 600, 500
    T, Td = 0.9, 1.1
    lp, lq, tok, ua, us = tree_inputs(rng, parent, B, V, T=T, Td=Td)
    sm = lambda l, t: np.exp(l / t - (l / t).max(-1, keepdims=True)) / np.exp(
        l / t - (l / t).max(-1, keepdims=True)).sum(-1, keepdims=True)
    P = sm(lp.astype(np.float64), T).astype(np.float32)
    Q = sm(lq.astype(np.float64), Td).astype(np.float32)
    k1, p1, o1, n1 = oracle_mod.spec_accept_tree(np.array(parent, np.int32), P, Q, tok, ua, us)
    # the probability rows differ from the fp64 softmax by fp32 rounding
    # alone (~1e-7 relative), so a band of 1e-6 covers the difference
    k2, p2, o2, n2 = run(oracle_mod, parent, lp, lq, tok, ua, us, temperature=T, draft_temperature=Td, band=1e-6)
    ok = ~(n1 | n2)
    assert ok.mean() > 0.95
    assert np.array_equal(k1[ok], k2[ok])
    assert np.array_equal(p1[ok], p2[ok])
    assert np.array_equal(o1[ok], o2[ok])
    assert len(set(k2.tolist())) >= 3  # several depths reached


def test_doubled_logits_at_temperature_two_are_identical(oracle_mod):
    rng = np.random.default_rng(43)
    parent = [-1, 0, 0, 1, 1, 2]
    lp, lq, tok, ua, us = tree_inputs(rng, parent, 300, 200)
    a = run(oracle_mod, parent, lp, lq, tok, ua, us)
    b = run(oracle_mod, parent, lp * 2, lq * 2, tok, ua, us, temperature=2.0)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def chi2_ok(tokens, probs):
    obs = np.bincount(tokens, minlength=probs.shape[0]).astype(np.float64)
    return stats.chisquare(obs, probs / probs.sum() * obs.sum()).pvalue > 1e-4


def test_emitted_tokens_follow_the_target(oracle_mod):
    rng = np.random.default_rng(44)
    parent = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]
    n, V, B = len(parent), 8, 200_000
    internal = [0, 1, 2, 3]
    lp1 = rng.normal(0, 1.2, (n, V))
    lq1 = lp1[internal] + rng.normal(0, 0.8, (len(internal), V))
    T, Td = 0.9, 1.2
    P = np.exp(lp1 / T) / np.exp(lp1 / T).sum(-1, keepdims=True)
    Q = np.exp(lq1 / Td) / np.exp(lq1 / Td).sum(-1, keepdims=True)
    tok = np.zeros((B, n), np.int32)
    for c in range(1, n):
        cdf = np.cumsum(Q[internal.index(parent[c])])
        tok[:, c] = np.minimum((rng.random((B, 1)) >= cdf[None, :]).sum(-1), V - 1)
    ua = rng.random((B, n)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    lp = np.ascontiguousarray(np.broadcast_to(lp1.astype(np.float32), (B, n, V)))
    lq = np.ascontiguousarray(np.broadcast_to(lq1.astype(np.float32), (B, len(internal), V)))
    k, path, out, near = run(oracle_mod, parent, lp, lq, tok, ua, us, temperature=T, draft_temperature=Td)
    assert chi2_ok(out[:, 0], P[0])
    sel = path[:, 1] == 1
    assert sel.sum() > 5000 and chi2_ok(out[sel, 1], P[1])
    # near flags: draws within the band of a running sum (at most ~2 band V / Z
    # of them) and tests within it
    assert near.mean() < 0.03


def test_outcome_sets(oracle_mod):
    rng = np.random.default_rng(45)
    parent = np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3, 4, 6], np.int32)
    n = len(parent)
    B, V = 300, 400
    lp, lq, tok, ua, us = tree_inputs(rng, parent.tolist(), B, V)
    k, path, out, near = run(oracle_mod, parent, lp, lq, tok, ua, us)
    end = path[np.arange(B), k]
    drawn = out[np.arange(B), k]
    ok0, lo0, hi0 = oracle_mod.tree_logits_outcomes(parent, lp, lq, tok, ua, us, band=0.0)
    assert np.array_equal(ok0.sum(1), np.ones(B))
    assert np.all(ok0[np.arange(B), end])
    assert np.array_equal(lo0[np.arange(B), end], drawn) and np.array_equal(hi0[np.arange(B), end], drawn)
    okd, lod, hid = oracle_mod.tree_logits_outcomes(parent, lp, lq, tok, ua, us)
    assert np.all(okd[np.arange(B), end])
    assert np.all((lod[np.arange(B), end] <= drawn) & (drawn <= hid[np.arange(B), end]))
    assert np.all(okd >= ok0)
    ok1, lo1, hi1 = oracle_mod.tree_logits_outcomes(parent, lp, lq, tok, ua, us, band=1.0)
    assert np.all(ok1) and np.all(lo1 == 0) and np.all(hi1 == V - 1)
    assert np.all(okd.sum(1) < n)  # the default band rules most outcomes out


def test_invalid_inputs_raise(oracle_mod):
    lp = np.zeros((1, 3, 4), np.float32)
    lq = np.zeros((1, 1, 4), np.float32)
    with pytest.raises(oracle_mod.OracleError):
        run(oracle_mod, [-1, 0, 0], lp, lq, [[0, 4, 0]], [[0, 0.5, 0.5]], [0.5])  # token out of range
    with pytest.raises(oracle_mod.OracleError):
        run(oracle_mod, [-1, 1, 0], lp, lq, [[0, 1, 1]], [[0, 0.5, 0.5]], [0.5])  # parent after child
    bad = lp.copy()
    bad[0, 0, :] = NEG  # the root's target row has no finite logit
    with pytest.raises(oracle_mod.OracleError):
        run(oracle_mod, [-1, 0, 0], bad, lq, [[0, 1, 1]], [[0, 0.5, 0.5]], [0.5])
