"""Pins for the oracle's sampler front-end that forms P and Q from logits (CPU only).

The target pass produces logits and each draft token's acceptance ratio takes
softmax(logits)[x] ("Speculative Decoding and KV-Cache Compression", section
2.3; "LOW-LATENCY INFERENCE: SPECULATIVE DECODING & PAGING", architecture:
target logits checked against draft logits).  Sampling temperatures divide the
logits, the target's and the draft's each on its own.

Pins that do not restate the oracle:
  * a two-token example worked by hand: P = (1/4, 3/4), Q = (3/4, 1/4), so
    draft token 0 is accepted iff u <= 1/3 and its correction is always token
    1; the same with a temperature of 2 on doubled logits;
  * softmax shift invariance, checked bit for bit on a shift of 4096 (exact
    in fp32 here) that would overflow exp() without the max subtracted;
  * on the same rows, the probability-input sampler (pinned on its own)
    makes the same decisions wherever neither flags a near-boundary case,
    and its every draw lies in the draw window (fixed cases, and 150 random
    shapes with temperatures and masked tokens);
  * the draw window of a worked example, and its definition (the running
    sums within the band) checked with numpy on larger rows;
  * Monte-Carlo: with drafts drawn from Q, the emitted tokens follow P at
    positions 0 and 1, the mean first acceptance is 1 - TV(P, Q), and masked
    (-inf) target tokens are never emitted;
  * special cases: V = 1; an exact tie u Q = P is accepted and flagged; a draw
    exactly on a boundary is flagged; invalid rows raise;
  * the band itself: an emulation of the fp32 formation at V = 128256 errs by
    well under half of it.
"""
import numpy as np
import pytest
from scipy import stats

LN3 = float(np.log(3.0))


def softmax64(l, T=1.0):
    x = l.astype(np.float64) / T
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def draw_rows(rng, probs):
    """One draw from each row of probs [R, V] (numpy RNG, inverse CDF)."""
    cdf = np.cumsum(probs, axis=-1)
    cdf /= cdf[:, -1:]
    u = rng.random((probs.shape[0], 1))
    return np.minimum((u >= cdf).sum(-1), probs.shape[1] - 1).astype(np.int32)


def run(o, lp, lq, x, ua, us, **kw):
    f = lambda a, t: np.ascontiguousarray(np.asarray(a, dtype=t))
    return o.spec_accept_logits(f(lp, np.float32), f(lq, np.float32), f(x, np.int32), f(ua, np.float32),
                                f(us, np.float32), **kw)


@pytest.mark.parametrize("T", [1.0, 2.0])
def test_two_token_worked_example(oracle_mod, T):
    # target logits (0, ln 3) -> P = (1/4, 3/4); draft (ln 3, 0) -> Q = (3/4, 1/4)
    lp = np.array([[[0.0, LN3 * T], [0.0, LN3 * T]]])
    lq = np.array([[[LN3 * T, 0.0]]])
    for u, want_k in ((0.30, 1), (0.333, 1), (0.334, 0), (0.9, 0)):
        for us, bonus in ((0.2, 0), (0.3, 1)):
            k, toks, near = run(oracle_mod, lp, lq, [[0]], [[u]], [us], temperature=T)
            assert k[0] == want_k
            if want_k == 1:  # accepted: bonus from P_1 = (1/4, 3/4): token 0 iff u_s < 1/4
                assert toks[0].tolist() == [0, bonus]
            else:  # rejected: residual max(0, P - Q) = (0, 1/2) -> token 1 whatever u_s
                assert toks[0].tolist() == [1, -1]
            assert not near[0]


def test_draft_temperature_is_its_own(oracle_mod):
    # draft logits (3 ln 3, 0) at draft temperature 3 -> Q = (3/4, 1/4) again;
    # at the target's temperature 1 the draft would be (27/28, 1/28) and
    # u = 0.3 would be rejected (0.3 * 27/28 > 1/4)
    lp = np.array([[[0.0, LN3], [0.0, LN3]]])
    lq = np.array([[[3 * LN3, 0.0]]])
    k, _, _ = run(oracle_mod, lp, lq, [[0]], [[0.3]], [0.5], temperature=1.0, draft_temperature=3.0)
    assert k[0] == 1
    k, _, _ = run(oracle_mod, lp, lq, [[0]], [[0.3]], [0.5], temperature=1.0)
    assert k[0] == 0


def test_shift_invariance_bit_exact(oracle_mod):
    rng = np.random.default_rng(3)
    B, g, V = 64, 3, 300
    # multiples of 2^-10 within +-16: exact after adding 4096 in fp32
    lp = np.round(rng.normal(0, 3, (B, g + 1, V)).clip(-15, 15) * 1024) / 1024
    lq = np.round((lp[:, :g] + rng.normal(0, 0.5, (B, g, V))).clip(-15, 15) * 1024) / 1024
    x = draw_rows(rng, softmax64(lq).reshape(-1, V)).reshape(B, g)
    ua, us = rng.random((B, g)), rng.random(B)
    a = run(oracle_mod, lp, lq, x, ua, us, temperature=0.8)
    sp = (4096.0 * rng.integers(-1, 2, (B, g + 1, 1))).astype(np.float64)
    sq = (4096.0 * rng.integers(-1, 2, (B, g, 1))).astype(np.float64)
    assert np.array_equal((lp + sp).astype(np.float32) - sp.astype(np.float32), lp.astype(np.float32))
    b = run(oracle_mod, lp + sp, lq + sq, x, ua, us, temperature=0.8)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


@pytest.mark.parametrize("T,Td", [(1.0, 1.0), (0.7, 0.7), (1.3, 0.5)])
def test_agrees_with_probability_sampler(oracle_mod, T, Td):
    rng = np.random.default_rng(11)
    B, g, V = 400, 4, 1000
    lp = rng.normal(0, 3, (B, g + 1, V)).astype(np.float32)
    lq = (lp[:, :g] + rng.normal(0, 0.7, (B, g, V))).astype(np.float32)
    P = softmax64(lp, T)
    Q = softmax64(lq, Td)
    x = draw_rows(rng, Q.reshape(-1, V)).reshape(B, g)
    ua, us = rng.random((B, g)).astype(np.float32), rng.random(B).astype(np.float32)
    # the probability sampler sees P and Q rounded to fp32 (~6e-8 relative), so a
    # band of 1e-6 covers the difference; the window check covers every row
    k1, t1, n1 = run(oracle_mod, lp, lq, x, ua, us, temperature=T, draft_temperature=Td, band=1e-6)
    k2, t2, n2, _ = oracle_mod.spec_accept(P.astype(np.float32), Q.astype(np.float32), x, ua, us)
    ok = ~(n1 | n2)
    assert ok.sum() >= 0.95 * B
    assert np.array_equal(k1[ok], k2[ok])
    assert np.array_equal(t1[ok], t2[ok])
    lo, hi = oracle_mod.logits_draw_window(lp, lq, k2, us, temperature=T, draft_temperature=Td, band=1e-6)
    drawn = t2[np.arange(B), k2]
    assert np.all((lo <= drawn) & (drawn <= hi))


def test_draw_window_worked_example(oracle_mod):
    # rejected at k = 0: residual (0, 1/2), Z = 1/2; accepted: P_1 = (1/4, 3/4)
    lp = np.array([[[0.0, LN3], [0.0, LN3]]] * 3)
    lq = np.array([[[LN3, 0.0]]] * 3)
    k = np.array([0, 1, 1], np.int32)
    us = np.array([0.5, 0.1, 0.2499], np.float32)
    f = lambda a: np.asarray(a, np.float32)
    lo, hi = oracle_mod.logits_draw_window(f(lp), f(lq), k, us, band=1e-3)
    assert lo.tolist() == [1, 0, 0] and hi.tolist() == [1, 0, 1]
    lo, hi = oracle_mod.logits_draw_window(f(lp), f(lq), k, us, band=0.0)
    assert lo.tolist() == [1, 0, 0] and hi.tolist() == [1, 0, 0]


def test_draw_window_holds_the_exact_draw(oracle_mod):
    rng = np.random.default_rng(17)
    B, g, V = 300, 3, 5000
    lp = rng.normal(0, 3, (B, g + 1, V)).astype(np.float32)
    lq = (lp[:, :g] + rng.normal(0, 0.5, (B, g, V))).astype(np.float32)
    x = draw_rows(rng, softmax64(lq).reshape(-1, V)).reshape(B, g)
    ua, us = rng.random((B, g)), rng.random(B)
    k, toks, near, acc, accn = run(oracle_mod, lp, lq, x, ua, us, tests=True)
    drawn = toks[np.arange(B), k]
    lo, hi = oracle_mod.logits_draw_window(lp, lq, k, us.astype(np.float32))
    assert np.all((lo <= drawn) & (drawn <= hi))
    # a window spans only the tokens whose running sums lie within the band
    P = softmax64(lp)
    Q = softmax64(lq)
    for b in range(0, B, 37):
        r = np.maximum(P[b, k[b]] - Q[b, k[b]], 0) if k[b] < g else P[b, g]
        C = np.cumsum(r)
        t = np.float32(us[b]) * C[-1]
        assert C[lo[b]] >= t - 5e-5 - 1e-12 and (lo[b] == 0 or C[lo[b] - 1] < t - 5e-5 + 1e-12)
        assert hi[b] == V - 1 or (C[hi[b]] > t + 5e-5 - 1e-12 and C[hi[b] - 1] <= t + 5e-5 + 1e-12)
    # the per-test decisions: accepted before k, rejected at k
    for b in range(B):
        assert acc[b, :k[b]].all()
        if k[b] < g:
            assert not acc[b, k[b]]


def test_monte_carlo_output_follows_target(oracle_mod):
    rng = np.random.default_rng(5)
    V, g, B, T, Td = 8, 2, 400_000, 0.8, 1.2
    lp1 = rng.normal(0, 1.5, (g + 1, V))
    lp1[0, 6] = -np.inf  # masked: never emitted at position 0
    lq1 = lp1[:g] + rng.normal(0, 0.8, (g, V))
    lq1[0, 6] = 0.5      # ... although the draft proposes it
    P, Q = softmax64(lp1, T), softmax64(lq1, Td)
    lp = np.broadcast_to(lp1, (B, g + 1, V))
    lq = np.broadcast_to(lq1, (B, g, V))
    x = np.stack([draw_rows(rng, np.broadcast_to(Q[i], (B, V))) for i in range(g)], 1)
    ua, us = rng.random((B, g)), rng.random(B)
    k, toks, near = run(oracle_mod, lp, lq, x, ua, us, temperature=T, draft_temperature=Td)
    assert not (toks[:, 0] == 6).any()
    for pos, sel in ((0, np.ones(B, bool)), (1, k >= 1)):
        obs = np.bincount(toks[sel, pos], minlength=V).astype(np.float64)
        keep = P[pos] > 0
        exp = P[pos][keep] * obs[keep].sum()
        assert stats.chisquare(obs[keep], exp).pvalue > 1e-4, pos
    # first acceptance probability sum_x min(P, Q) = 1 - TV(P_0, Q_0)
    acc0 = np.minimum(P[0], Q[0]).sum()
    se = np.sqrt(acc0 * (1 - acc0) / B)
    assert abs((k >= 1).mean() - acc0) < 5 * se
    assert near.mean() < 1e-3


def test_vocabulary_of_one(oracle_mod):
    k, toks, near = run(oracle_mod, [[[2.0], [-1.0]]], [[[5.0]]], [[0]], [[0.99]], [0.7])
    assert k[0] == 1 and toks[0].tolist() == [0, 0]


def test_exact_tie_is_accepted_and_flagged(oracle_mod):
    # P = (1/2, 1/2), Q = (1, 0) with the second draft token masked: u Q(0) = 1/2 = P(0)
    lp = np.zeros((1, 2, 2))
    lq = np.array([[[0.0, -np.inf]]])
    k, _, near = run(oracle_mod, lp, lq, [[0]], [[0.5]], [0.9])
    assert k[0] == 1 and near[0]


def test_draw_on_a_boundary_is_flagged(oracle_mod):
    # every draft accepted (P == Q), bonus row (1/2, 1/2), u_s = 1/2 exactly:
    # the strict rule picks token 1, and the draw is flagged
    lp = np.zeros((1, 2, 2))
    lq = np.zeros((1, 1, 2))
    k, toks, near = run(oracle_mod, lp, lq, [[1]], [[0.5]], [0.5])
    assert k[0] == 1 and toks[0].tolist() == [1, 1] and near[0]
    k, toks, near = run(oracle_mod, lp, lq, [[1]], [[0.5]], [0.25])
    assert toks[0].tolist() == [1, 0] and not near[0]


@pytest.mark.parametrize("bad", ["nan", "posinf", "all_masked", "token", "temperature"])
def test_invalid_inputs_raise(oracle_mod, bad):
    lp = np.zeros((2, 2, 4))
    lq = np.zeros((2, 1, 4))
    x = np.zeros((2, 1), np.int32)
    T = 1.0
    if bad == "nan":
        lp[1, 0, 2] = np.nan
    elif bad == "posinf":
        lq[0, 0, 1] = np.inf
    elif bad == "all_masked":
        lp[1, 1, :] = -np.inf
    elif bad == "token":
        x[1, 0] = 4
    else:
        T = 0.0
    with pytest.raises(oracle_mod.OracleError):
        run(oracle_mod, lp, lq, x, np.full((2, 1), 0.5), np.full(2, 0.5), temperature=T)


def _fp32_formation(l, T, rng):
    """P formed the way the GPU front-end forms it, emulated in numpy fp32:
    per 16 logits the max, then 2^((l - m) c) (exp2 perturbed by up to two
    units in the last place, the hardware approximation's bound) summed as a
    tree; groups merged in fp32 within a 4096-token slab; slabs merged with
    the rescaled sums in fp64; P = 2^((l - m) c) * fp32(1 / S)."""
    f32 = np.float32
    c = f32(np.log2(np.e) / T)

    def ex2(x):
        y = np.exp2(x.astype(f32)).astype(f32)
        return (y * (1 + rng.uniform(-2, 2, y.shape) * 2.0 ** -23)).astype(f32)

    V = l.shape[0]
    pad = (-V) % 4096
    lp = np.concatenate([l.astype(f32), np.full(pad, -np.inf, f32)])
    g = lp.reshape(-1, 16)
    gm = g.max(1)
    fin = gm > -np.inf  # an all -inf group adds nothing (the kernel skips it)
    ge = np.zeros_like(g)
    ge[fin] = ex2((g[fin] - gm[fin, None]) * c)
    while ge.shape[1] > 1:  # tree sum of the sixteen terms
        ge = (ge[:, 0::2] + ge[:, 1::2]).astype(f32)
    gs = ge[:, 0]

    def scale(mi, mm):  # 2^((mi - mm) c), 0 for an empty part
        out = np.zeros(mi.shape, f32)
        ok = mi > -np.inf
        out[ok] = ex2((mi[ok] - mm[ok]) * c)
        return out

    # groups -> slab, merged in fp32 pairwise (butterfly and warp order differ
    # in order only)
    m, s = gm.reshape(-1, 256), gs.reshape(-1, 256)
    while m.shape[1] > 1:
        m1, m2, s1, s2 = m[:, 0::2], m[:, 1::2], s[:, 0::2], s[:, 1::2]
        mm = np.maximum(m1, m2)
        s = (s1 * scale(m1, mm) + s2 * scale(m2, mm)).astype(f32)
        m = mm
    sm, ss = m[:, 0], s[:, 0]
    M = sm.max()
    S = float(np.sum(ss.astype(np.float64) * scale(sm, np.full_like(sm, M)).astype(np.float64)))
    return (ex2((l.astype(f32) - M) * c) * f32(1.0 / S)).astype(f32)


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_band_covers_fp32_formation(T):
    """The 5e-5 band against an emulation of the fp32 formation at V = 128256:
    the relative error of P over entries down to 2^-100 (the acceptance
    test's) and the absolute error of the residual's running sums (the
    draw's) must stay well inside it."""
    rng = np.random.default_rng(29)
    V = 128256
    worst_rel, worst_cdf = 0.0, 0.0
    for _ in range(6):
        lp = (rng.standard_normal(V) * 3).astype(np.float32)
        lq = (lp + rng.standard_normal(V) * 0.5).astype(np.float32)
        P32, Q32 = _fp32_formation(lp, T, rng), _fp32_formation(lq, T, rng)
        P64, Q64 = softmax64(lp, T), softmax64(lq, T)
        sig = P64 > 2.0 ** -100
        rel = float(np.max(np.abs(P32[sig] - P64[sig]) / P64[sig]))
        r32 = np.maximum(P32.astype(np.float64) - Q32, 0)
        r64 = np.maximum(P64 - Q64, 0)
        cdf = float(np.max(np.abs(np.cumsum(r32) - np.cumsum(r64))))
        assert np.isfinite(rel) and np.isfinite(cdf)
        worst_rel, worst_cdf = max(worst_rel, rel), max(worst_cdf, cdf)
    # an acceptance test compares P with u Q: both errors add
    assert 0 < worst_rel and 2 * worst_rel < 5e-5 / 2, worst_rel
    assert 0 < worst_cdf < 5e-5 / 10, worst_cdf


def test_agrees_with_probability_sampler_on_random_shapes(oracle_mod):
    """Property form of the agreement pin: random vocabularies (1..60), draft
    lengths (1..6), temperatures and masked tokens; wherever neither sampler
    flags a near decision they agree, and every draw of the probability
    sampler lies in the logits oracle's window."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=150, deadline=None, derandomize=True)
    @hyp.given(V=st.integers(1, 60), g=st.integers(1, 6), B=st.integers(1, 24),
               T=st.floats(0.3, 3.0), Td=st.floats(0.3, 3.0), seed=st.integers(0, 2**31 - 1),
               mask=st.booleans())
    def check(V, g, B, T, Td, seed, mask):
        rng = np.random.default_rng(seed)
        lp = rng.normal(0, 2, (B, g + 1, V)).astype(np.float32)
        lq = (lp[:, :g] + rng.normal(0, 0.7, (B, g, V))).astype(np.float32)
        if mask and V > 1:  # mask one target token per row (never the whole row)
            lp[np.arange(B)[:, None], np.arange(g + 1)[None, :], rng.integers(0, V, (B, g + 1))] = -np.inf
        P, Q = softmax64(lp, T), softmax64(lq, Td)
        x = draw_rows(rng, Q.reshape(-1, V)).reshape(B, g)
        ua, us = rng.random((B, g)).astype(np.float32), rng.random(B).astype(np.float32)
        k1, t1, n1 = run(oracle_mod, lp, lq, x, ua, us, temperature=T, draft_temperature=Td, band=1e-6)
        k2, t2, n2, _ = oracle_mod.spec_accept(P.astype(np.float32), Q.astype(np.float32), x, ua, us)
        ok = ~(n1 | n2)
        assert np.array_equal(k1[ok], k2[ok])
        assert np.array_equal(t1[ok], t2[ok])
        lo, hi = oracle_mod.logits_draw_window(lp, lq, k2, us, temperature=T, draft_temperature=Td, band=1e-6)
        drawn = t2[np.arange(B), k2]
        assert np.all((lo <= drawn) & (drawn <= hi))

    check()
