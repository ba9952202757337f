"""Pins of the oracle's acceptance telemetry and adaptive draft length
against what fixes them independently of the code: the estimator's limit
under simulated per-token acceptance (a geometric-truncation argument), the
threshold table at its edges, the moving average's closed form, and E[K] /
speed-up against their closed forms and the worked example on the pages."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def simulate_accepted(alpha, gamma, steps, rng):
    """Accepted prefix lengths of a per-token Bernoulli(alpha) accept chain."""
    passes = rng.random((steps, gamma)) < alpha
    first_fail = np.where(passes.all(1), gamma, np.argmin(passes, 1))
    return first_fail.astype(np.int32)


@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.8, 0.92])
def test_estimator_recovers_per_token_rate(alpha):
    # with no forgetting (decay 1), accepted / tests is the per-token rate's
    # maximum-likelihood estimate; counting gamma tests per step instead would
    # bias it low, counting only accepts / (k + 1) would bias it for k = gamma
    rng = np.random.default_rng(7)
    k = simulate_accepted(alpha, 4, 40000, rng)
    r = oracle.gamma_update(4, k, seq_state=np.zeros((k.size, 2), np.float32), decay=1.0)
    a, n = r["batch_state"]
    assert abs(a / n - alpha) < 0.01
    # the per-sequence states see one step each: k / (k + [k < gamma])
    ss = r["seq_state"]
    assert np.array_equal(ss[:, 0], k.astype(np.float32))
    assert np.array_equal(ss[:, 1], (k + (k < 4)).astype(np.float32))


def test_threshold_table_edges():
    f = lambda x: oracle.gamma_from_alpha(np.float32(x))
    assert [f(0.99), f(0.86), f(0.85), f(0.71), f(0.70), f(0.51), f(0.50)] == [5, 5, 4, 4, 3, 3, 2]
    assert [f(0.25), f(np.nextafter(np.float32(0.25), np.float32(0))), f(0.0)] == [2, 1, 1]
    # the page's switch: > 0.85 -> 5, > 0.70 -> 4, > 0.50 -> 3, otherwise 2
    assert f(np.nextafter(np.float32(0.85), np.float32(1))) == 5


def test_moving_average_closed_form():
    # constant k and tests every step: A_n = k (1 - d^n) / (1 - d)
    d, k, steps = 0.9, 3, 25
    st, bs = np.zeros((1, 2), np.float32), (0.0, 0.0)
    for _ in range(steps):
        r = oracle.gamma_update(5, [k], seq_state=st, batch_state=bs, decay=d)
        st, bs = r["seq_state"], r["batch_state"]
    want_a = k * (1 - d ** steps) / (1 - d)
    want_n = (k + 1) * (1 - d ** steps) / (1 - d)
    assert abs(st[0, 0] - want_a) < 1e-4 * want_a and abs(st[0, 1] - want_n) < 1e-4 * want_n
    assert r["seq_gamma"][0] == oracle.gamma_from_alpha(np.float32(st[0, 0]) / np.float32(st[0, 1]))
    assert r["seq_gamma"][0] == 4  # alpha = 3/4


def test_collapse_falls_back_to_one_and_recovers():
    st, bs = np.zeros((2, 2), np.float32), (0.0, 0.0)
    for _ in range(30):  # sequence 0 never accepts, sequence 1 always does
        r = oracle.gamma_update(5, [0, 5], seq_state=st, batch_state=bs, decay=0.8)
        st, bs = r["seq_state"], r["batch_state"]
    assert list(r["seq_gamma"]) == [1, 5]
    for _ in range(30):  # at gamma 1 every step is one test: recovery is possible
        r = oracle.gamma_update(1, [1, 1], seq_state=st, batch_state=bs, decay=0.8)
        st, bs = r["seq_state"], r["batch_state"]
    assert list(r["seq_gamma"]) == [5, 5]


def test_expected_accepted_and_speedup_closed_forms():
    # constant alpha: E[K] = alpha (1 - alpha^g) / (1 - alpha) at the batch's
    # own draft length, speed-up (E[K] + 1) / (g r + 1)
    for alpha in (0.86, 0.75, 0.6, 0.3):
        # a state whose updated batch alpha is close to `alpha`
        r = oracle.gamma_update(4, [4], batch_state=(np.float32(alpha * 2000), np.float32(2000)), decay=0.5, r=0.08)
        al, g = float(r["telemetry"][0]), r["batch_gamma"]
        assert g == oracle.gamma_from_alpha(np.float32(al))
        ek = al * (1 - al ** g) / (1 - al)
        assert abs(r["telemetry"][2] - ek) < 1e-5
        assert abs(r["telemetry"][3] - (ek + 1) / (g * 0.08 + 1)) < 1e-5
    # the page's worked example (alpha 0.85, r 0.08, 4 drafts: speed-up above 2.8),
    # through the oracle's own E[K] and speed-up functions
    alpha_s, r_s, g_s, eta_lo = open(os.path.join(GOLDEN, "eta_worked_example.txt")).read().split("\n")[-2].split()
    alpha, r_, g = float(alpha_s), float(r_s), int(g_s)
    assert oracle.gamma_from_alpha(np.float32(alpha)) == g  # 0.85 is not above 0.85: 4 drafts
    ek = oracle.expected_accepted([alpha] * g)
    assert oracle.speedup(ek, g, r_) >= float(eta_lo)


def test_mean_accepted_and_batch_gamma_use_integer_totals():
    k = np.array([0, 1, 2, 3, 4, 4, 4, 1], np.int32)
    r = oracle.gamma_update(4, k, decay=0.0)
    assert r["telemetry"][1] == np.float32(k.sum()) / np.float32(k.size)
    tests = (k + (k < 4)).sum()
    assert r["telemetry"][0] == np.float32(k.sum()) / np.float32(tests)
    assert r["batch_gamma"] == oracle.gamma_from_alpha(np.float32(k.sum()) / np.float32(tests))


def test_invalid_counts_are_rejected():
    with pytest.raises(oracle.OracleError):
        oracle.gamma_update(4, [5])
    with pytest.raises(oracle.OracleError):
        oracle.gamma_update(4, [-1])
