"""GPU parity of svpa_spec_accept / svpa_spec_accept_tree against the oracle.

Accepted lengths must be bit-exact everywhere (the acceptance test is one
rounded fp32 product on both sides).  Emitted tokens must be bit-exact on
every row whose final draw the oracle does not flag as within 1e-6 of a CDF
boundary; on flagged rows the GPU's token must still be one whose CDF
interval reaches within 1e-6 of the uniform.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

from tree_check import tree_walk_valid

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_linear(s):
    B, g1, V = s.p.shape
    d = {k: getattr(s, k).to(DEV) for k in ("p", "q", "tokens", "u_accept", "u_sample")}
    k = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    toks = torch.full((B, g1), -7, dtype=torch.int32, device=DEV)
    near = torch.zeros(B, dtype=torch.uint8, device=DEV)
    ws = torch.zeros(svpa.spec_accept_workspace_size(B, V), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):  # second call checks the self-cleaning tickets
        svpa.spec_accept(d["p"], d["q"], d["tokens"], d["u_accept"], d["u_sample"], k, toks,
                         workspace=ws, error_flag=err, near_boundary=near)
    assert svpa.check_error(err) == 0
    return k.cpu().numpy(), toks.cpu().numpy(), near.cpu().numpy().astype(bool)


def residual_cdf(s, b, k):
    """fp64 cumulative residual (or bonus) mass of row b at position k, normalised."""
    p = s.p[b, k].double().numpy()
    gamma = s.q.shape[1]
    if k < gamma:
        r = np.maximum(p - s.q[b, k].double().numpy(), 0.0)
        if r.sum() == 0:
            r = p
    else:
        r = p
    c = np.cumsum(r)
    return c / c[-1]


def check_linear(s):
    """Accepted lengths bit-exact; tokens bit-exact on every row the oracle does
    not flag; on flagged rows (u within 1e-6 of a CDF boundary, where fp32 and
    exact sums may resolve the draw differently) the GPU token must be one whose
    CDF interval reaches within 1e-6 of u."""
    k, toks, gnear = run_linear(s)
    rk, rt, rnear, _ = oracle.spec_accept(s.p.cpu(), s.q.cpu(), s.tokens.cpu(), s.u_accept.cpu(),
                                          s.u_sample.cpu())
    assert np.array_equal(k, rk)
    ok = ~rnear
    assert np.array_equal(toks[ok], rt[ok])
    for b in np.where(rnear)[0]:
        assert np.array_equal(toks[b, :k[b]], rt[b, :k[b]])
        assert np.all(toks[b, k[b] + 1:] == -1)
        if toks[b, k[b]] != rt[b, k[b]]:
            c = residual_cdf(s, b, k[b])
            t = toks[b, k[b]]
            u = float(s.u_sample[b])
            lo = c[t - 1] if t > 0 else 0.0
            assert lo - 1e-6 <= u <= c[t] + 1e-6, (b, t, u, lo, c[t])
    return k


@pytest.mark.parametrize("name", ["tiny", "7b", "70b"])
def test_linear_parity(name):
    wl = W.WORKLOADS[name]
    s = W.make_sampler(wl, W.SEEDS[name], device="cpu")
    check_linear(s)


def test_linear_fp8_workload_shape():
    wl = W.WORKLOADS["fp8"]
    s = W.make_sampler(wl, W.SEEDS["fp8"], device="cpu")
    check_linear(s)


def test_linear_many_rows_small_vocab():
    wl = W.WORKLOADS["7b"].scaled(batch=3000, vocab=257, gamma=6)
    s = W.make_sampler(wl, 44, device="cpu")
    k = check_linear(s)
    assert 0 < (k == wl.gamma).mean() < 1 and (k == 0).any()


def test_linear_all_accept_and_all_reject():
    wl = W.WORKLOADS["7b"].scaled(batch=8, vocab=5000)
    s = W.make_sampler(wl, 45, device="cpu")
    # P == Q: everything accepted, bonus from P_gamma
    s.q = s.p[:, :wl.gamma].clone()
    k, toks, _ = run_linear(s)
    assert np.all(k == wl.gamma)
    check_linear(s)
    # draft token impossible under P: rejected at 0
    s2 = W.make_sampler(wl, 46, device="cpu")
    x = s2.tokens[:, 0].long()
    s2.p[torch.arange(8), 0, x] = 0.0
    k, _, _ = run_linear(s2)
    assert np.all(k == 0)
    check_linear(s2)


def test_linear_uniform_edges():
    wl = W.WORKLOADS["7b"].scaled(batch=16, vocab=4099)
    s = W.make_sampler(wl, 47, device="cpu")
    s.u_sample[:4] = 0.0
    s.u_sample[4:8] = torch.nextafter(torch.tensor(1.0), torch.tensor(0.0))
    s.u_accept[8:12] = 0.0
    check_linear(s)


def run_tree(parent, s):
    B, n, V = s.p.shape
    W_ = oracle.tree_max_depth(np.array(parent, np.int32)) + 1
    k = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    path = torch.full((B, W_), -7, dtype=torch.int32, device=DEV)
    toks = torch.full((B, W_), -7, dtype=torch.int32, device=DEV)
    near = torch.zeros(B, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.spec_accept_tree(parent, s.p.to(DEV), s.q.to(DEV), s.tokens.to(DEV), s.u_accept.to(DEV),
                          s.u_sample.to(DEV), k, path, toks, error_flag=err, near_boundary=near)
    assert svpa.check_error(err) == 0
    return k.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy()


def check_tree(parent, s, max_near):
    """Rows the oracle does not flag: accepted length, path and tokens equal.
    Every row, flagged or not: the GPU's path and final token are valid under
    tree_walk_valid (every decision outside the band agrees with the exact one,
    the path agrees up to the first in-band decision, the final token lies in
    the 1e-6 window of the distribution the walk ends in)."""
    k, path, toks = run_tree(parent, s)
    rk, rpath, rtoks, rnear = oracle.spec_accept_tree(np.array(parent, np.int32), s.p, s.q, s.tokens,
                                                      s.u_accept, s.u_sample)
    ok = ~rnear
    print(f"tree sampler: {int(rnear.sum())} of {rnear.shape[0]} rows flagged near a boundary "
          f"({rnear.mean():.3f})")
    assert rnear.mean() <= max_near  # flagged draws are reported; a flood would mean a bug
    assert np.array_equal(k[ok], rk[ok])
    assert np.array_equal(path[ok], rpath[ok])
    assert np.array_equal(toks[ok], rtoks[ok])
    for b in range(k.shape[0]):
        valid, _ = tree_walk_valid(parent, s, b, int(k[b]), path[b], toks[b])
        assert valid, (b, k[b], path[b], toks[b], rk[b], rpath[b], rtoks[b])
    return k


# The oracle's flagged fractions on these seeded inputs (deterministic): batch
# 4 none, batch 128 2 rows (0.016); vocabulary 4099 none, 128256 1 of 6 rows.
# The bounds sit just above them: a flood of flags would mean a bug.
@pytest.mark.parametrize("batch,max_near", [(4, 0.01), (128, 0.02)])
def test_tree_parity(batch, max_near):
    wl = W.WORKLOADS["tree"].scaled(batch=batch)
    s = W.make_sampler(wl, W.SEEDS["tree"], device="cpu")
    check_tree(wl.parent, s, max_near=max_near)


@pytest.mark.parametrize("vocab,max_near", [(4099, 0.01), (128256, 0.17)])
def test_tree_vocab_edges(vocab, max_near):
    # 4099: rows not a multiple of 4 tokens (scalar loads); 128256: a
    # residual row larger than one CTA's shared memory would hold
    wl = W.WORKLOADS["tree"].scaled(batch=6)
    s = W.make_sampler(wl, 61, device="cpu", vocab=vocab)
    check_tree(wl.parent, s, max_near=max_near)


def test_tree_empty_residual_draws_from_target():
    # chain 0-1-2-3; at the root P = Q/2 (unnormalised) so the residual after
    # the rejection is empty and the token comes from P_root itself
    wl = W.WORKLOADS["7b"].scaled(batch=16, vocab=3000, gamma=3)
    s = W.make_sampler(wl, 62, device="cpu")
    parent = [-1, 0, 1, 2]
    B = 16
    tok = torch.cat([torch.zeros(B, 1, dtype=torch.int32), s.tokens], 1)
    ua = torch.cat([torch.zeros(B, 1), s.u_accept], 1)
    ua[:, 1] = 0.99
    p = s.p.clone()
    p[:, 0] = 0.5 * s.q[:, 0]
    t = W.SamplerInputs(p=p, q=s.q, tokens=tok, u_accept=ua, u_sample=s.u_sample)
    k = check_tree(parent, t, max_near=0.01)
    assert np.all(k == 0)


def test_tree_chain_matches_linear_kernel():
    wl = W.WORKLOADS["7b"].scaled(batch=64, vocab=3000, gamma=4)
    s = W.make_sampler(wl, 48, device="cpu")
    k, toks, _ = run_linear(s)
    B = 64
    parent = [-1, 0, 1, 2, 3]
    tok = torch.cat([torch.zeros(B, 1, dtype=torch.int32), s.tokens], 1)
    ua = torch.cat([torch.zeros(B, 1), s.u_accept], 1)
    kt = torch.empty(B, dtype=torch.int32, device=DEV)
    path = torch.empty((B, 5), dtype=torch.int32, device=DEV)
    outt = torch.empty((B, 5), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.spec_accept_tree(parent, s.p.to(DEV), s.q.to(DEV), tok.to(DEV), ua.to(DEV),
                          s.u_sample.to(DEV), kt, path, outt, error_flag=err)
    assert svpa.check_error(err) == 0
    assert np.array_equal(kt.cpu().numpy(), k)
    assert np.array_equal(outt.cpu().numpy(), toks)


def test_linear_empty_residual_draws_from_target():
    # P_0 = Q_0/2 (unnormalised): draft 0 is rejected for u > 1/2 and the
    # residual max(0, P_0 - Q_0) is empty, so the token is drawn from P_0
    wl = W.WORKLOADS["7b"].scaled(batch=16, vocab=5000)
    s = W.make_sampler(wl, 63, device="cpu")
    s.p[:, 0] = 0.5 * s.q[:, 0]
    s.u_accept[:, 0] = 0.9
    k = check_linear(s)
    assert np.all(k == 0)


def test_linear_unaligned_rows():
    # rows that start 4 bytes past a 16-byte boundary take the scalar loads
    wl = W.WORKLOADS["7b"].scaled(batch=12, vocab=6000)
    s = W.make_sampler(wl, 64, device="cpu")
    B, g1, V = s.p.shape
    d = {}
    for name in ("p", "q"):
        x = getattr(s, name)
        buf = torch.empty(x.numel() + 1, dtype=x.dtype, device=DEV)
        dv = buf[1:].view(x.shape)
        dv.copy_(x)
        d[name] = dv
    assert d["p"].data_ptr() % 16 != 0
    k = torch.empty(B, dtype=torch.int32, device=DEV)
    toks = torch.empty((B, g1), dtype=torch.int32, device=DEV)
    ws = torch.zeros(svpa.spec_accept_workspace_size(B, V), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.spec_accept(d["p"], d["q"], s.tokens.to(DEV), s.u_accept.to(DEV), s.u_sample.to(DEV), k, toks,
                     workspace=ws, error_flag=err)
    assert svpa.check_error(err) == 0
    rk, rt, rnear, _ = oracle.spec_accept(s.p, s.q, s.tokens, s.u_accept, s.u_sample)
    assert np.array_equal(k.cpu().numpy(), rk)
    assert np.array_equal(toks.cpu().numpy()[~rnear], rt[~rnear])


def test_linear_vocab_beyond_cluster_rows():
    # V > 262144 takes the one-CTA-per-row kernel
    wl = W.WORKLOADS["7b"].scaled(batch=3, vocab=300_000, gamma=2)
    s = W.make_sampler(wl, 65, device="cpu")
    check_linear(s)


def test_gpu_output_distribution_equals_target():
    # Monte-Carlo on the GPU path: first emitted token ~ P_0
    from scipy import stats
    rng = np.random.default_rng(17)
    B, gamma, V = 100_000, 2, 8
    logits = rng.normal(0, 1.5, size=(gamma + 1, V))
    P = np.exp(logits) / np.exp(logits).sum(-1, keepdims=True)
    ql = rng.normal(0, 1.5, size=(gamma, V))
    Q = np.exp(ql) / np.exp(ql).sum(-1, keepdims=True)
    P32 = torch.tensor(np.broadcast_to(P, (B, gamma + 1, V)).copy(), dtype=torch.float32)
    Q32 = torch.tensor(np.broadcast_to(Q, (B, gamma, V)).copy(), dtype=torch.float32)
    cdf = np.cumsum(Q, -1)
    x = torch.tensor((rng.random((B, gamma, 1)) >= cdf[None]).sum(-1), dtype=torch.int32)
    s = W.SamplerInputs(p=P32, q=Q32, tokens=x, u_accept=torch.tensor(rng.random((B, gamma)), dtype=torch.float32),
                        u_sample=torch.tensor(rng.random(B), dtype=torch.float32))
    k, toks, _ = run_linear(s)
    obs = np.bincount(toks[:, 0], minlength=V)
    assert stats.chisquare(obs, P[0] / P[0].sum() * B).pvalue > 1e-4
