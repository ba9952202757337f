"""The draft-tree sampler fed by logits, on the GPU through the C ABI, against the oracle.

P = softmax(target logits / T) at every node and Q = softmax(draft logits /
T_draft) at every internal node are formed inside the kernel in fp32 (the
statistics of the visited rows only); the oracle forms them in fp64.  Every
row is checked:
  * its path is a chain from the root (each node a child of the one before),
    the emitted tokens are the path's node tokens, then the drawn token, then
    -1, and the accepted count is the path's length;
  * the node it ended on is one where the oracle's outcome set says an fp32
    formation may end (each test on the way, and the rejections at the end,
    exact or within its band), and the drawn token lies in the oracle's draw
    window there -- both computed from the inputs alone;
  * where neither side flags a near decision, the accepted count, the path
    and the tokens are the oracle's exactly.
Plus the full-size draft-tree workload, the output distribution (chi-square
at V = 8), masked tokens, rows that are not 16-byte aligned, a vocabulary of
one, a row with no finite logit (an error, no fault) and graph replay.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def width_of(parent):
    return oracle.tree_max_depth(np.asarray(parent, np.int32)) + 1


def gpu_run(ti, offset=0):
    """Runs the kernel; with offset > 0 the logit rows start that many floats
    into their buffers (not 16-byte aligned)."""
    B, n, V = ti.lp.shape
    Wd = width_of(ti.parent.numpy())

    def dev(x):
        if not offset:
            return x.to(DEV).contiguous()
        buf = torch.empty(x.numel() + offset, dtype=x.dtype, device=DEV)
        buf[offset:] = x.reshape(-1).to(DEV)
        return buf[offset:].view(x.shape)

    k = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    path = torch.full((B, Wd), -7, dtype=torch.int32, device=DEV)
    toks = torch.full((B, Wd), -7, dtype=torch.int32, device=DEV)
    nb = torch.full((B,), 7, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.spec_accept_tree_logits(ti.parent.tolist(), dev(ti.lp), dev(ti.lq), ti.tokens.to(DEV),
                                 ti.u_accept.to(DEV), ti.u_sample.to(DEV), k, path, toks, error_flag=err,
                                 temperature=ti.temperature, draft_temperature=ti.draft_temperature,
                                 near_boundary=nb)
    torch.cuda.synchronize()
    return (k.cpu().numpy(), path.cpu().numpy(), toks.cpu().numpy(), nb.cpu().numpy(), svpa.check_error(err))


def check_against_oracle(ti, offset=0, min_same=0.95):
    kg, pg, tg, ng, e = gpu_run(ti, offset)
    assert e == 0
    assert set(np.unique(ng)) <= {0, 1}
    ng = ng.astype(bool)
    par = ti.parent.numpy()
    B, n, V = ti.lp.shape
    Wd = width_of(par)
    T, Td = ti.temperature, ti.draft_temperature
    ko, po, to, no = oracle.spec_accept_tree_logits(par, ti.lp, ti.lq, ti.tokens, ti.u_accept, ti.u_sample,
                                                    temperature=T, draft_temperature=Td)
    end_ok, lo, hi = oracle.tree_logits_outcomes(par, ti.lp, ti.lq, ti.tokens, ti.u_accept, ti.u_sample,
                                                 temperature=T, draft_temperature=Td)
    tok = ti.tokens.numpy()
    assert np.all((kg >= 0) & (kg < Wd))
    assert np.all(pg[:, 0] == 0)
    for b in range(B):
        k = kg[b]
        for d in range(1, k + 1):
            assert par[pg[b, d]] == pg[b, d - 1], (b, d)
            assert tg[b, d - 1] == tok[b, pg[b, d]], (b, d)
        assert np.all(pg[b, k + 1:] == -1) and np.all(tg[b, k + 1:] == -1)
    rows = np.arange(B)
    end = pg[rows, kg]
    drawn = tg[rows, kg]
    assert np.all(end_ok[rows, end]), np.nonzero(~end_ok[rows, end])
    inwin = (lo[rows, end] <= drawn) & (drawn <= hi[rows, end])
    assert np.all(inwin), np.nonzero(~inwin)
    ok = ~(ng | no)
    assert np.array_equal(kg[ok], ko[ok])
    assert np.array_equal(pg[ok], po[ok])
    assert np.array_equal(tg[ok], to[ok])
    same = (kg == ko) & np.all(pg == po, axis=1)
    assert same.mean() >= min_same
    return kg, pg, tg, ng


SMALL = [
    # (branching, B, V, T, T_draft)
    ((4, 2, 2), 48, 1000, 1.0, 1.0),
    ((4, 2, 2), 40, 4099, 0.8, 1.2),      # V % 4 != 0: scalar loads
    ((2, 2, 2, 2), 24, 32000, 1.0, 1.0),
    ((3, 2), 6, 50257, 1.3, 0.6),          # ragged tail of the last CTA's slice
    ((5,), 300, 2048, 1.0, 1.0),           # more rows than cluster slots
    ((1, 1, 1, 1), 32, 5000, 1.0, 1.0),    # a chain
    ((8, 2), 4, 262144, 1.0, 1.0),         # the largest vocabulary
    ((2, 1), 3, 7, 1.0, 1.0),
]


@pytest.mark.parametrize("br,B,V,T,Td", SMALL)
def test_matches_oracle(br, B, V, T, Td):
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 700 + B + V, batch=B, vocab=V, branching=br, temperature=T,
                            draft_temperature=Td)
    check_against_oracle(ti, min_same=0.0 if B < 30 else 0.95)


def test_full_size_tree_workload():
    wl = W.WORKLOADS["tree"]
    ti = W.make_tree_logits(wl, W.SEEDS["tree"] + 5)
    kg, _, _, _ = check_against_oracle(ti)
    assert kg.max() >= 2  # the walk goes deep on some rows


def test_unaligned_rows():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 81, batch=16, vocab=6000, branching=(3, 2))
    check_against_oracle(ti, offset=1, min_same=0.0)


def test_vocabulary_of_one():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 82, batch=5, vocab=1, branching=(2, 2))
    kg, pg, tg, _ = check_against_oracle(ti, min_same=0.0)
    # P = Q = (1): the first child is always accepted, down to a leaf
    assert np.all(kg == 2) and np.all(tg[:, :3] == 0) and np.all(pg[:, 1] == 1)


def test_masked_tokens_are_never_drawn():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 83, batch=64, vocab=3000, branching=(4, 2))
    thr = ti.lp.median(dim=-1, keepdim=True).values
    ti.lp[ti.lp > thr] = -float("inf")
    kg, pg, tg, _ = check_against_oracle(ti, min_same=0.9)
    rows = np.arange(64)
    lp = ti.lp.numpy()
    assert np.all(np.isfinite(lp[rows, pg[rows, kg], tg[rows, kg]]))


def test_output_distribution_is_target():
    rng = np.random.default_rng(3)
    parent = W.tree_parents((3, 2))
    n, V, B = len(parent), 8, 100_000
    internal = [0, 1, 2, 3]
    lp1 = torch.tensor(rng.normal(0, 1.2, (n, V)), dtype=torch.float32)
    lq1 = lp1[internal] + torch.tensor(rng.normal(0, 0.8, (len(internal), V)), dtype=torch.float32)
    T, Td = 0.9, 1.2
    P = torch.softmax(lp1.double() / T, -1).numpy()
    Q = torch.softmax(lq1.double() / Td, -1)
    tok = torch.zeros((B, n), dtype=torch.int32)
    for c in range(1, n):
        tok[:, c] = torch.multinomial(Q[internal.index(parent[c])], B, replacement=True,
                                      generator=torch.Generator().manual_seed(c)).to(torch.int32)
    ti = W.TreeLogitInputs(lp=lp1.expand(B, n, V).contiguous(), lq=lq1.expand(B, len(internal), V).contiguous(),
                           tokens=tok, u_accept=torch.rand((B, n), generator=torch.Generator().manual_seed(7)),
                           u_sample=torch.rand((B,), generator=torch.Generator().manual_seed(8)),
                           parent=torch.tensor(parent, dtype=torch.int32), temperature=T, draft_temperature=Td)
    kg, pg, tg, ng, e = gpu_run(ti)
    assert e == 0
    obs = np.bincount(tg[:, 0], minlength=V).astype(np.float64)
    assert stats.chisquare(obs, P[0] * B).pvalue > 1e-4
    sel = pg[:, 1] == 1  # node 1 accepted: the next token follows P at node 1
    obs = np.bincount(tg[sel, 1], minlength=V).astype(np.float64)
    assert sel.sum() > 5000 and stats.chisquare(obs, P[1] * obs.sum()).pvalue > 1e-4


def test_row_without_a_finite_logit_raises_the_error_flag():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 84, batch=3, vocab=2000, branching=(2, 2))
    ti.lp[1, 0, :] = -float("inf")  # the root's target row of sequence 1 (always visited)
    kg, pg, tg, ng, e = gpu_run(ti)
    assert e == 1  # SVPA_DEVERR_BAD_VALUE maps to SVPA_ERR_INVALID_ARG
    assert np.all((kg >= 0) & (kg <= 2))
    assert np.all((tg >= -1) & (tg < 2000))


def test_invalid_arguments_are_refused():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 85, batch=2, vocab=100, branching=(2,))
    lp, lq = ti.lp.to(DEV), ti.lq.to(DEV)
    k = torch.empty(2, dtype=torch.int32, device=DEV)
    path = torch.empty((2, 2), dtype=torch.int32, device=DEV)
    toks = torch.empty((2, 2), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    args = (lp, lq, ti.tokens.to(DEV), ti.u_accept.to(DEV), ti.u_sample.to(DEV), k, path, toks)
    assert svpa.spec_accept_tree_logits([-1, 1, 0], *args, error_flag=err, check=False) == 1  # parent after child
    assert svpa.spec_accept_tree_logits([-1, 0, 0], *args, error_flag=err, temperature=0.0, check=False) == 1
    assert svpa.spec_accept_tree_logits([-1, 0, 0], *args, error_flag=err, draft_temperature=float("nan"),
                                        check=False) == 1
    assert svpa.spec_accept_tree_logits([-1, 0, 0], *args, error_flag=None, check=False) == 1
    torch.cuda.synchronize()
    assert svpa.check_error(err) == 0


def test_graph_replay_matches_eager():
    ti = W.make_tree_logits(W.WORKLOADS["tree"], 86, batch=32, vocab=32000, temperature=0.9)
    B, n, V = ti.lp.shape
    Wd = width_of(ti.parent.numpy())
    ins = [t.to(DEV).contiguous() for t in (ti.lp, ti.lq, ti.tokens, ti.u_accept, ti.u_sample)]
    k = torch.empty(B, dtype=torch.int32, device=DEV)
    path = torch.empty((B, Wd), dtype=torch.int32, device=DEV)
    toks = torch.empty((B, Wd), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    par = ti.parent.tolist()
    run = lambda: svpa.spec_accept_tree_logits(par, *ins, k, path, toks, error_flag=err, temperature=0.9)
    run()
    torch.cuda.synchronize()
    want = (k.clone(), path.clone(), toks.clone())
    for t in (k, path, toks):
        t.fill_(-5)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run()
    graph.replay()
    torch.cuda.synchronize()
    assert svpa.check_error(err) == 0
    assert torch.equal(k, want[0]) and torch.equal(path, want[1]) and torch.equal(toks, want[2])
