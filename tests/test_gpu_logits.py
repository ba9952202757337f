"""The sampler fed by logits, on the GPU through the C ABI, against the oracle.

P = softmax(target logits / T) and Q = softmax(draft logits / T_draft) are
formed inside the kernel in fp32; the oracle forms them in fp64.  Every row is
checked:
  * its accepted count k is one the oracle allows: every test before k is an
    oracle accept or within the 5e-5 band, test k an oracle reject or within
    the band;
  * the tokens before k are the drafts, those after it -1;
  * its drawn token lies in the oracle's draw window at the kernel's own k
    (the tokens whose running-sum interval, widened by the band, holds u*Z;
    the oracle computes the window at every k from the inputs alone);
  * where neither side flags a near decision, k and the tokens are the
    oracle's exactly.
Plus the output distribution (chi-square at V = 8) and the edge cases: V = 1,
gamma = 32, rows that are not 16-byte aligned, masked (-inf) tokens, a row
with no finite logit (an error, no fault).
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


def gpu_run(li, offset=0):
    """Runs the kernel; with offset > 0 the logit rows start that many floats
    into their buffers (not 16-byte aligned)."""
    B, g1, V = li.lp.shape

    def dev(x):
        if not offset:
            return x.to(DEV).contiguous()
        buf = torch.empty(x.numel() + offset, dtype=x.dtype, device=DEV)
        buf[offset:] = x.reshape(-1).to(DEV)
        return buf[offset:].view(x.shape)

    k = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    toks = torch.full((B, g1), -7, dtype=torch.int32, device=DEV)
    nb = torch.full((B,), 7, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(svpa.spec_accept_logits_workspace_size(B, g1 - 1, V), dtype=torch.uint8, device=DEV)
    svpa.spec_accept_logits(dev(li.lp), dev(li.lq), li.tokens.to(DEV), li.u_accept.to(DEV), li.u_sample.to(DEV),
                            k, toks, workspace=ws, error_flag=err, temperature=li.temperature,
                            draft_temperature=li.draft_temperature, near_boundary=nb)
    torch.cuda.synchronize()
    return k.cpu().numpy(), toks.cpu().numpy(), nb.cpu().numpy(), svpa.check_error(err)


def check_against_oracle(li, offset=0, min_same_k=0.98):
    kg, tg, ng, e = gpu_run(li, offset)
    assert e == 0
    assert set(np.unique(ng)) <= {0, 1}
    ng = ng.astype(bool)
    B, g = li.tokens.shape
    T, Td = li.temperature, li.draft_temperature
    ko, to, no, acc, accn = oracle.spec_accept_logits(li.lp, li.lq, li.tokens, li.u_accept, li.u_sample,
                                                      temperature=T, draft_temperature=Td, tests=True)
    x = li.tokens.numpy()
    assert np.all((kg >= 0) & (kg <= g))
    allowed = acc | accn           # an accept is allowed
    rej_allowed = ~acc | accn      # a reject is allowed
    idx = np.arange(g)
    before = idx[None, :] < kg[:, None]
    assert np.all(allowed[before])
    at = kg < g
    assert np.all(rej_allowed[np.nonzero(at)[0], kg[at]])
    pos = np.arange(g + 1)[None, :]
    assert np.array_equal(np.where(pos < kg[:, None], np.pad(x, ((0, 0), (0, 1))), 0)[pos < kg[:, None]],
                          tg[pos < kg[:, None]])
    assert np.all(tg[pos > kg[:, None]] == -1)
    # the draw windows at every possible accepted count, from the inputs alone;
    # the row's own count picks one
    win = [oracle.logits_draw_window(li.lp, li.lq, np.full(B, kk, np.int32), li.u_sample, temperature=T,
                                     draft_temperature=Td) for kk in range(g + 1)]
    lo = np.stack([w[0] for w in win], 1)[np.arange(B), kg]
    hi = np.stack([w[1] for w in win], 1)[np.arange(B), kg]
    drawn = tg[np.arange(B), kg]
    assert np.all((lo <= drawn) & (drawn <= hi)), np.nonzero(~((lo <= drawn) & (drawn <= hi)))
    ok = ~(ng | no)
    assert np.array_equal(kg[ok], ko[ok])
    assert np.array_equal(tg[ok], to[ok])
    assert (kg == ko).mean() >= min_same_k
    return kg, tg, ng


SMALL = [
    # (B, gamma, V, T, T_draft)
    (3, 4, 1000, 1.0, 1.0),
    (40, 4, 4099, 1.0, 1.0),       # V % 4 != 0: scalar loads
    (5, 8, 32000, 0.7, 0.7),
    (2, 5, 50257, 1.3, 0.6),       # ragged tail of the last CTA's slice
    (400, 4, 32000, 1.0, 1.0),     # more rows than slots: fewer CTAs per row
    (4, 32, 2048, 1.0, 1.0),       # gamma = 32: 65 rows per sequence
    (1, 1, 7, 1.0, 1.0),
    (6, 3, 262144, 1.0, 1.0),      # the largest vocabulary
]


@pytest.mark.parametrize("B,g,V,T,Td", SMALL)
def test_matches_oracle(B, g, V, T, Td):
    wl = W.WORKLOADS["7b"]
    li = W.make_logits(wl, 900 + B + g + V, batch=B, vocab=V, gamma=g, temperature=T, draft_temperature=Td)
    check_against_oracle(li, min_same_k=0.0 if B < 20 else 0.98)


def test_unaligned_rows():
    li = W.make_logits(W.WORKLOADS["7b"], 77, batch=9, vocab=5000, gamma=3)
    check_against_oracle(li, offset=1)


def test_vocabulary_of_one():
    li = W.make_logits(W.WORKLOADS["tiny"], 5, batch=4, vocab=1, gamma=2)
    kg, tg, ng = check_against_oracle(li)
    assert np.all(kg == 2) and np.all(tg == 0)


def test_masked_tokens_are_never_drawn():
    li = W.make_logits(W.WORKLOADS["7b"], 13, batch=64, vocab=3000, gamma=4)
    # the top-scoring half of every target row masked out: only the other
    # half may be emitted (the drafts keep their own logits)
    thr = li.lp.median(dim=-1, keepdim=True).values
    li.lp[li.lp > thr] = -float("inf")
    kg, tg, _ = check_against_oracle(li)
    drawn = tg[np.arange(64), kg]
    lp = li.lp.numpy()
    assert np.all(np.isfinite(lp[np.arange(64), kg, drawn]))


@pytest.mark.parametrize("name", ["7b", "70b"])
def test_full_size(name):
    wl = W.WORKLOADS[name]
    li = W.make_logits(wl, W.SEEDS[name] + 3)
    check_against_oracle(li)


def test_output_distribution_is_target():
    rng = np.random.default_rng(2)
    V, g, B = 8, 2, 200_000
    lp1 = torch.tensor(rng.normal(0, 1.5, (g + 1, V)), dtype=torch.float32)
    lq1 = lp1[:g] + torch.tensor(rng.normal(0, 0.8, (g, V)), dtype=torch.float32)
    T, Td = 0.8, 1.1
    P = torch.softmax(lp1.double() / T, -1).numpy()
    Q = torch.softmax(lq1.double() / Td, -1)
    x = torch.stack([torch.multinomial(Q[i], B, replacement=True, generator=torch.Generator().manual_seed(i))
                     for i in range(g)], 1).to(torch.int32)
    li = W.LogitInputs(lp=lp1.expand(B, g + 1, V).contiguous(), lq=lq1.expand(B, g, V).contiguous(), tokens=x,
                       u_accept=torch.rand((B, g), generator=torch.Generator().manual_seed(7)),
                       u_sample=torch.rand((B,), generator=torch.Generator().manual_seed(8)),
                       temperature=T, draft_temperature=Td)
    kg, tg, ng, e = gpu_run(li)
    assert e == 0
    for pos, sel in ((0, np.ones(B, bool)), (1, kg >= 1)):
        obs = np.bincount(tg[sel, pos], minlength=V).astype(np.float64)
        assert stats.chisquare(obs, P[pos] * obs.sum()).pvalue > 1e-4, pos
    acc0 = np.minimum(P[0], Q[0].numpy()).sum()
    assert abs((kg >= 1).mean() - acc0) < 5 * np.sqrt(acc0 * (1 - acc0) / B)


def test_row_without_a_finite_logit_raises_the_error_flag():
    li = W.make_logits(W.WORKLOADS["7b"], 21, batch=3, vocab=2000, gamma=2)
    li.lp[1, 2, :] = -float("inf")  # the bonus row of sequence 1
    kg, tg, ng, e = gpu_run(li)
    assert e == 1  # SVPA_DEVERR_BAD_VALUE maps to SVPA_ERR_INVALID_ARG
    assert np.all((kg >= 0) & (kg <= 2))
    assert np.all((tg >= -1) & (tg < 2000))


def test_graph_replay_matches_eager():
    li = W.make_logits(W.WORKLOADS["7b"], 31, batch=16, vocab=32000, gamma=4, temperature=0.9)
    B, g1, V = li.lp.shape
    ins = [t.to(DEV).contiguous() for t in (li.lp, li.lq, li.tokens, li.u_accept, li.u_sample)]
    k = torch.empty(B, dtype=torch.int32, device=DEV)
    toks = torch.empty((B, g1), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(svpa.spec_accept_logits_workspace_size(B, g1 - 1, V), dtype=torch.uint8, device=DEV)
    run = lambda: svpa.spec_accept_logits(*ins, k, toks, workspace=ws, error_flag=err, temperature=0.9)
    run()
    torch.cuda.synchronize()
    want = (k.clone(), toks.clone())
    k.fill_(-5)
    toks.fill_(-5)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run()
    graph.replay()
    torch.cuda.synchronize()
    assert svpa.check_error(err) == 0
    assert torch.equal(k, want[0]) and torch.equal(toks, want[1])
