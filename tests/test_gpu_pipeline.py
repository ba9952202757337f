"""One whole verification step on the GPU, through the C ABI, against the same
step through the oracle: K/V append (with copy-on-write of a shared partly
filled page), paged verification attention over the appended cache, rejection
sampling, commit/rollback and the draft-length update.  Each side runs on its
own state, so block ids may differ; the attention output, accepted lengths and
tokens, committed lengths, the number of blocks held and the draft lengths
must not."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def gpu_step(inp, q, smp, wl):
    fp8 = wl.kv_fp8
    t = lambda x: x.to(DEV).clone()
    bt, cl, rc, fs = t(inp.block_table), t(inp.context_lens), t(inp.refcount), t(inp.free_stack)
    ft = torch.tensor([inp.free_top], dtype=torch.int32, device=DEV)
    kp, vp = t(inp.k_pool), t(inp.v_pool)
    if fp8:
        kp, vp = kp.view(torch.uint8), vp.view(torch.uint8)
    ks = t(inp.k_scale) if fp8 else None
    vs = t(inp.v_scale) if fp8 else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.kv_append(t(inp.new_k), t(inp.new_v), bt, cl, rc, fs, ft, kp, vp, error_flag=err, k_scale=ks,
                   v_scale=vs, scale_tile=wl.scale_tile)
    B, n_q, Hq, D = q.shape
    p = svpa.attn_params(B, n_q, Hq, wl.num_kv_heads, D, bt.shape[1], kp.shape[0], kv_fp8=fp8,
                         sm_scale=wl.sm_scale, scale_tile=wl.scale_tile)
    ws = torch.zeros(svpa.attn_workspace_size(p), dtype=torch.uint8, device=DEV)
    out = torch.empty((B, n_q, Hq, D), dtype=torch.bfloat16, device=DEV)
    svpa.paged_verify_attn(p, t(q), kp, vp, bt, cl, out, workspace=ws, error_flag=err, k_scale=ks, v_scale=vs)
    k = torch.empty(B, dtype=torch.int32, device=DEV)
    toks = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device=DEV)
    near = torch.zeros(B, dtype=torch.uint8, device=DEV)
    sws = torch.zeros(svpa.spec_accept_workspace_size(B, smp.p.shape[2]), dtype=torch.uint8, device=DEV)
    svpa.spec_accept(t(smp.p), t(smp.q), t(smp.tokens), t(smp.u_accept), t(smp.u_sample), k, toks,
                     workspace=sws, error_flag=err, near_boundary=near)
    svpa.block_table_commit(n_q, bt, cl, k, rc, fs, ft, error_flag=err)
    bs = torch.zeros(2, dtype=torch.float32, device=DEV)
    bg = torch.zeros(1, dtype=torch.int32, device=DEV)
    tel = torch.zeros(4, dtype=torch.float32, device=DEV)
    svpa.gamma_update(wl.gamma, k, bs, bg, tel, error_flag=err, draft_cost_ratio=0.08)
    assert svpa.check_error(err) == 0
    return dict(out=out.float().cpu().numpy(), k=k.cpu().numpy(), toks=toks.cpu().numpy(),
                near=near.cpu().numpy().astype(bool), bt=bt.cpu().numpy(), cl=cl.cpu().numpy(),
                rc=rc.cpu().numpy(), ft=int(ft.item()), fs=fs.cpu().numpy(), gamma=int(bg.item()))


def oracle_step(inp, q, smp, wl):
    c = lambda x: None if x is None else x.cpu()
    r = oracle.kv_append(c(inp.new_k), c(inp.new_v), inp.block_table.numpy(), inp.context_lens.numpy(),
                         inp.refcount.numpy(), inp.free_stack.numpy(), inp.free_top, c(inp.k_pool),
                         c(inp.v_pool), c(inp.k_scale), c(inp.v_scale), scale_tile=wl.scale_tile)
    out, _ = oracle.paged_verify_attn(q, r["k_pool"], r["v_pool"], r["block_table"], inp.context_lens.numpy(),
                                      num_kv_heads=wl.num_kv_heads, sm_scale=wl.sm_scale, kv_fp8=wl.kv_fp8,
                                      k_scale=r["k_scale"], v_scale=r["v_scale"], scale_tile=wl.scale_tile)
    k, toks, near, _ = oracle.spec_accept(smp.p, smp.q, smp.tokens, smp.u_accept, smp.u_sample)
    cm = oracle.block_table_commit(r["block_table"], inp.context_lens.numpy(), k, r["refcount"],
                                   r["free_stack"], r["free_top"], n_q=wl.n_q)
    g = oracle.gamma_update(wl.gamma, k, r=0.08)
    return dict(out=out, k=k, toks=toks, near=np.asarray(near).astype(bool), bt=cm["block_table"],
                cl=cm["context_lens"], rc=cm["refcount"], ft=cm["free_top"], gamma=g["batch_gamma"])


CASES = {
    # workload, contexts (private part), shared prefix (ends inside a page:
    # copy-on-write), factors of the appended rows.  bf16 rows are N(0, 1) as
    # in the task's workloads, so the plain attention bounds apply; the FP8
    # cases keep rows of 0.5x, 1x and 3x N(0, 1), so that page and tile scales
    # grow on some writes (requantised history) and not on others.
    "bf16": (W.WORKLOADS["7b"].scaled(num_q_heads=8, num_kv_heads=8, vocab=4000), (1, 3, 40, 250), 19, (1.0,)),
    "fp8": (W.WORKLOADS["fp8"].scaled(vocab=4000), (2, 6, 100, 700), 35, (0.5, 1.0, 3.0)),
    "fp8_t64": (W.WORKLOADS["fp8_t64"].scaled(vocab=4000), (0, 9, 64, 300), 21, (0.5, 1.0, 3.0)),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_verification_step_matches_oracle(name):
    wl, ctx, prefix, factors = CASES[name]
    inp = W.make_append(wl, 31 + len(name), contexts=ctx, shared_prefix=prefix, row_factors=factors)
    B = inp.new_k.shape[0]
    g = torch.Generator().manual_seed(5)
    q = torch.randn((B, wl.n_q, wl.num_q_heads, wl.head_dim), generator=g).to(torch.bfloat16)
    smp = W.make_sampler(wl, 77, batch=B)
    got = gpu_step(inp, q, smp, wl)
    ref = oracle_step(inp, q, smp, wl)
    # the attention bounds of every other parity test: bf16 max-abs 2e-2 and
    # rel-L2 5e-3, FP8 rel-L2 3e-2
    U.assert_attention_close(got["out"], ref["out"], fp8=wl.kv_fp8, what=f"{name} attention after append")
    assert np.array_equal(got["k"], ref["k"])
    ok = ~(got["near"] | ref["near"])
    assert np.array_equal(got["toks"][ok], ref["toks"][ok])
    assert np.array_equal(got["cl"], ref["cl"])
    assert got["ft"] == ref["ft"]
    # the same number of pages held per sequence, the same counts on them
    for b in range(B):
        gb, rb = got["bt"][b], ref["bt"][b]
        assert np.array_equal(gb >= 0, rb >= 0)
        assert np.array_equal(got["rc"][gb[gb >= 0]], ref["rc"][rb[rb >= 0]])
    assert got["gamma"] == ref["gamma"]
