"""A whole verification step captured in one CUDA graph and replayed gives the
results of the same step run eagerly: the entry points enqueue only device
work on the caller's stream (after the first call on a device), so a serving
loop can capture a step once and replay it.  The K/V append's second kernel
is a programmatic dependent launch, which the capture must keep."""
import numpy as np
import pytest
import torch

from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


class StepState:
    def __init__(self, wl, seed):
        inp = W.make_append(wl, seed, contexts=(3, 40, 77, 200, 9, 500), shared_prefix=19, device=DEV)
        self.inp, self.wl = inp, wl
        self.fp8 = wl.kv_fp8
        self.kp = inp.k_pool.view(torch.uint8) if self.fp8 else inp.k_pool
        self.vp = inp.v_pool.view(torch.uint8) if self.fp8 else inp.v_pool
        self.saved = {n: getattr(inp, n).clone() for n in ("block_table", "context_lens", "refcount", "free_stack")}
        self.pools = [t.clone() for t in (self.kp, self.vp)]
        self.scales = [t.clone() for t in (inp.k_scale, inp.v_scale)] if self.fp8 else []
        self.ft0 = torch.tensor([inp.free_top], dtype=torch.int32, device=DEV)
        self.ft = self.ft0.clone()
        B = inp.new_k.shape[0]
        g = torch.Generator(device=DEV)
        g.manual_seed(seed + 1)
        self.q = torch.randn((B, wl.n_q, wl.num_q_heads, wl.head_dim), generator=g, device=DEV).to(torch.bfloat16)
        self.smp = W.make_sampler(wl, seed, device=DEV, batch=B)
        self.params = svpa.attn_params(B, wl.n_q, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                       inp.block_table.shape[1], self.kp.shape[0], kv_fp8=self.fp8,
                                       sm_scale=wl.sm_scale)
        self.ws = torch.zeros(svpa.attn_workspace_size(self.params), dtype=torch.uint8, device=DEV)
        self.sws = torch.zeros(svpa.spec_accept_workspace_size(B, self.smp.p.shape[2]), dtype=torch.uint8,
                               device=DEV)
        self.out = torch.empty((B, wl.n_q, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=DEV)
        self.k = torch.empty(B, dtype=torch.int32, device=DEV)
        self.toks = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device=DEV)
        self.gs = torch.zeros((B, 2), dtype=torch.float32, device=DEV)
        self.gq = torch.zeros(B, dtype=torch.int32, device=DEV)
        self.gb = torch.zeros(2, dtype=torch.float32, device=DEV)
        self.gg = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.tel = torch.zeros(4, dtype=torch.float32, device=DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)

    def restore(self):
        for n, t in self.saved.items():
            getattr(self.inp, n).copy_(t)
        for dst, src in zip((self.kp, self.vp), self.pools):
            dst.copy_(src)
        if self.fp8:
            for dst, src in zip((self.inp.k_scale, self.inp.v_scale), self.scales):
                dst.copy_(src)
        self.ft.copy_(self.ft0)
        for t in (self.gs, self.gb):
            t.zero_()

    def step(self):
        inp, s, wl = self.inp, self.smp, self.wl
        svpa.kv_append(inp.new_k, inp.new_v, inp.block_table, inp.context_lens, inp.refcount, inp.free_stack,
                       self.ft, self.kp, self.vp, error_flag=self.err, k_scale=inp.k_scale, v_scale=inp.v_scale)
        svpa.paged_verify_attn(self.params, self.q, self.kp, self.vp, inp.block_table, inp.context_lens, self.out,
                               workspace=self.ws, error_flag=self.err, k_scale=inp.k_scale, v_scale=inp.v_scale)
        svpa.spec_accept(s.p, s.q, s.tokens, s.u_accept, s.u_sample, self.k, self.toks, workspace=self.sws,
                         error_flag=self.err)
        svpa.block_table_commit(wl.n_q, inp.block_table, inp.context_lens, self.k, inp.refcount, inp.free_stack,
                                self.ft, error_flag=self.err)
        svpa.gamma_update(wl.gamma, self.k, self.gb, self.gg, self.tel, error_flag=self.err, seq_state=self.gs,
                          seq_gamma=self.gq)

    def results(self):
        return dict(out=self.out.clone(), k=self.k.clone(), toks=self.toks.clone(),
                    cl=self.inp.context_lens.clone(), ft=self.ft.clone(), gq=self.gq.clone(),
                    gb=self.gb.clone(), tel=self.tel.clone())


@pytest.mark.parametrize("name", ["7b", "fp8"])
def test_step_replayed_from_a_cuda_graph_matches_eager(name):
    wl = W.WORKLOADS[name].scaled(num_q_heads=16 if name == "7b" else 64,
                                  num_kv_heads=16 if name == "7b" else 8, vocab=3000)
    st = StepState(wl, 61)
    st.restore()
    st.step()  # eager, also settles the per-device launch facts
    torch.cuda.synchronize()
    assert svpa.check_error(st.err) == 0
    eager = st.results()

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    st.restore()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        st.step()
    for _ in range(2):  # the same step replayed on the restored state
        st.restore()
        graph.replay()
        torch.cuda.synchronize()
        assert svpa.check_error(st.err) == 0
        got = st.results()
        assert torch.equal(got["out"], eager["out"])
        for key in ("k", "toks", "cl", "ft", "gq", "gb", "tel"):
            assert torch.equal(got[key], eager[key]), key
