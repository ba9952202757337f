"""GPU parity of svpa_gamma_update against the oracle: moving-average states,
draft lengths and telemetry, bit for bit (both sides make the same rounded
fp32 operations in the same order, and the batch uses integer totals)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_steps(ks, gammas, decay, r, with_seq=True):
    B = len(ks[0])
    ss = torch.zeros((B, 2), dtype=torch.float32, device=DEV) if with_seq else None
    sg = torch.zeros(B, dtype=torch.int32, device=DEV) if with_seq else None
    bs = torch.zeros(2, dtype=torch.float32, device=DEV)
    bg = torch.zeros(1, dtype=torch.int32, device=DEV)
    tel = torch.zeros(4, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_ss = np.zeros((B, 2), np.float32) if with_seq else None
    o_bs = np.zeros(2, np.float32)
    for k, g in zip(ks, gammas):
        kd = torch.as_tensor(np.asarray(k, np.int32), device=DEV)
        svpa.gamma_update(g, kd, bs, bg, tel, error_flag=err, seq_state=ss, seq_gamma=sg, decay=decay,
                          draft_cost_ratio=r)
        assert svpa.check_error(err) == 0
        ref = oracle.gamma_update(g, np.asarray(k, np.int32), seq_state=o_ss, batch_state=o_bs, decay=decay, r=r)
        o_ss, o_bs = ref["seq_state"], ref["batch_state"]
        if with_seq:
            assert np.array_equal(ss.cpu().numpy(), o_ss)
            assert np.array_equal(sg.cpu().numpy(), ref["seq_gamma"])
        assert np.array_equal(bs.cpu().numpy(), o_bs)
        assert int(bg.item()) == ref["batch_gamma"]
        assert np.array_equal(tel.cpu().numpy(), ref["telemetry"])


@pytest.mark.parametrize("B,decay", [(1, 0.9), (37, 0.8), (300, 0.95), (4099, 0.5)])
def test_gamma_update_matches_oracle(B, decay):
    rng = np.random.default_rng(B)
    alpha = rng.uniform(0.1, 0.95, B)
    ks, gs = [], []
    g = 4
    for step in range(12):
        passes = rng.random((B, g)) < alpha[:, None]
        ks.append(np.where(passes.all(1), g, np.argmin(passes, 1)).astype(np.int32))
        gs.append(g)
        g = [4, 5, 3, 1, 2, 4][step % 6]
    run_steps(ks, gs, decay, 0.08)
    run_steps(ks, gs, decay, 0.0, with_seq=False)


def test_collapse_and_recovery_on_device():
    ks = [[0, 5]] * 20 + [[1, 1]] * 20
    gs = [5] * 20 + [1] * 20
    run_steps(ks, gs, 0.8, 0.1)


def test_gamma_update_reads_the_sampler_output_in_place():
    wl = W.WORKLOADS["7b"]
    s = W.make_sampler(wl, W.SEEDS["7b"], device=DEV)
    B = s.p.shape[0]
    k = torch.empty(B, dtype=torch.int32, device=DEV)
    toks = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.zeros(svpa.spec_accept_workspace_size(B, s.p.shape[2]), dtype=torch.uint8, device=DEV)
    svpa.spec_accept(s.p, s.q, s.tokens, s.u_accept, s.u_sample, k, toks, workspace=ws, error_flag=err)
    ss = torch.zeros((B, 2), dtype=torch.float32, device=DEV)
    sg = torch.zeros(B, dtype=torch.int32, device=DEV)
    bs = torch.zeros(2, dtype=torch.float32, device=DEV)
    bg = torch.zeros(1, dtype=torch.int32, device=DEV)
    tel = torch.zeros(4, dtype=torch.float32, device=DEV)
    svpa.gamma_update(wl.gamma, k, bs, bg, tel, error_flag=err, seq_state=ss, seq_gamma=sg, draft_cost_ratio=0.08)
    assert svpa.check_error(err) == 0
    # the oracle's own sampler on the same rows gives the accepted lengths
    # (the kernel's are the same: its acceptance tests are bit-exact)
    ko, _, _, _ = oracle.spec_accept(s.p.cpu(), s.q.cpu(), s.tokens.cpu(), s.u_accept.cpu(), s.u_sample.cpu())
    assert np.array_equal(k.cpu().numpy(), ko)
    ref = oracle.gamma_update(wl.gamma, ko, seq_state=np.zeros((B, 2), np.float32), r=0.08)
    assert np.array_equal(sg.cpu().numpy(), ref["seq_gamma"])
    assert np.array_equal(tel.cpu().numpy(), ref["telemetry"])


def test_out_of_range_accepted_length_is_reported():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    bs = torch.tensor([1.0, 2.0], device=DEV)
    bg = torch.zeros(1, dtype=torch.int32, device=DEV)
    tel = torch.zeros(4, dtype=torch.float32, device=DEV)
    k = torch.tensor([1, 6, 2], dtype=torch.int32, device=DEV)
    svpa.gamma_update(4, k, bs, bg, tel, error_flag=err)
    assert svpa.check_error(err) == 1  # SVPA_DEVERR_BAD_VALUE maps to INVALID_ARG
    assert bs.cpu().tolist() == [1.0, 2.0]
