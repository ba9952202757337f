"""The allocation-free attention entry point (svpa_paged_verify_attn_noalloc).

Callers that may not allocate device memory -- code inside a host framework
that owns every device allocation and forbids cudaMalloc on its hot path, or
plugin code handed only its input and output buffers -- use this entry point,
which takes its scratch from a fixed array inside the library instead of a
caller workspace.  The test calls it through the C ABI twice in a row (the
second call reuses the scratch the first one left behind) and checks both
results against the workspace entry point and against the oracle, within the
attention tolerances the other tests use.  This file is collected last.
"""
import numpy as np
import pytest
import torch

from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

import gpu_util as U

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2   # the bf16 attention tolerance of the parity tests
REL_L2 = 5e-3
FP8_REL_L2 = 3e-2


def _close(a, b, fp8=False):
    assert np.isfinite(a).all()
    if fp8:
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= FP8_REL_L2
    else:
        assert np.max(np.abs(a - b)) <= MAX_ABS
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= REL_L2


CASES = {
    # split KV at a forced size (partials and the merge go through the array)
    "7b_split": (W.WORKLOADS["7b"].scaled(batch=4, ctx_lo=50, ctx_hi=900), 16),
    "70b_split": (W.WORKLOADS["70b"].scaled(batch=4, ctx_lo=50, ctx_hi=900), 32),
    # unsplit units outnumbering the resident CTAs: the library's split size
    # keeps one split per unit and the units are handed out longest first, from
    # an order written into the array by a ranking kernel
    "7b_ordered": (W.WORKLOADS["7b"].scaled(batch=32, ctx_lo=20, ctx_hi=200), 0),
    # FP8 pages with per-page scales (tcgen05 kernel), the library's split size
    "fp8": (W.WORKLOADS["fp8"].scaled(batch=2, ctx_lo=300, ctx_hi=900), 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_workspace_entry_point(name):
    wl, split = CASES[name]
    dev = torch.device("cuda:0")
    inp = W.make_attention(wl, 321)
    B, n_q, Hq, D = inp.q.shape
    q, kp, vp = inp.q.to(dev), inp.k_pool.to(dev), inp.v_pool.to(dev)
    if wl.kv_fp8:
        kp, vp = kp.view(torch.uint8), vp.view(torch.uint8)
    ks = None if inp.k_scale is None else inp.k_scale.to(dev)
    vs = None if inp.v_scale is None else inp.v_scale.to(dev)
    bt, cl = inp.block_table.to(dev), inp.context_lens.to(dev)
    p = svpa.attn_params(B, n_q, Hq, wl.num_kv_heads, D, bt.shape[1], inp.num_blocks, kv_fp8=wl.kv_fp8,
                         split_pages=split)
    if name == "7b_ordered":
        assert svpa.attn_launches(p) == 2  # the ranking kernel runs: the ordered path
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    ws = torch.zeros(svpa.attn_workspace_size(p), dtype=torch.uint8, device=dev)
    ref = torch.empty((B, n_q, Hq, D), dtype=torch.bfloat16, device=dev)
    ref_lse = torch.empty((B, n_q, Hq), dtype=torch.float32, device=dev)
    svpa.paged_verify_attn(p, q, kp, vp, bt, cl, ref, workspace=ws, error_flag=err, lse=ref_lse,
                           k_scale=ks, v_scale=vs)
    assert svpa.check_error(err) == 0
    ref_np = ref.float().cpu().numpy()
    # the oracle on the same inputs (fp64 on the CPU)
    orc, _ = U.run_oracle_attention(inp)

    for _ in range(2):
        out = torch.full((B, n_q, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, n_q, Hq), float("nan"), dtype=torch.float32, device=dev)
        svpa.paged_verify_attn_noalloc(p, q, kp, vp, bt, cl, out, error_flag=err, lse=lse,
                                       k_scale=ks, v_scale=vs)
        assert svpa.check_error(err) == 0
        got = out.float().cpu().numpy()
        _close(got, ref_np, fp8=wl.kv_fp8)
        _close(got, orc, fp8=wl.kv_fp8)
        assert np.max(np.abs(lse.cpu().numpy() - ref_lse.cpu().numpy())) < 2e-3


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 70B-shape GQA at 64 sequences of up to 32k tokens needs far more than 32 MiB
    p = svpa.attn_params(64, 6, 64, 8, 128, 2049, 100000, split_pages=16)
    assert svpa.attn_workspace_size(p) > (32 << 20)
    st = svpa.paged_verify_attn_noalloc(p, None, None, None, None, None, None,
                                        error_flag=None, check=False)
    assert st == 6  # SVPA_ERR_WORKSPACE
