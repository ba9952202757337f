"""The device-side wait limit: a kernel whose mbarrier wait can never complete
(no thread arrives, no copy is in flight) gives up after the limit, raises
SVPA_DEVERR_TIMEOUT, frees its tensor memory and returns; svpa_check_error
maps that to SVPA_ERR_TIMEOUT and the GPU stays usable -- the next attention
call on the same device still matches the oracle."""
import numpy as np
import pytest
import torch

from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

import gpu_util as U

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SVPA_ERR_TIMEOUT = 7
SVPA_DEVERR_TIMEOUT = 2


def test_wait_runs_out_then_attention_still_matches_oracle():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    reached = torch.zeros(1, dtype=torch.int32, device=DEV)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    svpa.wait_selftest(1_000_000, err, reached)  # 1 ms
    b.record()
    assert svpa.check_error(err) == SVPA_ERR_TIMEOUT
    assert int(err.item()) & SVPA_DEVERR_TIMEOUT
    assert int(reached.item()) == 1  # the wait returned, as timed out
    ms = a.elapsed_time(b)
    assert 1.0 <= ms < 1000.0, ms
    # the same device, right after: an attention call matches the oracle
    inp = W.make_attention(W.WORKLOADS["70b"].scaled(batch=3, ctx_lo=100, ctx_hi=700), 515)
    got, lse, st = U.run_attention(inp, split_pages=16)
    assert st == 0
    ref, ref_lse = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, what="attention after a timed-out wait")
    assert np.max(np.abs(lse - ref_lse)) < 2e-3


def test_wait_selftest_rejects_bad_arguments():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert svpa.wait_selftest(0, err, err, check=False) == 1
    assert svpa.wait_selftest(20_000_000_000, err, err, check=False) == 1
    assert svpa.wait_selftest(1000, None, err, check=False) == 1
