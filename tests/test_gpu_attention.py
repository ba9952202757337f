"""GPU parity of svpa_paged_verify_attn against the fp64 oracle.

Tolerances: bf16 K/V max-abs 2e-2 and rel-L2 5e-3; FP8 K/V rel-L2 3e-2
(against the oracle run on the same FP8 bytes and scales).  Small cases span
several pages, several KV splits and ragged last pages; the full-size
workloads run in the launch configuration the benchmark times and are checked
on sampled sequences.
"""
import numpy as np
import pytest
import torch

from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu

import gpu_util as U  # noqa: E402


def small(name, **kw):
    base = W.WORKLOADS[name]
    return base.scaled(**kw)


CASES = [
    ("tiny", W.WORKLOADS["tiny"], 0),
    ("tiny_split2", W.WORKLOADS["tiny"], 2),
    ("7b_small", small("7b", batch=5, ctx_lo=1, ctx_hi=700), 16),
    ("7b_small_auto", small("7b", batch=5, ctx_lo=1, ctx_hi=700), 0),
    ("70b_small", small("70b", batch=3, ctx_lo=200, ctx_hi=1500), 32),
    ("fp8_small", small("fp8", batch=2, ctx_lo=300, ctx_hi=1200), 16),
    # one FP8 scale per 64-element tile of a row (tcgen05 kernel)
    ("fp8_t64_small", small("fp8_t64", batch=3, ctx_lo=1, ctx_hi=900), 16),
    ("fp8_t64_nosplit", small("fp8_t64", batch=2, ctx_lo=100, ctx_hi=300), 1024),
    ("fp8_t64_g4", small("fp8_t64", batch=3, ctx_lo=40, ctx_hi=700, num_q_heads=32, num_kv_heads=8), 8),
    ("tree_small", small("tree", batch=4, ctx_lo=1, ctx_hi=400, shared_prefix=32), 16),
    ("tree_prefix800", small("tree", batch=3, ctx_lo=1024, ctx_hi=1300), 32),
    ("d64_gqa", small("tiny", num_q_heads=8, num_kv_heads=2, fixed_contexts=None, ctx_lo=0, ctx_hi=300,
                      batch=6, fixed_pool_blocks=None), 4),
]


@pytest.mark.parametrize("name,wl,split", CASES, ids=[c[0] for c in CASES])
def test_small_parity(name, wl, split):
    inp = W.make_attention(wl, 100 + len(name))
    got, lse, st = U.run_attention(inp, split_pages=split)
    assert st == 0
    ref, ref_lse = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, fp8=wl.kv_fp8, what=name)
    assert np.max(np.abs(lse - ref_lse)) < 2e-3


def test_block_permutation_gives_identical_bits():
    wl = small("70b", batch=3, ctx_lo=50, ctx_hi=600)
    inp = W.make_attention(wl, 7)
    out1, _, st = U.run_attention(inp, split_pages=8)
    assert st == 0
    nb = inp.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3))
    kp = torch.empty_like(inp.k_pool)
    vp = torch.empty_like(inp.v_pool)
    kp[perm] = inp.k_pool
    vp[perm] = inp.v_pool
    bt = inp.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    inp2 = W.AttnInputs(**{**inp.__dict__, "k_pool": kp, "v_pool": vp, "block_table": bt})
    out2, _, st = U.run_attention(inp2, split_pages=8)
    assert st == 0
    assert np.array_equal(out1, out2)


def test_split_size_invariance():
    wl = small("7b", batch=4, ctx_lo=300, ctx_hi=900)
    inp = W.make_attention(wl, 8)
    ref, _ = U.run_oracle_attention(inp)
    outs = []
    for sp in (16, 32, 64, 1024):
        o, _, st = U.run_attention(inp, split_pages=sp)
        assert st == 0
        U.assert_attention_close(o, ref, what=f"split {sp}")
        outs.append(o)
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 2e-2


def test_edge_lengths():
    # empty history, exact page multiples, one token short of a page
    wl = small("7b", batch=6, num_q_heads=8, num_kv_heads=8)
    inp = W.make_attention(wl, 9, contexts=[0, 11, 27, 43, 15, 1])
    got, _, st = U.run_attention(inp, split_pages=1)
    assert st == 0
    ref, _ = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, what="edges")


def test_single_query():
    wl = small("70b", gamma=0, batch=3, ctx_lo=5, ctx_hi=200)
    inp = W.make_attention(wl, 10)
    got, _, st = U.run_attention(inp, split_pages=4)
    assert st == 0
    ref, _ = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, what="n_q=1")


def test_bad_block_reported_not_faulted():
    inp = W.make_attention(W.WORKLOADS["tiny"], 11)
    inp.block_table[1, 2] = inp.num_blocks + 5
    _, _, st = U.run_attention(inp, split_pages=2)
    assert st == 5  # SVPA_ERR_BAD_BLOCK


FULL = ["7b", "70b", "fp8", "tree", "fp8_t64"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    wl = W.WORKLOADS[name]
    inp = W.make_attention(wl, W.SEEDS[name], device="cuda", poison=True)
    got, lse, st = U.run_attention(inp)
    assert st == 0
    assert np.isfinite(got).all()
    B = got.shape[0]
    rng = np.random.default_rng(0)
    seqs = sorted(set([0, B - 1] + list(rng.choice(B, size=2, replace=False))))
    sub = U.subset(inp, seqs)
    ref, ref_lse = U.run_oracle_attention(sub)
    U.assert_attention_close(got[seqs], ref, fp8=wl.kv_fp8, what=f"{name} sampled")
    assert np.max(np.abs(lse[seqs] - ref_lse)) < 5e-3
    del inp
    torch.cuda.empty_cache()


# Both kernels on the shapes where the library picks the tcgen05/TMEM one
# (many rows per kv head) and on a multi-head shape: 1 = warp-level MMA,
# 2 = tcgen05 with TMEM accumulators.
VARIANT_CASES = [
    ("gqa", small("70b", batch=3, ctx_lo=1, ctx_hi=900), 16),
    ("gqa_nosplit", small("70b", batch=2, ctx_lo=100, ctx_hi=300), 1024),
    ("tree", small("tree", batch=3, ctx_lo=1, ctx_hi=500, shared_prefix=32), 8),
    ("mha", small("7b", batch=3, ctx_lo=1, ctx_hi=300, num_q_heads=8, num_kv_heads=8), 8),
    ("fp8", small("fp8", batch=3, ctx_lo=1, ctx_hi=900), 16),
    ("fp8_nosplit", small("fp8", batch=2, ctx_lo=100, ctx_hi=300), 1024),
    ("fp8_g4", small("fp8", batch=3, ctx_lo=40, ctx_hi=700, num_q_heads=32, num_kv_heads=8), 8),
    # FP8 tensor-core kernel at other row counts: 64 rows (gamma 7, G 8), 12
    # rows (G 2, MMA N 16), 40 rows (gamma 4: rows 40..47 of the N = 48 tile
    # are padding)
    ("fp8_m64", small("fp8", gamma=7, batch=2, ctx_lo=1, ctx_hi=700), 16),
    ("fp8_m12", small("fp8", num_q_heads=16, num_kv_heads=8, batch=3, ctx_lo=1, ctx_hi=600), 8),
    ("fp8_m40", small("fp8", gamma=4, batch=3, ctx_lo=30, ctx_hi=500), 0),
]


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("name,wl,split", VARIANT_CASES, ids=[c[0] for c in VARIANT_CASES])
def test_kernel_variants(name, wl, split, variant):
    inp = W.make_attention(wl, 200 + len(name))
    got, lse, st = U.run_attention(inp, split_pages=split, variant=variant)
    assert st == 0
    ref, ref_lse = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, fp8=wl.kv_fp8, what=f"{name} variant {variant}")
    assert np.max(np.abs(lse - ref_lse)) < 2e-3


def test_fp8_page_scales_wide_range():
    # K and V page scales spread over eight decades and a few zero V scales:
    # the warp-level kernel applies the scales in fp32 and takes any of them;
    # the tcgen05 kernel (one scale per page) takes any K scale and V scales
    # up to 255 (its documented contract; larger ones are reported, see the
    # next test)
    wl = small("fp8", batch=3, ctx_lo=100, ctx_hi=900)
    inp = W.make_attention(wl, 17)
    g = torch.Generator().manual_seed(23)
    fk = 10.0 ** (torch.rand(inp.k_scale.shape, generator=g) * 8 - 3)
    fv = 10.0 ** (torch.rand(inp.v_scale.shape, generator=g) * 8 - 3)
    fv[torch.rand(inp.v_scale.shape, generator=g) < 0.05] = 0.0
    base_k, base_v = inp.k_scale.clone(), inp.v_scale.clone()
    inp.k_scale = (base_k * fk).contiguous()
    inp.v_scale = (base_v * fv).contiguous()
    assert float(inp.v_scale.max()) > 146 and float(inp.k_scale.max()) > 146
    got, _, st = U.run_attention(inp, split_pages=8, variant=1)
    assert st == 0
    ref, _ = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, fp8=True, what="wide scales, warp-level kernel")
    # the same spread, V scales capped at 255, on the tcgen05 kernel
    inp.v_scale = (base_v * fv).clamp(max=255.0).contiguous()
    got, _, st = U.run_attention(inp, split_pages=8, variant=2)
    assert st == 0
    ref, _ = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, fp8=True, what="K scales to 1e5, V scales to 255, tcgen05 kernel")


def test_fp8_query_rows_of_any_magnitude():
    # the tcgen05 kernel splits each query row into two E4M3 terms at a
    # power-of-two scale of its own: rows of very different norms (1e-4 ..
    # 1e4 times N(0, 1)) keep their relative accuracy
    wl = small("fp8", batch=3, ctx_lo=100, ctx_hi=900)
    inp = W.make_attention(wl, 19)
    g = torch.Generator().manual_seed(29)
    B, n_q, Hq, D = inp.q.shape
    f = 10.0 ** (torch.rand((B, n_q, Hq, 1), generator=g) * 8 - 4)
    inp.q = (inp.q.float() * f).to(torch.bfloat16).contiguous()
    got, lse, st = U.run_attention(inp, variant=2)
    assert st == 0
    ref, ref_lse = U.run_oracle_attention(inp)
    U.assert_attention_close(got, ref, fp8=True, what="query rows over eight decades, tcgen05 kernel")
    # the log-sum-exp is relative to the scores' scale here
    assert np.max(np.abs(lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse))) < 2e-3


def test_fp8_even_split_mixed_lengths():
    # the tcgen05 kernel for per-page FP8 scales splits all blocks evenly over
    # the SMs: sequences of mixed lengths (some shorter than one block, some
    # cut into several pieces) and a batch whose blocks are fewer than the SMs
    for seed, kw in ((31, dict(batch=9, ctx_lo=0, ctx_hi=6000)), (37, dict(batch=2, ctx_lo=1, ctx_hi=40)),
                     (41, dict(batch=5, ctx_lo=20000, ctx_hi=40000))):
        inp = W.make_attention(small("fp8", **kw), seed)
        got, lse, st = U.run_attention(inp, variant=2)
        assert st == 0
        ref, ref_lse = U.run_oracle_attention(inp)
        U.assert_attention_close(got, ref, fp8=True, what=f"even split, {kw}")
        assert np.max(np.abs(lse - ref_lse)) < 2e-3


def test_fp8_scale_beyond_f16_range_reported_on_tcgen05():
    wl = small("fp8", batch=2, ctx_lo=100, ctx_hi=300)
    inp = W.make_attention(wl, 18)
    inp.v_scale = inp.v_scale.clone()
    inp.v_scale[inp.block_table[0, 0].long(), 0] = 500.0
    _, _, st = U.run_attention(inp, split_pages=8, variant=2)
    assert st == 1  # SVPA_DEVERR_BAD_VALUE maps to SVPA_ERR_INVALID_ARG
