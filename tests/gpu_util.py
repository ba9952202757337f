"""Helpers shared by the GPU parity tests: run the CUDA library through its
C ABI, run the oracle on the same seeded inputs, and compare."""
import numpy as np
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

DEV = torch.device("cuda:0")

# Attention tolerances (output in bf16, fp32 accumulation, fp64 oracle)
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
FP8_REL_L2 = 3e-2


def to_dev(inp: W.AttnInputs) -> W.AttnInputs:
    d = dict(inp.__dict__)
    for k, v in d.items():
        if isinstance(v, torch.Tensor):
            d[k] = v.to(DEV)
    return W.AttnInputs(**d)


def to_cpu(inp: W.AttnInputs) -> W.AttnInputs:
    d = dict(inp.__dict__)
    for k, v in d.items():
        if isinstance(v, torch.Tensor):
            d[k] = v.cpu()
    return W.AttnInputs(**d)


def mask_list(inp):
    return None if inp.ancestor_mask is None else [int(x) for x in inp.ancestor_mask.cpu().tolist()]


def run_attention(inp: W.AttnInputs, split_pages=0, with_lse=True, variant=0):
    """Returns (out fp32 numpy [B, n_q, Hq, D], lse numpy or None, device error status)."""
    wl = inp.wl
    d = to_dev(inp)
    B, n_q, Hq, D = d.q.shape
    p = svpa.attn_params(B, n_q, Hq, wl.num_kv_heads, D, d.block_table.shape[1], d.num_blocks,
                         kv_fp8=wl.kv_fp8, sm_scale=wl.sm_scale, split_pages=split_pages,
                         variant=variant, scale_tile=wl.scale_tile)
    ws = torch.zeros(svpa.attn_workspace_size(p), dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.full((B, n_q, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, n_q, Hq), float("nan"), dtype=torch.float32, device=DEV) if with_lse else None
    kp = d.k_pool.view(torch.uint8) if wl.kv_fp8 else d.k_pool
    vp = d.v_pool.view(torch.uint8) if wl.kv_fp8 else d.v_pool
    svpa.paged_verify_attn(p, d.q, kp, vp, d.block_table, d.context_lens, out, workspace=ws,
                           error_flag=err, k_scale=d.k_scale, v_scale=d.v_scale,
                           ancestor_mask=mask_list(inp), lse=lse)
    st = svpa.check_error(err)
    # the scheduler counters and tickets are left at zero for the next call
    words = ws[: 256 + B * wl.num_kv_heads * 4].view(torch.int32)
    assert int(words[:2].abs().sum().item()) == 0
    assert int(words[64:].abs().sum().item()) == 0
    return out.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None), st


def run_oracle_attention(inp: W.AttnInputs):
    c = to_cpu(inp)
    wl = c.wl
    am = None if c.ancestor_mask is None else c.ancestor_mask.numpy().view(np.uint64)
    return oracle.paged_verify_attn(c.q, c.k_pool, c.v_pool, c.block_table, c.context_lens,
                                    num_kv_heads=wl.num_kv_heads, sm_scale=wl.sm_scale,
                                    kv_fp8=wl.kv_fp8, k_scale=c.k_scale, v_scale=c.v_scale,
                                    ancestor_mask=am, scale_tile=wl.scale_tile)


def rel_l2(a, b):
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


def assert_attention_close(got, ref, fp8=False, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.max(np.abs(got - ref))
    rl = rel_l2(got, ref)
    if fp8:
        assert rl <= FP8_REL_L2, f"{what}: rel-L2 {rl}"
    else:
        assert err <= BF16_MAX_ABS, f"{what}: max-abs {err}"
        assert rl <= BF16_REL_L2, f"{what}: rel-L2 {rl}"
    return err, rl


def subset(inp: W.AttnInputs, seqs) -> W.AttnInputs:
    """The selected sequences with a compacted pool holding only their pages
    (so the oracle need not copy a multi-GB pool to the host)."""
    seqs = list(seqs)
    bt = inp.block_table[seqs]
    used = torch.unique(bt[bt >= 0])
    remap = torch.full((inp.num_blocks,), -1, dtype=torch.int32, device=bt.device)
    remap[used.long()] = torch.arange(used.numel(), dtype=torch.int32, device=bt.device)
    nbt = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], bt)
    d = dict(inp.__dict__)
    d.update(q=inp.q[seqs], block_table=nbt, context_lens=inp.context_lens[seqs],
             k_pool=inp.k_pool[used.long()], v_pool=inp.v_pool[used.long()],
             k_scale=None if inp.k_scale is None else inp.k_scale[used.long()],
             v_scale=None if inp.v_scale is None else inp.v_scale[used.long()],
             refcount=inp.refcount[used.long()], free_stack=inp.free_stack[:0], free_top=0)
    return to_cpu(W.AttnInputs(**d))
