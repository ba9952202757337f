"""Pins for the oracle's paged verification attention (CPU only).

What the method computes is the masked softmax attention of each sequence's
n_q verification queries over its cached keys and values ("The
Sub-Millisecond Speculative Decoding Meltdown", section "Speculative Decoding
Mechanics & The K-Token Penalty": A = Softmax((Q K^T + M_tree)/sqrt(d_k)) V),
with the keys and values fetched page by page through a block table (same
page, section "Triton CUDA Fused Speculative Tree-Verification Kernel").

The oracle is pinned by things other than itself:
  * a library special case: torch's scaled_dot_product_attention in fp64 on
    tensors gathered here with torch indexing (an independent gather);
  * brute force on tiny inputs: pure-Python loops with exp() of the raw
    scores (no max subtraction) and math.fsum;
  * closed forms (all keys equal => mean of visible values; constant values;
    an empty history => the first query sees only itself);
  * invariance under relabelling of the physical blocks;
  * a draft-tree mask that is a chain equals the causal mask.
"""
import math

import numpy as np
import pytest
import torch

from speculative_verify_paged_attn_gb300 import workloads as W


def gathered_reference(inp: W.AttnInputs, fp8=False):
    """Independent reference: gather with torch indexing and call SDPA in fp64."""
    wl = inp.wl
    B, n_q, Hq, D = inp.q.shape
    G = Hq // wl.num_kv_heads
    outs = []
    for b in range(B):
        L = int(inp.context_lens[b])
        T = L + n_q
        p = torch.arange(T)
        blk = inp.block_table[b, p // W.BLOCK_SIZE].long()
        slot = p % W.BLOCK_SIZE
        if fp8:
            k = inp.k_pool[blk, :, slot, :].to(torch.float64) * inp.k_scale[blk].double()[:, :, None]
            v = inp.v_pool[blk, :, slot, :].to(torch.float64) * inp.v_scale[blk].double()[:, :, None]
        else:
            k = inp.k_pool[blk, :, slot, :].to(torch.float64)      # [T, Hkv, D]
            v = inp.v_pool[blk, :, slot, :].to(torch.float64)
        k = k.permute(1, 0, 2).repeat_interleave(G, dim=0)          # [Hq, T, D]
        v = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
        q = inp.q[b].to(torch.float64).permute(1, 0, 2)            # [Hq, n_q, D]
        mask = torch.zeros((n_q, T), dtype=torch.bool)
        mask[:, :L] = True
        for j in range(n_q):
            for i in range(n_q):
                if inp.ancestor_mask is not None:
                    vis = (int(inp.ancestor_mask[j]) >> i) & 1
                else:
                    vis = i <= j
                mask[j, L + i] = bool(vis)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=wl.sm_scale)
        outs.append(o.permute(1, 0, 2))
    return torch.stack(outs).numpy()


def run_oracle(oracle_mod, inp: W.AttnInputs):
    wl = inp.wl
    return oracle_mod.paged_verify_attn(
        inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.context_lens,
        num_kv_heads=wl.num_kv_heads, sm_scale=wl.sm_scale, kv_fp8=wl.kv_fp8,
        k_scale=inp.k_scale, v_scale=inp.v_scale,
        ancestor_mask=None if inp.ancestor_mask is None else inp.ancestor_mask.numpy().view(np.uint64))


def test_tiny_matches_sdpa(oracle_mod):
    inp = W.make_attention(W.WORKLOADS["tiny"], W.SEEDS["tiny"])
    out, lse = run_oracle(oracle_mod, inp)
    ref = gathered_reference(inp)
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("name", ["7b", "70b", "tree"])
def test_scaled_shapes_match_sdpa(oracle_mod, name):
    wl = W.WORKLOADS[name].scaled(batch=3, ctx_lo=20, ctx_hi=90, shared_prefix=min(W.WORKLOADS[name].shared_prefix, 32))
    inp = W.make_attention(wl, 77)
    out, _ = run_oracle(oracle_mod, inp)
    ref = gathered_reference(inp)
    assert np.max(np.abs(out - ref)) < 1e-11


def test_fp8_matches_sdpa_on_decoded_pages(oracle_mod):
    wl = W.WORKLOADS["fp8"].scaled(batch=2, ctx_lo=40, ctx_hi=70, fixed_contexts=None)
    inp = W.make_attention(wl, 5)
    out, _ = run_oracle(oracle_mod, inp)
    ref = gathered_reference(inp, fp8=True)
    assert np.max(np.abs(out - ref)) < 1e-11


def test_lse_matches_logsumexp(oracle_mod):
    wl = W.WORKLOADS["tiny"].scaled(batch=2, fixed_contexts=(3, 17))
    inp = W.make_attention(wl, 3)
    _, lse = run_oracle(oracle_mod, inp)
    b, j, h = 1, 2, 3
    L = int(inp.context_lens[b])
    T = L + wl.n_q
    scores = []
    for p in range(T):
        if p >= L and p - L > j:
            continue
        blk = int(inp.block_table[b, p // 16])
        k = inp.k_pool[blk, h, p % 16].double()
        scores.append(float((inp.q[b, j, h].double() * k).sum()) * wl.sm_scale)
    assert abs(lse[b, j, h] - math.log(math.fsum(math.exp(s) for s in scores))) < 1e-12


def brute_force(inp: W.AttnInputs):
    """Pure-Python triple loop, exp of raw scores, fsum; no numpy, no max-shift."""
    wl = inp.wl
    B, n_q, Hq, D = inp.q.shape
    G = Hq // wl.num_kv_heads
    qf = inp.q.double().tolist()
    kf = inp.k_pool.double().tolist()
    vf = inp.v_pool.double().tolist()
    out = np.zeros((B, n_q, Hq, D))
    for b in range(B):
        L = int(inp.context_lens[b])
        for h in range(Hq):
            g = h // G
            for j in range(n_q):
                ws, rows = [], []
                for p in range(L + n_q):
                    if p >= L and (p - L) > j:
                        continue
                    blk = int(inp.block_table[b, p // 16])
                    krow = kf[blk][g][p % 16]
                    s = math.fsum(qf[b][j][h][d] * krow[d] for d in range(D)) * wl.sm_scale
                    ws.append(math.exp(s))
                    rows.append(vf[blk][g][p % 16])
                z = math.fsum(ws)
                for d in range(D):
                    out[b, j, h, d] = math.fsum(w * r[d] for w, r in zip(ws, rows)) / z
    return out


def test_brute_force_tiny(oracle_mod):
    wl = W.WORKLOADS["tiny"].scaled(head_dim=8, num_q_heads=4, num_kv_heads=2,
                                    fixed_contexts=(0, 5, 21, 40), batch=4, fixed_pool_blocks=None)
    inp = W.make_attention(wl, 11)
    out, _ = run_oracle(oracle_mod, inp)
    assert np.max(np.abs(out - brute_force(inp))) < 1e-12


def test_block_permutation_invariance(oracle_mod):
    wl = W.WORKLOADS["70b"].scaled(batch=3, ctx_lo=30, ctx_hi=80, head_dim=64)
    inp = W.make_attention(wl, 21, poison=False)
    out1, lse1 = run_oracle(oracle_mod, inp)
    nb = inp.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(9))
    # relabel: new block id perm[old]; move the pages accordingly
    kp = torch.empty_like(inp.k_pool)
    vp = torch.empty_like(inp.v_pool)
    kp[perm] = inp.k_pool
    vp[perm] = inp.v_pool
    bt = inp.block_table.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    inp2 = W.AttnInputs(**{**inp.__dict__, "k_pool": kp, "v_pool": vp, "block_table": bt})
    out2, lse2 = run_oracle(oracle_mod, inp2)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)


def test_closed_form_equal_keys(oracle_mod):
    # all keys equal => uniform weights => output = mean of the visible values
    wl = W.WORKLOADS["tiny"].scaled(fixed_contexts=(9, 30))
    inp = W.make_attention(wl, 4, poison=False)
    inp.k_pool[:] = inp.k_pool[0, 0, 0]
    out, _ = run_oracle(oracle_mod, inp)
    b, j, h = 1, 3, 2
    L = int(inp.context_lens[b])
    vals = []
    for p in range(L + j + 1):
        blk = int(inp.block_table[b, p // 16])
        vals.append(inp.v_pool[blk, h, p % 16].double().numpy())
    assert np.max(np.abs(out[b, j, h] - np.mean(vals, axis=0))) < 1e-12


def test_closed_form_constant_values(oracle_mod):
    wl = W.WORKLOADS["tiny"].scaled(fixed_contexts=(9, 30))
    inp = W.make_attention(wl, 4, poison=False)
    row = inp.v_pool[3, 1, 5].clone()
    inp.v_pool[:] = row
    out, _ = run_oracle(oracle_mod, inp)
    assert np.max(np.abs(out - row.double().numpy())) < 1e-12


def test_empty_history_first_query_sees_itself(oracle_mod):
    wl = W.WORKLOADS["tiny"].scaled(fixed_contexts=(0, 0))
    inp = W.make_attention(wl, 8)
    out, _ = run_oracle(oracle_mod, inp)
    for b in range(2):
        blk = int(inp.block_table[b, 0])
        assert np.array_equal(out[b, 0], inp.v_pool[blk, :, 0].double().numpy())


def test_chain_tree_mask_equals_causal(oracle_mod):
    wl = W.WORKLOADS["7b"].scaled(batch=2, ctx_lo=10, ctx_hi=40, head_dim=64, num_q_heads=4,
                                  num_kv_heads=4)
    inp = W.make_attention(wl, 13)
    out1, _ = run_oracle(oracle_mod, inp)
    chain = [-1, 0, 1, 2, 3]
    am = torch.tensor(W.ancestor_masks(chain), dtype=torch.int64)
    inp2 = W.AttnInputs(**{**inp.__dict__, "ancestor_mask": am})
    out2, _ = run_oracle(oracle_mod, inp2)
    assert np.array_equal(out1, out2)


def test_rejects_bad_block(oracle_mod):
    wl = W.WORKLOADS["tiny"]
    inp = W.make_attention(wl, 1)
    inp.block_table[0, 0] = inp.num_blocks
    with pytest.raises(oracle_mod.OracleError):
        run_oracle(oracle_mod, inp)


def tile_scaled_reference(inp: W.AttnInputs):
    """SDPA in fp64 on pages decoded with one scale per 64-element tile of a
    row: the scale array [blocks, Hkv, 16, D/64] is broadcast to full rows."""
    ks = inp.k_scale.double().repeat_interleave(64, dim=3)  # [blocks, Hkv, 16, D]
    vs = inp.v_scale.double().repeat_interleave(64, dim=3)
    k = inp.k_pool.to(torch.float64) * ks
    v = inp.v_pool.to(torch.float64) * vs
    # the same gather as the per-page reference, on already decoded pages
    dec = W.AttnInputs(wl=inp.wl.scaled(kv_fp8=False, scale_tile=0), q=inp.q, k_pool=k, v_pool=v,
                       k_scale=None, v_scale=None, block_table=inp.block_table,
                       context_lens=inp.context_lens, ancestor_mask=inp.ancestor_mask,
                       refcount=inp.refcount, free_stack=inp.free_stack, free_top=inp.free_top)
    return gathered_reference(dec)


def run_oracle_tiles(oracle_mod, inp: W.AttnInputs):
    wl = inp.wl
    return oracle_mod.paged_verify_attn(
        inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.context_lens,
        num_kv_heads=wl.num_kv_heads, sm_scale=wl.sm_scale, kv_fp8=True, k_scale=inp.k_scale,
        v_scale=inp.v_scale, scale_tile=64,
        ancestor_mask=None if inp.ancestor_mask is None else inp.ancestor_mask.numpy().view(np.uint64))


@pytest.mark.parametrize("name", ["fp8", "tree"])
def test_fp8_tile_scales_match_sdpa(oracle_mod, name):
    # one scale per 64 consecutive elements of a token's row: a swapped slot,
    # head or tile index in the oracle's decode would change the values
    base = W.WORKLOADS[name]
    wl = base.scaled(batch=3, ctx_lo=20, ctx_hi=90, fixed_contexts=None, kv_fp8=True, scale_tile=64,
                     shared_prefix=min(base.shared_prefix, 32))
    inp = W.make_attention(wl, 9)
    assert tuple(inp.k_scale.shape[2:]) == (16, wl.head_dim // 64)
    # the tile scales really differ within every page a sequence maps
    used = inp.block_table[inp.block_table >= 0].long().unique()
    assert inp.k_scale[used].std(dim=(2, 3)).min() > 0
    out, _ = run_oracle_tiles(oracle_mod, inp)
    ref = tile_scaled_reference(inp)
    assert np.max(np.abs(out - ref)) < 1e-11


def test_fp8_tile_scales_equal_to_page_scale_reduce_to_per_page(oracle_mod):
    wl = W.WORKLOADS["fp8"].scaled(batch=2, ctx_lo=40, ctx_hi=70, fixed_contexts=None)
    inp = W.make_attention(wl, 5)
    out_page, _ = run_oracle(oracle_mod, inp)
    tiles = W.AttnInputs(**{**inp.__dict__,
                            "k_scale": inp.k_scale[:, :, None, None].expand(-1, -1, 16, 2).contiguous(),
                            "v_scale": inp.v_scale[:, :, None, None].expand(-1, -1, 16, 2).contiguous()})
    out_tile, _ = run_oracle_tiles(oracle_mod, tiles)
    assert np.array_equal(out_page, out_tile)
