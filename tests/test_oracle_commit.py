"""Pins for the oracle's block-table commit / rollback (CPU only).

Semantics: accepted tokens are committed to the block table, the KV blocks of
rejected tokens are discarded ("LOW-LATENCY INFERENCE: SPECULATIVE DECODING &
PAGING", architecture diagram); a dropped block's reference count falls by
one and the block returns to the free pool when it reaches zero
("Speculative Decoding & KV-Cache PagedAttention in Enterprise LLM Serving",
PagedKVCacheManager.ReleaseSession; shared prefix blocks carry a count equal
to the number of holders).
"""
import json
import os

import numpy as np
import torch

from speculative_verify_paged_attn_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hand_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "commit_worked_example.json")))
    r = oracle_mod.block_table_commit(np.array(g["block_table"]), np.array(g["context_lens"]),
                                      np.array(g["accepted_len"]), np.array(g["refcount"]),
                                      np.array(g["free_stack"]), g["free_top"], n_q=g["n_q"],
                                      block_size=g["block_size"])
    e = g["expect"]
    assert r["block_table"].tolist() == e["block_table"]
    assert r["context_lens"].tolist() == e["context_lens"]
    assert r["refcount"].tolist() == e["refcount"]
    assert r["free_top"] == e["free_top"]
    assert sorted(r["free_stack"][:r["free_top"]].tolist()) == e["free_stack_multiset"]


def invariants(bt, cl, rc, fs, ft, num_blocks, shared=()):
    held = {}
    for row in bt:
        for blk in row:
            if blk >= 0:
                held[int(blk)] = held.get(int(blk), 0) + 1
    free = fs[:ft].tolist()
    assert len(set(free)) == len(free)
    # conservation: every block is either referenced or free, never both
    assert sum(1 for b in range(num_blocks) if rc[b] > 0) + ft == num_blocks
    for b in range(num_blocks):
        assert rc[b] >= 0
        assert (rc[b] == 0) == (b in free)
        assert rc[b] >= held.get(b, 0)
    # each sequence holds exactly ceil(len / 16) leading pages
    for row, L in zip(bt, cl):
        n = -(-int(L) // 16)
        assert np.all(row[:n] >= 0) and np.all(row[n:] == -1)
    for blk in shared:
        assert rc[blk] > 0


def test_random_rollbacks_conserve_blocks(oracle_mod):
    wl = W.WORKLOADS["7b"].scaled(batch=40, ctx_lo=1, ctx_hi=200, head_dim=8, num_q_heads=2,
                                  num_kv_heads=2)
    inp = W.make_attention(wl, 17, poison=False)
    rng = np.random.default_rng(0)
    k = rng.integers(0, wl.n_q, size=wl.batch).astype(np.int32)
    r = oracle_mod.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                      inp.free_stack, inp.free_top, n_q=wl.n_q)
    invariants(r["block_table"], r["context_lens"], r["refcount"], r["free_stack"],
               r["free_top"], inp.num_blocks)
    assert np.array_equal(r["context_lens"], inp.context_lens.numpy() + k + 1)
    # freed exactly the pages past the new length
    freed = 0
    for b in range(wl.batch):
        L = int(inp.context_lens[b])
        freed += -(-(L + wl.n_q) // 16) - (-(-(L + int(k[b]) + 1) // 16))
    assert r["free_top"] - inp.free_top == freed


def test_full_accept_keeps_every_page(oracle_mod):
    wl = W.WORKLOADS["tiny"]
    inp = W.make_attention(wl, 2)
    k = np.full(2, wl.gamma, np.int32)
    r = oracle_mod.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                      inp.free_stack, inp.free_top, n_q=wl.n_q)
    assert np.array_equal(r["block_table"], inp.block_table.numpy())
    assert r["free_top"] == inp.free_top


def test_shared_prefix_never_freed(oracle_mod):
    wl = W.WORKLOADS["tree"].scaled(batch=6, ctx_lo=0, ctx_hi=30, head_dim=8, num_q_heads=4,
                                    num_kv_heads=2, shared_prefix=32)
    inp = W.make_attention(wl, 23, poison=False)
    shared = inp.block_table[0, :2].tolist()
    assert all(int(inp.refcount[b]) == 6 for b in shared)
    k = np.zeros(wl.batch, np.int32)
    r = oracle_mod.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                      inp.free_stack, inp.free_top, n_q=wl.n_q)
    invariants(r["block_table"], r["context_lens"], r["refcount"], r["free_stack"],
               r["free_top"], inp.num_blocks, shared=shared)


def test_tree_compaction_moves_path_rows(oracle_mod):
    wl = W.WORKLOADS["tree"].scaled(batch=5, ctx_lo=3, ctx_hi=60, head_dim=16, num_q_heads=4,
                                    num_kv_heads=2, shared_prefix=0)
    inp = W.make_attention(wl, 29, poison=False)
    parent = wl.parent
    rng = np.random.default_rng(1)
    # random root-to-node paths
    children = {i: [c for c in range(len(parent)) if parent[c] == i] for i in range(len(parent))}
    depth_max = 3
    paths = np.full((wl.batch, depth_max + 1), -1, np.int32)
    ks = np.zeros(wl.batch, np.int32)
    for b in range(wl.batch):
        node, path = 0, [0]
        for _ in range(int(rng.integers(0, depth_max + 1))):
            node = int(rng.choice(children[node]))
            path.append(node)
        paths[b, :len(path)] = path
        ks[b] = len(path) - 1
    kp = inp.k_pool.view(torch.int16).numpy()
    vp = inp.v_pool.view(torch.int16).numpy()
    r = oracle_mod.block_table_commit(inp.block_table, inp.context_lens, ks, inp.refcount,
                                      inp.free_stack, inp.free_top, n_q=wl.n_q,
                                      path_nodes=paths, k_pool=kp, v_pool=vp)
    bt = inp.block_table.numpy()

    def row(pool, b, pos):
        return pool[bt[b, pos // 16], :, pos % 16]

    for b in range(wl.batch):
        L = int(inp.context_lens[b])
        for d in range(1, ks[b] + 1):
            assert np.array_equal(row(r["k_pool"], b, L + d), row(kp, b, L + int(paths[b, d])))
            assert np.array_equal(row(r["v_pool"], b, L + d), row(vp, b, L + int(paths[b, d])))
        # history and the root slot are untouched
        for pos in range(L + 1):
            assert np.array_equal(row(r["k_pool"], b, pos), row(kp, b, pos))
    invariants(r["block_table"], r["context_lens"], r["refcount"], r["free_stack"],
               r["free_top"], inp.num_blocks)
