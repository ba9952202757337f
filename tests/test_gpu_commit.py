"""GPU parity of svpa_block_table_commit: bit-exact block tables, lengths and
reference counts; the free stack is compared as a multiset (the order of
concurrent pushes is unspecified) with an exact top."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def run_commit(inp, k, path=None):
    bt = inp.block_table.to(DEV).clone()
    cl = inp.context_lens.to(DEV).clone()
    rc = inp.refcount.to(DEV).clone()
    fs = inp.free_stack.to(DEV).clone()
    ft = torch.tensor([inp.free_top], dtype=torch.int32, device=DEV)
    kp = inp.k_pool.to(DEV).clone()
    vp = inp.v_pool.to(DEV).clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    wl = inp.wl
    svpa.block_table_commit(wl.n_q, bt, cl, torch.as_tensor(k, dtype=torch.int32).to(DEV), rc, fs, ft,
                            error_flag=err,
                            path_nodes=None if path is None else torch.as_tensor(path).to(DEV),
                            k_pool=kp, v_pool=vp, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim)
    st = svpa.check_error(err)
    return st, dict(block_table=bt.cpu().numpy(), context_lens=cl.cpu().numpy(),
                    refcount=rc.cpu().numpy(), free_stack=fs.cpu().numpy(), free_top=int(ft.item()),
                    k_pool=kp.cpu(), v_pool=vp.cpu())


def compare(g, r):
    assert np.array_equal(g["block_table"], r["block_table"])
    assert np.array_equal(g["context_lens"], r["context_lens"])
    assert np.array_equal(g["refcount"], r["refcount"])
    assert g["free_top"] == r["free_top"]
    n = g["free_top"]
    assert sorted(g["free_stack"][:n].tolist()) == sorted(r["free_stack"][:n].tolist())


@pytest.mark.parametrize("name", ["tiny", "7b", "70b"])
def test_linear_commit(name):
    wl = W.WORKLOADS[name]
    if name != "tiny":
        wl = wl.scaled(batch=min(wl.batch, 48), head_dim=64, num_q_heads=8, num_kv_heads=8)
    inp = W.make_attention(wl, 300, poison=False)
    rng = np.random.default_rng(1)
    k = rng.integers(0, wl.n_q, size=inp.q.shape[0]).astype(np.int32)
    st, g = run_commit(inp, k)
    assert st == 0
    r = oracle.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                  inp.free_stack, inp.free_top, n_q=wl.n_q)
    compare(g, r)


def test_shared_prefix_commit():
    wl = W.WORKLOADS["tree"].scaled(batch=16, head_dim=64, ctx_lo=0, ctx_hi=100)
    inp = W.make_attention(wl, 301, poison=False)
    k = np.zeros(16, np.int32)
    st, g = run_commit(inp, k)
    assert st == 0
    r = oracle.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                  inp.free_stack, inp.free_top, n_q=wl.n_q)
    compare(g, r)


def test_tree_commit_compacts_path():
    wl = W.WORKLOADS["tree"].scaled(batch=12, ctx_lo=1, ctx_hi=90, shared_prefix=32)
    inp = W.make_attention(wl, 302, poison=False)
    parent = wl.parent
    children = {i: [c for c in range(len(parent)) if parent[c] == i] for i in range(len(parent))}
    rng = np.random.default_rng(5)
    W_ = 4
    paths = np.full((12, W_), -1, np.int32)
    ks = np.zeros(12, np.int32)
    for b in range(12):
        node, path = 0, [0]
        for _ in range(int(rng.integers(0, 4))):
            node = int(rng.choice(children[node]))
            path.append(node)
        paths[b, :len(path)] = path
        ks[b] = len(path) - 1
    st, g = run_commit(inp, ks, paths)
    assert st == 0
    r = oracle.block_table_commit(inp.block_table, inp.context_lens, ks, inp.refcount, inp.free_stack,
                                  inp.free_top, n_q=wl.n_q, path_nodes=paths,
                                  k_pool=inp.k_pool.view(torch.int16).numpy(),
                                  v_pool=inp.v_pool.view(torch.int16).numpy())
    compare(g, r)
    assert np.array_equal(g["k_pool"].view(torch.int16).numpy(), r["k_pool"])
    assert np.array_equal(g["v_pool"].view(torch.int16).numpy(), r["v_pool"])


def test_full_size_commit_70b():
    wl = W.WORKLOADS["70b"]
    inp = W.make_attention(wl.scaled(head_dim=64, num_q_heads=8, num_kv_heads=1), W.SEEDS["70b"],
                           poison=False)
    rng = np.random.default_rng(2)
    k = rng.integers(0, wl.n_q, size=wl.batch).astype(np.int32)
    st, g = run_commit(inp, k)
    assert st == 0
    r = oracle.block_table_commit(inp.block_table, inp.context_lens, k, inp.refcount,
                                  inp.free_stack, inp.free_top, n_q=wl.n_q)
    compare(g, r)


def test_bad_accepted_len_reported():
    inp = W.make_attention(W.WORKLOADS["tiny"], 303, poison=False)
    st, _ = run_commit(inp, np.array([0, 9], np.int32))
    assert st == 1


def test_tree_commit_bad_path_leaves_sequence_untouched():
    # sequence 3's path names node 1 at depth 2 (a node's index is at least its
    # depth in BFS order): the call reports it and leaves that sequence's rows,
    # pages and length as they were; the other sequences commit normally
    wl = W.WORKLOADS["tree"].scaled(batch=6, ctx_lo=1, ctx_hi=90, shared_prefix=32)
    inp = W.make_attention(wl, 304, poison=False)
    paths = np.full((6, 4), -1, np.int32)
    paths[:, 0] = 0
    paths[:, 1] = 2
    paths[:, 2] = [c for c in range(len(wl.parent)) if wl.parent[c] == 2][0]
    ks = np.full(6, 2, np.int32)
    paths[3, 2] = 1
    st, g = run_commit(inp, ks, paths)
    assert st == 5  # SVPA_ERR_BAD_BLOCK
    good = [0, 1, 2, 4, 5]
    r = oracle.block_table_commit(inp.block_table[good], inp.context_lens[good], ks[good], inp.refcount,
                                  inp.free_stack, inp.free_top, n_q=wl.n_q, path_nodes=paths[good],
                                  k_pool=inp.k_pool.view(torch.int16).numpy(),
                                  v_pool=inp.v_pool.view(torch.int16).numpy())
    assert np.array_equal(g["block_table"][good], r["block_table"])
    assert np.array_equal(g["context_lens"][good], r["context_lens"])
    assert np.array_equal(g["block_table"][3], inp.block_table[3].numpy())
    assert g["context_lens"][3] == int(inp.context_lens[3])
    own = inp.block_table[3]
    own = own[own >= 0].long()
    assert torch.equal(g["k_pool"][own], inp.k_pool[own])
    assert torch.equal(g["v_pool"][own], inp.v_pool[own])
    assert np.array_equal(g["refcount"][own.numpy()], inp.refcount[own].numpy())
