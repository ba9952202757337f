"""The tree-sampler validity check (tests/tree_check.py) accepts the oracle's
own outputs and rejects planted mistakes, so that the GPU test built on it
cannot pass vacuously."""
import numpy as np
import torch

import oracle
from speculative_verify_paged_attn_gb300 import workloads as W

from tree_check import tree_walk_valid


def _case(batch=48, vocab=3000, seed=91):
    wl = W.WORKLOADS["tree"].scaled(batch=batch)
    s = W.make_sampler(wl, seed, device="cpu", vocab=vocab)
    k, path, toks, near = oracle.spec_accept_tree(np.array(wl.parent, np.int32), s.p, s.q, s.tokens,
                                                  s.u_accept, s.u_sample)
    return wl.parent, s, k, path, toks


def test_oracle_rows_are_valid():
    parent, s, k, path, toks = _case()
    assert 0 < (k == 0).sum() < k.shape[0] and (k == 3).any()
    for b in range(k.shape[0]):
        valid, in_band = tree_walk_valid(parent, s, b, int(k[b]), path[b], toks[b])
        assert valid and not in_band, b


def test_planted_mistakes_are_caught():
    parent, s, k, path, toks = _case()
    V = s.p.shape[2]
    caught = {"token": 0, "length": 0, "branch": 0}
    for b in range(k.shape[0]):
        kb = int(k[b])
        # a final token far from the drawn one
        t2 = toks[b].copy()
        t2[kb] = (t2[kb] + V // 2) % V
        caught["token"] += not tree_walk_valid(parent, s, b, kb, path[b], t2)[0]
        # one accepted node dropped (the walk would have accepted it)
        if kb > 0:
            p2, t3 = path[b].copy(), toks[b].copy()
            p2[kb] = -1
            t3[kb - 1] = toks[b][kb]
            t3[kb] = -1
            caught["length"] += not tree_walk_valid(parent, s, b, kb - 1, p2, t3)[0]
        # the first accepted node replaced by a sibling tested after it
        if kb > 0:
            c = int(path[b][1])
            sib = [x for x in range(len(parent)) if parent[x] == 0 and x > c]
            if sib:
                p2 = path[b].copy()
                p2[1] = sib[0]
                caught["branch"] += not tree_walk_valid(parent, s, b, kb, p2, toks[b])[0]
    n_acc = int((k > 0).sum())
    assert caught["token"] == k.shape[0]
    assert caught["length"] == n_acc
    assert caught["branch"] > 0
