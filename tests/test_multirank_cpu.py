"""Multi-rank host logic on CPU (gloo, world size 2).

The verification step has no cross-sequence dependency, so a batch shards by
sequence with no collective on the data path: each rank verifies its own
sequences against its own block table and pool.  These tests run two gloo
ranks, shard a batch, compute each shard with the oracle and check that the
union equals the single-process result; they also check the benchmark's
max/sum-over-ranks reductions.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def gathered_rows(r, b, n):
    """K and V bytes (and the FP8 scale of each row's page) of positions 0..n-1
    of sequence b in an append result, through its block table."""
    bt = r["block_table"][b]
    k = np.stack([r["k_pool"][bt[p // 16], :, p % 16] for p in range(n)])
    v = np.stack([r["v_pool"][bt[p // 16], :, p % 16] for p in range(n)])
    ks = np.stack([r["k_scale"][bt[p // 16]] for p in range(n)])
    return k, v, ks


def _worker(rank, world, port, outdir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    from speculative_verify_paged_attn_gb300 import workloads as W

    wl = W.WORKLOADS["70b"].scaled(batch=6, ctx_lo=10, ctx_hi=120, head_dim=64)
    inp = W.make_attention(wl, 55)
    smp = W.make_sampler(wl.scaled(vocab=500), 55)
    mine = list(range(rank, wl.batch, world))
    out, _ = oracle.paged_verify_attn(inp.q[mine], inp.k_pool, inp.v_pool, inp.block_table[mine],
                                      inp.context_lens[mine], num_kv_heads=wl.num_kv_heads,
                                      sm_scale=wl.sm_scale, nthreads=1)
    k, toks, _, _ = oracle.spec_accept(smp.p[mine], smp.q[mine], smp.tokens[mine],
                                       smp.u_accept[mine], smp.u_sample[mine], nthreads=1)
    # the sampler fed by logits on the shard's sequences
    li = W.make_logits(wl.scaled(vocab=700), 57, temperature=0.8)
    lk, lt, _ = oracle.spec_accept_logits(li.lp[mine], li.lq[mine], li.tokens[mine], li.u_accept[mine],
                                          li.u_sample[mine], temperature=0.8, nthreads=1)
    # K/V append on this rank's own copy of the cache (replicas: each GPU
    # owns its pool), for its sequences only; the gathered rows of each
    # sequence must not depend on which rank appended it
    ap = W.make_append(W.WORKLOADS["tiny"].scaled(kv_fp8=True), 56, contexts=(2, 5, 40, 9, 70, 3),
                       shared_prefix=19, n_new=5)
    ra = oracle.kv_append(ap.new_k[mine], ap.new_v[mine], ap.block_table.numpy()[mine],
                          ap.context_lens.numpy()[mine], ap.refcount.numpy(), ap.free_stack.numpy(),
                          ap.free_top, ap.k_pool, ap.v_pool, ap.k_scale, ap.v_scale)
    rows = [gathered_rows(ra, b_local, int(ap.context_lens[b]) + 5) for b_local, b in enumerate(mine)]
    # per-sequence acceptance averages and draft lengths on the shard
    gk = np.array([[0, 3, 4, 1, 2, 4], [1, 4, 4, 0, 2, 3]], np.int32)
    st = np.zeros((len(mine), 2), np.float32)
    for step in range(2):
        rg = oracle.gamma_update(4, gk[step][mine], seq_state=st, decay=0.8)
        st = rg["seq_state"]
    parts = [None] * world
    dist.all_gather_object(parts, (mine, out, k, toks, rows, st, rg["seq_gamma"], lk, lt))
    cpu = torch.device("cpu")
    mx = bench.max_over_ranks(float(rank + 1), world, cpu)
    sm = bench.sum_over_ranks(float(rank + 1), world, cpu)
    if rank == 0:
        np.save(os.path.join(outdir, "reduce.npy"), np.array([mx, sm]))
        B = wl.batch
        full_out = np.zeros((B,) + out.shape[1:])
        full_k = np.zeros(B, np.int32)
        full_t = np.zeros((B, toks.shape[1]), np.int32)
        app, gst, gg = [None] * 6, np.zeros((6, 2), np.float32), np.zeros(6, np.int32)
        full_lk = np.zeros(B, np.int32)
        full_lt = np.zeros((B, lt.shape[1]), np.int32)
        for idx, o, kk, tt, rr, ss, gq, lkk, ltt in parts:
            full_out[idx] = o
            full_k[idx] = kk
            full_t[idx] = tt
            full_lk[idx] = lkk
            full_lt[idx] = ltt
            for j, b in enumerate(idx):
                app[b] = rr[j]
            gst[idx], gg[idx] = ss, gq
        flat = np.empty(len(app), dtype=object)
        for b, r in enumerate(app):
            flat[b] = np.concatenate([a.ravel().view(np.uint8) for a in r])
        np.save(os.path.join(outdir, "append.npy"), flat, allow_pickle=True)
        np.save(os.path.join(outdir, "gstate.npy"), gst)
        np.save(os.path.join(outdir, "ggamma.npy"), gg)
        np.save(os.path.join(outdir, "out.npy"), full_out)
        np.save(os.path.join(outdir, "k.npy"), full_k)
        np.save(os.path.join(outdir, "t.npy"), full_t)
        np.save(os.path.join(outdir, "lk.npy"), full_lk)
        np.save(os.path.join(outdir, "lt.npy"), full_lt)
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_by_sequence_equals_single_process(tmp_path, oracle_mod):
    world = 2
    mp.start_processes(_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    from speculative_verify_paged_attn_gb300 import workloads as W
    wl = W.WORKLOADS["70b"].scaled(batch=6, ctx_lo=10, ctx_hi=120, head_dim=64)
    inp = W.make_attention(wl, 55)
    smp = W.make_sampler(wl.scaled(vocab=500), 55)
    ref, _ = oracle_mod.paged_verify_attn(inp.q, inp.k_pool, inp.v_pool, inp.block_table,
                                          inp.context_lens, num_kv_heads=wl.num_kv_heads,
                                          sm_scale=wl.sm_scale)
    k, toks, _, _ = oracle_mod.spec_accept(smp.p, smp.q, smp.tokens, smp.u_accept, smp.u_sample)
    assert np.array_equal(np.load(tmp_path / "out.npy"), ref)
    assert np.array_equal(np.load(tmp_path / "k.npy"), k)
    assert np.array_equal(np.load(tmp_path / "t.npy"), toks)
    li = W.make_logits(wl.scaled(vocab=700), 57, temperature=0.8)
    lk, lt, _ = oracle_mod.spec_accept_logits(li.lp, li.lq, li.tokens, li.u_accept, li.u_sample, temperature=0.8)
    assert np.array_equal(np.load(tmp_path / "lk.npy"), lk)
    assert np.array_equal(np.load(tmp_path / "lt.npy"), lt)
    mx, sm = np.load(tmp_path / "reduce.npy")
    assert mx == 2.0 and sm == 3.0
    # the append and the per-sequence draft-length state, single process
    ap = W.make_append(W.WORKLOADS["tiny"].scaled(kv_fp8=True), 56, contexts=(2, 5, 40, 9, 70, 3),
                       shared_prefix=19, n_new=5)
    ra = oracle_mod.kv_append(ap.new_k, ap.new_v, ap.block_table.numpy(), ap.context_lens.numpy(),
                              ap.refcount.numpy(), ap.free_stack.numpy(), ap.free_top, ap.k_pool, ap.v_pool,
                              ap.k_scale, ap.v_scale)
    got = np.load(tmp_path / "append.npy", allow_pickle=True)
    for b in range(6):
        want = np.concatenate([a.ravel().view(np.uint8) for a in gathered_rows(ra, b, int(ap.context_lens[b]) + 5)])
        assert np.array_equal(got[b], want), b
    gk = np.array([[0, 3, 4, 1, 2, 4], [1, 4, 4, 0, 2, 3]], np.int32)
    st = np.zeros((6, 2), np.float32)
    for step in range(2):
        rg = oracle_mod.gamma_update(4, gk[step], seq_state=st, decay=0.8)
        st = rg["seq_state"]
    assert np.array_equal(np.load(tmp_path / "gstate.npy"), st)
    assert np.array_equal(np.load(tmp_path / "ggamma.npy"), rg["seq_gamma"])
