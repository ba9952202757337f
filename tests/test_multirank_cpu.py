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
    parts = [None] * world
    dist.all_gather_object(parts, (mine, out, k, toks))
    cpu = torch.device("cpu")
    mx = bench.max_over_ranks(float(rank + 1), world, cpu)
    sm = bench.sum_over_ranks(float(rank + 1), world, cpu)
    if rank == 0:
        np.save(os.path.join(outdir, "reduce.npy"), np.array([mx, sm]))
        B = wl.batch
        full_out = np.zeros((B,) + out.shape[1:])
        full_k = np.zeros(B, np.int32)
        full_t = np.zeros((B, toks.shape[1]), np.int32)
        for idx, o, kk, tt in parts:
            full_out[idx] = o
            full_k[idx] = kk
            full_t[idx] = tt
        np.save(os.path.join(outdir, "out.npy"), full_out)
        np.save(os.path.join(outdir, "k.npy"), full_k)
        np.save(os.path.join(outdir, "t.npy"), full_t)
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
    mx, sm = np.load(tmp_path / "reduce.npy")
    assert mx == 2.0 and sm == 3.0
