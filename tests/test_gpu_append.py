"""GPU parity of svpa_kv_append (paged K/V append with block allocation,
copy-on-write and FP8 quantise-on-write) against the oracle.

Which free block a sequence receives, and which holder of a shared page keeps
it, depend on the order of concurrent pops; everything else is unique and
compared bit for bit: each sequence's gathered K/V bytes (and FP8 scales) on
every page it maps, the count of every block it maps, which table entries
share a block, the set of blocks in use and the free-stack top.  Small cases
run the oracle on the whole state; the full-size workloads check every
sequence's touched pages against an oracle run on that sequence alone, plus
block conservation."""
import numpy as np
import pytest
import torch

import oracle
from speculative_verify_paged_attn_gb300 import svpa
from speculative_verify_paged_attn_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BS = 16
CODE = {name: code for code, name in svpa.STATUS.items()}


def raw(pool):
    """uint16 (bf16 bits) or uint8 (E4M3 bytes) numpy view of a CPU/GPU pool."""
    t = pool.detach().cpu()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def run_gpu(inp, free_top=None, block_table=None, pools_on_device=False):
    fp8 = inp.wl.kv_fp8
    bt = (inp.block_table if block_table is None else block_table).to(DEV).clone()
    cl = inp.context_lens.to(DEV).clone()
    rc = inp.refcount.to(DEV).clone()
    fs = inp.free_stack.to(DEV).clone()
    ft = torch.tensor([inp.free_top if free_top is None else free_top], dtype=torch.int32, device=DEV)
    kp = inp.k_pool.to(DEV).clone()
    vp = inp.v_pool.to(DEV).clone()
    if fp8:
        kp, vp = kp.view(torch.uint8), vp.view(torch.uint8)
    ks = inp.k_scale.to(DEV).clone() if fp8 else None
    vs = inp.v_scale.to(DEV).clone() if fp8 else None
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    svpa.kv_append(inp.new_k.to(DEV), inp.new_v.to(DEV), bt, cl, rc, fs, ft, kp, vp, error_flag=err,
                   k_scale=ks, v_scale=vs, scale_tile=inp.wl.scale_tile)
    st = svpa.check_error(err)
    return st, dict(block_table=bt.cpu().numpy(), refcount=rc.cpu().numpy(), free_stack=fs.cpu().numpy(),
                    free_top=int(ft.item()),
                    k_pool=kp if pools_on_device else raw(kp), v_pool=vp if pools_on_device else raw(vp),
                    k_scale=None if ks is None else ks.cpu().numpy(),
                    v_scale=None if vs is None else vs.cpu().numpy())


def run_oracle(inp):
    c = lambda t: None if t is None else t.cpu()
    return oracle.kv_append(c(inp.new_k), c(inp.new_v), inp.block_table.cpu().numpy(),
                            inp.context_lens.cpu().numpy(), inp.refcount.cpu().numpy(),
                            inp.free_stack.cpu().numpy(), inp.free_top, c(inp.k_pool), c(inp.v_pool),
                            c(inp.k_scale), c(inp.v_scale), scale_tile=inp.wl.scale_tile)


def canon(bt):
    """Label blocks by first appearance: equal arrays = same sharing structure."""
    lab, out = {}, np.full(bt.shape, -1, np.int64)
    for idx, blk in np.ndenumerate(bt):
        if blk >= 0:
            out[idx] = lab.setdefault(int(blk), len(lab))
    return out


def check_conservation(res, num_blocks):
    bt = res["block_table"]
    used = {}
    for blk in bt[bt >= 0].tolist():
        used[blk] = used.get(blk, 0) + 1
    free = res["free_stack"][:res["free_top"]].tolist()
    assert len(set(free)) == len(free) and set(free).isdisjoint(used)
    assert set(free) | set(used) == set(range(num_blocks))
    rc = res["refcount"]
    for blk in range(num_blocks):
        assert rc[blk] == used.get(blk, 0), f"block {blk}"


def compare(g, r, inp):
    fp8 = inp.wl.kv_fp8
    L = inp.context_lens.cpu().numpy().astype(np.int64)
    end = L + inp.n_new
    gb, rb = g["block_table"], r["block_table"]
    assert np.array_equal(gb >= 0, rb >= 0)
    assert np.array_equal(canon(gb), canon(rb))
    assert g["free_top"] == r["free_top"]
    assert set(gb[gb >= 0].tolist()) == set(rb[rb >= 0].tolist())
    check_conservation(g, inp.k_pool.shape[0])
    for b in range(gb.shape[0]):
        for i in range(int((end[b] + BS - 1) // BS)):
            x, y = int(gb[b, i]), int(rb[b, i])
            assert g["refcount"][x] == r["refcount"][y]
            touched = i >= L[b] // BS
            upto = BS if (fp8 and touched) else int(min(BS, end[b] - i * BS))
            for name in ("k_pool", "v_pool"):
                assert np.array_equal(g[name][x, :, :upto], r[name][y, :, :upto]), (b, i, name)
            if fp8:
                # tile scales of slots past the last row are never written
                n_used = int(min(BS, end[b] - i * BS))
                for name in ("k_scale", "v_scale"):
                    gs, rs = g[name][x], r[name][y]
                    if inp.wl.scale_tile:
                        gs, rs = gs[:, :n_used], rs[:, :n_used]
                    assert np.array_equal(gs, rs), (b, i, name)


SMALL = {
    # name: (workload, contexts, shared prefix, n_new)
    "bf16_cow": (W.WORKLOADS["tiny"], (2, 50, 3, 12), 19, 7),
    "fp8_cow_d64": (W.WORKLOADS["tiny"].scaled(kv_fp8=True), (2, 50, 3, 12), 19, 7),
    "bf16_edges": (W.WORKLOADS["7b"].scaled(num_q_heads=4, num_kv_heads=4), (0, 1, 15, 16, 17, 31), 0, 40),
    "fp8_edges": (W.WORKLOADS["fp8"], (0, 1, 15, 16, 17, 31, 200), 0, 29),
    "fp8_rescale_cow": (W.WORKLOADS["fp8"], (0, 4, 9, 12, 300, 1000), 35, 6),
    "bf16_tree_cow": (W.WORKLOADS["tree"], (0, 3, 5, 700), 803, 29),
    "fp8_single_row": (W.WORKLOADS["fp8"], (5, 16, 95), 0, 1),
    # one scale per 64-element tile of a row
    "fp8_t64_cow": (W.WORKLOADS["fp8_t64"], (0, 4, 9, 12, 300, 1000), 35, 6),
    "fp8_t64_edges": (W.WORKLOADS["fp8_t64"].scaled(num_q_heads=4, num_kv_heads=2, head_dim=256),
                      (0, 1, 15, 16, 17, 31), 0, 29),
    "fp8_t64_d64": (W.WORKLOADS["tiny"].scaled(kv_fp8=True, scale_tile=64), (2, 50, 3, 12), 19, 7),
    # widest FP8 tile (16 x 256 bytes) and a copy-on-write at D = 256
    "fp8_d256_cow": (W.WORKLOADS["fp8"].scaled(num_q_heads=4, num_kv_heads=2, head_dim=256),
                     (1, 3, 16, 40), 21, 20),
    # odd head count (a partial group of units) and 9 chunks per bf16 row
    "bf16_hkv3_d72": (W.WORKLOADS["7b"].scaled(num_q_heads=3, num_kv_heads=3, head_dim=72), (5, 33, 0), 0, 9),
}


@pytest.mark.parametrize("case", sorted(SMALL))
def test_append_matches_oracle(case):
    wl, ctx, prefix, n_new = SMALL[case]
    inp = W.make_append(wl, 11 + len(case), contexts=ctx, shared_prefix=prefix, n_new=n_new)
    st, g = run_gpu(inp)
    assert st == 0
    r = run_oracle(inp)
    compare(g, r, inp)
    if prefix % BS:
        # the copy-on-write path really ran: some sequences started on the shared page
        L = inp.context_lens.numpy()
        on_shared = int(((L <= (prefix // BS + 1) * BS) & (L > prefix // BS * BS)).sum())
        assert on_shared >= 2
        assert g["free_top"] < inp.free_top


def test_append_batch_zero_is_a_noop():
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    z = torch.zeros(1, dtype=torch.int32, device=DEV)
    e = torch.empty((0, 5, 4, 64), dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros((4, 4, 16, 64), dtype=torch.bfloat16, device=DEV)
    bt = torch.zeros((0, 4), dtype=torch.int32, device=DEV)
    assert svpa.kv_append(e, e, bt, z[:0], z, z, z, pool, pool, error_flag=err) == 0
    assert svpa.check_error(err) == 0


def test_append_out_of_blocks_writes_no_rows():
    wl = W.WORKLOADS["tiny"]
    inp = W.make_append(wl, 21, contexts=(30, 40, 50), shared_prefix=0, n_new=40)
    before_k, before_v = raw(inp.k_pool), raw(inp.v_pool)
    st, g = run_gpu(inp, free_top=3)
    assert st == CODE["SVPA_ERR_OUT_OF_BLOCKS"]
    check_conservation_with_free(g, inp, 3)
    bt0 = inp.block_table.numpy()
    for blk in bt0[bt0 >= 0].tolist():  # pages mapped before the call are untouched
        assert np.array_equal(g["k_pool"][blk], before_k[blk])
        assert np.array_equal(g["v_pool"][blk], before_v[blk])


def check_conservation_with_free(g, inp, top):
    """Conservation when only the first `top` entries of the stack were offered."""
    bt = g["block_table"]
    used = {}
    for blk in bt[bt >= 0].tolist():
        used[blk] = used.get(blk, 0) + 1
    offered = set(inp.free_stack.numpy()[:top].tolist())
    free = set(g["free_stack"][:g["free_top"]].tolist())
    bt0 = inp.block_table.numpy()
    before = set(bt0[bt0 >= 0].tolist())
    assert set(used) == before | (offered - free)
    for blk, n in used.items():
        assert g["refcount"][blk] == n


def test_append_missing_history_page_and_bad_block_are_reported():
    wl = W.WORKLOADS["tiny"]
    inp = W.make_append(wl, 22, contexts=(30, 40), shared_prefix=0, n_new=3)
    bt = inp.block_table.clone()
    bt[0, 1] = -1  # L = 30: page 1 holds history and is where the rows land
    st, _ = run_gpu(inp, block_table=bt)
    assert st == CODE["SVPA_ERR_INVALID_ARG"]
    bt = inp.block_table.clone()
    bt[1, 2] = inp.k_pool.shape[0] + 5
    st, _ = run_gpu(inp, block_table=bt)
    assert st == CODE["SVPA_ERR_BAD_BLOCK"]


def sequence_oracle(inp, b, old_k, old_v, old_ks, old_vs):
    """The oracle on sequence b alone: its touched pages (old content) on a
    private pool, a free stack big enough for its new pages."""
    L = int(inp.context_lens[b])
    end = L + inp.n_new
    i0, i1 = L // BS, (end - 1) // BS
    n = i1 - i0 + 1
    nb = 2 * n
    fp8 = inp.wl.kv_fp8
    shape = (nb,) + tuple(inp.k_pool.shape[1:])
    dt = np.uint8 if fp8 else np.uint16
    kp, vp = np.zeros(shape, dt), np.zeros(shape, dt)
    sshape = (nb,) + tuple(inp.k_scale.shape[1:]) if fp8 else (nb, shape[1])
    ks, vs = np.ones(sshape, np.float32), np.ones(sshape, np.float32)
    bt = np.full((1, i1 + 1), -1, np.int32)
    rc = np.zeros(nb, np.int32)
    for j in range(n):
        if old_k[j] is not None:
            kp[j], vp[j] = old_k[j], old_v[j]
            if fp8:
                ks[j], vs[j] = old_ks[j], old_vs[j]
            bt[0, i0 + j] = j
            rc[j] = 1
    fs = np.arange(n, nb, dtype=np.int32)
    fs = np.concatenate([fs, np.full(nb - fs.size, -1, np.int32)])
    r = oracle.kv_append(inp.new_k[b:b + 1].cpu(), inp.new_v[b:b + 1].cpu(), bt,
                         np.array([L], np.int32), rc, fs, nb - n, kp, vp,
                         ks if fp8 else None, vs if fp8 else None, scale_tile=inp.wl.scale_tile)
    return r, i0, i1


@pytest.mark.parametrize("name", ["7b", "70b", "fp8", "tree", "fp8_t64"])
def test_append_full_size_workloads(name):
    """The bench's append state (full batch, n_new = n_q, contexts as drawn);
    every sequence's touched pages against the oracle on that sequence."""
    wl = W.WORKLOADS[name]
    inp = W.make_append(wl, W.SEEDS[name], device=DEV)
    fp8 = wl.kv_fp8
    L = inp.context_lens.cpu().numpy().astype(np.int64)
    bt0 = inp.block_table.cpu().numpy()
    B = bt0.shape[0]
    olds = []
    for b in range(B):
        i0, i1 = L[b] // BS, (L[b] + inp.n_new - 1) // BS
        ok, ov, oks, ovs = [], [], [], []
        for i in range(i0, i1 + 1):
            blk = int(bt0[b, i])
            if blk < 0:
                ok.append(None), ov.append(None), oks.append(None), ovs.append(None)
                continue
            ok.append(raw(inp.k_pool[blk]))
            ov.append(raw(inp.v_pool[blk]))
            oks.append(inp.k_scale[blk].cpu().numpy() if fp8 else None)
            ovs.append(inp.v_scale[blk].cpu().numpy() if fp8 else None)
        olds.append((ok, ov, oks, ovs))
    st, g = run_gpu(inp, pools_on_device=True)
    assert st == 0
    check_conservation(g, inp.k_pool.shape[0])
    new_pages = int(sum((L[b] + inp.n_new + BS - 1) // BS - (L[b] + BS - 1) // BS for b in range(B)))
    assert inp.free_top - g["free_top"] == new_pages
    for b in range(B):
        r, i0, i1 = sequence_oracle(inp, b, *olds[b])
        end = L[b] + inp.n_new
        for i in range(i0, i1 + 1):
            x, y = int(g["block_table"][b, i]), int(r["block_table"][0, i])
            assert g["refcount"][x] == 1
            upto = BS if fp8 else int(min(BS, end - i * BS))
            for nm in ("k_pool", "v_pool"):
                assert np.array_equal(raw(g[nm][x])[:, :upto], r[nm][y, :, :upto]), (b, i, nm)
            if fp8:
                n_used = int(min(BS, end - i * BS))
                for nm in ("k_scale", "v_scale"):
                    gs, rs = g[nm][x], r[nm][y]
                    if inp.wl.scale_tile:  # tile scales past the last row are never written
                        gs, rs = gs[:, :n_used], rs[:, :n_used]
                    assert np.array_equal(gs, rs), (b, i, nm)
        # pages before the append are untouched
        for i in range(0, int(i0)):
            assert g["block_table"][b, i] == bt0[b, i]
