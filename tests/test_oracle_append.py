"""Pins of the oracle's paged K/V append (allocation, copy-on-write, FP8
quantise-on-write) against what the method fixes independently of paging:
after the append, every sequence's gathered K/V is its old history followed by
its new rows; a shared page is cloned before a write, so the other holders'
view is unchanged; blocks are conserved; FP8 codes follow the scale rule and
the OCP E4M3 rounding (checked against torch's float8_e4m3fn cast)."""
import numpy as np
import pytest
import torch

import oracle

BS = 16


def gather(pool, table_row, n):
    """Positions 0..n-1 of one sequence, [n, Hkv, D], through its block table."""
    return np.stack([pool[table_row[p // BS], :, p % BS, :] for p in range(n)])


def make_state(seed, B=3, Hkv=2, D=8, num_blocks=24, L=(10, 16, 37), shared=None):
    g = torch.Generator().manual_seed(seed)
    kp = torch.randn(num_blocks, Hkv, BS, D, generator=g).to(torch.bfloat16)
    vp = torch.randn(num_blocks, Hkv, BS, D, generator=g).to(torch.bfloat16)
    max_blocks = 6
    bt = np.full((B, max_blocks), -1, np.int32)
    rc = np.zeros(num_blocks, np.int32)
    perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    nxt = 0
    for b in range(B):
        for i in range((L[b] + BS - 1) // BS):
            bt[b, i] = perm[nxt]
            rc[perm[nxt]] = 1
            nxt += 1
    if shared is not None:  # sequences (a, c) share their first page
        a, c = shared
        rc[bt[c, 0]] = 0
        bt[c, 0] = bt[a, 0]
        rc[bt[a, 0]] += 1
    free = np.array(sorted(set(range(num_blocks)) - set(bt[bt >= 0].tolist())), np.int32)
    fs = np.zeros(num_blocks, np.int32)
    fs[:free.size] = free
    return kp, vp, bt, rc, fs, free.size, np.array(L, np.int32)


def check_conservation(bt, rc, fs, ft, num_blocks):
    used = {}
    for blk in bt[bt >= 0].tolist():
        used[blk] = used.get(blk, 0) + 1
    for blk in range(num_blocks):
        assert rc[blk] == used.get(blk, 0)
    free = set(fs[:ft].tolist())
    assert len(free) == ft
    assert free.isdisjoint(used) and free | set(used) == set(range(num_blocks))


@pytest.mark.parametrize("n_new", [1, 5, 6, 29])
def test_append_gathers_history_then_new_rows(n_new):
    kp, vp, bt, rc, fs, ft, L = make_state(1)
    B, Hkv, D = 3, 2, 8
    g = torch.Generator().manual_seed(2)
    nk = torch.randn(B, n_new, Hkv, D, generator=g).to(torch.bfloat16)
    nv = torch.randn(B, n_new, Hkv, D, generator=g).to(torch.bfloat16)
    r = oracle.kv_append(nk, nv, bt, L, rc, fs, ft, kp, vp)
    k16, v16 = kp.view(torch.int16).numpy().view(np.uint16), vp.view(torch.int16).numpy().view(np.uint16)
    for b in range(B):
        old_k, old_v = gather(k16, bt[b], L[b]), gather(v16, bt[b], L[b])
        new_k, new_v = gather(r["k_pool"], r["block_table"][b], L[b] + n_new), gather(r["v_pool"], r["block_table"][b], L[b] + n_new)
        assert np.array_equal(new_k[:L[b]], old_k) and np.array_equal(new_v[:L[b]], old_v)
        assert np.array_equal(new_k[L[b]:], nk[b].view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(new_v[L[b]:], nv[b].view(torch.int16).numpy().view(np.uint16))
    check_conservation(r["block_table"], r["refcount"], r["free_stack"], r["free_top"], 24)
    pages_needed = sum(-(-(int(L[b]) + n_new) // BS) - (-(-int(L[b]) // BS)) for b in range(B))
    assert ft - r["free_top"] == pages_needed


def test_copy_on_write_keeps_the_other_holder_unchanged():
    # sequences 0 and 1 share a partially filled first page (both 10 tokens long)
    kp, vp, bt, rc, fs, ft, L = make_state(3, L=(10, 10, 37), shared=(0, 1))
    assert rc[bt[0, 0]] == 2
    nk = torch.randn(3, 4, 2, 8).to(torch.bfloat16)
    nv = torch.randn(3, 4, 2, 8).to(torch.bfloat16)
    shared_blk = int(bt[0, 0])
    before = kp[shared_blk].clone()
    r = oracle.kv_append(nk, nv, bt, L, rc, fs, ft, kp, vp)
    t0, t1 = r["block_table"][0, 0], r["block_table"][1, 0]
    assert t0 != t1  # one holder got a private copy
    assert shared_blk in (t0, t1) and r["refcount"][shared_blk] == 1
    # the history both share is intact in both views
    k16 = r["k_pool"]
    for t in (t0, t1):
        assert np.array_equal(k16[t, :, :10], before[:, :10].view(torch.int16).numpy().view(np.uint16))
    check_conservation(r["block_table"], r["refcount"], r["free_stack"], r["free_top"], 24)


def test_out_of_blocks_and_missing_history_page_are_errors():
    kp, vp, bt, rc, fs, ft, L = make_state(4)
    nk = torch.zeros(3, 64, 2, 8).to(torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(nk, nk, bt, L, rc, fs, 2, kp, vp)  # only two free blocks
    bt2 = bt.copy()
    bt2[2, 2] = -1  # sequence 2 has 37 tokens: page 2, where the append lands, holds history
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(nk[:, :1], nk[:, :1], bt2, L, rc, fs, ft, kp, vp)


def test_e4m3_encode_matches_torch_rounding():
    g = torch.Generator().manual_seed(5)
    # 10^6 values over five magnitudes, from the subnormal range to saturation
    x = torch.cat([torch.randn(200000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 200.0)])
    x = torch.cat([x[x.abs() <= 448], torch.tensor([0.0, -0.0, -2.0 ** -11, 2.0 ** -11])])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)
    # every finite code re-encodes to itself; beyond 448 saturates
    codes = torch.arange(256, dtype=torch.uint8)
    vals = codes.view(torch.float8_e4m3fn).float()
    fin = torch.isfinite(vals)
    assert np.array_equal(oracle.e4m3_encode(vals[fin].numpy()), codes[fin].numpy())
    assert list(oracle.e4m3_encode(np.array([449.0, 1e6, -500.0], np.float32))) == [0x7E, 0x7E, 0xFE]


def test_fp8_quantise_on_write_worked_page():
    # a fresh page: scale = amax / 448 over the new rows, code = e4m3(x / scale)
    Hkv, D, nb = 1, 4, 4
    kp = torch.zeros(nb, Hkv, BS, D, dtype=torch.uint8)
    vp = torch.zeros(nb, Hkv, BS, D, dtype=torch.uint8)
    ks = torch.ones(nb, Hkv)
    vs = torch.ones(nb, Hkv)
    bt = np.full((1, 2), -1, np.int32)
    rc = np.zeros(nb, np.int32)
    fs = np.arange(nb, dtype=np.int32)
    rows = torch.tensor([[[1.0, -2.0, 0.5, 3.5]], [[7.0, 0.0, -0.25, 1.0]]]).to(torch.bfloat16)  # [2, 1, 4]
    r = oracle.kv_append(rows[None], rows[None], bt, np.array([0], np.int32), rc, fs, nb, kp, vp, ks, vs)
    blk = r["block_table"][0, 0]
    assert r["k_scale"][blk, 0] == np.float32(7.0) / np.float32(448.0)
    want = (rows.float() / torch.tensor(np.float32(7.0) / np.float32(448.0))).to(torch.float8_e4m3fn)
    assert np.array_equal(r["k_pool"][blk, 0, :2], want.view(torch.uint8).numpy()[:, 0])
    assert not r["k_pool"][blk, 0, 2:].any()  # unused slots are zero
    # appending a row with a larger magnitude rescales the page and re-encodes the history
    more = torch.tensor([[[14.0, 1.0, 1.0, 1.0]]]).to(torch.bfloat16)
    r2 = oracle.kv_append(more[None], more[None], r["block_table"], np.array([2], np.int32), r["refcount"],
                          r["free_stack"], r["free_top"], r["k_pool"], r["v_pool"], r["k_scale"], r["v_scale"])
    s2 = r2["k_scale"][blk, 0]
    assert s2 == np.float32(14.0) / np.float32(448.0)
    dec = torch.from_numpy(r2["k_pool"][blk, 0, :3].copy()).view(torch.float8_e4m3fn).float().numpy() * s2
    data = torch.cat([rows[:, 0], more[:, 0]]).float().numpy()
    spacing = np.maximum(np.abs(data), 2.0 ** -6 * s2) * 2.0 ** -3  # worst case: two roundings
    assert np.all(np.abs(dec - data) <= spacing + 1e-7)
    # a row within the current range keeps the history codes as they are
    small = torch.tensor([[[1.0, 1.0, 1.0, 1.0]]]).to(torch.bfloat16)
    r3 = oracle.kv_append(small[None], small[None], r2["block_table"], np.array([3], np.int32), r2["refcount"],
                          r2["free_stack"], r2["free_top"], r2["k_pool"], r2["v_pool"], r2["k_scale"], r2["v_scale"])
    assert r3["k_scale"][blk, 0] == s2
    assert np.array_equal(r3["k_pool"][blk, 0, :3], r2["k_pool"][blk, 0, :3])


def test_fp8_tile_scales_quantise_each_new_row_tile():
    # one scale per 64 consecutive elements of a row: a new row's tiles get
    # amax/448 of their own values; history rows keep codes and scales
    Hkv, D, nb = 2, 128, 6
    g = torch.Generator().manual_seed(11)
    kp = torch.randint(0, 120, (nb, Hkv, BS, D), generator=g).to(torch.uint8)
    vp = torch.randint(0, 120, (nb, Hkv, BS, D), generator=g).to(torch.uint8)
    ks = torch.rand(nb, Hkv, BS, D // 64, generator=g) + 0.01
    vs = torch.rand(nb, Hkv, BS, D // 64, generator=g) + 0.01
    bt = np.array([[2, -1], [4, 5]], np.int32)  # sequence 1 shares nothing; pages hold 5 and 17 tokens
    rc = np.zeros(nb, np.int32)
    rc[[2, 4, 5]] = 1
    fs = np.array([0, 1, 3, -1, -1, -1], np.int32)
    L = np.array([5, 17], np.int32)
    rows = (torch.randn(2, 3, Hkv, D, generator=g) * torch.tensor([0.1, 1.0, 20.0])[None, :, None, None])
    rows[0, 1, 0, 64:] = 0.0  # an all-zero tile: scale 1
    rows = rows.to(torch.bfloat16)
    r = oracle.kv_append(rows, rows, bt, L, rc, fs, 3, kp, vp, ks, vs, scale_tile=64)
    ksr = r["k_scale"].reshape(nb, Hkv, BS, D // 64)
    for b, blk, s0 in [(0, 2, 5), (1, 5, 1)]:
        for t in range(3):
            for h in range(Hkv):
                for tile in range(2):
                    x = rows[b, t, h, 64 * tile:64 * tile + 64].float()
                    amax = x.abs().max()
                    sc = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
                    assert ksr[blk, h, s0 + t, tile] == sc
                    want = (x / torch.tensor(sc)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                    assert np.array_equal(r["k_pool"][blk, h, s0 + t, 64 * tile:64 * tile + 64], want)
    assert ksr[2, 0, 6, 1] == np.float32(1.0)
    # history rows and their scales are untouched; codes past the last row are 0
    assert np.array_equal(r["k_pool"][2, :, :5], kp[2, :, :5].numpy())
    assert np.array_equal(ksr[2, :, :5], ks[2, :, :5].numpy())
    assert not r["k_pool"][2, :, 8:].any()


def test_fp8_tile_scales_copy_on_write_carries_tile_scales():
    kp, vp, bt, rc, fs, ft, L = make_state(3, L=(10, 10, 37), shared=(0, 1))
    kp8 = torch.randint(0, 120, tuple(kp.shape)).to(torch.uint8)
    vp8 = torch.randint(0, 120, tuple(vp.shape)).to(torch.uint8)
    # D = 8 is not a multiple of 64: the tile mode needs D % 64 == 0
    nk = torch.randn(3, 2, 2, 8).to(torch.bfloat16)
    ks = torch.rand(24, 2, BS, 1)
    with pytest.raises(oracle.OracleError):
        oracle.kv_append(nk, nk, bt, L, rc, fs, ft, kp8, vp8, ks, ks, scale_tile=64)
    g = torch.Generator().manual_seed(4)
    kp8 = torch.randint(0, 120, (24, 2, BS, 64), generator=g).to(torch.uint8)
    ks = torch.rand(24, 2, BS, 1, generator=g)
    nk = torch.randn(3, 2, 2, 64, generator=g).to(torch.bfloat16)
    r = oracle.kv_append(nk, nk, bt, L, rc, fs, ft, kp8, kp8.clone(), ks, ks.clone(), scale_tile=64)
    shared = int(bt[0, 0])
    t0, t1 = r["block_table"][0, 0], r["block_table"][1, 0]
    ksr = r["k_scale"].reshape(24, 2, BS, 1)
    for t in (t0, t1):  # both views keep the shared history's codes and tile scales
        assert np.array_equal(r["k_pool"][t, :, :10], kp8[shared, :, :10].numpy())
        assert np.array_equal(ksr[t, :, :10], ks[shared, :, :10].numpy())
