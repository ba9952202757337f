"""The C-ABI library builds, loads and exports every entry point the header
declares; host-side validation answers without touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from speculative_verify_paged_attn_gb300 import build, svpa
    build.build()
    return svpa.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "svpa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(svpa_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from speculative_verify_paged_attn_gb300 import svpa
    for code in range(8):
        assert svpa.status_string(code)
    assert svpa.version() >= 100


def test_workspace_size_and_validation(lib):
    from speculative_verify_paged_attn_gb300 import svpa
    p = svpa.attn_params(64, 6, 64, 8, 128, 2049, 100000, split_pages=256)
    n = svpa.attn_workspace_size(p)
    # tickets + (max, sum) + accumulators for 9 splits of 48 rows
    assert n >= 64 * 8 * 9 * 48 * (128 + 2) * 4
    for bad in [dict(head_dim=96), dict(num_kv_heads=5), dict(n_q=65)]:
        kw = dict(batch=2, n_q=5, num_q_heads=4, num_kv_heads=4, head_dim=64,
                  max_blocks_per_seq=8, num_blocks=16, split_pages=4)
        kw.update(bad)
        with pytest.raises(svpa.SvpaError):
            svpa.attn_workspace_size(svpa.attn_params(**kw))
    # unsplit units with more units than resident CTAs are ranked first (2 launches)
    assert svpa.attn_launches(svpa.attn_params(128, 29, 32, 8, 128, 600, 100000)) in (1, 2)
    assert svpa.attn_launches(svpa.attn_params(2, 5, 4, 4, 64, 8, 16)) == 1
    assert svpa.attn_launches(svpa.attn_params(0, 5, 4, 4, 64, 8, 16)) == 0
    # which kernel runs: warp-level MMA for few rows per kv head, tcgen05 for many
    assert svpa.attn_kernel(svpa.attn_params(32, 5, 32, 32, 128, 256, 4096)) == 1
    assert svpa.attn_kernel(svpa.attn_params(64, 6, 64, 8, 128, 2049, 100000)) == 2
    assert svpa.attn_kernel(svpa.attn_params(64, 6, 64, 8, 128, 2049, 100000, variant=1)) == 1
    assert svpa.attn_kernel(svpa.attn_params(16, 6, 64, 8, 128, 2049, 100000, kv_fp8=True)) == 2
    assert svpa.attn_kernel(svpa.attn_params(16, 29, 32, 8, 128, 600, 100000, kv_fp8=True)) == 1
    # FP8 pages on the tcgen05 kernel take at most 64 rows per kv head
    with pytest.raises(svpa.SvpaError) as e:
        svpa.attn_workspace_size(svpa.attn_params(2, 9, 64, 8, 128, 8, 16, kv_fp8=True, variant=2))
    assert e.value.status == 2
    assert svpa.attn_workspace_size(svpa.attn_params(2, 8, 64, 8, 128, 8, 16, kv_fp8=True, variant=2)) > 0
    # 64-element FP8 tile scales run on the tcgen05 kernel only
    tile = dict(kv_fp8=True, scale_tile=64)
    assert svpa.attn_kernel(svpa.attn_params(16, 6, 64, 8, 128, 2049, 100000, **tile)) == 2
    for bad, code in [(dict(variant=1), 2), (dict(n_q=9), 2), (dict(kv_fp8=False), 2), (dict(scale_tile=32), 1)]:
        kw = dict(kv_fp8=True, scale_tile=64)
        kw.update(bad)
        n_q = kw.pop("n_q", 6)
        with pytest.raises(svpa.SvpaError) as e:
            svpa.attn_workspace_size(svpa.attn_params(2, n_q, 64, 8, 128, 8, 16, **kw))
        assert e.value.status == code, bad
    # GQA rows per CTA beyond 128 are not supported
    with pytest.raises(svpa.SvpaError) as e:
        svpa.attn_workspace_size(svpa.attn_params(1, 17, 64, 8, 128, 8, 16, split_pages=4))
    assert e.value.status == 2


def test_null_pointers_rejected_before_launch(lib):
    from speculative_verify_paged_attn_gb300 import svpa
    p = svpa.attn_params(2, 5, 4, 4, 64, 8, 16, split_pages=4)
    st = lib.svpa_paged_verify_attn(ctypes.byref(p), *([None] * 11), 0, None, None)
    assert st == 1
    st = lib.svpa_spec_accept(2, 4, 1000, *([None] * 9), 0, None, None)
    assert st == 1
    st = lib.svpa_spec_accept(2, 0, 1000, *([None] * 9), 0, None, None)
    assert st == 1
    st = lib.svpa_block_table_commit(2, 5, 16, 8, 16, *([None] * 7), 0, None, None, 4, 64, 0, None, None)
    assert st == 1
    # K/V append: sizes checked first, then pointers, then alignment
    nz = ctypes.c_void_p(16)  # never dereferenced: validation returns before any launch
    base = [2, 5, 4, 64, 16, 8, 16, 0, 0]
    assert lib.svpa_kv_append(*base, *([None] * 13)) == 1
    for bad in [dict(n=0), dict(n=4097), dict(d=60), dict(bs=32), dict(dt=2), dict(h=0), dict(tile=32)]:
        a = list(base)
        a[1], a[3], a[4], a[7], a[2], a[8] = (bad.get("n", 5), bad.get("d", 64), bad.get("bs", 16),
                                              bad.get("dt", 0), bad.get("h", 4), bad.get("tile", 0))
        assert lib.svpa_kv_append(*a, *([nz] * 13)) == 1, bad
    # FP8 tiles: head_dim a multiple of 16, at most 256
    for d in (72, 272):
        assert lib.svpa_kv_append(2, 5, 4, d, 16, 8, 16, 1, 0, *([nz] * 13)) == 1, d
    # 64-element tile scales: FP8 pools with head_dim a multiple of 64 only
    assert lib.svpa_kv_append(2, 5, 4, 64, 16, 8, 16, 0, 64, *([nz] * 13)) == 1
    assert lib.svpa_kv_append(2, 5, 4, 80, 16, 8, 16, 1, 64, *([nz] * 13)) == 1
    # FP8 pools need both scale arrays
    assert lib.svpa_kv_append(2, 5, 4, 64, 16, 8, 16, 1, 0, *([nz] * 9), None, None, nz, None) == 1
    # a pool that is not 16-byte aligned
    odd = ctypes.c_void_p(24)
    assert lib.svpa_kv_append(*base, nz, nz, nz, nz, nz, nz, nz, odd, nz, None, None, nz, None) == 1
    assert lib.svpa_kv_append(0, 5, 4, 64, 16, 8, 16, 0, 0, *([None] * 13)) == 0
    # adaptive draft length: sizes, decay and ratio checked before any launch
    F = ctypes.c_float
    for args in [(0, 4, F(0.9), F(0.0)), (2, 0, F(0.9), F(0.0)), (2, 64, F(0.9), F(0.0)),
                 (2, 4, F(1.5), F(0.0)), (2, 4, F(0.9), F(-1.0)), (2, 4, F(float("nan")), F(0.0))]:
        b, g, d, r = args
        assert lib.svpa_gamma_update(b, g, nz, None, None, nz, nz, nz, d, r, nz, None) == 1, args
    assert lib.svpa_gamma_update(2, 4, nz, None, nz, nz, nz, nz, F(0.9), F(0.0), nz, None) == 1
    assert lib.svpa_gamma_update(2, 4, None, None, None, nz, nz, nz, F(0.9), F(0.0), nz, None) == 1
    # logits front-end: sizes, temperatures, vocabulary, pointers, workspace
    for args in [(2, 0, 1000, F(1.0), F(1.0)), (2, 33, 1000, F(1.0), F(1.0)), (2, 4, 0, F(1.0), F(1.0)),
                 (2, 4, 1000, F(0.0), F(1.0)), (2, 4, 1000, F(1.0), F(-0.5)),
                 (2, 4, 1000, F(float("inf")), F(1.0)), (2, 4, 1000, F(1.0), F(float("nan"))),
                 (2, 4, 1000, F(1e-39), F(1.0))]:
        assert lib.svpa_spec_accept_logits(*args, *([nz] * 9), 256, nz, None) == 1, args
    assert lib.svpa_spec_accept_logits(2, 4, 262145, F(1.0), F(1.0), *([nz] * 9), 256, nz, None) == 2
    assert lib.svpa_spec_accept_logits(2, 4, 1000, F(1.0), F(1.0), *([None] * 9), 0, None, None) == 1
    assert lib.svpa_spec_accept_logits(2, 4, 1000, F(1.0), F(1.0), *([nz] * 8), None, 0, nz, None) == 6
    assert lib.svpa_spec_accept_logits(2, 4, 1000, F(1.0), F(1.0), *([nz] * 8), odd, 256, nz, None) == 6
    assert lib.svpa_spec_accept_logits(0, 4, 1000, F(0.7), F(1.0), *([None] * 9), 0, None, None) == 0
    # its workspace: one (max, sum) pair per 8192-token slab of each of the 2 gamma + 1 rows
    n = ctypes.c_size_t(0)
    assert lib.svpa_spec_accept_logits_workspace_size(2, 4, 32000, ctypes.byref(n)) == 0
    assert n.value == 768  # 2 * 9 * 4 * 8 = 576 bytes, in 256-byte units
    assert lib.svpa_spec_accept_logits_workspace_size(64, 5, 128256, ctypes.byref(n)) == 0
    assert n.value == 64 * 11 * 16 * 8
    assert lib.svpa_spec_accept_logits_workspace_size(1, 1, 1, ctypes.byref(n)) == 0 and n.value == 256
    assert lib.svpa_spec_accept_logits_workspace_size(2, 0, 1000, ctypes.byref(n)) == 1
    assert lib.svpa_spec_accept_logits_workspace_size(2, 4, 262145, ctypes.byref(n)) == 2
    ws = ctypes.c_void_p(256)
    assert lib.svpa_spec_accept_logits(2, 4, 32000, F(1.0), F(1.0), *([nz] * 8), ws, 512, nz, None) == 6
    # empty batch is a no-op
    p0 = svpa.attn_params(0, 5, 4, 4, 64, 8, 16, split_pages=4)
    assert lib.svpa_paged_verify_attn(ctypes.byref(p0), *([None] * 11), 0, None, None) == 0


def test_tree_topology_validated(lib):
    par = (ctypes.c_int32 * 3)(-1, 0, 2)   # node 2 names itself as parent
    st = lib.svpa_spec_accept_tree(1, 3, 10, ctypes.cast(par, ctypes.c_void_p), *([None] * 10),
                                   0, None, None)
    assert st == 1


def test_tree_logits_arguments_validated(lib):
    F = ctypes.c_float
    nz = ctypes.c_void_p(16)
    good = (ctypes.c_int32 * 3)(-1, 0, 0)
    bad = (ctypes.c_int32 * 3)(-1, 1, 0)  # a parent after its child
    g = ctypes.cast(good, ctypes.c_void_p)
    assert lib.svpa_spec_accept_tree_logits(1, 3, 10, ctypes.cast(bad, ctypes.c_void_p), F(1.0), F(1.0),
                                            *([nz] * 11)) == 1
    assert lib.svpa_spec_accept_tree_logits(1, 3, 10, None, F(1.0), F(1.0), *([nz] * 11)) == 1
    assert lib.svpa_spec_accept_tree_logits(1, 65, 10, g, F(1.0), F(1.0), *([nz] * 11)) == 1
    for t, td in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf")), (1e-39, 1.0)):
        assert lib.svpa_spec_accept_tree_logits(1, 3, 10, g, F(t), F(td), *([nz] * 11)) == 1, (t, td)
    assert lib.svpa_spec_accept_tree_logits(1, 3, 262145, g, F(1.0), F(1.0), *([nz] * 11)) == 2
    assert lib.svpa_spec_accept_tree_logits(1, 3, 10, g, F(1.0), F(1.0), *([None] * 11)) == 1
    # the error word is required
    assert lib.svpa_spec_accept_tree_logits(1, 3, 10, g, F(1.0), F(1.0), *([nz] * 9), None, None) == 1
    assert lib.svpa_spec_accept_tree_logits(0, 3, 10, g, F(1.0), F(1.0), *([None] * 11)) == 0


def test_library_is_not_the_oracle(lib):
    # the product library must not link or contain the CPU oracle
    from speculative_verify_paged_attn_gb300 import svpa
    data = open(svpa.LIB_PATH, "rb").read()
    assert b"oracle_" not in data


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_standalone(lang, std, tmp_path):
    """include/svpa.h is usable from plain C and from C++ with no other header
    (stdint/stddef only), with no warnings."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "svpa.h"\nint main(void) { return (int)SVPA_OK; }\n')
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                        os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
