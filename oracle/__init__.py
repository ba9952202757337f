"""CPU oracle for the paged speculative-verification step -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The library itself never does: it has no CPU fallback.

The arithmetic lives in ``svpa_oracle.c`` (plain C, fp64, OpenMP); this module
compiles it with gcc on first use and wraps it with numpy arrays.  It shares
no code with the CUDA library.

Parity status of each function (what pins it is in ``tests/test_oracle_*.py``):
  paged_verify_attn    pinned (library SDPA special case, brute force,
                       closed forms, block-permutation invariance, FP8 decode
                       table)
  spec_accept          pinned (Monte-Carlo output distribution = P, mean
                       accepted length = E[K] formula, special cases)
  spec_accept_logits   pinned (worked two-token example, softmax shift and
                       temperature identities, agreement with spec_accept on
                       the same rows, Monte-Carlo output distribution = P)
  spec_accept_tree     pinned (reduces to spec_accept on a chain; Monte-Carlo
                       distribution of the first emitted token = P[root])
  spec_accept_tree_logits
                       pinned (hand-worked three-token trees; reduces to
                       spec_accept_logits on a chain and to spec_accept_tree
                       on the softmax rows off the band; doubled logits at
                       temperature 2; Monte-Carlo distribution = P at the root
                       and at an accepted child)
  tree_logits_outcomes pinned (a zero band leaves exactly the sampler's own
                       outcome, a band of 1 every outcome, the default band
                       contains the sampler's outcome)
  block_table_commit   pinned (hand-worked example, conservation invariants,
                       tree compaction moves the path's K/V bytes)
  expected_accepted, speedup
                       pinned (the worked example: alpha >= 0.85, r ~ 0.08
                       gives eta >= 2.8)
  kv_append            pinned (gathered history ++ new rows, copy-on-write leaves
                       the other holders' pages untouched, conservation of
                       blocks; FP8: the scale rule on a worked page, decoded
                       values within half a code of the data)
  e4m3_encode          pinned (equals torch.float8_e4m3fn rounding on every
                       in-range value tested; saturation at 448)
  FP8 tile scales      pinned (attention: SDPA on pages decoded in the test
  (scale_tile=64)      with the scales broadcast to full rows; equal tile
                       scales reproduce the per-page result; append: every new
                       tile's scale and codes on a worked example)
  gamma_update,        pinned (estimator limit under simulated per-token
  gamma_from_alpha     acceptance, threshold edges, the moving average's closed
                       form, E[K] / speed-up closed forms and the worked example)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "svpa_oracle.c")
_LIB = os.path.join(_HERE, "libsvpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, OpenMP, no FMA contraction); return the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.oracle_paged_verify_attn.argtypes = [I] * 9 + [D] + [P] * 10 + [I]
            lib.oracle_paged_verify_attn.restype = I
            lib.oracle_spec_accept.argtypes = [I, I, I] + [P] * 9 + [I]
            lib.oracle_spec_accept.restype = I
            lib.oracle_spec_accept_logits.argtypes = [I, I, I, D, D, D] + [P] * 10 + [I]
            lib.oracle_spec_accept_logits.restype = I
            lib.oracle_logits_draw_window.argtypes = [I, I, I, D, D, D] + [P] * 6 + [I]
            lib.oracle_logits_draw_window.restype = I
            lib.oracle_spec_accept_tree.argtypes = [I, I, I] + [P] * 10 + [I]
            lib.oracle_spec_accept_tree.restype = I
            lib.oracle_spec_accept_tree_logits.argtypes = [I, I, I, P, D, D, D] + [P] * 9 + [I]
            lib.oracle_spec_accept_tree_logits.restype = I
            lib.oracle_tree_logits_outcomes.argtypes = [I, I, I, P, D, D, D] + [P] * 8 + [I]
            lib.oracle_tree_logits_outcomes.restype = I
            lib.oracle_block_table_commit.argtypes = [I] * 5 + [P] * 7 + [I, P, P, I, I, I]
            lib.oracle_block_table_commit.restype = I
            lib.oracle_tree_max_depth.argtypes = [P, I]
            lib.oracle_tree_max_depth.restype = I
            lib.oracle_expected_accepted.argtypes = [P, I]
            lib.oracle_expected_accepted.restype = D
            lib.oracle_speedup.argtypes = [D, I, D]
            lib.oracle_speedup.restype = D
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_double.restype = D
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_to_double.restype = D
            lib.oracle_kv_append.argtypes = [I] * 8 + [P] * 11
            lib.oracle_kv_append.restype = I
            lib.oracle_gamma_update.argtypes = [I, I] + [P] * 6 + [ctypes.c_float, ctypes.c_float]
            lib.oracle_gamma_update.restype = I
            lib.oracle_gamma_from_alpha.argtypes = [ctypes.c_float]
            lib.oracle_gamma_from_alpha.restype = I
            lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _c(a, dtype):
    """Contiguous numpy array of ``a`` as ``dtype`` (accepts torch CPU tensors).

    bf16 tensors become their uint16 bit patterns and FP8 tensors their bytes.
    """
    if a is None:
        return None
    if hasattr(a, "detach"):
        import torch
        t = a.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype.itemsize == 1 and t.dtype.is_floating_point:
            t = t.view(torch.uint8)
        a = t.numpy()
    a = np.asarray(a)
    dt = np.dtype(dtype)
    if a.dtype != dt and a.dtype.itemsize == dt.itemsize and dt.kind == "u" and a.dtype.kind in "iu":
        a = a.view(dt)
    return np.ascontiguousarray(a, dtype=dt)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    return _load().oracle_max_threads()


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def e4m3_to_double(byte: int) -> float:
    return _load().oracle_e4m3_to_double(int(byte))


def paged_verify_attn(q_bits, k_pool, v_pool, block_table, context_lens, *,
                      num_kv_heads, sm_scale, kv_fp8=False, k_scale=None,
                      v_scale=None, ancestor_mask=None, nthreads=0, scale_tile=0):
    """fp64 masked attention of each sequence's n_q queries over its paged history.

    q_bits: uint16 bf16 bits [B, n_q, Hq, D]; k_pool/v_pool: uint16 bf16 bits or
    uint8 E4M3 bytes [num_blocks, Hkv, BS, D]; block_table int32 [B, max_blocks];
    context_lens int32 [B]; ancestor_mask uint64 [n_q] or None (causal).
    FP8 scales: [num_blocks, Hkv] (scale_tile 0) or one per 64-element tile of
    a row, [num_blocks, Hkv, BS, D / 64] (scale_tile 64).
    Returns (out fp64 [B, n_q, Hq, D], lse fp64 [B, n_q, Hq]).
    """
    lib = _load()
    q = _c(q_bits, np.uint16)
    kp = _c(k_pool, np.uint8 if kv_fp8 else np.uint16)
    vp = _c(v_pool, np.uint8 if kv_fp8 else np.uint16)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    am = _c(ancestor_mask, np.uint64)
    B, n_q, Hq, D = q.shape
    num_blocks, Hkv, BS, D2 = kp.shape
    assert D2 == D and Hkv == num_kv_heads
    out = np.zeros((B, n_q, Hq, D), np.float64)
    lse = np.zeros((B, n_q, Hq), np.float64)
    rc = lib.oracle_paged_verify_attn(B, n_q, Hq, Hkv, D, BS, bt.shape[1], num_blocks,
                                      (2 if scale_tile == 64 else 1) if kv_fp8 else 0, float(sm_scale), _ptr(q),
                                      _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs), _ptr(bt),
                                      _ptr(cl), _ptr(am), _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_paged_verify_attn failed with status {rc}")
    return out, lse


def spec_accept(p_probs, q_probs, draft_tokens, u_accept, u_sample, nthreads=0):
    """Linear rejection sampler. Returns (accepted_len, out_tokens, near_boundary, dist)."""
    lib = _load()
    P = _c(p_probs, np.float32)
    Q = _c(q_probs, np.float32)
    x = _c(draft_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    B, g1, V = P.shape
    gamma = g1 - 1
    assert Q.shape == (B, gamma, V) and x.shape == (B, gamma)
    k = np.zeros(B, np.int32)
    out = np.zeros((B, gamma + 1), np.int32)
    near = np.zeros(B, np.uint8)
    dist = np.zeros(B, np.float64)
    rc = lib.oracle_spec_accept(B, gamma, V, _ptr(P), _ptr(Q), _ptr(x), _ptr(ua), _ptr(us),
                                _ptr(k), _ptr(out), _ptr(near), _ptr(dist), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_spec_accept failed with status {rc}")
    return k, out, near.astype(bool), dist


# Near-boundary band of the logits front-end: relative for the acceptance
# test, absolute (probability units) for the residual mass and the draw.  An
# fp32 formation of P and Q errs by ~1.2e-7 * |log2 P| relative per entry
# (exponent rounding, <= 1.6e-5 down to 2^-126) plus <= ~1e-5 in the
# normaliser (partial sums of <= 128 fp32 terms); 5e-5 covers both.
LOGIT_BAND = 5e-5


def spec_accept_logits(target_logits, draft_logits, draft_tokens, u_accept, u_sample, temperature=1.0,
                       draft_temperature=None, band=LOGIT_BAND, nthreads=0, tests=False):
    """Linear rejection sampler on P = softmax(Lp / T), Q = softmax(Lq / T_draft)
    formed in fp64.  Returns (accepted_len, out_tokens, near_boundary), and with
    tests=True also every acceptance test's decision and near flag [B, gamma]."""
    lib = _load()
    Lp = _c(target_logits, np.float32)
    Lq = _c(draft_logits, np.float32)
    x = _c(draft_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    B, g1, V = Lp.shape
    gamma = g1 - 1
    assert Lq.shape == (B, gamma, V) and x.shape == (B, gamma)
    assert ua.shape == (B, gamma) and us.shape == (B,)
    td = temperature if draft_temperature is None else draft_temperature
    k = np.zeros(B, np.int32)
    out = np.zeros((B, gamma + 1), np.int32)
    near = np.zeros(B, np.uint8)
    acc = np.zeros((B, gamma), np.uint8)
    accn = np.zeros((B, gamma), np.uint8)
    rc = lib.oracle_spec_accept_logits(B, gamma, V, float(temperature), float(td), float(band), _ptr(Lp),
                                       _ptr(Lq), _ptr(x), _ptr(ua), _ptr(us), _ptr(k), _ptr(out), _ptr(near),
                                       _ptr(acc), _ptr(accn), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_spec_accept_logits failed with status {rc}")
    if tests:
        return k, out, near.astype(bool), acc.astype(bool), accn.astype(bool)
    return k, out, near.astype(bool)


def logits_draw_window(target_logits, draft_logits, accepted_len, u_sample, temperature=1.0,
                       draft_temperature=None, band=LOGIT_BAND, nthreads=0):
    """For each row and its given accepted count k, the range [lo, hi] of
    tokens an fp32 formation of P and Q may draw (the running-sum intervals
    within `band` of u * Z).  Returns (lo, hi)."""
    lib = _load()
    Lp = _c(target_logits, np.float32)
    Lq = _c(draft_logits, np.float32)
    k = _c(accepted_len, np.int32)
    us = _c(u_sample, np.float32)
    B, g1, V = Lp.shape
    td = temperature if draft_temperature is None else draft_temperature
    lo = np.zeros(B, np.int32)
    hi = np.zeros(B, np.int32)
    rc = lib.oracle_logits_draw_window(B, g1 - 1, V, float(temperature), float(td), float(band), _ptr(Lp),
                                       _ptr(Lq), _ptr(k), _ptr(us), _ptr(lo), _ptr(hi), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_logits_draw_window failed with status {rc}")
    return lo, hi


def tree_max_depth(parent) -> int:
    par = _c(parent, np.int32)
    d = _load().oracle_tree_max_depth(_ptr(par), par.shape[0])
    if d < 0:
        raise OracleError("parent array is not a tree in node order")
    return d


def spec_accept_tree(parent, p_probs, q_probs, node_tokens, u_accept, u_sample, nthreads=0):
    """Tree rejection sampler. Returns (accepted_len, path_nodes, out_tokens, near)."""
    lib = _load()
    par = _c(parent, np.int32)
    P = _c(p_probs, np.float32)
    Q = _c(q_probs, np.float32)
    tok = _c(node_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    B, n_nodes, V = P.shape
    W = tree_max_depth(par) + 1
    k = np.zeros(B, np.int32)
    path = np.zeros((B, W), np.int32)
    out = np.zeros((B, W), np.int32)
    near = np.zeros(B, np.uint8)
    rc = lib.oracle_spec_accept_tree(B, n_nodes, V, _ptr(par), _ptr(P), _ptr(Q), _ptr(tok),
                                     _ptr(ua), _ptr(us), _ptr(k), _ptr(path), _ptr(out),
                                     _ptr(near), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_spec_accept_tree failed with status {rc}")
    return k, path, out, near.astype(bool)


def spec_accept_tree_logits(parent, target_logits, draft_logits, node_tokens, u_accept, u_sample, temperature=1.0,
                            draft_temperature=None, band=LOGIT_BAND, nthreads=0):
    """Tree rejection sampler on P = softmax(Lp / T) at every node and
    Q = softmax(Lq / T_draft) at every internal node, formed in fp64.
    Returns (accepted_len, path_nodes, out_tokens, near)."""
    lib = _load()
    par = _c(parent, np.int32)
    Lp = _c(target_logits, np.float32)
    Lq = _c(draft_logits, np.float32)
    tok = _c(node_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    B, n_nodes, V = Lp.shape
    assert par.shape == (n_nodes,) and tok.shape == (B, n_nodes) and ua.shape == (B, n_nodes)
    assert Lq.shape[0] == B and Lq.shape[2] == V and us.shape == (B,)
    td = temperature if draft_temperature is None else draft_temperature
    W = tree_max_depth(par) + 1
    k = np.zeros(B, np.int32)
    path = np.zeros((B, W), np.int32)
    out = np.zeros((B, W), np.int32)
    near = np.zeros(B, np.uint8)
    rc = lib.oracle_spec_accept_tree_logits(B, n_nodes, V, _ptr(par), float(temperature), float(td), float(band),
                                            _ptr(Lp), _ptr(Lq), _ptr(tok), _ptr(ua), _ptr(us), _ptr(k),
                                            _ptr(path), _ptr(out), _ptr(near), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_spec_accept_tree_logits failed with status {rc}")
    return k, path, out, near.astype(bool)


def tree_logits_outcomes(parent, target_logits, draft_logits, node_tokens, u_accept, u_sample, temperature=1.0,
                         draft_temperature=None, band=LOGIT_BAND, nthreads=0):
    """Per sequence and node: whether an fp32 formation of the tree sampler
    fed by logits may end its walk there, and the range [lo, hi] of tokens its
    final draw there may give.  Returns (end_ok [B, n_nodes] bool, lo, hi)."""
    lib = _load()
    par = _c(parent, np.int32)
    Lp = _c(target_logits, np.float32)
    Lq = _c(draft_logits, np.float32)
    tok = _c(node_tokens, np.int32)
    ua = _c(u_accept, np.float32)
    us = _c(u_sample, np.float32)
    B, n_nodes, V = Lp.shape
    td = temperature if draft_temperature is None else draft_temperature
    ok = np.zeros((B, n_nodes), np.uint8)
    lo = np.zeros((B, n_nodes), np.int32)
    hi = np.zeros((B, n_nodes), np.int32)
    rc = lib.oracle_tree_logits_outcomes(B, n_nodes, V, _ptr(par), float(temperature), float(td), float(band),
                                         _ptr(Lp), _ptr(Lq), _ptr(tok), _ptr(ua), _ptr(us), _ptr(ok), _ptr(lo),
                                         _ptr(hi), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_tree_logits_outcomes failed with status {rc}")
    return ok.astype(bool), lo, hi


def block_table_commit(block_table, context_lens, accepted_len, refcount, free_stack,
                       free_top, *, n_q, block_size=16, path_nodes=None, k_pool=None,
                       v_pool=None):
    """Commit/rollback on copies of the inputs; returns the updated copies.

    Returns dict(block_table, context_lens, refcount, free_stack, free_top,
    k_pool, v_pool) -- pools only when path_nodes is given (tree compaction).
    """
    lib = _load()
    bt = _c(block_table, np.int32).copy()
    cl = _c(context_lens, np.int32).copy()
    k = _c(accepted_len, np.int32)
    rcnt = _c(refcount, np.int32).copy()
    fs = _c(free_stack, np.int32).copy()
    ft = np.array([int(free_top)], np.int32)
    B, max_blocks = bt.shape
    num_blocks = rcnt.shape[0]
    path = _c(path_nodes, np.int32)
    kp = vp = None
    Hkv = D = eb = 0
    if path is not None:
        kp = np.ascontiguousarray(np.asarray(k_pool)).copy()
        vp = np.ascontiguousarray(np.asarray(v_pool)).copy()
        _, Hkv, _, D = kp.shape
        eb = kp.dtype.itemsize
    rc = lib.oracle_block_table_commit(B, n_q, block_size, max_blocks, num_blocks, _ptr(bt),
                                       _ptr(cl), _ptr(k), _ptr(rcnt), _ptr(fs), _ptr(ft),
                                       _ptr(path), 0 if path is None else path.shape[1],
                                       _ptr(kp), _ptr(vp), Hkv, D, eb)
    if rc != 0:
        raise OracleError(f"oracle_block_table_commit failed with status {rc}")
    return dict(block_table=bt, context_lens=cl, refcount=rcnt, free_stack=fs,
                free_top=int(ft[0]), k_pool=kp, v_pool=vp)


def kv_append(new_k, new_v, block_table, context_lens, refcount, free_stack, free_top, k_pool,
              v_pool, k_scale=None, v_scale=None, *, block_size=16, scale_tile=0):
    """Append the new rows on copies of the inputs; returns the updated copies.

    new_k, new_v: bf16 [B, n_new, Hkv, D]; pools bf16 or float8_e4m3fn (or raw
    uint16 / uint8 arrays) [num_blocks, Hkv, 16, D]; scales fp32 for FP8.
    Returns dict(block_table, refcount, free_stack, free_top, k_pool, v_pool,
    k_scale, v_scale) -- pools as raw uint16 (bf16 bits) or uint8 (E4M3 bytes).
    """
    lib = _load()
    nk = _c(new_k, np.uint16)
    nv = _c(new_v, np.uint16)
    B, n_new, Hkv, D = nk.shape
    bt = _c(block_table, np.int32).copy()
    cl = _c(context_lens, np.int32)
    rcnt = _c(refcount, np.int32).copy()
    fs = _c(free_stack, np.int32).copy()
    ft = np.array([int(free_top)], np.int32)
    isz = k_pool.element_size() if hasattr(k_pool, "element_size") else np.asarray(k_pool).itemsize
    raw = np.uint8 if isz == 1 else np.uint16
    kp = _c(k_pool, raw).copy()
    vp = _c(v_pool, raw).copy()
    fp8 = isz == 1
    ks = _c(k_scale, np.float32).copy() if fp8 else None
    vs = _c(v_scale, np.float32).copy() if fp8 else None
    mode = (2 if scale_tile == 64 else 1) if fp8 else 0
    rc = lib.oracle_kv_append(B, n_new, Hkv, D, block_size, bt.shape[1], rcnt.shape[0], mode,
                              _ptr(nk), _ptr(nv), _ptr(bt), _ptr(cl), _ptr(rcnt), _ptr(fs), _ptr(ft),
                              _ptr(kp), _ptr(vp), _ptr(ks), _ptr(vs))
    if rc != 0:
        raise OracleError(f"oracle_kv_append failed with status {rc}")
    return dict(block_table=bt, refcount=rcnt, free_stack=fs, free_top=int(ft[0]), k_pool=kp,
                v_pool=vp, k_scale=ks, v_scale=vs)


def e4m3_encode(x) -> np.ndarray:
    """OCP E4M3 codes (uint8) of fp32 values: nearest, ties to even, saturating at 448."""
    lib = _load()
    a = np.asarray(x, np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in a], np.uint8).reshape(np.shape(x))


def expected_accepted(alpha) -> float:
    a = np.ascontiguousarray(np.asarray(alpha, np.float64))
    return _load().oracle_expected_accepted(_ptr(a), a.shape[0])


def speedup(expected_k: float, gamma: int, r: float) -> float:
    return _load().oracle_speedup(float(expected_k), int(gamma), float(r))


def gamma_from_alpha(alpha: float) -> int:
    """Draft length for an acceptance-rate estimate (fp32 comparison)."""
    return int(_load().oracle_gamma_from_alpha(float(alpha)))


def gamma_update(gamma, accepted_len, seq_state=None, batch_state=(0.0, 0.0), *, decay=0.9, r=0.0):
    """One step of the acceptance moving averages on copies of the state.

    Returns dict(seq_state [B, 2] fp32 or None, seq_gamma [B] int32 or None,
    batch_state [2] fp32, batch_gamma int, telemetry [4] fp32: batch alpha,
    mean accepted this step, E[K], speed-up at ratio r)."""
    lib = _load()
    k = _c(accepted_len, np.int32)
    B = k.shape[0]
    ss = None if seq_state is None else _c(seq_state, np.float32).reshape(B, 2).copy()
    sg = None if seq_state is None else np.zeros(B, np.int32)
    bs = np.asarray(batch_state, np.float32).copy()
    bg = np.zeros(1, np.int32)
    tel = np.zeros(4, np.float32)
    rc = lib.oracle_gamma_update(B, int(gamma), _ptr(k), _ptr(ss), _ptr(sg), _ptr(bs), _ptr(bg), _ptr(tel),
                                 float(decay), float(r))
    if rc != 0:
        raise OracleError(f"oracle_gamma_update failed with status {rc}")
    return dict(seq_state=ss, seq_gamma=sg, batch_state=bs, batch_gamma=int(bg[0]), telemetry=tel)
