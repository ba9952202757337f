"""ctypes binding of libsvpa.so -- argument marshalling only.

Every function here forwards to the C entry point of the same name in
``include/svpa.h``: it checks nothing the library does not check itself,
computes nothing, and passes device pointers (``tensor.data_ptr()``) plus the
current CUDA stream.  Device memory is allocated by the caller (PyTorch).

There is no CPU fallback: if the compiled library is missing, importing the
library raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsvpa.so")

SVPA_KV_BF16 = 0
SVPA_KV_FP8_E4M3 = 1
STATUS = {0: "SVPA_OK", 1: "SVPA_ERR_INVALID_ARG", 2: "SVPA_ERR_UNSUPPORTED", 3: "SVPA_ERR_CUDA",
          4: "SVPA_ERR_OUT_OF_BLOCKS", 5: "SVPA_ERR_BAD_BLOCK", 6: "SVPA_ERR_WORKSPACE",
          7: "SVPA_ERR_TIMEOUT"}
EXPORTS = ("svpa_attn_workspace_size", "svpa_attn_kernel", "svpa_paged_verify_attn", "svpa_spec_accept_workspace_size",
           "svpa_spec_accept", "svpa_spec_accept_tree", "svpa_block_table_commit", "svpa_check_error",
           "svpa_status_string", "svpa_version", "svpa_paged_verify_attn_noalloc", "svpa_kv_append",
           "svpa_gamma_update", "svpa_attn_launches", "svpa_spec_accept_logits",
           "svpa_spec_accept_logits_workspace_size", "svpa_wait_selftest", "svpa_spec_accept_tree_logits")


class SvpaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class AttnParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("max_blocks_per_seq", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("split_pages", ctypes.c_int32),
                ("variant", ctypes.c_int32), ("scale_tile", ctypes.c_int32)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libsvpa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsvpa.so not found at {path}; build it with "
                           "`python -m speculative_verify_paged_attn_gb300.build`")
    L = ctypes.CDLL(path)
    P, I, U, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    L.svpa_attn_workspace_size.argtypes = [ctypes.POINTER(AttnParams), ctypes.POINTER(U)]
    L.svpa_attn_kernel.argtypes = [ctypes.POINTER(AttnParams), ctypes.POINTER(I)]
    L.svpa_attn_launches.argtypes = [ctypes.POINTER(AttnParams), ctypes.POINTER(I)]
    L.svpa_paged_verify_attn.argtypes = [ctypes.POINTER(AttnParams)] + [P] * 11 + [U, P, P]
    L.svpa_spec_accept_workspace_size.argtypes = [I, I, ctypes.POINTER(U)]
    L.svpa_spec_accept.argtypes = [I, I, I] + [P] * 9 + [U, P, P]
    L.svpa_spec_accept_tree.argtypes = [I, I, I] + [P] * 11 + [U, P, P]
    L.svpa_spec_accept_logits.argtypes = [I, I, I, ctypes.c_float, ctypes.c_float] + [P] * 9 + [U, P, P]
    L.svpa_spec_accept_logits_workspace_size.argtypes = [I, I, I, ctypes.POINTER(U)]
    L.svpa_spec_accept_tree_logits.argtypes = [I, I, I, P, ctypes.c_float, ctypes.c_float] + [P] * 11
    L.svpa_block_table_commit.argtypes = [I] * 5 + [P] * 7 + [I, P, P, I, I, I, P, P]
    L.svpa_paged_verify_attn_noalloc.argtypes = [ctypes.POINTER(AttnParams)] + [P] * 12
    L.svpa_kv_append.argtypes = [I] * 9 + [P] * 13
    L.svpa_gamma_update.argtypes = [I, I] + [P] * 6 + [ctypes.c_float, ctypes.c_float, P, P]
    L.svpa_check_error.argtypes = [P, P]
    L.svpa_wait_selftest.argtypes = [ctypes.c_uint64, P, P, P]
    L.svpa_status_string.argtypes = [I]
    L.svpa_status_string.restype = ctypes.c_char_p
    L.svpa_version.argtypes = []
    for name in EXPORTS:
        if name != "svpa_status_string":
            getattr(L, name).restype = I
    _lib = L
    return L


def _p(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != 0:
        raise SvpaError(status, what)


VARIANT_AUTO, VARIANT_MMA, VARIANT_TCGEN05 = 0, 1, 2


def attn_params(batch, n_q, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_blocks,
                kv_fp8=False, sm_scale=None, split_pages=0, block_size=16, variant=0,
                scale_tile=0) -> AttnParams:
    return AttnParams(batch, n_q, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_blocks, SVPA_KV_FP8_E4M3 if kv_fp8 else SVPA_KV_BF16,
                      1.0 / math.sqrt(head_dim) if sm_scale is None else sm_scale, split_pages,
                      variant, scale_tile)


def attn_workspace_size(params: AttnParams) -> int:
    n = ctypes.c_size_t(0)
    _check(load().svpa_attn_workspace_size(ctypes.byref(params), ctypes.byref(n)),
           "svpa_attn_workspace_size")
    return n.value


def attn_kernel(params: AttnParams) -> int:
    """The attention kernel the library runs for `params`: 1 warp-level MMA, 2 tcgen05."""
    k = ctypes.c_int32(0)
    _check(load().svpa_attn_kernel(ctypes.byref(params), ctypes.byref(k)), "svpa_attn_kernel")
    return k.value


def attn_launches(params: AttnParams) -> int:
    """Kernel launches of one svpa_paged_verify_attn call for `params` (1, or 2 with the unit ranking)."""
    n = ctypes.c_int32(0)
    _check(load().svpa_attn_launches(ctypes.byref(params), ctypes.byref(n)), "svpa_attn_launches")
    return n.value


def spec_accept_workspace_size(batch: int, vocab: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().svpa_spec_accept_workspace_size(batch, vocab, ctypes.byref(n)),
           "svpa_spec_accept_workspace_size")
    return n.value


def _mask_array(mask: Optional[Sequence[int]]):
    if mask is None:
        return None
    vals = [int(m) & ((1 << 64) - 1) for m in (mask.tolist() if hasattr(mask, "tolist") else mask)]
    return (ctypes.c_uint64 * len(vals))(*vals)


def paged_verify_attn(params: AttnParams, q, k_pool, v_pool, block_table, context_lens, out, *,
                      workspace, error_flag, k_scale=None, v_scale=None, ancestor_mask=None,
                      lse=None, stream=None, check=True) -> int:
    """svpa_paged_verify_attn.  ancestor_mask: host sequence of n_q 64-bit masks or None."""
    m = _mask_array(ancestor_mask)
    st = load().svpa_paged_verify_attn(
        ctypes.byref(params), _p(q), _p(k_pool), _p(v_pool), _p(k_scale), _p(v_scale),
        _p(block_table), _p(context_lens), None if m is None else ctypes.cast(m, ctypes.c_void_p),
        _p(out), _p(lse), _p(workspace), workspace.numel() * workspace.element_size(),
        _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_paged_verify_attn")
    return st


def paged_verify_attn_noalloc(params: AttnParams, q, k_pool, v_pool, block_table, context_lens, out,
                              *, error_flag, k_scale=None, v_scale=None, ancestor_mask=None,
                              lse=None, stream=None, check=True) -> int:
    """svpa_paged_verify_attn_noalloc: no workspace argument; the library's own
    fixed scratch array is used (for callers that may not allocate)."""
    m = _mask_array(ancestor_mask)
    st = load().svpa_paged_verify_attn_noalloc(
        ctypes.byref(params), _p(q), _p(k_pool), _p(v_pool), _p(k_scale), _p(v_scale),
        _p(block_table), _p(context_lens), None if m is None else ctypes.cast(m, ctypes.c_void_p),
        _p(out), _p(lse), _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_paged_verify_attn_noalloc")
    return st


def spec_accept(p_probs, q_probs, draft_tokens, u_accept, u_sample, accepted_len, out_tokens, *,
                workspace, error_flag, near_boundary=None, stream=None, check=True) -> int:
    B, g1, V = p_probs.shape
    st = load().svpa_spec_accept(B, g1 - 1, V, _p(p_probs), _p(q_probs), _p(draft_tokens),
                                 _p(u_accept), _p(u_sample), _p(accepted_len), _p(out_tokens),
                                 _p(near_boundary), _p(workspace),
                                 workspace.numel() * workspace.element_size(), _p(error_flag),
                                 _stream(stream))
    if check:
        _check(st, "svpa_spec_accept")
    return st


def spec_accept_logits_workspace_size(batch: int, gamma: int, vocab: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().svpa_spec_accept_logits_workspace_size(batch, gamma, vocab, ctypes.byref(n)),
           "svpa_spec_accept_logits_workspace_size")
    return n.value


def spec_accept_logits(target_logits, draft_logits, draft_tokens, u_accept, u_sample, accepted_len, out_tokens,
                       *, workspace, error_flag, temperature=1.0, draft_temperature=None, near_boundary=None,
                       stream=None, check=True) -> int:
    """The linear sampler on P = softmax(target_logits / T), Q = softmax(draft_logits / T_draft)."""
    B, g1, V = target_logits.shape
    td = temperature if draft_temperature is None else draft_temperature
    st = load().svpa_spec_accept_logits(B, g1 - 1, V, float(temperature), float(td), _p(target_logits),
                                        _p(draft_logits), _p(draft_tokens), _p(u_accept), _p(u_sample),
                                        _p(accepted_len), _p(out_tokens), _p(near_boundary), _p(workspace),
                                        workspace.numel() * workspace.element_size(), _p(error_flag),
                                        _stream(stream))
    if check:
        _check(st, "svpa_spec_accept_logits")
    return st


def spec_accept_tree(parent: Sequence[int], p_probs, q_probs, node_tokens, u_accept, u_sample,
                     accepted_len, path_nodes, out_tokens, *, error_flag, near_boundary=None,
                     workspace=None, stream=None, check=True) -> int:
    """parent: host sequence (parent[0] = -1)."""
    par = [int(x) for x in (parent.tolist() if hasattr(parent, "tolist") else parent)]
    arr = (ctypes.c_int32 * len(par))(*par)
    B, n, V = p_probs.shape
    st = load().svpa_spec_accept_tree(B, n, V, ctypes.cast(arr, ctypes.c_void_p), _p(p_probs),
                                      _p(q_probs), _p(node_tokens), _p(u_accept), _p(u_sample),
                                      _p(accepted_len), _p(path_nodes), _p(out_tokens),
                                      _p(near_boundary), _p(workspace),
                                      0 if workspace is None else workspace.numel() * workspace.element_size(),
                                      _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_spec_accept_tree")
    return st


def spec_accept_tree_logits(parent: Sequence[int], target_logits, draft_logits, node_tokens, u_accept, u_sample,
                            accepted_len, path_nodes, out_tokens, *, error_flag, temperature=1.0,
                            draft_temperature=None, near_boundary=None, stream=None, check=True) -> int:
    """The draft-tree sampler on P = softmax(target_logits / T) at every node and
    Q = softmax(draft_logits / T_draft) at every internal node; parent: host
    sequence (parent[0] = -1)."""
    par = [int(x) for x in (parent.tolist() if hasattr(parent, "tolist") else parent)]
    arr = (ctypes.c_int32 * len(par))(*par)
    B, n, V = target_logits.shape
    td = temperature if draft_temperature is None else draft_temperature
    st = load().svpa_spec_accept_tree_logits(B, n, V, ctypes.cast(arr, ctypes.c_void_p), float(temperature),
                                             float(td), _p(target_logits), _p(draft_logits), _p(node_tokens),
                                             _p(u_accept), _p(u_sample), _p(accepted_len), _p(path_nodes),
                                             _p(out_tokens), _p(near_boundary), _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_spec_accept_tree_logits")
    return st


def block_table_commit(n_q, block_table, context_lens, accepted_len, refcount, free_stack, free_top,
                       *, error_flag, path_nodes=None, k_pool=None, v_pool=None, num_kv_heads=0,
                       head_dim=0, kv_fp8=False, stream=None, check=True) -> int:
    B, max_blocks = block_table.shape
    st = load().svpa_block_table_commit(
        B, n_q, 16, max_blocks, refcount.shape[0], _p(block_table), _p(context_lens),
        _p(accepted_len), _p(refcount), _p(free_stack), _p(free_top), _p(path_nodes),
        0 if path_nodes is None else path_nodes.shape[1], _p(k_pool), _p(v_pool), num_kv_heads,
        head_dim, SVPA_KV_FP8_E4M3 if kv_fp8 else SVPA_KV_BF16, _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_block_table_commit")
    return st


def kv_append(new_k, new_v, block_table, context_lens, refcount, free_stack, free_top, k_pool, v_pool,
              *, error_flag, k_scale=None, v_scale=None, scale_tile=0, stream=None, check=True) -> int:
    """svpa_kv_append: write new_k/new_v [B, n_new, Hkv, D] (bf16) at positions
    context_lens[b] .. + n_new - 1, allocating and cloning pages as needed; the
    pools are bf16 or float8_e4m3fn/uint8 [num_blocks, Hkv, 16, D]."""
    B, n_new, Hkv, D = new_k.shape
    fp8 = k_pool.element_size() == 1
    st = load().svpa_kv_append(
        B, n_new, Hkv, D, 16, block_table.shape[1], k_pool.shape[0],
        SVPA_KV_FP8_E4M3 if fp8 else SVPA_KV_BF16, scale_tile, _p(new_k), _p(new_v), _p(block_table),
        _p(context_lens), _p(refcount), _p(free_stack), _p(free_top), _p(k_pool), _p(v_pool),
        _p(k_scale), _p(v_scale), _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_kv_append")
    return st


def gamma_update(gamma, accepted_len, batch_state, batch_gamma, telemetry, *, error_flag, seq_state=None,
                 seq_gamma=None, decay=0.9, draft_cost_ratio=0.0, stream=None, check=True) -> int:
    """svpa_gamma_update: acceptance moving averages (per sequence when
    seq_state [B, 2] is given, and for the batch in batch_state [2]) and the
    draft length of the next step (seq_gamma [B], batch_gamma [1])."""
    st = load().svpa_gamma_update(
        accepted_len.shape[0], gamma, _p(accepted_len), _p(seq_state), _p(seq_gamma), _p(batch_state),
        _p(batch_gamma), _p(telemetry), float(decay), float(draft_cost_ratio), _p(error_flag), _stream(stream))
    if check:
        _check(st, "svpa_gamma_update")
    return st


def check_error(error_flag, stream=None) -> int:
    """svpa_check_error: synchronise the stream and map the device error word."""
    return load().svpa_check_error(_p(error_flag), _stream(stream))


def wait_selftest(limit_ns: int, error_flag, reached, stream=None, check=True) -> int:
    """svpa_wait_selftest: one kernel waits, bounded by limit_ns, on an
    mbarrier no thread arrives on (the wait-limit path of every kernel)."""
    st = load().svpa_wait_selftest(int(limit_ns), _p(error_flag), _p(reached), _stream(stream))
    if check:
        _check(st, "svpa_wait_selftest")
    return st

def status_string(status: int) -> str:
    return load().svpa_status_string(status).decode()


def version() -> int:
    return load().svpa_version()
