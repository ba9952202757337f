"""Seeded synthetic inputs for the paged speculative-verification step.

This module only draws and lays out inputs: random queries and K/V pages, a
shuffled physical block pool with per-sequence block tables, draft/target
distributions, draft tokens and uniforms.  It contains none of the method's
arithmetic (no attention, no acceptance test, no resampling, no commit); the
CUDA library and the CPU oracle both consume what it produces.

The five named workloads follow the problem sizes the verification step is
studied at: a tiny case, a 7B-shaped multi-head model, a 70B-shaped
grouped-query model, the same with FP8-E4M3 K/V pages carrying one fp32 scale
per (page, kv head), and a draft-tree verification over a shared system
prompt.  No public dataset is involved: every tensor is seeded noise with the
stated distribution.

Determinism: the CPU generator gives identical inputs on any host.  Large
workloads may be drawn on a CUDA device with a CUDA generator seeded the same
way (identical on a given GPU model, not across CPU/GPU); both consumers then
read the same buffers.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch

BLOCK_SIZE = 16
FP8_MAX = 448.0  # largest finite OCP E4M3 magnitude


def tree_parents(branching) -> list:
    """Parent array (BFS order, children contiguous) of a full draft tree.

    Node 0 is the root (the last committed token); ``branching[d]`` is the
    number of children of every node at depth d.
    """
    parent = [-1]
    level = [0]
    for br in branching:
        nxt = []
        for node in level:
            for _ in range(br):
                parent.append(node)
                nxt.append(len(parent) - 1)
        level = nxt
    return parent


def ancestor_masks(parent) -> list:
    """Bit i of entry j is set when node i is j itself or an ancestor of j."""
    masks = []
    for j in range(len(parent)):
        m, n = 0, j
        while n >= 0:
            m |= 1 << n
            n = parent[n]
        masks.append(m)
    return masks


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    gamma: int                      # draft tokens per sequence (linear)
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    ctx_lo: int                     # committed history, uniform in [lo, hi]
    ctx_hi: int
    vocab: int
    sigma_target: float             # target logits ~ N(0, sigma_target)
    sigma_draft: float              # draft logits = target logits + N(0, sigma_draft)
    kv_fp8: bool = False
    scale_tile: int = 0             # FP8 scales: 0 = one per (page, kv head); 64 = one per 64-element tile
    tree_branching: Optional[tuple] = None
    shared_prefix: int = 0          # tokens of a refcounted prefix shared by all sequences
    fixed_pool_blocks: Optional[int] = None
    spare_frac: float = 0.10
    fixed_contexts: Optional[tuple] = None

    @property
    def parent(self):
        return tree_parents(self.tree_branching) if self.tree_branching else None

    @property
    def n_q(self) -> int:
        return len(self.parent) if self.tree_branching else self.gamma + 1

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def max_blocks_per_seq(self) -> int:
        hi = self.shared_prefix + (max(self.fixed_contexts) if self.fixed_contexts else self.ctx_hi)
        return -(-(hi + self.n_q) // BLOCK_SIZE)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", batch=2, gamma=4, num_q_heads=4, num_kv_heads=4, head_dim=64,
                     ctx_lo=37, ctx_hi=100, fixed_contexts=(37, 100), vocab=1000,
                     sigma_target=2.0, sigma_draft=0.5, fixed_pool_blocks=16),
    "7b": Workload("7b", batch=32, gamma=4, num_q_heads=32, num_kv_heads=32, head_dim=128,
                   ctx_lo=512, ctx_hi=4096, vocab=32000, sigma_target=3.0, sigma_draft=0.7),
    "70b": Workload("70b", batch=64, gamma=5, num_q_heads=64, num_kv_heads=8, head_dim=128,
                    ctx_lo=8192, ctx_hi=32768, vocab=128256, sigma_target=3.0, sigma_draft=0.5),
    "fp8": Workload("fp8", batch=16, gamma=5, num_q_heads=64, num_kv_heads=8, head_dim=128,
                    ctx_lo=32768, ctx_hi=32768, vocab=128256, sigma_target=3.0, sigma_draft=0.5,
                    kv_fp8=True),
    # the FP8 workload with one scale per 64-element tile of a row
    "fp8_t64": Workload("fp8_t64", batch=16, gamma=5, num_q_heads=64, num_kv_heads=8, head_dim=128,
                        ctx_lo=32768, ctx_hi=32768, vocab=128256, sigma_target=3.0, sigma_draft=0.5,
                        kv_fp8=True, scale_tile=64),
    "tree": Workload("tree", batch=128, gamma=3, num_q_heads=32, num_kv_heads=8, head_dim=128,
                     ctx_lo=1024, ctx_hi=8192, vocab=32000, sigma_target=3.0, sigma_draft=0.7,
                     tree_branching=(4, 2, 2), shared_prefix=800),
}

SEEDS = {"tiny": 1000, "7b": 1001, "70b": 1002, "fp8": 1003, "tree": 1004, "fp8_t64": 1005}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


@dataclass
class AttnInputs:
    """Device-agnostic bundle of one paged-attention problem (torch tensors)."""
    wl: Workload
    q: torch.Tensor                 # bf16 [B, n_q, Hq, D]
    k_pool: torch.Tensor            # bf16 or float8_e4m3fn [num_blocks, Hkv, 16, D]
    v_pool: torch.Tensor
    k_scale: Optional[torch.Tensor]  # fp32 [num_blocks, Hkv] (FP8 only)
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor       # int32 [B, max_blocks] (-1 past the last page)
    context_lens: torch.Tensor      # int32 [B] committed history L_b
    ancestor_mask: Optional[torch.Tensor]  # int64 [n_q] (uint64 bit patterns) or None
    refcount: torch.Tensor          # int32 [num_blocks]
    free_stack: torch.Tensor        # int32 [num_blocks] (first free_top entries valid)
    free_top: int
    extra: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]

    def kv_bytes(self) -> int:
        """Bytes of K/V (and FP8 scales) the step must read: valid tokens only."""
        wl = self.wl
        T = (self.context_lens.to(torch.int64) + wl.n_q)
        if wl.shared_prefix:
            # the shared prefix pages are one physical copy
            tokens = int((T - wl.shared_prefix).sum().item()) + wl.shared_prefix
        else:
            tokens = int(T.sum().item())
        eb = 1 if wl.kv_fp8 else 2
        b = tokens * wl.num_kv_heads * wl.head_dim * 2 * eb
        if wl.kv_fp8:
            pages = int(((T + BLOCK_SIZE - 1) // BLOCK_SIZE).sum().item())
            per_page = BLOCK_SIZE * (wl.head_dim // 64) if wl.scale_tile == 64 else 1
            b += pages * wl.num_kv_heads * per_page * 2 * 4
        return b


def make_attention(wl: Workload, seed: int, device="cpu", poison: bool = True,
                   batch: Optional[int] = None, contexts=None) -> AttnInputs:
    """Draw one paged-attention problem.

    contexts: optional explicit committed lengths (private part, before any
    shared prefix).  poison: fill K/V slots that no sequence owns (unused pool
    blocks and the slots past each sequence's last token) with NaN so that a
    kernel that reads them is caught.
    """
    B = batch if batch is not None else wl.batch
    g_cpu = _gen(seed, "cpu")
    n_q, BS = wl.n_q, BLOCK_SIZE
    if contexts is not None:
        priv = torch.as_tensor(contexts, dtype=torch.int64)
        B = priv.shape[0]
    elif wl.fixed_contexts is not None:
        priv = torch.tensor(wl.fixed_contexts, dtype=torch.int64)[:B]
    else:
        priv = torch.randint(wl.ctx_lo, wl.ctx_hi + 1, (B,), generator=g_cpu, dtype=torch.int64)
    L = priv + wl.shared_prefix
    T = L + n_q
    pages = (T + BS - 1) // BS
    max_blocks = max(wl.max_blocks_per_seq(), int(pages.max().item()))
    shared_pages = wl.shared_prefix // BS        # only whole pages are shared
    need = int((pages - shared_pages).sum().item()) + shared_pages
    if wl.fixed_pool_blocks is not None:
        num_blocks = max(wl.fixed_pool_blocks, need)
    else:
        num_blocks = int(math.ceil(need * (1.0 + wl.spare_frac)))
    perm = torch.randperm(num_blocks, generator=g_cpu).to(torch.int32)
    bt = torch.full((B, max_blocks), -1, dtype=torch.int32)
    refcount = torch.zeros(num_blocks, dtype=torch.int32)
    cursor = 0
    shared_ids = perm[cursor:cursor + shared_pages]
    cursor += shared_pages
    for b in range(B):
        bt[b, :shared_pages] = shared_ids
        own = int(pages[b].item()) - shared_pages
        bt[b, shared_pages:shared_pages + own] = perm[cursor:cursor + own]
        cursor += own
    used = bt[bt >= 0].to(torch.int64)
    refcount.index_add_(0, used, torch.ones_like(used, dtype=torch.int32))
    free = perm[cursor:].clone()
    free_stack = torch.full((num_blocks,), -1, dtype=torch.int32)
    free_stack[:free.shape[0]] = free

    Hq, Hkv, D = wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    dev = torch.device(device)
    g_dev = _gen(seed + 7919, dev)
    q = torch.randn((B, n_q, Hq, D), generator=g_dev, device=dev, dtype=torch.float32).to(torch.bfloat16)

    # which pool slots hold a token of some sequence
    valid = torch.zeros((num_blocks, BS), dtype=torch.bool)
    for b in range(B):
        t = int(T[b].item())
        for i in range(int(pages[b].item())):
            n = min(BS, t - i * BS)
            valid[int(bt[b, i].item()), :n] = True
    valid_d = valid.to(dev)

    kf = torch.randn((num_blocks, Hkv, BS, D), generator=g_dev, device=dev, dtype=torch.float32)
    vf = torch.randn((num_blocks, Hkv, BS, D), generator=g_dev, device=dev, dtype=torch.float32)
    k_scale = v_scale = None
    if wl.kv_fp8:
        mask = valid_d[:, None, :, None]
        kf = torch.where(mask, kf, torch.zeros((), device=dev))
        vf = torch.where(mask, vf, torch.zeros((), device=dev))

        def quantise(x):
            if wl.scale_tile == 64:
                # one scale per 64 consecutive elements of a token's row
                xt = x.unflatten(3, (Hd // 64, 64))
                amax = xt.abs().amax(dim=4)
                scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
                y = (xt / scale[..., None]).clamp(-FP8_MAX, FP8_MAX).flatten(3)
                return y.to(torch.float8_e4m3fn), scale.to(torch.float32).contiguous()
            amax = x.abs().amax(dim=(2, 3))
            scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
            y = (x / scale[:, :, None, None]).clamp(-FP8_MAX, FP8_MAX)
            return y.to(torch.float8_e4m3fn), scale.to(torch.float32).contiguous()

        Hd = D
        k_pool, k_scale = quantise(kf)
        v_pool, v_scale = quantise(vf)
        del kf, vf
        if poison:
            nan8 = torch.tensor(0x7F, dtype=torch.uint8, device=dev)
            kb = k_pool.view(torch.uint8)
            vb = v_pool.view(torch.uint8)
            kb.copy_(torch.where(mask, kb, nan8))
            vb.copy_(torch.where(mask, vb, nan8))
    else:
        k_pool = kf.to(torch.bfloat16)
        v_pool = vf.to(torch.bfloat16)
        del kf, vf
        if poison:
            mask = valid_d[:, None, :, None]
            nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=dev)
            k_pool = torch.where(mask, k_pool, nan)
            v_pool = torch.where(mask, v_pool, nan)

    am = None
    if wl.tree_branching:
        m = ancestor_masks(wl.parent)
        am = torch.tensor([x - (1 << 64) if x >= (1 << 63) else x for x in m], dtype=torch.int64)

    return AttnInputs(wl=wl, q=q, k_pool=k_pool.contiguous(), v_pool=v_pool.contiguous(),
                      k_scale=k_scale, v_scale=v_scale,
                      block_table=bt.to(dev), context_lens=L.to(torch.int32).to(dev),
                      ancestor_mask=None if am is None else am.to(dev),
                      refcount=refcount.to(dev), free_stack=free_stack.to(dev),
                      free_top=int(free.shape[0]))


@dataclass
class SamplerInputs:
    p: torch.Tensor          # fp32 [B, gamma+1, V]  (tree: [B, n_nodes, V])
    q: torch.Tensor          # fp32 [B, gamma, V]    (tree: [B, n_internal, V])
    tokens: torch.Tensor     # int32 [B, gamma]      (tree: [B, n_nodes], entry 0 unused)
    u_accept: torch.Tensor   # fp32 [B, gamma]       (tree: [B, n_nodes])
    u_sample: torch.Tensor   # fp32 [B]
    parent: Optional[torch.Tensor] = None  # int32 [n_nodes] (tree only)


def make_sampler(wl: Workload, seed: int, device="cpu", batch: Optional[int] = None,
                 vocab: Optional[int] = None) -> SamplerInputs:
    """Target P = softmax(N(0, s_t) logits); draft Q = softmax(target logits +
    N(0, s_d) noise); draft tokens drawn from Q; uniforms U[0, 1).

    Linear: gamma draft positions, P has one more row (the bonus position).
    Tree: P at every node, Q at every internal node, each node's children
    drawn independently from its parent's Q row.
    """
    B = batch if batch is not None else wl.batch
    V = vocab if vocab is not None else wl.vocab
    dev = torch.device(device)
    g = _gen(seed + 104729, dev)
    if wl.tree_branching:
        parent = wl.parent
        n = len(parent)
        internal = [i for i in range(n) if i in set(parent[1:])]
        row_of = {node: r for r, node in enumerate(internal)}
        logits = torch.randn((B, n, V), generator=g, device=dev) * wl.sigma_target
        p = torch.softmax(logits, dim=-1)
        dl = logits[:, internal, :] + torch.randn((B, len(internal), V), generator=g, device=dev) * wl.sigma_draft
        q = torch.softmax(dl, dim=-1)
        del logits, dl
        tokens = torch.zeros((B, n), dtype=torch.int32, device=dev)
        for c in range(1, n):
            tokens[:, c] = torch.multinomial(q[:, row_of[parent[c]], :], 1, generator=g).squeeze(1).to(torch.int32)
        ua = torch.rand((B, n), generator=g, device=dev)
        us = torch.rand((B,), generator=g, device=dev)
        return SamplerInputs(p=p.contiguous(), q=q.contiguous(), tokens=tokens, u_accept=ua,
                             u_sample=us, parent=torch.tensor(parent, dtype=torch.int32, device=dev))
    gm = wl.gamma
    logits = torch.randn((B, gm + 1, V), generator=g, device=dev) * wl.sigma_target
    p = torch.softmax(logits, dim=-1)
    dl = logits[:, :gm, :] + torch.randn((B, gm, V), generator=g, device=dev) * wl.sigma_draft
    q = torch.softmax(dl, dim=-1)
    del logits, dl
    x = torch.multinomial(q.reshape(B * gm, V), 1, generator=g).reshape(B, gm).to(torch.int32)
    ua = torch.rand((B, gm), generator=g, device=dev)
    us = torch.rand((B,), generator=g, device=dev)
    return SamplerInputs(p=p.contiguous(), q=q.contiguous(), tokens=x, u_accept=ua, u_sample=us)


@dataclass
class LogitInputs:
    lp: torch.Tensor         # fp32 [B, gamma+1, V] target logits
    lq: torch.Tensor         # fp32 [B, gamma, V]   draft logits
    tokens: torch.Tensor     # int32 [B, gamma] drawn from softmax(lq / draft_temperature)
    u_accept: torch.Tensor   # fp32 [B, gamma]
    u_sample: torch.Tensor   # fp32 [B]
    temperature: float
    draft_temperature: float


def make_logits(wl: Workload, seed: int, device="cpu", batch: Optional[int] = None, vocab: Optional[int] = None,
                gamma: Optional[int] = None, temperature: float = 1.0,
                draft_temperature: Optional[float] = None) -> LogitInputs:
    """Logits for the sampler's front-end: target N(0, s_t), draft = target +
    N(0, s_d) (the recipe of make_sampler, before the softmax); draft tokens
    drawn from softmax(draft / draft_temperature); uniforms U[0, 1)."""
    B = batch if batch is not None else wl.batch
    V = vocab if vocab is not None else wl.vocab
    gm = gamma if gamma is not None else wl.gamma
    td = temperature if draft_temperature is None else draft_temperature
    dev = torch.device(device)
    g = _gen(seed + 130363, dev)
    lp = torch.randn((B, gm + 1, V), generator=g, device=dev) * wl.sigma_target
    lq = lp[:, :gm, :] + torch.randn((B, gm, V), generator=g, device=dev) * wl.sigma_draft
    q = torch.softmax(lq.reshape(B * gm, V).double() / td, dim=-1)
    x = torch.multinomial(q, 1, generator=g).reshape(B, gm).to(torch.int32)
    del q
    ua = torch.rand((B, gm), generator=g, device=dev)
    us = torch.rand((B,), generator=g, device=dev)
    return LogitInputs(lp=lp.contiguous(), lq=lq.contiguous(), tokens=x, u_accept=ua, u_sample=us,
                       temperature=float(temperature), draft_temperature=float(td))


@dataclass
class TreeLogitInputs:
    lp: torch.Tensor         # fp32 [B, n_nodes, V] target logits at every node
    lq: torch.Tensor         # fp32 [B, n_internal, V] draft logits of each internal node's children
    tokens: torch.Tensor     # int32 [B, n_nodes] (entry 0 unused), drawn from the parent's draft softmax
    u_accept: torch.Tensor   # fp32 [B, n_nodes]
    u_sample: torch.Tensor   # fp32 [B]
    parent: torch.Tensor     # int32 [n_nodes]
    temperature: float
    draft_temperature: float


def make_tree_logits(wl: Workload, seed: int, device="cpu", batch: Optional[int] = None,
                     vocab: Optional[int] = None, branching: Optional[tuple] = None, temperature: float = 1.0,
                     draft_temperature: Optional[float] = None) -> TreeLogitInputs:
    """Logits for the draft-tree sampler's front-end (the recipe of
    make_sampler's tree, before the softmax): target N(0, s_t) at every node,
    draft = the node's target logits + N(0, s_d) at every internal node; each
    child's token drawn independently from softmax(parent's draft /
    draft_temperature); uniforms U[0, 1)."""
    B = batch if batch is not None else wl.batch
    V = vocab if vocab is not None else wl.vocab
    br = branching if branching is not None else wl.tree_branching
    parent = tree_parents(br)
    td = temperature if draft_temperature is None else draft_temperature
    dev = torch.device(device)
    g = _gen(seed + 151051, dev)
    n = len(parent)
    internal = [i for i in range(n) if i in set(parent[1:])]
    row_of = {node: r for r, node in enumerate(internal)}
    lp = torch.randn((B, n, V), generator=g, device=dev) * wl.sigma_target
    lq = lp[:, internal, :] + torch.randn((B, len(internal), V), generator=g, device=dev) * wl.sigma_draft
    tokens = torch.zeros((B, n), dtype=torch.int32, device=dev)
    for r, node in enumerate(internal):
        q = torch.softmax(lq[:, r, :].double() / td, dim=-1)
        kids = [c for c in range(1, n) if parent[c] == node]
        draws = torch.multinomial(q, len(kids), replacement=True, generator=g).to(torch.int32)
        for i, c in enumerate(kids):
            tokens[:, c] = draws[:, i]
        del q
    ua = torch.rand((B, n), generator=g, device=dev)
    us = torch.rand((B,), generator=g, device=dev)
    return TreeLogitInputs(lp=lp.contiguous(), lq=lq.contiguous(), tokens=tokens, u_accept=ua, u_sample=us,
                           parent=torch.tensor(parent, dtype=torch.int32, device=dev),
                           temperature=float(temperature), draft_temperature=float(td))


@dataclass
class AppendInputs:
    """The paged cache before an append and the rows to append (torch tensors)."""
    wl: Workload
    new_k: torch.Tensor             # bf16 [B, n_new, Hkv, D]
    new_v: torch.Tensor
    k_pool: torch.Tensor            # bf16 or float8_e4m3fn [num_blocks, Hkv, 16, D]
    v_pool: torch.Tensor
    k_scale: Optional[torch.Tensor]  # fp32 [num_blocks, Hkv] (FP8 only)
    v_scale: Optional[torch.Tensor]
    block_table: torch.Tensor       # int32 [B, max_blocks]; pages cover [0, L_b) only
    context_lens: torch.Tensor      # int32 [B]
    refcount: torch.Tensor          # int32 [num_blocks]
    free_stack: torch.Tensor        # int32 [num_blocks]
    free_top: int

    @property
    def n_new(self) -> int:
        return self.new_k.shape[1]

    def write_bytes(self) -> int:
        """Bytes the append must move at least: the new rows read once and
        written once (bf16), or, for FP8, each touched (page, head) tile read
        and written once plus the new rows read once (with 64-element tile
        scales: the new rows read, their codes and scales written)."""
        wl = self.wl
        B, n, Hkv, D = self.new_k.shape
        rows = B * n * Hkv * D * 2 * 2          # K and V, bf16
        if not wl.kv_fp8:
            return 2 * rows
        if wl.scale_tile == 64:                  # codes and tile scales of the new rows only
            return rows + rows // 2 + B * n * Hkv * (D // 64) * 4 * 2
        L = self.context_lens.to(torch.int64).cpu()
        first, last = L // BLOCK_SIZE, (L + n - 1) // BLOCK_SIZE
        tiles = int((last - first + 1).sum().item()) * Hkv * 2
        return rows + tiles * BLOCK_SIZE * D * 2 + tiles * 8


def make_append(wl: Workload, seed: int, device="cpu", batch: Optional[int] = None,
                n_new: Optional[int] = None, shared_prefix: Optional[int] = None,
                contexts=None, row_factors=(0.5, 1.0, 3.0)) -> AppendInputs:
    """Draw the cache state before an append of n_new rows (default n_q).

    The whole pages of the first shared_prefix tokens (default: the
    workload's) are mapped by every sequence, one reference each.  When the
    prefix ends inside a page, the sequences whose history ends on that page
    share it (so their append lands on a shared page and copy-on-write runs);
    the others hold a private copy of it.  Pages cover [0, L_b) only and every
    other block is on the free stack (shuffled); the pool holds enough blocks
    for every sequence to own all its pages after the append, plus 10%.
    New rows are N(0, 1) times a per-row factor drawn from `row_factors`
    (default {0.5, 1, 3}, so that FP8 page scales grow on some writes and not
    on others; (1,) gives plain N(0, 1) rows, as in the task's workloads).  Pool slots that hold
    no token are NaN (bf16) or the code of +448 (FP8): a kernel that took a
    page maximum over them would change the page's scale.
    """
    B = batch if batch is not None else wl.batch
    n_new = wl.n_q if n_new is None else n_new
    prefix = wl.shared_prefix if shared_prefix is None else shared_prefix
    g_cpu = _gen(seed, "cpu")
    BS = BLOCK_SIZE
    if contexts is not None:
        priv = torch.as_tensor(contexts, dtype=torch.int64)
        B = priv.shape[0]
    elif wl.fixed_contexts is not None:
        priv = torch.tensor(wl.fixed_contexts, dtype=torch.int64)[:B]
    else:
        priv = torch.randint(wl.ctx_lo, wl.ctx_hi + 1, (B,), generator=g_cpu, dtype=torch.int64)
    L = priv + prefix
    pages = (L + BS - 1) // BS
    after = (L + n_new + BS - 1) // BS
    max_blocks = int(after.max().item())
    full = prefix // BS                              # whole pages of the prefix
    # the prefix's partly filled page is shared by the sequences whose history
    # ends on it; a longer history holds its own copy of that page (the state
    # an earlier copy-on-write leaves)
    on_partial = (prefix % BS != 0) & (L <= (full + 1) * BS)
    num_blocks = int(math.ceil(int(after.sum().item()) * 1.10)) + 1
    perm = torch.randperm(num_blocks, generator=g_cpu).to(torch.int32)
    bt = torch.full((B, max_blocks), -1, dtype=torch.int32)
    bt[:, :full] = perm[:full]
    cursor = full
    if bool(on_partial.any()):
        bt[on_partial, full] = perm[cursor]
        cursor += 1
    for b in range(B):
        start = full + int(on_partial[b].item())
        own = int(pages[b].item()) - start
        bt[b, start:start + own] = perm[cursor:cursor + own]
        cursor += own
    refcount = torch.zeros(num_blocks, dtype=torch.int32)
    used = bt[bt >= 0].to(torch.int64)
    refcount.index_add_(0, used, torch.ones_like(used, dtype=torch.int32))
    free = perm[cursor:].clone()
    free_stack = torch.full((num_blocks,), -1, dtype=torch.int32)
    free_stack[:free.shape[0]] = free

    Hkv, D = wl.num_kv_heads, wl.head_dim
    dev = torch.device(device)
    g_dev = _gen(seed + 7919, dev)
    valid = torch.zeros((num_blocks, BS), dtype=torch.bool)
    for b in range(B):
        t = int(L[b].item())
        for i in range(int(pages[b].item())):
            valid[int(bt[b, i].item()), :min(BS, t - i * BS)] = True
    mask = valid.to(dev)[:, None, :, None]
    kf = torch.randn((num_blocks, Hkv, BS, D), generator=g_dev, device=dev, dtype=torch.float32)
    vf = torch.randn((num_blocks, Hkv, BS, D), generator=g_dev, device=dev, dtype=torch.float32)
    k_scale = v_scale = None
    if wl.kv_fp8:
        def quantise(x):
            x = torch.where(mask, x, torch.zeros((), device=dev))
            if wl.scale_tile == 64:
                xt = x.unflatten(3, (D // 64, 64))
                amax = xt.abs().amax(dim=4)
                scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
                y = (xt / scale[..., None]).clamp(-FP8_MAX, FP8_MAX).flatten(3).to(torch.float8_e4m3fn)
                yb = torch.where(mask, y.view(torch.uint8), torch.tensor(0x7E, dtype=torch.uint8, device=dev))
                return yb.view(torch.float8_e4m3fn).contiguous(), scale.to(torch.float32).contiguous()
            amax = x.abs().amax(dim=(2, 3))
            scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
            y = (x / scale[:, :, None, None]).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
            yb = torch.where(mask, y.view(torch.uint8), torch.tensor(0x7E, dtype=torch.uint8, device=dev))
            return yb.view(torch.float8_e4m3fn).contiguous(), scale.to(torch.float32).contiguous()

        k_pool, k_scale = quantise(kf)
        v_pool, v_scale = quantise(vf)
    else:
        nan = torch.tensor(float("nan"), device=dev)
        k_pool = torch.where(mask, kf, nan).to(torch.bfloat16).contiguous()
        v_pool = torch.where(mask, vf, nan).to(torch.bfloat16).contiguous()
    del kf, vf
    factor = torch.tensor(list(row_factors), dtype=torch.float32, device=dev)[
        torch.randint(0, len(row_factors), (B, n_new, 1, 1), generator=g_dev, device=dev)]
    new_k = (torch.randn((B, n_new, Hkv, D), generator=g_dev, device=dev) * factor).to(torch.bfloat16)
    new_v = (torch.randn((B, n_new, Hkv, D), generator=g_dev, device=dev) * factor).to(torch.bfloat16)
    return AppendInputs(wl=wl, new_k=new_k, new_v=new_v, k_pool=k_pool, v_pool=v_pool,
                        k_scale=k_scale, v_scale=v_scale, block_table=bt.to(dev),
                        context_lens=L.to(torch.int32).to(dev), refcount=refcount.to(dev),
                        free_stack=free_stack.to(dev), free_top=int(free.shape[0]))
