"""Seeded synthetic inputs for the tree-attention decode step.

This module only *generates inputs*: token trees (parent / node_len /
query_node arrays), a paged KV layout addressed by tree node, and seeded
Q / K / V tensors.  It holds none of the method's arithmetic (no ancestor
walks, no masks, no softmax), so both the fp64 oracle and the CUDA path may
consume what it produces.

The workloads follow the shapes of the DeFT pages (arXiv 2404.00242 abstract:
few-shot prompting, multi-step reasoning and speculative decoding trees;
the aifetchly "DeFT Guide", section "The Tree-Attention Bottleneck", for the
prefix + candidate-tree picture).  No dataset or model weights are used: the
trees and tensors below are synthetic stand-ins with those shapes.

Conventions (shared with the library's C-ABI):
  parent[n]      int32, -1 for a root (forests allowed)
  node_len[n]    int32 >= 0 tokens held by node n
  query_node[q]  int32 node at which query q sits
  KV pages       bf16 [num_pages][num_kv_heads][page_size][head_dim]
  node_page_off  int32 [num_nodes + 1]; node n owns page_id[off[n]:off[n+1]]
  page_id        int32 physical page index for each logical page
Token t of node n lives in page page_id[node_page_off[n] + t // P], slot t % P.
Every node starts on a fresh page.
"""
from __future__ import annotations

import math
import random
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

PAGE_SIZE = 16


@dataclass
class TreeSpec:
    """A token tree plus the head geometry of one attention layer."""
    name: str
    parent: np.ndarray          # int32 [N]
    node_len: np.ndarray        # int32 [N]
    query_node: np.ndarray      # int32 [Q]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    k_scale: float = 1.0        # K ~ N(0,1) * k_scale before the bf16 cast
    shuffle_pages: bool = False
    seed: int = 0
    notes: dict = field(default_factory=dict)
    # Per query, the token of its node it sits at (tree verification with
    # multi-token nodes: it attends tokens 0..p of its own node); None: every
    # query sits at its node's last token.
    query_pos: Optional[np.ndarray] = None

    @property
    def num_nodes(self) -> int:
        return int(self.parent.shape[0])

    @property
    def num_queries(self) -> int:
        return int(self.query_node.shape[0])

    @property
    def gqa_group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _arr(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


# ---------------------------------------------------------------------------
# The five workload shapes
# ---------------------------------------------------------------------------

def tiny_tree() -> TreeSpec:
    """Root prefix of 128 tokens, 2 children of 16 tokens, each with 2 leaves
    of 8 tokens; one query per leaf; 4 heads MHA, head_dim 64."""
    parent = [-1, 0, 0, 1, 1, 2, 2]
    node_len = [128, 16, 16, 8, 8, 8, 8]
    return TreeSpec("tiny_tree_7n_4q_h4_d64", _arr(parent), _arr(node_len),
                    _arr([3, 4, 5, 6]), 4, 4, 64, seed=1001)


def few_shot_tree(prefix: int = 4096, branches: int = 32, branch_len: int = 256,
                  heads: int = 32, head_dim: int = 128) -> TreeSpec:
    """Shared-prefix few-shot decode: one prefix node, `branches` children of
    `branch_len` tokens, one query at every branch tip.  K is scaled by
    1/sqrt(head_dim) before the bf16 cast."""
    parent = [-1] + [0] * branches
    node_len = [prefix] + [branch_len] * branches
    query = list(range(1, branches + 1))
    return TreeSpec(f"few_shot_{prefix}p_{branches}x{branch_len}_h{heads}_d{head_dim}",
                    _arr(parent), _arr(node_len), _arr(query), heads, heads,
                    head_dim, k_scale=1.0 / math.sqrt(head_dim), seed=1002)


def _grow_token_tree(rng: random.Random, target: int, max_depth: int,
                     branch_lo: int, branch_hi: int) -> Optional[List[int]]:
    """Breadth-first growth of a `target`-node tree of 1-token nodes.

    Returns parent indices local to the tree (-1 for the first node, which
    sits at depth 1 under the prefix) or None when the frontier empties
    before `target` nodes exist."""
    parents = [-1]
    depth = [1]
    frontier = [0]
    head = 0
    while len(parents) < target and head < len(frontier):
        node = frontier[head]
        head += 1
        if depth[node] >= max_depth:
            continue
        for _ in range(rng.randint(branch_lo, branch_hi)):
            if len(parents) >= target:
                break
            parents.append(node)
            depth.append(depth[node] + 1)
            frontier.append(len(parents) - 1)
    if len(parents) < target:
        return None
    return parents


def speculative_forest(requests: int = 8, prefix: int = 4000, tree_nodes: int = 64,
                       max_depth: int = 6, heads: int = 32, head_dim: int = 128,
                       seed: int = 3) -> TreeSpec:
    """Speculative-verification token trees: a forest of `requests` trees, each
    a `prefix`-token root followed by a `tree_nodes`-node tree of 1-token
    nodes grown breadth-first with branching U{1..4} and depth <= max_depth.
    Every 1-token tree node carries a query."""
    parent: List[int] = []
    node_len: List[int] = []
    query: List[int] = []
    resampled = []
    for r in range(requests):
        sub = 0
        while True:
            rng = random.Random(seed * 1000003 + r * 7919 + sub)
            local = _grow_token_tree(rng, tree_nodes, max_depth, 1, 4)
            if local is not None:
                break
            sub += 1
        resampled.append(sub)
        root = len(parent)
        parent.append(-1)
        node_len.append(prefix)
        base = len(parent)
        for p in local:
            parent.append(root if p < 0 else base + p)
            node_len.append(1)
        query.extend(range(base, base + tree_nodes))
    return TreeSpec(f"speculative_{requests}x({prefix}p+{tree_nodes}n)_h{heads}_d{head_dim}",
                    _arr(parent), _arr(node_len), _arr(query), heads, heads,
                    head_dim, seed=1003, notes={"resampled_subseeds": resampled})


def multitoken_speculative_forest(requests: int = 8, prefix: int = 4000, tree_nodes: int = 16,
                                  node_tokens: int = 4, max_depth: int = 6, heads: int = 32,
                                  head_dim: int = 128, seed: int = 7) -> TreeSpec:
    """Tree verification with multi-token nodes: like speculative_forest, but
    each tree node holds `node_tokens` candidate tokens and every token is a
    query that sits at its position (attending the prefix, its ancestors and
    its own node up to itself)."""
    parent: List[int] = []
    node_len: List[int] = []
    query: List[int] = []
    pos: List[int] = []
    for r in range(requests):
        sub = 0
        while True:
            rng = random.Random(seed * 1000003 + r * 7919 + sub)
            local = _grow_token_tree(rng, tree_nodes, max_depth, 1, 4)
            if local is not None:
                break
            sub += 1
        root = len(parent)
        parent.append(-1)
        node_len.append(prefix)
        base = len(parent)
        for p in local:
            parent.append(root if p < 0 else base + p)
            node_len.append(node_tokens)
        for n in range(base, base + tree_nodes):
            query.extend([n] * node_tokens)
            pos.extend(range(node_tokens))
    spec = TreeSpec(f"verify_{requests}x({prefix}p+{tree_nodes}n x{node_tokens}t)_h{heads}_d{head_dim}",
                    _arr(parent), _arr(node_len), _arr(query), heads, heads, head_dim, seed=1007)
    spec.query_pos = _arr(pos)
    return spec


def reasoning_tree(levels: int = 4, branch_lo: int = 3, branch_hi: int = 5,
                   len_lo: int = 100, len_hi: int = 600, num_queries: int = 128,
                   q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128,
                   seed: int = 4) -> TreeSpec:
    """Multi-step reasoning tree: `levels` levels (root + levels-1), every
    internal node has U{branch_lo..branch_hi} children, every node holds
    U{len_lo..len_hi} tokens.  `num_queries` queries are dealt round-robin to
    the leaves.  KV pages are placed in a seeded random page order."""
    rng = random.Random(seed)
    parent = [-1]
    node_len = [rng.randint(len_lo, len_hi)]
    level = [0]
    for _ in range(levels - 1):
        nxt = []
        for n in level:
            for _ in range(rng.randint(branch_lo, branch_hi)):
                parent.append(n)
                node_len.append(rng.randint(len_lo, len_hi))
                nxt.append(len(parent) - 1)
        level = nxt
    leaves = level
    query = [leaves[i % len(leaves)] for i in range(num_queries)]
    return TreeSpec(f"reasoning_{levels}lv_b{branch_lo}-{branch_hi}_len{len_lo}-{len_hi}"
                    f"_{num_queries}q_gqa{q_heads}/{kv_heads}_d{head_dim}",
                    _arr(parent), _arr(node_len), _arr(query), q_heads, kv_heads,
                    head_dim, shuffle_pages=True, seed=1004)


def imbalance_tree(prefix: int = 32768, leaves: int = 256, lo: int = 64, hi: int = 8192,
                   q_heads: int = 32, kv_heads: int = 8, head_dim: int = 128,
                   control: bool = False, control_len: int = 2048, seed: int = 5) -> TreeSpec:
    """Imbalance stress: a `prefix`-token root and `leaves` leaves whose lengths
    are round(exp(U[ln lo, ln hi])), one query per leaf.  The control variant
    has an empty root and `leaves` independent `control_len`-token leaves."""
    rng = random.Random(seed)
    parent = [-1] + [0] * leaves
    if control:
        node_len = [0] + [control_len] * leaves
        name = f"imbalance_control_{leaves}x{control_len}_gqa{q_heads}/{kv_heads}_d{head_dim}"
    else:
        lens = [int(round(math.exp(rng.uniform(math.log(lo), math.log(hi)))))
                for _ in range(leaves)]
        node_len = [prefix] + lens
        name = f"imbalance_{prefix}p+{leaves}leaves_{lo}-{hi}_gqa{q_heads}/{kv_heads}_d{head_dim}"
    query = list(range(1, leaves + 1))
    return TreeSpec(name, _arr(parent), _arr(node_len), _arr(query), q_heads, kv_heads,
                    head_dim, seed=1005 + (1 if control else 0))


def config(i: int) -> TreeSpec:
    """The benchmark workloads by number: 1 tiny tree, 2 few-shot prefix,
    3 speculative-decoding forest, 4 multi-step reasoning tree, 5 length
    imbalance under a long prefix, 6 the no-sharing control of 5, 7 tree
    verification with multi-token nodes (every token a query)."""
    return {1: tiny_tree, 2: few_shot_tree, 3: speculative_forest,
            4: reasoning_tree, 5: imbalance_tree,
            6: lambda: imbalance_tree(control=True),
            7: multitoken_speculative_forest}[i]()


# ---------------------------------------------------------------------------
# Small trees for tests
# ---------------------------------------------------------------------------

def random_tree(seed: int, max_nodes: int = 12, max_len: int = 40, max_queries: int = 10,
                q_heads: int = 4, kv_heads: int = 2, head_dim: int = 64,
                forest: bool = True, zero_len_prob: float = 0.15) -> TreeSpec:
    """A small random forest: random parents (always a lower id, so no cycles),
    random lengths including zero-length nodes, queries anywhere (internal
    nodes and repeated nodes included)."""
    rng = random.Random(seed)
    n = rng.randint(1, max_nodes)
    parent = []
    for i in range(n):
        if i == 0 or (forest and rng.random() < 0.1):
            parent.append(-1)
        else:
            parent.append(rng.randrange(i))
    node_len = [0 if rng.random() < zero_len_prob else rng.randint(1, max_len)
                for _ in range(n)]
    nq = rng.randint(1, max_queries)
    query = [rng.randrange(n) for _ in range(nq)]
    return TreeSpec(f"random_{seed}", _arr(parent), _arr(node_len), _arr(query),
                    q_heads, kv_heads, head_dim, shuffle_pages=bool(seed % 2),
                    seed=20000 + seed)


def chain_tree(lengths: List[int], q_heads: int = 2, kv_heads: int = 1,
               head_dim: int = 64) -> TreeSpec:
    """A single branch: node i is the child of node i-1; one query per node."""
    n = len(lengths)
    parent = [-1] + list(range(n - 1))
    return TreeSpec(f"chain_{n}", _arr(parent), _arr(lengths), _arr(list(range(n))),
                    q_heads, kv_heads, head_dim, seed=31337)


def causal_node_tree(length: int, q_heads: int = 2, kv_heads: int = 1, head_dim: int = 64,
                     parent_len: int = 0) -> TreeSpec:
    """Prefill of one node: a `length`-token node (under an optional
    `parent_len`-token root) with a query at every one of its positions, so
    that query i attends the root and tokens 0..i: causal self-attention."""
    if parent_len:
        parent, node_len, node = [-1, 0], [parent_len, length], 1
    else:
        parent, node_len, node = [-1], [length], 0
    spec = TreeSpec(f"causal_node_{parent_len}+{length}", _arr(parent), _arr(node_len),
                    _arr([node] * length), q_heads, kv_heads, head_dim, seed=3000 + length)
    spec.query_pos = _arr(list(range(length)))
    return spec


def positions_tree(seed: int, max_nodes: int = 12, max_len: int = 40, max_queries: int = 16,
                   q_heads: int = 2, kv_heads: int = 1, head_dim: int = 64) -> TreeSpec:
    """A random tree whose queries sit at random token positions of their
    nodes (-1 for some: the node's last token), several per node."""
    spec = random_tree(seed, max_nodes=max_nodes, max_len=max_len, max_queries=max_queries,
                       q_heads=q_heads, kv_heads=kv_heads, head_dim=head_dim, zero_len_prob=0.0)
    rng = random.Random(7000 + seed)
    pos = []
    for n in spec.query_node:
        L = int(spec.node_len[n])
        pos.append(-1 if L == 0 or rng.random() < 0.25 else rng.randrange(L))
    spec.query_pos = _arr(pos)
    spec.name = f"positions_{seed}"
    return spec


def heap_example_tree(prefix: int = 1024, tree_nodes: int = 16, head_dim: int = 64) -> TreeSpec:
    """The simulator example of the aifetchly "DeFT Guide" (section "End-to-End
    Implementation"): a 1024-token prefix and 16 one-token candidate nodes in
    a heap shape (node i's parent is (i-1)//2), one query per candidate node.
    Node 0 here is the prefix; candidate i is node i+1."""
    parent = [-1, 0] + [1 + (i - 1) // 2 for i in range(1, tree_nodes)]
    node_len = [prefix] + [1] * tree_nodes
    query = list(range(1, tree_nodes + 1))
    return TreeSpec("heap_example", _arr(parent), _arr(node_len), _arr(query),
                    1, 1, head_dim, seed=42)


def relabel(spec: TreeSpec, perm: np.ndarray) -> TreeSpec:
    """Renumber nodes: old node n becomes perm[n].  Queries keep their order."""
    perm = np.asarray(perm, dtype=np.int64)
    n = spec.num_nodes
    parent = np.full(n, -1, dtype=np.int32)
    node_len = np.zeros(n, dtype=np.int32)
    for old in range(n):
        p = spec.parent[old]
        parent[perm[old]] = -1 if p < 0 else perm[p]
        node_len[perm[old]] = spec.node_len[old]
    query = perm[spec.query_node].astype(np.int32)
    out = TreeSpec(spec.name + "_relabelled", parent, node_len, query, spec.num_q_heads,
                   spec.num_kv_heads, spec.head_dim, spec.k_scale, spec.shuffle_pages,
                   spec.seed)
    out.query_pos = None if spec.query_pos is None else spec.query_pos.copy()
    return out


# ---------------------------------------------------------------------------
# Paged layout and tensors
# ---------------------------------------------------------------------------

@dataclass
class PagedLayout:
    node_page_off: np.ndarray   # int32 [N+1]
    page_id: np.ndarray         # int32 [num_logical_pages]
    num_pages: int              # physical pages allocated
    page_size: int


def paged_layout(spec: TreeSpec, page_size: int = PAGE_SIZE, spare_pages: int = 0,
                 shuffle: Optional[bool] = None) -> PagedLayout:
    """Give every node ceil(len/P) pages (a fresh page per node).  Physical
    page numbers are sequential, or a seeded permutation when the spec (or
    `shuffle`) asks for a shuffled page order.  `spare_pages` extra physical
    pages are allocated and left unreferenced."""
    counts = (spec.node_len.astype(np.int64) + page_size - 1) // page_size
    off = np.zeros(spec.num_nodes + 1, dtype=np.int64)
    off[1:] = np.cumsum(counts)
    logical = int(off[-1])
    num_pages = logical + spare_pages
    shuffle = spec.shuffle_pages if shuffle is None else shuffle
    if shuffle:
        rng = np.random.default_rng(spec.seed + 77)
        page_id = rng.permutation(num_pages)[:logical]
    else:
        page_id = np.arange(logical)
    return PagedLayout(off.astype(np.int32), page_id.astype(np.int32), max(num_pages, 1),
                       page_size)


def unused_slot_mask(spec: TreeSpec, layout: PagedLayout) -> np.ndarray:
    """bool [num_pages, P]: True where a physical (page, slot) holds no token
    of any node (tails of last pages and unreferenced pages)."""
    used = np.zeros((layout.num_pages, layout.page_size), dtype=bool)
    P = layout.page_size
    for n in range(spec.num_nodes):
        L = int(spec.node_len[n])
        for j in range((L + P - 1) // P):
            pg = layout.page_id[layout.node_page_off[n] + j]
            used[pg, : min(P, L - j * P)] = True
    return ~used


@dataclass
class Tensors:
    q: "object"        # torch bf16 [Q, Hq, d]
    k_pages: "object"  # torch bf16 [num_pages, Hkv, P, d]
    v_pages: "object"  # torch bf16 [num_pages, Hkv, P, d]


def make_tensors(spec: TreeSpec, layout: PagedLayout, device="cpu", seed: Optional[int] = None,
                 poison_unused: bool = False, zero_q: bool = False, equal_keys: bool = False):
    """Seeded Q, K, V: iid N(0,1) in fp32 (K times spec.k_scale), rounded to
    bf16 (round to nearest even).  With `poison_unused`, every KV slot that
    holds no token is set to NaN, so any read of it shows up in the output.
    `zero_q` and `equal_keys` build the closed-form special cases."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(spec.seed if seed is None else seed)
    Q, Hq, Hkv, d = spec.num_queries, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = torch.randn((Q, Hq, d), generator=g, device=device, dtype=torch.float32)
    shape = (layout.num_pages, Hkv, layout.page_size, d)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * spec.k_scale
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if zero_q:
        q.zero_()
    if equal_keys:
        k[:] = k[0, :, 0:1, :].unsqueeze(0).clone()
        k = k.expand(shape).contiguous()
    q, k, v = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    if poison_unused:
        mask = torch.from_numpy(unused_slot_mask(spec, layout)).to(device)
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16, device=device)
        m = mask[:, None, :, None].expand(shape)
        k = torch.where(m, nan, k)
        v = torch.where(m, nan, v)
    return Tensors(q.contiguous(), k.contiguous(), v.contiguous())


def bf16_bits(t) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 torch tensor, as a host numpy array."""
    import torch
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
