"""Shared test helpers: inputs built from contiguous per-token arrays and then
scattered into the paged layout, so that tests index KV one way (contiguous)
while the oracle and the kernels index it another (through the page table)."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import workloads as W

BF16_NAN = np.uint16(0x7FC0)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass
class DenseInputs:
    spec: W.TreeSpec
    layout: W.PagedLayout
    q_bits: np.ndarray        # uint16 [Q, Hq, d]
    k_tok: np.ndarray         # float64 [T, Hkv, d]  every token of every node, node-major
    v_tok: np.ndarray
    tok_node: np.ndarray      # int [T]
    tok_pos: np.ndarray       # int [T]  position inside its node
    k_pages: np.ndarray       # uint16 [pages, Hkv, P, d]  unused slots are NaN
    v_pages: np.ndarray

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)


def dense_inputs(spec: W.TreeSpec, seed: int = 0, spare_pages: int = 3, zero_q=False,
                 equal_keys=False, poison=True, k_ramp: float = 0.0) -> DenseInputs:
    """k_ramp > 0 scales the key of the token at position p of its node by
    1 + k_ramp * p, so that logits grow along a node (later tiles of a chunk
    then exceed the column maxima of its first tile)."""
    rng = np.random.default_rng(seed)
    Q, Hq, Hkv, d = spec.num_queries, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    T = int(spec.node_len.sum())
    q = rng.standard_normal((Q, Hq, d), dtype=np.float32)
    if zero_q:
        q[:] = 0
    k = rng.standard_normal((T, Hkv, d), dtype=np.float32) * np.float32(spec.k_scale)
    if equal_keys:
        k[:] = k[:1]
    if k_ramp:
        pos = np.concatenate([np.arange(L) for L in spec.node_len]) if T else np.zeros(0, int)
        k *= (1.0 + k_ramp * pos).astype(np.float32)[:, None, None]
    v = rng.standard_normal((T, Hkv, d), dtype=np.float32)
    q_bits, k_bits, v_bits = to_bf16_bits(q), to_bf16_bits(k), to_bf16_bits(v)
    tok_node = np.repeat(np.arange(spec.num_nodes), spec.node_len)
    tok_pos = np.concatenate([np.arange(L) for L in spec.node_len]) if T else np.zeros(0, int)
    layout = W.paged_layout(spec, spare_pages=spare_pages)
    P = layout.page_size
    fill = BF16_NAN if poison else np.uint16(0)
    kp = np.full((layout.num_pages, Hkv, P, d), fill, dtype=np.uint16)
    vp = np.full_like(kp, fill)
    start = 0
    for n in range(spec.num_nodes):
        L = int(spec.node_len[n])
        for j in range((L + P - 1) // P):
            cnt = min(P, L - j * P)
            pg = layout.page_id[layout.node_page_off[n] + j]
            src = slice(start + j * P, start + j * P + cnt)
            # [cnt, Hkv, d] -> [Hkv, cnt, d]
            kp[pg, :, :cnt, :] = np.transpose(k_bits[src], (1, 0, 2))
            vp[pg, :, :cnt, :] = np.transpose(v_bits[src], (1, 0, 2))
        start += L
    return DenseInputs(spec, layout, q_bits, bits_to_f64(k_bits), bits_to_f64(v_bits),
                       tok_node, tok_pos, kp, vp)


def subtree_sets(parent: np.ndarray):
    """Descendant-or-self sets by a downward traversal from each node (built
    from child lists, not by walking parents)."""
    n = len(parent)
    children = [[] for _ in range(n)]
    for i, p in enumerate(parent):
        if p >= 0:
            children[p].append(i)
    sets = []
    for i in range(n):
        seen, stack = set(), [i]
        while stack:
            x = stack.pop()
            seen.add(x)
            stack.extend(children[x])
        sets.append(seen)
    return sets


def dense_reference(inp: DenseInputs):
    """Textbook masked softmax attention over ALL tokens with the tree mask
    M[q, j] = 0 if token j's node has query q's node in its subtree (and, in
    q's own node, j's position is at most q's position when it has one),
    else -inf.  fp64, numpy."""
    spec = inp.spec
    sub = subtree_sets(spec.parent)
    Q, Hq, Hkv, d = spec.num_queries, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    G = Hq // Hkv
    T = inp.k_tok.shape[0]
    mask = np.full((Q, T), -np.inf)
    for qi in range(Q):
        pos = -1 if spec.query_pos is None else int(spec.query_pos[qi])
        for j in range(T):
            if spec.query_node[qi] in sub[inp.tok_node[j]]:
                own = inp.tok_node[j] == spec.query_node[qi]
                if not (own and pos >= 0 and inp.tok_pos[j] > pos):
                    mask[qi, j] = 0.0
    qf = bits_to_f64(inp.q_bits)
    out = np.zeros((Q, Hq, d))
    lse = np.full((Q, Hq), -np.inf)
    for h in range(Hq):
        K = np.repeat(inp.k_tok, G, axis=1)[:, h, :]   # [T, d], q head h -> kv head h // G
        V = np.repeat(inp.v_tok, G, axis=1)[:, h, :]
        S = qf[:, h, :] @ K.T * inp.scale + mask      # [Q, T]
        for qi in range(Q):
            row = S[qi]
            if not np.isfinite(row).any():
                continue
            m = row.max()
            p = np.exp(row - m)
            out[qi, h] = p @ V / p.sum()
            lse[qi, h] = m + np.log(p.sum())
    return out, lse


def run_oracle(inp: DenseInputs, query_subset=None, threads=0, lib=None):
    import oracle
    s = inp.spec
    return oracle.tree_attn(inp.q_bits, inp.k_pages, inp.v_pages, inp.layout.node_page_off,
                            inp.layout.page_id, inp.layout.page_size, s.parent, s.node_len,
                            s.query_node, s.num_q_heads, s.num_kv_heads, s.head_dim, inp.scale,
                            query_subset=query_subset, threads=threads, lib=lib,
                            query_pos=s.query_pos)
