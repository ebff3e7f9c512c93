"""Pins of the fp64 oracle against things other than itself (no GPU).

* dense brute force with an explicit tree mask built from subtree sets
  (DeFT Guide, section "Deep Dive: Mathematical Formulation": tree-constrained
  attention with the causal tree mask);
* a single-branch tree equals ordinary causal decode attention, computed by
  torch's scaled_dot_product_attention;
* closed forms: one token, q = 0, equal keys, empty path;
* node relabelling and any split-and-merge partition leave results unchanged;
* the Guide's worked IO example (section "End-to-End Implementation").
"""
import json
import zlib
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits_to_f64, dense_inputs, dense_reference, run_oracle, subtree_sets

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY_SPECS = [W.random_tree(s) for s in range(24)] + [W.tiny_tree()]


@pytest.mark.parametrize("spec", TINY_SPECS, ids=lambda s: s.name)
def test_oracle_matches_dense_masked_attention(spec):
    inp = dense_inputs(spec, seed=zlib.crc32(spec.name.encode()) % 1000)
    out, lse = run_oracle(inp)
    ref_out, ref_lse = dense_reference(inp)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(lse), np.isinf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    assert np.isfinite(out).all(), "oracle read a poisoned (unused) KV slot"


def test_oracle_gqa_head_mapping_is_h_div_g():
    # With 4 query heads on 2 KV heads, q head h reads KV head h // 2.  A
    # dense check with G != 1 and distinct KV heads fails for h % Hkv.
    spec = W.random_tree(5, q_heads=4, kv_heads=2)
    inp = dense_inputs(spec, seed=9)
    out, _ = run_oracle(inp)
    ref, _ = dense_reference(inp)
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("lengths", [[5, 3, 7, 1, 4], [17, 16, 1, 33], [1], [40, 0, 9]])
def test_chain_tree_equals_causal_decode(lengths):
    spec = W.chain_tree(lengths, q_heads=2, kv_heads=1, head_dim=64)
    inp = dense_inputs(spec, seed=len(lengths))
    out, lse = run_oracle(inp)
    T = int(sum(lengths))
    ends = np.cumsum(lengths) - 1          # sequence position of each node's last token
    qf = torch.from_numpy(bits_to_f64(inp.q_bits))
    K = torch.from_numpy(inp.k_tok[:, 0, :])
    V = torch.from_numpy(inp.v_tok[:, 0, :])
    mask = torch.triu(torch.ones(T, T, dtype=torch.bool), 1)
    for h in range(spec.num_q_heads):
        for i, e in enumerate(ends):
            # Causal decode over the concatenated sequence: the query for node
            # i sits at position ends[i] and sees positions 0..ends[i].
            qfull = torch.zeros((T, spec.head_dim), dtype=torch.float64)
            qfull[e] = qf[i, h]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qfull[None, None], K[None, None], V[None, None], is_causal=True,
                scale=inp.scale)[0, 0]
            scores = ((qfull @ K.T) * inp.scale).masked_fill(mask, -math.inf)
            ref_lse = torch.logsumexp(scores, dim=-1)
            np.testing.assert_allclose(out[i, h], ref[e].numpy(), atol=1e-12, rtol=0)
            np.testing.assert_allclose(lse[i, h], ref_lse[e].item(), atol=1e-12, rtol=0)


def test_single_token_path_returns_that_value():
    spec = W.TreeSpec("one", np.array([-1], np.int32), np.array([1], np.int32),
                      np.array([0], np.int32), 2, 1, 64)
    inp = dense_inputs(spec, seed=3)
    out, lse = run_oracle(inp)
    qf = bits_to_f64(inp.q_bits)
    for h in range(2):
        np.testing.assert_array_equal(out[0, h], inp.v_tok[0, 0])
        s = float(np.dot(qf[0, h], inp.k_tok[0, 0])) * inp.scale
        assert abs(lse[0, h] - s) < 1e-12


@pytest.mark.parametrize("seed", range(6))
def test_zero_query_gives_mean_and_log_count(seed):
    spec = W.random_tree(100 + seed, zero_len_prob=0.0)
    inp = dense_inputs(spec, seed=seed, zero_q=True)
    out, lse = run_oracle(inp)
    sub = subtree_sets(spec.parent)
    G = spec.gqa_group
    for qi in range(spec.num_queries):
        vis = [j for j in range(len(inp.tok_node)) if spec.query_node[qi] in sub[inp.tok_node[j]]]
        for h in range(spec.num_q_heads):
            np.testing.assert_allclose(out[qi, h], inp.v_tok[vis, h // G].mean(axis=0),
                                       atol=1e-12, rtol=0)
            assert abs(lse[qi, h] - math.log(len(vis))) < 1e-12


def test_equal_keys_give_mean_and_shifted_log_count():
    spec = W.random_tree(7, zero_len_prob=0.0, kv_heads=1, q_heads=2)
    inp = dense_inputs(spec, seed=1, equal_keys=True)
    out, lse = run_oracle(inp)
    sub = subtree_sets(spec.parent)
    qf = bits_to_f64(inp.q_bits)
    for qi in range(spec.num_queries):
        vis = [j for j in range(len(inp.tok_node)) if spec.query_node[qi] in sub[inp.tok_node[j]]]
        for h in range(2):
            s = float(np.dot(qf[qi, h], inp.k_tok[0, 0])) * inp.scale
            np.testing.assert_allclose(out[qi, h], inp.v_tok[vis, 0].mean(axis=0), atol=1e-12)
            assert abs(lse[qi, h] - (s + math.log(len(vis)))) < 1e-12


def test_empty_path_gives_zero_and_minus_inf():
    # Query 0 at an empty root, query 1 at an empty child of it, query 2 at a
    # non-empty child.
    spec = W.TreeSpec("empty", np.array([-1, 0, 0], np.int32), np.array([0, 0, 3], np.int32),
                      np.array([0, 1, 2], np.int32), 2, 2, 64)
    inp = dense_inputs(spec, seed=4)
    out, lse = run_oracle(inp)
    assert np.all(out[:2] == 0) and np.all(np.isneginf(lse[:2]))
    assert np.isfinite(lse[2]).all()


@pytest.mark.parametrize("seed", range(5))
def test_relabelling_nodes_is_bit_identical(seed):
    spec = W.random_tree(200 + seed, max_nodes=14)
    inp = dense_inputs(spec, seed=seed)
    out, lse = run_oracle(inp)
    perm = np.random.default_rng(seed).permutation(spec.num_nodes)
    rs = W.relabel(spec, perm)
    # Same physical pages under the new numbering.
    lay = inp.layout
    counts = np.diff(lay.node_page_off)
    new_counts = np.zeros(spec.num_nodes, np.int64)
    new_counts[perm] = counts
    off = np.zeros(spec.num_nodes + 1, np.int64)
    off[1:] = np.cumsum(new_counts)
    pid = np.zeros(lay.page_id.shape[0], np.int32)
    for old in range(spec.num_nodes):
        new = perm[old]
        pid[off[new]:off[new + 1]] = lay.page_id[lay.node_page_off[old]:lay.node_page_off[old + 1]]
    out2, lse2 = oracle.tree_attn(inp.q_bits, inp.k_pages, inp.v_pages, off, pid, lay.page_size,
                                  rs.parent, rs.node_len, rs.query_node, rs.num_q_heads,
                                  rs.num_kv_heads, rs.head_dim, inp.scale)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


@pytest.mark.parametrize("seed", range(6))
def test_any_partition_merges_to_the_direct_result(seed):
    spec = W.random_tree(300 + seed, max_len=60)
    inp = dense_inputs(spec, seed=seed)
    out, lse = run_oracle(inp)
    rng = np.random.default_rng(seed)
    cut = (rng.random(int(spec.node_len.sum()) + 1) < [0.05, 0.3, 0.7][seed % 3]).astype(np.uint8)
    s = spec
    out2, lse2 = oracle.tree_attn_pieces(inp.q_bits, inp.k_pages, inp.v_pages,
                                         inp.layout.node_page_off, inp.layout.page_id,
                                         inp.layout.page_size, s.parent, s.node_len, s.query_node,
                                         s.num_q_heads, s.num_kv_heads, s.head_dim, inp.scale, cut)
    np.testing.assert_allclose(out2, out, atol=1e-12, rtol=0)
    fin = np.isfinite(lse)
    np.testing.assert_array_equal(fin, np.isfinite(lse2))
    np.testing.assert_allclose(lse2[fin], lse[fin], atol=1e-12, rtol=0)


@pytest.mark.parametrize("seed", range(20))
def test_cover_and_paths_match_subtree_enumeration(seed):
    spec = W.random_tree(400 + seed, max_nodes=30, max_queries=70)
    sub = subtree_sets(spec.parent)
    cov = oracle.cover(spec.parent, spec.query_node)
    paths = oracle.paths(spec.parent, spec.query_node)
    for n in range(spec.num_nodes):
        for qi in range(spec.num_queries):
            on_path = spec.query_node[qi] in sub[n]
            bit = (int(cov[n, qi // 64]) >> (qi % 64)) & 1
            assert bit == on_path
            assert (n in paths[qi]) == on_path
    for qi, p in enumerate(paths):
        assert p[-1] == spec.query_node[qi]
        assert spec.parent[p[0]] == -1
        for a, b in zip(p, p[1:]):
            assert spec.parent[b] == a
    uniq, naive = oracle.token_counts(spec.parent, spec.node_len, spec.query_node)
    on_any = [n for n in range(spec.num_nodes) if any(spec.query_node[q] in sub[n]
                                                      for q in range(spec.num_queries))]
    assert uniq == int(spec.node_len[on_any].sum())
    assert naive == sum(int(spec.node_len[n]) for qi in range(spec.num_queries)
                        for n in range(spec.num_nodes) if spec.query_node[qi] in sub[n])


def test_oracle_rejects_a_cycle():
    with pytest.raises(ValueError):
        oracle.paths(np.array([1, 0], np.int32), np.array([0], np.int32))


def test_worked_io_example_of_the_guide():
    with open(os.path.join(GOLDEN, "worked_example_io.json")) as f:
        g = json.load(f)
    setup, printed = g["setup"], g["printed"]
    prefix, nq = setup["prefix_length"], setup["num_candidate_nodes"]
    spec = W.heap_example_tree(prefix, nq)
    # The conventional count exactly as the page's formula states it.
    assert nq * prefix * 2 + nq * 4 * 2 == printed["conventional_reads"]
    # The script's count on this tree: prefix once, then 2 per (query, node in
    # its inclusive ancestor list) over the candidate nodes.
    paths = oracle.paths(spec.parent, spec.query_node)
    anc = sum(len(p) - 1 for p in paths)          # drop the prefix node
    assert anc == 54
    deft = 2 * prefix + 2 * anc
    assert round(100.0 * (1 - deft / printed["conventional_reads"]), 1) == printed["io_reduction_percent"]
    # An exclusive ancestor list would print 93.5%: the inclusive reading is pinned.
    excl = 2 * prefix + 2 * (anc - nq)
    assert round(100.0 * (1 - excl / printed["conventional_reads"]), 1) != printed["io_reduction_percent"]
    # The printed 2176 is the fixed-depth-4 figure, not this tree's count.
    assert printed["deft_reads"] == 2 * prefix + nq * 4 * 2 != deft
    uniq, naive = oracle.token_counts(spec.parent, spec.node_len, spec.query_node)
    assert uniq == prefix + nq
    assert naive == nq * prefix + anc


# ---------------------------------------------------------------------------
# Queries at token positions of multi-token nodes (tree verification / node
# prefill: the Guide's causal tree mask, section "Deep Dive", at token level)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_positions_match_dense_masked_attention(seed):
    """Random trees with queries at random positions of their nodes against
    the brute-force masked softmax (mask built from subtree sets and the
    token positions)."""
    spec = W.positions_tree(seed, q_heads=4, kv_heads=2)
    inp = dense_inputs(spec, seed=seed)
    out, lse = run_oracle(inp)
    ref, ref_lse = dense_reference(inp)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("length,parent_len", [(9, 0), (33, 5), (1, 16), (70, 17)])
def test_node_with_a_query_at_every_position_is_causal_attention(length, parent_len):
    """Queries at positions 0..L-1 of one node (under a root of parent_len
    tokens) equal causal self-attention over root + node, computed by torch's
    scaled_dot_product_attention."""
    spec = W.causal_node_tree(length, q_heads=2, kv_heads=1, parent_len=parent_len)
    inp = dense_inputs(spec, seed=length)
    out, _ = run_oracle(inp)
    T = parent_len + length
    K = torch.from_numpy(inp.k_tok[:, 0]); V = torch.from_numpy(inp.v_tok[:, 0])
    qf = torch.from_numpy(bits_to_f64(inp.q_bits))
    for h in range(spec.num_q_heads):
        qfull = torch.zeros((T, spec.head_dim), dtype=torch.float64)
        qfull[parent_len:] = qf[:, h]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qfull[None, None], K[None, None], V[None, None], is_causal=True,
            scale=inp.scale)[0, 0]
        np.testing.assert_allclose(out[:, h], ref[parent_len:].numpy(), rtol=0, atol=1e-12)


@pytest.mark.parametrize("length", [1, 6, 19])
def test_positions_equal_a_chain_of_one_token_nodes(length):
    """A node of L tokens with a query at each position gives bit for bit
    the results of a chain of L one-token nodes with a query at each node
    (the same tokens, attended in the same order)."""
    a = W.causal_node_tree(length, parent_len=4)
    b = W.chain_tree([4] + [1] * length, q_heads=a.num_q_heads, kv_heads=a.num_kv_heads,
                     head_dim=a.head_dim)
    b.query_node = np.arange(1, length + 1, dtype=np.int32)
    ia, ib = dense_inputs(a, seed=9), dense_inputs(b, seed=9)
    np.testing.assert_array_equal(ia.q_bits, ib.q_bits)
    oa, la = run_oracle(ia)
    ob, lb = run_oracle(ib)
    np.testing.assert_array_equal(oa, ob)
    np.testing.assert_array_equal(la, lb)


@pytest.mark.parametrize("seed", range(4))
def test_last_position_is_the_whole_node(seed):
    spec = W.positions_tree(seed)
    tip = spec.node_len[spec.query_node] - 1
    spec.query_pos = np.where(spec.node_len[spec.query_node] > 0, tip, -1).astype(np.int32)
    inp = dense_inputs(spec, seed=seed)
    out, lse = run_oracle(inp)
    spec.query_pos = None
    out2, lse2 = run_oracle(inp)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_position_token_counts_closed_form():
    L, P = 23, 7
    spec = W.causal_node_tree(L, parent_len=P)
    uniq, naive = oracle.token_counts(spec.parent, spec.node_len, spec.query_node,
                                      query_pos=spec.query_pos)
    assert uniq == P + L
    assert naive == sum(P + i + 1 for i in range(L))
    # only the first 3 tokens of the node attended by anyone
    pos = np.array([0, 2, 1], dtype=np.int32)
    uniq, naive = oracle.token_counts(spec.parent, spec.node_len, np.array([1, 1, 1], np.int32),
                                      query_pos=pos)
    assert uniq == P + 3 and naive == 3 * P + 1 + 3 + 2
    with pytest.raises(ValueError):
        oracle.token_counts(spec.parent, spec.node_len, np.array([1], np.int32),
                            query_pos=np.array([L], np.int32))
