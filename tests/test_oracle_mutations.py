"""Plant plausible mistakes in copies of the oracle's C source (on the CPU)
and check that the pins reject every one of them.  A pin set that a dropped
term, a wrong sign, a wrong index or a transposed operand slips through
would not be a pin."""
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from helpers import bits_to_f64, dense_inputs, dense_reference, run_oracle, subtree_sets

SRC = os.path.join(os.path.dirname(oracle.__file__), "deft_oracle.c")

MUTATIONS = {
    "path_excludes_the_node_itself": ("int32_t cur = n;\n", "int32_t cur = parent[n];\n"),
    "gqa_head_h_mod_hkv": ("head_dim, h / group, scale, tok_node, tok_idx, nt",
                           "head_dim, h % num_kv_heads, scale, tok_node, tok_idx, nt"),
    "scale_dropped": ("scores[j] = dot * scale;", "scores[j] = dot;"),
    "slot_off_by_one": ("int32_t slot = t % page_size;", "int32_t slot = (t + 1) % page_size;"),
    "head_and_slot_axes_swapped": (
        "return (((size_t)page * num_kv_heads + kvh) * page_size + slot) * head_dim;",
        "return (((size_t)page * page_size + slot) * num_kv_heads + kvh) * head_dim;"),
    "lse_without_max": ("return m + log(l);", "return log(l);"),
    "output_not_normalised": ("        out[i] /= l;\n    return", "        out[i] += 0.0;\n    return"),
    "exp_sign_flipped": ("double p = exp(scores[j] - m);", "double p = exp(m - scores[j]);"),
    "query_row_transposed": (
        "const uint16_t *qv = q + ((size_t)qi * num_q_heads + h) * head_dim;\n            double *o = out + ((size_t)i",
        "const uint16_t *qv = q + ((size_t)h * num_queries + qi) * head_dim;\n            double *o = out + ((size_t)i"),
    "cover_bit_uses_word_index": ("|= (uint64_t)1 << (q % 64);", "|= (uint64_t)1 << (q / 64);"),
    "unique_tokens_not_deduplicated": ("if (take > taken[buf[i]])\n                taken[buf[i]] = take;",
                                       "uniq += take;"),
    "path_not_reversed": ("for (int32_t i = 0; i < len / 2; ++i) {", "for (int32_t i = 0; i < 0; ++i) {"),
    "merge_weight_sign_flipped": ("double w = exp(piece_lse[p] - M);", "double w = exp(M - piece_lse[p]);"),
    "last_token_of_node_dropped": ("for (int32_t t = 0; t < tokens_taken(node_len, pathbuf[i], qnode, qpos); ++t) {",
                                   "for (int32_t t = 0; t + 1 < tokens_taken(node_len, pathbuf[i], qnode, qpos); ++t) {"),
    "own_node_position_off_by_one": ("        return pos + 1;\n", "        return pos;\n"),
}


def _close(a, b, tol=1e-9):
    a, b = np.asarray(a, float), np.asarray(b, float)
    if a.shape != b.shape:
        return False
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    return bool(np.all(both_inf | (np.abs(a - b) <= tol)))


def pins_pass(lib) -> bool:
    """A compact run of the oracle's pins against `lib`; False on any miss."""
    try:
        for spec in [W.random_tree(5, q_heads=4, kv_heads=2), W.random_tree(11), W.tiny_tree()]:
            inp = dense_inputs(spec, seed=7)
            out, lse = run_oracle(inp, lib=lib)
            ref, ref_lse = dense_reference(inp)
            if not (_close(out, ref) and _close(lse, ref_lse)):
                return False
        # chain == causal decode
        spec = W.chain_tree([5, 3, 7, 1, 4])
        inp = dense_inputs(spec, seed=1)
        out, _ = run_oracle(inp, lib=lib)
        T = int(spec.node_len.sum())
        qf = torch.from_numpy(bits_to_f64(inp.q_bits))
        K = torch.from_numpy(inp.k_tok[:, 0]); V = torch.from_numpy(inp.v_tok[:, 0])
        for i, e in enumerate(np.cumsum(spec.node_len) - 1):
            qfull = torch.zeros((T, spec.head_dim), dtype=torch.float64)
            qfull[e] = qf[i, 0]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qfull[None, None], K[None, None], V[None, None], is_causal=True,
                scale=inp.scale)[0, 0]
            if not _close(out[i, 0], ref[e].numpy()):
                return False
        # a node with a query at every position == causal self-attention
        spec = W.causal_node_tree(9, parent_len=5)
        inp = dense_inputs(spec, seed=6)
        out, _ = run_oracle(inp, lib=lib)
        K = torch.from_numpy(inp.k_tok[:, 0]); V = torch.from_numpy(inp.v_tok[:, 0])
        qf = torch.from_numpy(bits_to_f64(inp.q_bits))
        qfull = torch.zeros((14, spec.head_dim), dtype=torch.float64)
        qfull[5:] = qf[:, 0]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qfull[None, None], K[None, None], V[None, None], is_causal=True, scale=inp.scale)[0, 0]
        if not _close(out[:, 0], ref[5:].numpy()):
            return False
        # closed form: q = 0 -> mean, ln count
        spec = W.random_tree(101, zero_len_prob=0.0)
        inp = dense_inputs(spec, seed=2, zero_q=True)
        out, lse = run_oracle(inp, lib=lib)
        sub = subtree_sets(spec.parent)
        for qi in range(spec.num_queries):
            vis = [j for j in range(len(inp.tok_node)) if spec.query_node[qi] in sub[inp.tok_node[j]]]
            if abs(lse[qi, 0] - math.log(len(vis))) > 1e-9:
                return False
        # integer facts
        spec = W.random_tree(401, max_nodes=30, max_queries=70)
        sub = subtree_sets(spec.parent)
        cov = oracle.cover(spec.parent, spec.query_node, lib=lib)
        paths = oracle.paths(spec.parent, spec.query_node, lib=lib)
        for qi, p in enumerate(paths):
            if p[-1] != spec.query_node[qi] or spec.parent[p[0]] != -1:
                return False
        for n in range(spec.num_nodes):
            for qi in range(spec.num_queries):
                if ((int(cov[n, qi // 64]) >> (qi % 64)) & 1) != (spec.query_node[qi] in sub[n]):
                    return False
        uniq, _ = oracle.token_counts(spec.parent, spec.node_len, spec.query_node, lib=lib)
        on_any = [n for n in range(spec.num_nodes)
                  if any(spec.query_node[q] in sub[n] for q in range(spec.num_queries))]
        if uniq != int(spec.node_len[on_any].sum()):
            return False
        # worked example: 93.4% needs the inclusive ancestor count 54
        ex = W.heap_example_tree()
        anc = sum(len(p) - 1 for p in oracle.paths(ex.parent, ex.query_node, lib=lib))
        if round(100 * (1 - (2048 + 2 * anc) / 32896), 1) != 93.4:
            return False
        # split-and-merge equals direct
        spec = W.random_tree(302, max_len=60)
        inp = dense_inputs(spec, seed=3)
        out, lse = run_oracle(inp, lib=lib)
        cut = (np.random.default_rng(0).random(int(spec.node_len.sum()) + 1) < 0.3).astype(np.uint8)
        s = spec
        out2, lse2 = oracle.tree_attn_pieces(inp.q_bits, inp.k_pages, inp.v_pages,
                                             inp.layout.node_page_off, inp.layout.page_id,
                                             inp.layout.page_size, s.parent, s.node_len,
                                             s.query_node, s.num_q_heads, s.num_kv_heads,
                                             s.head_dim, inp.scale, cut, lib=lib)
        if not (_close(out2, out) and _close(lse2, lse)):
            return False
    except ValueError:
        return False
    return True


def test_unmutated_oracle_passes_the_compact_pins():
    assert pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(mutated), out=str(tmp_path / "libm.so")))
    assert not pins_pass(lib), f"planted mistake '{name}' passed every pin"
