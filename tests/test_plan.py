"""Host planner and C-ABI checks (no GPU).

The planner's integer outputs are compared bit-exactly with the oracle's
independent coverage bitsets and token counts, and its chunks are expanded
into (query, node, token) triples that must cover every query's path exactly
once (KV-Guided Grouping + Flattened Tree KV Splitting: DeFT abstract; DeFT
Guide, "The DeFT Architecture")."""
import ctypes
import os
import re
from collections import defaultdict

import numpy as np
import pytest

import oracle
import workloads as W

deft = pytest.importorskip("shared_prefix_kv_deft_gb300")
from shared_prefix_kv_deft_gb300 import build as deft_build  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    deft_build.build()
    deft.load()


def header_functions():
    src = open(os.path.join(ROOT, "include", "deft.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int32_t|int|size_t|void|const char \*)\s*(deft_\w+)\s*\(", src, re.M)))


def test_library_exports_every_declared_symbol():
    lib = deft.load()
    names = header_functions()
    assert set(names) == set(deft.EXPORTS)
    for n in names:
        assert hasattr(lib, n), f"libdeft.so does not export {n}"
    assert deft.version() == 200


@pytest.mark.parametrize("parent,node_len,query,ct,g,status", [
    ([1, 0], [3, 3], [0], 64, 1, -2),            # cycle
    ([-1, 0, 1, 2, 1], [1, 1, 1, 1, 1], [4], 64, 1, 0),
    ([-1, 5], [3, 3], [0], 64, 1, -3),           # parent out of range
    ([-1, -2], [3, 3], [0], 64, 1, -3),          # parent below -1
    ([-1, 0], [3, -1], [0], 64, 1, -1),          # negative length
    ([-1, 0], [3, 3], [2], 64, 1, -3),           # query node out of range
    ([-1, 0], [3, 3], [1], 0, 1, -1),            # chunk_target 0
    ([-1, 0], [3, 3], [1], 9000, 1, -1),         # chunk_target too large
    ([-1, 0], [3, 3], [1], 64, 0, -1),           # GQA group 0
    ([0], [3], [0], 64, 1, -2),                  # self loop
])
def test_plan_validation(parent, node_len, query, ct, g, status):
    lib = deft.load()
    p = np.array(parent, np.int32)
    L = np.array(node_len, np.int32)
    qn = np.array(query, np.int32)
    h = ctypes.c_void_p()
    rc = lib.deft_plan(p.ctypes.data_as(ctypes.c_void_p), L.ctypes.data_as(ctypes.c_void_p),
                       len(parent), qn.ctypes.data_as(ctypes.c_void_p), len(query), ct, g,
                       ctypes.byref(h))
    assert rc == status
    if rc == 0:
        lib.deft_plan_free(h)
    else:
        assert not h.value


def check_plan(spec: W.TreeSpec, chunk_target: int, G: int, tensor_pack: bool = False):
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, chunk_target, G,
                     query_pos=spec.query_pos, tensor_pack=tensor_pack)
    st = plan.stats
    Q, N = spec.num_queries, spec.num_nodes
    Wd = (Q + 63) // 64
    cover = oracle.cover(spec.parent, spec.query_node)
    uniq, naive = oracle.token_counts(spec.parent, spec.node_len, spec.query_node,
                                      query_pos=spec.query_pos)
    paths = oracle.paths(spec.parent, spec.query_node)

    def taken(q, n):
        """Tokens of node n (on q's path) that query q attends."""
        if spec.query_pos is not None and n == spec.query_node[q] and spec.query_pos[q] >= 0:
            return int(spec.query_pos[q]) + 1
        return int(spec.node_len[n])

    # Bit-exact coverage bitsets and token counts.
    np.testing.assert_array_equal(plan.get("node_cover").reshape(N, Wd), cover)
    assert st["unique_tokens"] == uniq and st["planned_tokens"] == uniq
    assert st["naive_tokens"] == naive
    order = plan.get("node_order")
    assert sorted(order.tolist()) == list(range(N))

    def bits(words):
        return [q for q in range(Q) if (int(words[q // 64]) >> (q % 64)) & 1]

    def check_partition(prefix, chunk_limit, naive_part):
        seg_off = plan.get(prefix + "chunk_seg_off")
        chunk_q = plan.get(prefix + "chunk_q")
        seg_node = plan.get(prefix + "seg_node")
        seg_b = plan.get(prefix + "seg_tok_begin")
        seg_l = plan.get(prefix + "seg_tok_len")
        q_off = plan.get(prefix + "q_slot_off")
        q_slot = plan.get(prefix + "q_slot")
        C = len(seg_off) - 1
        if naive_part:
            chunk_q_off = np.arange(C + 1)
            seg_mask = None
        else:
            chunk_q_off = plan.get("chunk_q_off")
            seg_mask = plan.get("seg_mask").reshape(-1, Wd)
            chunk_mask = plan.get("chunk_mask").reshape(-1, Wd)
        assert len(chunk_q) == chunk_q_off[-1]
        intervals = defaultdict(list)
        for c in range(C):
            qs = chunk_q[chunk_q_off[c]:chunk_q_off[c + 1]].tolist()
            assert qs == sorted(set(qs)) and len(qs) > 0
            if naive_part:
                assert len(qs) == 1
            tok = 0
            union = set()
            nseg = seg_off[c + 1] - seg_off[c]
            assert nseg >= 1
            nodes = set()
            for s in range(seg_off[c], seg_off[c + 1]):
                n, b, L = int(seg_node[s]), int(seg_b[s]), int(seg_l[s])
                assert L > 0 and 0 <= b and b + L <= spec.node_len[n]
                # A whole page (aligned in its node) sits at an aligned
                # position of the chunk: one copy moves it.
                if b % 16 == 0 and L >= 16:
                    assert tok % 16 == 0, f"chunk {c}: page of node {n} at position {tok}"
                tok += L
                nodes.add(n)
                if naive_part:
                    sq = qs
                else:
                    # A segment's bitmask is exactly the set of queries that
                    # attend its tokens: its node's coverage set, less the
                    # queries sitting in the node before the segment.
                    sq = bits(seg_mask[s])
                    want = [q for q in bits(cover[n]) if taken(q, n) > b]
                    assert sq == want
                    assert all(taken(q, n) >= b + L for q in sq)
                union |= set(sq)
                for q in sq:
                    intervals[(q, n)].append((b, L))
            assert union == set(qs)
            if not naive_part:
                assert bits(chunk_mask[c]) == qs
                if len(nodes) > 1:
                    # Chunks of several nodes: short nodes up to the chunk
                    # target, or tensor-packed pieces of up to
                    # max(256, limit / nodes) tokens.
                    limit = max(chunk_limit, 256 * len(nodes)) if tensor_pack else chunk_limit
                    assert tok <= limit and nseg <= 256
            else:
                assert tok <= chunk_limit
        # Exactly once: every (query, node on its path, token) in one chunk.
        expected = {(q, n) for q in range(Q) for n in paths[q] if taken(q, n) > 0}
        assert set(intervals) == expected
        for (q, n), iv in intervals.items():
            iv.sort()
            pos = 0
            for b, L in iv:
                assert b == pos, f"gap/overlap at query {q} node {n}"
                pos = b + L
            assert pos == taken(q, n)
        # Slot CSR: slot s of chunk_q belongs to query chunk_q[s].
        for q in range(Q):
            sl = q_slot[q_off[q]:q_off[q + 1]].tolist()
            assert sl == [s for s in range(len(chunk_q)) if chunk_q[s] == q]
        return C, chunk_q_off, chunk_q

    C, cqo, _ = check_partition("", chunk_target, False)
    check_partition("naive_", chunk_target, True)
    assert st["num_chunks"] == C

    # Work items: each chunk's query list covered once per family.
    def item_cover(name):
        it = plan.get(name).reshape(-1, 3)
        cov = defaultdict(list)
        for c, b, e in it:
            assert 0 <= b < e <= cqo[c + 1] - cqo[c]
            cov[int(c)].append((int(b), int(e)))
        return it, cov

    fma, fcov = item_cover("fma_items")
    mma, mcov = item_cover("mma_items")
    fb, bcov = item_cover("fallback_items")
    for c in range(C):
        k = cqo[c + 1] - cqo[c]
        if k * G < 16:
            assert c not in mcov and c not in bcov
            iv = sorted(fcov[c])
            pos = 0
            for b, e in iv:   # row blocks of at most 8 rows (whole queries)
                assert b == pos and (e - b) * G <= max(8, G)
                pos = e
            assert pos == k and len(iv) == -(-k // max(1, 8 // G))
        else:
            for fam, cap in ((mcov, 128), (bcov, 16)):
                iv = sorted(fam[c])
                pos = 0
                for b, e in iv:
                    assert b == pos and (e - b) * G <= max(cap, G)
                    pos = e
                assert pos == k
    for it in (fma, fb):   # sorted by row bucket
        rows = [(e - b) * G for _, b, e in it]
        buckets = [0 if r <= 1 else 1 if r <= 2 else 2 if r <= 4 else 3 if r <= 8 else 4 for r in rows]
        assert buckets == sorted(buckets)
    return plan


RANDOM = [W.random_tree(s, max_nodes=40, max_len=300, max_queries=90) for s in range(40)]


@pytest.mark.parametrize("spec", RANDOM, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [1, 16, 100, 512])
def test_plan_random_trees(spec, ct):
    check_plan(spec, ct, spec.gqa_group)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 6])
def test_plan_workload_shapes(cfg):
    spec = W.config(cfg)
    plan = check_plan(spec, 256, spec.gqa_group)
    st = plan.stats
    if cfg == 2:
        assert st["unique_tokens"] == 4096 + 32 * 256
        assert st["naive_tokens"] == 32 * (4096 + 256)


@pytest.mark.parametrize("seed", range(4))
def test_plan_relabelled_tree_has_the_same_coverage(seed):
    spec = W.random_tree(900 + seed, max_nodes=30, max_queries=40)
    perm = np.random.default_rng(seed).permutation(spec.num_nodes)
    check_plan(W.relabel(spec, perm), 64, 2)


def test_plan_worked_example_counts():
    spec = W.heap_example_tree()
    plan = check_plan(spec, 64, 1)
    assert plan.stats["unique_tokens"] == 1040
    assert plan.stats["naive_tokens"] == 16 * 1024 + 54


def test_plan_is_deterministic():
    spec = W.config(4)
    a = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, 4)
    b = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, 4)
    for name in deft.ARRAYS:
        np.testing.assert_array_equal(a.get(name), b.get(name))


def test_empty_query_list_plans():
    plan = deft.Plan([-1, 0], [5, 5], [], 64, 1)
    assert plan.stats["num_chunks"] == 0 and plan.stats["num_slots"] == 0


POSITIONS = [W.positions_tree(s, max_nodes=30, max_len=200, max_queries=70) for s in range(30)]
POSITIONS += [W.causal_node_tree(L, parent_len=P) for L, P in ((40, 0), (300, 1000), (17, 33))]


@pytest.mark.parametrize("spec", POSITIONS, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [1, 16, 100, 512])
def test_plan_with_query_positions(spec, ct):
    """Queries at token positions: the same exactly-once coverage of every
    (query, node, token) the query attends, segment masks equal to the
    attending query sets, and the oracle's token counts."""
    check_plan(spec, ct, 4)


def test_plan_rejects_positions_outside_the_node():
    spec = W.causal_node_tree(8)
    for bad in (8, -2):
        pos = spec.query_pos.copy()
        pos[3] = bad
        with pytest.raises(deft.DeftError):
            deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1, query_pos=pos)


def test_positions_at_the_last_token_plan_like_no_positions():
    spec = W.random_tree(7, max_nodes=20, max_len=120, max_queries=40, zero_len_prob=0.0)
    a = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 2)
    b = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 2,
                  query_pos=spec.node_len[spec.query_node] - 1)
    for name in ("chunk_seg_off", "chunk_q", "seg_node", "seg_tok_begin", "seg_tok_len",
                 "seg_mask", "q_slot", "mma_items", "fma_items"):
        np.testing.assert_array_equal(a.get(name), b.get(name))


@pytest.mark.parametrize("cfg", [2, 4, 7])
def test_tree_only_plan_matches_the_full_plan(cfg):
    """DEFT_PLAN_TREE_ONLY leaves the tree partition as it is and the naive
    one empty (no chunk, no slot; every query's slot list empty)."""
    spec = W.config(cfg)
    full = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group,
                     query_pos=spec.query_pos)
    tree = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group,
                     query_pos=spec.query_pos, naive=False)
    for name in deft.ARRAYS:
        if name.startswith("naive_"):
            continue
        np.testing.assert_array_equal(full.get(name), tree.get(name))
    for key, v in tree.stats.items():
        if key.startswith("naive_num_"):
            assert v == 0
        elif key != "device_bytes":
            assert v == full.stats[key], key
    assert tree.stats["device_bytes"] < full.stats["device_bytes"]
    assert tree.get("naive_chunk_seg_off").tolist() == [0]
    assert tree.get("naive_q_slot_off").tolist() == [0] * (spec.num_queries + 1)
    for name in ("naive_chunk_q", "naive_seg_node", "naive_q_slot"):
        assert tree.get(name).size == 0


def test_plan_ex_rejects_unknown_flags():
    lib = deft.load()
    p = np.array([-1, 0], np.int32)
    L = np.array([5, 5], np.int32)
    qn = np.array([1], np.int32)
    h = ctypes.c_void_p()
    vp = ctypes.c_void_p
    for bad in (4, 8, 1 << 20):
        rc = lib.deft_plan_ex(p.ctypes.data_as(vp), L.ctypes.data_as(vp), 2, qn.ctypes.data_as(vp), None, 1,
                              64, 1, bad, ctypes.byref(h))
        assert rc == -1 and not h.value
    for good in (deft.PLAN_TREE_ONLY, deft.PLAN_TENSOR_PACK, deft.PLAN_TREE_ONLY | deft.PLAN_TENSOR_PACK):
        rc = lib.deft_plan_ex(p.ctypes.data_as(vp), L.ctypes.data_as(vp), 2, qn.ctypes.data_as(vp), None, 1,
                              64, 1, good, ctypes.byref(h))
        assert rc == 0 and h.value
        lib.deft_plan_free(h)


REBUILDS = [(2, 4), (4, 7), (7, 1), (1, 3)]


@pytest.mark.parametrize("first,second", REBUILDS)
@pytest.mark.parametrize("naive", [True, False])
def test_rebuild_matches_a_fresh_plan(first, second, naive):
    """deft_plan_rebuild leaves exactly what deft_plan_ex builds for the new
    tree (every array and statistic)."""
    a, b = W.config(first), W.config(second)
    p = deft.Plan(a.parent, a.node_len, a.query_node, 256, a.gqa_group, query_pos=a.query_pos)
    p.rebuild(b.parent, b.node_len, b.query_node, 128, b.gqa_group, query_pos=b.query_pos, naive=naive)
    f = deft.Plan(b.parent, b.node_len, b.query_node, 128, b.gqa_group, query_pos=b.query_pos, naive=naive)
    assert p.stats == f.stats
    for name in deft.ARRAYS:
        np.testing.assert_array_equal(p.get(name), f.get(name))


def test_plans_rebuilt_in_turn_each_match_a_fresh_plan():
    """Rebuilds build into a spare host plan of the calling thread that the
    plans share (its arrays keep their storage): two plans rebuilt in turn
    over different trees, and one rebuilt after a failed rebuild, each hold
    exactly a fresh plan of their last tree."""
    specs = [W.config(c) for c in (2, 4, 7, 1)] + [W.random_tree(s, max_nodes=30, max_len=300, max_queries=50,
                                                                 q_heads=8, kv_heads=2, head_dim=128)
                                                   for s in range(4)]
    plans = [deft.Plan(specs[0].parent, specs[0].node_len, specs[0].query_node, 256, specs[0].gqa_group)
             for _ in range(2)]
    for k, s in enumerate(specs * 2):
        p = plans[k % 2]
        if k == 5:
            with pytest.raises(deft.DeftError):
                p.rebuild(s.parent, s.node_len, s.query_node, 0, s.gqa_group)
        tp = k % 3 == 0
        p.rebuild(s.parent, s.node_len, s.query_node, 100, s.gqa_group, query_pos=s.query_pos, tensor_pack=tp)
        f = deft.Plan(s.parent, s.node_len, s.query_node, 100, s.gqa_group, query_pos=s.query_pos, tensor_pack=tp)
        assert p.stats == f.stats
        for name in deft.ARRAYS:
            np.testing.assert_array_equal(p.get(name), f.get(name), err_msg=f"step {k} {name}")


def test_failed_rebuild_leaves_the_plan_unchanged():
    a = W.config(4)
    p = deft.Plan(a.parent, a.node_len, a.query_node, 256, a.gqa_group)
    before = {name: p.get(name).copy() for name in deft.ARRAYS}
    stats = dict(p.stats)
    bad_parent = a.parent.copy()
    bad_parent[3] = 3   # a self-loop: not a forest
    for kwargs in ({"parent": bad_parent}, {"chunk_target": 0}, {"query_node": a.query_node + 10 ** 6}):
        args = dict(parent=a.parent, node_len=a.node_len, query_node=a.query_node, chunk_target=256,
                    gqa_group=a.gqa_group)
        args.update(kwargs)
        with pytest.raises(deft.DeftError):
            p.rebuild(**args)
        assert p.stats == stats
        for name in deft.ARRAYS:
            np.testing.assert_array_equal(p.get(name), before[name])


# ---------------------------------------------------------------------------
# Host-side checks of the step ABI (no GPU: every case below returns before
# the library makes a CUDA call).
# ---------------------------------------------------------------------------

def _tiny_plan():
    spec = W.tiny_tree()
    return spec, deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, spec.gqa_group)


def test_workspace_holds_the_partials_of_the_larger_partition():
    spec, plan = _tiny_plan()
    st = plan.stats
    slots = max(st["num_slots"], st["naive_num_slots"])
    up = lambda x: (x + 255) // 256 * 256   # noqa: E731
    for hq, d in ((4, 64), (8, 128)):
        assert plan.workspace_bytes(hq, d) == up(slots * hq * d * 4) + up(slots * hq * 4)
    assert plan.workspace_bytes(0, 64) == 0


def test_direct_rows_and_merge_queries_follow_the_slot_counts():
    """A row goes to out / lse from phase 1 exactly when its query has one
    partial slot and that slot's chunk has fewer than 16 rows (a CUDA-core
    chunk); the merge launch takes every other query."""
    cases = [(W.tiny_tree(), 256), (W.tiny_tree(), 16), (W.config(2), 256),
             (W.reasoning_tree(levels=3, len_lo=5, len_hi=40, num_queries=12, q_heads=4, kv_heads=2), 32),
             (W.imbalance_tree(leaves=12, control=True, control_len=150, q_heads=8, kv_heads=2), 64),
             (W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128), 8192)]
    cases += [(s, ct) for s in RANDOM[:10] for ct in (1, 16, 512)]
    seen_direct = seen_merge = 0
    for spec, ct in cases:
        plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, ct, spec.gqa_group)
        G = spec.gqa_group
        nslots = np.diff(plan.get("q_slot_off"))
        chunk_q, q_off = plan.get("chunk_q"), plan.get("chunk_q_off")
        rows = np.diff(q_off) * G
        slot_chunk = np.repeat(np.arange(len(rows)), np.diff(q_off))
        first = plan.get("q_slot")[plan.get("q_slot_off")[:-1].clip(max=max(len(slot_chunk) - 1, 0))] \
            if len(slot_chunk) else np.zeros(len(nslots), int)
        direct_q = (nslots == 1) & (rows[slot_chunk[first]] < 16) if len(slot_chunk) else nslots < 0
        np.testing.assert_array_equal(plan.get("merge_q"), np.nonzero(~direct_q)[0])
        for kind in ("fma", "fallback"):
            items = plan.get(kind + "_items").reshape(-1, 3)
            direct = plan.get(kind + "_direct")
            assert len(direct) == len(items)
            for (c, b, e), dw in zip(items, direct):
                want = 0
                for r in range((e - b) * G):
                    want |= int(direct_q[chunk_q[q_off[c] + b + r // G]]) << r
                assert int(dw) == want, (spec.name, ct, kind, c)
                seen_direct += bin(want).count("1")
        seen_merge += len(plan.get("merge_q"))
    # The tiny tree in one 256-token chunk: every query single-slot, no merge launch.
    tiny = deft.Plan(cases[0][0].parent, cases[0][0].node_len, cases[0][0].query_node, 256, 1)
    assert tiny.stats["num_merge_queries"] == 0
    # One chunk of >= 16 rows holding whole paths: single-slot, but merged by phase 2.
    fs = cases[-1][0]
    big = deft.Plan(fs.parent, fs.node_len, fs.query_node, 8192, fs.gqa_group)
    assert big.stats["num_merge_queries"] > 0
    assert seen_direct > 0 and seen_merge > 0


def test_step_calls_reject_bad_flags_and_state_before_any_cuda_call():
    spec, plan = _tiny_plan()
    lib = deft.load()
    P = ctypes.c_void_p
    fake = P(1 << 20)   # 16-byte aligned, never dereferenced

    def call_ex(flags, handle=plan.handle):
        return lib.deft_tree_attn_ex(fake, fake, fake, fake, fake, 4, 4, 4, 64, 16, 0.125, handle, fake, 0,
                                     fake, fake, 1 << 20, flags, None)
    assert call_ex(8) == -1                 # unknown flag bit
    assert call_ex(1 << 30) == -1
    assert call_ex(0) == -8                 # never uploaded
    assert call_ex(deft.STEP_NAIVE | deft.STEP_SEPARATE_MERGE) == -8
    tree_only = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1, naive=False)
    assert call_ex(deft.STEP_NAIVE, tree_only.handle) == -8
    code = ctypes.c_int32(7)
    assert lib.deft_step_status(plan.handle, None, ctypes.byref(code)) == -8
    assert code.value == 0
    assert lib.deft_step_status(None, None, ctypes.byref(code)) == -1
    assert lib.deft_step_status(plan.handle, None, None) == -1

    def call_host(q_host, out_host, lse_host):
        return lib.deft_tree_attn_host(q_host, fake, fake, fake, fake, fake, 4, 4, 4, 64, 16, 0.125, plan.handle,
                                       fake, 0, fake, fake, 1 << 20, out_host, lse_host, None)
    assert call_host(None, fake, fake) == -1      # host buffers are required
    assert call_host(fake, None, fake) == -1
    assert call_host(fake, fake, None) == -1
    assert call_host(fake, fake, fake) == -8      # never uploaded: nothing enqueued


def _extreme_shapes():
    """The planner's limits: a comb of 300 one-token children (packed chunks
    close at 256 segments), a 600-node chain of one-token nodes with a query
    at every node, 1000 queries on six nodes (16 mask words)."""
    comb = W.TreeSpec("comb300", np.array([-1] + [0] * 300, np.int32), np.ones(301, np.int32),
                      np.arange(1, 301, dtype=np.int32), 4, 1, 128)
    chain = W.TreeSpec("chain600", np.array([-1] + list(range(599)), np.int32), np.ones(600, np.int32),
                       np.arange(600, dtype=np.int32), 8, 2, 128)
    rng = np.random.default_rng(7)
    manyq = W.TreeSpec("manyq1000", np.array([-1, 0, 0, 1, 1, 2], np.int32),
                       np.array([300, 17, 0, 65, 1, 129], np.int32),
                       rng.integers(0, 6, 1000).astype(np.int32), 8, 2, 128)
    return [comb, chain, manyq]


@pytest.mark.parametrize("spec", _extreme_shapes(), ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [16, 256])
@pytest.mark.parametrize("G", [1, 16, 64])
def test_extreme_shapes_keep_the_plan_invariants(spec, ct, G):
    for tp in (False, True):
        plan = check_plan(spec, ct, G, tensor_pack=tp)
        so = plan.get("chunk_seg_off")
        assert (np.diff(so) <= 256).all()   # kMaxSegsPerChunk


def test_gqa_group_is_limited_to_one_tensor_core_item():
    """A query's whole GQA group shares one tensor-core item (at most 64
    rows): groups up to 64 plan, one query per item at 64; larger groups are
    rejected (they once made items of more rows than the kernel's widths
    and wrote past the planner's bucket tables)."""
    spec = W.chain_tree([40, 30, 5], q_heads=64, kv_heads=1, head_dim=128)
    for g in (1, 16, 32, 64):
        for tp in (False, True):
            p = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, g, tensor_pack=tp)
            items = p.get("mma_items").reshape(-1, 3)
            rows = (items[:, 2] - items[:, 1]) * g
            assert (rows <= 64).all() and (rows >= 16).all()
    p = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, 64)
    for g in (65, 100, 128, 129):
        with pytest.raises(deft.DeftError) as e:
            deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, g, tensor_pack=True)
        assert e.value.status == -1
        with pytest.raises(deft.DeftError):
            p.rebuild(spec.parent, spec.node_len, spec.query_node, 256, g)
    assert p.stats["gqa_group"] == 64   # a failed rebuild leaves the plan as it was


def test_host_step_checks_its_tensors_once():
    """HostStep (deft_tree_attn_host bound to its buffers) makes the same
    checks as the plain call, at construction; host tensors where device
    ones belong, or the reverse, are rejected before any library call."""
    torch = pytest.importorskip("torch")
    spec = W.tiny_tree()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, spec.gqa_group)
    Q, Hq, Hkv, d = spec.num_queries, spec.num_q_heads, spec.num_kv_heads, spec.head_dim
    q = torch.zeros((Q, Hq, d), dtype=torch.bfloat16)
    kv = torch.zeros((4, Hkv, 16, d), dtype=torch.bfloat16)
    idx = torch.zeros(8, dtype=torch.int32)

    class Bufs:
        out = torch.zeros((Q, Hq, d), dtype=torch.bfloat16)
        lse = torch.zeros((Q, Hq), dtype=torch.float32)
        workspace = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensors"):
        deft.HostStep(q.clone(), q, kv, kv, idx, idx, plan, Bufs, Bufs.out.clone(), Bufs.lse.clone())
    with pytest.raises(ValueError, match="CUDA tensors"):
        deft.deft_tree_attn_host(q.clone(), q, kv, kv, idx, idx, plan, Bufs, Bufs.out.clone(), Bufs.lse.clone())


def test_check_pages_accepts_a_layout_and_rejects_each_bad_table():
    spec = W.reasoning_tree(levels=3, len_lo=5, len_hi=40, num_queries=12, q_heads=4, kv_heads=2)
    lay = W.paged_layout(spec)
    npo, pid, pages = lay.node_page_off, lay.page_id, int(lay.page_id.max()) + 1
    ln = spec.node_len
    assert deft.deft_check_pages(ln, npo, pid, pages) == 0
    assert deft.deft_check_pages(ln, npo, pid, pages + 5) == 0
    n = int(np.argmax(ln))                   # a node with tokens
    bad = pid.copy()
    bad[npo[n]] = pages                      # a page past the pool
    assert deft.deft_check_pages(ln, npo, bad, pages) == -3
    bad[npo[n]] = -1                         # a negative page id
    assert deft.deft_check_pages(ln, npo, bad, pages) == -3
    off = npo.copy()
    off[n] = -1                              # page-table offset before the table
    assert deft.deft_check_pages(ln, off, pid, pages) == -3
    off[n] = len(pid) - 1                    # the node's pages run past the table's end
    assert ln[n] > 16
    assert deft.deft_check_pages(ln, off, pid, pages) == -3
    last = int(np.argmax(npo[:-1]))          # the node whose pages end the table
    longer = ln.copy()
    longer[last] = (len(pid) - npo[last]) * 16 + 1   # one token more than its pages hold
    assert deft.deft_check_pages(longer, npo, pid, pages) == -3
    assert deft.deft_check_pages(ln, npo, pid, 0) == -1
    neg = ln.copy()
    neg[0] = -1
    assert deft.deft_check_pages(neg, npo, pid, pages) == -1
    # Zero-length nodes need no page.
    z = ln.copy()
    z[n] = 0
    off2 = npo.copy()
    off2[n] = -7
    assert deft.deft_check_pages(z, off2, pid, pages) == 0


@pytest.mark.parametrize("spec", RANDOM[:20], ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [1, 16, 100, 512])
def test_tensor_packed_plan_random_trees(spec, ct):
    """DEFT_PLAN_TENSOR_PACK keeps every (query, node, token) triple in
    exactly one chunk that lists the query, with exact segment masks."""
    check_plan(spec, ct, spec.gqa_group, tensor_pack=True)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5, 6, 7])
def test_tensor_packed_plan_workload_shapes(cfg):
    spec = W.config(cfg)
    plan = check_plan(spec, 256, spec.gqa_group, tensor_pack=True) if cfg != 5 else \
        deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group, tensor_pack=True)
    st = plan.stats
    plain = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group)
    assert st["unique_tokens"] == plain.stats["unique_tokens"] == st["planned_tokens"]
    # Segments of 4 to 15 rows and more than a quarter chunk no longer run
    # on CUDA cores, but for a remainder that could not reach 16 rows.
    G = spec.gqa_group
    q_off = plan.get("chunk_q_off")
    fma_chunks = set(plan.get("fma_items").reshape(-1, 3)[:, 0].tolist())
    seg_off, seg_l = plan.get("chunk_seg_off"), plan.get("seg_tok_len")
    rows = np.diff(q_off) * G
    left = sum(int(seg_l[seg_off[c]:seg_off[c + 1]].sum()) for c in fma_chunks
               if rows[c] >= 4 and (seg_l[seg_off[c]:seg_off[c + 1]] > 64).any())
    assert left <= 0.02 * st["unique_tokens"] or cfg == 1


def test_tensor_pack_rows_and_pieces():
    """GQA 4, one query per sequence (4 rows): four sequences per chunk, a
    256-token piece of each, so every chunk reaches 16 rows on the tensor
    path; one-row segments are left to the CUDA cores."""
    spec = W.imbalance_tree(leaves=12, control=True, control_len=1024, q_heads=8, kv_heads=2)
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group, tensor_pack=True)
    q_off, seg_off = plan.get("chunk_q_off"), plan.get("chunk_seg_off")
    seg_l = plan.get("seg_tok_len")
    assert plan.stats["num_fma_items"] == 0
    assert plan.stats["num_chunks"] == 3 * 4
    for c in range(len(q_off) - 1):
        assert (q_off[c + 1] - q_off[c]) * spec.gqa_group == 16
        assert (seg_l[seg_off[c]:seg_off[c + 1]] == 256).all()
    few = W.few_shot_tree(prefix=600, branches=32, branch_len=256, heads=4, head_dim=128)
    p1 = deft.Plan(few.parent, few.node_len, few.query_node, 256, 1, tensor_pack=True)
    p0 = deft.Plan(few.parent, few.node_len, few.query_node, 256, 1)
    for name in ("chunk_seg_off", "seg_node", "seg_tok_len", "fma_items", "mma_items"):
        np.testing.assert_array_equal(p1.get(name), p0.get(name))
