"""Incremental plan updates and the KV page pool (no GPU).

deft_plan_update (DeFT Guide, "Production Engineering and Kernel Deployment
Best Practices": the tree grows and is pruned between decode steps) must
give, array for array, the plan a fresh build of the new tree gives; the
page pool ("Tree Pruning Memory Management") must hand out and take back
pages by reference count."""
import random

import numpy as np
import pytest

import workloads as W

deft = pytest.importorskip("shared_prefix_kv_deft_gb300")
from shared_prefix_kv_deft_gb300 import build as deft_build  # noqa: E402

ARRAYS = ["chunk_seg_off", "chunk_q_off", "chunk_q", "seg_node", "seg_tok_begin", "seg_tok_len", "seg_mask",
          "chunk_mask", "q_slot_off", "q_slot", "node_cover", "node_order", "fma_items", "mma_items",
          "fallback_items", "naive_chunk_seg_off", "naive_chunk_q", "naive_seg_node", "naive_seg_tok_begin",
          "naive_seg_tok_len", "naive_q_slot_off", "naive_q_slot", "fma_direct", "fallback_direct", "merge_q"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    deft_build.build()
    deft.load()


def assert_same_plan(a, b, what=""):
    sa, sb = a.stats, b.stats
    assert sa == sb, what
    for name in ARRAYS:
        np.testing.assert_array_equal(a.get(name), b.get(name), err_msg=f"{what}: {name}")


def _grow_and_prune(spec, rng, len_, steps):
    """A decode-like sequence of new length vectors: a few nodes gain
    tokens, now and then a leaf subtree is pruned to length 0."""
    N = spec.num_nodes
    children = [[] for _ in range(N)]
    for n, p in enumerate(spec.parent):
        if p >= 0:
            children[p].append(n)
    for _ in range(steps):
        ln = len_.copy()
        for n in rng.sample(range(N), k=min(N, rng.randint(1, 4))):
            ln[n] += rng.randint(1, 40)
        if rng.random() < 0.3:
            stack = [rng.randrange(N)]
            while stack:
                n = stack.pop()
                ln[n] = 0
                stack.extend(children[n])
        len_ = ln
        yield ln


SHAPES = [W.random_tree(s, max_nodes=40, max_len=300, max_queries=90) for s in range(12)]
SHAPES += [W.config(c) for c in (1, 2, 4)]
SHAPES += [W.positions_tree(s, max_nodes=14, max_len=120, max_queries=24, q_heads=8, kv_heads=2,
                            head_dim=128) for s in range(3)]


@pytest.mark.parametrize("spec", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("ct,tp,naive", [(16, False, True), (256, False, False), (100, True, True),
                                         (256, True, False)])
def test_update_equals_a_fresh_plan(spec, ct, tp, naive):
    rng = random.Random(ct + spec.num_nodes)
    pos = spec.query_pos
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, ct, spec.gqa_group, query_pos=pos,
                     naive=naive, tensor_pack=tp)
    ln0 = spec.node_len.astype(np.int32)
    if pos is not None:
        # Positioned queries keep their token: their nodes only grow.
        keep = set(int(spec.query_node[q]) for q in range(spec.num_queries) if pos[q] >= 0)
    for k, ln in enumerate(_grow_and_prune(spec, rng, ln0, 6)):
        if pos is not None:
            ln = np.maximum(ln, np.where(np.isin(np.arange(spec.num_nodes), list(keep)), ln0, 0)).astype(np.int32)
        plan.update(ln)
        fresh = deft.Plan(spec.parent, ln, spec.query_node, ct, spec.gqa_group, query_pos=pos, naive=naive,
                          tensor_pack=tp)
        assert_same_plan(plan, fresh, f"step {k}")
        ln0 = ln


def test_update_without_a_change_keeps_the_upload_state_and_rejects_bad_lengths():
    spec = W.tiny_tree()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1)
    plan.update(spec.node_len)                       # no change: fine, nothing to do
    lib = deft.load()
    bad = spec.node_len.astype(np.int32).copy()
    bad[2] = -1
    assert lib.deft_plan_update(plan.handle, bad.ctypes.data, len(bad)) == -1
    assert lib.deft_plan_update(plan.handle, bad.ctypes.data, len(bad) - 1) == -1
    assert lib.deft_plan_update(None, bad.ctypes.data, len(bad)) == -1
    fresh = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1)
    assert_same_plan(plan, fresh, "after refused updates")
    # A positioned query beyond its node's new length.
    pspec = W.positions_tree(1, max_nodes=8, max_len=60, max_queries=10)
    pp = deft.Plan(pspec.parent, pspec.node_len, pspec.query_node, 32, pspec.gqa_group, query_pos=pspec.query_pos)
    q = int(np.argmax(pspec.query_pos))
    if pspec.query_pos[q] >= 0:
        short = pspec.node_len.astype(np.int32).copy()
        short[pspec.query_node[q]] = pspec.query_pos[q]
        assert lib.deft_plan_update(pp.handle, short.ctypes.data, len(short)) == -3


def test_update_resumes_late_for_a_late_change():
    """Growing only the last branch of the few-shot tree re-emits from that
    branch on: the leading chunks are the old plan's (and the result equals a
    fresh plan)."""
    spec = W.config(2)
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, 1, naive=False)
    old = plan.get("chunk_seg_off").copy()
    ln = spec.node_len.astype(np.int32).copy()
    ln[-1] += 1
    plan.update(ln)
    fresh = deft.Plan(spec.parent, ln, spec.query_node, 256, 1, naive=False)
    assert_same_plan(plan, fresh)
    new = plan.get("chunk_seg_off")
    np.testing.assert_array_equal(new[: len(old) - 1], old[:-1])


# ---------------------------------------------------------------------------
# Page pool
# ---------------------------------------------------------------------------

def test_page_pool_alloc_retain_release():
    pool = deft.PagePool(10)
    assert pool.free_count == 10
    a = pool.alloc(4)
    assert a.tolist() == [0, 1, 2, 3] and pool.free_count == 6
    assert all(pool.refcount(p) == 1 for p in a)
    with pytest.raises(deft.DeftError):
        pool.alloc(7)                                  # not enough free pages: nothing taken
    assert pool.free_count == 6
    pool.retain([1, 1, 2])                             # page 1 shared twice more, page 2 once
    assert [pool.refcount(p) for p in range(4)] == [1, 3, 2, 1]
    pool.release([0, 1, 2, 3])
    assert [pool.refcount(p) for p in range(4)] == [0, 2, 1, 0] and pool.free_count == 8
    with pytest.raises(deft.DeftError):
        pool.release([2, 2])                           # more releases than references: nothing released
    assert pool.refcount(2) == 1
    with pytest.raises(deft.DeftError):
        pool.release([0])                              # a free page
    with pytest.raises(deft.DeftError):
        pool.retain([10])                              # out of range
    pool.release([1, 1, 2])
    assert pool.free_count == 10 and pool.refcount(99) == -1
    b = pool.alloc(10)
    assert sorted(b.tolist()) == list(range(10)) and pool.free_count == 0


def test_pruned_branches_give_their_pages_back():
    """A speculative step: a draft tree gets pages from the pool, the rejected
    branches are pruned (length 0, pages released), the plan is updated, and
    the pool's free count is back where the kept nodes leave it."""
    spec = W.speculative_forest(requests=1, prefix=300, tree_nodes=32, heads=4)
    N = spec.num_nodes
    pool = deft.PagePool(1000)
    pages = [pool.alloc(-(-int(L) // 16)) for L in spec.node_len]
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1)
    children = [[] for _ in range(N)]
    for n, p in enumerate(spec.parent):
        if p >= 0:
            children[p].append(n)
    # Reject the subtree of the root's first child that has children.
    victim = next(c for c in children[0] if children[c])
    pruned, stack = [], [victim]
    while stack:
        n = stack.pop()
        pruned.append(n)
        stack.extend(children[n])
    before = pool.free_count
    for n in pruned:
        pool.release(pages[n])
    freed = sum(len(pages[n]) for n in pruned)
    assert pool.free_count == before + freed
    ln = spec.node_len.astype(np.int32).copy()
    ln[pruned] = 0
    plan.update(ln)
    fresh = deft.Plan(spec.parent, ln, spec.query_node, 64, 1)
    assert_same_plan(plan, fresh)
    assert plan.stats["unique_tokens"] < deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1).stats[
        "unique_tokens"]
