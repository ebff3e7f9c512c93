"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (stated for bf16 inputs, fp32 accumulation): max-abs error 1e-2
on outputs, 1e-3 on lse; bit-exact integer plan (checked without a GPU in
test_plan.py).  Unused KV slots are NaN-poisoned, so a kernel that reads a
slot past a node's last token fails here."""
import ctypes
import math

import numpy as np
import pytest

import oracle
import workloads as W
from helpers import dense_inputs, run_oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def deft():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import shared_prefix_kv_deft_gb300 as d
    from shared_prefix_kv_deft_gb300 import build
    build.build()
    d.load()
    return d


def bits_to_cuda(b: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()


class Case:
    """Device copies of one input set plus its plan."""

    def __init__(self, deft, inp, chunk_target, tensor_pack=False):
        self.inp, self.spec = inp, inp.spec
        self.q = bits_to_cuda(inp.q_bits)
        self.k = bits_to_cuda(inp.k_pages)
        self.v = bits_to_cuda(inp.v_pages)
        self.npo = torch.from_numpy(inp.layout.node_page_off).cuda()
        self.pid = torch.from_numpy(inp.layout.page_id).cuda()
        s = self.spec
        self.plan = deft.Plan(s.parent, s.node_len, s.query_node, chunk_target, s.gqa_group,
                              query_pos=s.query_pos, tensor_pack=tensor_pack)
        self.plan.upload()
        self.deft = deft

    def run(self, naive=False, out_dtype=0, flags=0):
        """One step; flags (STEP_*) go through deft_tree_attn_ex."""
        if flags:
            flags |= self.deft.STEP_NAIVE if naive else 0
            out, lse = self.deft.deft_tree_attn(self.q, self.k, self.v, self.npo, self.pid, self.plan,
                                                out_dtype=out_dtype, flags=flags)
        else:
            fn = self.deft.deft_naive_attn if naive else self.deft.deft_tree_attn
            out, lse = fn(self.q, self.k, self.v, self.npo, self.pid, self.plan, out_dtype=out_dtype)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_parity(out, lse, ref, ref_lse, what=""):
    assert np.isfinite(out).all(), f"{what}: non-finite output (poisoned slot read?)"
    err = np.abs(out - ref).max() if out.size else 0.0
    assert err <= OUT_TOL, f"{what}: out max-abs error {err}"
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref_lse), err_msg=what)
    fin = np.isfinite(ref_lse)
    lerr = np.abs(lse[fin] - ref_lse[fin]).max() if fin.any() else 0.0
    assert lerr <= LSE_TOL, f"{what}: lse max-abs error {lerr}"


def small_shapes():
    shapes = [W.tiny_tree()]
    shapes += [W.random_tree(s, max_nodes=16, max_len=90, max_queries=12) for s in range(16)]
    shapes += [W.random_tree(100 + s, max_nodes=20, max_len=200, max_queries=40, q_heads=8,
                             kv_heads=2, head_dim=128) for s in range(8)]
    # MHA with many queries sharing the root: chunks of >= 16 rows.
    shapes += [W.random_tree(200 + s, max_nodes=10, max_len=300, max_queries=60, q_heads=2,
                             kv_heads=2, head_dim=128, forest=False) for s in range(4)]
    shapes += [
        W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128),
        W.speculative_forest(requests=2, prefix=300, tree_nodes=64, heads=4),
        W.reasoning_tree(levels=3, len_lo=20, len_hi=90, num_queries=24, q_heads=8, kv_heads=2),
        W.imbalance_tree(prefix=700, leaves=24, lo=5, hi=400, q_heads=8, kv_heads=2),
        W.imbalance_tree(leaves=12, control=True, control_len=150, q_heads=8, kv_heads=2),
        W.chain_tree([5, 70, 1, 130], q_heads=4, kv_heads=4, head_dim=128),
    ]
    return shapes


SMALL = small_shapes()


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [16, 100, 256])
def test_tree_and_naive_match_oracle(deft, spec, ct):
    """Both partitions against the oracle; merging in phase 1 (the default)
    and in a separate launch give the same values (same partials, same merge
    arithmetic), and no kernel reports a failed wait."""
    inp = dense_inputs(spec, seed=ct + spec.num_nodes)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct)
    for naive in (False, True):
        what = f"{'naive' if naive else 'tree'} ct={ct}"
        out, lse = case.run(naive=naive)
        assert_parity(out, lse, ref, ref_lse, what)
        out_s, lse_s = case.run(naive=naive, flags=deft.STEP_SEPARATE_MERGE)
        np.testing.assert_array_equal(out_s, out, err_msg=what + " separate merge")
        np.testing.assert_array_equal(lse_s, lse, err_msg=what + " separate merge")
    assert case.plan.step_status() == 0


DIRECT_CASES = [
    # every query's path is one CUDA-core chunk: no merge launch at all
    ("all", W.imbalance_tree(leaves=12, control=True, control_len=150, q_heads=8, kv_heads=2), 256),
    # a mix of single-chunk paths and paths through shared nodes
    ("some", W.random_tree(1, max_nodes=16, max_len=90, max_queries=12), 256),
    ("some_gqa", W.random_tree(116, max_nodes=20, max_len=200, max_queries=40, q_heads=8, kv_heads=2,
                               head_dim=128), 64),
    # every path crosses the shared prefix: every query merged
    ("none", W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128), 256),
]


@pytest.mark.parametrize("which,spec,ct", DIRECT_CASES, ids=[c[0] for c in DIRECT_CASES])
def test_direct_rows_for_all_some_and_no_queries(deft, which, spec, ct):
    """Queries whose whole path is one CUDA-core chunk get their rows from
    phase 1 (the merge of one partial is the identity); the merge launch
    takes the others and is left out when there are none.  Against the
    oracle, and bitwise equal to merging every query in phase 2."""
    inp = dense_inputs(spec, seed=7 + ct)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct)
    merged = case.plan.stats["num_merge_queries"]
    Q = spec.num_queries
    assert {"all": merged == 0, "some": 0 < merged < Q, "some_gqa": 0 < merged < Q,
            "none": merged == Q}[which], (which, merged, Q)
    deft.trace_read()
    deft.trace_enable(True)
    out, lse = case.run()
    deft.trace_enable(False)
    launches = [r["kernel"] for r in deft.trace_read()]
    assert launches.count("phase2_merge") == (0 if merged == 0 else 1), launches
    assert_parity(out, lse, ref, ref_lse, f"direct rows ({which})")
    out_s, lse_s = case.run(flags=deft.STEP_SEPARATE_MERGE)
    np.testing.assert_array_equal(out_s, out)
    np.testing.assert_array_equal(lse_s, lse)
    assert case.plan.step_status() == 0


@pytest.mark.parametrize("spec", [W.tiny_tree(), W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4,
                                                                  head_dim=128)], ids=lambda s: s.name)
def test_host_buffer_step_equals_the_device_step(deft, spec):
    """deft_tree_attn_host (q in, out and lse back, all on the stream) gives
    the device step's values bit for bit, in both output dtypes."""
    inp = dense_inputs(spec, seed=11)
    case = Case(deft, inp, 64)
    for odt in (0, 1):
        out_d, lse_d = case.run(out_dtype=odt)
        bufs = deft.alloc_buffers(case.plan, spec.num_queries, spec.num_q_heads, spec.head_dim, out_dtype=odt)
        q_host = case.q.cpu().pin_memory()
        q_dev = torch.empty_like(case.q)
        out_h = torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory()
        lse_h = torch.empty(bufs.lse.shape, dtype=bufs.lse.dtype).pin_memory()
        deft.deft_tree_attn_host(q_host, q_dev, case.k, case.v, case.npo, case.pid, case.plan, bufs, out_h, lse_h)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out_h.float().numpy().astype(np.float64), out_d)
        np.testing.assert_array_equal(lse_h.numpy().astype(np.float64), lse_d)
        torch.testing.assert_close(q_dev, case.q, rtol=0, atol=0)
        # The same call bound once (HostStep), twice, into cleared buffers.
        step = deft.HostStep(q_host, q_dev, case.k, case.v, case.npo, case.pid, case.plan, bufs, out_h, lse_h)
        for _ in range(2):
            out_h.zero_()
            lse_h.zero_()
            q_dev.zero_()
            step()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(out_h.float().numpy().astype(np.float64), out_d)
            np.testing.assert_array_equal(lse_h.numpy().astype(np.float64), lse_d)
    assert case.plan.step_status() == 0


TENSOR_PACK_SHAPES = [s for s in SMALL if s.head_dim == 128]


@pytest.mark.parametrize("spec", TENSOR_PACK_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [16, 256])
def test_tensor_packed_plans_match_oracle(deft, spec, ct):
    """Plans built with DEFT_PLAN_TENSOR_PACK (thin segments laid side by
    side into chunks of >= 16 rows) against the oracle, on both kernel
    paths."""
    inp = dense_inputs(spec, seed=ct + 17 + spec.num_nodes)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct, tensor_pack=True)
    out, lse = case.run()
    assert_parity(out, lse, ref, ref_lse, f"tensor-packed ct={ct}")
    out, lse = case.run(flags=deft.STEP_CUDA_CORES)
    assert_parity(out, lse, ref, ref_lse, f"tensor-packed on CUDA cores ct={ct}")
    assert case.plan.step_status() == 0


EXTREME = [W.tiny_tree(),
           W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128),
           W.reasoning_tree(levels=3, len_lo=20, len_hi=90, num_queries=24, q_heads=8, kv_heads=2),
           W.random_tree(7, max_nodes=16, max_len=90, max_queries=12),
           W.chain_tree([5, 70, 1, 130], q_heads=4, kv_heads=4, head_dim=128)]


@pytest.mark.parametrize("spec", EXTREME, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [1, 8192])
def test_extreme_chunk_targets_match_oracle(deft, spec, ct):
    """chunk_target at its bounds: 1 (every node its own run of pieces) and
    8192 (the largest chunks the plan allows, page lists at their limit)."""
    inp = dense_inputs(spec, seed=ct + 3)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct)
    out, lse = case.run()
    assert_parity(out, lse, ref, ref_lse, f"tree ct={ct}")
    out, lse = case.run(naive=True)
    assert_parity(out, lse, ref, ref_lse, f"naive ct={ct}")


def test_fp32_output(deft):
    spec = W.reasoning_tree(levels=3, len_lo=20, len_hi=90, num_queries=24, q_heads=8, kv_heads=2)
    inp = dense_inputs(spec, seed=5)
    ref, ref_lse = run_oracle(inp)
    out, lse = Case(deft, inp, 64).run(out_dtype=1)
    assert_parity(out, lse, ref, ref_lse, "fp32 out")
    assert np.abs(out - ref).max() < 2e-3


def test_empty_paths_give_zero_and_minus_inf(deft):
    spec = W.TreeSpec("empty", np.array([-1, 0, 0, -1], np.int32), np.array([0, 0, 37, 0], np.int32),
                      np.array([0, 1, 2, 3, 2], np.int32), 4, 2, 128)
    inp = dense_inputs(spec, seed=1)
    ref, ref_lse = run_oracle(inp)
    for naive in (False, True):
        out, lse = Case(deft, inp, 16).run(naive=naive)
        assert np.all(out[[0, 1, 3]] == 0) and np.all(np.isneginf(lse[[0, 1, 3]]))
        assert_parity(out, lse, ref, ref_lse, "empty paths")


def test_results_are_bitwise_repeatable(deft):
    spec = W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128)
    case = Case(deft, dense_inputs(spec, seed=3), 64)
    a = case.run()
    b = case.run()
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_step_captured_in_a_cuda_graph(deft):
    """The step is graph-capturable: a captured step, replayed several times
    (the work queues reset themselves between launches), gives the eager
    step's results bit for bit, on a tree with both kernel families."""
    spec = W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128)
    case = Case(deft, dense_inputs(spec, seed=5), 64)
    ref_out, ref_lse = case.run()
    s = case.spec
    bufs = deft.alloc_buffers(case.plan, s.num_queries, s.num_q_heads, s.head_dim)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        deft.deft_tree_attn(case.q, case.k, case.v, case.npo, case.pid, case.plan, bufs=bufs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        deft.deft_tree_attn(case.q, case.k, case.v, case.npo, case.pid, case.plan, bufs=bufs)
    for _ in range(3):
        bufs.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bufs.out.float().cpu().numpy().astype(np.float64), ref_out)
        np.testing.assert_array_equal(bufs.lse.cpu().numpy().astype(np.float64), ref_lse)


def test_abi_rejects_bad_calls(deft):
    spec = W.tiny_tree()
    case = Case(deft, dense_inputs(spec, seed=2), 64)
    lib = deft.load()
    Q, Hq, d = case.q.shape
    out = torch.empty((Q, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((Q, Hq), dtype=torch.float32, device="cuda")
    ws_bytes = case.plan.workspace_bytes(Hq, d)
    ws = torch.zeros(ws_bytes + 512, dtype=torch.uint8, device="cuda")
    P = ctypes.c_void_p

    def call(plan=case.plan.handle, hq=Hq, hkv=4, hd=d, ps=16, wsp=ws.data_ptr(), wsb=ws_bytes,
             scale=0.125, odt=0, fn=lib.deft_tree_attn):
        return fn(P(case.q.data_ptr()), P(case.k.data_ptr()), P(case.v.data_ptr()),
                                  P(case.npo.data_ptr()), P(case.pid.data_ptr()), case.k.shape[0],
                                  hq, hkv, hd, ps, scale, plan, P(out.data_ptr()), odt,
                                  P(lse.data_ptr()), P(wsp), wsb,
                                  P(torch.cuda.current_stream().cuda_stream))
    assert call() == 0
    assert call(hkv=2) == -8           # GQA group differs from the plan's
    assert call(hkv=3) == -1           # heads not a multiple
    assert call(hd=96) == -5           # head_dim not compiled
    assert call(ps=8) == -5            # page size
    assert call(wsb=ws_bytes - 1) == -7
    assert call(wsp=ws.data_ptr() + 16) == -7
    assert call(scale=0.0) == -1
    assert call(odt=7) == -1
    unuploaded = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1)
    assert call(plan=unuploaded.handle) == -8
    tree_only = deft.Plan(spec.parent, spec.node_len, spec.query_node, 64, 1, naive=False)
    tree_only.upload()
    assert call(plan=tree_only.handle) == 0
    assert call(plan=tree_only.handle, fn=lib.deft_naive_attn) == -8   # no naive partition
    assert call(fn=lib.deft_naive_attn) == 0

    def call_ex(flags, plan=case.plan.handle):
        return lib.deft_tree_attn_ex(P(case.q.data_ptr()), P(case.k.data_ptr()), P(case.v.data_ptr()),
                                     P(case.npo.data_ptr()), P(case.pid.data_ptr()), case.k.shape[0],
                                     Hq, 4, d, 16, 0.125, plan, P(out.data_ptr()), 0,
                                     P(lse.data_ptr()), P(ws.data_ptr()), ws_bytes, flags,
                                     P(torch.cuda.current_stream().cuda_stream))
    assert call_ex(0) == 0
    assert call_ex(deft.STEP_NAIVE | deft.STEP_SEPARATE_MERGE | deft.STEP_CUDA_CORES) == 0
    assert call_ex(8) == -1             # unknown flag bit
    assert call_ex(deft.STEP_NAIVE, plan=tree_only.handle) == -8
    torch.cuda.synchronize()
    assert case.plan.step_status() == 0
    code = ctypes.c_int32(5)
    assert lib.deft_step_status(unuploaded.handle, None, ctypes.byref(code)) == -8
    assert lib.deft_step_status(case.plan.handle, None, None) == -1


@pytest.mark.parametrize("cfg", [2, 7])
def test_tree_only_plan_gives_the_same_step(deft, cfg):
    """A plan without the naive partition runs the tree step bit for bit as
    the full plan does (same partition, same launches)."""
    spec = W.config(cfg)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cuda")
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    res = []
    for naive in (True, False):
        plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group,
                         query_pos=spec.query_pos, naive=naive)
        plan.upload()
        out, lse = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)
        torch.cuda.synchronize()
        res.append((out.float().cpu().numpy(), lse.cpu().numpy()))
    np.testing.assert_array_equal(res[0][0], res[1][0])
    np.testing.assert_array_equal(res[0][1], res[1][1])


# ---------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times, every
# query and head against the oracle.
# ---------------------------------------------------------------------------

FULL = {2: 256, 3: 256, 4: 256, 5: 256, 6: 256, 1: 64, 7: 256}
# (config, tensor-packed plan): the plain plans, and the packed ones the
# benchmark runs at head_dim 128.
FULL_CASES = [(c, False) for c in sorted(FULL)] + [(c, True) for c in sorted(FULL) if c != 1]


@pytest.mark.parametrize("cfg,tp", FULL_CASES)
def test_full_size_workloads_every_query(deft, cfg, tp):
    spec = W.config(cfg)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cuda")
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, FULL[cfg], spec.gqa_group,
                     query_pos=spec.query_pos, tensor_pack=tp)
    plan.upload()
    out, lse = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)
    nout, nlse = deft.deft_naive_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)
    torch.cuda.synchronize()
    assert plan.step_status() == 0
    # Every query (the oracle takes a few seconds on the largest workload).
    sample = np.arange(spec.num_queries)
    ref, ref_lse = oracle.tree_attn(W.bf16_bits(t.q), W.bf16_bits(t.k_pages), W.bf16_bits(t.v_pages),
                                    layout.node_page_off, layout.page_id, layout.page_size,
                                    spec.parent, spec.node_len, spec.query_node, spec.num_q_heads,
                                    spec.num_kv_heads, spec.head_dim, 1.0 / math.sqrt(spec.head_dim),
                                    query_subset=sample, query_pos=spec.query_pos)
    for o, l, what in ((out, lse, "tree"), (nout, nlse, "naive")):
        o = o.float().cpu().numpy().astype(np.float64)
        l = l.cpu().numpy().astype(np.float64)
        assert np.isfinite(o).all() and np.isfinite(l).all(), what
        assert_parity(o[sample], l[sample], ref, ref_lse, f"config {cfg} {what}")


MMA_SHAPES = [
    W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128),
    W.speculative_forest(requests=2, prefix=300, tree_nodes=64, heads=4),
    W.random_tree(203, max_nodes=10, max_len=300, max_queries=60, q_heads=2, kv_heads=2,
                  head_dim=128, forest=False),
    W.reasoning_tree(levels=3, len_lo=20, len_hi=90, num_queries=40, q_heads=8, kv_heads=2),
    W.few_shot_tree(prefix=1000, branches=140, branch_len=20, heads=2, head_dim=128),
]


@pytest.mark.parametrize("spec", MMA_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [64, 256])
def test_tensor_core_and_cuda_core_paths_agree_with_oracle(deft, spec, ct):
    inp = dense_inputs(spec, seed=11 + ct)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct)
    assert case.plan.stats["num_mma_items"] > 0, "shape has no >= 16-row chunk"
    deft.trace_read()
    deft.trace_enable(True)
    out, lse = case.run()
    deft.trace_enable(False)
    kinds = {r["kernel"] for r in deft.trace_read()}
    assert "phase1_mma" in kinds
    assert_parity(out, lse, ref, ref_lse, "tcgen05 path")
    out2, lse2 = case.run(flags=deft.STEP_CUDA_CORES)
    assert_parity(out2, lse2, ref, ref_lse, "CUDA-core fallback")
    out3, lse3 = case.run(flags=deft.STEP_CUDA_CORES | deft.STEP_SEPARATE_MERGE)
    assert_parity(out3, lse3, ref, ref_lse, "CUDA-core fallback, separate merge")
    assert case.plan.step_status() == 0


@pytest.mark.parametrize("spec", MMA_SHAPES[:2], ids=lambda s: s.name)
@pytest.mark.parametrize("ct,tp", [(64, False), (256, False), (256, True)])
def test_growing_logits_take_the_rescale_path(deft, spec, ct, tp):
    """Keys scaled up along each node: a chunk's later tiles hold logits far
    above the maxima of its first tile, so the kernels' rescale of the
    running output and sums (online softmax) is exercised, not just the
    common path; both the tensor-core and CUDA-core steps against the
    oracle.  The softmax is then sharply peaked, so an output is close to a
    single value row (|out| up to ~5): fp32 output, since rounding such a
    value to bf16 alone can be 1.6e-2 off."""
    inp = dense_inputs(spec, seed=5, k_ramp=0.1)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct, tensor_pack=tp)
    assert case.plan.stats["num_mma_items"] > 0
    out, lse = case.run(out_dtype=1)
    assert_parity(out, lse, ref, ref_lse, "tcgen05 path, growing logits")
    out2, lse2 = case.run(flags=deft.STEP_CUDA_CORES, out_dtype=1)
    assert_parity(out2, lse2, ref, ref_lse, "CUDA-core path, growing logits")
    assert case.plan.step_status() == 0


# Large GQA groups: a query alone makes G rows (8 .. 64), so one query can
# fill a tensor-core item (G = 32, 64) and CUDA-core items hold one or two
# queries (G = 8, 16).
GQA_SHAPES = [
    W.reasoning_tree(levels=3, len_lo=20, len_hi=150, num_queries=nq, q_heads=q, kv_heads=kv, seed=g)
    for g, q, kv, nq in ((8, 16, 2, 12), (16, 32, 2, 9), (32, 32, 1, 7), (64, 64, 1, 5))
]


@pytest.mark.parametrize("spec", GQA_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("ct,tp", [(64, False), (256, False), (256, True)])
def test_large_gqa_groups_match_oracle(deft, spec, ct, tp):
    inp = dense_inputs(spec, seed=7 + ct)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct, tensor_pack=tp)
    out, lse = case.run()
    assert_parity(out, lse, ref, ref_lse, f"G={spec.gqa_group}")
    out_s, lse_s = case.run(flags=deft.STEP_SEPARATE_MERGE)
    np.testing.assert_array_equal(out_s, out)
    np.testing.assert_array_equal(lse_s, lse)
    if spec.gqa_group <= 16:
        out2, lse2 = case.run(flags=deft.STEP_CUDA_CORES)
        assert_parity(out2, lse2, ref, ref_lse, f"G={spec.gqa_group}, CUDA cores")
    assert case.plan.step_status() == 0


POSITION_SHAPES = [W.positions_tree(s, max_nodes=14, max_len=120, max_queries=24, q_heads=8,
                                    kv_heads=2, head_dim=128) for s in range(6)]
POSITION_SHAPES += [W.positions_tree(50 + s, max_nodes=10, max_len=60, max_queries=12)
                    for s in range(4)]
POSITION_SHAPES += [
    # node prefill: a query at every token of a 96-token node under a
    # 200-token root (GQA 4: the early pieces of the node have >= 16 rows)
    W.causal_node_tree(96, q_heads=8, kv_heads=2, head_dim=128, parent_len=200),
    W.causal_node_tree(40, q_heads=4, kv_heads=4, head_dim=64),
]


@pytest.mark.parametrize("spec", POSITION_SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("ct", [16, 128])
def test_queries_at_token_positions_match_oracle(deft, spec, ct):
    """Tree verification / node prefill: queries at token positions of
    multi-token nodes, tree and naive forms, against the fp64 oracle."""
    inp = dense_inputs(spec, seed=11)
    ref, ref_lse = run_oracle(inp)
    case = Case(deft, inp, ct)
    for naive in (False, True):
        out, lse = case.run(naive=naive)
        assert_parity(out, lse, ref, ref_lse, f"{spec.name} ct={ct} naive={naive}")


@pytest.mark.parametrize("cfg", [2, 4])
def test_kv_head_shards_give_the_same_step(deft, cfg):
    """The step splits by KV head with no exchange: a device holding half the
    KV heads (and their query heads) computes exactly the full step's rows
    for those heads, bit for bit (same units, same merge order)."""
    spec = W.config(cfg)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cuda")
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group, naive=False)
    plan.upload()
    out, lse = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)
    torch.cuda.synchronize()
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    Hkv, G = spec.num_kv_heads, spec.gqa_group
    for shard in range(2):
        kv = slice(shard * Hkv // 2, (shard + 1) * Hkv // 2)
        qh = slice(kv.start * G, kv.stop * G)
        o_s, l_s = deft.deft_tree_attn(t.q[:, qh].contiguous(), t.k_pages[:, kv].contiguous(),
                                       t.v_pages[:, kv].contiguous(), npo, pid, plan)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(o_s.float().cpu().numpy(), out[:, qh])
        np.testing.assert_array_equal(l_s.cpu().numpy(), lse[:, qh])


def test_rebuilt_plan_runs_like_a_fresh_one(deft):
    """A decode loop's plan reuse: rebuild into the same plan (smaller tree,
    then a larger one that grows the device copy), upload, step: bit for bit
    the step of a fresh plan; a rebuilt plan not yet uploaded is refused."""
    lib = deft.load()
    P = ctypes.c_void_p
    big, small = W.config(2), W.config(1)
    plan = deft.Plan(small.parent, small.node_len, small.query_node, 64, small.gqa_group, naive=False)
    plan.upload()
    for spec, ct in ((big, 256), (small, 64), (big, 128)):
        layout = W.paged_layout(spec)
        t = W.make_tensors(spec, layout, device="cuda")
        npo = torch.from_numpy(layout.node_page_off).cuda()
        pid = torch.from_numpy(layout.page_id).cuda()
        plan.rebuild(spec.parent, spec.node_len, spec.query_node, ct, spec.gqa_group, naive=False)
        bufs = deft.alloc_buffers(plan, spec.num_queries, spec.num_q_heads, spec.head_dim)
        rc = lib.deft_tree_attn(P(t.q.data_ptr()), P(t.k_pages.data_ptr()), P(t.v_pages.data_ptr()),
                                P(npo.data_ptr()), P(pid.data_ptr()), t.k_pages.shape[0], spec.num_q_heads,
                                spec.num_kv_heads, spec.head_dim, 16, 0.1, plan.handle,
                                P(bufs.out.data_ptr()), 0, P(bufs.lse.data_ptr()),
                                P(bufs.workspace.data_ptr()), bufs.workspace.numel(),
                                P(torch.cuda.current_stream().cuda_stream))
        assert rc == -8   # rebuilt, not uploaded
        plan.upload()
        out, lse = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan, bufs=bufs)
        fresh = deft.Plan(spec.parent, spec.node_len, spec.query_node, ct, spec.gqa_group, naive=False)
        fresh.upload()
        out2, lse2 = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, fresh)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.float().cpu().numpy(), out2.float().cpu().numpy())
        np.testing.assert_array_equal(lse.cpu().numpy(), lse2.cpu().numpy())


def test_updated_plan_runs_like_a_fresh_one(deft):
    """deft_plan_update across decode steps (tokens appended to branches,
    then a branch pruned to length 0): each updated plan, uploaded, runs the
    step of a fresh plan of the same tree bit for bit and matches the oracle
    on sampled queries."""
    spec0 = W.few_shot_tree(prefix=600, branches=20, branch_len=70, heads=4, head_dim=128)
    extra = 40   # room in every node's pages for the appended tokens
    grown = W.TreeSpec(spec0.name, spec0.parent, spec0.node_len + extra, spec0.query_node, spec0.num_q_heads,
                       spec0.num_kv_heads, spec0.head_dim, seed=spec0.seed)
    layout = W.paged_layout(grown)
    inp = dense_inputs(grown, seed=3)
    q, k, v = bits_to_cuda(inp.q_bits), bits_to_cuda(inp.k_pages), bits_to_cuda(inp.v_pages)
    npo = torch.from_numpy(inp.layout.node_page_off).cuda()
    pid = torch.from_numpy(inp.layout.page_id).cuda()
    plan = deft.Plan(spec0.parent, spec0.node_len, spec0.query_node, 128, 1, naive=False)
    ln = spec0.node_len.astype(np.int32).copy()
    rng = np.random.default_rng(0)
    for step in range(4):
        ln = ln.copy()
        ln[rng.choice(len(ln), size=3, replace=False)] += 10
        if step == 3:
            ln[5] = 0                                   # a branch pruned
        plan.update(ln)
        plan.upload()
        out, lse = deft.deft_tree_attn(q, k, v, npo, pid, plan)
        fresh = deft.Plan(spec0.parent, ln, spec0.query_node, 128, 1, naive=False)
        fresh.upload()
        out2, lse2 = deft.deft_tree_attn(q, k, v, npo, pid, fresh)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.float().cpu().numpy(), out2.float().cpu().numpy())
        np.testing.assert_array_equal(lse.cpu().numpy(), lse2.cpu().numpy())
        cur = W.TreeSpec(spec0.name, spec0.parent, ln, spec0.query_node, spec0.num_q_heads, spec0.num_kv_heads,
                         spec0.head_dim, seed=spec0.seed)
        ref, ref_lse = oracle.tree_attn(inp.q_bits, inp.k_pages, inp.v_pages, inp.layout.node_page_off,
                                        inp.layout.page_id, inp.layout.page_size, cur.parent, cur.node_len,
                                        cur.query_node, cur.num_q_heads, cur.num_kv_heads, cur.head_dim,
                                        1.0 / math.sqrt(cur.head_dim))
        assert_parity(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
                      ref, ref_lse, f"updated plan, step {step}")


def path_token_counts(spec):
    """|T(q)| per query from the oracle's own path walk: the tokens query q
    attends (its own node up to its position)."""
    counts = []
    for q, path in enumerate(oracle.paths(spec.parent, spec.query_node)):
        n_own = int(spec.query_node[q])
        c = 0
        for n in path:
            if n == n_own and spec.query_pos is not None and spec.query_pos[q] >= 0:
                c += int(spec.query_pos[q]) + 1
            else:
                c += int(spec.node_len[n])
        counts.append(c)
    return np.array(counts, dtype=np.int64)


@pytest.mark.parametrize("cfg", sorted(FULL))
def test_every_query_attends_each_of_its_tokens_once(deft, cfg):
    """An exact count of the (query, token) pairs the kernels process, for
    every query and head, at full size: with K = 0 every logit is 0, each
    attended token adds exactly 1 to its chunk's sum, and the merged lse is
    ln(number of tokens attended).  It must be |T(q)| (each pair once, none
    missed), in the tree and the naive forms."""
    spec = W.config(cfg)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cuda")
    t.k_pages.zero_()
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, FULL[cfg], spec.gqa_group,
                     query_pos=spec.query_pos)
    plan.upload()
    packed = deft.Plan(spec.parent, spec.node_len, spec.query_node, FULL[cfg], spec.gqa_group,
                       query_pos=spec.query_pos, tensor_pack=True, naive=False)
    packed.upload()
    want = path_token_counts(spec)
    runs = [("tree", lambda: deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)),
            ("naive", lambda: deft.deft_naive_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)),
            ("tree, tensor-packed", lambda: deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, packed))]
    for name, fn in runs:
        _, lse = fn()
        torch.cuda.synchronize()
        got = np.rint(np.exp(lse.cpu().numpy().astype(np.float64))).astype(np.int64)
        bad = np.argwhere(got != want[:, None])
        assert bad.size == 0, f"{name}: query {bad[0][0]} head {bad[0][1]} attends " \
                              f"{got[tuple(bad[0])]} tokens, expected {want[bad[0][0]]}"
