"""deft_tree_attn_noalloc: the step for callers that cannot allocate device
memory (graph-capture code, pool-owned memory, allocation-free loops).

It keeps the plan arrays and the partials in the library's fixed 64 MiB
device array instead of a caller workspace and an uploaded plan.  Its
results must equal those of deft_tree_attn, on two calls in a row (the array
keeps the previous call's contents), and a plan that does not fit must be
refused before anything runs.  This file is collected last on purpose."""
import ctypes
import math

import numpy as np
import pytest

import workloads as W

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


def _call_noalloc(deft, t, npo, pid, spec, plan, out, lse):
    P = ctypes.c_void_p
    return deft.load().deft_tree_attn_noalloc(
        P(t.q.data_ptr()), P(t.k_pages.data_ptr()), P(t.v_pages.data_ptr()),
        P(npo.data_ptr()), P(pid.data_ptr()), int(t.k_pages.shape[0]), spec.num_q_heads,
        spec.num_kv_heads, spec.head_dim, 16, 1.0 / math.sqrt(spec.head_dim), plan.handle,
        P(out.data_ptr()), 0, P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("cfg,shape", [
    (2, None),
    (None, dict(levels=3, len_lo=20, len_hi=90, num_queries=24, q_heads=8, kv_heads=2)),
    (None, "mha_many_queries"),
])
def test_noalloc_matches_tree_attn_twice(deft, cfg, shape):
    if cfg is not None:
        spec = W.config(cfg)
    elif shape == "mha_many_queries":
        spec = W.random_tree(203, max_nodes=10, max_len=300, max_queries=60, q_heads=2,
                             kv_heads=2, head_dim=128, forest=False)
    else:
        spec = W.reasoning_tree(**shape)
    layout = W.paged_layout(spec)
    t = W.make_tensors(spec, layout, device="cuda")
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group)
    plan.upload()
    ref_out, ref_lse = deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan)
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    # A separate plan that was never uploaded: the no-alloc call needs none.
    fresh = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group)
    for _ in range(2):
        out = torch.full_like(t.q, float("nan"))
        lse = torch.full((spec.num_queries, spec.num_q_heads), float("nan"), device="cuda")
        assert _call_noalloc(deft, t, npo, pid, spec, fresh, out, lse) == 0
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.isfinite(o).all()
        assert np.abs(o - ref_out).max() <= OUT_TOL
        assert np.abs(l - ref_lse).max() <= LSE_TOL


def test_noalloc_rejects_a_plan_larger_than_the_array(deft):
    # 256 queries sharing a 70000-token root with 32 heads of 128: the
    # partials alone are over 64 MiB.  The call must refuse before launching.
    spec = W.TreeSpec("big", np.array([-1] + [0] * 256, np.int32),
                      np.array([70000] + [1] * 256, np.int32),
                      np.arange(1, 257, dtype=np.int32), 32, 32, 128)
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, 1)
    need = plan.stats["num_slots"] * 32 * 129 * 4
    assert need > 64 << 20
    small = W.tiny_tree()
    layout = W.paged_layout(small)
    t = W.make_tensors(small, layout, device="cuda")
    npo = torch.from_numpy(layout.node_page_off).cuda()
    pid = torch.from_numpy(layout.page_id).cuda()
    out = torch.zeros((256, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((256, 32), dtype=torch.float32, device="cuda")
    P = ctypes.c_void_p
    rc = deft.load().deft_tree_attn_noalloc(
        P(t.q.data_ptr()), P(t.k_pages.data_ptr()), P(t.v_pages.data_ptr()), P(npo.data_ptr()),
        P(pid.data_ptr()), int(t.k_pages.shape[0]), 32, 32, 128, 16, 0.088, plan.handle,
        P(out.data_ptr()), 0, P(lse.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert rc == -7
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0
