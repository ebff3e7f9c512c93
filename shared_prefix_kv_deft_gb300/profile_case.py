"""Runs a few tree-attention steps of a named, seeded workload on cuda:0, for
profiling captures that must stay small (a few hundred MB on the device):

    python -m shared_prefix_kv_deft_gb300.profile_case <case> [steps] [--range]

--range brackets one more step, after the others, with cudaProfilerStart /
cudaProfilerStop, so that ncu's range replay (--replay-mode range
--profile-from-start off) measures the whole step, its launches running
concurrently as they do in the benchmark.

Cases (synthetic, seeded; the shapes of the benchmark workloads, fewer
requests):
    speculative_3req   3 requests x (4000-token prefix + 64-node token tree),
                       32/32 heads, d 128 (tensor-core launch, 64 rows)
    control_32x2048    32 independent 2048-token sequences, GQA 32/8, d 128
                       (CUDA-core launch, 4 rows)
    few_shot           the few-shot tree (4096-token prefix + 32 x 256)
    reasoning          the reasoning tree (4 levels, 128 queries, GQA 32/8):
                       CUDA-core launches with 8 and 12 rows
"""
import sys

import torch

import workloads as W
import shared_prefix_kv_deft_gb300 as deft

CASES = {
    "speculative_3req": lambda: W.speculative_forest(requests=3),
    "control_32x2048": lambda: W.imbalance_tree(control=True, leaves=32),
    "few_shot": lambda: W.config(2),
    "reasoning": lambda: W.config(4),
}


def main(argv):
    ranged = "--range" in argv
    argv = [x for x in argv if x != "--range"]
    spec = CASES[argv[1]]()
    steps = int(argv[2]) if len(argv) > 2 else 4
    lay = W.paged_layout(spec)
    t = W.make_tensors(spec, lay, device="cuda")
    npo = torch.from_numpy(lay.node_page_off).cuda()
    pid = torch.from_numpy(lay.page_id).cuda()
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group)
    plan.upload()
    bufs = deft.alloc_buffers(plan, spec.num_queries, spec.num_q_heads, spec.head_dim)
    for _ in range(steps):
        deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan, bufs=bufs)
    torch.cuda.synchronize()
    if ranged:
        torch.cuda.profiler.start()
        deft.deft_tree_attn(t.q, t.k_pages, t.v_pages, npo, pid, plan, bufs=bufs)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    print("ok", spec.name)


if __name__ == "__main__":
    main(sys.argv)
