"""The bench's host arithmetic (no GPU): algorithmic bytes of each launch
from the plan, KV-head shards, the whole-step roofline and the job value."""
import importlib.util
import os
import sys

import numpy as np
import pytest

import workloads as W
import shared_prefix_kv_deft_gb300 as deft

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


@pytest.mark.parametrize("cfg,tp", [(2, False), (4, False), (4, True), (3, True)])
def test_algorithmic_bytes_cover_the_unique_kv(bench, cfg, tp):
    """Each family's 'all buckets' entry reads every chunk of its items once:
    over both families the KV bytes equal the unique KV (a chunk cut into
    row blocks counts once), q and partial bytes follow the rows."""
    spec = W.config(cfg)
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group, tensor_pack=tp)
    alg = bench.algorithmic_bytes(plan, spec)
    kv_tok = 2 * spec.num_kv_heads * spec.head_dim * 2
    fam = [alg[k] for k in ((0, -1, 0), (1, -1, 0)) if k in alg]
    assert sum(f["kv"] for f in fam) == plan.stats["unique_tokens"] * kv_tok
    G = spec.gqa_group
    rows = 0
    for name in ("fma_items", "mma_items"):
        it = plan.get(name).reshape(-1, 3)
        rows += int(((it[:, 2] - it[:, 1]) * G).sum())
    assert sum(f["q"] for f in fam) == rows * spec.num_kv_heads * spec.head_dim * 2
    assert sum(f["partials"] for f in fam) == rows * spec.num_kv_heads * (spec.head_dim + 1) * 4
    for f in alg.values():
        assert f["total"] == f["kv"] + f["q"] + f["partials"]


def test_phase2_bytes_follow_the_slots(bench):
    spec = W.config(2)
    plan = deft.Plan(spec.parent, spec.node_len, spec.query_node, 256, spec.gqa_group)
    d, Hq, Q = spec.head_dim, spec.num_q_heads, spec.num_queries
    slots = plan.stats["num_slots"]
    assert bench.phase2_bytes(plan, spec) == slots * Hq * (d + 1) * 4 + Q * Hq * (d * 2 + 4) + (Q + 1 + slots) * 4


@pytest.mark.parametrize("hq,hkv,world", [(32, 8, 2), (32, 8, 4), (32, 32, 8), (8, 2, 2)])
def test_head_shards_cover_every_head_once(bench, hq, hkv, world):
    G = hq // hkv
    q_seen, k_seen = [], []
    for r in range(world):
        q0, q1, k0, k1 = bench.head_shard(hq, hkv, r, world)
        assert (q0, q1) == (k0 * G, k1 * G)
        q_seen += list(range(q0, q1))
        k_seen += list(range(k0, k1))
    assert q_seen == list(range(hq)) and k_seen == list(range(hkv))


def test_head_shards_refuse_an_uneven_split(bench):
    with pytest.raises(ValueError):
        bench.head_shard(32, 8, 0, 3)


def test_whole_step_roofline_and_job_value(bench):
    kernels = {"phase1_mma[bucket=0]": {"total_ms": 2.0, "achieved_gbs": 3000.0, "alg_bytes": 1, "avg_us": 1.0},
               "phase2_merge": {"total_ms": 0.5, "achieved_gbs": 100.0, "alg_bytes": 1, "avg_us": 1.0}}
    r = bench.roofline_of(kernels, ms_per_step=0.05, unique_kv=200e6, hbm_peak=8000.0, peak_kind="measured", cfg=99)
    assert r["kernel"] == "phase1_mma[bucket=0]"
    assert r["frac"] == pytest.approx(3000.0 / 8000.0)
    assert r["whole_step"]["achieved"] == pytest.approx(200e6 / 50e-6 / 1e9)
    assert r["whole_step"]["frac"] == pytest.approx(4000.0 / 8000.0)
    assert r["traffic"] is None          # no capture for an unknown workload
    # N replicas each finishing a step in the slowest rank's time.
    assert bench.job_us_per_step(0.05, 4) == pytest.approx(12.5)


def test_source_hash_ignores_comments_only(bench):
    """The counters in profiles/ncu_traffic.json are tied to a hash of the
    kernel sources; a change to comments alone must not detach them, any
    change to code must."""
    src = 'int a = 1; // note\n/* block\n   note */ const char *s = "x // y /* z */"; char q = \'"\';\n\n int b;\n'
    out = bench.strip_comments(src)
    assert "note" not in out and "block" not in out
    assert '"x // y /* z */"' in out and "'\"'" in out
    assert bench.strip_comments(src.replace("// note", "// another note")) == out
    assert bench.strip_comments(src.replace("int b;", "int b = 2;")) != out
