"""Host-side logic of bench.py, on CPU: algorithmic work counts, the
max-over-ranks timing reduction under a world_size-2 gloo group, and the
JSON contract of the reference (oracle) arm on a tiny workload."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from pod_workloads import make_config, make_custom  # noqa: E402


def test_allowed_and_touched_keys_closed_forms():
    # causal q = kv = n: n (n + 1) / 2 pairs, n keys touched
    assert bench.allowed_keys(100, 100, True, -1) == 100 * 101 // 2
    assert bench.touched_keys(100, 100, True, -1) == 100
    # decode q_len 1: every key
    assert bench.allowed_keys(777, 1, True, -1) == 777
    # window w: each row sees at most w + 1 keys
    assert bench.allowed_keys(50, 4, True, 3) == 4 * 4
    assert bench.touched_keys(50, 4, True, 3) == 4 + 3
    # non-causal: q_len * kv_len
    assert bench.allowed_keys(9, 5, False, -1) == 45


def test_work_matches_workload_figures():
    inp = make_config("c3", with_data=False)
    w = bench.work(inp)
    # 2 requests x causal 2048^2 / 2 pairs x 64 heads x 4 d flops
    assert w["p"]["flops"] == 2 * (2048 * 2049 // 2) * 64 * 4 * 128
    assert abs(w["p"]["flops"] - 137.5e9) / 137.5e9 < 2e-3
    assert w["d"]["kv_bytes"] == 128 * 2048 * 8 * 128 * 2 * 2


def _rank_main(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2",
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ws, r, _ = bench.dist_env()
    bench.barrier(ws)
    v = bench.max_over_ranks(1.5 + rank, ws)
    q.put((r, v))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    ps = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5), (1, 2.5)]


def test_reference_arm_json_contract():
    env = dict(os.environ)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "c1", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "cpu_baseline", "e2e", "impl"):
        assert k in line
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_variant_switches_reach_the_inputs():
    """bench.py's variant switches build the same workload with an HND cache,
    a soft cap, ALiBi slopes or a custom prefill mask, and name them in the
    JSON line's config."""
    import argparse
    from pod_workloads import make_config
    args = argparse.Namespace(kv_fp8=False, kv_layout="HND", soft_cap=0.0, alibi=True,
                              prefill_mask=0.3, rope=True)
    base = make_config("c1")
    inp = bench.with_kv_option(make_config("c1"), args)
    assert inp.p.kv_layout == inp.d.kv_layout == "HND"
    assert tuple(inp.p.kv.shape) == (base.p.kv.shape[0], 2, base.num_kv_heads, base.page_size,
                                      base.head_dim)
    assert inp.alibi is not None and inp.alibi.shape == (base.num_qo_heads,)
    bits = int(sum(int(q) * int(k) for q, k in zip(np.diff(inp.p.q_indptr), inp.p.kv_lens)))
    assert inp.p.packed_mask.nbytes == (bits + 7) // 8
    desc = bench.variant_desc(args)
    assert desc["kv_layout"] == "HND" and "alibi" in desc
    assert desc["prefill_custom_mask_density"] == 0.3
    assert inp.rope == (1.0, 1e4) and "ROPE_LLAMA" in desc["pos_encoding"]
