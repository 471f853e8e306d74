"""CUDA-graph replay across serving steps (POD walkthrough, "CUDAGraph 模式的
运行时约束": a fixed batch, page-table buffers reserved at their maximum size,
plan run outside capture).

One pod_run is captured in a CUDA graph on a capacity plan. Every later step
plans its new page tables (decode requests one key longer, a further prefill
chunk, new pages) into the same workspace with pod_replan, writes that
step's queries, cache pages and sinks into the captured tensors in place, replays
the graph, and checks both halves against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import prefill_decode_paged_pod_gb300 as pod
from pod_workloads import make_custom
from podtest_util import compare_half

pytestmark = pytest.mark.gpu

H, HK, D, PS = 16, 2, 128, 16
POOL = 1200          # pages in each half's pool (fixed: the graph holds its pointer)
CAPS = dict(max_p_batch=1, max_p_rows=256, max_p_pages=64,
            max_d_batch=6, max_d_rows=24, max_d_pages=POOL)


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_decode_paged_pod_gb300 import _build
    _build.build()
    pod.load_library()


def _step(i):
    """Inputs of serving step i: decode requests (one with 4 query tokens,
    bottom-right causal) grow by i keys, a prefill chunk of 64 + 64 i rows
    against 64 + 128 i keys; every step draws new values and pages."""
    d_kv = [300 + i, 1777 + i, 77 + i, 4000 + i, 13 + i, 900 + i]
    d_q = [1, 4, 1, 1, 1, 1]
    inp = make_custom(f"g{i}", torch.bfloat16, H, HK, D, PS, True, -1, [64 + 64 * i],
                      [64 + 128 * i], d_q, d_kv, seed=100 + i, sinks=True)
    assert inp.p.num_pages <= POOL and inp.d.num_pages <= POOL
    return inp


def test_graph_replay_across_replans():
    dev = torch.device("cuda")
    inp0 = _step(0)
    pools = {h: torch.zeros((POOL, 2, PS, HK, D), dtype=torch.bfloat16, device=dev) for h in "pd"}
    q = {"p": torch.zeros((CAPS["max_p_rows"], H, D), dtype=torch.bfloat16, device=dev),
         "d": torch.zeros((CAPS["max_d_rows"], H, D), dtype=torch.bfloat16, device=dev)}
    sinks = inp0.sinks.to(dev)

    def load(inp):
        sinks.copy_(inp.sinks.to(dev))
        for half in "pd":
            hh = getattr(inp, half)
            pools[half][: hh.kv.shape[0]].copy_(hh.kv.to(dev))
            q[half][: hh.rows].copy_(hh.q.to(dev))

    h = pod.pod_plan(inp0.p.q_indptr, inp0.p.kv_indptr, inp0.p.kv_indices, inp0.p.last_page_len,
                     inp0.d.q_indptr, inp0.d.kv_indptr, inp0.d.kv_indices, inp0.d.last_page_len,
                     H, HK, D, PS, True, -1, None, dtype=torch.bfloat16, p_num_pages=POOL,
                     d_num_pages=POOL, has_sinks=True, num_sms=16)
    pod.pod_plan_set_graph_capacity(h, **CAPS)
    ws = torch.empty(pod.pod_workspace_size(h), dtype=torch.uint8, device=dev)
    pod.pod_bind_workspace(h, ws)
    outs = pod.pod_run(h, q["p"], pools["p"], q["d"], pools["d"], ws, sinks=sinks)  # tensor maps
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        pod.pod_run(h, q["p"], pools["p"], q["d"], pools["d"], ws, sinks=sinks,
                    out_p=outs[0], lse_p=outs[1], out_d=outs[2], lse_d=outs[3])
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            pod.pod_run(h, q["p"], pools["p"], q["d"], pools["d"], ws, sinks=sinks,
                        out_p=outs[0], lse_p=outs[1], out_d=outs[2], lse_d=outs[3])
    torch.cuda.current_stream().wait_stream(s)

    splits = 0
    for i in range(4):
        inp = _step(i)
        if i > 0:
            pod.pod_replan(h, inp.p.q_indptr, inp.p.kv_indptr, inp.p.kv_indices,
                           inp.p.last_page_len, inp.d.q_indptr, inp.d.kv_indptr,
                           inp.d.kv_indices, inp.d.last_page_len)
        load(inp)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert pod.pod_read_device_status(h, ws) == 0
        splits += pod.plan_summary(h)["n_groups"] > 0
        op, lp, od, ld = [t.double().cpu().numpy() for t in outs]
        compare_half(inp, "p", op[: inp.p.rows], lp[: inp.p.rows], tag=f"step {i} ")
        compare_half(inp, "d", od[: inp.d.rows], ld[: inp.d.rows], tag=f"step {i} ")
    assert splits > 0, "expected at least one step with decode splits (merge kernel in the graph)"
    pod.pod_destroy(h)
