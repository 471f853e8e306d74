"""Benchmark of the fused POD launch on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--impl ours|reference]

A step is one fused POD launch (prefill tiles + decode items of one batch,
plus the split merge when the plan has one) over a batch of synthetic inputs
already resident in HBM. The default workload is c5 ("ragged stress", the
largest single-GPU configuration): bf16, 64/8 heads, head_dim 128, page_size 16,
4 causal prefill requests q = kv = {1000, 3000, 700, 4096}, 512 decode requests
with 4 query tokens each and lognormal KV lengths, window_left 4096, sinks.

Printed JSON (one line, rank 0): the metric is the fused-launch time in
microseconds (lower is better); `roofline` reports the fused kernel against the
measured HBM or tensor peak; extra keys give prefill TFLOP/s and decode GB/s
from single-half runs of the same kernel, the CPU oracle baseline, end-to-end
time through the public API with host buffers, and SM clocks sampled during
the measurement.

Under torchrun each rank runs its own independent batch of the same workload
(no collective on the data path); the job time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused POD launch µs; prefill TFLOP/s & decode KV GB/s vs GB300 roofline"
WORKLOAD_DESC = {
    "c1": "c1 tiny POD fp16 4/1/64/16: prefill 64/64, decode kv {17,29,5,48}",
    "c2": "c2 single-request POD fp16 64/8/128/16: prefill 1024/1024, 7 decode (docstring page table)",
    "c3": "c3 batch POD bf16 64/8/128/1: prefill 2x2048, decode 128x2048, contiguous pages",
    "c4": "c4 chunked-prefill overlap bf16 32/8/128/16: prefill 512 vs kv 8192, 256 decode kv~U[512,16384]",
    "c5": "c5 ragged stress bf16 64/8/128/16: prefill {1000,3000,700,4096}, 512 decode x 4 tokens, "
          "kv lognormal(median 2048), window 4096, sinks",
}


# ----------------------------------------------------------------- algorithmic work
def allowed_keys(kv_len, q_len, causal, window_left):
    """Number of (query row, key) pairs allowed per qo head, per request."""
    tot = 0
    for i in range(q_len):
        p = kv_len - q_len + i
        hi = min(kv_len, p + 1) if causal else kv_len
        lo = max(0, p - window_left) if window_left >= 0 else 0
        tot += max(0, hi - lo)
    return tot


def touched_keys(kv_len, q_len, causal, window_left):
    """Keys read at least once by a request (union over its query rows)."""
    if q_len == 0:
        return 0
    p0, p1 = kv_len - q_len, kv_len - 1
    hi = min(kv_len, p1 + 1) if causal else kv_len
    lo = max(0, p0 - window_left) if window_left >= 0 else 0
    return max(0, hi - lo)


def work(inp):
    """Algorithmic FLOPs and bytes of one launch (per half)."""
    H, Hk, d = inp.num_qo_heads, inp.num_kv_heads, inp.head_dim
    el = 2
    out = {}
    for name, h in (("p", inp.p), ("d", inp.d)):
        el_kv = h.kv.element_size() if hasattr(h.kv, "element_size") else el
        pairs = keys = 0
        for r in range(h.batch):
            ql, kl = int(h.q_lens[r]), int(h.kv_lens[r])
            pairs += allowed_keys(kl, ql, inp.causal, inp.window_left)
            keys += touched_keys(kl, ql, inp.causal, inp.window_left)
        flops = 4.0 * d * H * pairs
        kv_bytes = keys * Hk * d * el_kv * 2.0
        qo_bytes = h.rows * H * (d * el * 2 + 4)
        out[name] = dict(pairs=pairs, keys=keys, flops=flops, kv_bytes=kv_bytes,
                         bytes=kv_bytes + qo_bytes, rows=h.rows)
    return out


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
              "utilization.gpu")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        load = [r for r in rows if (num(r[9]) or 0) >= 50] or rows
        sm = [num(r[1]) for r in load if num(r[1]) is not None]
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in load:
            for i, nm in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len(load),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ----------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), tc=float(d["bf16_tflops"]),
                    tc_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    source="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, source="fallback")


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "prefill_decode_paged_pod_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".hpp", ".cpp")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int, device=None) -> float:
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def sample_pairs(inp, half, n, seed):
    """Deterministic sample of (token, head) pairs of one half."""
    h = inp.p if half == "p" else inp.d
    if h.rows == 0 or n <= 0:
        return np.zeros(0, np.int64), np.zeros(0, np.int32)
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, h.rows, size=n).astype(np.int64)
    hd = rng.integers(0, inp.num_qo_heads, size=n).astype(np.int32)
    return tok, hd


def pairs_work(inp, half, tok, hd):
    """Allowed keys summed over the sampled pairs (oracle cost units)."""
    h = inp.p if half == "p" else inp.d
    req = np.searchsorted(h.q_indptr, tok, side="right") - 1
    tot = 0
    for t, r in zip(tok, req):
        ql, kl = int(h.q_lens[r]), int(h.kv_lens[r])
        i = int(t - h.q_indptr[r])
        p = kl - ql + i
        hi = min(kl, p + 1) if inp.causal else kl
        lo = max(0, p - inp.window_left) if inp.window_left >= 0 else 0
        tot += max(0, hi - lo)
    return tot


def oracle_launch_estimate(inp, w, target_s=10.0, seed=0, nthreads=None):
    """Time the fp64 oracle on a bounded sample of (token, head) pairs of both
    halves and scale to one whole launch. Returns (us_per_launch, info)."""
    import oracle
    nthreads = nthreads or os.cpu_count() or 1
    total_work = (w["p"]["pairs"] + w["d"]["pairs"]) * inp.num_qo_heads
    # calibrate on a small sample, then size the main sample for ~target_s
    n = 64
    spent, done_work, n_pairs = 0.0, 0, 0
    while True:
        t0 = time.perf_counter()
        for half, frac in (("p", 0.5), ("d", 0.5)):
            tok, hd = sample_pairs(inp, half, max(1, int(n * frac)), seed + n)
            if len(tok) == 0:
                continue
            oracle.attention_half(inp, half, sel_token=tok, sel_head=hd, nthreads=nthreads)
            done_work += pairs_work(inp, half, tok, hd)
            n_pairs += len(tok)
        spent += time.perf_counter() - t0
        if spent >= target_s or n >= 1 << 20:
            break
        rate = done_work / max(spent, 1e-6)
        want = (target_s - spent) * rate
        per_pair = done_work / max(n_pairs, 1)
        n = int(min(max(64, want / max(per_pair, 1)), 1 << 20))
    us = spent / max(done_work, 1) * total_work * 1e6
    info = dict(pairs=n_pairs, key_work=done_work, seconds=spent)
    return us, info


# ----------------------------------------------------------------- arms
def run_reference(args, ws, rank):
    """The fp64 CPU oracle as the reference arm, on the host cores."""
    from pod_workloads import make_config
    if rank != 0:
        return 0
    inp = with_kv_option(make_config(args.workload), args)
    w = work(inp)
    nthreads = os.cpu_count() or 1
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    vals = []
    info = None
    for s in range(args.warmup + args.steps):
        us, info = oracle_launch_estimate(inp, w, target_s=per_step, seed=1000 * s, nthreads=nthreads)
        if s >= args.warmup:
            vals.append(us)
    v = float(np.mean(vals))
    sample = (f"per step ~{per_step:.0f} s of fp64 oracle on random (token, head) pairs of both "
              f"halves (last step: {info['pairs']} pairs), scaled by allowed (row, key) pairs to one launch")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD_DESC[args.workload],
                                            **variant_desc(args)},
            "cpu_baseline": {"value": v, "unit": "us", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def with_kv_option(inp, args):
    """Variant switches of the same workload:
    --kv-fp8: the decode half's cache as FP8 E4M3 codes (scales 0.05);
    --kv-layout HND: both caches stored [pages, 2, Hk, ps, d];
    --soft-cap C: logits soft cap C on both halves;
    --alibi: geometric ALiBi slopes on both halves;
    --prefill-mask P: a random custom prefill mask, each bit set with probability P;
    --rope: ROPE_LLAMA (rope_scale 1, rope_theta 1e4) on both halves;
    --decode-requests N: only the first N decode requests (compact page pool),
    the smaller case the ncu captures use."""
    from pod_workloads import (alibi_slopes, with_fp8_decode_cache, with_kv_layout,
                               with_prefill_custom_mask)
    if getattr(args, "kv_layout", "NHD") == "HND":
        inp = with_kv_layout(inp, "HND")
    if getattr(args, "kv_fp8", False):
        inp = with_fp8_decode_cache(inp, k_scale=0.05, v_scale=0.05)
    if getattr(args, "soft_cap", 0.0):
        inp.soft_cap = float(args.soft_cap)
    if getattr(args, "alibi", False):
        inp.alibi = alibi_slopes(inp.num_qo_heads)
    if getattr(args, "prefill_mask", None) is not None:
        inp = with_prefill_custom_mask(inp, seed=7, density=float(args.prefill_mask))
    if getattr(args, "rope", False):
        inp.rope = (1.0, 1e4)
    if getattr(args, "decode_requests", None) is not None:
        from pod_workloads import with_decode_subset
        inp = with_decode_subset(inp, args.decode_requests)
    return inp


def variant_desc(args) -> dict:
    """The variant switches of a run, for the JSON line's config."""
    v = {"decode_kv": "fp8 e4m3 (k_scale 0.05, v_scale 0.05)" if args.kv_fp8 else "16-bit"}
    if getattr(args, "kv_layout", "NHD") != "NHD":
        v["kv_layout"] = args.kv_layout
    if getattr(args, "soft_cap", 0.0):
        v["logits_soft_cap"] = float(args.soft_cap)
    if getattr(args, "alibi", False):
        v["alibi"] = "geometric slopes 2^(-8h/H)"
    if getattr(args, "prefill_mask", None) is not None:
        v["prefill_custom_mask_density"] = float(args.prefill_mask)
    if getattr(args, "rope", False):
        v["pos_encoding"] = ("ROPE_LLAMA (scale 1, theta 1e4): hi/lo rotated queries and prefill "
                             "pages from a pre-pass, decode keys rotated in the kernel")
    if getattr(args, "decode_requests", None) is not None:
        v["decode_requests"] = int(args.decode_requests)
    return v


def time_loop(fn, steps, stream, per_launch=True, pre=None):
    """Run fn() `steps` times; returns (total_ms, list of per-call ms). pre(),
    when given, runs before each call outside the per-call events (an L2
    flush); the total includes it."""
    import torch
    if per_launch:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # Hold the stream on a short device-side spin so the host can queue the
    # launches ahead of the GPU: the events then time kernels, not the host's
    # per-call overhead (that is what the end-to-end figure measures).
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(min(steps * 200_000, 100_000_000)))
    start.record(stream)
    for i in range(steps):
        if pre is not None:
            pre()
        if per_launch:
            evs[i][0].record(stream)
        fn()
        if per_launch:
            evs[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in evs] if per_launch else []
    return start.elapsed_time(end), per


def e2e_pipelined(pod, inp, h, wsb, dev, outs, hq, device, steps):
    """End to end through the public API, steps overlapped on three streams:
    while step i computes, the host->device copy of step i+1's queries and
    the device->host copy of step i-1's outputs run on their own streams.
    Two device buffer sets (and two plan handles on the one workspace, so
    each keeps its tensor maps) alternate; events order every reuse. Every
    step still copies its queries in and its outputs out inside the timed
    region. Returns (ms per step, host outputs of the last step)."""
    import torch
    Ev = torch.cuda.Event
    h_b = pod.plan_inputs(inp)
    pod.pod_bind_workspace(h_b, wsb)
    handles = (h, h_b)
    like = lambda t: torch.empty_like(t) if t is not None else None
    qbuf = [dict(q_p=dev["q_p"], q_d=dev["q_d"]), dict(q_p=like(dev["q_p"]), q_d=like(dev["q_d"]))]
    obuf = [tuple(outs), tuple(torch.empty_like(t) for t in outs)]
    hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] for _ in range(2)]
    s_in, s_c, s_out = (torch.cuda.Stream(device) for _ in range(3))
    q_ready, q_free, done, out_free = ([Ev(), Ev()] for _ in range(4))

    def one(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(q_free[b])          # step i-2 has read this buffer set
            for k in ("q_p", "q_d"):
                if hq[k] is not None:
                    qbuf[b][k].copy_(hq[k], non_blocking=True)
            q_ready[b].record(s_in)
        with torch.cuda.stream(s_c):
            s_c.wait_event(q_ready[b])
            s_c.wait_event(out_free[b])         # step i-2's outputs have left
            op, lp, od, ld = obuf[b]
            pod.pod_run(handles[b], qbuf[b]["q_p"], dev["kv_p"], qbuf[b]["q_d"], dev["kv_d"], wsb,
                        sinks=dev["sinks"], out_p=op, lse_p=lp, out_d=od, lse_d=ld)
            q_free[b].record(s_c)
            done[b].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            for dst, src in zip(hout[b], obuf[b]):
                if src.numel():
                    dst.copy_(src, non_blocking=True)
            out_free[b].record(s_out)

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream(device)
    start, end = Ev(enable_timing=True), Ev(enable_timing=True)
    start.record(main)
    for st in (s_in, s_c, s_out):
        st.wait_stream(main)
    for i in range(steps):
        one(i)
    for st in (s_in, s_c, s_out):
        main.wait_stream(st)
    end.record(main)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, hout[(steps - 1) & 1]


def run_ours(args, ws, rank, local):
    import torch
    import prefill_decode_paged_pod_gb300 as pod
    from prefill_decode_paged_pod_gb300 import _build
    from pod_workloads import make_config

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    _build.build()
    pod.load_library()
    idx = ["c1", "c2", "c3", "c4", "c5"].index(args.workload) + 1
    inp = with_kv_option(make_config(args.workload, seed=idx + 1000 * rank), args)
    w = work(inp)
    stream = torch.cuda.current_stream(device)
    dev = dict(q_p=inp.p.q.to(device) if inp.p.rows else None,
               kv_p=inp.p.kv.to(device) if inp.p.rows else None,
               q_d=inp.d.q.to(device) if inp.d.rows else None,
               kv_d=inp.d.kv.to(device) if inp.d.rows else None,
               sinks=inp.sinks.to(device) if inp.sinks is not None else None)
    h = pod.plan_inputs(inp)
    summ = pod.plan_summary(h)
    # host planning time of this batch (once per serving step), through the
    # binding, on the calling thread
    plan_ts = []
    for _ in range(5):
        t0 = time.perf_counter()
        hp = pod.plan_inputs(inp)
        plan_ts.append(time.perf_counter() - t0)
        pod.pod_destroy(hp)
    plan_us = float(np.median(plan_ts)) * 1e6
    wsb = torch.empty(pod.pod_workspace_size(h), dtype=torch.uint8, device=device)
    pod.pod_bind_workspace(h, wsb)
    H, d = inp.num_qo_heads, inp.head_dim
    out_p = torch.empty((inp.p.rows, H, d), dtype=inp.dtype, device=device)
    lse_p = torch.empty((inp.p.rows, H), dtype=torch.float32, device=device)
    out_d = torch.empty((inp.d.rows, H, d), dtype=inp.dtype, device=device)
    lse_d = torch.empty((inp.d.rows, H), dtype=torch.float32, device=device)

    def step():
        pod.pod_run(h, dev["q_p"], dev["kv_p"], dev["q_d"], dev["kv_d"], wsb, sinks=dev["sinks"],
                    out_p=out_p, lse_p=lse_p, out_d=out_d, lse_d=lse_d)

    kv_total = inp.p.kv.numel() * inp.p.kv.element_size() + inp.d.kv.numel() * inp.d.kv.element_size()
    l2_bytes = 129 * 1024 * 1024
    flush = flush_r = None
    if kv_total < 2 * l2_bytes:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
        flush_r = torch.ones(256 * 1024 * 1024, dtype=torch.uint8, device=device)

    def flush_l2():
        # write a buffer larger than L2, then read another one: the read evicts
        # the write's dirty lines, so the timed launch pays for its own misses
        # and not for writing back the flush
        if flush is not None:
            flush.zero_()
            flush_r.sum()

    def step_flush():
        flush_l2()
        step()

    for _ in range(max(args.warmup, 3)):
        step_flush()
    torch.cuda.synchronize()
    assert pod.pod_read_device_status(h, wsb) == 0

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    # --- main timed region: K steps (flush between steps only when inputs fit in L2)
    barrier(ws)
    torch.cuda.synchronize()
    if flush is None:
        total_ms, per = time_loop(step, args.steps, stream)
    else:
        # per-launch events exclude the flush; the total includes it
        total_ms, per = time_loop(step, args.steps, stream, pre=flush_l2)
    torch.cuda.synchronize()
    barrier(ws)
    kernel_ms = float(np.mean(per))
    step_ms = total_ms / args.steps if flush is None else kernel_ms
    step_ms = max_over_ranks(step_ms, ws, device)
    # the fused kernel, the merge kernel when the plan splits, and under RoPE
    # the pre-pass (queries of each non-empty half, pages of the prefill half;
    # the angle table runs once per bound workspace, before the timed steps)
    launches = 1 + (1 if summ["n_mrows"] > 0 else 0)
    if summ.get("rope"):
        launches += (2 if inp.p.rows else 0) + (1 if inp.d.rows else 0)

    # --- single-half runs of the same kernel: prefill TFLOP/s and decode GB/s
    halves = {}
    for half in ("p", "d"):
        hh = inp.p if half == "p" else inp.d
        if hh.rows == 0:
            continue
        import copy
        sub = copy.copy(inp)
        empty = copy.copy(inp.d if half == "p" else inp.p)
        empty.q_indptr = np.zeros(1, np.int32)
        empty.kv_indptr = np.zeros(1, np.int32)
        empty.kv_indices = np.zeros(0, np.int32)
        empty.last_page_len = np.zeros(0, np.int32)
        if half == "p":
            sub.d = empty
        else:
            sub.p = empty
        hs = pod.plan_inputs(sub)
        wss = torch.empty(pod.pod_workspace_size(hs), dtype=torch.uint8, device=device)
        pod.pod_bind_workspace(hs, wss)

        def step_half(hs=hs, wss=wss, half=half):
            if half == "p":
                pod.pod_run(hs, dev["q_p"], dev["kv_p"], None, None, wss, sinks=dev["sinks"],
                            out_p=out_p, lse_p=lse_p)
            else:
                pod.pod_run(hs, None, None, dev["q_d"], dev["kv_d"], wss, sinks=dev["sinks"],
                            out_d=out_d, lse_d=lse_d)

        for _ in range(3):
            step_half()
        torch.cuda.synchronize()
        n = max(10, args.steps // 2)
        _, per_h = time_loop(step_half, n, stream, pre=flush_l2)  # same cache state
        halves[half] = float(np.median(per_h))

    # --- end to end through the public API with host buffers
    pin = lambda t: t.pin_memory() if t is not None else None
    hq_p, hq_d = pin(inp.p.q) if inp.p.rows else None, pin(inp.d.q) if inp.d.rows else None
    ho = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (out_p, lse_p, out_d, lse_d)]
    h2d = (inp.p.q.numel() + inp.d.q.numel()) * inp.p.q.element_size()
    d2h = sum(t.numel() * t.element_size() for t in (out_p, lse_p, out_d, lse_d))

    def step_e2e():
        if hq_p is not None:
            dev["q_p"].copy_(hq_p, non_blocking=True)
        if hq_d is not None:
            dev["q_d"].copy_(hq_d, non_blocking=True)
        step()
        for dst, src in zip(ho, (out_p, lse_p, out_d, lse_d)):
            if src.numel():
                dst.copy_(src, non_blocking=True)

    for _ in range(3):
        step_e2e()
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms, _ = time_loop(step_e2e, args.steps, stream, per_launch=False)
    barrier(ws)
    e2e_serial_ms = max_over_ranks(e2e_ms / args.steps, ws, device)
    # the same, with the copies of neighbouring steps overlapping the compute;
    # a candidate only if its outputs equal the serial loop's bit for bit
    e2e_mode = "3-stream pipelined"
    try:
        pipe_ms, last = e2e_pipelined(pod, inp, h, wsb, dev, (out_p, lse_p, out_d, lse_d),
                                      dict(q_p=hq_p, q_d=hq_d), device, args.steps)
        if not all(torch.equal(a, b) for a, b in zip(last, ho)):
            raise RuntimeError("pipelined outputs differ from the serial loop")
    except Exception as ex:  # noqa: BLE001 - report and keep the serial figure
        print(f"[bench] pipelined end-to-end not used: {ex!r}", file=sys.stderr)
        pipe_ms = float("inf")
    barrier(ws)
    pipe_ms = max_over_ranks(pipe_ms, ws, device)
    # the faster of the two schedules (tiny launches lose more to the three
    # streams' synchronisation than the overlap gains)
    if pipe_ms >= e2e_serial_ms:
        e2e_mode, pipe_ms = "serial", e2e_serial_ms
    e2e_step_ms = pipe_ms
    clk = clocks.stop()
    assert pod.pod_read_device_status(h, wsb) == 0

    # --- roofline of the fused kernel
    peaks = measured_peaks()
    B = w["p"]["bytes"] + w["d"]["bytes"]
    F = w["p"]["flops"]
    t_s = kernel_ms / 1e3
    t_hbm = B / (peaks["hbm"] * 1e9)
    t_tc = F / (peaks["tc"] * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": B / t_s / 1e9, "peak": peaks["hbm"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": F / t_s / 1e12, "peak": peaks["tc"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(args.workload)
    roof["peak_source"] = peaks["source"]
    roof["fused_frac"] = max(t_hbm, t_tc) / t_s
    roof["algorithmic_bytes_per_launch"] = B
    roof["algorithmic_prefill_flops_per_launch"] = F
    extra = {}
    if "p" in halves:
        tf = w["p"]["flops"] / (halves["p"] / 1e3) / 1e12
        extra["prefill_only_us"] = halves["p"] * 1e3
        extra["prefill_tflops"] = tf
        extra["prefill_frac_of_measured_bf16"] = tf / peaks["tc"]
    if "d" in halves:
        gbs = w["d"]["bytes"] / (halves["d"] / 1e3) / 1e9
        extra["decode_only_us"] = halves["d"] * 1e3
        extra["decode_gbs"] = gbs
        extra["decode_frac_of_measured_hbm"] = gbs / peaks["hbm"]

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        nthreads = os.cpu_count() or 1
        us, info = oracle_launch_estimate(inp, w, target_s=args.cpu_seconds, nthreads=nthreads)
        cpu = {"value": us, "unit": "us", "cores": nthreads, "kind": "oracle",
               "sample": f"{info['pairs']} random (token, head) pairs of both halves "
                         f"({info['seconds']:.1f} s, fp64), scaled by allowed (row, key) pairs to one launch"}

    value_us = step_ms * 1e3
    line = {
        "metric": METRIC, "value": value_us, "unit": "us", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if inp.dtype.__repr__().endswith("bfloat16") else "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "num_qo_heads": H,
                   "num_kv_heads": inp.num_kv_heads, "head_dim": d, "page_size": inp.page_size,
                   "prefill_rows": inp.p.rows, "decode_rows": inp.d.rows,
                   "l2": ("inputs larger than L2" if flush is None else
                          "L2 flushed (256 MB write + 256 MB read) between timed launches"),
                   "kv_cache_bytes": kv_total, "parallelism": f"replicas x{ws} (independent batches)",
                   **variant_desc(args)},
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": e2e_step_ms * 1e3, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "mode": e2e_mode,
                "serial_value": e2e_serial_ms * 1e3},
        "gpu_launches": launches * args.steps, "clocks": clk,
        "plan": {k: summ[k] for k in ("grid", "n_p_ctas", "n_d_ctas", "n_tiles", "n_items",
                                       "n_groups", "decode_chunk")},
        "launch_us_median": float(np.median(per)) * 1e3,
        "plan_us": plan_us,
    }
    line.update(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile(args):
    """Launch one variant of the workload --warmup + --steps times with nothing
    else on the GPU (no flush, no timing beyond a summary line): the command
    the ncu captures under profiles/ run. fused = both halves; prefill or
    decode = that half alone, planned as the single-half runs of run_ours."""
    import copy
    import torch
    import prefill_decode_paged_pod_gb300 as pod
    from prefill_decode_paged_pod_gb300 import _build
    from pod_workloads import make_config

    _build.build()
    pod.load_library()
    torch.cuda.set_device(0)
    idx = ["c1", "c2", "c3", "c4", "c5"].index(args.workload) + 1
    inp = with_kv_option(make_config(args.workload, seed=idx), args)
    sub = copy.copy(inp)
    if args.profile != "fused":
        empty = copy.copy(inp.d if args.profile == "prefill" else inp.p)
        empty.q_indptr = np.zeros(1, np.int32)
        empty.kv_indptr = np.zeros(1, np.int32)
        empty.kv_indices = np.zeros(0, np.int32)
        empty.last_page_len = np.zeros(0, np.int32)
        if args.profile == "prefill":
            sub.d = empty
        else:
            sub.p = empty
    use_p, use_d = sub.p.rows > 0, sub.d.rows > 0
    q_p = inp.p.q.cuda() if use_p else None
    kv_p = inp.p.kv.cuda() if use_p else None
    q_d = inp.d.q.cuda() if use_d else None
    kv_d = inp.d.kv.cuda() if use_d else None
    sinks = inp.sinks.cuda() if inp.sinks is not None else None
    h = pod.plan_inputs(sub)
    wsb = torch.empty(pod.pod_workspace_size(h), dtype=torch.uint8, device="cuda")
    pod.pod_bind_workspace(h, wsb)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup + args.steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            s.record()
        pod.pod_run(h, q_p, kv_p, q_d, kv_d, wsb, sinks=sinks)
    e.record()
    torch.cuda.synchronize()
    status = pod.pod_read_device_status(h, wsb)
    summ = pod.plan_summary(h)
    print(json.dumps({"profile": args.profile, "workload": args.workload,
                      "launch_us_mean": s.elapsed_time(e) * 1e3 / max(args.steps, 1),
                      "grid": summ["grid"], "status": status}), flush=True)
    return 0 if status == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="c5", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--kv-fp8", action="store_true",
                    help="decode cache in FP8 E4M3 (per-tensor K and V scales)")
    ap.add_argument("--kv-layout", choices=["NHD", "HND"], default="NHD",
                    help="page layout of both caches")
    ap.add_argument("--soft-cap", type=float, default=0.0, help="logits soft cap (0 = off)")
    ap.add_argument("--alibi", action="store_true", help="ALiBi with geometric head slopes")
    ap.add_argument("--prefill-mask", type=float, default=None, metavar="DENSITY",
                    help="random custom prefill mask with this fraction of allowed keys")
    ap.add_argument("--rope", action="store_true", help="ROPE_LLAMA on both halves")
    ap.add_argument("--decode-requests", type=int, default=None, metavar="N",
                    help="only the first N decode requests (a smaller case for profiler captures)")
    ap.add_argument("--profile", choices=["fused", "prefill", "decode"], default=None,
                    help="only launch this variant (for ncu captures); prints a summary line")
    args = ap.parse_args(argv)
    if args.profile:
        return run_profile(args)
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
