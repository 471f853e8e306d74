"""Shared helpers of the GPU tests: run the POD library through its C-ABI
binding and compare with the fp64 oracle under the stated tolerances.

Tolerances (from the build's accuracy target): outputs |gpu - ref| <=
2e-2 + 2e-2 |ref| elementwise; base-2 LSE |gpu - ref| <= 1e-3.
"""
from __future__ import annotations

import os
import subprocess

import numpy as np
import torch

import oracle
import prefill_decode_paged_pod_gb300 as pod

OUT_ATOL = 2e-2
OUT_RTOL = 2e-2
LSE_ATOL = 1e-3

HERE = os.path.dirname(os.path.abspath(__file__))


def to_dev(inp, device="cuda"):
    return dict(
        q_p=inp.p.q.to(device) if inp.p.rows else None,
        kv_p=inp.p.kv.to(device) if inp.p.rows else None,
        q_d=inp.d.q.to(device) if inp.d.rows else None,
        kv_d=inp.d.kv.to(device) if inp.d.rows else None,
        sinks=inp.sinks.to(device) if inp.sinks is not None else None)


def run_pod(inp, dev=None, num_sms=0, repeat=1):
    """Plan (host), bind a fresh workspace, run; returns CPU fp64 numpy outputs
    (out_p, lse_p, out_d, lse_d), the handle and the workspace."""
    dev = dev or to_dev(inp)
    h = pod.plan_inputs(inp, workspace=None, num_sms=num_sms)
    ws = torch.empty(max(pod.pod_workspace_size(h), 256), dtype=torch.uint8, device="cuda")
    pod.pod_bind_workspace(h, ws)
    res = None
    for _ in range(repeat):
        res = pod.pod_run(h, dev["q_p"], dev["kv_p"], dev["q_d"], dev["kv_d"], ws, sinks=dev["sinks"])
    torch.cuda.synchronize()
    status = pod.pod_read_device_status(h, ws)
    assert status == 0, f"device status {status}"
    out_p, lse_p, out_d, lse_d = [t.double().cpu().numpy() for t in res]
    return (out_p, lse_p, out_d, lse_d), h, ws


def compare_half(inp, half, out, lse, sel_token=None, sel_head=None, tag=""):
    """Oracle on the selected (token, head) pairs (all when None) and compare."""
    h = inp.p if half == "p" else inp.d
    if h.rows == 0:
        return 0.0, 0.0
    H = inp.num_qo_heads
    if sel_token is None:
        sel_token = np.repeat(np.arange(h.rows), H)
        sel_head = np.tile(np.arange(H), h.rows)
    ro, rl, st = oracle.attention_half(inp, half, sel_token=sel_token, sel_head=sel_head)
    assert st == 0, f"oracle status {st}"
    go = out[sel_token, sel_head].astype(np.float64)
    gl = lse[sel_token, sel_head].astype(np.float64)
    err = np.abs(go - ro)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ro)
    # rows a custom mask leaves without keys: lse = -inf on both sides
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(gl), ~fin), f"{tag}{half}: -inf LSE rows differ"
    lerr = np.abs(gl[fin] - rl[fin]) if fin.any() else np.zeros(1)
    msg = f"{tag}{half}: max|out err| {err.max():.3e}, max|lse err| {lerr.max():.3e}"
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{msg}; first bad (token {sel_token[i[0]]}, head {sel_head[i[0]]}, "
                             f"col {i[1]}): gpu {go[i[0], i[1]]} ref {ro[i[0], i[1]]}")
    assert np.all(np.isfinite(go)), msg
    assert lerr.max() <= LSE_ATOL, msg
    return float(err.max()), float(lerr.max())


def sample_rows(h, H, n_tok, seed, include_last=True):
    """Deterministic sample: n_tok tokens (first/last of every request
    included), every head."""
    rng = np.random.default_rng(seed)
    toks = set()
    for r in range(h.batch):
        a, b = int(h.q_indptr[r]), int(h.q_indptr[r + 1])
        if b > a:
            toks.add(a)
            if include_last:
                toks.add(b - 1)
    rest = max(0, n_tok - len(toks))
    if h.rows:
        toks.update(rng.choice(h.rows, size=min(rest, h.rows), replace=False).tolist())
    toks = np.array(sorted(toks), dtype=np.int64)
    sel_token = np.repeat(toks, H)
    sel_head = np.tile(np.arange(H), len(toks))
    return sel_token, sel_head


_SELFTEST = None


def selftest_lib():
    global _SELFTEST
    if _SELFTEST is None:
        import ctypes
        from prefill_decode_paged_pod_gb300 import _build
        out = os.path.join(HERE, "csrc", "_build")
        os.makedirs(out, exist_ok=True)
        so = os.path.join(out, "libumma_selftest.so")
        src = os.path.join(HERE, "csrc", "umma_selftest.cu")
        hdr = os.path.join(_build.CSRC, "pod_device.cuh")
        if (not os.path.exists(so) or os.path.getmtime(so) < os.path.getmtime(src)
                or os.path.getmtime(so) < os.path.getmtime(hdr)):
            cmd = [_build.nvcc()] + _build.ARCH + ["-O2", "-std=c++17", "-shared", "-Xcompiler",
                                                   "-fPIC", "-I", _build.CSRC, src, "-o", so]
            subprocess.check_call(cmd)
        L = ctypes.CDLL(so)
        L.umma_selftest.restype = ctypes.c_int
        L.umma_selftest.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
        L.e4m3_selftest.restype = ctypes.c_int
        L.e4m3_selftest.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
        _SELFTEST = L
    return _SELFTEST
