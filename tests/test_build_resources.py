"""Register budget of the fused kernel (CPU: nvcc cross-compiles for sm_103a).

Two CTAs of 256 threads share an SM, so each thread has at most 128
registers. The decode role runs at that limit; a change that makes the
compiler spill (a value held in registers across the decode loop) costs a
few per cent of decode bandwidth on GB300. This test compiles the
instantiations without a logits transform or RoPE and fails on any spill.
"""
import os
import re
import subprocess

import pytest

from prefill_decode_paged_pod_gb300 import _build


def test_plain_kernels_do_not_spill(tmp_path):
    try:
        cc = _build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    src = os.path.join(_build.CSRC, "pod_k1_plain.cu")
    cmd = [cc] + _build._flags(True) + ["-c", src, "-o", str(tmp_path / "k1.o")]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    entries = re.findall(r"Compiling entry function '([^']+)'.*?(\d+) bytes spill stores, "
                         r"(\d+) bytes spill loads", r.stderr, re.S)
    kernels = [e for e in entries if "pod_kernel" in e[0]]
    assert len(kernels) == 8, r.stderr
    # The FP8-cache instantiations (template flag F8 = true, "Lb1" after the
    # head_dim in the mangled name) hold 16 fp32 logits of a 32-key slice next
    # to the 64 O accumulators and sit at the 128-register cap of two CTAs per
    # SM: a bounded spill is accepted there (the 16-bit kernels must not spill).
    fp8 = [(n, int(st), int(ld)) for n, st, ld in kernels if "Li128ELb1E" in n]
    assert len(fp8) == 2, kernels
    assert all(st <= 256 and ld <= 256 for _, st, ld in fp8), fp8
    spilled = [(name, st, ld) for name, st, ld in kernels
               if "Li128ELb1E" not in name and (int(st) or int(ld))]
    assert not spilled, spilled
