"""GPU parity of the layout and encoding variants against the fp64 oracle:
HND pages, the logits soft cap and ALiBi, and ROPE_LLAMA. The file sorts
after the other GPU tests so that they all run first.
"""
import numpy as np
import pytest
import torch

import prefill_decode_paged_pod_gb300 as pod
from pod_workloads import make_custom
from podtest_util import compare_half, run_pod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_decode_paged_pod_gb300 import _build
    _build.build()
    pod.load_library()


# ------------------------------------------------------------- HND page layout
HND_CASES = [
    # name, dtype, H, Hk, d, ps, causal, window, sinks, p_q, p_kv, d_q, d_kv, layouts (p, d), fp8
    ("h16", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [100, 37], [300, 37], [1, 4], [500, 900],
     ("HND", "HND"), False),
    ("h4", torch.float16, 8, 2, 64, 4, True, 40, False, [70], [150], [1, 2, 1], [33, 64, 90],
     ("HND", "HND"), False),
    ("h3", torch.bfloat16, 8, 8, 128, 3, False, -1, False, [20], [50], [3], [77], ("HND", "HND"), False),
    ("hmix", torch.bfloat16, 32, 8, 128, 16, True, -1, False, [64], [64], [1, 1], [129, 700],
     ("NHD", "HND"), False),
    ("h1", torch.float16, 4, 2, 64, 1, True, -1, False, [64], [64], [1, 1], [17, 29], ("HND", "HND"), False),
    ("h1c", torch.bfloat16, 16, 2, 128, 1, True, -1, False, [80], [200], [2, 1], [300, 129],
     ("HND", "HND"), False),
    ("f8h16", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [33], [33], [1, 4, 2], [700, 300, 64],
     ("HND", "HND"), True),
    ("f8h4", torch.bfloat16, 16, 2, 128, 4, True, -1, False, [], [], [1, 4], [200, 51],
     ("NHD", "HND"), True),
    ("h256", torch.bfloat16, 16, 2, 256, 16, True, -1, True, [100, 37], [300, 37], [1, 4],
     [500, 900], ("HND", "HND"), False),
    ("h256g", torch.float16, 8, 4, 256, 3, True, 60, False, [40], [90], [1, 2], [77, 130],
     ("HND", "HND"), False),
]


@pytest.mark.parametrize("case", HND_CASES, ids=[c[0] for c in HND_CASES])
def test_hnd_layout(case):
    """Caches stored HND ([pages, 2, Hk, ps, d]) on either half: TMA page boxes
    (page_size 16, and contiguous page_size 1 where both layouts are the
    same bytes) and the cp.async gather (page sizes 1, 3 and 4), 16-bit and
    FP8 decode caches."""
    from pod_workloads import with_fp8_decode_cache, with_kv_layout
    name, dt, H, Hk, d, ps, causal, window, sinks, pq, pkv, dq, dkv, (lp, ld), fp8 = case
    inp = make_custom(name, dt, H, Hk, d, ps, causal, window, pq, pkv, dq, dkv, seed=31,
                      sinks=sinks, pages="contig" if name == "h1c" else "perm")
    if lp == "HND":
        inp = with_kv_layout(inp, "HND", "p")
    if ld == "HND":
        inp = with_kv_layout(inp, "HND", "d")
    if fp8:
        inp = with_fp8_decode_cache(inp)
    (op, lp_, od, ld_), h, ws = run_pod(inp)
    compare_half(inp, "p", op, lp_, tag=name + " ")
    compare_half(inp, "d", od, ld_, tag=name + " ")


# ------------------------------------------------------------- logits soft cap and ALiBi
LT_CASES = [
    # name, dtype, H, Hk, d, ps, causal, window, sinks, p_q, p_kv, d_q, d_kv, cap, alibi, num_sms
    ("cap30", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [100, 37], [300, 37], [1, 4],
     [500, 900], 30.0, False, 0),
    ("cap5", torch.float16, 8, 2, 64, 16, False, 64, False, [70], [150], [1, 2, 1], [33, 64, 90],
     5.0, False, 0),
    ("capsplit", torch.bfloat16, 32, 8, 128, 16, True, -1, False, [64], [64], [1, 4], [9000, 12000],
     20.0, False, 16),
    ("alibi", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [100, 37], [300, 37], [1, 4],
     [500, 900], 0.0, True, 0),
    ("alibi64", torch.float16, 8, 8, 64, 1, False, -1, False, [70], [150], [3], [77], 0.0, True, 0),
    ("alibisplit", torch.bfloat16, 32, 8, 128, 16, True, 4096, True, [], [], [1, 4], [9000, 7000],
     0.0, True, 16),
]


@pytest.mark.parametrize("case", LT_CASES, ids=[c[0] for c in LT_CASES])
def test_logits_transform(case):
    """Logits soft cap (cap * tanh(x / cap) of the scaled logit) and ALiBi
    (geometric head slopes, bias slope * (t - p)) on both halves, including
    decode splits merged by the second kernel (few SMs, long keys)."""
    from pod_workloads import alibi_slopes
    name, dt, H, Hk, d, ps, causal, window, sinks, pq, pkv, dq, dkv, cap, alibi, nsm = case
    inp = make_custom(name, dt, H, Hk, d, ps, causal, window, pq, pkv, dq, dkv, seed=41,
                      sinks=sinks)
    inp.soft_cap = cap
    inp.alibi = alibi_slopes(H) if alibi else None
    (op, lp, od, ld), h, ws = run_pod(inp, num_sms=nsm)
    if name.endswith("split"):
        assert pod.plan_summary(h)["n_groups"] > 0, "expected decode splits"
    compare_half(inp, "p", op, lp, tag=name + " ")
    compare_half(inp, "d", od, ld, tag=name + " ")


# ------------------------------------------------------------- ROPE_LLAMA
ROPE_CASES = [
    # name, dtype, H, Hk, d, ps, causal, window, sinks, p_q, p_kv, d_q, d_kv, rope, extra
    ("r16", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [100, 37], [300, 37], [1, 4],
     [500, 900], (1.0, 1e4), {}),
    ("r64nc", torch.float16, 8, 2, 64, 4, False, -1, False, [70], [50], [2, 1], [33, 90],
     (2.0, 500.0), {}),
    ("rhnd", torch.bfloat16, 16, 2, 128, 16, True, 256, False, [64], [64], [1, 2], [700, 300],
     (1.0, 1e4), {"hnd": True, "soft_cap": 30.0}),
    ("rlong", torch.bfloat16, 32, 8, 128, 16, True, -1, False, [], [], [1, 4], [20000, 17000],
     (1.0, 1e6), {"num_sms": 16}),
    ("r1", torch.float16, 4, 2, 64, 1, True, -1, False, [80], [200], [2], [129],
     (4.0, 1e4), {"pages": "contig"}),
]


@pytest.mark.parametrize("case", ROPE_CASES, ids=[c[0] for c in ROPE_CASES])
def test_rope(case):
    """ROPE_LLAMA on both halves through the rotated-copy pre-pass: TMA and
    gather page sizes, a non-causal prefill with more queries than keys
    (negative positions), an HND source cache with a soft cap, positions
    past 16 Ki with decode splits, and contiguous page_size 1."""
    from pod_workloads import with_kv_layout
    name, dt, H, Hk, d, ps, causal, window, sinks, pq, pkv, dq, dkv, rope, extra = case
    inp = make_custom(name, dt, H, Hk, d, ps, causal, window, pq, pkv, dq, dkv, seed=51,
                      sinks=sinks, pages=extra.get("pages", "perm"))
    if extra.get("hnd"):
        inp = with_kv_layout(inp, "HND")
    inp.soft_cap = extra.get("soft_cap", 0.0)
    inp.rope = rope
    (op, lp, od, ld), h, ws = run_pod(inp, num_sms=extra.get("num_sms", 0))
    assert pod.plan_summary(h)["rope"] == 1
    compare_half(inp, "p", op, lp, tag=name + " ")
    compare_half(inp, "d", od, ld, tag=name + " ")
