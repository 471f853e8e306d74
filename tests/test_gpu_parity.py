"""GPU parity: the POD library (through its C-ABI binding) against the fp64
oracle on the same seeded inputs, element by element.

Covers the five benchmark workloads (every row of c1-c5 at full size, and of
the c5 decode half with an FP8 cache), a randomized sweep shaped like the FlashInfer
POD test grid (page size 1/16, GQA groups, decode batches 1/17/127, prefill
lengths that are not tile multiples), edge cases, determinism and the tcgen05
building blocks in isolation.
"""
import numpy as np
import pytest
import torch

import prefill_decode_paged_pod_gb300 as pod
from pod_workloads import make_config, make_custom
from podtest_util import compare_half, run_pod, sample_rows, selftest_lib, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from prefill_decode_paged_pod_gb300 import _build
    _build.build()
    pod.load_library()


# ------------------------------------------------------------- building blocks
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bf16", [0, 1])
@pytest.mark.parametrize("variant", [0, 1, 2])
def test_umma_building_blocks(d, bf16, variant):
    L = selftest_lib()
    dt = torch.bfloat16 if bf16 else torch.float16
    g = torch.Generator().manual_seed(7 + d + bf16)
    q = torch.randn(128, d, generator=g).to(dt).cuda()
    k = torch.randn(64, d, generator=g).to(dt).cuda()
    v = torch.randn(64, d, generator=g).to(dt).cuda()
    p = torch.rand(128, 64, generator=g).to(dt).cuda()
    s = torch.zeros(128, 64, device="cuda")
    o = torch.zeros(128, d, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.umma_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), p.data_ptr(), s.data_ptr(),
                         o.data_ptr(), d, bf16, variant, st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    s_ref = q.float() @ k.float().T
    o_ref = p.float() @ v.float()
    assert torch.allclose(s, s_ref, atol=1e-2, rtol=1e-3), (s - s_ref).abs().max()
    assert torch.allclose(o, o_ref, atol=1e-2, rtol=1e-3), (o - o_ref).abs().max()


# ------------------------------------------------------------- workloads
@pytest.mark.parametrize("name", ["c1", "c2"])
def test_config_full(name):
    inp = make_config(name)
    (op, lp, od, ld), h, ws = run_pod(inp)
    assert op.shape == (inp.p.rows, inp.num_qo_heads, inp.head_dim)
    assert od.shape == (inp.d.rows, inp.num_qo_heads, inp.head_dim)
    compare_half(inp, "p", op, lp, tag=name)
    compare_half(inp, "d", od, ld, tag=name)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["c3", "c4", "c5"])
def test_config_full_size(name):
    """Every output row and LSE of both halves of c3-c5 at full size, in the
    launch configuration the benchmark times, against the fp64 oracle element
    by element (the oracle takes about half a minute for c5 on 16 host
    cores)."""
    inp = make_config(name)
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "p", op, lp, tag=name)
    compare_half(inp, "d", od, ld, tag=name)
    assert np.isfinite(op).all() and np.isfinite(od).all()
    assert np.isfinite(lp).all() and np.isfinite(ld).all()


# ------------------------------------------------------------- sweep (M1-like)
SWEEP = []
for ps in (1, 16):
    for G in (1, 4, 8):
        for db in (1, 17, 127):
            SWEEP.append((ps, G, db))


@pytest.mark.parametrize("ps,G,db", SWEEP)
def test_sweep(ps, G, db):
    rng = np.random.default_rng(ps * 1000 + G * 10 + db)
    Hk = 2
    d = int(rng.choice([64, 128]))
    dt = torch.bfloat16 if rng.integers(0, 2) else torch.float16
    window = int(rng.choice([-1, -1, 37, 300]))
    sinks = bool(rng.integers(0, 2))
    pl = [int(x) for x in rng.choice([1, 127, 300], size=int(rng.integers(1, 3)))]
    pkv = [q + int(rng.integers(0, 200)) for q in pl]
    dkv = [int(x) for x in rng.integers(1, 700, size=db)]
    dq = [int(min(k, rng.choice([1, 1, 3]))) for k in dkv]
    inp = make_custom("sweep", dt, G * Hk, Hk, d, ps, True, window, pl, pkv, dq, dkv,
                      seed=int(rng.integers(0, 1 << 30)), sinks=sinks, extra_pages=3)
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "p", op, lp, tag=f"ps{ps} G{G} db{db} d{d} w{window} ")
    compare_half(inp, "d", od, ld, tag=f"ps{ps} G{G} db{db} d{d} w{window} ")


@pytest.mark.parametrize("ps,pages", [(1, "contig"), (2, "contig"), (4, "perm"), (3, "perm"),
                                      (8, "perm"), (32, "perm"), (128, "perm")])
def test_page_layouts(ps, pages):
    """Every page geometry: TMA page boxes (ps >= 8), TMA runs of consecutive
    pages (ps 1 both halves, ps 2 prefill only), and the cp.async gather (ps 3,
    ps 4 permuted, ps 2 decode)."""
    inp = make_custom("pl", torch.bfloat16, 16, 2, 128, ps, True, -1, [130, 67], [200, 67],
                      [1, 3, 1, 2], [1000, 517, 96, 33], seed=ps, sinks=True, pages=pages,
                      extra_pages=5)
    (op, lp, od, ld), h, ws = run_pod(inp)
    s = pod.plan_summary(h)
    assert bool(s["p_tma"]) == (ps in (1, 2, 8, 32, 128)), s
    assert bool(s["d_tma"]) == (ps in (1, 8, 32, 128)), s  # decode boxes: ps 1 runs or ps >= 8
    compare_half(inp, "p", op, lp, tag=f"ps{ps} ")
    compare_half(inp, "d", od, ld, tag=f"ps{ps} ")


def test_unused_page_slots_do_not_leak():
    """Slots past kv_len in a request's last page hold non-finite values; TMA
    copies whole pages, so the kernels must keep them out of the result."""
    inp = make_custom("nan", torch.float16, 16, 2, 64, 16, True, -1, [40, 7], [45, 7],
                      [1, 2], [37, 70], seed=3, pages="perm")
    for h in (inp.p, inp.d):
        for r in range(h.batch):
            last = int(h.kv_indices[h.kv_indptr[r + 1] - 1])
            n = int(h.last_page_len[r])
            h.kv[last, :, n:] = float("nan")
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "p", op, lp)
    compare_half(inp, "d", od, ld)


@pytest.mark.parametrize("causal", [True, False])
def test_non_causal_and_long_decode_split(causal):
    """Long decode KV on few SMs forces split chunks and the merge kernel."""
    inp = make_custom("split", torch.bfloat16, 16, 2, 128, 16, causal, -1, [40], [300],
                      [1, 2, 1], [5000, 7000, 3000], seed=11, sinks=True)
    (op, lp, od, ld), h, ws = run_pod(inp, num_sms=4)
    s = pod.plan_summary(h)
    assert s["n_groups"] > 0, s
    compare_half(inp, "p", op, lp)
    compare_half(inp, "d", od, ld)


# ------------------------------------------------------------- edge cases
def test_empty_prefill_half():
    inp = make_custom("ed", torch.float16, 8, 2, 128, 16, True, -1, [], [], [1, 1], [33, 1], seed=3)
    (op, lp, od, ld), h, ws = run_pod(inp)
    assert op.shape[0] == 0
    compare_half(inp, "d", od, ld)


def test_empty_decode_half():
    inp = make_custom("ep", torch.bfloat16, 8, 8, 64, 1, True, 5, [65, 3], [70, 3], [], [], seed=4)
    (op, lp, od, ld), h, ws = run_pod(inp)
    assert od.shape[0] == 0
    compare_half(inp, "p", op, lp)


def test_zero_length_requests_and_tiny_kv():
    # request 1 of each half has no queries; kv_len == 1 and kv_len == q_len cases
    inp = make_custom("z", torch.float16, 4, 1, 64, 4, True, 0, [1, 0, 5], [1, 4, 5],
                      [1, 0, 1], [1, 2, 9], seed=5, sinks=True)
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "p", op, lp)
    compare_half(inp, "d", od, ld)


def test_determinism():
    inp = make_config("c1")
    r1, h, ws = run_pod(inp)
    r2, _, _ = run_pod(inp)
    for x, y in zip(r1, r2):
        assert np.array_equal(x, y)


def test_run_many_times_one_plan():
    """plan once, run many (the walkthrough's per-layer reuse)."""
    inp = make_config("c1")
    dev = to_dev(inp)
    (op, lp, od, ld), h, ws = run_pod(inp, dev=dev, repeat=5)
    compare_half(inp, "p", op, lp)
    compare_half(inp, "d", od, ld)


def test_cuda_graph_capture_and_replan_in_place():
    """pod_run captured in a CUDA graph, then the graph replayed after a new
    plan was written into the same workspace: same lengths, a different page
    permutation and new cache contents in the same buffers (the serving loop's
    fixed-batch mode: plan outside the graph, replay inside it)."""
    def inputs(seed):
        return make_custom("graph", torch.bfloat16, 16, 2, 128, 16, True, -1, [77, 300], [90, 300],
                           [1, 4, 1, 2, 1], [1000, 517, 96, 33, 2500], seed=seed, sinks=True)
    a, b = inputs(21), inputs(22)
    assert not np.array_equal(a.d.kv_indices, b.d.kv_indices)
    dev = to_dev(a)
    h = pod.plan_inputs(a)
    ws = torch.empty(pod.pod_workspace_size(h), dtype=torch.uint8, device="cuda")
    pod.pod_bind_workspace(h, ws)
    H, d = a.num_qo_heads, a.head_dim
    outs = dict(out_p=torch.empty((a.p.rows, H, d), dtype=a.dtype, device="cuda"),
                lse_p=torch.empty((a.p.rows, H), dtype=torch.float32, device="cuda"),
                out_d=torch.empty((a.d.rows, H, d), dtype=a.dtype, device="cuda"),
                lse_d=torch.empty((a.d.rows, H), dtype=torch.float32, device="cuda"))

    def run():
        pod.pod_run(h, dev["q_p"], dev["kv_p"], dev["q_d"], dev["kv_d"], ws, sinks=dev["sinks"],
                    **outs)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()  # warm-up outside the capture (function attributes, tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for inp in (a, b):
        if inp is b:
            # new contents in the captured buffers, new tables in the same workspace
            for k, t in (("q_p", b.p.q), ("kv_p", b.p.kv), ("q_d", b.d.q), ("kv_d", b.d.kv),
                         ("sinks", b.sinks)):
                dev[k].copy_(t.to("cuda"))
            h2 = pod.plan_inputs(b, workspace=ws)
            assert pod.pod_workspace_size(h2) == pod.pod_workspace_size(h)
            for which in (0, 1, 8, 9):
                assert np.array_equal(pod.pod_plan_table(h2, which), pod.pod_plan_table(h, which))
            torch.cuda.synchronize()
        for o in outs.values():
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pod.pod_read_device_status(h, ws) == 0
        op, lp, od, ld = [outs[k].double().cpu().numpy() for k in ("out_p", "lse_p", "out_d", "lse_d")]
        compare_half(inp, "p", op, lp, tag="graph ")
        compare_half(inp, "d", od, ld, tag="graph ")


# ------------------------------------------------------------- FP8 decode cache
def test_e4m3_widening_against_torch():
    """The decode path's E4M3 -> fp16 / bf16 widening, on every pair of codes
    (NaN codes excepted), against torch's conversion."""
    L = selftest_lib()
    pairs = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    codes = pairs.view(torch.uint8).reshape(-1, 2)           # low byte first
    src = pairs.cuda()
    out_h = torch.empty(65536, dtype=torch.int32, device="cuda")
    out_b = torch.empty(65536, dtype=torch.int32, device="cuda")
    assert L.e4m3_selftest(src.data_ptr(), out_h.data_ptr(), out_b.data_ptr(), 65536) == 0
    f8 = codes.contiguous().view(torch.float8_e4m3fn)
    ref = f8.float()
    gh = out_h.cpu().view(torch.float16).reshape(-1, 2).float()
    gb = out_b.cpu().view(torch.bfloat16).reshape(-1, 2).float()
    live = ~torch.isnan(ref)
    assert torch.equal(gh[live], ref[live]) and torch.equal(gb[live], ref[live])
    assert torch.isnan(gh[~live]).all() and torch.isnan(gb[~live]).all()


FP8_CASES = [
    # ps, pages, G, Hk, decode q_len, dtype, window, sinks, num_sms
    (16, "perm", 8, 2, 4, torch.bfloat16, 4096, True, 0),     # TMA page boxes, 32-row items
    (16, "perm", 4, 2, 1, torch.float16, -1, False, 0),
    (1, "contig", 4, 2, 1, torch.bfloat16, -1, True, 0),       # TMA runs of pages
    (3, "perm", 2, 2, 2, torch.bfloat16, 37, True, 0),         # cp.async gather
    (16, "perm", 8, 2, 1, torch.bfloat16, -1, True, 4),        # split KV + merge
    (32, "perm", 4, 1, 3, torch.float16, 300, False, 0),
    (32, "perm", 4, 1, 3, torch.float16, -1, False, 4),
]


@pytest.mark.parametrize("ps,pages,G,Hk,ql,dt,window,sinks,nsm", FP8_CASES)
def test_fp8_decode_cache(ps, pages, G, Hk, ql, dt, window, sinks, nsm):
    from pod_workloads import with_fp8_decode_cache
    rng = np.random.default_rng(ps * 100 + G * 10 + ql)
    if nsm:   # few long requests on few SMs: the plan splits their keys
        dkv = [9000, 12000, 7000]
    else:
        dkv = [int(x) for x in rng.integers(ql, 3000, size=9)]
    base = make_custom("fp8", dt, G * Hk, Hk, 128, ps, True, window, [70], [90], [ql] * len(dkv),
                       dkv, seed=ps + G, sinks=sinks, pages=pages, extra_pages=2)
    inp = with_fp8_decode_cache(base, k_scale=0.05, v_scale=0.02)
    (op, lp, od, ld), h, ws = run_pod(inp, num_sms=nsm)
    s = pod.plan_summary(h)
    if nsm:
        assert s["n_groups"] > 0, s
    compare_half(inp, "p", op, lp, tag="fp8 ")
    compare_half(inp, "d", od, ld, tag=f"fp8 ps{ps} G{G} q{ql} ")


def test_fp8_unused_page_slots_do_not_leak():
    """E4M3 NaN codes in the unused slots of the last pages stay out."""
    from pod_workloads import with_fp8_decode_cache
    base = make_custom("nan8", torch.bfloat16, 16, 2, 128, 16, True, -1, [20], [20],
                       [1, 2, 1], [37, 70, 5], seed=9, pages="perm")
    inp = with_fp8_decode_cache(base, k_scale=0.1, v_scale=0.1)
    raw = inp.d.kv.view(torch.uint8)
    for r in range(inp.d.batch):
        last = int(inp.d.kv_indices[inp.d.kv_indptr[r + 1] - 1])
        raw[last, :, int(inp.d.last_page_len[r]):] = 0x7F
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "d", od, ld, tag="fp8 nan ")


@pytest.mark.slow
def test_fp8_decode_c5_full_size():
    """The FP8 (E4M3) decode cache on c5 at full size: every decode row."""
    from pod_workloads import with_fp8_decode_cache
    inp = with_fp8_decode_cache(make_config("c5"), k_scale=0.05, v_scale=0.05)
    (op, lp, od, ld), h, ws = run_pod(inp)
    compare_half(inp, "d", od, ld, tag="fp8 c5 ")
    assert np.isfinite(od).all() and np.isfinite(ld).all()


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_key_split_and_merge(causal):
    """A small prefill half (few tiles, long keys) is split along the keys
    and merged (half-0 merge groups), next to a decode half."""
    inp = make_custom("psplit", torch.bfloat16, 16, 2, 128, 16, causal, -1, [200, 37], [3000, 1200],
                      [1, 2], [500, 900], seed=13, sinks=True)
    (op, lp, od, ld), h, ws = run_pod(inp)
    groups = pod.pod_plan_table(h, 5).reshape(-1, 8)
    assert np.any(groups[:, 0] == 0), "expected a prefill key split"
    compare_half(inp, "p", op, lp, tag="psplit ")
    compare_half(inp, "d", od, ld, tag="psplit ")


def test_prefill_alone_split_at_c4_shape():
    """c4's prefill half alone (32/8/128/16, 512 rows against 8192 keys):
    every one of its 128 tiles is split along the keys and merged."""
    inp = make_custom("p4", torch.bfloat16, 32, 8, 128, 16, True, -1, [512], [8192], [], [], seed=14)
    (op, lp, od, ld), h, ws = run_pod(inp)
    groups = pod.pod_plan_table(h, 5).reshape(-1, 8)
    assert int((groups[:, 0] == 0).sum()) == 128
    st, sh = sample_rows(inp.p, inp.num_qo_heads, 64, seed=5)
    compare_half(inp, "p", op, lp, st, sh, tag="p4 ")
    assert np.isfinite(op).all() and np.isfinite(lp).all()


# ------------------------------------------------------------- custom prefill mask
MASK_CASES = [
    # name, dtype, H, Hk, d, ps, causal, window, sinks, p_q, p_kv, d_q, d_kv
    ("mA", torch.float16, 8, 2, 128, 16, True, -1, False, [100, 37], [300, 37], [1, 2], [50, 60]),
    ("mB", torch.bfloat16, 16, 2, 128, 1, True, 64, True, [200], [900], [4], [500]),
    ("mC", torch.bfloat16, 4, 4, 64, 16, False, -1, True, [130, 1], [130, 260], [], []),
    ("mD", torch.bfloat16, 16, 2, 128, 16, True, -1, True, [40], [6000], [1], [30]),
]


@pytest.mark.parametrize("case", MASK_CASES, ids=[c[0] for c in MASK_CASES])
def test_custom_prefill_mask(case):
    """A packed custom mask on the prefill half (random bits plus a row with
    no key and a row with every key in each request), next to a decode half
    that keeps the causal rule. mD is a small prefill with long keys whose
    tiles the planner splits: merged partials of rows that some chunks
    leave empty."""
    from pod_workloads import with_prefill_custom_mask
    name, dt, H, Hk, d, ps, causal, window, sinks, pq, pkv, dq, dkv = case
    inp = make_custom(name, dt, H, Hk, d, ps, causal, window, pq, pkv, dq, dkv, seed=21,
                      sinks=sinks)
    inp = with_prefill_custom_mask(inp, seed=22, density=0.5)
    (op, lp, od, ld), h, ws = run_pod(inp)
    assert pod.plan_summary(h)["p_mask"] == 1
    if name == "mD":
        groups = pod.pod_plan_table(h, 5).reshape(-1, 8)
        assert np.any(groups[:, 0] == 0), "expected a prefill key split"
    compare_half(inp, "p", op, lp, tag=name + " ")
    compare_half(inp, "d", od, ld, tag=name + " ")
    # the first row of every request allows no key: out = 0, lse = -inf
    first = inp.p.q_indptr[:-1][np.diff(inp.p.q_indptr) > 2]
    assert np.all(op[first] == 0.0) and np.all(np.isneginf(lp[first]))



# ------------------------------------------------------------- head_dim 256
D256_CASES = [
    # name, dtype, H, Hk, ps, causal, window, sinks, p_q, p_kv, d_q, d_kv, pages, num_sms
    ("b16", torch.bfloat16, 16, 2, 16, True, -1, True, [300, 33], [300, 40], [1, 4, 1],
     [900, 77, 2000], "perm", 0),
    ("f8g", torch.float16, 64, 8, 16, True, 500, False, [129], [700], [1, 1, 3], [1500, 64, 300],
     "perm", 0),
    ("mha1", torch.bfloat16, 4, 4, 1, False, -1, True, [70], [90], [2, 1], [400, 17], "contig", 0),
    ("gather", torch.float16, 8, 2, 3, True, -1, False, [50], [80], [1, 2], [250, 33], "perm", 0),
    ("split", torch.bfloat16, 16, 2, 16, True, -1, True, [40], [300], [1, 4], [6000, 9000],
     "perm", 8),
]


@pytest.mark.parametrize("case", D256_CASES, ids=[c[0] for c in D256_CASES])
def test_head_dim_256(case):
    """head_dim 256 on both halves (one CTA per SM, O over 256 TMEM columns,
    PV at N = 256): GQA groups 2, 8 and MHA, page boxes, runs of single-token
    pages and the cp.async gather (page size 3), windows, sinks, and decode
    splits merged by the second kernel."""
    name, dt, H, Hk, ps, causal, window, sinks, pq, pkv, dq, dkv, pages, nsm = case
    inp = make_custom(name, dt, H, Hk, 256, ps, causal, window, pq, pkv, dq, dkv, seed=61,
                      sinks=sinks, pages=pages, extra_pages=3)
    (op, lp, od, ld), h, ws = run_pod(inp, num_sms=nsm)
    if name == "split":
        assert pod.plan_summary(h)["n_groups"] > 0, "expected decode splits"
    compare_half(inp, "p", op, lp, tag=name + " ")
    compare_half(inp, "d", od, ld, tag=name + " ")
