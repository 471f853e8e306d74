"""CPU tests of the C-ABI library: it loads, exports every declared symbol, and
its host planner matches the plain restatement in oracle/planner_ref.py bit for
bit. No GPU is needed: plans are made host-only (workspace NULL, num_sms given).
"""
import copy
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
from oracle import planner_ref
import prefill_decode_paged_pod_gb300 as pod
from prefill_decode_paged_pod_gb300 import _build
from pod_workloads import make_config, make_custom

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REC = 8


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pod.load_library()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pod.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pod_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert "pod_plan" in syms and "pod_run" in syms and len(syms) >= 8
    for s in syms:
        assert hasattr(lib, s), f"{s} is declared in include/pod.h but not exported"


def plan_host(inp, num_sms=152):
    return pod.plan_inputs(inp, workspace=None, num_sms=num_sms)


def check_against_reference(inp, h):
    s = pod.plan_summary(h)
    # kv_len: library == oracle C == python restatement
    for half, which in (("p", 6), ("d", 7)):
        hh = inp.p if half == "p" else inp.d
        got = pod.pod_plan_table(h, which)
        if hh.batch == 0:
            continue
        assert np.array_equal(got, oracle.seq_lens(hh.kv_indptr, hh.last_page_len, inp.page_size))
        assert np.array_equal(got, planner_ref.seq_lens(hh.kv_indptr, hh.last_page_len, inp.page_size))
    H, Hk = inp.num_qo_heads, inp.num_kv_heads
    kvl_p = planner_ref.seq_lens(inp.p.kv_indptr, inp.p.last_page_len, inp.page_size)
    kvl_d = planner_ref.seq_lens(inp.d.kv_indptr, inp.d.last_page_len, inp.page_size)
    G = H // Hk
    groups = pod.pod_plan_table(h, 5).reshape(-1, REC)
    # prefill tiles: in the restated order; per tile, the chunks partition
    # [lo, hi) in order (one chunk unless the planner split it, then with a
    # merge group of half 0)
    tiles = pod.pod_plan_table(h, 1).reshape(-1, REC)
    # a custom mask replaces the causal rule on the prefill half
    p_causal = inp.causal and getattr(inp.p, "packed_mask", None) is None
    ref = planner_ref.prefill_tiles(inp.p.q_indptr, kvl_p, H, Hk, p_causal, inp.window_left)
    i = 0
    gi = 0
    prows = 0
    for (r, g, t0, nt, lo, hi) in ref:
        start = i
        k = lo
        while i < len(tiles) and tuple(tiles[i, :4]) == (r, g, t0, nt) and tiles[i, 4] == k:
            assert tiles[i, 5] > tiles[i, 4] or lo == hi
            k = int(tiles[i, 5])
            i += 1
            if k == hi:
                break
        assert k == hi and i > start, f"tile {(r, g, t0, nt, lo, hi)} not covered"
        n = i - start
        assert all(int(tiles[j, 4]) % 64 == 0 for j in range(start + 1, i))
        if n == 1:
            assert tiles[start, 6] == -1
        else:
            R = nt * G
            assert tuple(groups[gi]) == (0, r, g, t0, nt, prows, n, R)
            for j in range(n):
                assert tiles[start + j, 6] == prows + j * R
            prows += n * R
            gi += 1
    assert i == len(tiles) == s["n_tiles"]
    # decode items: per unit, the chunks partition [lo, hi) in order
    items = pod.pod_plan_table(h, 2).reshape(-1, REC)
    units = planner_ref.decode_units(inp.d.q_indptr, kvl_d, H, Hk, inp.causal, inp.window_left)
    i = 0
    for (r, g, t0, nt, lo, hi) in units:
        start = i
        k = lo
        while i < len(items) and tuple(items[i, :4]) == (r, g, t0, nt) and items[i, 4] == k:
            assert items[i, 5] > items[i, 4]
            k = int(items[i, 5])
            i += 1
            if k == hi:
                break
        assert k == hi, f"unit {(r, g, t0, nt, lo, hi)} not covered"
        n = i - start
        inner = [int(items[j, 4]) for j in range(start + 1, i)]
        assert all(b % 64 == 0 for b in inner)
        if n == 1:
            assert items[start, 6] == -1
        else:
            R = nt * G
            assert tuple(groups[gi]) == (1, r, g, t0, nt, prows, n, R)
            for j in range(n):
                assert items[start + j, 6] == prows + j * R
            prows += n * R
            gi += 1
    assert i == len(items) == s["n_items"]
    assert gi == len(groups) == s["n_groups"]
    assert prows == s["n_prows"]
    # CTA lists: every record exactly once, prefill CTAs first
    ptr = pod.pod_plan_table(h, 3)
    lst = pod.pod_plan_table(h, 4)
    npc, ndc = s["n_p_ctas"], s["n_d_ctas"]
    assert len(ptr) == s["grid"] + 1 and s["grid"] == npc + ndc
    assert sorted(lst[: ptr[npc]].tolist()) == list(range(s["n_tiles"]))
    assert sorted(lst[ptr[npc]:].tolist()) == list(range(s["n_items"]))
    assert s["grid"] <= 2 * s["num_sms"]
    # work queues: each a permutation of its records (the kernel serves both
    # through atomic counters, so every record runs exactly once)
    assert sorted(pod.pod_plan_table(h, 8).tolist()) == list(range(s["n_tiles"]))
    dq = pod.pod_plan_table(h, 9)
    assert sorted(dq.tolist()) == list(range(s["n_items"]))
    # decode queue records: the item record, then its request's fields, in queue order
    dqrec = pod.pod_plan_table(h, 10).reshape(-1, 16)
    assert dqrec.shape[0] == s["n_items"]
    if len(dq):
        assert np.array_equal(dqrec[:, :REC], items[dq])
        r = dqrec[:, 0]
        d = inp.d
        assert np.array_equal(dqrec[:, 8], kvl_d[r])
        assert np.array_equal(dqrec[:, 9], d.q_indptr[r])
        assert np.array_equal(dqrec[:, 10], d.q_indptr[r + 1] - d.q_indptr[r])
        assert np.array_equal(dqrec[:, 11], d.kv_indptr[r])
        assert np.array_equal(dqrec[:, 12], d.kv_indptr[r + 1] - d.kv_indptr[r])
        assert np.all(dqrec[:, 13:] == 0)
    return s


@pytest.mark.parametrize("name", ["c1", "c2"])
def test_planner_small_configs(lib, name):
    inp = make_config(name)
    h = plan_host(inp)
    s = check_against_reference(inp, h)
    assert s["p_rows"] == inp.p.rows and s["d_rows"] == inp.d.rows
    pod.pod_destroy(h)


def test_planner_docstring_kv_lens(lib):
    inp = make_config("c2")
    h = plan_host(inp)
    assert pod.pod_plan_table(h, 7).tolist() == [257, 183, 238, 52, 275, 529, 448]


@pytest.mark.parametrize("seed", range(8))
def test_planner_random(lib, seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 8]))
    Hk = int(rng.choice([1, 2, 8]))
    ps = int(rng.choice([1, 3, 16]))
    causal = bool(rng.integers(0, 2))
    window = int(rng.choice([-1, 0, 100, 4096]))
    pb, db = int(rng.integers(0, 4)), int(rng.integers(0, 40))
    pkv = rng.integers(1, 3000, size=pb)
    pq = [int(rng.integers(1, k + 1)) if causal else int(rng.integers(1, 3000)) for k in pkv]
    dkv = rng.integers(5, 20000, size=db)
    dq = [int(rng.integers(1, min(5, k) + 1)) for k in dkv]
    inp = make_custom("r", torch.float16, G * Hk, Hk, 64, ps, causal, window, pq, pkv, dq, dkv,
                      seed=seed)
    h = plan_host(inp, num_sms=int(rng.choice([8, 152])))
    check_against_reference(inp, h)


def test_planner_deterministic(lib):
    inp = make_config("c1")
    a = plan_host(inp)
    b = plan_host(inp)
    for w in range(6):
        assert np.array_equal(pod.pod_plan_table(a, w), pod.pod_plan_table(b, w))


def test_planner_large_configs_host_only(lib):
    # c4: 256 decode requests of U[512,16384] keys; plan must split decode KV
    inp = make_config("c4")
    h = plan_host(inp)
    s = check_against_reference(inp, h)
    assert s["n_items"] >= s["n_d_ctas"] > 0 and s["n_p_ctas"] > 0


def _bad(lib, **over):
    inp = make_custom("v", torch.float16, 4, 2, 64, 4, True, -1, [3], [5], [1, 1], [6, 9], seed=0)
    args = dict(p_q_indptr=inp.p.q_indptr, p_kv_indptr=inp.p.kv_indptr, p_kv_indices=inp.p.kv_indices,
                p_last_page_len=inp.p.last_page_len, d_q_indptr=inp.d.q_indptr,
                d_kv_indptr=inp.d.kv_indptr, d_kv_indices=inp.d.kv_indices,
                d_last_page_len=inp.d.last_page_len, num_qo_heads=4, num_kv_heads=2, head_dim=64,
                page_size=4, causal=True, window_left=-1, sm_scale=None, dtype=torch.float16,
                p_num_pages=inp.p.num_pages, d_num_pages=inp.d.num_pages, num_sms=4)
    args.update(over)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan(**args)
    return e.value.code


def test_plan_error_codes(lib):
    assert _bad(lib, num_qo_heads=5) == 1                      # H % Hk != 0
    assert _bad(lib, head_dim=96) == 2                         # unsupported head_dim
    assert _bad(lib, d_last_page_len=np.array([5, 1])) == 1    # last_page_len > page_size
    assert _bad(lib, d_last_page_len=np.array([0, 1])) == 1    # last_page_len < 1
    assert _bad(lib, d_kv_indices=np.array([0, 1, 99])) == 1   # page outside the pool
    assert _bad(lib, d_q_indptr=np.array([0, 2, 1])) == 1      # non-monotone indptr
    assert _bad(lib, p_q_indptr=np.array([0, 9])) == 1         # kv_len < q_len under causal
    assert _bad(lib, num_qo_heads=256, num_kv_heads=1) == 2    # group > 128
    assert _bad(lib, num_qo_heads=128, num_kv_heads=2) == 2    # decode group > 32
    assert _bad(lib, window_left=-2) == 1


def test_reference_validation_agrees(lib):
    """The restated validation rules reject exactly what the library rejects."""
    rng = np.random.default_rng(3)
    for trial in range(40):
        b = int(rng.integers(1, 4))
        ps = int(rng.choice([1, 4]))
        q_indptr = np.concatenate([[0], np.cumsum(rng.integers(0, 4, size=b))]).astype(np.int32)
        kv_indptr = np.concatenate([[0], np.cumsum(rng.integers(0, 3, size=b))]).astype(np.int32)
        last = rng.integers(0, ps + 2, size=b).astype(np.int32)
        npages = 6
        idx = rng.integers(-1, npages + 1, size=int(kv_indptr[-1])).astype(np.int32)
        reason = planner_ref.validate_half(q_indptr, kv_indptr, idx, last, npages, ps, True)
        ok = True
        try:
            pod.pod_plan(None, None, None, None, q_indptr, kv_indptr, idx, last, 2, 1, 64, ps,
                         True, -1, None, dtype=torch.float16, p_num_pages=1, d_num_pages=npages,
                         num_sms=4)
        except pod.PodError as e:
            ok = False
            assert e.code == 1
        assert ok == (reason is None), (trial, reason)


def test_decode_fp8_switch_host_checks(lib):
    """pod_plan_set_decode_fp8 accepts head_dim 128 with positive scales and
    refuses the rest with the documented codes (host-only plans)."""
    from pod_workloads import with_fp8_decode_cache
    inp = with_fp8_decode_cache(make_custom("f8", torch.bfloat16, 16, 2, 128, 16, True, -1, [5], [9],
                                            [1, 2], [40, 70], seed=1))
    h = plan_host(inp, num_sms=4)
    pod.pod_plan_set_decode_fp8(h, 0.5, 2.0)
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(pod.PodError) as e:
            pod.pod_plan_set_decode_fp8(h, ks, vs)
        assert e.value.code == 1
    inp64 = make_custom("f8", torch.bfloat16, 16, 2, 64, 16, True, -1, [5], [9], [1], [40], seed=1)
    h64 = plan_host(inp64, num_sms=4)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_decode_fp8(h64, 1.0, 1.0)
    assert e.value.code == 2


def _without_decode(inp):
    sub = copy.copy(inp)
    empty = copy.copy(inp.d)
    empty.q_indptr = np.zeros(1, np.int32)
    empty.kv_indptr = np.zeros(1, np.int32)
    empty.kv_indices = np.zeros(0, np.int32)
    empty.last_page_len = np.zeros(0, np.int32)
    sub.d = empty
    return sub


def test_small_prefill_alone_is_split_and_starts_at_once(lib):
    """c4's prefill half alone: 512 rows (below the 1536-row colocation
    cutoff) in 128 tiles of 8192 keys, whose longest tile outlasts the
    balanced makespan. The planner splits every tile's key range into chunks
    merged like decode splits (half-0 merge groups), so that the grid has
    about one prefill job per CTA."""
    h = plan_host(_without_decode(make_config("c4", with_data=False)))
    s = pod.plan_summary(h)
    groups = pod.pod_plan_table(h, 5).reshape(-1, REC)
    pgroups = groups[groups[:, 0] == 0]
    assert len(pgroups) == 128 and np.all(pgroups[:, 6] >= 2), s
    assert s["n_tiles"] == int(pgroups[:, 6].sum()) and s["n_p_ctas"] >= s["num_sms"], s


def test_small_prefill_next_to_long_decode_is_not_split(lib):
    """c4 fused: the decode stream (about 9 GB) sets the makespan and the
    unsplit 8192-key tiles finish well inside it, so a split would only add
    the merge. Every long tile still gets a CTA that starts on it."""
    h = plan_host(make_config("c4", with_data=False))
    s = pod.plan_summary(h)
    groups = pod.pod_plan_table(h, 5).reshape(-1, REC)
    assert not np.any(groups[:, 0] == 0) if len(groups) else True
    assert s["n_tiles"] == 128 and s["n_p_ctas"] >= 128, s
    assert s["grid"] <= 2 * s["num_sms"] and s["n_d_ctas"] > 0


def test_large_prefill_is_not_split(lib):
    """c3 and c5 have more than 1536 prefill rows: no prefill merge group."""
    for name in ("c3", "c5"):
        h = plan_host(make_config(name, with_data=False))
        groups = pod.pod_plan_table(h, 5).reshape(-1, REC)
        assert not np.any(groups[:, 0] == 0) if len(groups) else True


def test_split_follows_decode_item_width(lib):
    """The split depends on how decode CTAs share an SM with prefill CTAs.
    c5's decode items have 32 rows (both m-tiles, all 8 decode warps busy),
    and a decode CTA next to a prefill CTA is measured 11 % slower: the plan
    starts nearly every CTA on decode and lets them cross to the prefill
    queue afterwards. c3's items have 8 rows (half the decode warps idle):
    the split stays near the CTA-time balance (a quarter to a half of the
    grid starts on prefill). Every CTA has work in both (grid = 2 x SMs)."""
    for name, lo, hi in (("c5", 1, 0.1), ("c3", 0.25, 0.5)):
        h = plan_host(make_config(name, with_data=False))
        s = pod.plan_summary(h)
        assert s["grid"] == 2 * s["num_sms"], s
        assert lo * (s["grid"] if lo < 1 else 1) <= s["n_p_ctas"] <= hi * s["grid"], (name, s)


# ------------------------------------------------------------- custom prefill mask
def _mask_offsets(inp):
    ql = np.diff(inp.p.q_indptr).astype(np.int64)
    kvl = planner_ref.seq_lens(inp.p.kv_indptr, inp.p.last_page_len, inp.page_size).astype(np.int64)
    return np.concatenate([[0], np.cumsum(ql * kvl)])


@pytest.mark.parametrize("seed", range(4))
def test_custom_mask_plan(lib, seed):
    """With a custom mask the prefill tiles span every key the window allows
    (the restated planner run non-causal on that half), the decode half keeps
    the causal rule, and plan table 11 holds each request's first mask bit."""
    from pod_workloads import with_prefill_custom_mask
    rng = np.random.default_rng(100 + seed)
    window = int(rng.choice([-1, 50]))
    pkv = rng.integers(1, 900, size=int(rng.integers(1, 4)))
    pq = [int(rng.integers(1, k + 1)) for k in pkv]
    inp = make_custom("m", torch.bfloat16, 16, 2, 128, int(rng.choice([1, 16])), True, window,
                      pq, pkv, [1, 3], [300, 40], seed=seed)
    inp = with_prefill_custom_mask(inp, seed=seed)
    h = plan_host(inp, num_sms=int(rng.choice([8, 152])))
    s = check_against_reference(inp, h)
    assert s["p_mask"] == 1 and s["causal"] == 1
    off = pod.pod_plan_table(h, 11).view(np.int64)
    assert np.array_equal(off, _mask_offsets(inp))
    # removing the mask gives the causal plan back
    pod.pod_plan_set_prefill_mask(h, None)
    inp.p.packed_mask = None
    s = check_against_reference(inp, h)
    assert s["p_mask"] == 0 and len(pod.pod_plan_table(h, 11)) == 0


def test_custom_mask_host_checks(lib):
    """A mask shorter than the prefill requests' bits is refused; switching
    the mask on releases the bound workspace (host-only here: the size may
    change, so the caller binds again)."""
    inp = make_custom("m", torch.float16, 8, 2, 64, 16, True, -1, [70], [100],
                      [1], [40], seed=1)
    h = plan_host(inp, num_sms=4)
    need = (70 * 100 + 7) // 8
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_prefill_mask(h, np.zeros(need - 1, np.uint8))
    assert e.value.code == 1
    causal_hi = sorted(set(pod.pod_plan_table(h, 1).reshape(-1, REC)[:, 5].tolist()))
    pod.pod_plan_set_prefill_mask(h, np.zeros(need, np.uint8))
    masked_hi = sorted(set(pod.pod_plan_table(h, 1).reshape(-1, REC)[:, 5].tolist()))
    # tiles of 32 tokens (G = 4): causal ranges end at the tiles' last
    # diagonals 62, 94, 100; under the mask every tile reads all 100 keys
    assert causal_hi == [62, 94, 100] and masked_hi == [100]
    assert h.workspace_ptr is None and pod.plan_summary(h)["p_mask"] == 1


def test_kv_layout_switch_host_checks(lib):
    """pod_plan_set_kv_layout takes 0 (NHD) or 1 (HND) per half, leaves the
    plan as it is (the page tables do not depend on the layout) and refuses
    other codes."""
    inp = make_custom("l", torch.bfloat16, 16, 2, 128, 16, True, -1, [40], [90], [1, 2], [60, 70],
                      seed=2)
    h = plan_host(inp, num_sms=8)
    before = [pod.pod_plan_table(h, w).copy() for w in range(11)]
    pod.pod_plan_set_kv_layout(h, "HND", "NHD")
    pod.pod_plan_set_kv_layout(h, 1, 1)
    assert all(np.array_equal(b, pod.pod_plan_table(h, w)) for w, b in enumerate(before))
    L = pod.load_library()
    for p_l, d_l in ((2, 0), (0, -1)):
        assert L.pod_plan_set_kv_layout(ctypes.c_void_p(h.ptr), p_l, d_l) == 1
    assert L.pod_plan_set_kv_layout(None, 0, 0) == 1
    with pytest.raises(pod.PodError):
        pod.pod_plan_set_kv_layout(h, "NDH", "NHD")


def test_logits_transform_host_checks(lib):
    """pod_plan_set_logits_transform takes a non-negative finite soft cap or
    ALiBi slopes, not both, and neither next to an FP8 decode cache."""
    from pod_workloads import with_fp8_decode_cache
    inp = make_custom("t", torch.bfloat16, 16, 2, 128, 16, True, -1, [5], [9], [1, 2], [40, 70],
                      seed=1)
    h = plan_host(inp, num_sms=4)
    slopes = torch.full((16,), 0.5)
    pod.pod_plan_set_logits_transform(h, 30.0)
    pod.pod_plan_set_logits_transform(h, 0.0, slopes)
    pod.pod_plan_set_logits_transform(h, 0.0)
    for cap in (-1.0, float("nan"), float("inf")):
        with pytest.raises(pod.PodError) as e:
            pod.pod_plan_set_logits_transform(h, cap)
        assert e.value.code == 1
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_logits_transform(h, 5.0, slopes)
    assert e.value.code == 2
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_logits_transform(h, 0.0, torch.zeros(8))
    assert e.value.code == 1
    # FP8 decode cache: either order is refused
    pod.pod_plan_set_logits_transform(h, 5.0)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_decode_fp8(h, 1.0, 1.0)
    assert e.value.code == 2
    h8 = plan_host(with_fp8_decode_cache(inp), num_sms=4)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_logits_transform(h8, 5.0)
    assert e.value.code == 2


def test_plain_c_client(lib, tmp_path):
    """include/pod.h compiles as strict C99, and a C program makes, inspects,
    switches and destroys a host-only plan through the ABI alone."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(pod.LIB_PATH)
    exe = str(tmp_path / "abi_c_client")
    subprocess.check_call([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "csrc", "abi_c_client.c"),
                           "-L", libdir, "-lpod_gb300", f"-Wl,-rpath,{libdir}", "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_plan_is_deterministic_across_processes(lib):
    """The schedule search runs on integer times on the calling thread: two
    processes plan c3-c5 bit for bit alike."""
    import subprocess
    import sys
    code = (
        "import hashlib, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "import prefill_decode_paged_pod_gb300 as pod\n"
        "from pod_workloads import make_config\n"
        "pod.load_library()\n"
        "h = hashlib.sha256()\n"
        "for n in ('c3', 'c4', 'c5'):\n"
        "    p = pod.plan_inputs(make_config(n, with_data=False), num_sms=152)\n"
        "    for w in range(12):\n"
        "        h.update(pod.pod_plan_table(p, w).tobytes())\n"
        "print(h.hexdigest())\n")
    digests = set()
    for _ in range(2):
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr
        digests.add(r.stdout.strip())
    assert len(digests) == 1


def test_plan_latency(lib):
    """Planning is on the serving path (once per batch): the c5 plan (4408
    tiles, 4096 decode items) takes a few ms on one host thread. The bound
    here is loose (shared CI hosts); bench.py reports the measured time."""
    import time
    inp = make_config("c5", with_data=False)
    ts = []
    for _ in range(5):
        t0 = time.perf_counter()
        h = pod.plan_inputs(inp, num_sms=152)
        ts.append(time.perf_counter() - t0)
        pod.pod_destroy(h)
    assert min(ts) < 0.02, ts


def test_binding_refuses_host_mask_and_slopes_before_launch(lib):
    """A custom mask or ALiBi slopes that live in host memory serve host-only
    plans, but pod_run refuses them before any launch (the kernels read them
    from device memory)."""
    from pod_workloads import alibi_slopes, with_prefill_custom_mask
    inp = with_prefill_custom_mask(
        make_custom("b", torch.bfloat16, 8, 2, 64, 16, True, -1, [5], [9], [1], [20], seed=3))
    h = plan_host(inp, num_sms=4)          # the mask stays a CPU tensor without a GPU
    q = inp.p.q
    with pytest.raises(pod.PodError, match="CUDA uint8"):
        pod.pod_run(h, q, inp.p.kv, inp.d.q, inp.d.kv, torch.empty(256, dtype=torch.uint8))
    h2 = plan_host(make_custom("b", torch.bfloat16, 8, 2, 64, 16, True, -1, [5], [9], [1], [20],
                               seed=3), num_sms=4)
    pod.pod_plan_set_logits_transform(h2, 0.0, alibi_slopes(8))
    with pytest.raises(pod.PodError, match="ALiBi"):
        pod.pod_run(h2, q, inp.p.kv, inp.d.q, inp.d.kv, torch.empty(256, dtype=torch.uint8))


# ------------------------------------------------------------- RoPE pre-pass plan
def test_rope_plan_tables(lib):
    """With RoPE the plan keeps its tiles and items and runs one CTA per SM;
    its tables give each prefill page-table entry the position of its slot 0
    and its slots below kv_len (the decode half has no page copies: its keys
    are rotated in the kernel), and each query row of either half its
    bottom-right position (negative for a non-causal row before the keys);
    the workspace grows by the prefill page copies (K_hi, V, K_lo) and the
    high and low parts of both halves' rotated queries."""
    inp = make_custom("rp", torch.bfloat16, 8, 2, 128, 16, False, -1, [5, 70], [40, 33],
                      [1, 4], [300, 17], seed=5)
    h = plan_host(inp, num_sms=8)
    base = pod.pod_workspace_size(h)
    tiles0 = pod.pod_plan_table(h, 1).copy()
    items0 = pod.pod_plan_table(h, 2).copy()
    pod.pod_plan_set_rope(h, 2.0, 500.0)
    s = pod.plan_summary(h)
    assert s["rope"] == 1 and np.array_equal(pod.pod_plan_table(h, 1), tiles0)
    assert np.array_equal(pod.pod_plan_table(h, 2), items0)
    assert s["grid"] <= 8, "one CTA per SM under RoPE"
    ps = inp.page_size
    for half, hh, te, tq in (("p", inp.p, 12, 14), ("d", inp.d, 13, 15)):
        ent = pod.pod_plan_table(h, te).reshape(-1, 2)
        want, qpos = [], []
        for r in range(hh.batch):
            kvl = int(hh.kv_lens[r])
            for i in range(int(hh.kv_indptr[r + 1] - hh.kv_indptr[r])):
                want.append((i * ps, max(0, min(ps, kvl - i * ps))))
            ql = int(hh.q_indptr[r + 1] - hh.q_indptr[r])
            qpos += [kvl - ql + i for i in range(ql)]
        if half == "d":
            want = []
        assert [tuple(x) for x in ent.tolist()] == want, half
        assert pod.pod_plan_table(h, tq).tolist() == qpos, half
    # prefill page copies (3 rows a page) and both halves' queries (hi + lo)
    page = 3 * ps * 2 * 128 * 2
    grow = len(inp.p.kv_indices) * page + (inp.p.rows + inp.d.rows) * 8 * 128 * 2 * 2
    assert pod.pod_workspace_size(h) >= base + grow
    # the decode page table is the caller's (no identity over copies)
    assert min(pod.pod_plan_table(h, 14)) < 0          # request 1: 70 queries, 33 keys
    pod.pod_plan_set_rope(h, 0.0, 0.0)
    assert pod.plan_summary(h)["rope"] == 0 and pod.pod_workspace_size(h) == base


def test_rope_host_checks(lib):
    from pod_workloads import with_fp8_decode_cache
    inp = make_custom("rp", torch.bfloat16, 16, 2, 128, 16, True, -1, [5], [9], [1], [40], seed=1)
    h = plan_host(inp, num_sms=4)
    for sc, th in ((-1.0, 1e4), (1.0, 0.0), (float("nan"), 1e4), (1.0, float("inf"))):
        with pytest.raises(pod.PodError) as e:
            pod.pod_plan_set_rope(h, sc, th)
        assert e.value.code == 1
    h8 = plan_host(with_fp8_decode_cache(inp), num_sms=4)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_rope(h8, 1.0, 1e4)
    assert e.value.code == 2
    pod.pod_plan_set_rope(h, 1.0, 1e4)
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_decode_fp8(h, 1.0, 1.0)
    assert e.value.code == 2
    # RoPE and ALiBi are two position encodings: one at a time
    from pod_workloads import alibi_slopes
    with pytest.raises(pod.PodError) as e:
        pod.pod_plan_set_logits_transform(h, 0.0, alibi_slopes(16))
    assert e.value.code == 2


def test_replanning_switches_keep_each_other(lib):
    """The custom mask and RoPE each plan the handle again; switching one
    keeps the other, and switching both off gives the original plan back."""
    from pod_workloads import with_prefill_custom_mask
    inp = with_prefill_custom_mask(
        make_custom("sw", torch.bfloat16, 16, 2, 128, 16, True, 100, [70, 20], [300, 20],
                    [1, 3], [500, 60], seed=8))
    h = plan_host(inp, num_sms=8)                  # plan_inputs sets the mask
    orig = make_custom("sw", torch.bfloat16, 16, 2, 128, 16, True, 100, [70, 20], [300, 20],
                       [1, 3], [500, 60], seed=8)
    h0 = plan_host(orig, num_sms=8)
    pod.pod_plan_set_rope(h, 1.0, 1e4)
    s = pod.plan_summary(h)
    assert s["p_mask"] == 1 and s["rope"] == 1
    pod.pod_plan_set_prefill_mask(h, None)
    s = pod.plan_summary(h)
    assert s["p_mask"] == 0 and s["rope"] == 1
    pod.pod_plan_set_rope(h, 0.0, 0.0)
    assert pod.pod_workspace_size(h) == pod.pod_workspace_size(h0)
    for w in range(12):
        assert np.array_equal(pod.pod_plan_table(h, w), pod.pod_plan_table(h0, w)), w


# ------------------------------------------------------------- CUDA-graph capacity mode
def _caps_case(seed, d_kv, p_q, p_kv):
    return make_custom("gc", torch.bfloat16, 16, 2, 128, 16, True, -1, [p_q], [p_kv],
                       [1] * len(d_kv), d_kv, seed=seed)


def test_graph_capacity_layout_is_fixed(lib):
    """Under a CUDA-graph capacity the workspace layout and the launch shape
    depend on the capacities only: two plans of different lengths within the
    same capacities have the same workspace size and the full grid, and their
    counts sit in the status block the kernels read."""
    caps = (2, 256, 64, 8, 8, 800)
    sizes, grids = set(), set()
    for seed, d_kv, pq, pkv in ((1, [300, 500, 77, 1000], 64, 64),
                                (2, [301, 501, 78, 1001, 17, 3000], 128, 192)):
        inp = _caps_case(seed, d_kv, pq, pkv)
        h = plan_host(inp, num_sms=8)
        pod.pod_plan_set_graph_capacity(h, *caps)
        s = pod.plan_summary(h)
        sizes.add(pod.pod_workspace_size(h))
        grids.add(s["grid"])
        assert s["grid"] == 16                      # 2 CTAs x 8 SMs, whatever the work
        check_against_reference(inp, h)
        pod.pod_destroy(h)
    assert len(sizes) == 1 and grids == {16}


def test_graph_capacity_and_replan_errors(lib):
    inp = _caps_case(1, [300, 500], 64, 64)
    h = plan_host(inp, num_sms=8)
    with pytest.raises(pod.PodError) as e:             # no capacity mode
        pod.pod_replan(h, inp.p.q_indptr, inp.p.kv_indptr, inp.p.kv_indices, inp.p.last_page_len,
                       inp.d.q_indptr, inp.d.kv_indptr, inp.d.kv_indices, inp.d.last_page_len)
    assert e.value.code == 1
    with pytest.raises(pod.PodError) as e:             # the current plan exceeds a capacity
        pod.pod_plan_set_graph_capacity(h, 1, 256, 64, 1, 8, 800)
    assert e.value.code == 1
    pod.pod_plan_set_graph_capacity(h, 2, 256, 64, 8, 8, 800)
    with pytest.raises(pod.PodError) as e:             # no bound workspace yet
        pod.pod_replan(h, inp.p.q_indptr, inp.p.kv_indptr, inp.p.kv_indices, inp.p.last_page_len,
                       inp.d.q_indptr, inp.d.kv_indptr, inp.d.kv_indices, inp.d.last_page_len)
    assert e.value.code == 3
    with pytest.raises(pod.PodError) as e:             # one capacity mode at a time with RoPE
        pod.pod_plan_set_rope(h, 1.0, 1e4)
    assert e.value.code == 2
    pod.pod_plan_set_graph_capacity(h, 0, 0, 0, 0, 0, 0)   # off again
    assert pod.plan_summary(h)["grid"] <= 16
    pod.pod_destroy(h)


def test_head_dim_256_plans_one_cta_per_sm(lib):
    """head_dim 256 (a 256-column O in TMEM, 224 KB of prefill stages) plans
    one CTA per SM; the logits transforms and RoPE are refused there."""
    from pod_workloads import alibi_slopes
    inp = make_custom("d256", torch.bfloat16, 16, 2, 256, 16, True, -1, [300, 33], [300, 40],
                      [1, 4], [900, 77], seed=3, sinks=True)
    h = plan_host(inp, num_sms=16)
    s = check_against_reference(inp, h)
    assert s["grid"] <= 16
    for call in (lambda: pod.pod_plan_set_logits_transform(h, 30.0, None),
                 lambda: pod.pod_plan_set_logits_transform(h, 0.0, alibi_slopes(16)),
                 lambda: pod.pod_plan_set_rope(h, 1.0, 1e4),
                 lambda: pod.pod_plan_set_decode_fp8(h, 1.0, 1.0)):
        with pytest.raises(pod.PodError) as e:
            call()
        assert e.value.code == 2
    pod.pod_destroy(h)
