"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each check here is either a closed form, a hand-worked example, an invariant
that the definition implies (page permutation, page size, split/merge), an
exhaustive check of a decoder against a library routine, or brute-force dense
attention written independently with numpy/scipy (sink as an explicit extra
key column with a zero value row).

``test_planted_mistakes`` compiles mutated copies of the oracle's C source
(each with one plausible mistake) and checks that at least one pin fails for
every mutant, so the pins are shown to be sensitive.
"""
import json
import math
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from pod_workloads import (HalfInputs, alibi_slopes, make_custom, pack_mask,
                           page_table_from_lens, with_kv_layout, with_prefill_custom_mask)

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


# --------------------------------------------------------------------------
# helpers (independent of the oracle)
# --------------------------------------------------------------------------

def dense_kv(h: HalfInputs, r: int, ps: int):
    """Dense K, V [kv_len, Hk, d] of request r, gathered with numpy indexing
    (NHD pages [2, ps, Hk, d] or HND pages [2, Hk, ps, d])."""
    kv = h.kv.double().numpy()
    lo, hi = int(h.kv_indptr[r]), int(h.kv_indptr[r + 1])
    pages = h.kv_indices[lo:hi]
    kvl = int(h.kv_lens[r])
    t = np.arange(kvl)
    pg = pages[t // ps]
    sl = t % ps
    if h.kv_layout == "HND":
        return kv[pg, 0, :, sl], kv[pg, 1, :, sl]
    return kv[pg, 0, sl], kv[pg, 1, sl]


def brute_force(inp, half="d", soft_cap=0.0, alibi=None):
    """Textbook masked softmax(QK^T)V per request/head, all rows; optional
    logits soft cap (cap * tanh(x / cap) of the scaled logits) and ALiBi
    bias slope * (t - p)."""
    h = inp.p if half == "p" else inp.d
    H, Hk, d = inp.num_qo_heads, inp.num_kv_heads, inp.head_dim
    G = H // Hk
    q = h.q.float().numpy().astype(np.float64)
    rows = h.rows
    out = np.zeros((rows, H, d))
    lse = np.zeros((rows, H))
    for r in range(h.batch):
        q0, q1 = int(h.q_indptr[r]), int(h.q_indptr[r + 1])
        ql = q1 - q0
        if ql == 0:
            continue
        K, V = dense_kv(h, r, inp.page_size)
        kvl = K.shape[0]
        i = np.arange(ql)[:, None]
        t = np.arange(kvl)[None, :]
        p = kvl - ql + i
        mask = np.ones((ql, kvl), dtype=bool)
        if h.packed_mask is not None:
            # custom mask: this request's bits of the little-bit-order array,
            # unpacked by numpy; it takes the place of the causal rule
            bits = np.unpackbits(h.packed_mask, bitorder="little").astype(bool)
            off = int(sum(int(h.q_indptr[j + 1] - h.q_indptr[j]) * int(h.kv_lens[j])
                          for j in range(r)))
            mask &= bits[off:off + ql * kvl].reshape(ql, kvl)
        elif inp.causal:
            mask &= t <= p
        if inp.window_left >= 0:
            mask &= t >= p - inp.window_left
        live = mask.any(axis=1)          # rows a custom mask left with keys
        for hh in range(H):
            S = inp.sm_scale * (q[q0:q1, hh, :] @ K[:, hh // G, :].T)
            if soft_cap > 0:
                S = soft_cap * np.tanh(S / soft_cap)
            if alibi is not None:
                S = S + float(alibi[hh]) * (t - p)
            S = np.where(mask, S, -np.inf)[live]
            lse[q0:q1, hh] = -np.inf
            out[q0:q1, hh] = 0.0
            if not live.any():
                continue
            rows_idx = np.arange(q0, q1)[live]
            lse[rows_idx, hh] = logsumexp(S, axis=1) / math.log(2.0)
            if inp.sinks is not None:
                sink_col = np.full((S.shape[0], 1), float(inp.sinks[hh]))
                Vz = np.concatenate([V[:, hh // G, :], np.zeros((1, d))], axis=0)
                P = softmax(np.concatenate([S, sink_col], axis=1), axis=1)
                out[rows_idx, hh] = P @ Vz
            else:
                out[rows_idx, hh] = softmax(S, axis=1) @ V[:, hh // G, :]
    return out, lse


def run_oracle(inp, half="d", fn=None, **kw):
    fn = fn or oracle.attention_rows
    h = inp.p if half == "p" else inp.d
    out, lse, st = fn(h.q, h.kv, h.q_indptr, h.kv_indptr, h.kv_indices, h.last_page_len,
                      inp.num_qo_heads, inp.num_kv_heads, inp.head_dim, inp.page_size,
                      inp.causal, inp.window_left, inp.sm_scale, sinks=inp.sinks, nthreads=2, **kw)
    assert st == 0
    return out.reshape(h.rows, inp.num_qo_heads, inp.head_dim), lse.reshape(h.rows, inp.num_qo_heads)


def tiny_case(seed, G=None, ps=None, causal=None, window=None, sinks=None, d=None, dtype=torch.float16):
    rng = np.random.default_rng(seed)
    G = G or int(rng.choice([1, 2, 3]))
    Hk = int(rng.choice([1, 2]))
    d = d or int(rng.choice([4, 8, 16]))
    ps = ps or int(rng.choice([1, 3, 4, 16]))
    causal = bool(rng.integers(0, 2)) if causal is None else causal
    window = int(rng.choice([-1, 0, 2, 5])) if window is None else window
    sinks = bool(rng.integers(0, 2)) if sinks is None else sinks
    B = int(rng.integers(1, 4))
    kv = rng.integers(1, 41, size=B)
    ql = np.array([int(rng.integers(1, k + 1)) for k in kv])
    return make_custom("tiny", dtype, G * Hk, Hk, d, ps, causal, window,
                       [], [], ql, kv, seed=seed, sinks=sinks, extra_pages=3)


# --------------------------------------------------------------------------
# pins, written as functions of an attention callable so mutants can be run
# --------------------------------------------------------------------------

def pin_two_token(fn):
    g = json.load(open(os.path.join(GOLDEN, "two_token.json")))
    for case in g["cases"]:
        ql = case["q_len"]
        e = math.e
        # closed forms recomputed here; the fixture decimals must agree with them
        if case["name"] == "no_sink":
            cf = [[(e + 3) / (e + 1), (2 * e + 4) / (e + 1), math.log2(e + 1)]]
        elif case["name"] == "sink_zero":
            cf = [[(e + 3) / (e + 2), (2 * e + 4) / (e + 2), math.log2(e + 1)]]
        else:
            cf = [[1.0, 2.0, 1.0 / math.log(2.0)],
                  [(e + 3) / (e + 1), (2 * e + 4) / (e + 1), math.log2(e + 1)]]
        for row, c in zip(case["rows"], cf):
            assert np.allclose(row["out"] + [row["lse"]], c, rtol=0, atol=1e-15)
        # page_size 1, pages 0 and 1 hold keys 0 and 1
        kv = torch.zeros(2, 2, 1, 1, 2, dtype=torch.float16)
        kv[0, 0, 0, 0] = torch.tensor([1.0, 0.0])
        kv[1, 0, 0, 0] = torch.tensor([0.0, 1.0])
        kv[0, 1, 0, 0] = torch.tensor([1.0, 2.0])
        kv[1, 1, 0, 0] = torch.tensor([3.0, 4.0])
        q = torch.tensor([[[1.0, 0.0]]] * ql, dtype=torch.float16)
        sinks = None if case["sink"] is None else torch.tensor([case["sink"]], dtype=torch.float32)
        out, lse, st = fn(q, kv, np.array([0, ql]), np.array([0, 2]), np.array([0, 1]), np.array([1]),
                          1, 1, 2, 1, case["causal"], -1, 1.0, sinks=sinks, nthreads=1)
        assert st == 0
        for i, row in enumerate(case["rows"]):
            assert np.allclose(out[i], row["out"], rtol=0, atol=1e-12), (case["name"], out[i])
            assert abs(lse[i] - row["lse"]) < 1e-12, (case["name"], lse[i])


def pin_brute_force(fn, seeds=range(12)):
    for s in seeds:
        inp = tiny_case(s)
        ref_o, ref_l = brute_force(inp, "d")
        o, l = run_oracle(inp, "d", fn)
        assert np.max(np.abs(o - ref_o)) < 1e-12, f"seed {s}: out differs"
        assert np.max(np.abs(l - ref_l)) < 1e-12, f"seed {s}: lse differs"


def pin_closed_forms(fn):
    # q = 0: uniform weights over the allowed keys, lse = log2(n_allowed)
    inp = make_custom("q0", torch.bfloat16, 4, 2, 8, 4, True, 3, [], [], [2, 1], [9, 6], seed=5,
                      extra_pages=2)
    inp.d.q.zero_()
    o, l = run_oracle(inp, "d", fn)
    for r in range(2):
        K, V = dense_kv(inp.d, r, inp.page_size)
        q0, ql, kvl = inp.d.q_indptr[r], inp.d.q_lens[r], inp.d.kv_lens[r]
        for i in range(ql):
            p = kvl - ql + i
            allowed = [t for t in range(kvl) if t <= p and t >= p - 3]
            for hh in range(4):
                assert np.allclose(o[q0 + i, hh], V[allowed, hh // 2].mean(axis=0), atol=1e-13)
                assert abs(l[q0 + i, hh] - math.log2(len(allowed))) < 1e-13
    # window_left = 0: only the diagonal key; out = v_p, lse = s_p / ln 2
    inp = make_custom("w0", torch.float16, 2, 1, 8, 3, True, 0, [], [], [3], [7], seed=6)
    o, l = run_oracle(inp, "d", fn)
    K, V = dense_kv(inp.d, 0, 3)
    q = inp.d.q.double().numpy()
    for i in range(3):
        p = 7 - 3 + i
        for hh in range(2):
            assert np.allclose(o[i, hh], V[p, 0], atol=0)
            assert abs(l[i, hh] - inp.sm_scale * float(q[i, hh] @ K[p, 0]) / math.log(2)) < 1e-13
    # kv_len = 1: out = v_0
    inp = make_custom("kv1", torch.bfloat16, 3, 3, 16, 16, False, -1, [], [], [1], [1], seed=7)
    o, l = run_oracle(inp, "d", fn)
    K, V = dense_kv(inp.d, 0, 16)
    for hh in range(3):
        assert np.allclose(o[0, hh], V[0, hh], atol=0)
    # equal keys: uniform weights, lse = s + log2(n)
    inp = make_custom("eqk", torch.float16, 2, 1, 8, 4, False, -1, [], [], [1], [10], seed=8)
    inp.d.kv[:, 0] = inp.d.kv[0, 0, 0]
    o, l = run_oracle(inp, "d", fn)
    K, V = dense_kv(inp.d, 0, 4)
    q = inp.d.q.double().numpy()
    for hh in range(2):
        assert np.allclose(o[0, hh], V[:, 0].mean(axis=0), atol=1e-13)
        s = inp.sm_scale * float(q[0, hh] @ K[0, 0])
        assert abs(l[0, hh] - (s / math.log(2) + math.log2(10))) < 1e-12
    # sink with q = 0: out = sum v / (n + e^sink)
    inp = make_custom("sq0", torch.float16, 2, 1, 4, 2, False, -1, [], [], [1], [5], seed=9, sinks=True)
    inp.d.q.zero_()
    o, l = run_oracle(inp, "d", fn)
    K, V = dense_kv(inp.d, 0, 2)
    for hh in range(2):
        ref = V[:, 0].sum(axis=0) / (5 + math.exp(float(inp.sinks[hh])))
        assert np.allclose(o[0, hh], ref, atol=1e-13)
        assert abs(l[0, hh] - math.log2(5)) < 1e-13


def pin_gqa(fn):
    inp = make_custom("gqa", torch.bfloat16, 8, 2, 16, 4, True, -1, [], [], [3, 2], [11, 17], seed=10)
    q = inp.d.q
    for g in range(2):
        q[:, g * 4 + 1: g * 4 + 4] = q[:, g * 4: g * 4 + 1]
    o, l = run_oracle(inp, "d", fn)
    for g in range(2):
        for j in range(1, 4):
            assert np.array_equal(o[:, g * 4 + j], o[:, g * 4])
            assert np.array_equal(l[:, g * 4 + j], l[:, g * 4])
    # different groups read different kv heads: outputs must differ
    assert not np.allclose(o[:, 0], o[:, 4])


def pin_page_invariance(fn):
    inp = make_custom("perm", torch.float16, 4, 2, 8, 4, True, 6, [], [], [3, 1, 5], [13, 22, 9],
                      seed=11, sinks=True, extra_pages=5)
    o0, l0 = run_oracle(inp, "d", fn)
    h = inp.d
    rng = np.random.default_rng(1)
    perm = rng.permutation(h.num_pages)
    kv2 = torch.empty_like(h.kv)
    kv2[torch.from_numpy(perm)] = h.kv
    h2 = HalfInputs(h.q_indptr, h.kv_indptr, perm[h.kv_indices].astype(np.int32), h.last_page_len,
                    h.num_pages, h.q, kv2, h.q_lens, h.kv_lens)
    inp.d = h2
    o1, l1 = run_oracle(inp, "d", fn)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    # re-page the same token sequence with other page sizes
    inp.d = h
    for ps2 in (1, 3, 16):
        ks, vs = [], []
        for r in range(h.batch):
            K, V = dense_kv(h, r, 4)
            ks.append(K)
            vs.append(V)
        indptr, last = page_table_from_lens(h.kv_lens, ps2)
        npg = int(indptr[-1])
        kvn = torch.zeros(npg, 2, ps2, 2, 8, dtype=torch.float16)
        for r in range(h.batch):
            for t in range(int(h.kv_lens[r])):
                pg, sl = indptr[r] + t // ps2, t % ps2
                kvn[pg, 0, sl] = torch.from_numpy(ks[r][t]).half()
                kvn[pg, 1, sl] = torch.from_numpy(vs[r][t]).half()
        inp.d = HalfInputs(h.q_indptr, indptr, np.arange(npg, dtype=np.int32), last, npg,
                           h.q, kvn, h.q_lens, h.kv_lens)
        inp.page_size = ps2
        o2, l2 = run_oracle(inp, "d", fn)
        assert np.array_equal(o0, o2) and np.array_equal(l0, l2), ps2
    inp.page_size = 4
    inp.d = h


def pin_split_merge(fn, merge=None):
    merge = merge or oracle.merge
    for seed, sinks in ((12, False), (13, True)):
        inp = make_custom("sm", torch.bfloat16, 2, 1, 8, 4, True, -1, [], [], [2], [37],
                          seed=seed, sinks=sinks)
        o, l = run_oracle(inp, "d", fn)
        h = inp.d
        cuts = [0, 5, 16, 17, 30, 37]
        for tok in range(2):
            for hh in range(2):
                parts_o, parts_l = [], []
                for a, b in zip(cuts[:-1], cuts[1:]):
                    po, pl, st = fn(h.q, h.kv, h.q_indptr, h.kv_indptr, h.kv_indices, h.last_page_len,
                                    2, 1, 8, 4, True, -1, inp.sm_scale, sinks=None,
                                    sel_token=[tok], sel_head=[hh], key_lo=[a], key_hi=[b], nthreads=1)
                    if st == 2:      # every key of this chunk is masked for this row
                        continue
                    assert st == 0
                    parts_o.append(po[0])
                    parts_l.append(pl[0])
                sink = float(inp.sinks[hh]) if sinks else None
                mo, ml = merge(np.array(parts_o), np.array(parts_l), sink)
                assert np.max(np.abs(mo - o[tok, hh])) < 1e-12
                assert abs(ml - l[tok, hh]) < 1e-12


def pin_fp8(fn, seeds=range(6)):
    """FP8 (E4M3) decode cache: the attention callable on codes and scales
    equals textbook attention over the dequantized cache."""
    for seed in seeds:
        inp = _fp8_tiny(seed)
        ref_out, ref_lse = brute_force_scaled(inp)
        out, lse = run_oracle(inp, "d", fn=fn, k_scale=inp.k_scale, v_scale=inp.v_scale)
        assert np.allclose(out, ref_out, atol=1e-12, rtol=1e-12), seed
        assert np.allclose(lse, ref_lse, atol=1e-12, rtol=0), seed


def _masked_tiny(seed, **kw):
    inp = tiny_case(seed, **kw)
    # the prefill half of the tiny cases is empty: move the requests there
    inp.p, inp.d = inp.d, inp.p
    return with_prefill_custom_mask(inp, seed=seed, density=0.6)


def pin_custom_mask(fn, seeds=range(8)):
    """Custom prefill mask (POD walkthrough, run parameters custom_mask_p /
    packed_custom_mask_p, little bit order):
    - random masks with empty and full rows against brute force over the
      mask numpy unpacks;
    - a mask with one set bit picks exactly that key: out = v_t and
      lse = s_t / ln 2, which fixes the bit order and the row stride;
    - the bottom-right lower-triangular mask reproduces the causal result and
      the all-ones mask the non-causal one, bit for bit."""
    for seed in seeds:
        inp = _masked_tiny(seed)
        ref_out, ref_lse = brute_force(inp, "p")
        out, lse = run_oracle(inp, "p", fn=fn, packed_mask=inp.p.packed_mask)
        assert np.allclose(out, ref_out, atol=1e-12, rtol=1e-12), seed
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse)), seed
        assert np.allclose(lse[fin], ref_lse[fin], atol=1e-12, rtol=0), seed
    # one set bit per request, at a chosen (row, key)
    inp = _masked_tiny(3, causal=False, window=-1, sinks=False)
    h = inp.p
    mats, picks = [], []
    for r in range(h.batch):
        ql = int(h.q_indptr[r + 1] - h.q_indptr[r])
        kl = int(h.kv_lens[r])
        m = np.zeros((ql, kl), dtype=bool)
        i, t = ql - 1, (7 * r + 5) % kl
        m[i, t] = True
        mats.append(m)
        picks.append((r, i, t))
    h.packed_mask = pack_mask(mats)
    out, lse = run_oracle(inp, "p", fn=fn, packed_mask=h.packed_mask)
    G = inp.num_qo_heads // inp.num_kv_heads
    qf = h.q.double().numpy()
    for r, i, t in picks:
        K, V = dense_kv(h, r, inp.page_size)
        row = int(h.q_indptr[r]) + i
        for hh in range(inp.num_qo_heads):
            assert np.array_equal(out[row, hh], V[t, hh // G]), (r, hh)
            s_t = inp.sm_scale * float(qf[row, hh] @ K[t, hh // G])
            assert abs(lse[row, hh] - s_t / math.log(2.0)) < 1e-12, (r, hh)
    # triangular and all-ones masks against the mask-free rules
    for seed in (1, 2, 5):
        inp = _masked_tiny(seed, window=-1)
        h = inp.p
        tri, ones = [], []
        for r in range(h.batch):
            ql = int(h.q_indptr[r + 1] - h.q_indptr[r])
            kl = int(h.kv_lens[r])
            i = np.arange(ql)[:, None]
            t = np.arange(kl)[None, :]
            tri.append(t <= kl - ql + i)
            ones.append(np.ones((ql, kl), dtype=bool))
        for mats, causal in ((tri, True), (ones, False)):
            inp.causal = causal
            o_ref, l_ref = run_oracle(inp, "p", fn=fn)
            inp.causal = not causal
            o_m, l_m = run_oracle(inp, "p", fn=fn, packed_mask=pack_mask(mats))
            assert np.array_equal(o_m, o_ref) and np.array_equal(l_m, l_ref), seed


def pin_hnd_layout(fn, seeds=range(6)):
    """HND pages ([2, Hk, ps, d]): the same keys stored the other way give the
    NHD result bit for bit, and brute force over a gather written for HND."""
    for seed in seeds:
        inp = tiny_case(seed)
        o_n, l_n = run_oracle(inp, "d", fn=fn)
        hnd = with_kv_layout(inp, "HND")
        o_h, l_h = run_oracle(hnd, "d", fn=fn, kv_layout=1)
        assert np.array_equal(o_h, o_n) and np.array_equal(l_h, l_n), seed
        if inp.num_kv_heads > 1 and inp.page_size > 1:
            # reading HND pages as NHD must change the result
            o_x, _ = run_oracle(hnd, "d", fn=fn, kv_layout=0)
            assert not np.array_equal(o_x, o_n), seed
        ref_o, ref_l = brute_force(hnd, "d")
        assert np.allclose(o_h, ref_o, atol=1e-12, rtol=1e-12), seed
        assert np.allclose(l_h, ref_l, atol=1e-12, rtol=0), seed


def pin_alibi(fn, seeds=range(6)):
    """ALiBi (pos_encoding_mode ALIBI): brute force with the bias
    slope * (t - p); with q = 0 on a causal row the weights are
    e^{-m (p - t)}, so the lse is log2 of the geometric sum
    (1 - e^{-m (p + 1)}) / (1 - e^{-m}); slope 0 is the plain result."""
    for seed in seeds:
        inp = tiny_case(seed)
        sl = alibi_slopes(inp.num_qo_heads)
        ref_o, ref_l = brute_force(inp, "d", alibi=sl.numpy())
        out, lse = run_oracle(inp, "d", fn=fn, alibi_slopes=sl)
        assert np.allclose(out, ref_o, atol=1e-12, rtol=1e-12), seed
        assert np.allclose(lse, ref_l, atol=1e-12, rtol=0), seed
        o0, l0 = run_oracle(inp, "d", fn=fn, alibi_slopes=np.zeros(inp.num_qo_heads, np.float32))
        o1, l1 = run_oracle(inp, "d", fn=fn)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1), seed
    inp = tiny_case(2, causal=True, window=-1, sinks=False)
    inp.d.q = torch.zeros_like(inp.d.q)
    sl = alibi_slopes(inp.num_qo_heads)
    _, lse = run_oracle(inp, "d", fn=fn, alibi_slopes=sl)
    h = inp.d
    for r in range(h.batch):
        ql = int(h.q_indptr[r + 1] - h.q_indptr[r])
        kvl = int(h.kv_lens[r])
        for i in range(ql):
            p = kvl - ql + i
            for hh in range(inp.num_qo_heads):
                m = float(sl[hh])
                z = (1.0 - math.exp(-m * (p + 1))) / (1.0 - math.exp(-m))
                assert abs(lse[int(h.q_indptr[r]) + i, hh] - math.log2(z)) < 1e-12


def pin_soft_cap(fn, seeds=range(6)):
    """Logits soft cap (cap * tanh(x / cap) of the scaled logit x): brute
    force; two keys whose scaled logits are +-L with L far above the cap get
    weights 1 / (1 + e^{-2 cap}) and e^{-2 cap} / (1 + e^{-2 cap}); a cap far
    above every logit leaves the result unchanged to 1e-9."""
    for seed in seeds:
        inp = tiny_case(seed)
        ref_o, ref_l = brute_force(inp, "d", soft_cap=1.5)
        out, lse = run_oracle(inp, "d", fn=fn, soft_cap=1.5)
        assert np.allclose(out, ref_o, atol=1e-12, rtol=1e-12), seed
        assert np.allclose(lse, ref_l, atol=1e-12, rtol=0), seed
        o_big, l_big = run_oracle(inp, "d", fn=fn, soft_cap=1e7)
        o_pl, l_pl = run_oracle(inp, "d", fn=fn)
        assert np.allclose(o_big, o_pl, atol=1e-9) and np.allclose(l_big, l_pl, atol=1e-9), seed
    # one request, two keys, d = 2: q = [1, 0], k0 = [L, 0], k1 = [-L, 0], sm_scale = 1
    H = Hk = 1
    q_indptr = np.array([0, 1], np.int32)
    kv_indptr = np.array([0, 1], np.int32)
    kv = torch.zeros((1, 2, 2, 1, 2), dtype=torch.float16)
    L, cap = 1000.0, 2.0
    kv[0, 0, 0, 0] = torch.tensor([L, 0.0])
    kv[0, 0, 1, 0] = torch.tensor([-L, 0.0])
    kv[0, 1, 0, 0] = torch.tensor([1.0, 0.0])
    kv[0, 1, 1, 0] = torch.tensor([0.0, 1.0])
    q = torch.tensor([[[1.0, 0.0]]], dtype=torch.float16)
    out, lse, st = fn(q, kv, q_indptr, kv_indptr, np.array([0], np.int32), np.array([2], np.int32),
                      H, Hk, 2, 2, False, -1, 1.0, nthreads=1, soft_cap=cap)
    assert st == 0
    c0, c1 = cap * math.tanh(L / cap), cap * math.tanh(-L / cap)   # = +-cap in fp64
    w0 = 1.0 / (1.0 + math.exp(c1 - c0))
    assert abs(out[0, 0] - w0) < 1e-15 and abs(out[0, 1] - (1.0 - w0)) < 1e-15
    assert abs(lse[0] - (c0 + math.log1p(math.exp(c1 - c0))) / math.log(2.0)) < 1e-12


def _set_row(h, r, t, kind, vec):
    """Write key/value vector of request r, position t (all kv heads), NHD."""
    ps = h.kv.shape[2]
    page = int(h.kv_indices[int(h.kv_indptr[r]) + t // ps])
    h.kv[page, kind, t % ps, :, :] = torch.as_tensor(vec, dtype=h.kv.dtype)


def _rope_closed_case(q, k, n, sm_scale=1.0):
    """One request, one query at p = n - 1, n keys all equal to k, value row
    t = (t, 1, ...); H = Hk = 1, d = len(q)."""
    d = len(q)
    inp = make_custom("rope", torch.float16, 1, 1, d, 4, True, -1, [], [], [1], [n], seed=0,
                      sm_scale=sm_scale)
    h = inp.d
    h.q[0, 0] = torch.tensor(q, dtype=h.q.dtype)
    for t in range(n):
        _set_row(h, 0, t, 0, k)
        v = np.zeros(d)
        v[0], v[1] = t, 1.0
        _set_row(h, 0, t, 1, v)
    return inp


def pin_rope(fn):
    """ROPE_LLAMA: pins that do not restate the rotation.
    - d = 4, q = k = e1 (pair 1: elements 1 and 3): the logit of key t is
      cos((p - t) * theta^(-1/2) / rope_scale); q = k = e0 gives
      cos((p - t) / rope_scale); q = e0, k = e2 gives sin((p - t) / rope_scale)
      (fixes pairing, frequency exponent, scale and direction);
    - a query and its keys moved 5 positions later give the same output
      (only relative positions matter);
    - at position 0 (kv_len = 1) the rotation is the identity."""
    rs, th, n = 2.0, 100.0, 6
    e = np.eye(4)
    for qv, kv_, f in ((e[1], e[1], lambda x: math.cos(x * th ** -0.5 / rs)),
                       (e[0], e[0], lambda x: math.cos(x / rs)),
                       (e[0], e[2], lambda x: math.sin(x / rs))):
        inp = _rope_closed_case(qv, kv_, n)
        out, lse = run_oracle(inp, "d", fn=fn, rope=True, rope_scale=rs, rope_theta=th)
        s_t = np.array([f(n - 1 - t) for t in range(n)])
        w = np.exp(s_t - s_t.max())
        w /= w.sum()
        assert abs(out[0, 0, 0] - float(w @ np.arange(n))) < 1e-12
        assert abs(out[0, 0, 1] - 1.0) < 1e-12
        assert abs(lse[0, 0] - math.log2(np.exp(s_t).sum())) < 1e-12
    # shift: request 1 = request 0 moved 5 positions later, a window hides the rest
    inp = make_custom("ropeshift", torch.float16, 4, 2, 8, 4, True, 6, [], [], [1, 1], [7, 12],
                      seed=5)
    h = inp.d
    h.q[1] = h.q[0]
    for t in range(7):
        for kind in (0, 1):
            ps = inp.page_size
            src = int(h.kv_indices[int(h.kv_indptr[0]) + t // ps])
            _set_row(h, 1, t + 5, kind, h.kv[src, kind, t % ps].clone())
    out, lse = run_oracle(inp, "d", fn=fn, rope=True, rope_scale=1.0, rope_theta=1e4)
    assert np.allclose(out[1], out[0], atol=1e-12, rtol=0) and np.allclose(lse[1], lse[0], atol=1e-12)
    plain_o, _ = run_oracle(inp, "d", fn=fn)
    assert not np.allclose(plain_o[0], out[0], atol=1e-6)
    # position 0
    inp = make_custom("rope0", torch.float16, 2, 1, 8, 4, True, -1, [], [], [1], [1], seed=6)
    o_r, l_r = run_oracle(inp, "d", fn=fn, rope=True, rope_scale=3.0, rope_theta=50.0)
    o_p, l_p = run_oracle(inp, "d", fn=fn)
    assert np.allclose(o_r, o_p, atol=1e-14) and np.allclose(l_r, l_p, atol=1e-14)


ALL_PINS = (pin_two_token, pin_brute_force, pin_closed_forms, pin_gqa, pin_page_invariance,
            pin_split_merge, pin_fp8, pin_custom_mask, pin_hnd_layout, pin_alibi, pin_soft_cap,
            pin_rope)


# --------------------------------------------------------------------------
# tests
# --------------------------------------------------------------------------

def test_f16_decoder_exhaustive():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(c)) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_bf16_decoder_exhaustive():
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    ref = codes.double().numpy()
    got = np.array([oracle.bf16_to_f64(c) for c in range(65536)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_seq_lens_docstring_page_table():
    g = json.load(open(os.path.join(GOLDEN, "docstring_page_table.json")))
    got = oracle.seq_lens(g["kv_page_indptr"], g["kv_last_page_len"], g["page_size"])
    assert got.tolist() == g["kv_len"]


def test_two_token_example():
    pin_two_token(oracle.attention_rows)


def test_brute_force_dense():
    pin_brute_force(oracle.attention_rows, seeds=range(40))


@pytest.mark.parametrize("ps", [1, 5, 16])
@pytest.mark.parametrize("window", [-1, 0, 7])
def test_brute_force_grid(ps, window):
    for s in range(3):
        inp = tiny_case(100 + s, ps=ps, window=window, causal=True, sinks=(s == 1), d=16,
                        dtype=torch.bfloat16)
        ref_o, ref_l = brute_force(inp, "d")
        o, l = run_oracle(inp, "d")
        assert np.max(np.abs(o - ref_o)) < 1e-12
        assert np.max(np.abs(l - ref_l)) < 1e-12


def test_closed_forms():
    pin_closed_forms(oracle.attention_rows)


def test_gqa_duplication():
    pin_gqa(oracle.attention_rows)


def test_page_permutation_and_size_invariance():
    pin_page_invariance(oracle.attention_rows)


def test_split_merge_identity():
    pin_split_merge(oracle.attention_rows)


def test_prefill_half_matches_brute_force():
    inp = make_custom("pf", torch.float16, 6, 2, 16, 4, True, 9, [7, 12, 1], [7, 20, 3], [], [],
                      seed=21, sinks=True)
    ref_o, ref_l = brute_force(inp, "p")
    o, l = run_oracle(inp, "p")
    assert np.max(np.abs(o - ref_o)) < 1e-12 and np.max(np.abs(l - ref_l)) < 1e-12


# --------------------------------------------------------------------------
# planted mistakes: every mutant of the oracle must fail at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "causal_off_by_one": ("} else if (causal && t > p) {", "} else if (causal && t >= p) {"),
    "window_excludes_diagonal_bound": ("t < p - window_left) ok = 0;", "t <= p - window_left) ok = 0;"),
    "gqa_modulo": ("int hk = h / group;", "int hk = h % Hk;"),
    "top_left_causal": ("int64_t p = kv_len - q_len + i;", "int64_t p = i;"),
    "natural_log_lse": ("lse[s] = (m + log(z)) / log(2.0);", "lse[s] = (m + log(z));"),
    "sink_in_lse": ("lse[s] = (m + log(z)) / log(2.0);", "lse[s] = (m + log(denom)) / log(2.0);"),
    "sink_dropped": ("if (sinks) denom += exp((double)sinks[h] - m);", ""),
    "sink_scaled": ("denom += exp((double)sinks[h] - m);", "denom += exp(sm_scale * (double)sinks[h] - m);"),
    "k_for_v": ("row_offset(kv_layout, page, 1, slot", "row_offset(kv_layout, page, 0, slot"),
    "last_page_off": ("return (pages - 1) * (int64_t)page_size + last_page_len[r];",
                      "return pages * (int64_t)page_size;"),
    "scale_dropped": ("            logit[t] = sm_scale * dot;", "            logit[t] = dot;"),
    "merge_natural_weights": ("double w = pow(2.0, lse_parts[i] - M);", "double w = exp(lse_parts[i] - M);"),
    "f16_bias": ("e - 25", "e - 24"),
    "e4m3_bias": ("ldexp((double)(8 + f), e - 10)", "ldexp((double)(8 + f), e - 9)"),
    "e4m3_subnormal": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "fp8_v_with_k_scale": ("kv_elem(kv, v0 + e, dtype, kv_fp8, v_scale)",
                           "kv_elem(kv, v0 + e, dtype, kv_fp8, k_scale)"),
    "mask_big_endian_bits": ("(packed[pos >> 3] >> (int)(pos & 7)) & 1",
                             "(packed[pos >> 3] >> (int)(7 - (pos & 7))) & 1"),
    "mask_no_request_offset": ("for (int rr = 0; rr < r; ++rr)", "for (int rr = 0; rr < 0; ++rr)"),
    "mask_row_stride_q_len": ("mask_row += i * kv_len;", "mask_row += i * q_len;"),
    "mask_and_causal": ("} else if (causal && t > p) {", "} if (causal && t > p) {"),
    "hnd_read_as_nhd": ("return (((page * 2 + kv) * Hk + hk) * (int64_t)page_size + slot) * (int64_t)d;",
                        "return (((page * 2 + kv) * (int64_t)page_size + slot) * Hk + hk) * (int64_t)d;"),
    "alibi_sign": ("(double)alibi_slopes[h] * (double)(t - p)", "(double)alibi_slopes[h] * (double)(p - t)"),
    "alibi_top_left": ("(double)alibi_slopes[h] * (double)(t - p)", "(double)alibi_slopes[h] * (double)(t - i)"),
    "soft_cap_outside_scale": ("soft_cap * tanh(sm_scale * dot / soft_cap)",
                               "sm_scale * soft_cap * tanh(dot / soft_cap)"),
    "rope_interleaved_pairs": ("double a = x[j], b = x[j + half];\n        x[j] = a * c - b * sn;\n        x[j + half] = b * c + a * sn;",
                               "double a = x[2 * j], b = x[2 * j + 1];\n        x[2 * j] = a * c - b * sn;\n        x[2 * j + 1] = b * c + a * sn;"),
    "rope_freq_exponent": ("-2.0 * (double)j / (double)d", "-1.0 * (double)j / (double)d"),
    "rope_scale_multiplies": ("(pos / rope_scale)", "(pos * rope_scale)"),
    "rope_query_at_row_index": ("rope_rotate(qv, d, (double)p,", "rope_rotate(qv, d, (double)i,"),
    "rope_reverse_direction": ("x[j] = a * c - b * sn;\n        x[j + half] = b * c + a * sn;",
                               "x[j] = a * c + b * sn;\n        x[j + half] = b * c - a * sn;"),
}


def _mutant_fns(tmpdir, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "pod_oracle.c")).read()
    assert old in src, name
    so = os.path.join(tmpdir, f"m_{name}.so")
    cpath = os.path.join(tmpdir, f"m_{name}.c")
    open(cpath, "w").write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", so, cpath, "-lm"])
    import ctypes
    L = ctypes.CDLL(so)
    # reuse the wrapper by swapping the library object temporarily
    def fn(*a, **k):
        saved = oracle._lib
        oracle._lib = L
        L.oracle_attention_rows.restype = ctypes.c_int
        L.oracle_attention_rows.argtypes = saved.oracle_attention_rows.argtypes
        L.oracle_attention_rows_kv.restype = ctypes.c_int
        L.oracle_attention_rows_kv.argtypes = saved.oracle_attention_rows_kv.argtypes
        L.oracle_attention_rows_masked.restype = ctypes.c_int
        L.oracle_attention_rows_masked.argtypes = saved.oracle_attention_rows_masked.argtypes
        L.oracle_attention_rows_ext.restype = ctypes.c_int
        L.oracle_attention_rows_ext.argtypes = saved.oracle_attention_rows_ext.argtypes
        L.oracle_merge.argtypes = saved.oracle_merge.argtypes
        L.oracle_merge.restype = None
        try:
            return oracle.attention_rows(*a, **k)
        finally:
            oracle._lib = saved

    def mg(*a, **k):
        saved = oracle._lib
        oracle._lib = L
        L.oracle_merge.argtypes = saved.oracle_merge.argtypes
        L.oracle_merge.restype = None
        try:
            return oracle.merge(*a, **k)
        finally:
            oracle._lib = saved
    return fn, mg


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name):
    oracle.lib()
    old, new = MUTANTS[name]
    with tempfile.TemporaryDirectory() as td:
        fn, mg = _mutant_fns(td, name, old, new)
        failures = 0
        for pin in ALL_PINS:
            try:
                if pin is pin_split_merge:
                    pin(fn, mg)
                elif pin is pin_brute_force:
                    pin(fn, seeds=range(12))
                else:
                    pin(fn)
            except AssertionError:
                failures += 1
        assert failures > 0, f"mutant {name} passed every pin"


# --------------------------------------------------------------------------
# FP8 (E4M3) decode cache
# --------------------------------------------------------------------------

def test_e4m3_decoder_exhaustive():
    """All 256 E4M3 codes against torch's float8_e4m3fn and against values the
    format's definition fixes (bias 7, 3 fraction bits, S.1111.111 = NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    assert np.array_equal(ref[~np.isnan(ref)], got[~np.isnan(got)])
    fixed = {0x38: 1.0, 0x40: 2.0, 0x7E: 448.0, 0x08: 2.0 ** -6, 0x01: 2.0 ** -9,
             0x07: 7 * 2.0 ** -9, 0x3C: 1.5, 0xC0: -2.0, 0x00: 0.0}
    for c, v in fixed.items():
        assert oracle.e4m3_to_f64(c) == v, hex(c)
    assert math.isnan(oracle.e4m3_to_f64(0x7F)) and math.isnan(oracle.e4m3_to_f64(0xFF))
    assert math.copysign(1.0, oracle.e4m3_to_f64(0x80)) == -1.0


def _fp8_tiny(seed):
    from pod_workloads import with_fp8_decode_cache
    base = tiny_case(seed, dtype=torch.bfloat16)
    rng = np.random.default_rng(seed)
    return with_fp8_decode_cache(base, k_scale=float(rng.choice([0.02, 0.5, 3.0])),
                                 v_scale=float(rng.choice([0.03, 1.0, 4.0])))


@pytest.mark.parametrize("seed", range(10))
def test_fp8_cache_matches_dequantized_brute_force(seed):
    """Textbook attention over code * scale (K and V dequantized separately)
    equals the oracle's FP8 path."""
    inp = _fp8_tiny(seed)
    ref_out, ref_lse = brute_force_scaled(inp)
    out, lse, st = oracle.attention_half(inp, "d", nthreads=2)
    assert st == 0
    h = inp.d
    out = out.reshape(h.rows, inp.num_qo_heads, inp.head_dim)
    lse = lse.reshape(h.rows, inp.num_qo_heads)
    assert np.allclose(out, ref_out, atol=1e-12, rtol=1e-12)
    assert np.allclose(lse, ref_lse, atol=1e-12, rtol=0)


def brute_force_scaled(inp):
    """brute_force over a copy of the decode half whose cache holds the
    dequantized values (codes * k_scale for K, codes * v_scale for V) in fp64."""
    import copy
    h = copy.copy(inp.d)
    kv = h.kv.double()
    kv[:, 0] *= inp.k_scale
    kv[:, 1] *= inp.v_scale
    h.kv = kv
    inp2 = copy.copy(inp)
    inp2.d = h
    return brute_force(inp2, "d")


def test_fp8_scale_folding():
    """k_scale acts as a factor on the logits (same result as folding it into
    sm_scale with k_scale = 1); v_scale scales the output and leaves the LSE."""
    inp = _fp8_tiny(3)
    h = inp.d
    args = (h.q, h.kv, h.q_indptr, h.kv_indptr, h.kv_indices, h.last_page_len,
            inp.num_qo_heads, inp.num_kv_heads, inp.head_dim, inp.page_size, inp.causal,
            inp.window_left)
    o1, l1, _ = oracle.attention_rows(*args, inp.sm_scale, sinks=inp.sinks, k_scale=2.5,
                                      v_scale=1.0, nthreads=2)
    o2, l2, _ = oracle.attention_rows(*args, inp.sm_scale * 2.5, sinks=inp.sinks, k_scale=1.0,
                                      v_scale=1.0, nthreads=2)
    assert np.allclose(o1, o2, atol=1e-12, rtol=1e-12) and np.allclose(l1, l2, atol=1e-12)
    o3, l3, _ = oracle.attention_rows(*args, inp.sm_scale, sinks=inp.sinks, k_scale=2.5,
                                      v_scale=0.25, nthreads=2)
    assert np.allclose(o3, 0.25 * o1, atol=1e-12, rtol=1e-12) and np.array_equal(l3, l1)


# --------------------------------------------------------------------------
# custom prefill mask
# --------------------------------------------------------------------------

def test_custom_mask_pins():
    pin_custom_mask(oracle.attention_rows)


def test_pack_mask_bit_order():
    """pack_mask puts element k of the flattened masks at bit k % 8 of byte
    k // 8 (little bit order), the layout the pages name."""
    m = np.zeros((3, 5), dtype=bool)
    m[0, 0] = m[1, 2] = m[2, 4] = True     # flat positions 0, 7, 14
    b = pack_mask([m])
    assert b.tolist() == [0b10000001, 0b01000000]


def test_custom_mask_with_window_and_sinks():
    """An all-ones mask with a window equals the non-causal windowed result;
    sinks leave a row the mask empties at out = 0 (its only weight is on the
    sink's zero value row) and lse = -inf."""
    inp = _masked_tiny(4, window=2, sinks=True)
    h = inp.p
    ones = [np.ones((int(h.q_indptr[r + 1] - h.q_indptr[r]), int(h.kv_lens[r])), dtype=bool)
            for r in range(h.batch)]
    inp.causal = False
    o_ref, l_ref = run_oracle(inp, "p")
    inp.causal = True
    o_m, l_m = run_oracle(inp, "p", packed_mask=pack_mask(ones))
    assert np.array_equal(o_m, o_ref) and np.array_equal(l_m, l_ref)
    zeros = [np.zeros_like(m) for m in ones]
    o_z, l_z = run_oracle(inp, "p", packed_mask=pack_mask(zeros))
    assert np.all(o_z == 0.0) and np.all(l_z == -np.inf)


# --------------------------------------------------------------------------
# NEXT variants: HND layout, ALiBi, logits soft cap
# --------------------------------------------------------------------------

def test_hnd_layout_pins():
    pin_hnd_layout(oracle.attention_rows)


def test_alibi_pins():
    pin_alibi(oracle.attention_rows)


def test_soft_cap_pins():
    pin_soft_cap(oracle.attention_rows)


def test_rope_pins():
    pin_rope(oracle.attention_rows)
