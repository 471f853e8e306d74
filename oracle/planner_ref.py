"""Plain restatement of the POD planner's integer rules — TEST INFRASTRUCTURE ONLY.

Used to check the library's host planner bit for bit. It restates, in the
simplest loops, what the plan must contain:

* kv_len per request: (pages - 1) * page_size + last_page_len (POD
  walkthrough, "plan 内部做了什么", get_seq_lens);
* the query rows of every prefill tile: 128 // G tokens of one request times
  the G qo heads of one kv head (G = num_qo_heads / num_kv_heads, "plan/run
  生命周期" GQA rule), tiles ordered by request, token block, kv head;
* the key range [lo, hi) each tile or decode unit needs: the bottom-right
  diagonal p = kv_len - q_len + i bounds it above when causal, the window
  keeps keys t >= p - window_left (flashinfer.cudnn page, "Decode 能力矩阵与参数");
* decode units: 32 // G tokens x G heads, same ordering;
* the validation rules of the walkthrough ("CUDAGraph 模式的运行时约束",
  "plan/run 生命周期") and the page-table invariants 1 <= last_page_len <= page_size.
"""
from __future__ import annotations

import numpy as np

TILE_ROWS = 128
DECODE_ROWS = 32


def seq_lens(kv_indptr, last_page_len, page_size):
    out = []
    for r in range(len(kv_indptr) - 1):
        pages = int(kv_indptr[r + 1]) - int(kv_indptr[r])
        out.append(0 if pages <= 0 else (pages - 1) * page_size + int(last_page_len[r]))
    return np.array(out, dtype=np.int32)


def key_range(kv_len, q_len, t0, ntok, causal, window_left):
    p_first = kv_len - q_len + t0
    p_last = p_first + ntok - 1
    hi = min(kv_len, p_last + 1) if causal else kv_len
    lo = max(0, p_first - window_left) if window_left >= 0 else 0
    return min(lo, hi), hi


def prefill_tiles(q_indptr, kv_lens, H, Hk, causal, window_left):
    G = H // Hk
    tq = max(1, TILE_ROWS // G)
    tiles = []
    for r in range(len(q_indptr) - 1):
        ql = int(q_indptr[r + 1]) - int(q_indptr[r])
        for t0 in range(0, ql, tq):
            nt = min(tq, ql - t0)
            lo, hi = key_range(int(kv_lens[r]), ql, t0, nt, causal, window_left)
            for g in range(Hk):
                tiles.append((r, g, t0, nt, lo, hi))
    return tiles


def decode_units(q_indptr, kv_lens, H, Hk, causal, window_left):
    G = H // Hk
    tu = max(1, DECODE_ROWS // G)
    units = []
    for r in range(len(q_indptr) - 1):
        ql = int(q_indptr[r + 1]) - int(q_indptr[r])
        for t0 in range(0, ql, tu):
            nt = min(tu, ql - t0)
            lo, hi = key_range(int(kv_lens[r]), ql, t0, nt, causal, window_left)
            for g in range(Hk):
                units.append((r, g, t0, nt, lo, hi))
    return units


def validate_half(q_indptr, kv_indptr, kv_indices, last_page_len, num_pages, page_size, causal):
    """Return None when the half is valid, else a short reason."""
    b = len(q_indptr) - 1
    if b == 0:
        return None
    if q_indptr[0] != 0 or kv_indptr[0] != 0:
        return "indptr must start at 0"
    if np.any(np.diff(q_indptr) < 0) or np.any(np.diff(kv_indptr) < 0):
        return "indptr not monotone"
    if len(kv_indices) and (np.min(kv_indices) < 0 or np.max(kv_indices) >= num_pages):
        return "page index outside the pool"
    for r in range(b):
        pages = kv_indptr[r + 1] - kv_indptr[r]
        ql = q_indptr[r + 1] - q_indptr[r]
        if pages > 0 and not (1 <= last_page_len[r] <= page_size):
            return "last_page_len outside [1, page_size]"
        kl = 0 if pages == 0 else (pages - 1) * page_size + last_page_len[r]
        if ql > 0 and kl == 0:
            return "queries without keys"
        if ql > 0 and causal and kl < ql:
            return "kv_len < q_len under causal"
    return None
