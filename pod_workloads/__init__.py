"""Seeded synthetic inputs for POD (prefill-on-decode) paged attention.

This module only draws random numbers and builds page tables. It holds none of
the attention arithmetic, so both the CUDA path (tests, bench) and the CPU
oracle can consume what it produces without sharing any of the method.

Workloads follow the shapes on the FlashInfer ``flashinfer.pod`` walkthrough
(page "POD 是什么", the single-request docstring example and the batch POD
docstring example) and the five configurations of this library's benchmark:

  c1  tiny fp16, H/Hk/d/ps = 4/1/64/16; prefill 64/64; decode kv {17,29,5,48}
  c2  fp16 64/8/128/16; prefill 1024/1024 (pages 0..63); 7 decode requests with
      kv_page_indptr [0,17,29,44,48,66,100,128], last_page_len [1,7,14,4,3,1,16]
  c3  bf16 64/8/128/1; 2 x 2048 prefill; 128 x 2048 decode; contiguous pages
  c4  bf16 32/8/128/16; 1 chunk q=512 vs kv=8192; 256 decode kv ~ U{512..16384}
  c5  bf16 64/8/128/16; prefill q=kv {1000,3000,700,4096}; 512 decode x 4 tokens,
      kv ~ round(exp(ln 2048 + N(0,1))) clipped to [8, 32768]; window_left 4096;
      per-head fp32 sinks ~ N(0,1)

Values are N(0,1) drawn in fp32 from a seeded ``torch.Generator`` (CPU) and
rounded to the element type. Page ids are a random permutation of the pool
unless the workload says contiguous.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

__all__ = ["HalfInputs", "PODInputs", "make_half", "make_config", "make_custom",
           "CONFIG_NAMES", "page_table_from_lens", "pack_mask", "with_prefill_custom_mask",
           "with_kv_layout", "alibi_slopes", "with_decode_subset"]

CONFIG_NAMES = ("c1", "c2", "c3", "c4", "c5")


@dataclass
class HalfInputs:
    """One half (prefill or decode) of a POD call: host page tables + tensors."""
    q_indptr: np.ndarray          # int32 [B+1]
    kv_indptr: np.ndarray         # int32 [B+1] (in pages)
    kv_indices: np.ndarray        # int32 [kv_indptr[-1]]
    last_page_len: np.ndarray     # int32 [B]
    num_pages: int                # size of the page pool
    q: torch.Tensor               # [q_indptr[-1], H, d] fp16/bf16, CPU
    kv: torch.Tensor              # [num_pages, 2, ps, Hk, d] fp16/bf16, CPU
    q_lens: np.ndarray = field(default=None)   # int32 [B]
    kv_lens: np.ndarray = field(default=None)  # int32 [B]
    # custom mask (prefill half): uint8, the requests' [q_len, kv_len] boolean
    # matrices laid end to end, packed eight to a byte, little bit order
    packed_mask: Optional[np.ndarray] = None
    # page layout of kv: "NHD" [pages, 2, ps, Hk, d] or "HND" [pages, 2, Hk, ps, d]
    kv_layout: str = "NHD"

    @property
    def batch(self) -> int:
        return int(self.q_indptr.shape[0] - 1)

    @property
    def rows(self) -> int:
        return int(self.q_indptr[-1])


@dataclass
class PODInputs:
    name: str
    dtype: torch.dtype
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    causal: bool
    window_left: int
    sm_scale: float
    p: HalfInputs
    d: HalfInputs
    sinks: Optional[torch.Tensor]   # fp32 [H] or None
    # decode cache in FP8 E4M3: d.kv holds the codes; K = code * k_scale, V = code * v_scale
    k_scale: float = 1.0
    v_scale: float = 1.0
    # logits transform of both halves: soft cap (> 0) or per-head ALiBi slopes [H] fp32
    soft_cap: float = 0.0
    alibi: Optional[torch.Tensor] = None
    # rotary position encoding of both halves: (rope_scale, rope_theta) or None
    rope: Optional[tuple] = None


def page_table_from_lens(kv_lens: Sequence[int], page_size: int):
    """indptr / last_page_len for the given KV lengths, in the form the
    batch-POD docstring example builds them: pages = ceil(len / ps) and
    last = (len - 1) % ps + 1."""
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    pages = (kv_lens + page_size - 1) // page_size
    indptr = np.zeros(len(kv_lens) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(pages)
    last = np.where(kv_lens > 0, (kv_lens - 1) % page_size + 1, 0)
    return indptr.astype(np.int32), last.astype(np.int32)


def _randn(gen: torch.Generator, shape, dtype: torch.dtype, chunk: int = 1 << 26) -> torch.Tensor:
    """N(0,1) in fp32 rounded to ``dtype``, drawn in chunks so that multi-GB
    caches never need an fp32 copy of the whole tensor."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = torch.randn(e - s, generator=gen, dtype=torch.float32).to(dtype)
    return out.view(*shape)


def make_half(gen: torch.Generator, q_lens, kv_lens, H, Hk, d, ps, dtype,
              pages: str = "perm", extra_pages: int = 0,
              kv_indptr=None, last_page_len=None, with_data: bool = True) -> HalfInputs:
    """Build one half. ``pages`` is "perm" (random permutation of the pool),
    "contig" (0..n-1 in order). ``kv_indptr``/``last_page_len`` may be given
    directly (the single-request docstring example prints them)."""
    q_lens = np.asarray(q_lens, dtype=np.int64)
    if kv_indptr is None:
        kv_indptr, last_page_len = page_table_from_lens(kv_lens, ps)
    kv_indptr = np.asarray(kv_indptr, dtype=np.int32)
    last_page_len = np.asarray(last_page_len, dtype=np.int32)
    n_used = int(kv_indptr[-1])
    num_pages = n_used + int(extra_pages)
    if pages == "perm":
        perm = torch.randperm(num_pages, generator=gen).numpy()[:n_used]
        kv_indices = perm.astype(np.int32)
    elif pages == "contig":
        kv_indices = np.arange(n_used, dtype=np.int32)
    else:
        raise ValueError(pages)
    q_indptr = np.zeros(len(q_lens) + 1, dtype=np.int64)
    q_indptr[1:] = np.cumsum(q_lens)
    rows = int(q_indptr[-1])
    if with_data:
        q = _randn(gen, (rows, H, d), dtype)
        kv = _randn(gen, (max(num_pages, 1), 2, ps, Hk, d), dtype)
    else:   # page tables only (planner tests); tensors are empty placeholders
        q = torch.empty((0, H, d), dtype=dtype)
        kv = torch.empty((0, 2, ps, Hk, d), dtype=dtype)
    npg = kv_indptr[1:] - kv_indptr[:-1]
    kv_lens_arr = np.where(npg > 0, (npg - 1) * ps + last_page_len, 0).astype(np.int32)
    return HalfInputs(q_indptr=q_indptr.astype(np.int32), kv_indptr=kv_indptr,
                      kv_indices=kv_indices, last_page_len=last_page_len,
                      num_pages=max(num_pages, 1), q=q, kv=kv,
                      q_lens=q_lens.astype(np.int32), kv_lens=kv_lens_arr)


def _empty_half(gen, H, Hk, d, ps, dtype) -> HalfInputs:
    return make_half(gen, [], [], H, Hk, d, ps, dtype)


def make_custom(name, dtype, H, Hk, d, ps, causal, window_left,
                p_q_lens, p_kv_lens, d_q_lens, d_kv_lens, seed=0,
                sinks=False, pages="perm", sm_scale=None, extra_pages=0) -> PODInputs:
    gen = torch.Generator().manual_seed(int(seed))
    p = make_half(gen, p_q_lens, p_kv_lens, H, Hk, d, ps, dtype, pages, extra_pages)
    dd = make_half(gen, d_q_lens, d_kv_lens, H, Hk, d, ps, dtype, pages, extra_pages)
    s = torch.randn(H, generator=gen, dtype=torch.float32) if sinks else None
    return PODInputs(name=name, dtype=dtype, num_qo_heads=H, num_kv_heads=Hk, head_dim=d,
                     page_size=ps, causal=bool(causal), window_left=int(window_left),
                     sm_scale=(1.0 / math.sqrt(d)) if sm_scale is None else float(sm_scale),
                     p=p, d=dd, sinks=s)


def make_config(name: str, seed: Optional[int] = None, with_data: bool = True) -> PODInputs:
    """The five benchmark workloads. Seed defaults to the config index (1..5).
    ``with_data=False`` builds the page tables only (same page ids as with data
    only for the "contig" workloads, since tensor draws share the generator)."""
    idx = CONFIG_NAMES.index(name) + 1
    gen = torch.Generator().manual_seed(idx if seed is None else int(seed))
    import functools
    make_half_l = functools.partial(make_half, with_data=with_data)
    if name == "c1":
        H, Hk, d, ps, dt = 4, 1, 64, 16, torch.float16
        p = make_half_l(gen, [64], [64], H, Hk, d, ps, dt, "perm")
        dd = make_half_l(gen, [1] * 4, [17, 29, 5, 48], H, Hk, d, ps, dt, "perm")
        return PODInputs(name, dt, H, Hk, d, ps, True, -1, 1.0 / math.sqrt(d), p, dd, None)
    if name == "c2":
        H, Hk, d, ps, dt = 64, 8, 128, 16, torch.float16
        p = make_half_l(gen, [1024], [1024], H, Hk, d, ps, dt, "contig")
        dd = make_half_l(gen, [1] * 7, None, H, Hk, d, ps, dt, "contig",
                       kv_indptr=[0, 17, 29, 44, 48, 66, 100, 128],
                       last_page_len=[1, 7, 14, 4, 3, 1, 16])
        return PODInputs(name, dt, H, Hk, d, ps, True, -1, 1.0 / math.sqrt(d), p, dd, None)
    if name == "c3":
        H, Hk, d, ps, dt = 64, 8, 128, 1, torch.bfloat16
        p = make_half_l(gen, [2048] * 2, [2048] * 2, H, Hk, d, ps, dt, "contig")
        dd = make_half_l(gen, [1] * 128, [2048] * 128, H, Hk, d, ps, dt, "contig")
        return PODInputs(name, dt, H, Hk, d, ps, True, -1, 1.0 / math.sqrt(d), p, dd, None)
    if name == "c4":
        H, Hk, d, ps, dt = 32, 8, 128, 16, torch.bfloat16
        kv_d = torch.randint(512, 16384 + 1, (256,), generator=gen).numpy()
        p = make_half_l(gen, [512], [8192], H, Hk, d, ps, dt, "perm")
        dd = make_half_l(gen, [1] * 256, kv_d, H, Hk, d, ps, dt, "perm")
        return PODInputs(name, dt, H, Hk, d, ps, True, -1, 1.0 / math.sqrt(d), p, dd, None)
    if name == "c5":
        H, Hk, d, ps, dt = 64, 8, 128, 16, torch.bfloat16
        z = torch.randn(512, generator=gen, dtype=torch.float64).numpy()
        kv_d = np.clip(np.rint(np.exp(math.log(2048.0) + z)), 8, 32768).astype(np.int64)
        p = make_half_l(gen, [1000, 3000, 700, 4096], [1000, 3000, 700, 4096], H, Hk, d, ps, dt, "perm")
        dd = make_half_l(gen, [4] * 512, kv_d, H, Hk, d, ps, dt, "perm")
        sinks = torch.randn(H, generator=gen, dtype=torch.float32)
        return PODInputs(name, dt, H, Hk, d, ps, True, 4096, 1.0 / math.sqrt(d), p, dd, sinks)
    raise ValueError(f"unknown workload {name!r}")


def with_fp8_decode_cache(inp: PODInputs, k_scale: float = 0.02, v_scale: float = 0.03) -> PODInputs:
    """The same inputs with the decode half's cache stored as FP8 E4M3 codes:
    K / k_scale and V / v_scale rounded to E4M3 (torch's conversion), so the
    dequantized cache code * scale is close to the 16-bit one. Returns a new
    PODInputs; the prefill half is untouched."""
    import copy
    out = copy.copy(inp)
    d = copy.copy(inp.d)
    kv = inp.d.kv.float()
    scaled = torch.empty_like(kv)
    scaled[:, 0] = kv[:, 0] / k_scale
    scaled[:, 1] = kv[:, 1] / v_scale
    d.kv = scaled.to(torch.float8_e4m3fn)
    out.d = d
    out.k_scale = float(k_scale)
    out.v_scale = float(v_scale)
    return out


def pack_mask(mats: Sequence[np.ndarray]) -> np.ndarray:
    """Boolean [q_len, kv_len] matrices, one per request, laid end to end in
    row-major order and packed eight to a byte with the first element in the
    least significant bit (numpy's little bit order)."""
    flat = [np.asarray(m, dtype=bool).reshape(-1) for m in mats]
    bits = np.concatenate(flat) if flat else np.zeros(0, dtype=bool)
    return np.packbits(bits, bitorder="little")


def with_prefill_custom_mask(inp: PODInputs, seed: int = 0, density: float = 0.5,
                             empty_rows: int = 1, full_rows: int = 1) -> PODInputs:
    """The same inputs with a random custom mask on the prefill half: each
    (query row, key) allowed with probability ``density``; in every request
    with enough rows, the first ``empty_rows`` rows allow no key and the next
    ``full_rows`` rows allow every key. Returns a new PODInputs."""
    import copy
    gen = torch.Generator().manual_seed(int(seed))
    mats = []
    for r in range(inp.p.batch):
        ql = int(inp.p.q_indptr[r + 1] - inp.p.q_indptr[r])
        kl = int(inp.p.kv_lens[r])
        m = (torch.rand((ql, kl), generator=gen) < density).numpy()
        if ql > empty_rows + full_rows:
            m[:empty_rows] = False
            m[empty_rows:empty_rows + full_rows] = True
        mats.append(m)
    out = copy.copy(inp)
    p = copy.copy(inp.p)
    p.packed_mask = pack_mask(mats)
    out.p = p
    return out


def with_kv_layout(inp: PODInputs, layout: str = "HND", halves: str = "pd") -> PODInputs:
    """The same inputs with the caches of ``halves`` ("p", "d" or "pd") stored
    in ``layout``: the same keys and values, pages reordered from
    [2, ps, Hk, d] (NHD) to [2, Hk, ps, d] (HND) or back. Returns a new
    PODInputs."""
    import copy
    out = copy.copy(inp)
    for name in halves:
        h = copy.copy(getattr(inp, name))
        if h.kv_layout != layout:
            h.kv = h.kv.permute(0, 1, 3, 2, 4).contiguous()
            h.kv_layout = layout
        setattr(out, name, h)
    return out


def alibi_slopes(num_heads: int) -> torch.Tensor:
    """The geometric head slopes of the ALiBi paper for a power-of-two head
    count: 2^(-8 (h + 1) / H), h = 0..H-1 (fp32)."""
    h = torch.arange(1, num_heads + 1, dtype=torch.float64)
    return torch.pow(2.0, -8.0 * h / num_heads).to(torch.float32)


def with_decode_subset(inp: PODInputs, n: int) -> PODInputs:
    """The same inputs with only the first ``n`` decode requests. Their pages
    are copied into a compact pool (the pages keep their relative order, so a
    permuted pool stays permuted), so the device holds only what they use; a
    smaller case of the same decode distribution for profiler captures.
    Returns a new PODInputs; the prefill half is untouched."""
    import copy
    n = max(0, min(int(n), inp.d.batch))
    out = copy.copy(inp)
    d = copy.copy(inp.d)
    used = np.asarray(inp.d.kv_indices[: int(inp.d.kv_indptr[n])], dtype=np.int64)
    keep = np.unique(used)
    d.q_indptr = np.ascontiguousarray(inp.d.q_indptr[: n + 1])
    d.kv_indptr = np.ascontiguousarray(inp.d.kv_indptr[: n + 1])
    d.last_page_len = np.ascontiguousarray(inp.d.last_page_len[:n])
    d.kv_indices = np.searchsorted(keep, used).astype(np.int32)
    d.num_pages = max(int(len(keep)), 1)
    # gathered as bytes: CPU indexing has no float8 kernels
    raw = inp.d.kv.view(torch.uint8)
    raw = raw[torch.from_numpy(keep)] if len(keep) else raw[:1].clone()
    d.kv = raw.view(inp.d.kv.dtype)
    d.q = inp.d.q[: int(inp.d.q_indptr[n])].clone()
    d.q_lens = np.ascontiguousarray(inp.d.q_lens[:n])
    d.kv_lens = np.ascontiguousarray(inp.d.kv_lens[:n])
    out.d = d
    return out
