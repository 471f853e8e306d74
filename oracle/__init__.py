"""fp64 CPU oracle for POD paged attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package. The product path
(``prefill_decode_paged_pod_gb300``) never imports, links or calls it, and this
package imports nothing from the product.

The arithmetic lives in ``pod_oracle.c`` (plain C, fp64); this module only
compiles it with gcc, marshals numpy arrays through ctypes and offers the
convenience wrappers the tests use. ``planner_ref`` restates the integer
planning rules for the bit-exact check of the host planner.

Parity status per function (see the pins in tests/test_oracle_pins.py):
  attention_rows / attention_half   pinned (brute force, invariances, closed
                                    forms, hand-worked example, split/merge)
  merge                             pinned (split/merge identity)
  seq_lens                          pinned (closed form from the page tables)
  FP8 (E4M3) cache path             pinned (exhaustive decoder check against the
                                    format's definition and torch; dequantized
                                    brute force; scale folding identities)
  sink-in-LSE convention            pinned to the reading taken (sink excluded)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pod_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpod_oracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            _lib.oracle_attention_rows.restype = ctypes.c_int
            _lib.oracle_attention_rows.argtypes = [
                P, P, ctypes.c_int,
                P, P, P, P, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                P, ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int]
            _lib.oracle_merge.restype = None
            _lib.oracle_merge.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
                                          ctypes.c_double, P, P]
            _lib.oracle_seq_lens.restype = None
            _lib.oracle_seq_lens.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P]
            _lib.oracle_f16_to_f64.restype = ctypes.c_double
            _lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            _lib.oracle_bf16_to_f64.restype = ctypes.c_double
            _lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            _lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            _lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            _lib.oracle_attention_rows_masked.restype = ctypes.c_int
            _lib.oracle_attention_rows_masked.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                P, P, P, P, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                P, P, ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int]
            _lib.oracle_attention_rows_ext.restype = ctypes.c_int
            _lib.oracle_attention_rows_ext.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                P, P, P, P, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double, P,
                ctypes.c_int, ctypes.c_double, ctypes.c_double,
                P, P, ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int]
            _lib.oracle_attention_rows_kv.restype = ctypes.c_int
            _lib.oracle_attention_rows_kv.argtypes = [
                P, P, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                P, P, P, P, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double,
                P, ctypes.c_int64, P, P, P, P, P, P, ctypes.c_int]
        return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _codes(t) -> np.ndarray:
    """16-bit codes of an fp16/bf16 torch tensor (or numpy uint16 array)."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t.view(np.uint16))
    import torch
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def is_fp8(t) -> bool:
    """True for an FP8 E4M3 torch tensor (the cache format the oracle reads
    as E4M3 codes)."""
    import torch
    return getattr(t, "dtype", None) == torch.float8_e4m3fn


def _codes8(t) -> np.ndarray:
    """8-bit codes of an E4M3 torch tensor (or numpy uint8 array)."""
    if isinstance(t, np.ndarray):
        return np.ascontiguousarray(t.view(np.uint8))
    import torch
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.uint8).numpy())


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"oracle takes fp16/bf16 inputs, got {t.dtype}")


def attention_rows(q, kv, q_indptr, kv_indptr, kv_indices, last_page_len,
                   num_qo_heads, num_kv_heads, head_dim, page_size,
                   causal, window_left, sm_scale, sinks=None,
                   sel_token=None, sel_head=None, key_lo=None, key_hi=None,
                   nthreads: Optional[int] = None, dtype: Optional[int] = None,
                   k_scale: float = 1.0, v_scale: float = 1.0, packed_mask=None,
                   kv_layout: int = 0, soft_cap: float = 0.0, alibi_slopes=None,
                   rope: bool = False, rope_scale: float = 1.0, rope_theta: float = 1e4):
    """fp64 outputs for selected (token, head) pairs; all pairs if no selection.
    An E4M3 ``kv`` is read as codes times ``k_scale`` (K) / ``v_scale`` (V).
    ``packed_mask`` (uint8, little bit order) is a custom mask over every
    request's [q_len, kv_len] matrix; it replaces the causal rule.
    ``kv_layout`` 0 = NHD pages [2, ps, Hk, d], 1 = HND [2, Hk, ps, d];
    ``soft_cap`` > 0 caps the scaled logits (cap * tanh(x / cap));
    ``alibi_slopes`` [H] adds slope * (t - p) to each logit;
    ``rope`` rotates q (at p) and keys (at t) by the LLaMA rotary embedding.

    Returns (out [n, d] float64, lse [n] float64, status int).
    """
    qc = _codes(q)
    kv_fp8 = is_fp8(kv)
    kvc = _codes8(kv) if kv_fp8 else _codes(kv)
    if dtype is None:
        dtype = dtype_code(q)
    q_indptr = np.ascontiguousarray(q_indptr, dtype=np.int32)
    kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
    last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
    batch = len(q_indptr) - 1
    rows = int(q_indptr[-1]) if batch >= 0 and len(q_indptr) else 0
    H, d = int(num_qo_heads), int(head_dim)
    if sel_token is None:
        tok = np.repeat(np.arange(rows, dtype=np.int64), H)
        hd = np.tile(np.arange(H, dtype=np.int32), rows)
    else:
        tok = np.ascontiguousarray(sel_token, dtype=np.int64)
        hd = np.ascontiguousarray(sel_head, dtype=np.int32)
    n = int(tok.shape[0])
    out = np.zeros((max(n, 1), d), dtype=np.float64)
    lse = np.zeros(max(n, 1), dtype=np.float64)
    if key_lo is not None:
        key_lo = np.ascontiguousarray(key_lo, dtype=np.int64)
        key_hi = np.ascontiguousarray(key_hi, dtype=np.int64)
    sk = None
    if sinks is not None:
        sk = np.ascontiguousarray(np.asarray(sinks.cpu() if hasattr(sinks, "cpu") else sinks,
                                             dtype=np.float32))
    num_pages = int(kvc.shape[0]) if kvc.ndim >= 1 else 0
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    pm = None
    if packed_mask is not None:
        pm = np.ascontiguousarray(np.asarray(packed_mask.cpu() if hasattr(packed_mask, "cpu")
                                             else packed_mask, dtype=np.uint8))
        npg = np.diff(kv_indptr).astype(np.int64)
        kvl = np.where(npg > 0, (npg - 1) * int(page_size) + last_page_len, 0)
        need = int(np.sum(np.diff(q_indptr).astype(np.int64) * kvl))
        if pm.size * 8 < need:
            raise ValueError(f"packed_mask holds {pm.size * 8} bits, the requests need {need}")
    al = None
    if alibi_slopes is not None:
        al = np.ascontiguousarray(np.asarray(alibi_slopes.cpu() if hasattr(alibi_slopes, "cpu")
                                             else alibi_slopes, dtype=np.float32))
    st = lib().oracle_attention_rows_ext(
        _ptr(qc), _ptr(kvc), int(dtype), int(kv_fp8), float(k_scale), float(v_scale),
        _ptr(q_indptr), _ptr(kv_indptr), _ptr(kv_indices), _ptr(last_page_len),
        batch, num_pages, H, int(num_kv_heads), d, int(page_size), int(kv_layout),
        int(bool(causal)), int(window_left), float(sm_scale), float(soft_cap), _ptr(al),
        int(bool(rope)), float(rope_scale), float(rope_theta),
        _ptr(sk), _ptr(pm), n, _ptr(tok), _ptr(hd), _ptr(key_lo), _ptr(key_hi),
        _ptr(out), _ptr(lse), int(nthreads))
    return out[:n], lse[:n], int(st)


def attention_half(inp, half: str, sel_token=None, sel_head=None, nthreads=None, **kw):
    """Oracle for one half ("p" or "d") of a ``pod_workloads.PODInputs``."""
    h = inp.p if half == "p" else inp.d
    scales = {}
    if is_fp8(h.kv):
        scales = dict(k_scale=getattr(inp, "k_scale", 1.0), v_scale=getattr(inp, "v_scale", 1.0))
    if getattr(h, "packed_mask", None) is not None and "packed_mask" not in kw:
        scales["packed_mask"] = h.packed_mask
    if getattr(h, "kv_layout", "NHD") == "HND" and "kv_layout" not in kw:
        scales["kv_layout"] = 1
    if getattr(inp, "soft_cap", 0.0) and "soft_cap" not in kw:
        scales["soft_cap"] = float(inp.soft_cap)
    if getattr(inp, "alibi", None) is not None and "alibi_slopes" not in kw:
        scales["alibi_slopes"] = inp.alibi
    if getattr(inp, "rope", None) is not None and "rope" not in kw:
        scales.update(rope=True, rope_scale=float(inp.rope[0]), rope_theta=float(inp.rope[1]))
    return attention_rows(h.q, h.kv, h.q_indptr, h.kv_indptr, h.kv_indices, h.last_page_len,
                          inp.num_qo_heads, inp.num_kv_heads, inp.head_dim, inp.page_size,
                          inp.causal, inp.window_left, inp.sm_scale, sinks=inp.sinks,
                          sel_token=sel_token, sel_head=sel_head, nthreads=nthreads,
                          **scales, **kw)


def merge(o_parts: np.ndarray, lse_parts: np.ndarray, sink: Optional[float] = None):
    """Merge split partials (o_i, lse_i) of one (row, head) -> (o, lse)."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib().oracle_merge(n, d, _ptr(o_parts), _ptr(lse_parts), int(sink is not None),
                       float(sink) if sink is not None else 0.0, _ptr(o), _ptr(lse))
    return o, float(lse[0])


def seq_lens(kv_indptr, last_page_len, page_size) -> np.ndarray:
    kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
    b = len(kv_indptr) - 1
    out = np.zeros(max(b, 1), dtype=np.int32)
    lib().oracle_seq_lens(_ptr(kv_indptr), _ptr(last_page_len), b, int(page_size), _ptr(out))
    return out[:b]


def f16_to_f64(code: int) -> float:
    return lib().oracle_f16_to_f64(int(code))


def bf16_to_f64(code: int) -> float:
    return lib().oracle_bf16_to_f64(int(code))


def e4m3_to_f64(code: int) -> float:
    return lib().oracle_e4m3_to_f64(int(code))
