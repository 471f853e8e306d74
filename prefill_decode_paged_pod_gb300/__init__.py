"""GB300 (sm_103a) POD paged attention: Python binding of the C ABI in include/pod.h.

This module only marshals arguments: host page tables as int32 numpy arrays,
device tensors as raw pointers, the current torch CUDA stream as a handle.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback. If the shared library is missing or cannot be loaded
the import of the binding raises.

    h = pod_plan(p_q_indptr, p_kv_indptr, p_kv_indices, p_last_page_len,
                 d_q_indptr, d_kv_indptr, d_kv_indices, d_last_page_len,
                 num_qo_heads, num_kv_heads, head_dim, page_size,
                 causal, window_left, sm_scale, dtype=torch.bfloat16,
                 p_num_pages=..., d_num_pages=..., has_sinks=False, workspace=ws)
    out_p, lse_p, out_d, lse_d = pod_run(h, q_p, kv_p, q_d, kv_d, ws, sinks=None)

The names and the plan-once / run-many life cycle follow the POD walkthrough
("plan/run 生命周期", "BatchPOD 的 run 差异").
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

__all__ = [
    "POD_OK", "PodError", "load_library", "pod_plan", "pod_run", "pod_destroy",
    "pod_workspace_size", "pod_bind_workspace", "pod_last_error", "pod_read_device_status",
    "pod_plan_table", "PodHandle", "LIB_PATH", "DEFAULT_WORKSPACE_BYTES",
    "pod_run_static_scratch", "pod_static_scratch_capacity", "pod_plan_set_decode_fp8",
    "pod_plan_set_prefill_mask", "pod_plan_set_kv_layout", "pod_plan_set_logits_transform",
    "pod_plan_set_rope", "pod_plan_set_graph_capacity", "pod_replan",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libpod_gb300.so")
POD_OK = 0
_STATUS = {0: "POD_OK", 1: "POD_ERR_INVALID_ARG", 2: "POD_ERR_UNSUPPORTED", 3: "POD_ERR_WORKSPACE",
           4: "POD_ERR_CUDA", 5: "POD_ERR_DEVICE_STATUS"}
# the pages recommend a 128 MB workspace for typical POD use
DEFAULT_WORKSPACE_BYTES = 128 * 1024 * 1024

_lib = None


class PodError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_STATUS.get(code, code)}: {msg}")
        self.code = code


def load_library(path: Optional[str] = None):
    """Load the C-ABI library (built by ``__graft_entry__.build()``). Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"POD CUDA library not built: {p} is missing "
                           "(run __graft_entry__.build() or prefill_decode_paged_pod_gb300/_build.py)")
    lib = ctypes.CDLL(p)
    V, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    lib.pod_plan.restype = ctypes.c_int
    lib.pod_plan.argtypes = [V, V, V, V, I32, I32, V, V, V, V, I32, I32,
                             I32, I32, I32, I32, I32, I32, ctypes.c_float, ctypes.c_int, I32, I32,
                             V, SZ, V, ctypes.POINTER(V), ctypes.POINTER(SZ)]
    lib.pod_workspace_size.restype = SZ
    lib.pod_workspace_size.argtypes = [V]
    lib.pod_bind_workspace.restype = ctypes.c_int
    lib.pod_bind_workspace.argtypes = [V, V, SZ, V]
    lib.pod_run.restype = ctypes.c_int
    lib.pod_run.argtypes = [V, V, V, V, V, V, V, V, V, V, V, V]
    lib.pod_destroy.restype = ctypes.c_int
    lib.pod_destroy.argtypes = [V]
    lib.pod_last_error.restype = ctypes.c_char_p
    lib.pod_last_error.argtypes = []
    lib.pod_read_device_status.restype = ctypes.c_int
    lib.pod_read_device_status.argtypes = [V, V, V, ctypes.POINTER(I32)]
    lib.pod_plan_table.restype = ctypes.c_int
    lib.pod_plan_table.argtypes = [V, I32, V, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
    lib.pod_run_static_scratch.restype = ctypes.c_int
    lib.pod_run_static_scratch.argtypes = [V, V, V, V, V, V, V, V, V, V, V]
    lib.pod_static_scratch_capacity.restype = SZ
    lib.pod_static_scratch_capacity.argtypes = []
    lib.pod_plan_set_decode_fp8.restype = ctypes.c_int
    lib.pod_plan_set_decode_fp8.argtypes = [V, ctypes.c_float, ctypes.c_float]
    lib.pod_plan_set_rope.restype = ctypes.c_int
    lib.pod_plan_set_rope.argtypes = [V, ctypes.c_float, ctypes.c_float]
    lib.pod_plan_set_logits_transform.restype = ctypes.c_int
    lib.pod_plan_set_logits_transform.argtypes = [V, ctypes.c_float, V]
    lib.pod_plan_set_kv_layout.restype = ctypes.c_int
    lib.pod_plan_set_kv_layout.argtypes = [V, I32, I32]
    lib.pod_plan_set_prefill_mask.restype = ctypes.c_int
    lib.pod_plan_set_prefill_mask.argtypes = [V, V, ctypes.c_int64]
    lib.pod_plan_set_graph_capacity.restype = ctypes.c_int
    lib.pod_plan_set_graph_capacity.argtypes = [V] + [I32] * 6
    lib.pod_replan.restype = ctypes.c_int
    lib.pod_replan.argtypes = [V, V, V, V, V, I32, V, V, V, V, I32, V]
    if path is None:
        _lib = lib
    return lib


def pod_last_error() -> str:
    return load_library().pod_last_error().decode()


def _check(code: int):
    if code != POD_OK:
        raise PodError(code, pod_last_error())


def _i32(a) -> Optional[np.ndarray]:
    if a is None:
        return None
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return a.data_ptr()


def _stream(stream=None) -> Optional[int]:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    if not torch.cuda.is_available():
        return None
    return torch.cuda.current_stream().cuda_stream


def _dtype_code(dtype) -> int:
    import torch
    if dtype in (torch.float16, "float16", "fp16", 0):
        return 0
    if dtype in (torch.bfloat16, "bfloat16", "bf16", 1):
        return 1
    raise PodError(2, f"unsupported dtype {dtype}")


@dataclass
class PodHandle:
    """Owns a plan handle of the C library (released by ``pod_destroy``)."""
    ptr: int
    workspace_bytes: int
    p_rows: int
    d_rows: int
    num_qo_heads: int
    head_dim: int
    dtype: object
    has_sinks: bool
    workspace_ptr: Optional[int] = None
    d_kv_fp8: bool = False      # set by pod_plan_set_decode_fp8
    p_mask: object = None       # custom prefill mask, kept alive while the plan uses it
    alibi: object = None        # ALiBi slopes, kept alive while the plan uses them

    def __del__(self):
        if self.ptr and _lib is not None:
            _lib.pod_destroy(ctypes.c_void_p(self.ptr))
            self.ptr = 0


def pod_plan(p_q_indptr, p_kv_indptr, p_kv_indices, p_last_page_len,
             d_q_indptr, d_kv_indptr, d_kv_indices, d_last_page_len,
             num_qo_heads, num_kv_heads, head_dim, page_size,
             causal=True, window_left=-1, sm_scale=None, *, dtype, p_num_pages, d_num_pages,
             has_sinks=False, num_sms=0, workspace=None, stream=None) -> PodHandle:
    """Plan a POD launch. Index arrays are host int32 (numpy or CPU tensors).

    ``workspace`` is a device uint8 tensor (or None for a host-only plan that
    can be bound later with ``pod_bind_workspace``).
    """
    lib = load_library()
    arrs = [_i32(x) for x in (p_q_indptr, p_kv_indptr, p_kv_indices, p_last_page_len,
                              d_q_indptr, d_kv_indptr, d_kv_indices, d_last_page_len)]
    p_batch = 0 if arrs[0] is None else len(arrs[0]) - 1
    d_batch = 0 if arrs[4] is None else len(arrs[4]) - 1
    handle = ctypes.c_void_p()
    req = ctypes.c_size_t(0)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    code = lib.pod_plan(*[_ptr(a) for a in arrs[:4]], p_batch, int(p_num_pages),
                        *[_ptr(a) for a in arrs[4:]], d_batch, int(d_num_pages),
                        int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size),
                        int(bool(causal)), int(window_left),
                        float(sm_scale) if sm_scale is not None else 0.0,
                        _dtype_code(dtype), int(bool(has_sinks)), int(num_sms),
                        ws_ptr, ws_bytes, _stream(stream) if ws_ptr else None,
                        ctypes.byref(handle), ctypes.byref(req))
    if code != POD_OK:
        err = PodError(code, pod_last_error())
        err.required_workspace_bytes = int(req.value)
        raise err
    p_rows = 0 if arrs[0] is None or p_batch == 0 else int(arrs[0][-1])
    d_rows = 0 if arrs[4] is None or d_batch == 0 else int(arrs[4][-1])
    return PodHandle(ptr=handle.value, workspace_bytes=int(req.value), p_rows=p_rows,
                     d_rows=d_rows, num_qo_heads=int(num_qo_heads), head_dim=int(head_dim),
                     dtype=dtype, has_sinks=bool(has_sinks), workspace_ptr=ws_ptr)


def pod_workspace_size(h: PodHandle) -> int:
    return int(load_library().pod_workspace_size(ctypes.c_void_p(h.ptr)))


def pod_bind_workspace(h: PodHandle, workspace, stream=None):
    lib = load_library()
    _check(lib.pod_bind_workspace(ctypes.c_void_p(h.ptr), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))
    h.workspace_ptr = workspace.data_ptr()


def pod_run(h: PodHandle, q_p, kv_p, q_d, kv_d, workspace, sinks=None,
            out_p=None, lse_p=None, out_d=None, lse_d=None, stream=None):
    """One fused POD launch. Returns (out_p, lse_p, out_d, lse_d); outputs are
    allocated with torch on the inputs' device when not given."""
    import torch
    lib = load_library()
    H, d = h.num_qo_heads, h.head_dim
    dev = None
    for t in (q_p, q_d, workspace):
        if t is not None:
            dev = t.device
            break
    if out_p is None:
        out_p = torch.empty((h.p_rows, H, d), dtype=h.dtype, device=dev)
    if lse_p is None:
        lse_p = torch.empty((h.p_rows, H), dtype=torch.float32, device=dev)
    if out_d is None:
        out_d = torch.empty((h.d_rows, H, d), dtype=h.dtype, device=dev)
    if lse_d is None:
        lse_d = torch.empty((h.d_rows, H), dtype=torch.float32, device=dev)
    for name, t in (("q_p", q_p), ("kv_p", kv_p), ("q_d", q_d), ("kv_d", kv_d)):
        want = torch.float8_e4m3fn if (name == "kv_d" and h.d_kv_fp8) else h.dtype
        if t is not None and (not t.is_contiguous() or t.dtype != want):
            raise PodError(1, f"{name} must be contiguous {want}")
    _check_mask_device(h)
    p_empty, d_empty = h.p_rows == 0, h.d_rows == 0
    code = lib.pod_run(ctypes.c_void_p(h.ptr),
                       None if p_empty else _ptr(q_p), None if p_empty else _ptr(kv_p),
                       None if d_empty else _ptr(q_d), None if d_empty else _ptr(kv_d),
                       _ptr(sinks), _ptr(workspace),
                       None if p_empty else _ptr(out_p), None if p_empty else _ptr(lse_p),
                       None if d_empty else _ptr(out_d), None if d_empty else _ptr(lse_d),
                       _stream(stream))
    _check(code)
    return out_p, lse_p, out_d, lse_d


def pod_static_scratch_capacity() -> int:
    return int(load_library().pod_static_scratch_capacity())


def pod_run_static_scratch(h: PodHandle, q_p, kv_p, q_d, kv_d, sinks=None,
                           out_p=None, lse_p=None, out_d=None, lse_d=None, stream=None):
    """Like pod_run, but the kernels' scratch is the library's fixed device
    array instead of a caller-allocated workspace (for callers that cannot
    allocate device memory). Output tensors are allocated here when not given;
    pass them to keep the call free of allocations. Calls sharing a device must
    not overlap on the GPU."""
    import torch
    lib = load_library()
    H, d = h.num_qo_heads, h.head_dim
    dev = q_p.device if q_p is not None else (q_d.device if q_d is not None else None)
    if out_p is None:
        out_p = torch.empty((h.p_rows, H, d), dtype=h.dtype, device=dev)
    if lse_p is None:
        lse_p = torch.empty((h.p_rows, H), dtype=torch.float32, device=dev)
    if out_d is None:
        out_d = torch.empty((h.d_rows, H, d), dtype=h.dtype, device=dev)
    if lse_d is None:
        lse_d = torch.empty((h.d_rows, H), dtype=torch.float32, device=dev)
    _check_mask_device(h)
    p_empty, d_empty = h.p_rows == 0, h.d_rows == 0
    code = lib.pod_run_static_scratch(
        ctypes.c_void_p(h.ptr),
        None if p_empty else _ptr(q_p), None if p_empty else _ptr(kv_p),
        None if d_empty else _ptr(q_d), None if d_empty else _ptr(kv_d), _ptr(sinks),
        None if p_empty else _ptr(out_p), None if p_empty else _ptr(lse_p),
        None if d_empty else _ptr(out_d), None if d_empty else _ptr(lse_d), _stream(stream))
    _check(code)
    return out_p, lse_p, out_d, lse_d


def pod_destroy(h: PodHandle):
    if h.ptr:
        load_library().pod_destroy(ctypes.c_void_p(h.ptr))
        h.ptr = 0


def pod_read_device_status(h: PodHandle, workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    code = load_library().pod_read_device_status(ctypes.c_void_p(h.ptr), workspace.data_ptr(),
                                                 _stream(stream), ctypes.byref(v))
    if code not in (POD_OK, 5):
        _check(code)
    return int(v.value)


def pod_plan_table(h: PodHandle, which: int) -> np.ndarray:
    lib = load_library()
    n = ctypes.c_int64(0)
    _check(lib.pod_plan_table(ctypes.c_void_p(h.ptr), int(which), None, 0, ctypes.byref(n)))
    out = np.zeros(max(n.value, 1), dtype=np.int32)
    _check(lib.pod_plan_table(ctypes.c_void_p(h.ptr), int(which), out.ctypes.data, n.value,
                              ctypes.byref(n)))
    return out[:n.value]


# summary indices of pod_plan_table(h, 0), mirroring enum PodSummary in csrc/pod_plan.h
SUMMARY_FIELDS = ("H", "Hk", "d", "ps", "causal", "window", "dtype", "sinks", "num_sms", "grid",
                  "n_p_ctas", "n_d_ctas", "n_tiles", "n_items", "n_groups", "n_mrows", "n_prows",
                  "p_rows", "d_rows", "p_batch", "d_batch", "decode_chunk", "ws_lo", "ws_hi",
                  "p_tma", "d_tma", "p_mask", "rope")


def plan_summary(h: PodHandle) -> dict:
    s = pod_plan_table(h, 0)
    return {k: int(v) for k, v in zip(SUMMARY_FIELDS, s)}


def pod_plan_set_decode_fp8(h: PodHandle, k_scale: float, v_scale: float):
    """The decode cache is FP8 E4M3 codes; K = code * k_scale, V = code * v_scale."""
    _check(load_library().pod_plan_set_decode_fp8(ctypes.c_void_p(h.ptr), float(k_scale),
                                                  float(v_scale)))
    h.d_kv_fp8 = True


def pod_plan_set_prefill_mask(h: PodHandle, packed_mask):
    """Custom prefill mask: uint8 bits (little bit order) of every prefill
    request's [q_len, kv_len] matrix, end to end; None removes it. A CUDA
    tensor for runs; a CPU tensor or numpy array serves host-only plans
    (inspection), whose pointer the library never reads. Switching the mask
    on or off re-plans the handle and releases its workspace: bind again."""
    lib = load_library()
    if packed_mask is None:
        _check(lib.pod_plan_set_prefill_mask(ctypes.c_void_p(h.ptr), None, 0))
        h.p_mask = None
    else:
        if isinstance(packed_mask, np.ndarray):
            packed_mask = np.ascontiguousarray(packed_mask, dtype=np.uint8)
            ptr, nbytes = packed_mask.ctypes.data, packed_mask.nbytes
        else:
            import torch
            if packed_mask.dtype != torch.uint8 or not packed_mask.is_contiguous():
                raise PodError(1, "packed_mask must be a contiguous uint8 tensor")
            ptr, nbytes = packed_mask.data_ptr(), packed_mask.numel()
        _check(lib.pod_plan_set_prefill_mask(ctypes.c_void_p(h.ptr), ptr, int(nbytes)))
        h.p_mask = packed_mask
    h.workspace_bytes = pod_workspace_size(h)
    h.workspace_ptr = None


def pod_plan_set_logits_transform(h: PodHandle, soft_cap: float = 0.0, alibi_slopes=None):
    """Logits soft cap (cap * tanh(x / cap) of the scaled logit; 0 = off) or
    ALiBi slopes (fp32 [H]; a CUDA tensor for runs, any tensor for host-only
    plans), applied by both halves."""
    ptr = None
    if alibi_slopes is not None:
        import torch
        if alibi_slopes.dtype != torch.float32 or not alibi_slopes.is_contiguous() \
                or alibi_slopes.numel() != h.num_qo_heads:
            raise PodError(1, "alibi_slopes must be a contiguous float32 tensor of num_qo_heads")
        ptr = alibi_slopes.data_ptr()
    _check(load_library().pod_plan_set_logits_transform(ctypes.c_void_p(h.ptr), float(soft_cap),
                                                        ptr))
    h.alibi = alibi_slopes


def pod_plan_set_rope(h: PodHandle, rope_scale: float = 1.0, rope_theta: float = 1e4):
    """ROPE_LLAMA on both halves (rope_scale 0 turns it off). Plans the handle
    again and releases its workspace: bind again."""
    _check(load_library().pod_plan_set_rope(ctypes.c_void_p(h.ptr), float(rope_scale),
                                            float(rope_theta)))
    h.workspace_bytes = pod_workspace_size(h)
    h.workspace_ptr = None


_LAYOUTS = {"NHD": 0, "HND": 1, 0: 0, 1: 1}


def pod_plan_set_kv_layout(h: PodHandle, p_layout="NHD", d_layout="NHD"):
    """Page layout of each half's cache: "NHD" [pages, 2, ps, Hk, d] or
    "HND" [pages, 2, Hk, ps, d]."""
    if p_layout not in _LAYOUTS or d_layout not in _LAYOUTS:
        raise PodError(1, f"unknown kv layout {p_layout!r} / {d_layout!r}")
    _check(load_library().pod_plan_set_kv_layout(ctypes.c_void_p(h.ptr), _LAYOUTS[p_layout],
                                                 _LAYOUTS[d_layout]))


def _check_mask_device(h: PodHandle):
    m = h.p_mask
    if m is not None and h.p_rows and not getattr(m, "is_cuda", False):
        raise PodError(1, "the custom prefill mask must be a CUDA uint8 tensor to run")
    if h.alibi is not None and not getattr(h.alibi, "is_cuda", False):
        raise PodError(1, "the ALiBi slopes must be a CUDA float32 tensor to run")


def plan_inputs(inp, workspace=None, num_sms=0, stream=None) -> PodHandle:
    """pod_plan for a ``pod_workloads.PODInputs``-shaped object (tests, bench);
    an FP8 (float8_e4m3fn) decode cache gets pod_plan_set_decode_fp8 with the
    inputs' scales, a packed custom mask on the prefill half
    pod_plan_set_prefill_mask (moved to the GPU when there is one)."""
    mask = getattr(inp.p, "packed_mask", None)
    rope = getattr(inp, "rope", None)
    replans = mask is not None or rope is not None
    h = _plan_inputs(inp, None if replans else workspace, num_sms, stream)
    if rope is not None:
        pod_plan_set_rope(h, *rope)
    import torch
    if inp.d.rows and getattr(inp.d.kv, "dtype", None) == torch.float8_e4m3fn:
        pod_plan_set_decode_fp8(h, inp.k_scale, inp.v_scale)
    cap, slopes = float(getattr(inp, "soft_cap", 0.0) or 0.0), getattr(inp, "alibi", None)
    if cap > 0 or slopes is not None:
        if slopes is not None and torch.cuda.is_available():
            slopes = slopes.to(device="cuda", dtype=torch.float32).contiguous()
        pod_plan_set_logits_transform(h, cap, slopes)
    lp, ld = getattr(inp.p, "kv_layout", "NHD"), getattr(inp.d, "kv_layout", "NHD")
    if (lp, ld) != ("NHD", "NHD"):
        pod_plan_set_kv_layout(h, lp, ld)
    if mask is not None:
        t = torch.from_numpy(np.ascontiguousarray(mask, dtype=np.uint8))
        if torch.cuda.is_available():
            t = t.cuda()
        pod_plan_set_prefill_mask(h, t)
    if replans and workspace is not None:
        pod_bind_workspace(h, workspace, stream)
    return h


def _plan_inputs(inp, workspace, num_sms, stream) -> PodHandle:
    return pod_plan(inp.p.q_indptr, inp.p.kv_indptr, inp.p.kv_indices, inp.p.last_page_len,
                    inp.d.q_indptr, inp.d.kv_indptr, inp.d.kv_indices, inp.d.last_page_len,
                    inp.num_qo_heads, inp.num_kv_heads, inp.head_dim, inp.page_size,
                    inp.causal, inp.window_left, inp.sm_scale, dtype=inp.dtype,
                    p_num_pages=inp.p.num_pages, d_num_pages=inp.d.num_pages,
                    has_sinks=inp.sinks is not None, num_sms=num_sms, workspace=workspace,
                    stream=stream)


def pod_plan_set_graph_capacity(h: PodHandle, max_p_batch: int, max_p_rows: int, max_p_pages: int,
                                max_d_batch: int, max_d_rows: int, max_d_pages: int):
    """Capacity mode for CUDA-graph replay: the workspace layout and launch
    shapes depend on these maxima only; rebind the workspace afterwards. The
    q/out tensors given to pod_run then hold max_*_rows rows."""
    _check(load_library().pod_plan_set_graph_capacity(
        ctypes.c_void_p(h.ptr), int(max_p_batch), int(max_p_rows), int(max_p_pages),
        int(max_d_batch), int(max_d_rows), int(max_d_pages)))
    h.workspace_bytes = pod_workspace_size(h)
    h.p_rows, h.d_rows = int(max_p_rows), int(max_d_rows)


def pod_replan(h: PodHandle, p_q_indptr, p_kv_indptr, p_kv_indices, p_last_page_len,
               d_q_indptr, d_kv_indptr, d_kv_indices, d_last_page_len, stream=None):
    """Plan new page tables into a capacity handle's bound workspace (outside
    any capture); a pod_run captured earlier then replays the new plan."""
    arrs = [_i32(x) for x in (p_q_indptr, p_kv_indptr, p_kv_indices, p_last_page_len,
                              d_q_indptr, d_kv_indptr, d_kv_indices, d_last_page_len)]
    p_batch = 0 if arrs[0] is None else len(arrs[0]) - 1
    d_batch = 0 if arrs[4] is None else len(arrs[4]) - 1
    _check(load_library().pod_replan(ctypes.c_void_p(h.ptr), *[_ptr(a) for a in arrs[:4]], p_batch,
                                     *[_ptr(a) for a in arrs[4:]], d_batch, _stream(stream)))
