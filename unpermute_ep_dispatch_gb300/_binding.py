"""ctypes binding of libepd (``include/epd.h``): argument marshalling only.

Each function checks tensor dtypes, shapes, devices and contiguity, passes raw
pointers and the current CUDA stream to the C call of the same name and raises
``EpdError`` when the call returns a non-zero status. Every step of the path
runs in libepd's kernels; there is no fallback. Output tensors may be passed in
(for CUDA-graph capture and allocation-free steps) or are allocated here with
torch.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libepd.so")

EPD_OK = 0
EPD_ERR_INVALID_ARG = 1
EPD_ERR_UNSUPPORTED = 2
EPD_ERR_CUDA = 3
EPD_ERR_INVALID_EXPERT = 4
EPD_ERR_TIMEOUT = 5
EPD_ERR_CAPACITY = 6
EPD_BF16 = 0
EPD_FP8_E4M3 = 1
EPD_MAX_EXPERTS = 4096
EPD_MAX_TOPK = 64

class PermuteView(ctypes.Structure):
    """epd_permute_view_t."""
    _fields_ = [("expert_begin", ctypes.c_int), ("expert_end", ctypes.c_int),
                ("scale_cols", ctypes.c_int), ("scale_col_major", ctypes.c_int),
                ("scale_ld", ctypes.c_int64)]


# name -> (restype, argtypes); mirrors include/epd.h
_P, _I, _I64, _U32, _SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                           ctypes.c_size_t)
SIGNATURES = {
    "epd_status_string": (ctypes.c_char_p, [_I]),
    "epd_version": (_I, []),
    "epd_last_cuda_error": (_I, []),
    "epd_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "epd_workspace_init": (_I, [_P, _SZ, _P]),
    "ep_dispatch_layout": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "ep_dispatch_layout_offsets": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P,
                                        _P, _P]),
    "ep_scan_offsets": (_I, [_P, _I, _P, _P, _P, _P]),
    "ep_scan_offsets_aligned": (_I, [_P, _I, _I, _P, _P, _P, _P]),
    "ep_permute": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _I64, _P, _P, _P, _P, _P, _P]),
    "ep_dispatch": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                         _I64, _P, _P, _P, _P, _P, _P]),
    "ep_permute_ex": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P, _I64, ctypes.POINTER(PermuteView),
                           _P, _P, _P, _P, _P, _P]),
    "ep_unpermute": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _P, _P]),
    "ep_permute_lowlatency": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I64, _P, _P, _P, _P, _P, _P,
                                   _P, _P]),
    "ep_dispatch_lowlatency": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I64, _P, _P, _P, _P,
                                    _P, _P, _P, _P]),
    "ep_dispatch_layout_noalloc": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "epd_test_layout_stalled_tile": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                                          _U32, _P]),
}

_lock = threading.Lock()
_lib = None


class EpdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {status_string(code)} (status {code})"
        if code == EPD_ERR_CUDA:
            msg += f", cudaError {load_library().epd_last_cuda_error()}"
        super().__init__(msg)


def load_library(path: str = LIB_PATH):
    """Load libepd.so (built in-tree by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libepd.so is not built ({path}); run `python -m unpermute_ep_dispatch_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().epd_status_string(int(code)).decode()


def version() -> int:
    return int(load_library().epd_version())


def _check(rc: int, where: str):
    if rc != EPD_OK:
        raise EpdError(rc, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _want(t, name, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _out(t, name, dtype, shape, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _want(t, name, dtype, shape, device)


# ----------------------------------------------------------------------------- workspace
def epd_workspace_bytes(num_tokens: int, num_topk: int, num_experts: int, num_ranks: int,
                        num_rdma_ranks: int) -> int:
    n = int(load_library().epd_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks,
                                               num_rdma_ranks))
    if n == 0:
        raise EpdError(EPD_ERR_INVALID_ARG, "epd_workspace_bytes")
    return n


def new_workspace(num_tokens, num_topk, num_experts, num_ranks, num_rdma_ranks, device=None):
    """A zero-filled workspace tensor (uint8) for one stream's layout -> permute chain."""
    n = epd_workspace_bytes(num_tokens, num_topk, num_experts, num_ranks, num_rdma_ranks)
    return torch.zeros(n, dtype=torch.uint8, device=device or torch.device("cuda"))


def epd_workspace_init(workspace: torch.Tensor, stream=None):
    _want(workspace, "workspace", torch.uint8)
    _check(load_library().epd_workspace_init(_ptr(workspace), workspace.numel(),
                                             _stream(stream, workspace.device)),
           "epd_workspace_init")


def new_status(device=None) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=device or torch.device("cuda"))


def check_status(status: torch.Tensor, where: str = "libepd"):
    """Read the device status word (synchronises) and raise if a kernel flagged an error."""
    code = int(status.item())
    if code != EPD_OK:
        raise EpdError(code, where)


# ----------------------------------------------------------------------------- the four steps
def ep_dispatch_layout(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                       num_rdma_ranks: int, workspace: torch.Tensor, status: torch.Tensor,
                       tokens_per_expert=None, tokens_per_rank=None, tokens_per_rdma_rank=None,
                       is_token_in_rank=None, with_rdma: Optional[bool] = None,
                       with_is_token_in_rank: bool = True, stream=None):
    """Step 1. Returns (tokens_per_rank [R] i32, tokens_per_rdma_rank [N] i32 or None,
    tokens_per_expert [E] i32, is_token_in_rank [T, R] bool or None), the order of
    DeepEP's get_dispatch_layout. tokens_per_rdma_rank is None for one node unless
    with_rdma=True."""
    _want(topk_idx, "topk_idx", torch.int64)
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [num_tokens, num_topk]")
    dev = topk_idx.device
    T, k = topk_idx.shape
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    if workspace.numel() < epd_workspace_bytes(T, k, E, R, N):
        raise ValueError("workspace too small for this layout")
    if with_rdma is None:
        with_rdma = N > 1 or tokens_per_rdma_rank is not None
    per_e = _out(tokens_per_expert, "tokens_per_expert", torch.int32, (E,), dev)
    per_r = _out(tokens_per_rank, "tokens_per_rank", torch.int32, (R,), dev)
    per_n = _out(tokens_per_rdma_rank, "tokens_per_rdma_rank", torch.int32, (N,), dev) \
        if with_rdma else None
    itr = _out(is_token_in_rank, "is_token_in_rank", torch.bool, (T, R), dev) \
        if with_is_token_in_rank else None
    rc = load_library().ep_dispatch_layout(_ptr(topk_idx), T, k, E, R, N, _ptr(per_e),
                                           _ptr(per_r), _ptr(per_n), _ptr(itr), _ptr(workspace),
                                           _ptr(status), _stream(stream, dev))
    _check(rc, "ep_dispatch_layout")
    return per_r, per_n, per_e, itr


def ep_dispatch_layout_offsets(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                               num_rdma_ranks: int, workspace: torch.Tensor, status: torch.Tensor,
                               alignment: int = 1, tokens_per_expert=None, tokens_per_rank=None,
                               tokens_per_rdma_rank=None, is_token_in_rank=None,
                               expert_start_loc=None, total_rows=None,
                               with_rdma: Optional[bool] = None,
                               with_is_token_in_rank: bool = True, stream=None):
    """Steps 1 and 2 in one launch. Returns (tokens_per_rank, tokens_per_rdma_rank or
    None, tokens_per_expert, is_token_in_rank or None, expert_start_loc, total_rows)."""
    _want(topk_idx, "topk_idx", torch.int64)
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [num_tokens, num_topk]")
    dev = topk_idx.device
    T, k = topk_idx.shape
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    if workspace.numel() < epd_workspace_bytes(T, k, E, R, N):
        raise ValueError("workspace too small for this layout")
    if with_rdma is None:
        with_rdma = N > 1 or tokens_per_rdma_rank is not None
    per_e = _out(tokens_per_expert, "tokens_per_expert", torch.int32, (E,), dev)
    per_r = _out(tokens_per_rank, "tokens_per_rank", torch.int32, (R,), dev)
    per_n = _out(tokens_per_rdma_rank, "tokens_per_rdma_rank", torch.int32, (N,), dev) \
        if with_rdma else None
    itr = _out(is_token_in_rank, "is_token_in_rank", torch.bool, (T, R), dev) \
        if with_is_token_in_rank else None
    start = _out(expert_start_loc, "expert_start_loc", torch.int32, (E,), dev)
    total = _out(total_rows, "total_rows", torch.int32, (1,), dev)
    rc = load_library().ep_dispatch_layout_offsets(
        _ptr(topk_idx), T, k, E, R, N, _ptr(per_e), _ptr(per_r), _ptr(per_n), _ptr(itr),
        int(alignment), _ptr(start), _ptr(total), _ptr(workspace), _ptr(status),
        _stream(stream, dev))
    _check(rc, "ep_dispatch_layout_offsets")
    return per_r, per_n, per_e, itr, start, total


def ep_scan_offsets(tokens_per_expert: torch.Tensor, status: torch.Tensor,
                    expert_start_loc=None, total_rows=None, stream=None):
    """Step 2. Returns (expert_start_loc [E] i32, total_rows [1] i32), both on the device."""
    _want(tokens_per_expert, "tokens_per_expert", torch.int32)
    dev = tokens_per_expert.device
    E = tokens_per_expert.numel()
    _want(status, "status", torch.int32, (1,), dev)
    start = _out(expert_start_loc, "expert_start_loc", torch.int32, (E,), dev)
    total = _out(total_rows, "total_rows", torch.int32, (1,), dev)
    rc = load_library().ep_scan_offsets(_ptr(tokens_per_expert), E, _ptr(start), _ptr(total),
                                        _ptr(status), _stream(stream, dev))
    _check(rc, "ep_scan_offsets")
    return start, total


def ep_scan_offsets_aligned(tokens_per_expert: torch.Tensor, alignment: int,
                            status: torch.Tensor, expert_start_loc=None, total_rows=None,
                            stream=None):
    """Step 2 with every expert's region padded to a multiple of `alignment`.
    Returns (expert_start_loc [E] i32, total_rows [1] i32), both on the device."""
    _want(tokens_per_expert, "tokens_per_expert", torch.int32)
    dev = tokens_per_expert.device
    E = tokens_per_expert.numel()
    _want(status, "status", torch.int32, (1,), dev)
    start = _out(expert_start_loc, "expert_start_loc", torch.int32, (E,), dev)
    total = _out(total_rows, "total_rows", torch.int32, (1,), dev)
    rc = load_library().ep_scan_offsets_aligned(_ptr(tokens_per_expert), E, int(alignment),
                                                _ptr(start), _ptr(total), _ptr(status),
                                                _stream(stream, dev))
    _check(rc, "ep_scan_offsets_aligned")
    return start, total


def aligned_capacity(num_tokens: int, num_topk: int, num_experts: int, alignment: int) -> int:
    """Rows that always hold the padded regions: round_up(T*k + E*(alignment-1), alignment)."""
    a = int(alignment)
    return (num_tokens * num_topk + num_experts * (a - 1) + a - 1) // a * a


def ep_permute(x: torch.Tensor, x_scale: Optional[torch.Tensor], topk_idx: torch.Tensor,
               num_experts: int, expert_start_loc: torch.Tensor, workspace: torch.Tensor,
               status: torch.Tensor, capacity_rows: Optional[int] = None, out=None,
               out_scale=None, m_indices=None, output_index=None, stream=None):
    """Step 3 (ep_scatter). x: [T, H] bfloat16, or float8_e4m3fn with x_scale
    [T, H/128] float32. Returns (out [M, H], out_scale [M, H/128] or None,
    m_indices [M] i32, output_index [T, k] i32), M = capacity_rows (default T*k)."""
    if x.dtype == torch.bfloat16:
        dt = EPD_BF16
        if x_scale is not None:
            raise ValueError("bf16 rows take no scales")
    elif x.dtype == torch.float8_e4m3fn:
        dt = EPD_FP8_E4M3
        if x_scale is None:
            raise ValueError("fp8 rows need x_scale [T, H/128] float32")
    else:
        raise ValueError(f"x must be bfloat16 or float8_e4m3fn, got {x.dtype}")
    _want(x, "x", x.dtype)
    dev = x.device
    T, H = x.shape
    _want(topk_idx, "topk_idx", torch.int64, device=dev)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, k] with the T of x")
    k = topk_idx.shape[1]
    M = T * k if capacity_rows is None else int(capacity_rows)
    _want(expert_start_loc, "expert_start_loc", torch.int32, (num_experts,), dev)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    out = _out(out, "out", x.dtype, (M, H), dev)
    if dt == EPD_FP8_E4M3:
        _want(x_scale, "x_scale", torch.float32, (T, H // 128), dev)
        out_scale = _out(out_scale, "out_scale", torch.float32, (M, H // 128), dev)
    else:
        out_scale = None
    m_indices = _out(m_indices, "m_indices", torch.int32, (M,), dev)
    output_index = _out(output_index, "output_index", torch.int32, (T, k), dev)
    rc = load_library().ep_permute(_ptr(x), dt, _ptr(x_scale), _ptr(topk_idx), T, k, H,
                                   int(num_experts), _ptr(expert_start_loc), _ptr(workspace), M,
                                   _ptr(out), _ptr(out_scale), _ptr(m_indices),
                                   _ptr(output_index), _ptr(status), _stream(stream, dev))
    _check(rc, "ep_permute")
    return out, out_scale, m_indices, output_index


def ep_dispatch(x: torch.Tensor, x_scale: Optional[torch.Tensor], topk_idx: torch.Tensor,
                num_experts: int, num_ranks: int, num_rdma_ranks: int, workspace: torch.Tensor,
                status: torch.Tensor, alignment: int = 1, capacity_rows: Optional[int] = None,
                tokens_per_expert=None, tokens_per_rank=None, tokens_per_rdma_rank=None,
                is_token_in_rank=None, expert_start_loc=None, total_rows=None, out=None,
                out_scale=None, m_indices=None, output_index=None,
                with_rdma: Optional[bool] = None, with_is_token_in_rank: bool = True,
                stream=None):
    """Steps 1 to 3 in one call (layout, offsets, permute; see epd.h). x: [T, H]
    bfloat16, or float8_e4m3fn with x_scale [T, H/128] float32. Returns a dict with
    tokens_per_rank, tokens_per_rdma_rank (or None), tokens_per_expert,
    is_token_in_rank (or None), expert_start_loc, total_rows, out, out_scale (or
    None), m_indices and output_index."""
    if x.dtype == torch.bfloat16:
        dt = EPD_BF16
        if x_scale is not None:
            raise ValueError("bf16 rows take no scales")
    elif x.dtype == torch.float8_e4m3fn:
        dt = EPD_FP8_E4M3
        if x_scale is None:
            raise ValueError("fp8 rows need x_scale [T, H/128] float32")
    else:
        raise ValueError(f"x must be bfloat16 or float8_e4m3fn, got {x.dtype}")
    _want(x, "x", x.dtype)
    dev = x.device
    T, H = x.shape
    _want(topk_idx, "topk_idx", torch.int64, device=dev)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, k] with the T of x")
    k = topk_idx.shape[1]
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    M = T * k if capacity_rows is None else int(capacity_rows)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    if workspace.numel() < epd_workspace_bytes(T, k, E, R, N):
        raise ValueError("workspace too small for this layout")
    if with_rdma is None:
        with_rdma = N > 1 or tokens_per_rdma_rank is not None
    per_e = _out(tokens_per_expert, "tokens_per_expert", torch.int32, (E,), dev)
    per_r = _out(tokens_per_rank, "tokens_per_rank", torch.int32, (R,), dev)
    per_n = _out(tokens_per_rdma_rank, "tokens_per_rdma_rank", torch.int32, (N,), dev) \
        if with_rdma else None
    itr = _out(is_token_in_rank, "is_token_in_rank", torch.bool, (T, R), dev) \
        if with_is_token_in_rank else None
    start = _out(expert_start_loc, "expert_start_loc", torch.int32, (E,), dev)
    total = _out(total_rows, "total_rows", torch.int32, (1,), dev)
    out = _out(out, "out", x.dtype, (M, H), dev)
    if dt == EPD_FP8_E4M3:
        _want(x_scale, "x_scale", torch.float32, (T, H // 128), dev)
        out_scale = _out(out_scale, "out_scale", torch.float32, (M, H // 128), dev)
    else:
        out_scale = None
    m_indices = _out(m_indices, "m_indices", torch.int32, (M,), dev)
    output_index = _out(output_index, "output_index", torch.int32, (T, k), dev)
    rc = load_library().ep_dispatch(
        _ptr(x), dt, _ptr(x_scale), _ptr(topk_idx), T, k, H, E, R, N, int(alignment),
        _ptr(per_e), _ptr(per_r), _ptr(per_n), _ptr(itr), _ptr(start), _ptr(total),
        _ptr(workspace), M, _ptr(out), _ptr(out_scale), _ptr(m_indices), _ptr(output_index),
        _ptr(status), _stream(stream, dev))
    _check(rc, "ep_dispatch")
    return dict(tokens_per_rank=per_r, tokens_per_rdma_rank=per_n, tokens_per_expert=per_e,
                is_token_in_rank=itr, expert_start_loc=start, total_rows=total, out=out,
                out_scale=out_scale, m_indices=m_indices, output_index=output_index)


def ep_permute_ex(x: torch.Tensor, x_scale: Optional[torch.Tensor], topk_idx: torch.Tensor,
                  num_experts: int, expert_start_loc: torch.Tensor, workspace: torch.Tensor,
                  status: torch.Tensor, capacity_rows: Optional[int] = None,
                  expert_begin: int = 0, expert_end: Optional[int] = None,
                  scale_col_major: bool = False, scale_ld: Optional[int] = None, out=None,
                  out_scale=None, m_indices=None, output_index=None, stream=None):
    """Step 3 with a per-rank view [expert_begin, expert_end) and a scale layout.
    x: [T, *] rows of any dtype (row bytes a multiple of 16); x_scale: [T, C]
    float32 (fp32 scales) or int32 (UE8M0-packed words), or None. Returns (out
    [M, *], out_scale ([M, C] row-major or [C, scale_ld] column-major) or None,
    m_indices [M] (local expert ids), output_index [T, k] (rows of the view))."""
    _want(x, "x", x.dtype)
    dev = x.device
    T = x.shape[0]
    row_bytes = int(torch.Size(x.shape[1:]).numel()) * x.element_size()
    _want(topk_idx, "topk_idx", torch.int64, device=dev)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, k] with the T of x")
    k = topk_idx.shape[1]
    E = int(num_experts)
    e_end = E if expert_end is None else int(expert_end)
    M = T * k if capacity_rows is None else int(capacity_rows)
    _want(expert_start_loc, "expert_start_loc", torch.int32, (E,), dev)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    out = _out(out, "out", x.dtype, (M, *x.shape[1:]), dev)
    C = 0
    if x_scale is not None:
        if x_scale.dtype not in (torch.float32, torch.int32) or x_scale.dim() != 2:
            raise ValueError("x_scale must be [T, C] float32 or int32")
        _want(x_scale, "x_scale", x_scale.dtype, (T, x_scale.shape[1]), dev)
        C = x_scale.shape[1]
        ld = M if scale_ld is None else int(scale_ld)
        shape = (C, ld) if scale_col_major else (M, C)
        out_scale = _out(out_scale, "out_scale", x_scale.dtype, shape, dev)
    else:
        ld = 0
        out_scale = None
    m_indices = _out(m_indices, "m_indices", torch.int32, (M,), dev)
    output_index = _out(output_index, "output_index", torch.int32, (T, k), dev)
    view = PermuteView(int(expert_begin), e_end, C, int(bool(scale_col_major)), ld)
    rc = load_library().ep_permute_ex(_ptr(x), row_bytes, _ptr(x_scale), _ptr(topk_idx), T, k, E,
                                      _ptr(expert_start_loc), _ptr(workspace), M,
                                      ctypes.byref(view), _ptr(out), _ptr(out_scale),
                                      _ptr(m_indices), _ptr(output_index), _ptr(status),
                                      _stream(stream, dev))
    _check(rc, "ep_permute_ex")
    return out, out_scale, m_indices, output_index


def ep_permute_lowlatency(x: torch.Tensor, topk_idx: torch.Tensor, num_experts: int,
                          rows_per_expert: int, workspace: torch.Tensor, status: torch.Tensor,
                          expert_begin: int = 0, expert_end: Optional[int] = None, out_q=None,
                          out_scale=None, recv_count=None, output_index=None, src_token=None,
                          with_src_token: bool = True, stream=None):
    """Fixed-rectangle layout with the fused bf16 -> e4m3 cast (see epd.h).
    x: [T, H] bfloat16. Returns (out_q [E_view, rows, H] float8_e4m3fn, out_scale
    [E_view, H/128, rows] f32, recv_count [E_view] i32, output_index [T, k] i32,
    src_token [E_view, rows] i32 or None)."""
    _want(x, "x", torch.bfloat16)
    dev = x.device
    T, H = x.shape
    _want(topk_idx, "topk_idx", torch.int64, device=dev)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, k] with the T of x")
    k = topk_idx.shape[1]
    E = int(num_experts)
    e_end = E if expert_end is None else int(expert_end)
    EV = e_end - int(expert_begin)
    rows = int(rows_per_expert)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    out_q = _out(out_q, "out_q", torch.float8_e4m3fn, (EV, rows, H), dev)
    out_scale = _out(out_scale, "out_scale", torch.float32, (EV, H // 128, rows), dev)
    recv_count = _out(recv_count, "recv_count", torch.int32, (EV,), dev)
    output_index = _out(output_index, "output_index", torch.int32, (T, k), dev)
    if with_src_token:
        src_token = _out(src_token, "src_token", torch.int32, (EV, rows), dev)
    rc = load_library().ep_permute_lowlatency(
        _ptr(x), _ptr(topk_idx), T, k, H, E, int(expert_begin), e_end, rows, _ptr(workspace),
        _ptr(out_q), _ptr(out_scale), _ptr(recv_count), _ptr(output_index), _ptr(src_token),
        _ptr(status), _stream(stream, dev))
    _check(rc, "ep_permute_lowlatency")
    return out_q, out_scale, recv_count, output_index, src_token



def ep_dispatch_lowlatency(x: torch.Tensor, topk_idx: torch.Tensor, num_experts: int,
                           num_ranks: int, num_rdma_ranks: int, rows_per_expert: int,
                           workspace: torch.Tensor, status: torch.Tensor, expert_begin: int = 0,
                           expert_end: Optional[int] = None, out_q=None, out_scale=None,
                           recv_count=None, output_index=None, src_token=None,
                           with_src_token: bool = True, stream=None):
    """The low-latency dispatch in one call (layout pair ranks, then the fixed-
    rectangle permute with the fused cast; one kernel for a decode batch; see
    epd.h). Returns what ep_permute_lowlatency returns."""
    _want(x, "x", torch.bfloat16)
    dev = x.device
    T, H = x.shape
    _want(topk_idx, "topk_idx", torch.int64, device=dev)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError("topk_idx must be [T, k] with the T of x")
    k = topk_idx.shape[1]
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    e_end = E if expert_end is None else int(expert_end)
    EV = e_end - int(expert_begin)
    rows = int(rows_per_expert)
    _want(workspace, "workspace", torch.uint8, device=dev)
    _want(status, "status", torch.int32, (1,), dev)
    if workspace.numel() < epd_workspace_bytes(T, k, E, R, N):
        raise ValueError("workspace too small for this layout")
    out_q = _out(out_q, "out_q", torch.float8_e4m3fn, (EV, rows, H), dev)
    out_scale = _out(out_scale, "out_scale", torch.float32, (EV, H // 128, rows), dev)
    recv_count = _out(recv_count, "recv_count", torch.int32, (EV,), dev)
    output_index = _out(output_index, "output_index", torch.int32, (T, k), dev)
    if with_src_token:
        src_token = _out(src_token, "src_token", torch.int32, (EV, rows), dev)
    rc = load_library().ep_dispatch_lowlatency(
        _ptr(x), _ptr(topk_idx), T, k, H, E, R, N, int(expert_begin), e_end, rows,
        _ptr(workspace), _ptr(out_q), _ptr(out_scale), _ptr(recv_count), _ptr(output_index),
        _ptr(src_token), _ptr(status), _stream(stream, dev))
    _check(rc, "ep_dispatch_lowlatency")
    return out_q, out_scale, recv_count, output_index, src_token


def ep_unpermute(expert_out: torch.Tensor, output_index: torch.Tensor,
                 topk_weights: torch.Tensor, status: torch.Tensor, y=None, stream=None):
    """Step 4 (combine). expert_out [M, H] bf16, output_index / topk_weights [T, k].
    Returns y [T, H] bf16."""
    _want(expert_out, "expert_out", torch.bfloat16)
    dev = expert_out.device
    M, H = expert_out.shape
    _want(output_index, "output_index", torch.int32, device=dev)
    if output_index.dim() != 2:
        raise ValueError("output_index must be [T, k]")
    T, k = output_index.shape
    _want(topk_weights, "topk_weights", torch.float32, (T, k), dev)
    _want(status, "status", torch.int32, (1,), dev)
    y = _out(y, "y", torch.bfloat16, (T, H), dev)
    rc = load_library().ep_unpermute(_ptr(expert_out), M, _ptr(output_index), _ptr(topk_weights),
                                     T, k, H, _ptr(y), _ptr(status), _stream(stream, dev))
    _check(rc, "ep_unpermute")
    return y


def ep_dispatch_layout_noalloc(topk_idx: torch.Tensor, num_experts: int, num_ranks: int,
                               num_rdma_ranks: int, status: torch.Tensor, tokens_per_expert,
                               tokens_per_rank, tokens_per_rdma_rank=None, is_token_in_rank=None,
                               stream=None):
    """ep_dispatch_layout without a caller workspace (its scratch is a fixed
    device array inside libepd, see epd.h). The caller passes every output
    tensor; nothing is allocated. Returns the outputs in DeepEP's order."""
    _want(topk_idx, "topk_idx", torch.int64)
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [num_tokens, num_topk]")
    dev = topk_idx.device
    T, k = topk_idx.shape
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    _want(status, "status", torch.int32, (1,), dev)
    _want(tokens_per_expert, "tokens_per_expert", torch.int32, (E,), dev)
    _want(tokens_per_rank, "tokens_per_rank", torch.int32, (R,), dev)
    if tokens_per_rdma_rank is not None:
        _want(tokens_per_rdma_rank, "tokens_per_rdma_rank", torch.int32, (N,), dev)
    if is_token_in_rank is not None:
        _want(is_token_in_rank, "is_token_in_rank", torch.bool, (T, R), dev)
    rc = load_library().ep_dispatch_layout_noalloc(
        _ptr(topk_idx), T, k, E, R, N, _ptr(tokens_per_expert), _ptr(tokens_per_rank),
        _ptr(tokens_per_rdma_rank), _ptr(is_token_in_rank), _ptr(status), _stream(stream, dev))
    _check(rc, "ep_dispatch_layout_noalloc")
    return tokens_per_rank, tokens_per_rdma_rank, tokens_per_expert, is_token_in_rank


def epd_test_layout_stalled_tile(topk_idx, num_experts, num_ranks, num_rdma_ranks, workspace,
                                 status, stalled_tile: int, spin_limit: int, stream=None):
    """Failure-detection hook: the layout with one tile that never publishes (see epd.h)."""
    dev = topk_idx.device
    T, k = topk_idx.shape
    E, R, N = int(num_experts), int(num_ranks), int(num_rdma_ranks)
    per_e = torch.empty(E, dtype=torch.int32, device=dev)
    per_r = torch.empty(R, dtype=torch.int32, device=dev)
    per_n = torch.empty(N, dtype=torch.int32, device=dev)
    itr = torch.empty(T, R, dtype=torch.bool, device=dev)
    rc = load_library().epd_test_layout_stalled_tile(
        _ptr(topk_idx), T, k, E, R, N, _ptr(per_e), _ptr(per_r), _ptr(per_n), _ptr(itr),
        _ptr(workspace), _ptr(status), int(stalled_tile), int(spin_limit), _stream(stream, dev))
    _check(rc, "epd_test_layout_stalled_tile")
    return per_r, per_n, per_e, itr
