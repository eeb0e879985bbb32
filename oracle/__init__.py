"""CPU oracle for the single-GPU MoE expert-parallel permute / unpermute path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package. The product
(``unpermute_ep_dispatch_gb300``) never imports it, and the two share no code:
the arithmetic lives in ``epd_oracle.c`` (plain single-threaded C, built with
``-O2 -ffp-contract=off``), written from the pages' definitions:

* layout  -- "[MoE] Deepseek的All-to-all通信: DeepEP代码解读", section "Dispatch"
  (get_dispatch_layout docstring);
* offsets -- "高性能专家并行（EP）内核解剖学解读", section "5. 缓冲区布局与发送";
* permute -- "参考sglang代码，重构vllm021中EP高吞吐代码，消除空泡问题", sections
  2.2 and 3.3 (ep_scatter / deepgemm_moe_permute);
* combine -- DeepEP reading, section "Dispatch" (combine mirrors dispatch;
  fp32 topk_weights), formed in fp64 and rounded once to bf16.

This module only marshals numpy arrays into the C functions.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "epd_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

ORC_OK = 0
ORC_ERR_INVALID_ARG = 1
ORC_ERR_INVALID_EXPERT = 4
ORC_ERR_CAPACITY = 6


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (a second or so). Returns the library path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        lib.oracle_dispatch_layout.argtypes = [P, I, I, I, I, I, P, P, P, P]
        lib.oracle_dispatch_layout.restype = I
        lib.oracle_scan_offsets.argtypes = [P, I, P, P]
        lib.oracle_scan_offsets.restype = I
        lib.oracle_scan_offsets_aligned.argtypes = [P, I, I, P, P]
        lib.oracle_scan_offsets_aligned.restype = I
        lib.oracle_permute.argtypes = [P, I64, P, I, P, I, I, I, P, I64, P, P, P, P]
        lib.oracle_permute.restype = I
        lib.oracle_permute_ex.argtypes = [P, I64, P, I, I, I64, P, I, I, I, I, I, P, I64, P, P, P,
                                          P]
        lib.oracle_permute_ex.restype = I
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_permute_lowlatency.argtypes = [P, I, I, I, P, I, I, I, I64, P, P, P, P, P, P]
        lib.oracle_permute_lowlatency.restype = I
        lib.oracle_unpermute.argtypes = [P, I64, P, P, I, I, I, P]
        lib.oracle_unpermute.restype = I
        lib.oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_double_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_double_from_bf16.restype = ctypes.c_double
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != ORC_OK:
        raise OracleError(f"{what}: oracle status {rc}")


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def dispatch_layout(topk_idx, num_experts: int, num_ranks: int, num_rdma_ranks: int):
    """Returns dict(tokens_per_expert [E] i32, tokens_per_rank [R] i32,
    tokens_per_rdma_rank [N] i32, is_token_in_rank [T, R] bool)."""
    topk = _c(topk_idx, np.int64)
    T, k = topk.shape
    E, R, N = num_experts, num_ranks, num_rdma_ranks
    per_e = np.zeros(E, np.int32)
    per_r = np.zeros(R, np.int32)
    per_n = np.zeros(N, np.int32)
    in_rank = np.zeros((T, R), np.uint8)
    rc = _load().oracle_dispatch_layout(_ptr(topk), T, k, E, R, N, _ptr(per_e), _ptr(per_r),
                                        _ptr(per_n), _ptr(in_rank))
    _check(rc, "dispatch_layout")
    return dict(tokens_per_expert=per_e, tokens_per_rank=per_r, tokens_per_rdma_rank=per_n,
                is_token_in_rank=in_rank.astype(bool))


def scan_offsets(tokens_per_expert):
    """Returns (expert_start_loc [E] i32, total_rows int)."""
    cnt = _c(tokens_per_expert, np.int32)
    start = np.zeros(cnt.shape[0], np.int32)
    total = np.zeros(1, np.int32)
    _check(_load().oracle_scan_offsets(_ptr(cnt), cnt.shape[0], _ptr(start), _ptr(total)),
           "scan_offsets")
    return start, int(total[0])


def scan_offsets_aligned(tokens_per_expert, alignment: int):
    """Returns (expert_start_loc [E] i32 of the padded regions, total padded rows)."""
    cnt = _c(tokens_per_expert, np.int32)
    start = np.zeros(cnt.shape[0], np.int32)
    total = np.zeros(1, np.int32)
    _check(_load().oracle_scan_offsets_aligned(_ptr(cnt), cnt.shape[0], int(alignment),
                                               _ptr(start), _ptr(total)), "scan_offsets_aligned")
    return start, int(total[0])


def aligned_capacity(T: int, k: int, E: int, alignment: int) -> int:
    """Rows that always suffice for padded regions: round_up(T*k + E*(alignment-1),
    alignment) -- the upper bound of vLLM's compute_aligned_M."""
    a = int(alignment)
    return (T * k + E * (a - 1) + a - 1) // a * a


def permute(x_rows, x_scale, topk_idx, num_experts: int, expert_start_loc, capacity: int):
    """x_rows: [T, row_bytes] uint8 (the raw bytes of each token row, any dtype);
    x_scale: [T, C] float32 or None. Returns dict(out [capacity, row_bytes] u8,
    out_scale [capacity, C] f32 or None, m_indices [capacity] i32,
    output_index [T, k] i32). Rows of out beyond the filled ones stay zero."""
    xb = _c(x_rows, np.uint8)
    topk = _c(topk_idx, np.int64)
    T, k = topk.shape
    assert xb.shape[0] == T
    row_bytes = xb.shape[1]
    sc = None if x_scale is None else _c(x_scale, np.float32)
    scale_cols = 0 if sc is None else sc.shape[1]
    start = _c(expert_start_loc, np.int32)
    out = np.zeros((capacity, row_bytes), np.uint8)
    out_scale = None if sc is None else np.zeros((capacity, scale_cols), np.float32)
    m_indices = np.zeros(capacity, np.int32)
    output_index = np.zeros((T, k), np.int32)
    rc = _load().oracle_permute(_ptr(xb), row_bytes, _ptr(sc), scale_cols, _ptr(topk), T, k,
                                num_experts, _ptr(start), capacity, _ptr(out), _ptr(out_scale),
                                _ptr(m_indices), _ptr(output_index))
    _check(rc, "permute")
    return dict(out=out, out_scale=out_scale, m_indices=m_indices, output_index=output_index)


def permute_ex(x_rows, x_scale_words, topk_idx, num_experts: int, expert_start_loc,
               capacity: int, expert_begin: int = 0, expert_end=None, scale_col_major=False,
               scale_ld=None):
    """Permute with output options: only experts [expert_begin, expert_end) with local
    rows and local ids (expert - expert_begin); scale rows of 32-bit words (fp32 or
    UE8M0-packed) copied row-major or column-major with leading dimension scale_ld.
    Returns dict(out, out_scale (uint32 words: [capacity, C] row-major or
    [C, scale_ld] column-major) or None, m_indices, output_index)."""
    xb = _c(x_rows, np.uint8)
    topk = _c(topk_idx, np.int64)
    T, k = topk.shape
    E = num_experts
    e_end = E if expert_end is None else expert_end
    sc = None if x_scale_words is None else np.ascontiguousarray(x_scale_words).view(np.uint32)
    C = 0 if sc is None else sc.shape[1]
    ld = capacity if scale_ld is None else int(scale_ld)
    start = _c(expert_start_loc, np.int32)
    out = np.zeros((capacity, xb.shape[1]), np.uint8)
    if sc is None:
        out_scale = None
    elif scale_col_major:
        out_scale = np.zeros((C, ld), np.uint32)
    else:
        out_scale = np.zeros((capacity, C), np.uint32)
    m_indices = np.zeros(capacity, np.int32)
    output_index = np.zeros((T, k), np.int32)
    rc = _load().oracle_permute_ex(_ptr(xb), xb.shape[1], _ptr(sc), C, int(bool(scale_col_major)),
                                   ld, _ptr(topk), T, k, E, int(expert_begin), int(e_end),
                                   _ptr(start), capacity, _ptr(out), _ptr(out_scale),
                                   _ptr(m_indices), _ptr(output_index))
    _check(rc, "permute_ex")
    return dict(out=out, out_scale=out_scale, m_indices=m_indices, output_index=output_index)


def e4m3_from_float(v: float) -> int:
    return int(_load().oracle_e4m3_from_float(float(v)))


def permute_lowlatency(x_bf16, topk_idx, num_experts: int, rows_per_expert: int,
                       expert_begin: int = 0, expert_end=None):
    """Fixed-rectangle layout with the fused cast. x_bf16: [T, H] uint16 (bf16 bits).
    Returns dict(out_q [E_view, rows, H] uint8 (e4m3 bytes), out_scale [E_view, H/128,
    rows] f32, recv_count [E_view] i32, output_index [T, k] i32, src_token
    [E_view, rows] i32, overflow bool). Unwritten rows are zero (scales) / zero
    bytes / -1 (src_token)."""
    x = _c(x_bf16, np.uint16)
    topk = _c(topk_idx, np.int64)
    T, k = topk.shape
    H = x.shape[1]
    e_end = num_experts if expert_end is None else expert_end
    EV = e_end - expert_begin
    C = H // 128
    out_q = np.zeros((EV, rows_per_expert, H), np.uint8)
    out_scale = np.zeros((EV, C, rows_per_expert), np.float32)
    recv = np.zeros(EV, np.int32)
    oi = np.zeros((T, k), np.int32)
    src = -np.ones((EV, rows_per_expert), np.int32)
    ovf = ctypes.c_int(0)
    rc = _load().oracle_permute_lowlatency(_ptr(x), T, k, H, _ptr(topk), num_experts,
                                           int(expert_begin), int(e_end), int(rows_per_expert),
                                           _ptr(out_q), _ptr(out_scale), _ptr(recv), _ptr(oi),
                                           _ptr(src), ctypes.byref(ovf))
    _check(rc, "permute_lowlatency")
    return dict(out_q=out_q, out_scale=out_scale, recv_count=recv, output_index=oi,
                src_token=src, overflow=bool(ovf.value))


def unpermute(expert_out_bf16, output_index, topk_weights):
    """expert_out_bf16: [M, H] uint16 (bf16 bit patterns); output_index [T, k] i32;
    topk_weights [T, k] f32. Returns y [T, H] uint16 (bf16 bit patterns)."""
    eo = _c(expert_out_bf16, np.uint16)
    oi = _c(output_index, np.int32)
    w = _c(topk_weights, np.float32)
    T, k = oi.shape
    H = eo.shape[1]
    y = np.zeros((T, H), np.uint16)
    rc = _load().oracle_unpermute(_ptr(eo), eo.shape[0], _ptr(oi), _ptr(w), T, k, H, _ptr(y))
    _check(rc, "unpermute")
    return y


def bf16_from_double(v: float) -> int:
    return int(_load().oracle_bf16_from_double(float(v)))


def double_from_bf16(b: int) -> float:
    return float(_load().oracle_double_from_bf16(int(b)))


def run_path(x_rows, x_scale, topk_idx, topk_weights, num_experts, num_ranks, num_rdma_ranks,
             capacity=None, expert_out=None, alignment=1):
    """The whole path: layout -> offsets -> permute -> combine.
    expert_out: [capacity, H] uint16 bf16 bits, or None for identity experts
    (the permuted rows themselves, which must then be bf16)."""
    topk = _c(topk_idx, np.int64)
    T, k = topk.shape
    if capacity is None:
        capacity = T * k if alignment == 1 else aligned_capacity(T, k, num_experts, alignment)
    lay = dispatch_layout(topk, num_experts, num_ranks, num_rdma_ranks)
    if alignment == 1:
        start, total = scan_offsets(lay["tokens_per_expert"])
    else:
        start, total = scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    per = permute(x_rows, x_scale, topk, num_experts, start, capacity)
    if expert_out is None:
        eo = per["out"].view(np.uint16)
    else:
        eo = expert_out
    y = unpermute(eo, per["output_index"], topk_weights)
    res = dict(lay)
    res.update(per)
    res.update(expert_start_loc=start, total_rows=total, y=y)
    return res
