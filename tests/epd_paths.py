"""Run one workload through the CUDA path (via the C ABI binding) and through the
CPU oracle, and compare: bit-exact for counts, offsets, indices and permuted
bytes; within |gpu - ref| <= 1e-3 + 1e-2 |ref| per element for the combine."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import unpermute_ep_dispatch_gb300 as epd

ATOL = 1e-3
RTOL = 1e-2


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def row_bytes(t: torch.Tensor) -> np.ndarray:
    """[T, H] tensor of any dtype -> [T, row_bytes] uint8 view of its bytes."""
    t = t.detach().cpu().contiguous()
    return t.view(torch.uint8).numpy().reshape(t.shape[0], t.shape[1] * t.element_size())


def default_capacity(case, alignment=1):
    if alignment == 1:
        return case.capacity
    return oracle.aligned_capacity(case.T, case.k, case.E, alignment)


def oracle_path(case, capacity=None, topk_override=None, alignment=1):
    topk = (case.topk_idx if topk_override is None else topk_override).numpy()
    eo = None if case.expert_out is None else bits16(case.expert_out)
    cap = default_capacity(case, alignment) if capacity is None else capacity
    if eo is not None and eo.shape[0] < cap:
        eo = np.concatenate([eo, np.zeros((cap - eo.shape[0], eo.shape[1]), np.uint16)])
    xs = None if case.x_scale is None else case.x_scale.numpy()
    return oracle.run_path(row_bytes(case.x), xs, topk, case.topk_weights.numpy(), case.E,
                           case.R, case.N, capacity=cap, expert_out=eo, alignment=alignment)


class GpuPath:
    """Device-resident buffers for one case and the four C ABI calls on them."""

    def __init__(self, case, device="cuda", capacity=None, stream=None, alignment=1,
                 fused=False):
        self.case = case
        self.dev = torch.device(device)
        self.alignment = alignment
        self.fused = fused  # step() runs ep_dispatch_layout_offsets instead of layout + scan
        self.cap = default_capacity(case, alignment) if capacity is None else int(capacity)
        self.stream = stream
        d = self.dev
        self.topk = case.topk_idx.to(d)
        self.w = case.topk_weights.to(d)
        self.x = case.x.to(d)
        self.xs = None if case.x_scale is None else case.x_scale.to(d)
        if case.expert_out is None:
            self.eo = None
        else:
            eo = torch.zeros(self.cap, case.H, dtype=torch.bfloat16)
            eo[: case.expert_out.shape[0]] = case.expert_out[: self.cap]
            self.eo = eo.to(d)
        T, k, E, R, N = case.T, case.k, case.E, case.R, case.N
        self.ws = epd.new_workspace(T, k, E, R, N, d)
        self.status = epd.new_status(d)
        self.per_e = torch.empty(E, dtype=torch.int32, device=d)
        self.per_r = torch.empty(R, dtype=torch.int32, device=d)
        self.per_n = torch.empty(N, dtype=torch.int32, device=d)
        self.itr = torch.empty(T, R, dtype=torch.bool, device=d)
        self.start = torch.empty(E, dtype=torch.int32, device=d)
        self.total = torch.empty(1, dtype=torch.int32, device=d)
        self.out = torch.empty(self.cap, case.H, dtype=case.x.dtype, device=d)
        self.out_scale = None if self.xs is None else torch.empty(
            self.cap, case.H // 128, dtype=torch.float32, device=d)
        self.m_indices = torch.empty(self.cap, dtype=torch.int32, device=d)
        self.output_index = torch.empty(T, k, dtype=torch.int32, device=d)
        self.y = torch.empty(T, case.H, dtype=torch.bfloat16, device=d)

    def layout(self):
        c = self.case
        epd.ep_dispatch_layout(self.topk, c.E, c.R, c.N, self.ws, self.status,
                               tokens_per_expert=self.per_e, tokens_per_rank=self.per_r,
                               tokens_per_rdma_rank=self.per_n, is_token_in_rank=self.itr,
                               stream=self.stream)

    def scan(self):
        if self.alignment == 1:
            epd.ep_scan_offsets(self.per_e, self.status, expert_start_loc=self.start,
                                total_rows=self.total, stream=self.stream)
        else:
            epd.ep_scan_offsets_aligned(self.per_e, self.alignment, self.status,
                                        expert_start_loc=self.start, total_rows=self.total,
                                        stream=self.stream)

    def permute(self):
        c = self.case
        epd.ep_permute(self.x, self.xs, self.topk, c.E, self.start, self.ws, self.status,
                       capacity_rows=self.cap, out=self.out, out_scale=self.out_scale,
                       m_indices=self.m_indices, output_index=self.output_index,
                       stream=self.stream)

    def unpermute(self):
        eo = self.out if self.eo is None else self.eo
        epd.ep_unpermute(eo, self.output_index, self.w, self.status, y=self.y,
                         stream=self.stream)

    def layout_offsets(self):
        c = self.case
        epd.ep_dispatch_layout_offsets(self.topk, c.E, c.R, c.N, self.ws, self.status,
                                       alignment=self.alignment, tokens_per_expert=self.per_e,
                                       tokens_per_rank=self.per_r, tokens_per_rdma_rank=self.per_n,
                                       is_token_in_rank=self.itr, expert_start_loc=self.start,
                                       total_rows=self.total, stream=self.stream)

    def step(self):
        if self.fused:
            self.layout_offsets()
        else:
            self.layout()
            self.scan()
        self.permute()
        self.unpermute()

    def results(self):
        torch.cuda.synchronize(self.dev)
        r = dict(
            tokens_per_expert=self.per_e.cpu().numpy(), tokens_per_rank=self.per_r.cpu().numpy(),
            tokens_per_rdma_rank=self.per_n.cpu().numpy(),
            is_token_in_rank=self.itr.cpu().numpy(), expert_start_loc=self.start.cpu().numpy(),
            total_rows=int(self.total.item()), out=row_bytes(self.out),
            m_indices=self.m_indices.cpu().numpy(), output_index=self.output_index.cpu().numpy(),
            y=bits16(self.y), status=int(self.status.item()))
        r["out_scale"] = None if self.out_scale is None else self.out_scale.cpu().numpy()
        return r


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def combine_error(got_bits, want_bits):
    """Largest |gpu - ref| / (ATOL + RTOL |ref|) over all elements (<= 1 passes)."""
    g = bf16_to_f64(got_bits)
    w = bf16_to_f64(want_bits)
    if g.size == 0:
        return 0.0
    return float(np.max(np.abs(g - w) / (ATOL + RTOL * np.abs(w))))


def compare(got, want, check_status=True):
    if check_status:
        assert got["status"] == 0, f"device status {got['status']}"
    for key in ("tokens_per_expert", "tokens_per_rank", "tokens_per_rdma_rank",
                "expert_start_loc", "m_indices", "output_index"):
        assert np.array_equal(got[key], want[key]), key
    assert np.array_equal(got["is_token_in_rank"], want["is_token_in_rank"]), "is_token_in_rank"
    assert got["total_rows"] == want["total_rows"], "total_rows"
    filled = want["output_index"][want["output_index"] >= 0]   # rows some pair fills
    assert np.array_equal(got["out"][filled], want["out"][filled]), "permuted rows"
    if want["out_scale"] is not None:
        assert np.array_equal(got["out_scale"][filled], want["out_scale"][filled]), \
            "permuted scales"
    err = combine_error(got["y"], want["y"])
    assert err <= 1.0, f"combine off by {err:.3f}x the tolerance"
    return err
