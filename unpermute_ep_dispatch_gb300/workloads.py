"""Seeded synthetic inputs for the MoE expert-parallel permute / unpermute path.

This module is the one piece shared by the CUDA path's tests / benchmark and
the CPU oracle: it only draws inputs (router picks, weights, token rows,
expert outputs). It holds none of the path's arithmetic -- no counting,
offsets, slot assignment, copying or combining.

Every workload is built on the CPU from ``torch.Generator`` seeds, so one
process always feeds the same bytes to the GPU and to the oracle.

Workload shapes follow the pages' own settings:

* ``tiny``   -- the worked setting of "高性能专家并行（EP）内核解剖学解读",
  section "任务设定与数据流": 16 experts as 8 ranks x 2 experts on 2 nodes,
  each token routed to its top-2 of 16 router logits.
* ``prefill_bf16``, ``dsv3_fp8``, ``skew_bf16``, ``decode_fp8`` -- prefill- and
  decode-sized batches ("吞吐量与延迟的权衡"), the DeepSeek-V3 shape with fp8
  rows and one fp32 scale per 128 columns ("[MoE] Deepseek的All-to-all通信:
  DeepEP代码解读", "Dispatch", dispatch docstring: x as (e4m3 [T, H],
  float [T, H/128])), and lumpy routing ("2. 核心难点：未知的大小": one expert
  may get 1000 tokens, another none).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

FP8_MAX = 448.0  # largest finite float8_e4m3fn value

CONFIGS = {
    # T=64, H=256 bf16; E=16 = 8 ranks x 2 experts on 2 nodes; top-2 of N(0,1) logits
    "tiny": dict(T=64, H=256, dtype="bf16", E=16, R=8, N=2, k=2, routing="uniform",
                 p_invalid=0.0, experts="random", seed=0),
    # T=4096, H=4096 bf16; 64 experts on 8 ranks of one node; top-6; ~2% picks dropped
    "prefill_bf16": dict(T=4096, H=4096, dtype="bf16", E=64, R=8, N=1, k=6, routing="uniform",
                         p_invalid=0.02, experts="identity", seed=1),
    # DeepSeek-V3 shape: T=8192, H=7168 e4m3 + [T,56] scales; 256 experts, 32 ranks, 4 nodes
    "dsv3_fp8": dict(T=8192, H=7168, dtype="fp8", E=256, R=32, N=4, k=8, routing="uniform",
                     p_invalid=0.0, experts="random", seed=2),
    # Zipf(1.2) expert popularity, 20 experts never picked; T=16384, H=7168 bf16
    "skew_bf16": dict(T=16384, H=7168, dtype="bf16", E=256, R=32, N=4, k=8, routing="zipf",
                      zipf_s=1.2, zero_experts=20, p_invalid=0.0, experts="identity", seed=3),
    # decode: many independent steps of T=128 (seeds 1000 + step)
    "decode_fp8": dict(T=128, H=7168, dtype="fp8", E=256, R=32, N=4, k=8, routing="uniform",
                       p_invalid=0.0, experts="random", seed=1000, steps=512),
}


@dataclass
class Case:
    name: str
    T: int
    H: int
    k: int
    E: int
    R: int
    N: int
    dtype: str                       # "bf16" or "fp8"
    topk_idx: torch.Tensor           # [T, k] int64, -1 = no selection
    topk_weights: torch.Tensor       # [T, k] float32 (0 where topk_idx == -1)
    x: torch.Tensor                  # [T, H] bfloat16 or float8_e4m3fn
    x_scale: Optional[torch.Tensor]  # [T, H/128] float32, or [T, ceil(H/512)] int32 UE8M0 (fp8)
    expert_out: Optional[torch.Tensor]  # [T*k, H] bfloat16, or None = identity experts
    meta: dict = field(default_factory=dict)

    @property
    def capacity(self) -> int:
        return self.T * self.k

    @property
    def row_bytes(self) -> int:
        return self.H * (1 if self.dtype == "fp8" else 2)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _masked_softmax(logits: torch.Tensor, valid: torch.Tensor) -> torch.Tensor:
    """Softmax over the valid entries of each row (float64 internally), 0 elsewhere."""
    l = logits.double().masked_fill(~valid, float("-inf"))
    m = l.max(dim=1, keepdim=True).values
    m = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    ex = torch.exp(l - m).masked_fill(~valid, 0.0)
    s = ex.sum(dim=1, keepdim=True)
    w = torch.where(s > 0, ex / torch.where(s > 0, s, torch.ones_like(s)), torch.zeros_like(ex))
    return w.float()


def route_uniform(g, T, E, k, p_invalid=0.0):
    """Top-k of seeded N(0,1) router logits [T, E]; ties go to the lower expert
    index (stable sort). Each pick is independently dropped to -1 with
    probability p_invalid; weights are the softmax over the remaining picks."""
    logits = torch.randn(T, E, generator=g)
    order = torch.argsort(-logits, dim=1, stable=True)[:, :k]
    picked = torch.gather(logits, 1, order)
    valid = torch.ones(T, k, dtype=torch.bool)
    if p_invalid > 0:
        valid = torch.rand(T, k, generator=g) >= p_invalid
    topk = torch.where(valid, order, torch.full_like(order, -1)).to(torch.int64)
    return topk, _masked_softmax(picked, valid)


def route_zipf(g, T, E, k, s=1.2, zero_experts=20):
    """Expert popularity Zipf(s) over ranks 1..E-zero_experts, assigned to a
    seeded permutation of the experts; the remaining zero_experts are never
    picked. k distinct experts per token by Gumbel-top-k on log p; weights are
    the softmax over the perturbed scores of the picks."""
    perm = torch.randperm(E, generator=g)
    n_live = E - zero_experts
    ranks = torch.arange(1, n_live + 1, dtype=torch.float64)
    p = torch.zeros(E, dtype=torch.float64)
    p[perm[:n_live]] = ranks.pow(-s) / ranks.pow(-s).sum()
    u = torch.rand(T, E, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0 - 1e-16)
    gumbel = -torch.log(-torch.log(u))
    scores = torch.log(p).unsqueeze(0) + gumbel          # -inf for the zero experts
    order = torch.argsort(-scores, dim=1, stable=True)[:, :k]
    picked = torch.gather(scores, 1, order)
    valid = torch.ones(T, k, dtype=torch.bool)
    return order.to(torch.int64), _masked_softmax(picked.float(), valid), p


def quantize_fp8_per128(x: torch.Tensor):
    """Per-(row, 128-column block) e4m3 quantisation of a float32 [T, H] matrix:
    scale = amax(block) / 448 (1 where the block is all zero), q = e4m3(x / scale)
    with round-to-nearest-even and saturation at +-448."""
    T, H = x.shape
    blocks = x.reshape(T, H // 128, 128)
    amax = blocks.abs().amax(dim=2)
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = (blocks / scale.unsqueeze(2)).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.reshape(T, H), scale.float().contiguous()


def quantize_fp8_per128_ue8m0(x: torch.Tensor):
    """Per-(row, 128-column block) e4m3 quantisation with power-of-two scales, the
    form whose scales pack as UE8M0 bytes (an 8-bit biased exponent, no mantissa):
    scale = 2^ceil(log2(amax / 448)) (1 where the block is all zero), q = e4m3(x /
    scale). Returns (q [T, H] e4m3, words [T, ceil(H/512)] int32), four exponent
    bytes per word, block 4g in the lowest byte, missing blocks padded with 127
    (scale 1)."""
    T, H = x.shape
    C = H // 128
    blocks = x.reshape(T, C, 128).double()
    amax = blocks.abs().amax(dim=2)
    expo = torch.where(amax > 0, torch.ceil(torch.log2(amax / FP8_MAX)), torch.zeros_like(amax))
    scale = torch.pow(2.0, expo)
    q = (blocks / scale.unsqueeze(2)).clamp_(-FP8_MAX, FP8_MAX).float().to(torch.float8_e4m3fn)
    G = (C + 3) // 4
    byte = torch.full((T, 4 * G), 127, dtype=torch.int64)
    byte[:, :C] = (expo + 127).to(torch.int64)
    b = byte.reshape(T, G, 4)
    words = (b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24))
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32)
    return q.reshape(T, H), words.contiguous()


def _randn_bf16(g, rows, cols, chunk_rows=8192):
    out = torch.empty(rows, cols, dtype=torch.bfloat16)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn(r1 - r0, cols, generator=g).to(torch.bfloat16)
    return out


def make_rows(g, T, H, dtype, scales="f32"):
    if dtype == "bf16":
        return _randn_bf16(g, T, H), None
    if dtype == "fp8":
        if H % 128:
            raise ValueError("fp8 rows need H % 128 == 0")
        if scales == "ue8m0":
            return quantize_fp8_per128_ue8m0(torch.randn(T, H, generator=g))
        return quantize_fp8_per128(torch.randn(T, H, generator=g))
    raise ValueError(dtype)


def make_case(name: str = "tiny", seed: Optional[int] = None, T: Optional[int] = None,
              experts: Optional[str] = None, scales: str = "f32",
              dtype: Optional[str] = None) -> Case:
    """Build one named workload (see CONFIGS). ``T`` overrides the token count
    (smaller instances of the same routing shape); ``experts`` overrides the
    expert-output mode ("identity" or "random")."""
    cfg = dict(CONFIGS[name])
    if seed is None:
        seed = cfg["seed"]
    if T is not None:
        cfg["T"] = int(T)
    if experts is not None:
        cfg["experts"] = experts
    if dtype is not None:
        cfg["dtype"] = dtype
    return make_random_case(T=cfg["T"], H=cfg["H"], k=cfg["k"], E=cfg["E"], R=cfg["R"],
                            N=cfg["N"], dtype=cfg["dtype"], seed=seed,
                            routing=cfg["routing"], p_invalid=cfg.get("p_invalid", 0.0),
                            experts=cfg["experts"], zipf_s=cfg.get("zipf_s", 1.2),
                            zero_experts=cfg.get("zero_experts", 20), name=name, scales=scales)


def make_random_case(T, H, k, E, R, N, dtype="bf16", seed=0, routing="uniform", p_invalid=0.0,
                     experts="random", zipf_s=1.2, zero_experts=20, name="random",
                     scales="f32") -> Case:
    """scales: "f32" (one fp32 scale per 128 columns) or "ue8m0" (power-of-two scales
    packed as exponent bytes, four per int32 word; x_scale is then int32)."""
    g = _gen(seed)
    meta = {}
    if T == 0 or k == 0:
        topk = torch.zeros(T, k, dtype=torch.int64)
        w = torch.zeros(T, k, dtype=torch.float32)
    elif routing == "uniform":
        if k > E:
            raise ValueError("uniform routing draws k distinct experts: need k <= E")
        topk, w = route_uniform(g, T, E, k, p_invalid)
    elif routing == "zipf":
        topk, w, p = route_zipf(g, T, E, k, zipf_s, zero_experts)
        meta["popularity"] = p
    elif routing == "repeats":          # picks drawn with replacement (an expert may repeat)
        topk = torch.randint(0, E, (T, k), generator=g, dtype=torch.int64)
        valid = torch.rand(T, k, generator=g) >= p_invalid
        topk = torch.where(valid, topk, torch.full_like(topk, -1))
        w = _masked_softmax(torch.randn(T, k, generator=g), valid)
    elif routing == "invalid":          # every pick dropped
        topk = torch.full((T, k), -1, dtype=torch.int64)
        w = torch.zeros(T, k, dtype=torch.float32)
    else:
        raise ValueError(routing)
    x, x_scale = make_rows(g, T, H, dtype, scales)
    if experts == "random":
        eo = _randn_bf16(g, T * k, H)
    elif experts == "identity":
        if dtype != "bf16":
            raise ValueError("identity experts need bf16 rows")
        eo = None
    else:
        raise ValueError(experts)
    return Case(name=name, T=T, H=H, k=k, E=E, R=R, N=N, dtype=dtype, topk_idx=topk,
                topk_weights=w, x=x, x_scale=x_scale, expert_out=eo, meta=meta)


def decode_cases(steps: int, first_seed: int = 1000):
    """The decode workload: independent T=128 steps with seeds first_seed + i."""
    return [make_case("decode_fp8", seed=first_seed + i) for i in range(steps)]
