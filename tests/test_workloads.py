"""The seeded input generator produces the shapes and routing the workloads name (no GPU)."""
import numpy as np
import torch

import oracle
from unpermute_ep_dispatch_gb300 import workloads


def test_skew_routing_is_lumpy():
    """Zipf(1.2) popularity: some expert takes >10% of the rows and >=20 take none."""
    c = workloads.make_case("skew_bf16", T=16384, experts="identity")
    lay = oracle.dispatch_layout(c.topk_idx.numpy(), c.E, c.R, c.N)
    cnt = lay["tokens_per_expert"]
    assert cnt.max() / cnt.sum() > 0.10
    assert (cnt == 0).sum() >= 20
    # k distinct experts per token
    srt = np.sort(c.topk_idx.numpy(), axis=1)
    assert np.all(np.diff(srt, axis=1) > 0)


def test_prefill_drops_about_two_percent():
    c = workloads.make_case("prefill_bf16", T=4096)
    frac = (c.topk_idx == -1).float().mean().item()
    assert 0.015 < frac < 0.025
    w = c.topk_weights
    assert torch.all(w[c.topk_idx == -1] == 0)
    has = (c.topk_idx >= 0).any(dim=1)
    assert torch.allclose(w[has].double().sum(dim=1), torch.ones(int(has.sum()), dtype=torch.float64),
                          atol=1e-6)


def test_fp8_rows_and_scales():
    c = workloads.make_case("dsv3_fp8", T=64)
    assert c.x.dtype == torch.float8_e4m3fn and c.x.shape == (64, 7168)
    assert c.x_scale.shape == (64, 56) and c.x_scale.dtype == torch.float32
    deq = c.x.float().reshape(64, 56, 128) * c.x_scale.unsqueeze(2)
    assert torch.isfinite(deq).all()
    assert c.x.float().abs().max().item() <= 448.0
    assert c.expert_out.shape == (64 * 8, 7168) and c.expert_out.dtype == torch.bfloat16


def test_tiny_matches_worked_setting():
    c = workloads.make_case("tiny")
    assert (c.T, c.H, c.E, c.R, c.N, c.k) == (64, 256, 16, 8, 2, 2)
    assert torch.all(c.topk_idx >= 0)
    assert torch.allclose(c.topk_weights.sum(dim=1), torch.ones(64), atol=1e-6)


def test_seeded_and_repeatable():
    a = workloads.make_case("decode_fp8", seed=1003)
    b = workloads.make_case("decode_fp8", seed=1003)
    assert torch.equal(a.topk_idx, b.topk_idx)
    assert torch.equal(a.x.view(torch.uint8), b.x.view(torch.uint8))
    c = workloads.make_case("decode_fp8", seed=1004)
    assert not torch.equal(a.topk_idx, c.topk_idx)
