"""The allocation-free layout entry point, called through the C ABI.

ep_dispatch_layout_noalloc serves callers that own their inputs and outputs but
cannot allocate the workspace (device memory planned up front by a host
framework, or no allocator on a hot path). Its scratch is a fixed device array
inside libepd, shared by every call. Two calls in a row must each give what
ep_dispatch_layout gives with a caller workspace (counts and masks are integer
results: bit-exact). This file is collected last so that a run stopping at the
first failure has already run every other test; it passes alone in a fresh
process too (the array starts zeroed when the library loads).
"""
import ctypes

import pytest
import torch

import unpermute_ep_dispatch_gb300 as epd
from unpermute_ep_dispatch_gb300 import _binding, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from unpermute_ep_dispatch_gb300 import build
    build.build()
    return epd.load_library()


def _outputs(T, E, R, N, dev, fill):
    return (torch.full((E,), fill, dtype=torch.int32, device=dev),
            torch.full((R,), fill, dtype=torch.int32, device=dev),
            torch.full((N,), fill, dtype=torch.int32, device=dev),
            torch.zeros(T, R, dtype=torch.bool, device=dev))


@pytest.mark.parametrize("name,T", [("dsv3_fp8", 8192), ("skew_bf16", 4096), ("tiny", 64)])
def test_noalloc_layout_matches_workspace_layout_twice(lib, name, T):
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    for call, seed in enumerate((101, 202)):            # two calls in a row
        case = workloads.make_case(name, T=T, seed=seed, experts="identity"
                                   if name != "dsv3_fp8" else "random")
        topk = case.topk_idx.to(dev)
        E, R, N = case.E, case.R, case.N
        status_a = epd.new_status(dev)
        status_b = epd.new_status(dev)
        ws = epd.new_workspace(T, case.k, E, R, N, dev)
        per_e_a, per_r_a, per_n_a, itr_a = _outputs(T, E, R, N, dev, -7)
        per_e_b, per_r_b, per_n_b, itr_b = _outputs(T, E, R, N, dev, -9)
        rc = lib.ep_dispatch_layout(
            ctypes.c_void_p(topk.data_ptr()), T, case.k, E, R, N,
            ctypes.c_void_p(per_e_a.data_ptr()), ctypes.c_void_p(per_r_a.data_ptr()),
            ctypes.c_void_p(per_n_a.data_ptr()), ctypes.c_void_p(itr_a.data_ptr()),
            ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(status_a.data_ptr()),
            ctypes.c_void_p(stream.cuda_stream))
        assert rc == epd.EPD_OK
        rc = lib.ep_dispatch_layout_noalloc(
            ctypes.c_void_p(topk.data_ptr()), T, case.k, E, R, N,
            ctypes.c_void_p(per_e_b.data_ptr()), ctypes.c_void_p(per_r_b.data_ptr()),
            ctypes.c_void_p(per_n_b.data_ptr()), ctypes.c_void_p(itr_b.data_ptr()),
            ctypes.c_void_p(status_b.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert rc == epd.EPD_OK, f"call {call}: {_binding.status_string(rc)}"
        torch.cuda.synchronize(dev)
        assert int(status_a.item()) == 0 and int(status_b.item()) == 0
        assert torch.equal(per_e_a, per_e_b), f"call {call}: tokens_per_expert"
        assert torch.equal(per_r_a, per_r_b), f"call {call}: tokens_per_rank"
        assert torch.equal(per_n_a, per_n_b), f"call {call}: tokens_per_rdma_rank"
        assert torch.equal(itr_a, itr_b), f"call {call}: is_token_in_rank"
        assert int(per_e_b.sum().item()) == int((case.topk_idx >= 0).sum().item())


def test_noalloc_binding_and_size_limit(lib):
    dev = torch.device("cuda")
    case = workloads.make_case("tiny", seed=3)
    topk = case.topk_idx.to(dev)
    E, R, N = case.E, case.R, case.N
    st = epd.new_status(dev)
    per_e, per_r, per_n, itr = _outputs(case.T, E, R, N, dev, 0)
    _binding.ep_dispatch_layout_noalloc(topk, E, R, N, st, per_e, per_r, per_n, itr)
    ref = epd.ep_dispatch_layout(topk, E, R, N, epd.new_workspace(case.T, case.k, E, R, N, dev),
                                 epd.new_status(dev))
    torch.cuda.synchronize(dev)
    assert torch.equal(per_r, ref[0]) and torch.equal(per_n, ref[1])
    assert torch.equal(per_e, ref[2]) and torch.equal(itr, ref[3])
    # beyond the fixed scratch: rejected on the host with a clear error, nothing launched
    T_big, k_big = 1 << 21, 8
    assert lib.epd_workspace_bytes(T_big, k_big, 256, 32, 4) > (8 << 20)
    rc = lib.ep_dispatch_layout_noalloc(
        ctypes.c_void_p(topk.data_ptr()), T_big, k_big, 256, 32, 4,
        ctypes.c_void_p(per_e.data_ptr()), ctypes.c_void_p(per_r.data_ptr()), None, None,
        ctypes.c_void_p(st.data_ptr()), None)
    assert rc == epd.EPD_ERR_UNSUPPORTED


def test_noalloc_shape_changes_leave_no_stale_state(lib):
    """The shared array keeps each call's leftovers. A big call writes its pair ranks
    where a smaller call keeps its look-back state words or its clusters' published
    counts; the smaller call must not read them as published. Repeated, alternating
    shapes -- the tile form (320 000 pairs), several clusters (131 072 pairs) and one
    cluster -- each result against the oracle."""
    import numpy as np

    import oracle
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    E, R, N, k = 256, 32, 4, 8
    shapes = [(40000, 305), (8192, 301), (16384, 306), (2048, 302), (4096, 303),
              (1100, 304)]                                          # (T, seed)
    cases = [workloads.make_random_case(T=T, H=16, k=k, E=E, R=R, N=N, dtype="bf16", seed=s,
                                        routing="repeats", p_invalid=0.05, experts="identity")
             for T, s in shapes]
    want = [oracle.dispatch_layout(c.topk_idx.numpy(), E, R, N) for c in cases]
    tops = [c.topk_idx.to(dev) for c in cases]
    st = epd.new_status(dev)
    for rep in range(100):
        outs = []
        for c, topk in zip(cases, tops):            # six calls back to back, then one sync
            o = _outputs(c.T, E, R, N, dev, -3)
            per_e, per_r, per_n, itr = o
            rc = lib.ep_dispatch_layout_noalloc(
                ctypes.c_void_p(topk.data_ptr()), c.T, k, E, R, N,
                ctypes.c_void_p(per_e.data_ptr()), ctypes.c_void_p(per_r.data_ptr()),
                ctypes.c_void_p(per_n.data_ptr()), ctypes.c_void_p(itr.data_ptr()),
                ctypes.c_void_p(st.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
            assert rc == epd.EPD_OK
            outs.append(o)
        torch.cuda.synchronize(dev)
        assert int(st.item()) == 0, f"rep {rep}: status {int(st.item())}"
        for c, w, (per_e, per_r, per_n, itr) in zip(cases, want, outs):
            what = f"rep {rep} T={c.T}"
            assert np.array_equal(per_e.cpu().numpy(), w["tokens_per_expert"]), what
            assert np.array_equal(per_r.cpu().numpy(), w["tokens_per_rank"]), what
            assert np.array_equal(per_n.cpu().numpy(), w["tokens_per_rdma_rank"]), what
            assert np.array_equal(itr.cpu().numpy(), w["is_token_in_rank"]), what
