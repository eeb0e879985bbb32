"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Bit-exact for counts, is_token_in_rank, offsets, m_indices, output_index and the
permuted rows / scales; the bf16 combine within 1e-3 + 1e-2 |ref| per element.
"""
import numpy as np
import pytest
import torch

import unpermute_ep_dispatch_gb300 as epd
from epd_paths import GpuPath, bits16, compare, oracle_path, row_bytes
from unpermute_ep_dispatch_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from unpermute_ep_dispatch_gb300 import build
    build.build()
    epd.load_library()


def run_both(case, capacity=None, stream=None, alignment=1):
    g = GpuPath(case, capacity=capacity, stream=stream, alignment=alignment)
    g.step()
    got = g.results()
    want = oracle_path(case, capacity=capacity, alignment=alignment)
    return got, want, g


# ----------------------------------------------------------------------------- the five workloads
@pytest.mark.parametrize("name", ["tiny", "prefill_bf16", "dsv3_fp8", "skew_bf16"])
def test_workload_full_size(name):
    case = workloads.make_case(name)
    got, want, _ = run_both(case)
    err = compare(got, want)
    print(f"{name}: P={want['total_rows']} combine error {err:.3f} of tolerance")


def test_decode_steps():
    for i in range(8):
        case = workloads.make_case("decode_fp8", seed=1000 + i)
        got, want, _ = run_both(case)
        compare(got, want)


def test_identity_experts_give_back_x():
    """Weights that sum to 1 over identity experts: y == x exactly (0 for no pick)."""
    case = workloads.make_case("prefill_bf16")
    g = GpuPath(case)
    g.step()
    r = g.results()
    xb = bits16(case.x)
    has = (case.topk_idx >= 0).any(dim=1).numpy()
    assert np.array_equal(r["y"][has], xb[has])
    assert np.all(r["y"][~has] == 0)


# ----------------------------------------------------------------------------- edge cases
EDGE_T = [0, 1, 2, 3, 31, 33, 65, 257, 1000]
EDGE_TOPO = [(1, 1, 1), (2, 2, 1), (16, 8, 2), (256, 32, 4)]   # (E, R, N)


@pytest.mark.parametrize("T", EDGE_T)
@pytest.mark.parametrize("k", [1, 2, 8])
@pytest.mark.parametrize("topo", EDGE_TOPO)
@pytest.mark.parametrize("p_invalid", [0.0, 0.5, 1.0])
def test_edge_matrix_bf16(T, k, topo, p_invalid):
    E, R, N = topo
    case = workloads.make_random_case(T=T, H=136, k=k, E=E, R=R, N=N, dtype="bf16",
                                      seed=T * 7 + k * 131 + E, routing="repeats",
                                      p_invalid=p_invalid, experts="random")
    got, want, _ = run_both(case)
    compare(got, want)


@pytest.mark.parametrize("T", [0, 1, 33, 257])
@pytest.mark.parametrize("k,E,R,N", [(1, 16, 8, 2), (8, 256, 32, 4), (6, 64, 8, 1)])
@pytest.mark.parametrize("H", [128, 384])
def test_edge_fp8(T, k, E, R, N, H):
    case = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype="fp8",
                                      seed=T + k + H, routing="uniform", p_invalid=0.25,
                                      experts="random")
    got, want, _ = run_both(case)
    compare(got, want)


@pytest.mark.parametrize("T", [1, 300, 2100])
@pytest.mark.parametrize("topo", [(16, 8, 2), (256, 32, 4)])
def test_zero_topk(T, topo):
    """k = 0: no pairs, zero counts and masks, an empty buffer and y = 0 (2100 tokens
    are two layout tiles)."""
    E, R, N = topo
    case = workloads.make_random_case(T=T, H=136, k=0, E=E, R=R, N=N, dtype="bf16", seed=T,
                                      routing="uniform", experts="random")
    got, want, _ = run_both(case)
    compare(got, want)
    assert not got["y"].any()


def test_large_topk_and_repeated_experts():
    """k = 64 (the limit) over 4 experts: long runs of the same expert in a row."""
    case = workloads.make_random_case(T=300, H=64, k=64, E=4, R=2, N=1, dtype="bf16", seed=4,
                                      routing="repeats", p_invalid=0.1, experts="random")
    got, want, _ = run_both(case)
    compare(got, want)


def test_many_experts():
    case = workloads.make_random_case(T=700, H=64, k=8, E=4096, R=512, N=8, dtype="bf16",
                                      seed=6, routing="uniform", experts="random")
    got, want, _ = run_both(case)
    compare(got, want)


def test_capacity_above_tk_fills_tail():
    case = workloads.make_random_case(T=200, H=64, k=4, E=16, R=4, N=2, dtype="bf16", seed=8,
                                      routing="uniform", p_invalid=0.3, experts="random")
    got, want, _ = run_both(case, capacity=200 * 4 + 333)
    compare(got, want)
    assert np.all(got["m_indices"][want["total_rows"]:] == -1)


def test_ragged_hidden_bf16():
    for H in (8, 24, 7176):
        case = workloads.make_random_case(T=45, H=H, k=3, E=8, R=4, N=2, dtype="bf16", seed=H,
                                          routing="uniform", experts="random")
        got, want, _ = run_both(case)
        compare(got, want)


def test_very_wide_rows_use_the_register_permute():
    """Rows too wide for two shared-memory stages (128 KiB bf16 rows) take the
    register-copy permute; the result is the same."""
    case = workloads.make_random_case(T=33, H=65536, k=2, E=8, R=4, N=2, dtype="bf16", seed=12,
                                      routing="uniform", p_invalid=0.2, experts="random")
    got, want, _ = run_both(case)
    compare(got, want)


def test_side_stream():
    s = torch.cuda.Stream()
    case = workloads.make_case("tiny")
    with torch.cuda.stream(s):
        got, want, _ = run_both(case, stream=s)
    compare(got, want)


# ----------------------------------------------------------------------------- determinism & reuse
def test_deterministic_and_workspace_reuse():
    case = workloads.make_case("dsv3_fp8", T=3000)
    g = GpuPath(case)
    g.step()
    first = g.results()
    for _ in range(3):
        g.step()
    again = g.results()
    for key in first:
        a, b = first[key], again[key]
        if isinstance(a, np.ndarray):
            P = first["total_rows"]
            if key in ("out", "out_scale"):
                a, b = a[:P], b[:P]
            assert np.array_equal(a, b), key
        else:
            assert a == b, key


def test_workspace_shared_across_shapes():
    """One workspace, sized for the largest shape, reused for smaller ones; one-tile
    calls (which take no ticket and publish nothing) between many-tile calls leave the
    ticket and call counter as the next many-tile call needs them."""
    big = workloads.make_case("dsv3_fp8", T=2048)
    ws = epd.new_workspace(2048, 8, 256, 32, 4)
    for T in (2048, 17, 17, 1500, 1, 2048, 256):
        case = workloads.make_case("dsv3_fp8", T=T, seed=T)
        g = GpuPath(case)
        g.ws = ws[: epd.epd_workspace_bytes(T, 8, 256, 32, 4)]
        g.step()
        compare(g.results(), oracle_path(case))
    del big


# ----------------------------------------------------------------------------- failure paths
def test_invalid_expert_ids_are_reported_and_skipped():
    case = workloads.make_random_case(T=150, H=64, k=4, E=16, R=8, N=2, dtype="bf16", seed=2,
                                      routing="uniform", experts="random")
    bad = case.topk_idx.clone()
    bad[3, 1] = 16
    bad[77, 0] = -5
    bad[149, 3] = 1 << 40
    case_bad = workloads.Case(**{**case.__dict__, "topk_idx": bad})
    g = GpuPath(case_bad)
    g.step()
    got = g.results()
    assert got["status"] == epd.EPD_ERR_INVALID_EXPERT
    clean = torch.where((bad >= -1) & (bad < 16), bad, torch.full_like(bad, -1))
    want = oracle_path(case, topk_override=clean)
    compare(got, want, check_status=False)


def test_lookback_wait_gives_up_and_workspace_recovers():
    """A tile that never publishes: later tiles stop waiting after a bounded number
    of polls and report EPD_ERR_TIMEOUT; the next normal call is correct."""
    case = workloads.make_case("dsv3_fp8", T=2048)
    g = GpuPath(case)
    epd._binding.epd_test_layout_stalled_tile(g.topk, case.E, case.R, case.N, g.ws, g.status,
                                              stalled_tile=0, spin_limit=2000)
    torch.cuda.synchronize()
    assert int(g.status.item()) == epd.EPD_ERR_TIMEOUT
    g.status.zero_()
    g.step()
    compare(g.results(), oracle_path(case))


def test_permute_rejects_workspace_of_another_layout():
    a = workloads.make_case("tiny")
    b = workloads.make_case("tiny", T=32, seed=5)
    ga = GpuPath(a)
    ga.layout()
    gb = GpuPath(b)
    gb.ws = ga.ws[: gb.ws.numel()]
    gb.per_e.zero_()
    gb.scan()
    gb.output_index.fill_(123)
    gb.permute()
    torch.cuda.synchronize()
    assert int(gb.status.item()) == epd.EPD_ERR_INVALID_ARG
    assert torch.all(gb.output_index == 123)


def test_binding_validates_tensors():
    case = workloads.make_case("tiny")
    g = GpuPath(case)
    with pytest.raises(ValueError):
        epd.ep_dispatch_layout(g.topk.to(torch.int32), 16, 8, 2, g.ws, g.status)
    with pytest.raises(ValueError):
        epd.ep_dispatch_layout(g.topk, 16, 8, 2, g.ws[:16], g.status)
    with pytest.raises(epd.EpdError):
        epd.ep_dispatch_layout(g.topk, 16, 3, 1, g.ws, g.status)
    with pytest.raises(ValueError):
        epd.ep_unpermute(g.out.float(), g.output_index, g.w, g.status)


def test_cuda_graph_replay_of_the_step():
    """One step captured in a CUDA graph, replayed on fresh inputs copied into the
    captured buffers (the decode pattern): every replay matches the oracle."""
    cases = [workloads.make_case("decode_fp8", seed=2000 + i) for i in range(3)]
    g = GpuPath(cases[0])
    g.step()                                     # warm: library loaded, attributes set
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g.stream = s
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.step()
    for case in cases:
        g.case = case
        g.topk.copy_(case.topk_idx)
        g.w.copy_(case.topk_weights)
        g.x.copy_(case.x)
        g.xs.copy_(case.x_scale)
        g.eo.copy_(case.expert_out)
        torch.cuda.synchronize()
        graph.replay()
        compare(g.results(), oracle_path(case))


def test_cuda_graph_replay_of_the_cluster_layout_step():
    """A dsv3-shaped step (T=2048: the layout's cluster form, 16 blocks) with the
    layout and offsets in one launch, captured in a CUDA graph and replayed on fresh
    routings copied into the captured buffers: every replay matches the oracle."""
    cases = [workloads.make_case("dsv3_fp8", T=2048, seed=3000 + i) for i in range(3)]
    g = GpuPath(cases[0], fused=True)
    g.step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g.stream = s
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.step()
    for case in cases:
        g.case = case
        g.topk.copy_(case.topk_idx)
        g.w.copy_(case.topk_weights)
        g.x.copy_(case.x)
        g.xs.copy_(case.x_scale)
        g.eo.copy_(case.expert_out)
        torch.cuda.synchronize()
        for _ in range(2):          # two replays in a row on one workspace
            graph.replay()
        compare(g.results(), oracle_path(case))


# ----------------------------------------------------------------------------- expert alignment
@pytest.mark.parametrize("alignment", [4, 128, 256])
@pytest.mark.parametrize("name,T", [("tiny", None), ("dsv3_fp8", 2048), ("prefill_bf16", 1000),
                                    ("skew_bf16", 2048)])
def test_aligned_layouts(name, T, alignment):
    case = workloads.make_case(name, T=T)
    got, want, _ = run_both(case, alignment=alignment)
    compare(got, want)
    start = got["expert_start_loc"]
    assert np.all(start % alignment == 0)


def test_aligned_hand_example_on_gpu():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "hand_example_aligned4.json")))
    topk = torch.tensor(g["topk_idx"], dtype=torch.int64)
    case = workloads.make_random_case(T=4, H=64, k=2, E=16, R=8, N=2, dtype="bf16", seed=1,
                                      routing="uniform", experts="random")
    case = workloads.Case(**{**case.__dict__, "topk_idx": topk})
    got, want, _ = run_both(case, alignment=4)
    compare(got, want)
    assert got["expert_start_loc"].tolist() == g["expert_start_loc"]
    assert got["output_index"].tolist() == g["output_index"]
    assert got["m_indices"][:20].tolist() == g["m_indices_first_20"]


@pytest.mark.parametrize("T", [0, 1, 33])
@pytest.mark.parametrize("p_invalid", [0.0, 0.5, 1.0])
def test_aligned_edges(T, p_invalid):
    case = workloads.make_random_case(T=T, H=128, k=8, E=16, R=4, N=2, dtype="fp8", seed=T + 7,
                                      routing="repeats", p_invalid=p_invalid, experts="random")
    got, want, _ = run_both(case, alignment=64)
    compare(got, want)


# ----------------------------------------------------------------------------- views and scale layouts
def _words(t):
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)


@pytest.mark.parametrize("scales", ["f32", "ue8m0"])
@pytest.mark.parametrize("col_major", [False, True])
@pytest.mark.parametrize("alignment", [1, 128])
def test_permute_views_and_scale_layouts(scales, col_major, alignment):
    import oracle
    case = workloads.make_case("dsv3_fp8", T=2048, scales=scales)
    g = GpuPath(case, alignment=alignment)
    g.layout()
    g.scan()
    torch.cuda.synchronize()
    lay = oracle.dispatch_layout(case.topk_idx.numpy(), case.E, case.R, case.N)
    if alignment == 1:
        ostart, _ = oracle.scan_offsets(lay["tokens_per_expert"])
    else:
        ostart, _ = oracle.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    assert np.array_equal(g.start.cpu().numpy(), ostart)
    xs = case.x_scale.to(g.dev)
    xrows = row_bytes(case.x)
    for r in (0, 13, 31):
        b, e = r * 8, r * 8 + 8
        cap = 2048 * 8 // 4 + 8 * alignment         # a rank's rows stay far below this here
        ld = cap + 4 if col_major else None
        out, osc, mi, oi = epd.ep_permute_ex(g.x, xs, g.topk, case.E, g.start, g.ws, g.status,
                                             capacity_rows=cap, expert_begin=b, expert_end=e,
                                             scale_col_major=col_major, scale_ld=ld)
        torch.cuda.synchronize()
        assert int(g.status.item()) == 0
        want = oracle.permute_ex(xrows, _words(case.x_scale), case.topk_idx.numpy(), case.E,
                                 ostart, cap, expert_begin=b, expert_end=e,
                                 scale_col_major=col_major, scale_ld=ld)
        got_oi = oi.cpu().numpy()
        assert np.array_equal(got_oi, want["output_index"])
        assert np.array_equal(mi.cpu().numpy(), want["m_indices"])
        rows = got_oi[got_oi >= 0]
        assert np.array_equal(row_bytes(out)[rows], want["out"][rows])
        gs = _words(osc)
        if col_major:
            assert np.array_equal(gs[:, rows], want["out_scale"][:, rows])
        else:
            assert np.array_equal(gs[rows], want["out_scale"][rows])


@pytest.mark.parametrize("shape", ["whole", "whole_aligned", "half_view", "wide_rows", "no_picks"])
def test_permute_ex_column_major_scale_pass(shape):
    """Column-major scales of more than 16 words per row over a view of at least a
    quarter of the experts take the separate scale pass (the row copy parks each
    filled row's source token in m_indices; the pass writes the scales down their
    columns and the final m_indices). Rows, scales, m_indices and output_index equal
    the oracle's, on the bulk-copy kernel and on the register kernel (rows wider
    than two 32 KiB stages)."""
    import oracle
    alignment = 128 if shape == "whole_aligned" else 1
    if shape == "wide_rows":
        case = workloads.make_case("prefill_bf16", T=300)
    else:
        case = workloads.make_case("dsv3_fp8", T=2048)
    if shape == "no_picks":
        case = workloads.Case(**{**case.__dict__, "topk_idx": torch.full_like(case.topk_idx, -1)})
    g = GpuPath(case, alignment=alignment)
    g.layout()
    g.scan()
    torch.cuda.synchronize()
    T, k, E = case.T, case.k, case.E
    gen = torch.Generator().manual_seed(71)
    if shape == "wide_rows":
        x = torch.randint(0, 256, (T, 33024), generator=gen, dtype=torch.uint8)
        words = torch.randint(-2**31, 2**31 - 1, (T, 40), generator=gen, dtype=torch.int32)
    else:
        x = case.x
        words = case.x_scale.contiguous().view(torch.int32)
    b, e = (0, E // 2) if shape == "half_view" else (0, E)
    cap = oracle.aligned_capacity(T, k, E, alignment) if alignment > 1 else T * k
    ld = cap + 12
    lay = oracle.dispatch_layout(case.topk_idx.numpy(), E, case.R, case.N)
    if alignment == 1:
        ostart, _ = oracle.scan_offsets(lay["tokens_per_expert"])
    else:
        ostart, _ = oracle.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    assert np.array_equal(g.start.cpu().numpy(), ostart)
    dx, dw = x.to(g.dev), words.to(g.dev)
    out, osc, mi, oi = epd.ep_permute_ex(dx, dw, g.topk, E, g.start, g.ws, g.status,
                                         capacity_rows=cap, expert_begin=b, expert_end=e,
                                         scale_col_major=True, scale_ld=ld)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    want = oracle.permute_ex(row_bytes(x), _words(words), case.topk_idx.numpy(), E, ostart, cap,
                             expert_begin=b, expert_end=e, scale_col_major=True, scale_ld=ld)
    got_oi = oi.cpu().numpy()
    assert np.array_equal(got_oi, want["output_index"])
    assert np.array_equal(mi.cpu().numpy(), want["m_indices"])
    rows = got_oi[got_oi >= 0]
    if shape == "no_picks":
        assert rows.size == 0 and (mi.cpu().numpy() == -1).all()
    assert np.array_equal(row_bytes(out)[rows], want["out"][rows])
    assert np.array_equal(_words(osc)[:, rows], want["out_scale"][:, rows])


def test_permute_ex_whole_range_equals_permute():
    case = workloads.make_case("prefill_bf16", T=1500)
    g = GpuPath(case)
    g.step()
    ref = g.results()
    out, _, mi, oi = epd.ep_permute_ex(g.x, None, g.topk, case.E, g.start, g.ws, g.status,
                                       capacity_rows=g.cap)
    torch.cuda.synchronize()
    assert np.array_equal(oi.cpu().numpy(), ref["output_index"])
    assert np.array_equal(mi.cpu().numpy(), ref["m_indices"])
    rows = ref["output_index"][ref["output_index"] >= 0]
    assert np.array_equal(row_bytes(out)[rows], ref["out"][rows])


# ----------------------------------------------------------------------------- low-latency layout
def _ll_compare(case, rows, b=0, e_end=None, expect_status=0):
    import oracle
    dev = torch.device("cuda")
    E = case.E
    e_end = E if e_end is None else e_end
    topk = case.topk_idx.to(dev)
    x = case.x.to(dev)
    ws = epd.new_workspace(case.T, case.k, E, case.R, case.N, dev)
    st = epd.new_status(dev)
    epd.ep_dispatch_layout(topk, E, case.R, case.N, ws, st)
    q, sc, rc, oi, src = epd.ep_permute_lowlatency(x, topk, E, rows, ws, st, expert_begin=b,
                                                   expert_end=e_end)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    want = oracle.permute_lowlatency(bits16(case.x), case.topk_idx.numpy(), E, rows, b, e_end)
    assert want["overflow"] == (expect_status == epd.EPD_ERR_CAPACITY)
    got_oi = oi.cpu().numpy()
    assert np.array_equal(got_oi, want["output_index"])
    rcount = rc.cpu().numpy()
    assert np.array_equal(rcount, want["recv_count"])
    qb = q.cpu().view(torch.uint8).numpy().reshape(-1, case.H)
    used = got_oi[got_oi >= 0]
    assert np.array_equal(qb[used], want["out_q"].reshape(-1, case.H)[used])
    gs = sc.cpu().numpy()
    for e in range(e_end - b):
        n = rcount[e]
        assert np.array_equal(gs[e, :, :n], want["out_scale"][e, :, :n])
        assert np.array_equal(src.cpu().numpy()[e, :n], want["src_token"][e, :n])
    return oi, want


def _bf16_decode_case(T=128, seed=3000, **kw):
    return workloads.make_random_case(T=T, H=kw.pop("H", 7168), k=8, E=256, R=32, N=4,
                                      dtype="bf16", seed=seed, routing=kw.pop("routing", "uniform"),
                                      experts="random", **kw)


def test_lowlatency_decode_shape():
    case = _bf16_decode_case()
    _ll_compare(case, rows=128)


def test_lowlatency_rank_view():
    case = _bf16_decode_case(T=300, seed=3001)
    _ll_compare(case, rows=300, b=64, e_end=72)


def test_lowlatency_overflow_is_reported_and_dropped():
    case = _bf16_decode_case(T=200, seed=3002)
    _ll_compare(case, rows=3, expect_status=epd.EPD_ERR_CAPACITY)


@pytest.mark.parametrize("T", [0, 1, 33])
@pytest.mark.parametrize("H", [128, 384])
def test_lowlatency_edges(T, H):
    case = _bf16_decode_case(T=T, seed=3003 + T, H=H, routing="repeats", p_invalid=0.3)
    _ll_compare(case, rows=max(T, 1))


def test_lowlatency_half_view():
    """A view of half the experts loads rows before their slots are known."""
    case = _bf16_decode_case(T=300, seed=3006)
    _ll_compare(case, rows=300, b=128, e_end=256)


@pytest.mark.parametrize("T", [0, 5, 130])
def test_lowlatency_zero_topk(T):
    case = workloads.make_random_case(T=T, H=256, k=0, E=16, R=8, N=2, dtype="bf16", seed=T,
                                      routing="uniform", experts="random")
    _ll_compare(case, rows=4)


def test_lowlatency_rejects_workspace_of_another_layout():
    """A workspace whose header names another T: EPD_ERR_INVALID_ARG and no output
    written (each warp checks the header before its first store)."""
    dev = torch.device("cuda")
    a = _bf16_decode_case(T=64, seed=3007)
    b = _bf16_decode_case(T=96, seed=3008)
    ws = epd.new_workspace(b.T, b.k, b.E, b.R, b.N, dev)
    st = epd.new_status(dev)
    epd.ep_dispatch_layout(a.topk_idx.to(dev), a.E, a.R, a.N, ws, st)
    torch.cuda.synchronize()
    oi = torch.full((b.T, b.k), 123, dtype=torch.int32, device=dev)
    rc = torch.full((b.E,), 77, dtype=torch.int32, device=dev)
    epd.ep_permute_lowlatency(b.x.to(dev), b.topk_idx.to(dev), b.E, 16, ws, st,
                              output_index=oi, recv_count=rc)
    torch.cuda.synchronize()
    assert int(st.item()) == epd.EPD_ERR_INVALID_ARG
    assert torch.all(oi == 123) and torch.all(rc == 77)


def test_lowlatency_prefill_size():
    case = _bf16_decode_case(T=2048, seed=3004)
    _ll_compare(case, rows=256)


def test_combine_over_rectangles():
    import oracle
    case = _bf16_decode_case(T=128, seed=3005)
    oi, want = _ll_compare(case, rows=128)
    dev = torch.device("cuda")
    eo = torch.randn(256 * 128, case.H, generator=torch.Generator().manual_seed(7)).to(
        torch.bfloat16)
    st = epd.new_status(dev)
    y = epd.ep_unpermute(eo.to(dev), oi, case.topk_weights.to(dev), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.unpermute(bits16(eo), want["output_index"], case.topk_weights.numpy())
    from epd_paths import combine_error
    assert combine_error(bits16(y), ref) <= 1.0


# ----------------------------------------------------------------------------- fused layout + offsets
@pytest.mark.parametrize("alignment", [1, 128])
@pytest.mark.parametrize("name,T", [("dsv3_fp8", None), ("skew_bf16", 3000), ("tiny", None),
                                    ("decode_fp8", None), ("prefill_bf16", 0)])
def test_fused_layout_offsets_match_separate_steps(name, T, alignment):
    case = workloads.make_case(name, T=T)
    g = GpuPath(case, alignment=alignment)
    g.layout()
    g.scan()
    torch.cuda.synchronize()
    ws2 = epd.new_workspace(case.T, case.k, case.E, case.R, case.N)
    st2 = epd.new_status()
    per_r, per_n, per_e, itr, start, total = epd.ep_dispatch_layout_offsets(
        g.topk, case.E, case.R, case.N, ws2, st2, alignment=alignment, with_rdma=True)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.equal(per_e, g.per_e) and torch.equal(per_r, g.per_r)
    assert torch.equal(per_n, g.per_n) and torch.equal(itr, g.itr)
    assert torch.equal(start, g.start) and torch.equal(total, g.total)
    # and the permute / combine on the fused layout's workspace match the oracle
    g.ws = ws2
    g.start.copy_(start)
    g.permute()
    g.unpermute()
    compare(g.results(), oracle_path(case, alignment=alignment))


# ----------------------------------------------------------------------------- seeded random sweep
_TOPOS = [(1, 1, 1), (2, 2, 1), (4, 2, 2), (16, 8, 2), (64, 8, 1), (96, 12, 3), (256, 32, 4),
          (512, 64, 8), (1024, 128, 16), (4096, 512, 8)]


def _sweep_config(i):
    """Configuration i of the sweep, drawn from its own seed: topology, k (0 and 64
    included), T across tile boundaries, dtype and row width, routing style, dropped
    picks, alignment, whether the offsets are fused into the layout launch, and
    whether ep_dispatch runs the first three steps. Rows are kept to a few MB so
    that the oracle finishes in well under a second."""
    rng = np.random.default_rng(9000 + i)
    E, R, N = _TOPOS[int(rng.integers(len(_TOPOS)))]
    k = int(rng.choice([0, 1, 2, 3, 4, 6, 8, 9, 16, 64]))
    T = int(rng.choice([0, 1, 7, 31, 32, 33, 100, 257, 1000, 2049, 4097]))
    if k == 64:
        T = min(T, 300)
    dtype = str(rng.choice(["bf16", "fp8"]))
    widths = [128, 256, 384] if dtype == "fp8" else [8, 64, 136, 1024]
    elem = 1 if dtype == "fp8" else 2
    widths = [h for h in widths if T * max(k, 1) * h * elem <= 8 << 20] or widths[:1]
    H = int(rng.choice(widths))
    routing = str(rng.choice(["uniform", "repeats", "zipf", "invalid"]))
    if routing == "uniform" and k > E:
        routing = "repeats"
    if routing == "zipf" and (E < 256 or k > 16):
        routing = "repeats"
    p_invalid = float(rng.choice([0.0, 0.1, 0.5]))
    alignment = int(rng.choice([1, 1, 4, 64, 128]))
    fused = bool(rng.integers(2))
    dispatch = bool(rng.integers(3) == 0)  # layout, offsets and permute through ep_dispatch
    return dict(E=E, R=R, N=N, k=k, T=T, dtype=dtype, H=H, routing=routing,
                p_invalid=p_invalid, alignment=alignment, fused=fused, dispatch=dispatch)


@pytest.mark.parametrize("i", range(40))
def test_random_sweep(i):
    cfg = _sweep_config(i)
    case = workloads.make_random_case(T=cfg["T"], H=cfg["H"], k=cfg["k"], E=cfg["E"],
                                      R=cfg["R"], N=cfg["N"], dtype=cfg["dtype"], seed=9100 + i,
                                      routing=cfg["routing"], p_invalid=cfg["p_invalid"],
                                      experts="random", zero_experts=20)
    if cfg["dispatch"]:
        g = _dispatch_path(case, alignment=cfg["alignment"])
    else:
        g = GpuPath(case, alignment=cfg["alignment"], fused=cfg["fused"])
        g.step()
    got = g.results()
    want = oracle_path(case, alignment=cfg["alignment"])
    compare(got, want)


def _sweep_view(rng, E, R):
    kind = str(rng.choice(["whole", "half", "rank", "quarter"]))
    if kind == "whole":
        return 0, E
    if kind == "half":
        return (0, E // 2) if E >= 2 and rng.integers(2) else (E - max(1, E // 2), E)
    if kind == "quarter":
        q = max(1, E // 4)
        b = int(rng.integers(0, E - q + 1))
        return b, b + q
    r = int(rng.integers(R))
    return r * (E // R), (r + 1) * (E // R)


@pytest.mark.parametrize("i", range(16))
def test_random_sweep_permute_ex(i):
    """ep_permute_ex over random views, scale word counts and layouts (row- or
    column-major, leading dimension with slack) and alignments, against the oracle."""
    import oracle
    rng = np.random.default_rng(9500 + i)
    E, R, N = _TOPOS[int(rng.integers(3, 8))]
    k = int(rng.choice([1, 2, 6, 8]))
    T = int(rng.choice([1, 33, 257, 1000, 2049]))
    alignment = int(rng.choice([1, 4, 128]))
    scales = str(rng.choice(["f32", "ue8m0", "words"]))
    H = int(rng.choice([128, 256, 1024]))
    case = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype="fp8", seed=9600 + i,
                                      routing="repeats", p_invalid=0.2, experts="random",
                                      scales="ue8m0" if scales == "ue8m0" else "f32")
    if scales == "words":  # opaque 32-bit words, more than 16 per row
        words = torch.randint(-2**31, 2**31 - 1, (T, int(rng.choice([17, 40]))),
                              generator=torch.Generator().manual_seed(i), dtype=torch.int32)
    else:
        words = case.x_scale.contiguous()
        if words.dtype == torch.float32:
            words = words.view(torch.int32)
    g = GpuPath(case, alignment=alignment, fused=True)
    g.layout_offsets()
    torch.cuda.synchronize()
    b, e = _sweep_view(rng, E, R)
    cap = oracle.aligned_capacity(T, k, E, alignment) if alignment > 1 else T * k
    col = bool(rng.integers(2))
    ld = cap + int(rng.integers(0, 40)) if col else None
    ostart = g.start.cpu().numpy()
    out, osc, mi, oi = epd.ep_permute_ex(g.x, words.to(g.dev), g.topk, E, g.start, g.ws, g.status,
                                         capacity_rows=cap, expert_begin=b, expert_end=e,
                                         scale_col_major=col, scale_ld=ld)
    torch.cuda.synchronize()
    assert int(g.status.item()) == 0
    lay = oracle.dispatch_layout(case.topk_idx.numpy(), E, R, N)
    if alignment == 1:
        want_start, _ = oracle.scan_offsets(lay["tokens_per_expert"])
    else:
        want_start, _ = oracle.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    assert np.array_equal(ostart, want_start)
    want = oracle.permute_ex(row_bytes(case.x), _words(words), case.topk_idx.numpy(), E,
                             want_start, cap, expert_begin=b, expert_end=e,
                             scale_col_major=col, scale_ld=ld)
    got_oi = oi.cpu().numpy()
    assert np.array_equal(got_oi, want["output_index"])
    assert np.array_equal(mi.cpu().numpy(), want["m_indices"])
    rows = got_oi[got_oi >= 0]
    assert np.array_equal(row_bytes(out)[rows], want["out"][rows])
    gs = _words(osc)
    if col:
        assert np.array_equal(gs[:, rows], want["out_scale"][:, rows])
    else:
        assert np.array_equal(gs[rows], want["out_scale"][rows])


@pytest.mark.parametrize("i", range(12))
def test_random_sweep_lowlatency(i):
    """ep_permute_lowlatency (even i) and ep_dispatch_lowlatency (odd i) over random
    sizes, views and rectangle heights (some too small, which must report
    EPD_ERR_CAPACITY and drop exactly the oracle's picks), against the oracle."""
    import oracle
    rng = np.random.default_rng(9700 + i)
    E, R, N = _TOPOS[int(rng.integers(3, 8))]
    k = int(rng.choice([1, 2, 4, 8]))
    T = int(rng.choice([1, 31, 128, 300, 1000]))
    H = int(rng.choice([128, 384, 1024]))
    case = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype="bf16",
                                      seed=9800 + i, routing="repeats", p_invalid=0.1,
                                      experts="random")
    b, e = _sweep_view(rng, E, R)
    rows = int(rng.choice([1, 4, max(1, T * k // max(E, 1)), T]))
    if i % 2:  # the one-call form (one kernel for these sizes)
        _ll_dispatch_compare(case, rows, b, e)
        return
    want = oracle.permute_lowlatency(bits16(case.x), case.topk_idx.numpy(), E, rows, b, e)
    _ll_compare(case, rows=rows, b=b, e_end=e,
                expect_status=epd.EPD_ERR_CAPACITY if want["overflow"] else 0)


# ----------------------------------------------------------------------------- ep_dispatch
def _dispatch_path(case, alignment=1, capacity=None):
    """ep_dispatch then ep_unpermute; results in the GpuPath.results() form."""
    g = GpuPath(case, alignment=alignment, capacity=capacity)
    r = epd.ep_dispatch(g.x, g.xs, g.topk, case.E, case.R, case.N, g.ws, g.status,
                        alignment=alignment, capacity_rows=g.cap, tokens_per_expert=g.per_e,
                        tokens_per_rank=g.per_r, tokens_per_rdma_rank=g.per_n,
                        is_token_in_rank=g.itr, expert_start_loc=g.start, total_rows=g.total,
                        out=g.out, out_scale=g.out_scale, m_indices=g.m_indices,
                        output_index=g.output_index)
    assert r["out"] is g.out
    g.unpermute()
    return g


DISPATCH_CASES = [
    # (name, T, H, k, E, R, N, dtype, routing, p_invalid, alignment)
    ("decode", 128, 7168, 8, 256, 32, 4, "fp8", "uniform", 0.0, 1),
    ("decode_aligned", 128, 7168, 8, 256, 32, 4, "fp8", "uniform", 0.0, 128),
    ("tiny", 64, 256, 2, 16, 8, 2, "bf16", "uniform", 0.0, 1),
    ("prefill_small", 500, 4096, 6, 64, 8, 1, "bf16", "repeats", 0.02, 1),
    ("k1_many_tokens", 1024, 136, 1, 16, 4, 2, "bf16", "repeats", 0.1, 4),
    ("k4_4096_pairs", 1024, 128, 4, 1024, 64, 64, "fp8", "repeats", 0.2, 1),
    ("k64", 40, 64, 64, 4, 2, 1, "bf16", "repeats", 0.1, 1),
    ("k0", 77, 64, 0, 16, 8, 2, "bf16", "uniform", 0.0, 1),
    ("T0", 0, 64, 8, 16, 8, 2, "bf16", "uniform", 0.0, 1),
    ("all_dropped", 50, 64, 4, 16, 8, 2, "bf16", "repeats", 1.0, 64),
    ("scale_words_past_threads", 1000, 9216, 4, 64, 8, 2, "fp8", "uniform", 0.0, 1),
    ("block_rows_64KiB", 1000, 8192, 4, 64, 8, 2, "bf16", "uniform", 0.0, 1),
    ("two_kernels_dsv3", 2048, 7168, 8, 256, 32, 4, "fp8", "uniform", 0.0, 1),
    ("two_kernels_many_experts", 300, 64, 8, 4096, 512, 8, "bf16", "uniform", 0.0, 1),
    ("two_kernels_wide_ranks", 200, 64, 8, 256, 128, 4, "bf16", "uniform", 0.0, 1),
]


@pytest.mark.parametrize("cfg", DISPATCH_CASES, ids=[c[0] for c in DISPATCH_CASES])
def test_dispatch_matches_oracle(cfg):
    """ep_dispatch (one kernel for a small batch, the two kernels beyond) gives the
    oracle's counts, masks, offsets, rows, scales, m_indices and output_index."""
    _, T, H, k, E, R, N, dtype, routing, p_invalid, alignment = cfg
    case = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype=dtype,
                                      seed=T * 13 + k + E, routing=routing,
                                      p_invalid=p_invalid, experts="random")
    g = _dispatch_path(case, alignment=alignment)
    compare(g.results(), oracle_path(case, alignment=alignment))


@pytest.mark.parametrize("T", [1, 128, 700])
def test_dispatch_equals_separate_calls_and_workspace(T):
    """Same bytes as ep_dispatch_layout_offsets + ep_permute, workspace pair ranks and
    header included (a later ep_permute on the workspace gives the same rows)."""
    case = workloads.make_random_case(T=T, H=256, k=8, E=256, R=32, N=4, dtype="fp8",
                                      seed=T, routing="uniform", experts="random")
    a = _dispatch_path(case)
    b = GpuPath(case, fused=True)
    b.step()
    ra, rb = a.results(), b.results()
    for key in ("tokens_per_expert", "tokens_per_rank", "tokens_per_rdma_rank",
                "is_token_in_rank", "expert_start_loc", "m_indices", "output_index"):
        assert np.array_equal(ra[key], rb[key]), key
    n = T * 8 * 4
    off = 256  # per-pair ranks follow the 256-byte header block
    assert torch.equal(a.ws[off:off + n], b.ws[off:off + n])
    # the header names this layout: ep_permute on a's workspace succeeds and agrees
    out, _, mi, oi = epd.ep_permute(a.x, a.xs, a.topk, case.E, a.start, a.ws, a.status)
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0
    assert np.array_equal(oi.cpu().numpy(), rb["output_index"])
    assert np.array_equal(mi.cpu().numpy(), rb["m_indices"])


def test_dispatch_reports_invalid_ids_and_capacity():
    case = workloads.make_random_case(T=100, H=64, k=4, E=16, R=8, N=2, dtype="bf16", seed=5,
                                      routing="uniform", experts="random")
    bad = case.topk_idx.clone()
    bad[7, 2] = 16
    bad[90, 0] = -3
    case_bad = workloads.Case(**{**case.__dict__, "topk_idx": bad})
    g = _dispatch_path(case_bad)
    got = g.results()
    assert got["status"] == epd.EPD_ERR_INVALID_EXPERT
    clean = torch.where((bad >= -1) & (bad < 16), bad, torch.full_like(bad, -1))
    compare(got, oracle_path(case, topk_override=clean), check_status=False)
    # aligned offsets with a buffer of only T*k rows: slots past it are reported
    g2 = _dispatch_path(case, alignment=64, capacity=100 * 4)
    assert g2.results()["status"] == epd.EPD_ERR_CAPACITY


# ----------------------------------------------------------------------------- ep_dispatch_lowlatency
def _ll_dispatch_compare(case, rows, b=0, e_end=None):
    """ep_dispatch_lowlatency against the oracle (status from the oracle's overflow)."""
    import oracle
    dev = torch.device("cuda")
    E = case.E
    e_end = E if e_end is None else e_end
    topk = case.topk_idx.to(dev)
    x = case.x.to(dev)
    ws = epd.new_workspace(case.T, case.k, E, case.R, case.N, dev)
    st = epd.new_status(dev)
    q, sc, rc, oi, src = epd.ep_dispatch_lowlatency(x, topk, E, case.R, case.N, rows, ws, st,
                                                    expert_begin=b, expert_end=e_end)
    torch.cuda.synchronize()
    want = oracle.permute_lowlatency(bits16(case.x), case.topk_idx.numpy(), E, rows, b, e_end)
    assert int(st.item()) == (epd.EPD_ERR_CAPACITY if want["overflow"] else 0)
    got_oi = oi.cpu().numpy()
    assert np.array_equal(got_oi, want["output_index"])
    rcount = rc.cpu().numpy()
    assert np.array_equal(rcount, want["recv_count"])
    qb = q.cpu().view(torch.uint8).numpy().reshape(-1, case.H)
    used = got_oi[got_oi >= 0]
    assert np.array_equal(qb[used], want["out_q"].reshape(-1, case.H)[used])
    gs = sc.cpu().numpy()
    for e in range(e_end - b):
        n = rcount[e]
        assert np.array_equal(gs[e, :, :n], want["out_scale"][e, :, :n])
        assert np.array_equal(src.cpu().numpy()[e, :n], want["src_token"][e, :n])
    return oi


LL_DISPATCH_CASES = [
    # (name, T, H, k, E, R, N, routing, p_invalid, rows, view)
    ("decode", 128, 7168, 8, 256, 32, 4, "uniform", 0.0, 128, None),
    ("decode_rank_view", 128, 7168, 8, 256, 32, 4, "uniform", 0.0, 128, (40, 48)),
    ("decode_overflow", 128, 1024, 8, 256, 32, 4, "repeats", 0.1, 3, None),
    ("small_e", 300, 384, 4, 16, 8, 2, "repeats", 0.2, 300, (4, 12)),
    ("k1_many_tokens", 1024, 256, 1, 64, 8, 1, "repeats", 0.1, 64, None),
    ("k0", 50, 128, 0, 16, 8, 2, "uniform", 0.0, 4, None),
    ("T0", 0, 128, 8, 16, 8, 2, "uniform", 0.0, 4, None),
    ("two_kernels_prefill", 2048, 1024, 8, 256, 32, 4, "uniform", 0.0, 256, None),
    ("two_kernels_many_experts", 200, 256, 8, 2048, 256, 8, "uniform", 0.0, 8, (0, 1024)),
]


@pytest.mark.parametrize("cfg", LL_DISPATCH_CASES, ids=[c[0] for c in LL_DISPATCH_CASES])
def test_dispatch_lowlatency_matches_oracle(cfg):
    _, T, H, k, E, R, N, routing, p_invalid, rows, view = cfg
    case = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype="bf16",
                                      seed=T * 7 + k + E + rows, routing=routing,
                                      p_invalid=p_invalid, experts="random")
    b, e = view if view else (0, E)
    _ll_dispatch_compare(case, rows, b, e)


def test_dispatch_lowlatency_equals_two_calls():
    """Same rows, scales, counts and sources as ep_dispatch_layout + ep_permute_lowlatency."""
    case = _bf16_decode_case(T=128, seed=3100)
    dev = torch.device("cuda")
    topk, x = case.topk_idx.to(dev), case.x.to(dev)
    ws1 = epd.new_workspace(case.T, case.k, case.E, case.R, case.N, dev)
    ws2 = epd.new_workspace(case.T, case.k, case.E, case.R, case.N, dev)
    st = epd.new_status(dev)
    a = epd.ep_dispatch_lowlatency(x, topk, case.E, case.R, case.N, 128, ws1, st)
    epd.ep_dispatch_layout(topk, case.E, case.R, case.N, ws2, st)
    b = epd.ep_permute_lowlatency(x, topk, case.E, 128, ws2, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    oi = a[3].cpu().numpy()
    used = oi[oi >= 0]
    qa = a[0].view(torch.uint8).reshape(-1, case.H)
    qb = b[0].view(torch.uint8).reshape(-1, case.H)
    assert torch.equal(qa[used], qb[used])
    for e in range(case.E):
        n = int(a[2][e])
        assert torch.equal(a[1][e, :, :n], b[1][e, :, :n])
        assert torch.equal(a[4][e, :n], b[4][e, :n])


def test_dispatch_lowlatency_reports_invalid_ids():
    case = _bf16_decode_case(T=64, seed=3101)
    bad = case.topk_idx.clone()
    bad[5, 3] = 256
    bad[60, 0] = -7
    dev = torch.device("cuda")
    ws = epd.new_workspace(case.T, case.k, case.E, case.R, case.N, dev)
    st = epd.new_status(dev)
    epd.ep_dispatch_lowlatency(case.x.to(dev), bad.to(dev), case.E, case.R, case.N, 64, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == epd.EPD_ERR_INVALID_EXPERT
