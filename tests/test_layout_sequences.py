"""Layout calls in sequence on one workspace, on the GPU through the C ABI.

"[MoE] Deepseek的All-to-all通信: DeepEP代码解读", section "Dispatch": every
get_dispatch_layout call computes the layout of its own topk_idx. Here two layout
calls are issued back to back on one stream and one workspace, with different
topk_idx and nothing in between, and each call's outputs are compared element by
element with the oracle -- the counts, masks and offsets, and the second call's
per-pair ranks through the permute that follows it (output_index, m_indices).
Sizes span the cluster form (dsv3: one cluster of 16 blocks), several clusters
(131 072 pairs: their counts meet through global memory) and the tile form with
its ticket and look-back (524 288 pairs: 128 tiles of 4096 pairs).

A second group plants leftovers in the look-back state region of a workspace, or
in the region where several clusters publish their counts (values an earlier call
of another shape, or an earlier call, leaves there) and checks that the next call
ignores them.
"""
import numpy as np
import pytest
import torch

import oracle
import unpermute_ep_dispatch_gb300 as epd
from unpermute_ep_dispatch_gb300 import workloads

pytestmark = pytest.mark.gpu

E, R, N = 256, 32, 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from unpermute_ep_dispatch_gb300 import build
    build.build()
    epd.load_library()


def _case(T, k, seed, routing="uniform"):
    # 16-column bf16 rows (32 bytes): the permute after the layout reads out the ranks
    return workloads.make_random_case(T=T, H=16, k=k, E=E, R=R, N=N, dtype="bf16", seed=seed,
                                      routing=routing, p_invalid=0.05, experts="identity")


class Outs:
    """Device outputs of one layout call (filled with a sentinel first)."""

    def __init__(self, T, dev):
        self.per_e = torch.full((E,), -7, dtype=torch.int32, device=dev)
        self.per_r = torch.full((R,), -7, dtype=torch.int32, device=dev)
        self.per_n = torch.full((N,), -7, dtype=torch.int32, device=dev)
        self.itr = torch.ones(T, R, dtype=torch.bool, device=dev)
        self.start = torch.full((E,), -7, dtype=torch.int32, device=dev)
        self.total = torch.full((1,), -7, dtype=torch.int32, device=dev)


def _launch(kind, topk, ws, st, o):
    if kind == "layout":
        epd.ep_dispatch_layout(topk, E, R, N, ws, st, tokens_per_expert=o.per_e,
                               tokens_per_rank=o.per_r, tokens_per_rdma_rank=o.per_n,
                               is_token_in_rank=o.itr)
    else:
        epd.ep_dispatch_layout_offsets(topk, E, R, N, ws, st, tokens_per_expert=o.per_e,
                                       tokens_per_rank=o.per_r, tokens_per_rdma_rank=o.per_n,
                                       is_token_in_rank=o.itr, expert_start_loc=o.start,
                                       total_rows=o.total)


def _check_layout(kind, case, o, what):
    want = oracle.dispatch_layout(case.topk_idx.numpy(), E, R, N)
    for key, got in (("tokens_per_expert", o.per_e), ("tokens_per_rank", o.per_r),
                     ("tokens_per_rdma_rank", o.per_n), ("is_token_in_rank", o.itr)):
        assert np.array_equal(got.cpu().numpy(), want[key]), f"{what}: {key}"
    if kind == "offsets":
        start, total = oracle.scan_offsets(want["tokens_per_expert"])
        assert np.array_equal(o.start.cpu().numpy(), start), f"{what}: expert_start_loc"
        assert int(o.total.item()) == total, f"{what}: total_rows"
    return want


def _check_ranks(case, ws, st, start, what):
    """ep_permute_ex over the whole expert range after the layout: its slots are
    start[e] + the pair ranks the layout left in the workspace."""
    dev = ws.device
    x = case.x.to(dev)
    topk = case.topk_idx.to(dev)
    out, _, m_idx, out_idx = epd.ep_permute_ex(x, None, topk, E, start, ws, st)
    torch.cuda.synchronize()
    want_start, _ = oracle.scan_offsets(
        oracle.dispatch_layout(case.topk_idx.numpy(), E, R, N)["tokens_per_expert"])
    want = oracle.permute(case.x.view(torch.uint8).numpy().reshape(case.T, -1), None,
                          case.topk_idx.numpy(), E, want_start, case.T * case.k)
    assert np.array_equal(out_idx.cpu().numpy(), want["output_index"]), f"{what}: output_index"
    assert np.array_equal(m_idx.cpu().numpy(), want["m_indices"]), f"{what}: m_indices"


PAIRS = [("layout", "layout"), ("layout", "offsets"), ("offsets", "layout"),
         ("offsets", "offsets")]


@pytest.mark.parametrize("first,second", PAIRS)
@pytest.mark.parametrize("T,k", [(8192, 8), (16384, 8), (65536, 8)])
def test_two_layout_calls_back_to_back(first, second, T, k):
    dev = torch.device("cuda")
    a, b = _case(T, k, seed=T + 1), _case(T, k, seed=T + 2, routing="repeats")
    ws = epd.new_workspace(T, k, E, R, N, dev)
    st = epd.new_status(dev)
    oa, ob = Outs(T, dev), Outs(T, dev)
    ta, tb = a.topk_idx.to(dev), b.topk_idx.to(dev)
    torch.cuda.synchronize()
    for rep in range(3):
        _launch(first, ta, ws, st, oa)
        _launch(second, tb, ws, st, ob)        # issued right behind the first, same workspace
        if second == "layout":
            epd.ep_scan_offsets(ob.per_e, st, expert_start_loc=ob.start, total_rows=ob.total)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"rep {rep}: status {int(st.item())}"
        _check_layout(first, a, oa, f"rep {rep} first call")
        _check_layout("offsets", b, ob, f"rep {rep} second call")
        _check_ranks(b, ws, st, ob.start, f"rep {rep} second call")


def test_many_back_to_back_layouts_then_permute():
    """Twenty layout calls in a row on one workspace, alternating two routings and
    both entry points; only the last call's ranks reach the permute."""
    dev = torch.device("cuda")
    T, k = 16384, 8
    cases = [_case(T, k, seed=31), _case(T, k, seed=32, routing="repeats")]
    tops = [c.topk_idx.to(dev) for c in cases]
    ws = epd.new_workspace(T, k, E, R, N, dev)
    st = epd.new_status(dev)
    outs = [Outs(T, dev) for _ in range(20)]
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        _launch("offsets" if i % 3 else "layout", tops[i % 2], ws, st, o)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for i, o in enumerate(outs):
        _check_layout("offsets" if i % 3 else "layout", cases[i % 2], o, f"call {i}")
    last = outs[-1]
    _check_ranks(cases[1], ws, st, last.start, "last call")


def test_lowlatency_large_path_then_layout():
    """ep_dispatch_lowlatency on a batch beyond its one-kernel form (layout kernel +
    rectangle permute), then a layout of other routing on the same workspace."""
    dev = torch.device("cuda")
    T, k, H = 2048, 8, 128
    ll = workloads.make_random_case(T=T, H=H, k=k, E=E, R=R, N=N, dtype="bf16", seed=41,
                                    routing="uniform", experts="identity")
    b = _case(T, k, seed=42, routing="repeats")
    ws = epd.new_workspace(T, k, E, R, N, dev)
    st = epd.new_status(dev)
    rows = T
    ob = Outs(T, dev)
    x = ll.x.to(dev)
    ta, tb = ll.topk_idx.to(dev), b.topk_idx.to(dev)
    torch.cuda.synchronize()
    q, qs, recv, oi, src = epd.ep_dispatch_lowlatency(x, ta, E, R, N, rows, ws, st)
    _launch("offsets", tb, ws, st, ob)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want_ll = oracle.permute_lowlatency(ll.x.view(torch.int16).numpy().view(np.uint16),
                                        ll.topk_idx.numpy(), E, rows)
    assert np.array_equal(recv.cpu().numpy(), want_ll["recv_count"])
    assert np.array_equal(oi.cpu().numpy(), want_ll["output_index"])
    _check_layout("offsets", b, ob, "layout after the low-latency dispatch")
    _check_ranks(b, ws, st, ob.start, "layout after the low-latency dispatch")


# ----------------------------------------------------------------------------- leftovers
def _tile_tokens(k):
    # tokens per tile of the layout's tile form at E = 256 (32-warp blocks): 4096
    # (token, pick) pairs, at most 2048 tokens
    return max(1, min(2048, 4096 // k)) if k > 0 else 2048


def _state_region(T, k):
    """Byte range of the per-tile look-back state words in a workspace laid out for
    (T, k, E, R, N): after the 256-byte header block, the T*k pair ranks and the E
    counts, each region 256-byte aligned; one 64-bit word per tile."""
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    counts_off = up(256 + T * k * 4)
    state_off = up(counts_off + E * 4)
    tiles = (T + _tile_tokens(k) - 1) // _tile_tokens(k)
    return state_off, tiles


@pytest.mark.parametrize("plant", ["old_small_tags", "previous_call_tags", "minus_one"])
def test_leftover_state_words_are_ignored(plant):
    """A workspace sized for a big layout, a big call first (its pair ranks fill the
    region where the smaller call keeps its state words), then planted leftovers
    over the smaller call's state words, then the smaller many-tile call: its
    counts, offsets and ranks match the oracle."""
    dev = torch.device("cuda")
    # batches beyond one thread-block cluster (more than 131 072 pairs at E = 256): both
    # calls run the tile form, whose look-back reads the state words
    TB, TS = 32768, 20000
    big = _case(TB, 8, seed=51)
    small = _case(TS, 8, seed=52, routing="repeats")
    ws = epd.new_workspace(TB, 8, E, R, N, dev)
    st = epd.new_status(dev)
    ob, os_ = Outs(TB, dev), Outs(TS, dev)
    _launch("offsets", big.topk_idx.to(dev), ws, st, ob)
    torch.cuda.synchronize()
    off, tiles = _state_region(TS, 8)
    assert off + 8 * tiles <= 256 + TB * 8 * 4     # inside the big call's pair ranks
    assert tiles > 1
    words = ws[off: off + 8 * tiles].view(torch.int64)
    epoch = int(ws[8:16].view(torch.int64).item())     # the header's call counter
    if plant == "old_small_tags":      # 32-bit words an untagged scheme would accept
        w32 = ws[off: off + 8 * tiles].view(torch.int32)
        w32.copy_(torch.tensor([5, 6, 9, 10] * (2 * tiles // 4 + 1), dtype=torch.int32)[
            : 2 * tiles])
    elif plant == "previous_call_tags":  # states of the call before, marked and published
        assert epoch >= 1
        prev = (1 << 63) | (((epoch - 1) & ((1 << 61) - 1)) << 2) | 1
        words.fill_(prev - (1 << 64))               # the same 64 bits as a signed value
    else:                               # pair ranks of -1 (no selection) everywhere
        words.fill_(-1)
    _launch("offsets", small.topk_idx.to(dev), ws, st, os_)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws[8:16].view(torch.int64).item()) == epoch + 1   # the tile form ran
    _check_layout("offsets", small, os_, f"after planting {plant}")
    _check_ranks(small, ws, st, os_.start, f"after planting {plant}")


def _cluster_region(T, k):
    """Byte offset of the words several clusters publish their counts in: the tile
    form's aggregate rows, after the state words (256-byte aligned)."""
    up = lambda v: (v + 255) // 256 * 256  # noqa: E731
    state_off, tiles = _state_region(T, k)
    return up(state_off + 8 * tiles)


@pytest.mark.parametrize("plant", ["small_ints", "previous_call_tags", "minus_one"])
def test_leftover_cluster_words_are_ignored(plant):
    """131 072 pairs run as several clusters, whose last blocks publish each
    cluster's counts as self-tagged 64-bit words. Leftovers planted over those words
    between two calls -- small 32-bit values, words tagged with the previous call's
    counter, -1 everywhere -- are not taken for this call's counts."""
    dev = torch.device("cuda")
    T, k = 16384, 8
    a = _case(T, k, seed=61)
    b = _case(T, k, seed=62, routing="repeats")
    ws = epd.new_workspace(T, k, E, R, N, dev)
    st = epd.new_status(dev)
    oa, ob = Outs(T, dev), Outs(T, dev)
    _launch("offsets", a.topk_idx.to(dev), ws, st, oa)
    torch.cuda.synchronize()
    epoch = int(ws[8:16].view(torch.int64).item())
    assert epoch >= 1                                   # the call ran as several clusters
    off = _cluster_region(T, k)
    n = 8 * 320                                          # 8 clusters x padded columns
    words = ws[off: off + 8 * n].view(torch.int64)
    if plant == "small_ints":
        ws[off: off + 8 * n].view(torch.int32).copy_(
            torch.arange(2 * n, dtype=torch.int32, device=dev) % 7 + 1)
    elif plant == "previous_call_tags":
        prev = (1 << 63) | (((epoch - 1) & ((1 << 42) - 1)) << 21) | 12345
        words.fill_(prev - (1 << 64))
    else:
        words.fill_(-1)
    _launch("offsets", b.topk_idx.to(dev), ws, st, ob)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(ws[8:16].view(torch.int64).item()) == epoch + 1
    _check_layout("offsets", a, oa, "first call")
    _check_layout("offsets", b, ob, f"after planting {plant}")
    _check_ranks(b, ws, st, ob.start, f"after planting {plant}")


# ----------------------------------------------------------------------------- the two layout forms
# Batches of up to 16 x 8192 (token, pick) pairs (E <= 1024, <= 2048 tokens per block)
# run the cluster form -- as several clusters where one cluster of 16 blocks would need
# eight chunks per warp -- and larger ones the tile form. Each case below sits on an
# edge of those choices or of the forms themselves, and the whole path is compared
# with the oracle (counts, masks, offsets, slots, rows, combine).
FORM_EDGES = [
    # T, k, E, R, N
    (129, 64, 16, 8, 2),        # 16 blocks; the last one holds no token
    (3000, 8, 640, 64, 8),      # 16 warps per block (E > 512), four chunks per warp
    (2048, 8, 256, 128, 2),     # R > 64: distinct ranks counted by comparing picks
    (1500, 8, 512, 256, 128),   # R and N > 64
    (1000, 6, 90, 9, 3),        # E/R and R/N not powers of two (table look-ups)
    (32768, 1, 256, 32, 4),     # k = 1 at the 2048-token block limit
    (32769, 1, 256, 32, 4),     # one token over it: the tile form
    (16385, 8, 256, 32, 4),     # one token over the cluster's pairs: the tile form
    (1025, 1, 16, 8, 2),        # just over one tile: a cluster of two
    (8200, 8, 256, 32, 4),      # just over 16 x 4096 pairs: several clusters
    (9000, 8, 256, 32, 4),      # several clusters, the last tiles of the last one empty
    (16384, 8, 256, 32, 4),     # several clusters at the cluster form's largest batch
    (4000, 16, 1024, 32, 4),    # several clusters of 16-warp blocks (E > 512)
    (1100, 64, 256, 32, 4),     # several clusters at k = 64 (tiles of 9 tokens)
    (9000, 8, 90, 9, 3),        # several clusters, table look-ups for ranks and nodes
]


@pytest.mark.parametrize("T,k,E,R,N", FORM_EDGES)
@pytest.mark.parametrize("fused", [True, False])
def test_layout_form_edges(T, k, E, R, N, fused):
    from epd_paths import GpuPath, compare, oracle_path
    case = workloads.make_random_case(T=T, H=16, k=k, E=E, R=R, N=N, dtype="bf16",
                                      seed=T + 31 * k + E, routing="repeats", p_invalid=0.1,
                                      experts="random")
    g = GpuPath(case, fused=fused)
    g.step()
    compare(g.results(), oracle_path(case))


@pytest.mark.parametrize("alignment", [4, 128])
def test_several_clusters_with_aligned_offsets(alignment):
    """Several clusters with the fused, per-expert aligned offset scan (padding rows
    at -1 in m_indices): the whole path against the oracle."""
    from epd_paths import GpuPath, compare, oracle_path
    case = workloads.make_random_case(T=12000, H=16, k=8, E=256, R=32, N=4, dtype="bf16",
                                      seed=alignment + 7, routing="repeats", p_invalid=0.05,
                                      experts="random")
    g = GpuPath(case, fused=True, alignment=alignment)
    g.step()
    compare(g.results(), oracle_path(case, alignment=alignment))


def test_several_clusters_without_optional_outputs():
    """Several clusters with no tokens_per_rdma_rank and no is_token_in_rank: the
    counts that are asked for, and the ranks, still match the oracle."""
    dev = torch.device("cuda")
    T, k = 16384, 8
    case = _case(T, k, seed=71, routing="repeats")
    ws = epd.new_workspace(T, k, E, R, N, dev)
    st = epd.new_status(dev)
    per_r, per_n, per_e, itr = epd.ep_dispatch_layout(case.topk_idx.to(dev), E, R, N, ws, st,
                                                      with_rdma=False,
                                                      with_is_token_in_rank=False)
    assert per_n is None and itr is None
    start, _ = epd.ep_scan_offsets(per_e, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = oracle.dispatch_layout(case.topk_idx.numpy(), E, R, N)
    assert np.array_equal(per_e.cpu().numpy(), want["tokens_per_expert"])
    assert np.array_equal(per_r.cpu().numpy(), want["tokens_per_rank"])
    _check_ranks(case, ws, st, start, "no optional outputs")
