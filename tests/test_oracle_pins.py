"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest
import torch

import oracle
from oracle_pins import (check_against_sort, check_bf16_rounding, check_bruteforce,
                         check_combine_exact_sums, check_combine_identity, check_combine_one_hot,
                         check_hand_example, check_hand_example_aligned, check_invariants)
from unpermute_ep_dispatch_gb300 import workloads


def test_hand_example():
    """16 experts as 8 ranks x 2, 2 nodes, top-2 (the pages' worked setting)."""
    check_hand_example(oracle)


@pytest.mark.parametrize("T,k,E,R,N", [
    (3, 2, 4, 1, 1), (3, 2, 4, 2, 1), (3, 2, 4, 4, 2), (2, 2, 3, 3, 1),
    (1, 4, 4, 2, 2), (5, 1, 4, 4, 4),
])
def test_bruteforce_tiny(T, k, E, R, N):
    """Every topk_idx over {-1..E-1} (repeats included) against a sort-based definition."""
    n = check_bruteforce(oracle, T, k, E, R, N)
    assert n == (E + 1) ** (T * k)


@pytest.mark.parametrize("seed", range(6))
def test_sort_definition_random(seed):
    rng = np.random.default_rng(seed)
    T = int(rng.integers(1, 60))
    k = int(rng.integers(1, 9))
    R = int(rng.choice([1, 2, 4, 8]))
    E = R * int(rng.integers(1, 5))
    N = int(rng.choice([d for d in (1, 2, 4) if R % d == 0]))
    topk = rng.integers(-1, E, size=(T, k)).astype(np.int64)
    check_against_sort(oracle, topk, E, R, N)


@pytest.mark.parametrize("name,T", [("tiny", None), ("prefill_bf16", 300), ("dsv3_fp8", 200),
                                    ("skew_bf16", 500), ("decode_fp8", None)])
def test_invariants_workloads(name, T):
    cfg = workloads.CONFIGS[name]
    c = workloads.make_case(name, T=T, experts="random") if cfg["dtype"] == "fp8" or T else \
        workloads.make_case(name)
    check_invariants(oracle, c.topk_idx.numpy(), c.E, c.R, c.N)


@pytest.mark.parametrize("p_invalid", [0.0, 0.5, 1.0])
def test_invariants_invalid_density(p_invalid):
    rng = np.random.default_rng(int(p_invalid * 10))
    topk = rng.integers(0, 32, size=(97, 6)).astype(np.int64)
    topk[rng.random(topk.shape) < p_invalid] = -1
    check_invariants(oracle, topk, 32, 8, 2)


def test_invariants_larger_capacity():
    rng = np.random.default_rng(11)
    topk = rng.integers(-1, 16, size=(33, 3)).astype(np.int64)
    check_invariants(oracle, topk, 16, 4, 2, capacity=33 * 3 + 40)


def test_degenerate_sizes():
    empty = np.zeros((0, 4), np.int64)
    lay = oracle.dispatch_layout(empty, 8, 4, 2)
    assert lay["tokens_per_expert"].sum() == 0 and lay["tokens_per_rank"].sum() == 0
    start, total = oracle.scan_offsets(lay["tokens_per_expert"])
    assert total == 0 and np.all(start == 0)
    kzero = np.zeros((5, 0), np.int64)
    lay = oracle.dispatch_layout(kzero, 8, 4, 2)
    assert lay["is_token_in_rank"].sum() == 0
    y = oracle.unpermute(np.zeros((0, 16), np.uint16), np.zeros((5, 0), np.int32),
                         np.zeros((5, 0), np.float32))
    assert y.shape == (5, 16) and np.all(y == 0)


def test_rejects_bad_inputs():
    with pytest.raises(oracle.OracleError):
        oracle.dispatch_layout(np.array([[0, 8]], np.int64), 8, 4, 1)       # id == E
    with pytest.raises(oracle.OracleError):
        oracle.dispatch_layout(np.array([[0, -2]], np.int64), 8, 4, 1)      # id < -1
    with pytest.raises(oracle.OracleError):
        oracle.dispatch_layout(np.array([[0, 1]], np.int64), 8, 3, 1)       # E % R
    topk = np.array([[0, 1], [0, 1]], np.int64)
    start = np.array([0, 2] + [4] * 6, np.int32)
    with pytest.raises(oracle.OracleError):                                  # capacity short
        oracle.permute(np.zeros((2, 16), np.uint8), None, topk, 8, start, 3)


def test_combine_identity_experts():
    check_combine_identity(oracle)


def test_combine_one_hot():
    check_combine_one_hot(oracle)


def test_combine_exact_sums_and_ties():
    check_combine_exact_sums(oracle)


def test_bf16_rounding_matches_torch():
    check_bf16_rounding(oracle)


def test_combine_identity_on_prefill_shape():
    """Identity experts on a prefill-shaped slice (2% dropped picks, softmax over
    the rest): y == x for every token with a pick."""
    c = workloads.make_case("prefill_bf16", T=256)
    xb = c.x.view(torch.int16).numpy().view(np.uint16)
    res = oracle.run_path(xb.view(np.uint8), None, c.topk_idx.numpy(), c.topk_weights.numpy(),
                          c.E, c.R, c.N)
    has = (c.topk_idx >= 0).any(dim=1).numpy()
    assert np.array_equal(res["y"][has], xb[has])
    assert np.all(res["y"][~has] == 0)


# ----------------------------------------------------------------------------- expert alignment
def test_hand_example_aligned():
    """The worked routing with every expert padded to a multiple of 4."""
    check_hand_example_aligned(oracle)


@pytest.mark.parametrize("T,k,E,R,N,alignment", [
    (3, 2, 4, 2, 1, 2), (3, 2, 4, 4, 2, 4), (2, 2, 3, 3, 1, 3), (1, 4, 4, 2, 2, 8),
])
def test_bruteforce_tiny_aligned(T, k, E, R, N, alignment):
    n = check_bruteforce(oracle, T, k, E, R, N, alignment=alignment)
    assert n == (E + 1) ** (T * k)


@pytest.mark.parametrize("alignment", [2, 16, 128, 256])
def test_invariants_aligned(alignment):
    c = workloads.make_case("dsv3_fp8", T=300)
    check_invariants(oracle, c.topk_idx.numpy(), c.E, c.R, c.N, alignment=alignment)
    rng = np.random.default_rng(alignment)
    topk = rng.integers(-1, 16, size=(77, 5)).astype(np.int64)
    check_invariants(oracle, topk, 16, 4, 2, alignment=alignment)


def test_alignment_one_is_the_plain_scan():
    rng = np.random.default_rng(3)
    cnt = rng.integers(0, 50, size=64).astype(np.int32)
    a, ta = oracle.scan_offsets_aligned(cnt, 1)
    b, tb = oracle.scan_offsets(cnt)
    assert a.tolist() == b.tolist() and ta == tb


# ----------------------------------------------------------------------------- views and scale layouts
from oracle_pins import (check_hand_example_rank3, check_view_against_reference,  # noqa: E402
                         check_views_tile_the_buffer)


def test_hand_example_rank3():
    """The worked routing seen from simulated rank 3 (experts 6 and 7, local ids 0, 1)."""
    check_hand_example_rank3(oracle)


@pytest.mark.parametrize("b,e_end,alignment,col_major", [
    (0, 4, 1, False), (1, 3, 1, True), (2, 4, 2, False), (0, 2, 4, True), (3, 4, 1, True),
])
def test_views_bruteforce(b, e_end, alignment, col_major):
    import itertools
    for n, flat in enumerate(itertools.product(range(-1, 4), repeat=6)):
        if n % 3:
            continue
        topk = np.array(flat, np.int64).reshape(3, 2)
        check_view_against_reference(oracle, topk, 4, b, e_end, alignment, col_major, seed=n)


@pytest.mark.parametrize("alignment", [1, 8, 128])
def test_views_tile_the_buffer(alignment):
    c = workloads.make_case("dsv3_fp8", T=200)
    check_views_tile_the_buffer(oracle, c.topk_idx.numpy(), c.E, c.R, alignment)


def test_views_on_workload_shapes():
    c = workloads.make_case("skew_bf16", T=300, experts="identity")
    for b, e in [(0, 8), (64, 72), (248, 256)]:
        check_view_against_reference(oracle, c.topk_idx.numpy(), c.E, b, e, 1, True)


# ----------------------------------------------------------------------------- low-latency layout
from oracle_pins import (check_e4m3_rounding, check_lowlatency_against_exact_layout,  # noqa: E402
                         check_lowlatency_cast_exact, check_lowlatency_hand)


def test_e4m3_rounding_matches_torch():
    check_e4m3_rounding(oracle)


def test_lowlatency_hand_example():
    check_lowlatency_hand(oracle)


def test_lowlatency_cast_exact_values():
    check_lowlatency_cast_exact(oracle)


@pytest.mark.parametrize("rows,b,e_end", [(64, 0, None), (3, 0, None), (40, 8, 16), (1, 4, 6)])
def test_lowlatency_against_exact_layout(rows, b, e_end):
    c = workloads.make_case("decode_fp8", seed=1001)
    topk = c.topk_idx.numpy()
    E = 32
    topk = np.where(topk >= 0, topk % E, -1)
    check_lowlatency_against_exact_layout(oracle, topk, E, rows, b, e_end, seed=rows)
