"""Checks that pin the CPU oracle to what the pages and the mathematics fix.

Each ``check_*`` function takes the oracle module as an argument so that the
same checks can be run against deliberately broken copies of the oracle (see
``test_oracle_mutants.py``). None of them re-types the oracle's formulas: the
expected values come from the hand-worked example in ``tests/golden``, from an
independent definition (a sort of the (expert, token, slot) pairs), from
invariants, from closed forms of the combine, or from torch's own bf16
rounding.
"""
from __future__ import annotations

import itertools
import json
import os
from collections import Counter
from fractions import Fraction

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name="hand_example.json"):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def token_id_rows(T, row_bytes=16):
    """Rows whose bytes spell the token index, so a permuted row names its source."""
    rows = np.zeros((T, row_bytes), np.uint8)
    for t in range(T):
        rows[t, :4] = np.frombuffer(np.int32(t).tobytes(), np.uint8)
        rows[t, 4:] = (t * 7 + np.arange(row_bytes - 4)) % 251
    return rows


def rows_to_token_ids(rows):
    return [int(np.frombuffer(r[:4].tobytes(), np.int32)[0]) for r in rows]


# ----------------------------------------------------------------------------- hand example
def check_hand_example(orc):
    g = load_golden()
    topk = np.array(g["topk_idx"], np.int64)
    E, R, N, k = g["E"], g["R"], g["N"], g["k"]
    T = topk.shape[0]
    lay = orc.dispatch_layout(topk, E, R, N)
    assert lay["tokens_per_expert"].tolist() == g["tokens_per_expert"]
    assert lay["tokens_per_rank"].tolist() == g["tokens_per_rank"]
    assert lay["tokens_per_rdma_rank"].tolist() == g["tokens_per_rdma_rank"]
    sets = [sorted(np.nonzero(row)[0].tolist()) for row in lay["is_token_in_rank"]]
    assert sets == g["is_token_in_rank_sets"]
    start, total = orc.scan_offsets(lay["tokens_per_expert"])
    assert start.tolist() == g["expert_start_loc"]
    assert total == g["total_rows"]
    x = token_id_rows(T)
    per = orc.permute(x, None, topk, E, start, T * k)
    assert per["output_index"].tolist() == g["output_index"]
    assert per["m_indices"].tolist() == g["m_indices"]
    assert rows_to_token_ids(per["out"][:total]) == g["permuted_source_tokens"]


def check_hand_example_aligned(orc):
    g = load_golden("hand_example_aligned4.json")
    topk = np.array(g["topk_idx"], np.int64)
    T = topk.shape[0]
    lay = orc.dispatch_layout(topk, g["E"], g["R"], g["N"])
    start, total = orc.scan_offsets_aligned(lay["tokens_per_expert"], g["alignment"])
    assert start.tolist() == g["expert_start_loc"]
    assert total == g["total_rows"]
    assert orc.aligned_capacity(T, g["k"], g["E"], g["alignment"]) == g["capacity"]
    per = orc.permute(token_id_rows(T), None, topk, g["E"], start, g["capacity"])
    assert per["output_index"].tolist() == g["output_index"]
    mi = per["m_indices"]
    assert mi[:20].tolist() == g["m_indices_first_20"]
    assert np.all(mi[20:] == -1)
    src = rows_to_token_ids(per["out"])
    for row, tok in g["permuted_source_tokens_by_row"].items():
        assert src[int(row)] == tok


# ----------------------------------------------------------------------------- independent definition
def reference_by_sort(topk, E, R, N, alignment=1, capacity=None):
    """Layout and slots from an independent formulation: sort all valid pairs by
    (expert, token, slot); walking the sorted list, an expert's first pair opens a
    region at the next multiple of the alignment, and the buffer is read off."""
    T, k = topk.shape
    pairs = [(int(topk[t, j]), t, j) for t in range(T) for j in range(k) if topk[t, j] >= 0]
    order = sorted(pairs)
    cnt = Counter(e for (e, _, _) in order)
    counts = [cnt.get(e, 0) for e in range(E)]
    if capacity is None:
        capacity = T * k
    slot, m_indices, row, prev = {}, [-1] * capacity, 0, None
    for (e, t, j) in order:
        if e != prev:
            row = -(-row // alignment) * alignment      # next region starts aligned
            prev = e
        slot[(t, j)] = row
        m_indices[row] = e
        row += 1
    output_index = [[slot.get((t, j), -1) for j in range(k)] for t in range(T)]
    start = []
    acc = 0
    for e in range(E):
        start.append(acc)
        acc += -(-counts[e] // alignment) * alignment
    total_aligned = acc
    epr = E // R
    rpn = R // N
    token_ranks = [{int(e) // epr for e in topk[t] if e >= 0} for t in range(T)]
    token_nodes = [{r // rpn for r in rs} for rs in token_ranks]
    per_rank = [sum(r in rs for rs in token_ranks) for r in range(R)]
    per_node = [sum(n in ns for ns in token_nodes) for n in range(N)]
    return dict(output_index=output_index, m_indices=m_indices, counts=counts, start=start,
                per_rank=per_rank, per_node=per_node, token_ranks=token_ranks,
                total=len(order) if alignment == 1 else total_aligned, slot=slot)


def check_against_sort(orc, topk, E, R, N, alignment=1):
    T, k = topk.shape
    cap = T * k if alignment == 1 else orc.aligned_capacity(T, k, E, alignment)
    ref = reference_by_sort(topk, E, R, N, alignment, cap)
    lay = orc.dispatch_layout(topk, E, R, N)
    assert lay["tokens_per_expert"].tolist() == ref["counts"], "counts"
    assert lay["tokens_per_rank"].tolist() == ref["per_rank"], "per_rank"
    assert lay["tokens_per_rdma_rank"].tolist() == ref["per_node"], "per_node"
    sets = [set(np.nonzero(row)[0].tolist()) for row in lay["is_token_in_rank"]]
    assert sets == ref["token_ranks"], "is_token_in_rank"
    if alignment == 1:
        start, total = orc.scan_offsets(lay["tokens_per_expert"])
    else:
        start, total = orc.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    assert start.tolist() == ref["start"], "start"
    assert total == ref["total"], "total"
    x = token_id_rows(T)
    per = orc.permute(x, None, topk, E, start, cap)
    assert per["output_index"].tolist() == ref["output_index"], "output_index"
    assert per["m_indices"].tolist() == ref["m_indices"], "m_indices"
    src = rows_to_token_ids(per["out"])
    for (t, j), row in ref["slot"].items():
        assert src[row] == t, "permuted row source"


def check_bruteforce(orc, T, k, E, R, N, limit=None, alignment=1):
    """Every topk_idx in {-1..E-1}^(T x k) (with repeats) against the sort definition."""
    n = 0
    for flat in itertools.product(range(-1, E), repeat=T * k):
        check_against_sort(orc, np.array(flat, np.int64).reshape(T, k), E, R, N, alignment)
        n += 1
        if limit is not None and n >= limit:
            break
    return n


# ----------------------------------------------------------------------------- invariants
def check_invariants(orc, topk, E, R, N, row_bytes=32, with_scale=True, capacity=None,
                     alignment=1):
    T, k = topk.shape
    if capacity is None:
        capacity = T * k if alignment == 1 else orc.aligned_capacity(T, k, E, alignment)
    valid = topk >= 0
    P = int(valid.sum())
    lay = orc.dispatch_layout(topk, E, R, N)
    cnt = lay["tokens_per_expert"].astype(np.int64)
    assert cnt.sum() == P                                    # counts sum to the valid picks
    if alignment == 1:
        start, total = orc.scan_offsets(lay["tokens_per_expert"])
        assert total == P
        padded = cnt
    else:
        start, total = orc.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
        padded = -(-cnt // alignment) * alignment
        assert np.all(start % alignment == 0)                # regions start aligned
        assert total <= capacity                             # compute_aligned_M bound holds
        assert total == padded.sum()
    if E > 0:
        assert start[0] == 0
        assert np.all(np.diff(start.astype(np.int64)) == padded[:-1])  # regions tile [0, total)
        assert int(start[-1]) + int(padded[-1]) == total
    rng = np.random.default_rng(T * 131 + k)
    x = rng.integers(0, 256, size=(T, row_bytes), dtype=np.uint8)
    sc = rng.standard_normal((T, 3)).astype(np.float32) if with_scale else None
    per = orc.permute(x, sc, topk, E, start, capacity)
    oi = per["output_index"]
    mi = per["m_indices"]
    assert np.all(oi[~valid] == -1)
    slots = oi[valid]
    filled = np.concatenate([np.arange(start[e], start[e] + cnt[e]) for e in range(E)]) \
        if E else np.zeros(0, np.int64)
    assert sorted(slots.tolist()) == sorted(filled.tolist())  # bijection onto the filled rows
    assert np.all(mi[slots] == topk[valid])                  # row -> expert
    empty = np.ones(capacity, bool)
    empty[slots] = False
    assert np.all(mi[empty] == -1)                           # padding and tail rows
    assert np.array_equal(per["out"][slots], np.repeat(x, k, axis=0)[valid.reshape(-1)])
    if with_scale:
        assert np.array_equal(per["out_scale"][slots], np.repeat(sc, k, axis=0)[valid.reshape(-1)])
    # slots grow with (t, j) inside each expert
    for e in np.unique(topk[valid]):
        s_e = oi[topk == e]            # row-major order of (t, j)
        assert np.all(np.diff(s_e) > 0)
        assert s_e[0] == start[e]
    per_rank = lay["tokens_per_rank"].astype(np.int64)
    in_rank = lay["is_token_in_rank"]
    assert np.array_equal(in_rank.sum(axis=0), per_rank)
    epr, rpn = E // R, R // N
    per_node = lay["tokens_per_rdma_rank"].astype(np.int64)
    for r in range(R):
        assert per_rank[r] <= cnt[r * epr:(r + 1) * epr].sum()
    for n in range(N):
        block = per_rank[n * rpn:(n + 1) * rpn]
        assert block.sum() >= per_node[n] >= (block.max() if block.size else 0)
        assert per_node[n] <= T
    return lay, start, per


# ----------------------------------------------------------------------------- combine
def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def check_combine_identity(orc, T=40, H=64, k=4, E=8, p_invalid=0.3, seed=5):
    """Identity experts and weights summing to 1: y equals x bit for bit, and a
    token whose picks were all dropped gives +0."""
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    topk = torch.argsort(-logits, dim=1, stable=True)[:, :k]
    valid = torch.rand(T, k, generator=g) >= p_invalid
    valid[0] = False                                  # one token with no pick at all
    topk = torch.where(valid, topk, torch.full_like(topk, -1)).numpy().astype(np.int64)
    picked = torch.gather(logits, 1, torch.as_tensor(np.maximum(topk, 0)))
    w = torch.softmax(picked.masked_fill(~valid, float("-inf")), dim=1)
    w = torch.nan_to_num(w, nan=0.0).float().numpy()
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    xb = bf16_bits(x)
    res = orc.run_path(xb.view(np.uint8), None, topk, w, E, 1, 1)
    y = res["y"]
    has = valid.numpy().any(axis=1)
    assert np.array_equal(y[has], xb[has])
    assert np.all(y[~has] == 0)


def check_combine_one_hot(orc, T=24, H=32, k=3, E=6, seed=9):
    """One weight 1, the others 0: y is the selected expert-output row exactly."""
    rng = np.random.default_rng(seed)
    topk = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int64)
    hot = rng.integers(0, k, size=T)
    w = np.zeros((T, k), np.float32)
    w[np.arange(T), hot] = 1.0
    x = np.zeros((T, 2 * H), np.uint8)
    lay = orc.dispatch_layout(topk, E, 1, 1)
    start, _ = orc.scan_offsets(lay["tokens_per_expert"])
    per = orc.permute(x, None, topk, E, start, T * k)
    eo = bf16_bits(torch.randn(T * k, H, generator=torch.Generator().manual_seed(seed))
                   .to(torch.bfloat16))
    y = orc.unpermute(eo, per["output_index"], w)
    sel = per["output_index"][np.arange(T), hot]
    assert np.array_equal(y, eo[sel])


def _bf16_of_fraction(q: Fraction) -> int:
    """Round an exact rational to bf16 with torch's float32 -> bf16 conversion.
    Only used where q is exactly representable in float32, so the one rounding
    is torch's."""
    f = np.float32(float(q))
    assert Fraction(float(f)) == q
    return int(bf16_bits(torch.tensor([f]).to(torch.bfloat16))[0])


def _bf16_bits_of(v: float) -> int:
    return int(bf16_bits(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16))[0])


def check_combine_exact_sums(orc):
    """Dyadic weights and values: the exact weighted sum is known as a fraction;
    it includes bf16 round-to-nearest-even ties in both directions, cancellation
    to zero, and a sign change."""
    one = 1.0
    cases = [
        # (values (bf16-exact), weights) -> exact sum
        ([1.0, 2.0 ** -8], [1.0, 1.0]),                 # 1 + 2^-8: tie -> even (1.0)
        ([1.0, 3 * 2.0 ** -8], [1.0, 1.0]),             # 1 + 3*2^-8: tie -> even (1 + 2^-6)
        ([1.0, 2.0 ** -8], [1.0, 1.5]),                 # above the tie -> up
        ([3.0, -1.5], [0.5, 1.0]),                      # 1.5 - 1.5 = 0
        ([2.0, -3.0], [0.25, 0.5]),                     # 0.5 - 1.5 = -1
        ([0.75, 0.125, -0.0625], [0.5, 0.25, 2.0]),     # 0.375 + 0.03125 - 0.125
        ([one] * 8, [0.125] * 8),                       # eight eighths
        ([float(2 ** 120), float(2 ** 120)], [1.0, 1.0]),   # large magnitude
    ]
    for vals, ws in cases:
        k = len(vals)
        eo = np.array([[_bf16_bits_of(v)] for v in vals], np.uint16)      # [k, 1]
        oi = np.arange(k, dtype=np.int32).reshape(1, k)
        w = np.array([ws], np.float32)
        y = orc.unpermute(eo, oi, w)
        exact = sum(Fraction(wv) * Fraction(v) for wv, v in zip(ws, vals))
        assert int(y[0, 0]) == _bf16_of_fraction(exact), (vals, ws)
    # the order and sign of terms matter: w * x with x negative
    eo = np.array([[_bf16_bits_of(-2.5)], [_bf16_bits_of(1.25)]], np.uint16)
    y = orc.unpermute(eo, np.array([[1, 0]], np.int32), np.array([[2.0, 0.5]], np.float32))
    assert int(y[0, 0]) == _bf16_bits_of(2.0 * 1.25 + 0.5 * -2.5)


def check_bf16_rounding(orc, n=20000, seed=3):
    """The oracle's bf16 rounding against torch's float32 -> bf16 conversion."""
    rng = np.random.default_rng(seed)
    mant = rng.integers(0, 1 << 23, size=n, dtype=np.int64)
    expo = rng.integers(0, 255, size=n, dtype=np.int64)        # incl. subnormals, no inf/nan
    sign = rng.integers(0, 2, size=n, dtype=np.int64)
    bits = ((sign << 31) | (expo << 23) | mant).astype(np.uint32)
    # force exact ties and near-ties on a quarter of them
    tie = (bits & ~np.uint32(0xFFFF)) | np.uint32(0x8000)
    bits[: n // 4] = tie[: n // 4]
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    want = bf16_bits(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = np.array([orc.bf16_from_double(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, want)
    # every finite bf16 pattern survives a round trip through double
    for b in range(0, 1 << 16, 97):
        if (b & 0x7F80) == 0x7F80:
            continue
        assert orc.bf16_from_double(orc.double_from_bf16(b)) == b


def check_combine_all(orc):
    check_combine_identity(orc)
    check_combine_one_hot(orc)
    check_combine_exact_sums(orc)


# ----------------------------------------------------------------------------- views and scale layouts
def check_hand_example_rank3(orc):
    g = load_golden("hand_example_rank3.json")
    topk = np.array(g["topk_idx"], np.int64)
    T = topk.shape[0]
    lay = orc.dispatch_layout(topk, g["E"], g["R"], g["N"])
    start, _ = orc.scan_offsets(lay["tokens_per_expert"])
    r = orc.permute_ex(token_id_rows(T), None, topk, g["E"], start, g["capacity"],
                       expert_begin=g["expert_begin"], expert_end=g["expert_end"])
    assert r["output_index"].tolist() == g["output_index"]
    assert r["m_indices"].tolist() == g["m_indices"]
    n = len(g["permuted_source_tokens"])
    assert rows_to_token_ids(r["out"][:n]) == g["permuted_source_tokens"]


def reference_view(topk, E, b, e_end, alignment=1, scale_words=None, capacity=None):
    """Independent definition of one view: counts by Counter, offsets by numpy's
    cumulative sum of the (padded) counts, slots by sorting the view's pairs by
    (expert, token, slot); scale rows placed by numpy indexing."""
    T, k = topk.shape
    pairs = [(int(topk[t, j]), t, j) for t in range(T) for j in range(k) if topk[t, j] >= 0]
    cnt = Counter(e for (e, _, _) in pairs)
    counts = np.array([cnt.get(e, 0) for e in range(E)], np.int64)
    padded = -(-counts // alignment) * alignment
    start = np.concatenate([[0], np.cumsum(padded)[:-1]]).astype(np.int64)
    base = start[b]
    if capacity is None:
        capacity = T * k
    oi = -np.ones((T, k), np.int64)
    mi = -np.ones(capacity, np.int64)
    seen = Counter()
    for (e, t, j) in sorted(p for p in pairs if b <= p[0] < e_end):
        s = start[e] - base + seen[e]
        seen[e] += 1
        oi[t, j] = s
        mi[s] = e - b
    res = dict(output_index=oi, m_indices=mi, start=start)
    if scale_words is not None:
        C = scale_words.shape[1]
        rm = np.zeros((capacity, C), np.uint32)
        valid = oi >= 0
        rows = oi[valid]
        toks = np.nonzero(valid)[0]
        rm[rows] = scale_words[toks]
        res["scale_row_major"] = rm
    return res


def check_view_against_reference(orc, topk, E, b, e_end, alignment=1, col_major=False, seed=0):
    T, k = topk.shape
    cap = T * k if alignment == 1 else orc.aligned_capacity(T, k, E, alignment)
    rng = np.random.default_rng(seed)
    words = rng.integers(0, 2 ** 32, size=(T, 5), dtype=np.uint64).astype(np.uint32)
    ref = reference_view(topk, E, b, e_end, alignment, words, cap)
    lay = orc.dispatch_layout(topk, E, 1, 1)
    if alignment == 1:
        start, _ = orc.scan_offsets(lay["tokens_per_expert"])
    else:
        start, _ = orc.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    assert start.tolist() == ref["start"].tolist()
    ld = cap + 12 if col_major else None
    x = token_id_rows(T)
    r = orc.permute_ex(x, words, topk, E, start, cap, expert_begin=b, expert_end=e_end,
                       scale_col_major=col_major, scale_ld=ld)
    assert r["output_index"].tolist() == ref["output_index"].tolist(), "output_index"
    assert r["m_indices"].tolist() == ref["m_indices"].tolist(), "m_indices"
    valid = ref["output_index"] >= 0
    rows = ref["output_index"][valid]
    assert rows_to_token_ids(r["out"][rows]) == np.nonzero(valid)[0].tolist(), "rows"
    if col_major:
        got = r["out_scale"][:, :cap].T          # [C, ld] column-major -> [cap, C]
    else:
        got = r["out_scale"]
    assert np.array_equal(got[rows], ref["scale_row_major"][rows]), "scales"


def check_views_tile_the_buffer(orc, topk, E, R, alignment=1):
    """The per-rank views, placed at their region offsets, rebuild the whole buffer."""
    T, k = topk.shape
    cap = T * k if alignment == 1 else orc.aligned_capacity(T, k, E, alignment)
    lay = orc.dispatch_layout(topk, E, R, 1)
    if alignment == 1:
        start, total = orc.scan_offsets(lay["tokens_per_expert"])
    else:
        start, total = orc.scan_offsets_aligned(lay["tokens_per_expert"], alignment)
    x = token_id_rows(T)
    full = orc.permute(x, None, topk, E, start, cap)
    epr = E // R
    oi_all = -np.ones((T, k), np.int64)
    for r in range(R):
        b, e_end = r * epr, (r + 1) * epr
        v = orc.permute_ex(x, None, topk, E, start, cap, expert_begin=b, expert_end=e_end)
        base = int(start[b])
        end = int(start[e_end]) if e_end < E else total
        n = end - base
        mi = v["m_indices"][:n]
        want = full["m_indices"][base:end]
        assert np.array_equal(np.where(mi >= 0, mi + b, -1), want)
        assert np.all(v["m_indices"][n:] == -1)
        sel = v["output_index"] >= 0
        oi_all[sel] = v["output_index"][sel] + base
        rows = v["output_index"][sel]
        assert np.array_equal(v["out"][rows], full["out"][rows + base])
    assert np.array_equal(oi_all, full["output_index"])


# ----------------------------------------------------------------------------- low-latency layout
def check_e4m3_rounding(orc, n=20000, seed=4):
    """The oracle's e4m3 rounding against torch's float32 -> float8_e4m3fn conversion,
    inside the finite range (torch does not saturate; the oracle clamps to 448)."""
    rng = np.random.default_rng(seed)
    v = np.concatenate([rng.uniform(-448, 448, n // 2),
                        rng.standard_normal(n // 4) * 3,
                        rng.uniform(-2 ** -6, 2 ** -6, n // 4)]).astype(np.float32)
    # exact midpoints between neighbouring e4m3 values (ties) of every binade
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = ((grid[:-1].astype(np.float64) + grid[1:]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, grid, -grid])
    want = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_from_float(float(x)) for x in v], np.uint8)
    assert np.array_equal(got, want)
    assert orc.e4m3_from_float(1e9) == 0x7E and orc.e4m3_from_float(-500.0) == 0xFE  # saturate


def check_lowlatency_hand(orc):
    """[P2] setting (E=16, top-2), rectangles of 2 rows: experts 3 and 7 each take two
    picks, 0, 6 and 15 one; with 1 row per expert the second pick of 3 and of 7 is
    dropped."""
    topk = np.array([[3, 7], [3, -1], [0, 15], [7, 6]], np.int64)
    x = np.zeros((4, 128), np.uint16)
    r = orc.permute_lowlatency(x, topk, 16, 2)
    assert r["output_index"].tolist() == [[6, 14], [7, -1], [0, 30], [15, 12]]
    assert r["recv_count"].tolist() == [1, 0, 0, 2, 0, 0, 1, 2, 0, 0, 0, 0, 0, 0, 0, 1]
    assert r["src_token"][3].tolist() == [0, 1] and r["src_token"][7].tolist() == [0, 3]
    assert not r["overflow"]
    r1 = orc.permute_lowlatency(x, topk, 16, 1)
    assert r1["output_index"].tolist() == [[3, 7], [-1, -1], [0, 15], [-1, 6]]
    assert r1["overflow"]
    v = orc.permute_lowlatency(x, topk, 16, 2, expert_begin=6, expert_end=8)  # rank 3's view
    assert v["output_index"].tolist() == [[-1, 2], [-1, -1], [-1, -1], [3, 0]]
    assert v["recv_count"].tolist() == [1, 2]


def check_lowlatency_cast_exact(orc):
    """A block with amax 7 has scale 7/448 = 2^-6 exactly, so q = e4m3(64 x): values
    whose 64x is an e4m3 value come back exactly; the amax maps to 448."""
    vals = np.array([7.0, -7.0, 1.0, 0.5, -0.25, 3.5, 0.0, 2 ** -9], np.float32)
    row = np.resize(vals, 256).astype(np.float32)
    row[128:] = row[128:] * 0.5                         # second block: amax 3.5 -> 2^-7
    xb = bf16_bits(torch.from_numpy(row).to(torch.bfloat16)).reshape(1, 256)
    r = orc.permute_lowlatency(xb, np.array([[0]], np.int64), 1, 1)
    assert r["out_scale"][0, :, 0].tolist() == [2.0 ** -6, 2.0 ** -7]
    q = torch.from_numpy(r["out_q"][0, 0].copy()).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(q[:128], np.resize(vals * 64, 128).astype(np.float32).clip(-448, 448))
    assert np.array_equal(q[128:], np.resize(vals * 64, 128).astype(np.float32).clip(-448, 448))
    assert abs(q).max() == 448.0


def check_lowlatency_against_exact_layout(orc, topk, E, rows, b=0, e_end=None, seed=0):
    """Rectangle rows are the exact layout's rows shifted to fixed per-expert bases:
    the r-th pick of expert e (token-major) sits at (e - b) * rows + r; the cast
    dequantises to within e4m3's spacing."""
    T, k = topk.shape
    e_end = E if e_end is None else e_end
    rng = np.random.default_rng(seed)
    H = 256
    xf = (rng.standard_normal((T, H)) * rng.uniform(0.01, 10, size=(T, 1))).astype(np.float32)
    xb = bf16_bits(torch.from_numpy(xf).to(torch.bfloat16))
    r = orc.permute_lowlatency(xb, topk, E, rows, b, e_end)
    seen = Counter()
    overflow = False
    for t in range(T):
        for j in range(k):
            e = int(topk[t, j])
            if not (b <= e < e_end):
                assert r["output_index"][t, j] == -1
                continue
            rank = seen[e]
            seen[e] += 1
            if rank >= rows:
                overflow = True
                assert r["output_index"][t, j] == -1
                continue
            row = (e - b) * rows + rank
            assert r["output_index"][t, j] == row
            assert r["src_token"].reshape(-1)[row] == t
            xs = (xb[t].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            q = torch.from_numpy(r["out_q"].reshape(-1, H)[row].copy()).view(
                torch.float8_e4m3fn).double().numpy()
            sc = r["out_scale"][e - b, :, rank].astype(np.float64)
            deq = q * np.repeat(sc, 128)
            tol = np.maximum(np.abs(xs) * 2.0 ** -4, np.repeat(sc, 128) * 2.0 ** -9) * 1.0001
            assert np.all(np.abs(deq - xs) <= tol)
    assert r["overflow"] == overflow
    assert r["recv_count"].tolist() == [min(seen[e], rows) for e in range(b, e_end)]
