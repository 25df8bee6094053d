"""Pins of the oracle's multi-source receive layout (S source ranks, R
destination ranks, one worst-case region of T = S*Ts rows per destination,
rows in (source, token) order).

Expected values come from a hand-derived worked example (tests/golden), a
construction by sorting (r, g) pairs that shares nothing with the oracle's
per-rank walk, exhaustive enumeration of tiny routings, and the relation to
the independent single-source layout: both send the same tokens to the same
ranks, and their expert-major outputs agree."""
import itertools
import os

import numpy as np
import pytest

from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing, random_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden():
    d = {}
    with open(os.path.join(GOLDEN, "layout_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, *vals = line.split()
                d[k] = vals
    return d


def sorted_pairs_layout(idx: np.ndarray, S: int, E: int, R: int):
    """Receive side by sorting: collect the distinct (r, g) pairs, sort them,
    and number each rank's pairs from its region start; source offsets by
    binary search of the source boundaries in each rank's sorted token list."""
    T, K = idx.shape
    m = E // R
    Ts = T // S
    pairs = sorted({(int(e) // m, g) for g in range(T) for e in idx[g] if 0 <= e < E})
    recv_slot = -np.ones((T, R), np.int64)
    recv_src = -np.ones(R * T, np.int64)
    per_rank = {r: [] for r in range(R)}
    for r, g in pairs:
        per_rank[r].append(g)
    for r, gs in per_rank.items():
        for j, g in enumerate(gs):
            recv_slot[g, r] = r * T + j
            recv_src[r * T + j] = g
    src_off = np.array([[int(np.searchsorted(per_rank[r], s * Ts)) for s in range(S + 1)] for r in range(R)])
    counts = np.array([len(per_rank[r]) for r in range(R)])
    return recv_slot, recv_src, src_off, counts


def _check_against_sorting(o, idx, w, S, E, R):
    T, K = idx.shape
    L = o.layout_sources(idx, w, S, E, R)
    rs, src, off, cnt = sorted_pairs_layout(idx, S, E, R)
    assert L.capacity == R * T and L.num_sources == S
    assert np.array_equal(L.recv_slot, rs)
    assert np.array_equal(L.recv_src_token, src)
    assert np.array_equal(L.recv_source_offset, off)
    assert np.array_equal(L.tokens_per_rank, cnt)
    assert np.array_equal(L.rank_offset, np.arange(R + 1) * T)
    # expert-major rows map to the receive row of their token on their rank
    m = E // R
    for g in range(T):
        for k in range(K):
            e = int(idx[g, k])
            if 0 <= e < E:
                assert L.expert_src_row[L.expert_slot[g, k]] == rs[g, e // m]
    return L


def test_sources_worked_example(oracle_lib):
    import oracle
    g = _read_golden()
    T, K, E, R = (int(g[k][0]) for k in ("T", "K", "E", "R"))
    S = int(g["msrc_S"][0])
    idx = np.array(g["topk_idx"], np.int32).reshape(T, K)
    w = np.array(g["topk_w"], np.float32).reshape(T, K)
    L = oracle.layout_sources(idx, w, S, E, R)
    assert L.status == 0
    assert L.capacity == int(g["msrc_capacity"][0])
    ints = lambda k: np.array(g[k], np.int64)
    assert np.array_equal(L.tokens_per_rank, ints("msrc_tokens_per_rank"))
    assert np.array_equal(L.rank_offset, ints("msrc_rank_offset"))
    assert np.array_equal(L.recv_source_offset.ravel(), ints("msrc_recv_source_offset"))
    assert np.array_equal(L.recv_slot.ravel(), ints("msrc_recv_slot"))
    assert np.array_equal(L.recv_src_token, ints("msrc_recv_src_token"))
    assert np.array_equal(L.expert_src_row, ints("msrc_expert_src_row"))
    # the expert-major side is the single-source example's
    assert np.array_equal(L.tokens_per_expert, ints("tokens_per_expert"))
    assert np.array_equal(L.expert_offset, ints("expert_offset"))
    assert np.array_equal(L.expert_slot.ravel(), ints("expert_slot"))
    assert np.array_equal(L.expert_weight, np.array(g["expert_weight"], np.float32))


@pytest.mark.parametrize("S,Ts,K,E,R,mask,dups,seed", [
    (1, 37, 3, 8, 4, 0.0, False, 0),
    (3, 20, 4, 16, 4, 0.2, True, 1),
    (5, 7, 2, 6, 3, 0.1, False, 2),
    (8, 16, 8, 32, 8, 0.0, False, 3),
    (4, 1, 6, 12, 12, 0.3, True, 4),        # one token per source, one expert per rank
    (2, 0, 2, 4, 2, 0.0, False, 5),          # empty sources
])
def test_sources_vs_sorting(oracle_lib, S, Ts, K, E, R, mask, dups, seed):
    import oracle
    T = S * Ts
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups).numpy() if T else np.zeros((0, K), np.int32)
    w = random_weights(T, K, seed).numpy() if T else np.zeros((0, K), np.float32)
    L = _check_against_sorting(oracle, idx, w, S, E, R)
    assert L.status == 0


def test_sources_exhaustive_tiny(oracle_lib):
    """Every routing of 4 tokens (2 sources x 2), top-2 over 4 experts with
    masks, on 2 ranks."""
    import oracle
    S, E, R, K = 2, 4, 2, 2
    choices = list(itertools.product(range(-1, E), repeat=K))
    rng = np.random.default_rng(7)
    for _ in range(400):
        rows = [choices[i] for i in rng.integers(0, len(choices), size=4)]
        idx = np.array(rows, np.int32)
        _check_against_sorting(oracle, idx, None, S, E, R)


def test_sources_match_single_source_layout(oracle_lib):
    """Same routing, two layouts: the same (token, rank) pairs, the same
    per-rank counts and the same expert-major side; each expert-major row
    reads the same token in both."""
    import oracle
    wl = WORKLOADS["dsv3"].scaled(512)
    inp = make_inputs(wl, with_y=False)
    idx, w = inp.topk_idx.numpy(), inp.topk_w.numpy()
    ss = oracle.layout(idx, w, wl.E, wl.R)
    ms = oracle.layout_sources(idx, w, 8, wl.E, wl.R)
    assert ss.status == 0 and ms.status == 0
    assert np.array_equal(ss.recv_slot >= 0, ms.recv_slot >= 0)
    assert np.array_equal(ss.tokens_per_rank, ms.tokens_per_rank)
    assert ss.n_pairs == ms.n_pairs
    for f in ("tokens_per_expert", "expert_offset", "expert_slot", "expert_weight"):
        assert np.array_equal(getattr(ss, f), getattr(ms, f)), f
    nv = int(ss.expert_offset[-1])
    assert np.array_equal(ss.recv_src_token[ss.expert_src_row[:nv]], ms.recv_src_token[ms.expert_src_row[:nv]])
    assert np.all(ms.expert_src_row[nv:] == -1)


def test_one_expert_per_rank_single_source_is_the_packed_layout(oracle_lib):
    """With one expert per rank the primary expert of (t, r) is r's expert, so
    the single-source layout also orders each rank's rows by token: with S = 1
    the two layouts differ only in where each rank's rows start."""
    import oracle
    T, K, E = 300, 4, 16
    idx = random_routing(T, K, E, 11, mask_frac=0.1).numpy()
    ss = oracle.layout(idx, None, E, E)
    ms = oracle.layout_sources(idx, None, 1, E, E)
    for r in range(E):
        a, b = ss.recv_slot[:, r], ms.recv_slot[:, r]
        assert np.array_equal(a >= 0, b >= 0)
        assert np.array_equal(a[a >= 0] - ss.rank_offset[r], b[b >= 0] - r * T)


def test_sources_region_invariants(oracle_lib):
    """Every region: used rows first, tokens strictly increasing, -1 tail;
    source s's rows hold exactly the tokens of source s that reach r."""
    import oracle
    S, Ts, K, E, R = 6, 50, 6, 64, 16
    T = S * Ts
    idx = random_routing(T, K, E, 3, mask_frac=0.05, allow_duplicates=True).numpy()
    L = oracle.layout_sources(idx, None, S, E, R)
    m = E // R
    for r in range(R):
        reg = L.recv_src_token[r * T:(r + 1) * T]
        n = int(L.tokens_per_rank[r])
        assert np.all(np.diff(reg[:n]) > 0) and np.all(reg[n:] == -1)
        for s in range(S):
            lo, hi = L.recv_source_offset[r, s], L.recv_source_offset[r, s + 1]
            want = [g for g in range(s * Ts, (s + 1) * Ts) if any(0 <= e < E and e // m == r for e in idx[g])]
            assert list(reg[lo:hi]) == want


def test_sources_flag_bad_ids(oracle_lib):
    import oracle
    idx = np.array([[0, 5], [9, -1], [-3, 1], [2, 3]], np.int32)
    L = oracle.layout_sources(idx, None, 2, 4, 2)
    assert L.status & 2
    clean = np.where((idx >= 0) & (idx < 4), idx, -1).astype(np.int32)
    M = oracle.layout_sources(clean, None, 2, 4, 2)
    assert M.status == 0
    assert np.array_equal(L.recv_slot, M.recv_slot) and np.array_equal(L.expert_slot, M.expert_slot)
