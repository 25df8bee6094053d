"""Pins for the oracle's dispatch layout.

Expected values come from a hand-derived worked example (tests/golden), a
brute-force construction by sorting tuples (written independently of the
oracle's counting loops), exhaustive enumeration of tiny routings, and
invariants that any correct layout satisfies.
"""
import itertools
import os

import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing, random_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def brute_force_layout(idx: np.ndarray, w, E: int, R: int, capacity: int):
    """Layout by sorting.  Receive rows: the (primary expert, token) tuples in
    sorted order; expert rows: the (expert, token, k) tuples in sorted order."""
    T, K = idx.shape
    m = E // R
    pairs = []                                   # (primary, t, r)
    for t in range(T):
        by_rank = {}
        for k in range(K):
            e = int(idx[t, k])
            if 0 <= e < E:
                by_rank.setdefault(e // m, []).append(e)
        for r, es in by_rank.items():
            pairs.append((min(es), t, r))
    pairs.sort()
    recv_slot = -np.ones((T, R), np.int64)
    recv_src = -np.ones(capacity, np.int64)
    for row, (p, t, r) in enumerate(pairs):
        recv_slot[t, r] = row
        recv_src[row] = t
    ents = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K) if 0 <= idx[t, k] < E)
    expert_slot = -np.ones((T, K), np.int64)
    src_row = -np.ones(T * K, np.int64)
    ew = np.zeros(T * K, np.float32)
    for row, (e, t, k) in enumerate(ents):
        expert_slot[t, k] = row
        src_row[row] = recv_slot[t, e // m]
        if w is not None:
            ew[row] = w[t, k]
    tpe = np.bincount([e for e, _, _ in ents], minlength=E)
    prim = np.bincount([p for p, _, _ in pairs], minlength=E)
    tpr = np.bincount([r for _, _, r in pairs], minlength=R)
    return dict(tokens_per_expert=tpe, expert_offset=np.concatenate([[0], np.cumsum(tpe)]),
                tokens_per_rank=tpr, rank_offset=np.concatenate([[0], np.cumsum(tpr)]),
                recv_expert_offset=np.concatenate([[0], np.cumsum(prim)]),
                recv_slot=recv_slot, expert_slot=expert_slot, recv_src_token=recv_src,
                expert_src_row=src_row, expert_weight=ew)


def assert_layout_equal(L, ref, check_weight=True):
    for k, v in ref.items():
        if k == "expert_weight" and not check_weight:
            continue
        got = getattr(L, k)
        assert np.array_equal(np.asarray(got).ravel(), np.asarray(v).ravel()), k


def check_invariants(L, idx, E, R):
    T, K = idx.shape
    valid = (idx >= 0) & (idx < E)
    n_valid = int(valid.sum())
    assert L.tokens_per_expert.sum() == n_valid
    assert L.expert_offset[-1] == n_valid
    n_pairs = int((L.recv_slot >= 0).sum())
    assert L.rank_offset[R] == n_pairs == L.tokens_per_rank.sum()
    # every valid (t, r) pair appears exactly once; slots are a permutation of [0, n_pairs)
    slots = L.recv_slot[L.recv_slot >= 0]
    assert np.array_equal(np.sort(slots), np.arange(n_pairs))
    assert n_pairs <= L.capacity
    # recv_src_token is the inverse of recv_slot
    for t, r in zip(*np.nonzero(L.recv_slot >= 0)):
        assert L.recv_src_token[L.recv_slot[t, r]] == t
    assert np.all(L.recv_src_token[n_pairs:] == -1)
    # rows of rank r lie in [rank_offset[r], rank_offset[r+1])
    for r in range(R):
        s = L.recv_slot[:, r]
        s = s[s >= 0]
        assert np.all((s >= L.rank_offset[r]) & (s < L.rank_offset[r + 1]))
    # expert rows: a permutation of [0, n_valid), inside the expert's range
    es = L.expert_slot[valid]
    assert np.array_equal(np.sort(es), np.arange(n_valid))
    assert np.all(L.expert_slot[~valid] == -1)
    e_of = idx[valid]
    assert np.all((es >= L.expert_offset[e_of]) & (es < L.expert_offset[e_of + 1]))
    # expert rows point at the receive row of the same token on the expert's rank
    m = E // R
    ts = np.nonzero(valid)[0]
    assert np.array_equal(L.expert_src_row[es], L.recv_slot[ts, e_of // m])
    assert np.all(L.expert_src_row[n_valid:] == -1)


def _read_golden():
    d = {}
    with open(os.path.join(GOLDEN, "layout_worked_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, *vals = line.split()
                d[k] = vals
    return d


def test_layout_worked_example(oracle_lib):
    g = _read_golden()
    T, K, E, R, cap = (int(g[k][0]) for k in ("T", "K", "E", "R", "capacity"))
    idx = np.array(g["topk_idx"], np.int32).reshape(T, K)
    w = np.array(g["topk_w"], np.float32).reshape(T, K)
    L = oracle_lib.layout(idx, w, E, R, cap)
    assert L.status == 0
    for k in ("tokens_per_expert", "expert_offset", "tokens_per_rank", "rank_offset",
              "recv_expert_offset", "recv_slot", "expert_slot", "recv_src_token", "expert_src_row"):
        assert np.array_equal(np.asarray(getattr(L, k)).ravel(), np.array(g[k], np.int64)), k
    assert np.array_equal(L.expert_weight, np.array(g["expert_weight"], np.float32))
    # the brute-force construction agrees with the hand derivation too
    assert_layout_equal(L, brute_force_layout(idx, w, E, R, cap))


@pytest.mark.parametrize("T,K,E,R,mask,dups,seed", [
    (1, 1, 1, 1, 0.0, False, 0),
    (16, 3, 8, 4, 0.0, False, 1),
    (16, 3, 8, 4, 0.3, False, 2),
    (13, 4, 8, 2, 0.2, True, 3),      # duplicate expert ids inside a row
    (9, 2, 6, 3, 0.0, True, 4),
    (64, 8, 16, 8, 0.1, False, 5),
    (33, 6, 64, 32, 0.0, False, 6),
    (40, 8, 8, 8, 0.0, False, 7),     # every token to every expert
    (0, 2, 4, 2, 0.0, False, 8),      # no tokens
])
def test_layout_vs_brute_force(oracle_lib, T, K, E, R, mask, dups, seed):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups).numpy() if T else np.zeros((0, K), np.int32)
    w = random_weights(T, K, seed).numpy() if T else np.zeros((0, K), np.float32)
    cap = T * min(K, R)
    L = oracle_lib.layout(idx, w, E, R, cap)
    assert L.status == 0
    assert_layout_equal(L, brute_force_layout(idx, w, E, R, cap))
    if T:
        check_invariants(L, idx, E, R)


def test_layout_exhaustive_two_tokens(oracle_lib):
    """All ordered pairs of entries (including masked and duplicate ids) for two
    tokens, E=4 experts on R=2 ranks, top-2."""
    E, R, K = 4, 2, 2
    rows = list(itertools.product(range(-1, E), repeat=K))
    w = np.full((2, K), 0.5, np.float32)
    for a in rows:
        for b in rows:
            idx = np.array([a, b], np.int32)
            L = oracle_lib.layout(idx, w, E, R, 2 * min(K, R))
            assert L.status == 0
            assert_layout_equal(L, brute_force_layout(idx, w, E, R, 2 * min(K, R)))


@pytest.mark.parametrize("name", ["tiny", "dsv3", "qwen_skew", "ds16_wide"])
def test_layout_invariants_on_workloads(oracle_lib, name):
    wl = WORKLOADS[name]
    if wl.T > 4096:
        wl = wl.scaled(2048)       # keep the CPU suite quick; the routing recipe is unchanged
    inp = make_inputs(wl, with_y=False)
    idx = inp.topk_idx.numpy()
    L = oracle_lib.layout(idx, inp.topk_w.numpy(), wl.E, wl.R, wl.capacity)
    assert L.status == 0
    check_invariants(L, idx, wl.E, wl.R)
    assert L.tokens_per_expert.sum() == wl.T * wl.K        # no masked entries in routed inputs


def test_layout_flags_out_of_range_ids(oracle_lib):
    idx = np.array([[0, 5], [-2, 1], [3, 2]], np.int32)     # 5 and -2 are invalid for E=4
    L = oracle_lib.layout(idx, None, 4, 2, 6)
    assert L.status & oracle_lib.ERR_EXPERT_ID
    cleaned = np.where((idx >= 0) & (idx < 4), idx, -1)
    assert_layout_equal(L, brute_force_layout(cleaned, None, 4, 2, 6), check_weight=False)


def test_layout_flags_capacity(oracle_lib):
    idx = np.array([[0, 2], [1, 3]], np.int32)              # 4 (t, r) pairs
    L = oracle_lib.layout(idx, None, 4, 2, 3)
    assert L.status & oracle_lib.ERR_CAPACITY


def test_layout_rejects_bad_sizes(oracle_lib):
    idx = np.zeros((2, 2), np.int32)
    assert oracle_lib.layout(idx, None, 6, 4, 4).status & oracle_lib.ERR_ARG   # E % R != 0
