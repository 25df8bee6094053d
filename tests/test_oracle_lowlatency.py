"""Pins for the oracle's low-latency (fixed per-expert capacity) dispatch: the
hand-derived worked example, brute force by sorting, capacity overflow, and
the dispatch -> identity expert -> combine round trip on this layout."""
import os

import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import bf16_bits, random_routing, random_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_worked_example.txt")


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, *v = line.split()
            d[k] = v
    return d


def brute_force_ll(idx, E, cap):
    T, K = idx.shape
    ents = sorted((int(idx[t, k]), t, k) for t in range(T) for k in range(K) if 0 <= idx[t, k] < E)
    slot = -np.ones((T, K), np.int64)
    count = np.zeros(E, np.int64)
    for e, t, k in ents:                       # sorted by (expert, token, k)
        if count[e] < cap:
            slot[t, k] = e * cap + count[e]
            count[e] += 1
    return slot, count


def test_ll_worked_example(oracle_lib):
    g = _golden()
    T, K, E, cap = int(g["T"][0]), int(g["K"][0]), int(g["E"][0]), int(g["ll_cap"][0])
    idx = np.array(g["topk_idx"], np.int32).reshape(T, K)
    x = np.arange(T * 8, dtype=np.uint16).reshape(T, 8)
    recv, tpe, slot, st = oracle_lib.ll_dispatch(x, idx, E, cap)
    assert st == 0
    assert np.array_equal(slot.ravel(), np.array(g["ll_slot"], np.int64))
    assert np.array_equal(tpe, np.array(g["ll_tokens_per_expert"], np.int64))
    for t in range(T):
        for k in range(K):
            if slot[t, k] >= 0:
                assert np.array_equal(recv[slot[t, k]], x[t])


@pytest.mark.parametrize("T,K,E,cap,mask,dups,seed", [
    (50, 4, 16, 50, 0.1, False, 0), (33, 8, 8, 33, 0.0, False, 1), (20, 3, 4, 8, 0.0, True, 2), (0, 2, 4, 4, 0.0, False, 3)])
def test_ll_vs_brute_force(oracle_lib, T, K, E, cap, mask, dups, seed):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups).numpy() if T else np.zeros((0, K), np.int32)
    x = np.random.default_rng(seed).integers(0, 65535, (T, 16)).astype(np.uint16)
    recv, tpe, slot, st = oracle_lib.ll_dispatch(x, idx, E, cap)
    want_slot, want_cnt = brute_force_ll(idx, E, cap)
    assert np.array_equal(slot, want_slot) and np.array_equal(tpe, want_cnt)
    overflow = any(np.sum(idx == e) > cap for e in range(E))
    assert (st != 0) == overflow


def test_ll_round_trip(oracle_lib):
    """dispatch -> identity expert -> combine on the low-latency layout returns x
    (weights renormalised to 1)."""
    T, K, E, H = 128, 8, 256, 64
    idx = random_routing(T, K, E, 5).numpy()
    w = random_weights(T, K, 5).numpy()
    xb = bf16_bits(torch.randn(T, H).to(torch.bfloat16))
    recv, tpe, slot, st = oracle_lib.ll_dispatch(xb, idx, E, T)
    assert st == 0
    out, st = oracle_lib.combine(recv, slot, w)            # the expert output is its input
    assert st == 0 and np.array_equal(out, xb)
