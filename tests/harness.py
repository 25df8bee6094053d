"""Shared test plumbing: run the CUDA path (through the C ABI) and the CPU
oracle on the same seeded inputs and compare.  The two sides share only the
input generator; neither computes anything for the other."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from combine_moe_dispatch_02_gb300 import ep
from combine_moe_dispatch_02_gb300.inputs import bf16_bits

LAYOUT_FIELDS = ("tokens_per_expert", "expert_offset", "tokens_per_rank", "rank_offset", "recv_expert_offset",
                 "recv_slot", "expert_slot", "recv_src_token", "expert_src_row", "expert_weight")


def gpu_run(x, topk_idx, topk_w, y, E, R, fp8=False, capacity=None, reps=1, **tuning):
    """Layout -> dispatch -> combine on cuda:0.  `fp8` is a receive format
    (False/0 bf16, True/1 FP8 1x128, 2 MXFP8).  Returns numpy copies of every
    output, the receive buffers and the status."""
    dev = torch.device("cuda", 0)
    T, K = topk_idx.shape
    H = x.shape[1]
    L = ep.Layout(T, K, E, R, capacity, device=dev)
    idx_d = topk_idx.to(dev)
    w_d = topk_w.to(dev) if topk_w is not None else None
    x_d = x.to(dev)
    recv_x, recv_s = ep.alloc_recv(L, H, fp8, device=dev)
    out_d = torch.empty(T, H, dtype=torch.bfloat16, device=dev) if y is not None else None
    y_d = y.to(dev) if y is not None else None
    for _ in range(reps):
        ep.moe_dispatch_layout(idx_d, w_d, E, R, L, **tuning)
        ep.moe_dispatch(x_d, L, fp8, recv_x, recv_s, **tuning)
        if y is not None:
            ep.moe_combine(y_d, L, w_d, out_d, **tuning)
    st, flags = ep.moe_layout_read_status(L)
    res = {f: getattr(L, f).cpu().numpy() for f in LAYOUT_FIELDS}
    n_pairs = int(res["rank_offset"][R])
    if fp8:
        res["recv_q"] = recv_x[:n_pairs].cpu().numpy()
        res["recv_scales"] = recv_s[:n_pairs].cpu().numpy().copy()
    else:
        res["recv_x"] = bf16_bits(recv_x[:n_pairs].cpu())
    if y is not None:
        res["out"] = bf16_bits(out_d.cpu())
    res["status"], res["flags"] = st, flags
    res["n_pairs"] = n_pairs
    return res


def oracle_run(x, topk_idx, topk_w, y, E, R, fp8=False, capacity=None):
    idx = topk_idx.numpy()
    w = topk_w.numpy() if topk_w is not None else None
    L = oracle.layout(idx, w, E, R, capacity)
    res = {f: getattr(L, f) for f in LAYOUT_FIELDS}
    xb = bf16_bits(x)
    n_pairs = L.n_pairs
    if int(fp8) == 2:
        q, s, st = oracle.dispatch_mxfp8(xb, L)
        res["recv_q"], res["recv_scales"] = q[:n_pairs], s[:n_pairs]
    elif fp8:
        q, s, st = oracle.dispatch_fp8(xb, L)
        res["recv_q"], res["recv_scales"] = q[:n_pairs], s[:n_pairs]
    else:
        rx, st = oracle.dispatch_bf16(xb, L)
        res["recv_x"] = rx[:n_pairs]
    if y is not None:
        res["out"], st2 = oracle.combine(bf16_bits(y), L.expert_slot, topk_w.numpy())
        st |= st2
    res["status"] = L.status | st
    res["n_pairs"] = n_pairs
    return res


def bf16_ulp_diff(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between bf16 bit patterns (ordered
    integer mapping of the sign-magnitude encoding)."""
    def ordered(u):
        u = u.astype(np.int32)
        return np.where(u & 0x8000, 0x8000 - (u & 0x7FFF), 0x8000 + (u & 0x7FFF))
    return np.abs(ordered(a_bits) - ordered(b_bits))


def assert_parity(g, o, fp8=False, combine_ulps=1):
    for f in LAYOUT_FIELDS:
        assert np.array_equal(np.asarray(g[f]).ravel(), np.asarray(o[f]).ravel()), f"layout field {f} differs"
    assert g["n_pairs"] == o["n_pairs"]
    if fp8:
        assert np.array_equal(g["recv_q"], o["recv_q"]), "FP8 codes differ"
        gs, os_ = np.ascontiguousarray(g["recv_scales"]), np.ascontiguousarray(o["recv_scales"])
        assert gs.dtype == os_.dtype and np.array_equal(gs.view(np.uint8), os_.view(np.uint8)), "FP8 scales differ"
    else:
        assert np.array_equal(g["recv_x"], o["recv_x"]), "bf16 receive rows differ"
    if "out" in o:
        d = bf16_ulp_diff(g["out"], o["out"])
        assert d.max(initial=0) <= combine_ulps, f"combine differs by {d.max()} ulp"
