"""moe_dispatch_with_layout: the layout and the dispatch in one call, whose
dispatch may read x before the layout's outputs exist.  Its results must be
the oracle's (layout arrays, receive rows, FP8 / MXFP8 codes and scales bit
for bit), equal to the two separate calls', on the full-size workloads,
edge cases, every kernel variant, 16-byte-only alignment (no early loads),
the multi-source layout, and a CUDA graph replayed on new inputs."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_dispatch_02_gb300 import ep
from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, bf16_bits, make_inputs, random_routing, random_weights
from harness import LAYOUT_FIELDS, assert_parity, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()
    oracle.build()


def _fused(x, idx, w, E, R, fmt, x_dev=None, **tuning):
    """Layout + dispatch through the one call; returns the outputs as numpy."""
    T, K = idx.shape
    H = x.shape[1]
    L = ep.Layout(T, K, E, R)
    recv, scales = ep.alloc_recv(L, H, fmt)
    xd = x.cuda() if x_dev is None else x_dev
    ep.moe_dispatch_with_layout(idx.cuda(), w.cuda() if w is not None else None, E, R, L, xd, fmt, recv, scales,
                                **tuning)
    st, flags = ep.moe_layout_read_status(L)
    res = {f: getattr(L, f).cpu().numpy() for f in LAYOUT_FIELDS}
    n = int(res["rank_offset"][R])
    res["n_pairs"] = n
    if fmt:
        res["recv_q"] = recv[:n].cpu().numpy()
        res["recv_scales"] = scales[:n].cpu().numpy().copy()
    else:
        res["recv_x"] = bf16_bits(recv[:n].cpu())
    res["status"] = st
    return res


def _separate(x, idx, w, E, R, fmt):
    T, K = idx.shape
    L = ep.Layout(T, K, E, R)
    recv, scales = ep.alloc_recv(L, x.shape[1], fmt)
    ep.moe_dispatch_layout(idx.cuda(), w.cuda(), E, R, L)
    ep.moe_dispatch(x.cuda(), L, fmt, recv, scales)
    n = int(L.rank_offset[R].item())
    return recv[:n].cpu(), None if scales is None else scales[:n].cpu()


@pytest.mark.parametrize("name", ["tiny", "dsv3", "qwen_skew", "ds16_wide"])
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_workload_parity(name, fmt):
    wl = WORKLOADS[name]
    if fmt and wl.H % 128:
        pytest.skip("FP8 formats need hidden % 128 == 0")
    inp = make_inputs(wl, with_y=False)
    g = _fused(inp.x, inp.topk_idx, inp.topk_w, wl.E, wl.R, fmt)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=fmt)
    assert g["status"] == 0 and o["status"] == 0
    assert_parity(g, o, fp8=bool(fmt))
    # and the two separate calls write the same bytes
    rx, rs = _separate(inp.x, inp.topk_idx, inp.topk_w, wl.E, wl.R, fmt)
    if fmt:
        assert np.array_equal(rx.numpy(), g["recv_q"])
        assert np.array_equal(np.ascontiguousarray(rs.numpy()).view(np.uint8),
                              np.ascontiguousarray(g["recv_scales"]).view(np.uint8))
    else:
        assert np.array_equal(bf16_bits(rx), g["recv_x"])


@pytest.mark.parametrize("T,H,E,R,K,mask,dups,fmt,seed", [
    (1, 128, 4, 2, 2, 0.0, False, 1, 1),
    (777, 136, 16, 4, 3, 0.1, False, 0, 2),       # bf16 hidden % 16 != 0: the TMA kernel, no early loads
    (300, 48, 16, 4, 4, 0.0, False, 0, 13),       # rows ending half-way through a lane
    (257, 3200, 16, 8, 4, 0.05, True, 1, 14),     # FP8 rows ending inside a 1024-column segment
    (257, 3200, 16, 8, 4, 0.05, True, 2, 15),
    (700, 256, 128, 64, 8, 0.1, False, 1, 12),    # more than 32 destination ranks
    (2500, 128, 256, 32, 8, 0.0, False, 0, 10),   # many scan tiles
    (4096, 64, 1024, 256, 32, 0.0, False, 0, 11),  # the maxima of E, R and K
    (100, 256, 8, 4, 3, 1.0, False, 1, 16),       # every entry masked
])
@pytest.mark.parametrize("variant", [0, 1, 2, 3])
def test_edge_case_parity(T, H, E, R, K, mask, dups, fmt, seed, variant):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups)
    w = random_weights(T, K, seed)
    g_ = torch.Generator().manual_seed(seed + 1)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    g = _fused(x, idx, w, E, R, fmt, variant=variant)
    o = oracle_run(x, idx, w, None, E, R, fp8=fmt)
    assert g["status"] == 0 and o["status"] == 0
    assert_parity(g, o, fp8=bool(fmt))


def test_zero_tokens():
    idx = torch.zeros(0, 2, dtype=torch.int32)
    x = torch.zeros(0, 128, dtype=torch.bfloat16)
    g = _fused(x, idx, torch.zeros(0, 2), 8, 2, 1)
    assert g["status"] == 0 and g["n_pairs"] == 0


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_only_16_byte_aligned_x(fmt):
    """x at a 16-byte offset: the dispatch falls back to the 16-byte kernels
    (which load nothing early); the results are unchanged."""
    T, H, E, R, K = 300, 1024, 32, 8, 6
    idx = random_routing(T, K, E, 31, mask_frac=0.05)
    w = random_weights(T, K, 31)
    g_ = torch.Generator().manual_seed(32)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    xbuf = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
    x_off = xbuf[8:].view(T, H)
    x_off.copy_(x.cuda())
    assert x_off.data_ptr() % 32 == 16
    g = _fused(x, idx, w, E, R, fmt, x_dev=x_off)
    o = oracle_run(x, idx, w, None, E, R, fp8=fmt)
    assert_parity(g, o, fp8=bool(fmt))


@pytest.mark.parametrize("fmt", [0, 1])
def test_multi_source_layout(fmt):
    """8 sources of 512 tokens at the DeepSeek-V3 hidden size: the layout's
    third kernel sits between it and the dispatch."""
    wl = WORKLOADS["dsv3"].scaled(4096)
    inp = make_inputs(wl, with_y=False)
    S = 8
    L = ep.Layout(wl.T, wl.K, wl.E, wl.R, sources=S)
    recv, scales = ep.alloc_recv(L, wl.H, fmt)
    ep.moe_dispatch_with_layout(inp.topk_idx.cuda(), inp.topk_w.cuda(), wl.E, wl.R, L, inp.x.cuda(), fmt, recv,
                                scales)
    assert ep.moe_layout_read_status(L) == (0, 0)
    o = oracle.layout_sources(inp.topk_idx.numpy(), inp.topk_w.numpy(), S, wl.E, wl.R)
    assert np.array_equal(L.recv_slot.cpu().numpy().ravel(), o.recv_slot.ravel())
    assert np.array_equal(L.recv_source_offset.cpu().numpy().ravel(), o.recv_source_offset.ravel())
    rows = np.nonzero(o.recv_src_token >= 0)[0]
    rows_d = torch.from_numpy(rows).cuda()
    xb = bf16_bits(inp.x)
    if fmt == 0:
        rx, st = oracle.dispatch_bf16(xb, o)
        assert st == 0 and np.array_equal(bf16_bits(recv[rows_d].cpu()), rx[rows])
    else:
        q, s, st = oracle.dispatch_fp8(xb, o)
        assert st == 0 and np.array_equal(recv[rows_d].cpu().numpy(), q[rows])
        assert np.array_equal(np.ascontiguousarray(scales[rows_d].cpu().numpy()).view(np.uint8),
                              np.ascontiguousarray(s[rows]).view(np.uint8))


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_graph_replays_on_new_inputs(fmt):
    """Captured once (with the combine, as a training step would run it) and
    replayed on three new routings and activations."""
    T, H, E, R, K = 2000, 1024, 64, 8, 6
    dev = torch.device("cuda", 0)
    L = ep.Layout(T, K, E, R, device=dev)

    def inputs(seed):
        idx = random_routing(T, K, E, seed, mask_frac=0.05)
        w = random_weights(T, K, seed)
        g = torch.Generator().manual_seed(seed + 1)
        return idx, w, (torch.randn(T, H, generator=g) * 2).to(torch.bfloat16), \
            torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    idx0, w0, x0, y0 = inputs(700)
    idx_d, w_d, x_d, y_d = idx0.to(dev), w0.to(dev), x0.to(dev), y0.to(dev)
    recv, scales = ep.alloc_recv(L, H, fmt, device=dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ep.moe_dispatch_with_layout(idx_d, w_d, E, R, L, x_d, fmt, recv, scales)
    ep.moe_combine(y_d, L, w_d, out)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        ep.moe_dispatch_with_layout(idx_d, w_d, E, R, L, x_d, fmt, recv, scales, s)
        ep.moe_combine(y_d, L, w_d, out, s)
    for seed in (701, 702, 703):
        idx, w, x, y = inputs(seed)
        idx_d.copy_(idx)
        w_d.copy_(w)
        x_d.copy_(x)
        y_d.copy_(y)
        g.replay()
        torch.cuda.synchronize()
        assert ep.moe_layout_read_status(L) == (0, 0)
        res = {f: getattr(L, f).cpu().numpy() for f in LAYOUT_FIELDS}
        n = int(res["rank_offset"][R])
        res["n_pairs"] = n
        if fmt:
            res["recv_q"] = recv[:n].cpu().numpy()
            res["recv_scales"] = scales[:n].cpu().numpy().copy()
        else:
            res["recv_x"] = bf16_bits(recv[:n].cpu())
        res["out"] = bf16_bits(out.cpu())
        o = oracle_run(x, idx, w, y, E, R, fp8=fmt)
        assert_parity(res, o, fp8=bool(fmt))
        assert np.array_equal(res["out"], o["out"])


def test_timeout_is_reported_and_recoverable():
    """The layout's bounded wait made to run out (test hook) inside the one
    call: the timeout is reported, and the next call is healthy."""
    wl = WORKLOADS["dsv3"].scaled(2048)
    inp = make_inputs(wl, with_y=False)
    L = ep.Layout(2048, wl.K, wl.E, wl.R)
    recv, scales = ep.alloc_recv(L, wl.H, 1)
    idx, w, x = inp.topk_idx.cuda(), inp.topk_w.cuda(), inp.x.cuda()
    ep.moe_dispatch_with_layout(idx, w, wl.E, wl.R, L, x, 1, recv, scales, wait_timeout_ns=20_000_000,
                                debug_flags=ep.MOE_DEBUG_STALL_FIRST_TILE)
    st, flags = ep.moe_layout_read_status(L)
    assert st == ep.MOE_ERR_TIMEOUT and flags & ep.MOE_DEVERR_TIMEOUT
    ep.moe_dispatch_with_layout(idx, w, wl.E, wl.R, L, x, 1, recv, scales)
    assert ep.moe_layout_read_status(L) == (0, 0)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=1)
    n = o["n_pairs"]
    assert np.array_equal(recv[:n].cpu().numpy(), o["recv_q"])


def _check_layout_and_rows(L, recv, scales, x, idx, w, E, R, fmt):
    assert ep.moe_layout_read_status(L) == (0, 0)
    res = {f: getattr(L, f).cpu().numpy() for f in LAYOUT_FIELDS}
    n = int(res["rank_offset"][R])
    res["n_pairs"] = n
    if fmt:
        res["recv_q"] = recv[:n].cpu().numpy()
        res["recv_scales"] = scales[:n].cpu().numpy().copy()
    else:
        res["recv_x"] = bf16_bits(recv[:n].cpu())
    o = oracle_run(x, idx, w, None, E, R, fp8=fmt)
    assert_parity(res, o, fp8=bool(fmt))


def test_call_kinds_interleaved_on_one_layout():
    """The one call (early loads for bf16 and MXFP8, not for FP8), the
    separate calls, a one call on another grid (few channels) and the layout
    alone, alternating on one workspace with new routings: every call
    matches the oracle, so no call reads a word another call left behind."""
    T, H, E, R, K = 1500, 1024, 64, 8, 6
    L = ep.Layout(T, K, E, R)
    bufs = {fmt: ep.alloc_recv(L, H, fmt) for fmt in (0, 1, 2)}
    kinds = ["fused", "separate", "fused", "fused_channels", "fused", "layout_only", "fused", "fused"]
    fmts = [0, 0, 1, 2, 2, 0, 0, 1]
    for step, (kind, fmt) in enumerate(zip(kinds, fmts)):
        seed = 900 + step
        idx = random_routing(T, K, E, seed, mask_frac=0.05)
        w = random_weights(T, K, seed)
        g_ = torch.Generator().manual_seed(seed + 1)
        x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
        idx_d, w_d, x_d = idx.cuda(), w.cuda(), x.cuda()
        recv, scales = bufs[fmt]
        if kind == "fused":
            ep.moe_dispatch_with_layout(idx_d, w_d, E, R, L, x_d, fmt, recv, scales)
        elif kind == "fused_channels":
            ep.moe_dispatch_with_layout(idx_d, w_d, E, R, L, x_d, fmt, recv, scales, num_channels=40)
        elif kind == "separate":
            ep.moe_dispatch_layout(idx_d, w_d, E, R, L)
            ep.moe_dispatch(x_d, L, fmt, recv, scales)
        else:
            ep.moe_dispatch_layout(idx_d, w_d, E, R, L)
            assert ep.moe_layout_read_status(L) == (0, 0)
            o = oracle_run(x, idx, w, None, E, R, fp8=0)
            assert np.array_equal(L.recv_slot.cpu().numpy().ravel(), o["recv_slot"].ravel())
            continue
        _check_layout_and_rows(L, recv, scales, x, idx, w, E, R, fmt)


@pytest.mark.parametrize("T", [20000, 40000])
@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_many_scan_tiles(T, fmt):
    """79 scan tiles (flag look-back, tiles by block index) and 157 (more
    than the SMs: tiles from the ticket) in the one call."""
    H, E, R, K = 256, 256, 8, 8
    idx = random_routing(T, K, E, 41, mask_frac=0.02)
    w = random_weights(T, K, 41)
    g_ = torch.Generator().manual_seed(42)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    L = ep.Layout(T, K, E, R)
    assert L.c.num_tiles in (79, 157)
    recv, scales = ep.alloc_recv(L, H, fmt)
    ep.moe_dispatch_with_layout(idx.cuda(), w.cuda(), E, R, L, x.cuda(), fmt, recv, scales)
    _check_layout_and_rows(L, recv, scales, x, idx, w, E, R, fmt)


@pytest.mark.parametrize("fmt", [0, 2])
def test_timeout_is_reported_and_recoverable_bf16_mx(fmt):
    """As above for the formats whose dispatch loads early (its grid is
    resident while the scan gives up)."""
    wl = WORKLOADS["dsv3"].scaled(2048)
    inp = make_inputs(wl, with_y=False)
    L = ep.Layout(2048, wl.K, wl.E, wl.R)
    recv, scales = ep.alloc_recv(L, wl.H, fmt)
    idx, w, x = inp.topk_idx.cuda(), inp.topk_w.cuda(), inp.x.cuda()
    ep.moe_dispatch_with_layout(idx, w, wl.E, wl.R, L, x, fmt, recv, scales, wait_timeout_ns=20_000_000,
                                debug_flags=ep.MOE_DEBUG_STALL_FIRST_TILE)
    st, flags = ep.moe_layout_read_status(L)
    assert st == ep.MOE_ERR_TIMEOUT and flags & ep.MOE_DEVERR_TIMEOUT
    ep.moe_dispatch_with_layout(idx, w, wl.E, wl.R, L, x, fmt, recv, scales)
    _check_layout_and_rows(L, recv, scales, inp.x, inp.topk_idx, inp.topk_w, wl.E, wl.R, fmt)
