"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
the same seeded inputs.  Layout, indices, bf16 rows, FP8 bytes and scales
must match bit for bit; combine within 1 bf16 ulp (and in practice bit for
bit: both sides run the same fp32 fma chain in ascending k)."""
import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing, random_weights
from harness import assert_parity, bf16_ulp_diff, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from combine_moe_dispatch_02_gb300 import build, ep
    build.build()
    ep.lib()
    import oracle
    oracle.build()


@pytest.mark.parametrize("name", ["tiny", "dsv3", "dsv3_fp8", "qwen_skew", "ds16_wide"])
def test_workload_parity_full_size(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R, fp8=wl.fp8)
    assert o["status"] == 0
    for variant in (0, 1, 2, 3, 4):
        g = gpu_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R, fp8=wl.fp8, variant=variant)
        assert g["status"] == 0
        assert_parity(g, o, fp8=wl.fp8)
        # combine is bit-exact in practice (same fma chain)
        assert np.array_equal(g["out"], o["out"])


@pytest.mark.parametrize("T,H,E,R,K,mask,dups,fp8,seed", [
    (1, 8, 1, 1, 1, 0.0, False, False, 0),          # smallest everything
    (1, 128, 4, 2, 2, 0.0, False, True, 1),
    (777, 136, 16, 4, 3, 0.1, False, False, 2),      # ragged tokens, odd-ish hidden
    (1000, 256, 32, 8, 6, 0.2, True, False, 3),      # masked + duplicate ids
    (1000, 384, 32, 8, 6, 0.2, True, True, 4),       # same for FP8
    (513, 64, 8, 8, 8, 0.0, False, False, 5),        # one expert per rank, every expert
    (600, 64, 12, 1, 5, 0.0, False, False, 6),       # a single rank
    (300, 96, 64, 4, 16, 0.05, False, False, 7),     # top-16: generic combine path
    (200, 8200, 16, 4, 4, 0.0, False, False, 8),     # rows split into two column chunks
    (128, 9216, 16, 4, 4, 0.0, False, True, 9),      # FP8 rows split into chunks
    (2500, 128, 256, 32, 8, 0.0, False, False, 10),  # many tiles, wide ranks
    (4096, 64, 1024, 256, 32, 0.0, False, False, 11),  # the documented maxima of E, R and K
    (700, 256, 128, 64, 8, 0.1, False, True, 12),   # FP8 with more than 32 destination ranks
    (300, 48, 16, 4, 4, 0.0, False, False, 13),      # bf16 rows ending half-way through a 32-column lane
    (257, 3200, 16, 8, 4, 0.05, False, True, 14),    # FP8 rows ending inside a 1024-column segment
    (250, 64, 6, 3, 5, 0.1, False, False, 15),       # E and tile_tokens * R (1227) not multiples of 4:
                                                     # the scan's padded shared-memory tables
])
@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_edge_case_parity(T, H, E, R, K, mask, dups, fp8, seed, variant):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups)
    w = random_weights(T, K, seed)
    g_ = torch.Generator().manual_seed(seed + 1)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    y = torch.randn(T * K, H, generator=g_).to(torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R, fp8=fp8, variant=variant)
    o = oracle_run(x, idx, w, y, E, R, fp8=fp8)
    assert g["status"] == 0 and o["status"] == 0
    assert_parity(g, o, fp8=fp8)


@pytest.mark.parametrize("T,H,E,R,K,mask,seed", [
    (777, 144, 16, 4, 3, 0.1, 30),            # one partial 512-column segment, one batch of rows
    (1000, 784, 32, 8, 6, 0.2, 31),           # a 272-column last segment, masked entries
    (300, 96, 64, 4, 16, 0.05, 32),           # K = 16: six batches per token
    (4096, 64, 1024, 256, 32, 0.0, 33),       # K = 32: one full 32-slot window
])
def test_combine_gather(T, H, E, R, K, mask, seed):
    """The combine as the 32-byte gather (variant 4) against the oracle, bit
    for bit."""
    idx = random_routing(T, K, E, seed, mask_frac=mask)
    w = random_weights(T, K, seed)
    g_ = torch.Generator().manual_seed(seed + 1)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    y = torch.randn(T * K, H, generator=g_).to(torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R, variant=4)
    o = oracle_run(x, idx, w, y, E, R)
    assert g["status"] == 0 and o["status"] == 0
    assert_parity(g, o)
    assert np.array_equal(g["out"], o["out"])


@pytest.mark.parametrize("T,H,E,R,K,mask,fp8,seed", [
    (262144, 8, 256, 8, 8, 0.0, False, 20),    # 1,024 scan tiles: the flag look-back at length
    (100003, 16, 64, 4, 6, 0.05, False, 21),   # ragged last tile, masked entries
    (65536, 128, 256, 8, 8, 0.0, True, 22),    # FP8 over 256 tiles
    (20000, 16, 256, 8, 8, 0.02, False, 23),   # 79 tiles: the flag look-back with block-index tiles
    (8449, 32, 256, 8, 8, 0.0, False, 24),     # 34 tiles: the first count past the tagged look-back
])
def test_large_token_counts(T, H, E, R, K, mask, fp8, seed):
    idx = random_routing(T, K, E, seed, mask_frac=mask)
    w = random_weights(T, K, seed)
    g_ = torch.Generator().manual_seed(seed + 1)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    y = torch.randn(T * K, H, generator=g_).to(torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R, fp8=fp8)
    o = oracle_run(x, idx, w, y, E, R, fp8=fp8)
    assert g["status"] == 0 and o["status"] == 0
    assert_parity(g, o, fp8=fp8)
    assert np.array_equal(g["out"], o["out"])


def test_zero_tokens():
    E, R, K, H = 8, 2, 2, 64
    idx = torch.zeros(0, K, dtype=torch.int32)
    w = torch.zeros(0, K)
    x = torch.zeros(0, H, dtype=torch.bfloat16)
    y = torch.zeros(0, H, dtype=torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R)
    assert g["status"] == 0
    assert np.all(g["tokens_per_expert"] == 0) and np.all(g["expert_offset"] == 0)
    assert np.all(g["rank_offset"] == 0) and g["n_pairs"] == 0


def test_all_entries_masked():
    T, E, R, K, H = 100, 8, 4, 3, 32
    idx = torch.full((T, K), -1, dtype=torch.int32)
    w = random_weights(T, K, 3)
    x = torch.randn(T, H).to(torch.bfloat16)
    y = torch.randn(T * K, H).to(torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R)
    o = oracle_run(x, idx, w, y, E, R)
    assert_parity(g, o)
    assert np.all(g["out"] == 0)                     # every token sums nothing: +0


def test_fp8_special_blocks():
    """All-zero blocks, signed zeros, a block whose max sits in one element,
    large and tiny magnitudes."""
    T, H, E, R, K = 64, 512, 8, 4, 2
    idx = random_routing(T, K, E, 5)
    x = torch.randn(T, H)
    x[0] = 0.0
    x[1, :128] = -0.0
    x[2, 128:256] = 0.0
    x[2, 200] = -3.0
    x[3] *= 1e4
    x[4] *= 1e-30
    x[5, 256:384] = torch.tensor([1e-38] * 127 + [1.0])
    x = x.to(torch.bfloat16)
    o = oracle_run(x, idx, None, None, E, R, fp8=True)
    for variant in (0, 1, 2, 3, 4):
        g = gpu_run(x, idx, None, None, E, R, fp8=True, variant=variant)
        assert_parity(g, o, fp8=True)


def test_repeated_calls_reuse_workspace():
    """Several layout calls on one workspace (ticket and generation reuse) give
    identical results, also when routings alternate."""
    wl = WORKLOADS["tiny"]
    a = make_inputs(wl, seed=0)
    b = make_inputs(wl, seed=1)
    from combine_moe_dispatch_02_gb300 import ep
    L = ep.Layout(wl.T, wl.K, wl.E, wl.R)
    for inp in (a, b, a, b, a):
        ep.moe_dispatch_layout(inp.topk_idx.cuda(), inp.topk_w.cuda(), wl.E, wl.R, L)
        assert ep.moe_layout_read_status(L) == (0, 0)
        o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R)
        assert np.array_equal(L.recv_slot.cpu().numpy(), o["recv_slot"])
        assert np.array_equal(L.expert_slot.cpu().numpy(), o["expert_slot"])


def test_dispatch_identity_combine_roundtrip_on_gpu():
    """bf16 dispatch -> identity expert (y row = its receive row) -> combine
    with renormalised weights returns x exactly."""
    wl = WORKLOADS["dsv3"]
    inp = make_inputs(wl, with_y=False)
    from combine_moe_dispatch_02_gb300 import ep
    L = ep.Layout(wl.T, wl.K, wl.E, wl.R)
    x = inp.x.cuda()
    w = inp.topk_w.cuda()
    ep.moe_dispatch_layout(inp.topk_idx.cuda(), w, wl.E, wl.R, L)
    recv, _ = ep.alloc_recv(L, wl.H, False)
    ep.moe_dispatch(x, L, False, recv)
    y = recv[L.expert_src_row.long()].contiguous()      # test-only identity expert
    out = torch.empty_like(x)
    ep.moe_combine(y, L, w, out)
    assert ep.moe_layout_read_status(L) == (0, 0)
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))


def test_tuning_variants_agree():
    """Channel counts and stage depths change scheduling only, not results."""
    wl = WORKLOADS["dsv3"].scaled(512)
    inp = make_inputs(wl)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R)
    for ch, st, cb, var in [(1, 2, 0, 1), (4, 3, 2048, 1), (16, 8, 4096, 1), (1000, 0, 0, 1), (100000, 0, 2048, 1),
                            (1, 0, 0, 2), (5, 0, 0, 2), (3000, 0, 0, 2), (0, 4, 0, 2), (7, 4, 0, 2), (0, 8, 0, 2),
                            (5, 2, 0, 2), (1, 0, 0, 4), (7, 0, 0, 4), (100000, 0, 0, 4)]:
        g = gpu_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R, num_channels=ch, stages=st,
                    chunk_bytes=cb, variant=var)
        assert_parity(g, o)
    o8 = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=True)
    for ch, st, cb, var in [(1, 2, 0, 1), (7, 4, 2048, 1), (3, 0, 0, 2), (999, 0, 0, 2),
                            (1, 0, 0, 3), (7, 0, 2048, 3), (999, 0, 4096, 3), (0, 4, 0, 2), (9, 4, 0, 2),
                            (0, 8, 0, 2), (3, 2, 0, 2),
                            (100000, 0, 0, 1), (100000, 0, 2048, 1),     # one item per channel: one stage
                            (1, 0, 0, 4), (7, 0, 0, 4), (100000, 0, 0, 4), (5, 0, 0, 0)]:
        g = gpu_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=True, num_channels=ch, stages=st,
                    chunk_bytes=cb, variant=var)
        assert_parity(g, o8, fp8=True)


def test_over_provisioned_capacity():
    wl = WORKLOADS["tiny"]
    inp = make_inputs(wl)
    cap = wl.capacity + 333
    g = gpu_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R, capacity=cap)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, inp.y, wl.E, wl.R, capacity=cap)
    assert_parity(g, o)


# ---------------------------------------------------------------- MXFP8 dispatch

@pytest.mark.parametrize("name", ["dsv3", "qwen_skew", "ds16_wide"])
def test_mxfp8_parity_full_size(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, with_y=False)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=2)
    for variant in (0, 1, 2, 3, 4):
        g = gpu_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R, fp8=2, variant=variant)
        assert g["status"] == 0
        assert_parity(g, o, fp8=True)


@pytest.mark.parametrize("T,H,E,R,K,seed", [(1, 128, 4, 2, 2, 0), (333, 384, 32, 8, 6, 1), (128, 9216, 16, 4, 4, 2)])
@pytest.mark.parametrize("variant", [1, 2, 3, 4])
def test_mxfp8_edge_cases(T, H, E, R, K, seed, variant):
    idx = random_routing(T, K, E, seed, mask_frac=0.1)
    g_ = torch.Generator().manual_seed(seed + 5)
    x = torch.randn(T, H, generator=g_) * 3
    x[0, :32] = 0.0                                           # zero MX block
    x[0, 32:64] = -0.0                                        # negative zeros: codes 0x80
    if T > 1:
        x[1, :32] = torch.randn(32, generator=g_) * 1e-38     # bf16 subnormal-range block
        x[1, 64] = 3.3e38                                     # near the bf16 maximum
    x = x.to(torch.bfloat16)
    g = gpu_run(x, idx, None, None, E, R, fp8=2, variant=variant)
    o = oracle_run(x, idx, None, None, E, R, fp8=2)
    assert g["status"] == 0
    assert_parity(g, o, fp8=True)


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_wide_dispatch_falls_back_when_only_16_byte_aligned(fmt):
    """The 32-byte vector dispatch (the FP8 / MXFP8 default, variant 4) needs
    32-byte aligned rows; x and the receive buffer at a 16-byte offset take
    the 16-byte kernel instead, with the same results."""
    from combine_moe_dispatch_02_gb300 import ep
    T, H, E, R, K = 300, 1024, 32, 8, 6
    idx = random_routing(T, K, E, 31, mask_frac=0.05)
    g_ = torch.Generator().manual_seed(32)
    x = (torch.randn(T, H, generator=g_) * 2).to(torch.bfloat16)
    o = oracle_run(x, idx, None, None, E, R, fp8=fmt)
    L = ep.Layout(T, K, E, R)
    ep.moe_dispatch_layout(idx.cuda(), None, E, R, L)
    xbuf = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
    x_off = xbuf[8:].view(T, H)                                  # 16 bytes past a 256-byte boundary
    x_off.copy_(x.cuda())
    assert x_off.data_ptr() % 32 == 16
    esz = 2 if fmt == 0 else 1
    rbuf = torch.empty(L.capacity * H * esz + 16, dtype=torch.uint8, device="cuda")
    recv = rbuf[16:].view(torch.bfloat16).view(L.capacity, H) if fmt == 0 else rbuf[16:].view(L.capacity, H)
    assert recv.data_ptr() % 32 == 16
    scales = None if fmt == 0 else ep.alloc_recv(L, H, fmt)[1]
    for variant in (0, 4):
        ep.moe_dispatch(x_off, L, fmt, recv, scales, variant=variant)
        assert ep.moe_layout_read_status(L) == (0, 0)
        n = o["n_pairs"]
        if fmt == 0:
            assert np.array_equal(recv[:n].cpu().view(torch.int16).numpy().view(np.uint16), o["recv_x"])
        else:
            assert np.array_equal(recv[:n].cpu().numpy(), o["recv_q"])
            assert np.array_equal(np.ascontiguousarray(scales[:n].cpu().numpy()).view(np.uint8),
                                  np.ascontiguousarray(o["recv_scales"]).view(np.uint8))


def test_wide_gathers_fall_back_when_only_16_byte_aligned():
    """The 32-byte gather (the dispatch backward's default, the combine's
    variant 4) needs 32-byte aligned rows; inputs and outputs at a 16-byte
    offset take the 16-byte gather instead, with the same results."""
    import oracle
    from combine_moe_dispatch_02_gb300 import ep
    from combine_moe_dispatch_02_gb300.inputs import bf16_bits
    T, H, E, R, K = 300, 1024, 32, 8, 6
    idx = random_routing(T, K, E, 33, mask_frac=0.05)
    w = random_weights(T, K, 33)
    g_ = torch.Generator().manual_seed(34)
    L = ep.Layout(T, K, E, R)
    ep.moe_dispatch_layout(idx.cuda(), w.cuda(), E, R, L)
    Lo = oracle.layout(idx.numpy(), w.numpy(), E, R, None)
    # dispatch backward: grad_recv and grad_x 16 bytes past a 32-byte boundary
    grad_recv = (torch.randn(L.capacity, H, generator=g_) * 2).to(torch.bfloat16)
    gr_buf = torch.empty(L.capacity * H + 8, dtype=torch.bfloat16, device="cuda")
    gr = gr_buf[8:].view(L.capacity, H)
    gr.copy_(grad_recv.cuda())
    gx_buf = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
    gx = gx_buf[8:].view(T, H)
    assert gr.data_ptr() % 32 == 16 and gx.data_ptr() % 32 == 16
    ep.moe_dispatch_backward(gr, L, gx)
    ox, s1 = oracle.dispatch_backward(bf16_bits(grad_recv), Lo.recv_slot)
    assert s1 == 0 and np.array_equal(bf16_bits(gx.cpu()), ox)
    # combine, variant 4: y and out at the same offset
    y = torch.randn(T * K, H, generator=g_).to(torch.bfloat16)
    y_buf = torch.empty(T * K * H + 8, dtype=torch.bfloat16, device="cuda")
    yd = y_buf[8:].view(T * K, H)
    yd.copy_(y.cuda())
    out_buf = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
    out = out_buf[8:].view(T, H)
    ep.moe_combine(yd, L, w.cuda(), out, variant=4)
    oo, s2 = oracle.combine(bf16_bits(y), Lo.expert_slot, w.numpy())
    assert s2 == 0 and np.array_equal(bf16_bits(out.cpu()), oo)
    assert ep.moe_layout_read_status(L) == (0, 0)


@pytest.mark.parametrize("T,E,R,K,tiles", [
    (12000, 32, 8, 8, 47),      # E = 32: eight threads share a column of the tagged look-back
    (30000, 32, 4, 8, 118),
    (32900, 32, 8, 8, 129),     # the last tile count of the tagged look-back for E <= 32
    (33000, 32, 8, 8, 129),
    (33100, 32, 8, 8, 130),     # one more: progress flags
    (16640, 64, 8, 8, 65),      # E = 64: four threads share a column; 65 tiles tagged
    (16641, 64, 8, 8, 66),      # 66: progress flags
])
def test_lookback_tile_counts(T, E, R, K, tiles):
    """Layouts whose scan tiles sum their predecessors with several threads
    per column (few experts), up to and past the last tile count of the
    tagged look-back, against the oracle."""
    import oracle
    from combine_moe_dispatch_02_gb300 import ep
    from harness import LAYOUT_FIELDS
    idx = random_routing(T, K, E, T, mask_frac=0.03)
    w = random_weights(T, K, T)
    L = ep.Layout(T, K, E, R)
    assert L.c.num_tiles == tiles
    ep.moe_dispatch_layout(idx.cuda(), w.cuda(), E, R, L)
    assert ep.moe_layout_read_status(L) == (0, 0)
    o = oracle.layout(idx.numpy(), w.numpy(), E, R, None)
    for f in LAYOUT_FIELDS:
        got = getattr(L, f).cpu().numpy().ravel()
        want = np.asarray(getattr(o, f)).ravel()
        if f == "expert_weight":
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), f
        else:
            assert np.array_equal(got, want), f
