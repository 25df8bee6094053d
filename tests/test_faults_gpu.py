"""Failure handling on the GPU without faulting it: bad expert ids and a
bounded wait that is made to run out (a scan tile that never publishes)
come back as status bits; host argument errors come back as status codes
before anything is enqueued.  Nothing here traps, faults or hangs."""
import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing, random_weights
from harness import assert_parity, gpu_run, oracle_run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()


def test_out_of_range_expert_ids_are_flagged_and_masked():
    from combine_moe_dispatch_02_gb300 import ep
    T, H, E, R, K = 300, 64, 16, 4, 3
    idx = random_routing(T, K, E, 1)
    idx[5, 1] = 16          # == E
    idx[77, 0] = -7         # below the mask value
    idx[299, 2] = 1 << 30
    w = random_weights(T, K, 1)
    x = torch.randn(T, H).to(torch.bfloat16)
    y = torch.randn(T * K, H).to(torch.bfloat16)
    g = gpu_run(x, idx, w, y, E, R)
    o = oracle_run(x, idx, w, y, E, R)
    assert g["status"] == ep.MOE_ERR_EXPERT_ID and g["flags"] & ep.MOE_DEVERR_EXPERT_ID
    assert o["status"] & 2                              # the oracle flags them too
    assert_parity(g, o)                                  # both treat them as masked


def test_scan_wait_timeout_is_reported_and_recoverable():
    from combine_moe_dispatch_02_gb300 import ep
    wl = WORKLOADS["dsv3"]                               # 32 scan tiles
    inp = make_inputs(wl.scaled(2048), with_y=False)
    L = ep.Layout(2048, wl.K, wl.E, wl.R)
    assert L.c.num_tiles >= 2
    idx, w = inp.topk_idx.cuda(), inp.topk_w.cuda()
    ep.moe_dispatch_layout(idx, w, wl.E, wl.R, L, wait_timeout_ns=20_000_000,
                           debug_flags=ep.MOE_DEBUG_STALL_FIRST_TILE)
    st, flags = ep.moe_layout_read_status(L)
    assert st == ep.MOE_ERR_TIMEOUT and flags & ep.MOE_DEVERR_TIMEOUT
    # the context is intact and the next call on the same workspace is healthy
    ep.moe_dispatch_layout(idx, w, wl.E, wl.R, L)
    assert ep.moe_layout_read_status(L) == (0, 0)
    o = oracle_run(inp.x, inp.topk_idx, inp.topk_w, None, wl.E, wl.R)
    assert np.array_equal(L.recv_slot.cpu().numpy(), o["recv_slot"])
    assert np.array_equal(L.expert_slot.cpu().numpy(), o["expert_slot"])


def test_host_argument_errors():
    from combine_moe_dispatch_02_gb300 import ep
    T, H, E, R, K = 64, 256, 8, 4, 2
    L = ep.Layout(T, K, E, R)
    idx = random_routing(T, K, E, 0).cuda()
    w = random_weights(T, K, 0).cuda()
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    recv, _ = ep.alloc_recv(L, H, False)
    with pytest.raises(ep.MoeError) as e:
        ep.moe_dispatch_layout(idx, w, E + 1, R, L)
    assert e.value.status == ep.MOE_ERR_INVALID_ARG
    ep.moe_dispatch_layout(idx, w, E, R, L)
    # misaligned source
    xb = torch.empty(T * H + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ep.MoeError):
        ep.moe_dispatch(xb[1:1 + T * H].view(T, H), L, False, recv)
    # hidden not a multiple of 8
    with pytest.raises(ep.MoeError):
        ep.moe_dispatch(torch.zeros(T, 12, dtype=torch.bfloat16, device="cuda"), L, False, recv)
    # FP8 needs hidden % 128 == 0 and a scale buffer
    with pytest.raises(ep.MoeError):
        ep.moe_dispatch(torch.zeros(T, 64, dtype=torch.bfloat16, device="cuda"), L, True,
                        torch.empty(L.capacity, 64, dtype=torch.uint8, device="cuda"),
                        torch.empty(L.capacity, 1, device="cuda"))
    with pytest.raises(ep.MoeError):
        ep.moe_dispatch(x, L, True, torch.empty(L.capacity, H, dtype=torch.uint8, device="cuda"), None)
    # bf16 dispatch must not get a scale buffer
    with pytest.raises(ep.MoeError):
        ep.moe_dispatch(x, L, False, recv, torch.empty(L.capacity, 2, device="cuda"))
    assert ep.moe_layout_read_status(L) == (0, 0)
