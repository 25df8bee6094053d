"""GPU parity of the low-latency (fixed per-expert capacity) dispatch and its
combine against the CPU oracle, bit for bit: slot map, counts, receive rows,
combine output; plus capacity overflow and bad ids reported in the status."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, bf16_bits, make_inputs, random_routing, random_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()
    oracle.build()


def _run(x, idx, w, E, cap, channels=0):
    from combine_moe_dispatch_02_gb300 import ep
    T, H = x.shape
    K = idx.shape[1]
    sentinel = -3.0
    recv = torch.full((E * cap, H), sentinel, dtype=torch.bfloat16, device="cuda")
    tpe = torch.full((E,), -5, dtype=torch.int32, device="cuda")
    slot = torch.full((T, K), -5, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 0x7, dtype=torch.int32, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ep.moe_ll_dispatch(x.cuda(), idx.cuda(), E, cap, recv, tpe, slot, status, num_channels=channels)
    # identity expert: y = recv; combine over the same layout
    ep.moe_ll_combine(recv, slot, w.cuda(), E, cap, out, status)
    torch.cuda.synchronize()
    xb = bf16_bits(x)
    o_recv0 = np.full((E * cap, H), bf16_bits(torch.tensor([sentinel]).to(torch.bfloat16))[0], np.uint16)
    o_recv, o_tpe, o_slot, o_st = oracle.ll_dispatch(xb, idx.numpy(), E, cap, o_recv0)
    o_out, _ = oracle.combine(o_recv, o_slot, w.numpy())
    assert np.array_equal(slot.cpu().numpy(), o_slot)
    assert np.array_equal(tpe.cpu().numpy(), o_tpe)
    assert np.array_equal(bf16_bits(recv.cpu()), o_recv)
    assert np.array_equal(bf16_bits(out.cpu()), o_out)
    return int(status.item()), o_st


@pytest.mark.parametrize("T", [1, 64, 128, 512])
def test_ll_parity_decode_batches(T):
    wl = WORKLOADS["dsv3"].scaled(T)
    inp = make_inputs(wl, with_y=False)
    st, ost = _run(inp.x, inp.topk_idx, inp.topk_w, wl.E, T)
    assert st == 0 and ost == 0


@pytest.mark.parametrize("T,H,E,K,cap,mask,dups,seed,channels", [
    (100, 136, 16, 3, 100, 0.2, True, 1, 0),
    (300, 64, 1024, 8, 32, 0.0, False, 2, 0),
    (200, 64, 300, 6, 64, 0.05, True, 6, 0),     # duplicate ids with 300 experts: equal experts inside one warp chunk
    (256, 8, 4, 16, 1024, 0.1, True, 3, 7),     # few experts, many entries each
    (0, 64, 8, 2, 4, 0.0, False, 4, 0),
    (40, 9224, 16, 4, 16, 0.1, False, 5, 300),    # rows wider than one column group; more channels than tokens
])
def test_ll_edge_cases(T, H, E, K, cap, mask, dups, seed, channels):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups) if T else torch.zeros(0, K, dtype=torch.int32)
    w = random_weights(T, K, seed) if T else torch.zeros(0, K)
    x = torch.randn(T, H).to(torch.bfloat16)
    st, ost = _run(x, idx, w, E, cap, channels)
    assert st == 0 and ost == 0


def test_ll_capacity_overflow_and_bad_ids():
    from combine_moe_dispatch_02_gb300 import ep
    T, K, E, H = 64, 4, 8, 32
    idx = random_routing(T, K, E, 9)
    idx[3, 1] = 99                                     # out of range
    w = random_weights(T, K, 9)
    x = torch.randn(T, H).to(torch.bfloat16)
    st, ost = _run(x, idx, w, E, 5)                    # 5 rows per expert: overflows
    assert st & ep.MOE_DEVERR_CAPACITY and st & ep.MOE_DEVERR_EXPERT_ID
    assert ost & 4 and ost & 2
