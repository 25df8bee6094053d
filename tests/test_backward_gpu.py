"""GPU parity of the backward pair against the CPU oracle: dispatch backward
and the expert-row gradients bit for bit; the router-weight gradients (fp32
dot products whose summation order is an implementation choice) within the
fp32 error bound of a dot product of length H: |err| <= H * 2^-24 * sum|g*y|
(plus the fp32 rounding of the result)."""
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


def _run(idx, w, E, R, H, seed, capacity=None, **tuning):
    from combine_moe_dispatch_02_gb300 import ep
    T, K = idx.shape
    g = torch.Generator().manual_seed(seed)
    L = ep.Layout(T, K, E, R, capacity)
    idx_d, w_d = idx.cuda(), w.cuda()
    ep.moe_dispatch_layout(idx_d, w_d, E, R, L)
    grad_recv = (torch.randn(L.capacity, H, generator=g) * 2).to(torch.bfloat16)
    grad_out = torch.randn(T, H, generator=g).to(torch.bfloat16)
    y = torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    gx = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    gy = torch.full((T * K, H), -1.0, dtype=torch.bfloat16, device="cuda")
    gw = torch.full((T, K), 7.0, dtype=torch.float32, device="cuda")
    ep.moe_dispatch_backward(grad_recv.cuda(), L, gx, **tuning)
    ep.moe_combine_backward(grad_out.cuda(), y.cuda(), L, w_d, gy, gw)
    st = ep.moe_layout_read_status(L)
    Lo = oracle.layout(idx.numpy(), w.numpy(), E, R, capacity)
    ox, s1 = oracle.dispatch_backward(bf16_bits(grad_recv), Lo.recv_slot)
    oy0 = np.full((T * K, H), bf16_bits(torch.tensor([-1.0]).to(torch.bfloat16))[0], np.uint16)
    oy, ow, s2 = oracle.combine_backward(bf16_bits(grad_out), bf16_bits(y), Lo.expert_slot, w.numpy(), oy0)
    assert st == (0, 0) and s1 == 0 and s2 == 0
    assert np.array_equal(bf16_bits(gx.cpu()), ox), "dispatch backward differs"
    assert np.array_equal(bf16_bits(gy.cpu()), oy), "expert-row gradients differ"
    # router-weight gradients: fp32 dot products against the fp64 oracle
    go, yy = grad_out.double().numpy(), y.double().numpy()
    absdot = np.zeros_like(ow)
    for t in range(T):
        for k in range(K):
            s = Lo.expert_slot[t, k]
            if s >= 0:
                absdot[t, k] = np.abs(go[t] * yy[s]).sum()
    tol = H * 2.0 ** -24 * absdot + 2.0 ** -24 * np.abs(ow) + 1e-30
    gwn = gw.cpu().double().numpy()
    assert np.all(np.abs(gwn - ow) <= tol), float(np.max(np.abs(gwn - ow) / tol))
    assert np.all(gwn[Lo.expert_slot < 0] == 0.0)


@pytest.mark.parametrize("name", ["tiny", "dsv3", "ds16_wide"])
def test_backward_parity_workloads(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, with_y=False)
    _run(inp.topk_idx, inp.topk_w, wl.E, wl.R, wl.H, 3)


@pytest.mark.parametrize("T,H,E,R,K,mask,dups,seed", [
    (1, 8, 1, 1, 1, 0.0, False, 0),
    (517, 136, 16, 4, 3, 0.2, True, 1),
    (300, 64, 64, 32, 12, 0.1, False, 2),     # K > 8: entries in groups of 8; R = 32
    (200, 8200, 16, 4, 4, 0.0, False, 3),
    (400, 784, 64, 64, 8, 0.1, False, 4),     # R = 64: two 32-rank windows; a 272-column last segment
    (257, 2064, 256, 256, 8, 0.0, False, 5),  # R = 256, one expert per rank: eight windows
])
def test_backward_edge_cases(T, H, E, R, K, mask, dups, seed):
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups)
    _run(idx, random_weights(T, K, seed), E, R, H, seed + 10)


@pytest.mark.parametrize("T,H,E,R,K,seed", [
    (4096, 7168, 256, 8, 8, 6),               # DeepSeek-V3 shape: ~5 ranks per token, two batches of rows
    (700, 1024, 64, 32, 6, 7),                # 32 ranks, about six of them per token
    (300, 1040, 16, 4, 2, 8),                 # at most two ranks: one batch; a 16-column last segment
])
def test_dispatch_backward_gather(T, H, E, R, K, seed):
    """The 32-byte gather of the dispatch backward (rows 32-byte aligned,
    hidden % 16 == 0): bit for bit the oracle's add chain."""
    idx = random_routing(T, K, E, seed)
    _run(idx, random_weights(T, K, seed), E, R, H, seed + 10)
