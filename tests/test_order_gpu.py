"""Summation order on the GPU, pinned by values that fp32 cannot add in any
other order without a different result: 2^24, 1 and -2^24 give
(2^24 + 1) - 2^24 = 0 when added in that order (2^24 + 1 rounds to the even
2^24), and 1 in any order that adds -2^24 before the 1.

- combine: ascending k (the entry order of the token's routing row), not the
  order of the expert-major rows: expert ids out of k order make the two differ;
- dispatch backward: ascending destination rank."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

B24, ONE, NEG24 = 0x4B80, 0x3F80, 0xCB80           # bf16 2^24, 1, -2^24


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()


def _bf16(bits, shape):
    return torch.from_numpy(np.asarray(bits, np.uint16).astype(np.int16).reshape(shape)).view(torch.bfloat16)


@pytest.mark.parametrize("variant", [0, 1])
def test_combine_sums_in_ascending_k(variant):
    from combine_moe_dispatch_02_gb300 import ep
    H = 16
    idx = torch.tensor([[2, 0, 1]], dtype=torch.int32)   # k = 0, 1, 2 -> experts 2, 0, 1
    w = torch.ones(1, 3, dtype=torch.float32)
    L = ep.Layout(1, 3, 3, 3)
    ep.moe_dispatch_layout(idx.cuda(), w.cuda(), 3, 3, L)
    es = L.expert_slot.cpu().numpy()[0]
    assert list(es) == [2, 0, 1]                        # expert-major rows: (expert, token, k)
    rows = np.zeros((3, H), np.uint16)
    for k, bits in enumerate((B24, ONE, NEG24)):        # the k-th entry's value, at its expert row
        rows[es[k]] = bits
    out = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    ep.moe_combine(_bf16(rows, (3, H)).cuda(), L, w.cuda(), out, variant=variant)
    assert ep.moe_layout_read_status(L) == (0, 0)
    got = out.cpu().view(torch.int16).numpy().astype(np.uint16)
    assert np.all(got == 0x0000), got                   # rows in slot order would sum to 1 (0x3F80)


def test_dispatch_backward_sums_in_ascending_rank():
    from combine_moe_dispatch_02_gb300 import ep
    H = 16
    idx = torch.tensor([[0, 1, 2]], dtype=torch.int32)   # one expert per rank: ranks 0, 1, 2
    L = ep.Layout(1, 3, 3, 3)
    ep.moe_dispatch_layout(idx.cuda(), None, 3, 3, L)
    rs = L.recv_slot.cpu().numpy()[0]
    g = np.zeros((L.capacity, H), np.uint16)
    for r, bits in enumerate((B24, ONE, NEG24)):
        g[rs[r]] = bits
    gx = torch.empty(1, H, dtype=torch.bfloat16, device="cuda")
    ep.moe_dispatch_backward(_bf16(g, (L.capacity, H)).cuda(), L, gx)
    assert ep.moe_layout_read_status(L) == (0, 0)
    got = gx.cpu().view(torch.int16).numpy().astype(np.uint16)
    assert np.all(got == 0x0000), got
