"""Multi-source receive on the GPU against the oracle: S source ranks of Ts
tokens each, one worst-case region of S*Ts rows per destination rank, rows
in (source, token) order.  The layout is compared field by field (integer,
bit-exact); dispatch (bf16, FP8, MXFP8), combine and the backward pair run
unchanged on this layout and are compared on the rows in use."""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, bf16_bits, make_inputs, random_routing, random_weights
from harness import bf16_ulp_diff

pytestmark = pytest.mark.gpu

FIELDS = ("tokens_per_expert", "expert_offset", "tokens_per_rank", "rank_offset", "recv_source_offset",
          "recv_slot", "expert_slot", "recv_src_token", "expert_src_row", "expert_weight")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()
    oracle.build()


def _layout(idx, w, S, E, R, noalloc=False):
    from combine_moe_dispatch_02_gb300 import ep
    T, K = idx.shape
    L = ep.Layout(T, K, E, R, sources=S)
    idx_d = idx.cuda()
    w_d = w.cuda() if w is not None else None
    if noalloc:
        ep.moe_dispatch_layout_noalloc(idx_d, w_d, E, R, L.c)
    else:
        ep.moe_dispatch_layout(idx_d, w_d, E, R, L)
    return L, idx_d, w_d


def _assert_layout_equal(L, o):
    from combine_moe_dispatch_02_gb300 import ep
    assert ep.moe_layout_read_status(L) == (0, 0)
    for f in FIELDS:
        g = getattr(L, f).cpu().numpy()
        assert np.array_equal(g.ravel(), np.asarray(getattr(o, f)).ravel()), f"layout field {f} differs"
    assert L.recv_expert_offset is None


@pytest.mark.parametrize("S,Ts,K,E,R,mask,dups,seed", [
    (1, 1, 1, 1, 1, 0.0, False, 0),             # smallest everything
    (2, 0, 2, 8, 4, 0.0, False, 1),             # empty sources
    (3, 333, 4, 16, 4, 0.1, True, 2),           # ragged, masked, duplicate ids
    (8, 512, 8, 256, 8, 0.0, False, 3),         # DeepSeek-V3 routing, 8 sources
    (5, 700, 6, 64, 32, 0.05, False, 4),        # wide ranks, many tiles
    (32, 64, 8, 64, 64, 0.0, False, 5),         # one expert per rank
    (7, 100, 16, 256, 256, 0.0, False, 6),      # the rank maximum
    (1024, 2, 2, 8, 2, 0.2, False, 7),          # the source maximum
])
def test_layout_parity(S, Ts, K, E, R, mask, dups, seed):
    T = S * Ts
    idx = random_routing(T, K, E, seed, mask_frac=mask, allow_duplicates=dups)
    w = random_weights(T, K, seed)
    L, _, _ = _layout(idx, w, S, E, R)
    o = oracle.layout_sources(idx.numpy(), w.numpy(), S, E, R)
    assert o.status == 0
    _assert_layout_equal(L, o)


def test_layout_parity_noalloc():
    S, Ts, K, E, R = 4, 1000, 8, 256, 8
    idx = random_routing(S * Ts, K, E, 9, mask_frac=0.05)
    w = random_weights(S * Ts, K, 9)
    L, _, _ = _layout(idx, w, S, E, R, noalloc=True)
    _assert_layout_equal(L, oracle.layout_sources(idx.numpy(), w.numpy(), S, E, R))


def test_bad_ids_flagged():
    from combine_moe_dispatch_02_gb300 import ep
    S, Ts, K, E, R = 3, 50, 3, 12, 4
    idx = random_routing(S * Ts, K, E, 2)
    idx[7, 1] = E
    idx[100, 0] = -9
    L, _, _ = _layout(idx, None, S, E, R)
    st, flags = ep.moe_layout_read_status(L)
    assert st == ep.MOE_ERR_EXPERT_ID and flags & ep.MOE_DEVERR_EXPERT_ID
    o = oracle.layout_sources(idx.numpy(), None, S, E, R)
    assert o.status & 2
    for f in ("recv_slot", "expert_slot", "recv_src_token", "recv_source_offset", "tokens_per_rank"):
        assert np.array_equal(getattr(L, f).cpu().numpy().ravel(), np.asarray(getattr(o, f)).ravel()), f


def _used_rows(o):
    return np.nonzero(o.recv_src_token >= 0)[0]


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_dispatch_combine_parity(fmt):
    """DeepSeek-V3 hidden size and routing, 8 sources of 512 tokens."""
    from combine_moe_dispatch_02_gb300 import ep
    wl = WORKLOADS["dsv3"].scaled(4096)
    inp = make_inputs(wl)
    S = 8
    L, idx_d, w_d = _layout(inp.topk_idx, inp.topk_w, S, wl.E, wl.R)
    o = oracle.layout_sources(inp.topk_idx.numpy(), inp.topk_w.numpy(), S, wl.E, wl.R)
    _assert_layout_equal(L, o)
    rows = _used_rows(o)
    x_d = inp.x.cuda()
    recv, scales = ep.alloc_recv(L, wl.H, fmt)
    ep.moe_dispatch(x_d, L, fmt, recv, scales)
    xb = bf16_bits(inp.x)
    rows_d = torch.from_numpy(rows).cuda()
    if fmt == 0:
        rx, st = oracle.dispatch_bf16(xb, o)
        assert st == 0
        assert np.array_equal(bf16_bits(recv[rows_d].cpu()), rx[rows])
    else:
        q, s, st = (oracle.dispatch_fp8 if fmt == 1 else oracle.dispatch_mxfp8)(xb, o)
        assert st == 0
        assert np.array_equal(recv[rows_d].cpu().numpy(), q[rows]), "codes differ"
        gs = np.ascontiguousarray(scales[rows_d].cpu().numpy())
        assert np.array_equal(gs.view(np.uint8), np.ascontiguousarray(s[rows]).view(np.uint8)), "scales differ"
    out = torch.empty_like(x_d)
    ep.moe_combine(inp.y.cuda(), L, w_d, out)
    ref, st = oracle.combine(bf16_bits(inp.y), o.expert_slot, inp.topk_w.numpy())
    assert st == 0
    assert bf16_ulp_diff(bf16_bits(out.cpu()), ref).max() <= 1
    assert ep.moe_layout_read_status(L) == (0, 0)


def test_backward_pair_parity():
    """The backward pair on a multi-source layout: dispatch backward sums each
    token's rows over its destination regions; combine backward as usual."""
    from combine_moe_dispatch_02_gb300 import ep
    S, Ts, H, K, E, R = 4, 200, 256, 6, 32, 8
    T = S * Ts
    idx = random_routing(T, K, E, 13, mask_frac=0.1)
    w = random_weights(T, K, 13)
    L, _, w_d = _layout(idx, w, S, E, R)
    o = oracle.layout_sources(idx.numpy(), w.numpy(), S, E, R)
    _assert_layout_equal(L, o)
    g = torch.Generator().manual_seed(14)
    grad_recv = (torch.randn(R * T, H, generator=g) * 2).to(torch.bfloat16)
    gx = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ep.moe_dispatch_backward(grad_recv.cuda(), L, gx)
    ref, st = oracle.dispatch_backward(bf16_bits(grad_recv), o.recv_slot)
    assert st == 0 and np.array_equal(bf16_bits(gx.cpu()), ref)
    grad_out = torch.randn(T, H, generator=g).to(torch.bfloat16)
    y = torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    gy = torch.full((T * K, H), -1.0, dtype=torch.bfloat16, device="cuda")
    gw = torch.full((T, K), 7.0, dtype=torch.float32, device="cuda")
    ep.moe_combine_backward(grad_out.cuda(), y.cuda(), L, w_d, gy, gw)
    oy0 = np.full((T * K, H), bf16_bits(torch.tensor([-1.0]).to(torch.bfloat16))[0], np.uint16)
    ry, rw, st = oracle.combine_backward(bf16_bits(grad_out), bf16_bits(y), o.expert_slot, w.numpy(), oy0)
    assert st == 0
    assert np.array_equal(bf16_bits(gy.cpu()), ry)
    # fp32 dot products against the fp64 oracle: |error| <= H * 2^-24 * sum |terms| (+ the final rounding)
    go, yy = grad_out.double().numpy(), y.double().numpy()
    es = o.expert_slot
    absdot = np.where(es >= 0, np.abs(go[:, None, :] * yy[np.maximum(es, 0)]).sum(-1), 0.0)
    tol = H * 2.0 ** -24 * absdot + 2.0 ** -24 * np.abs(rw) + 1e-30
    gwn = gw.cpu().double().numpy()
    assert np.all(np.abs(gwn - rw) <= tol)
    assert np.all(gwn[es < 0] == 0.0)
    assert ep.moe_layout_read_status(L) == (0, 0)


def test_full_exchange_shadow_sampled():
    """All eight DeepSeek-V3 ranks' tokens at once (S = 8 sources of 4096
    tokens, R = 8 destinations): the layout exactly; dispatch and combine on
    sampled rows and tokens."""
    from combine_moe_dispatch_02_gb300 import ep
    wl = WORKLOADS["dsv3"]
    S, T = 8, 8 * wl.T
    g = torch.Generator().manual_seed(21)
    parts = [make_inputs(wl, seed=s, with_y=False) for s in range(S)]
    idx = torch.cat([p.topk_idx for p in parts]).contiguous()
    w = torch.cat([p.topk_w for p in parts]).contiguous()
    x = torch.cat([p.x for p in parts]).contiguous()
    L, _, w_d = _layout(idx, w, S, wl.E, wl.R)
    o = oracle.layout_sources(idx.numpy(), w.numpy(), S, wl.E, wl.R)
    _assert_layout_equal(L, o)
    x_d = x.cuda()
    recv, _ = ep.alloc_recv(L, wl.H, 0)
    ep.moe_dispatch(x_d, L, 0, recv)
    rows = _used_rows(o)
    pick = torch.from_numpy(rows[torch.randperm(rows.size, generator=g)[:3000].numpy()])
    got = bf16_bits(recv[pick.cuda()].cpu())
    want = bf16_bits(x[torch.from_numpy(o.recv_src_token[pick.numpy()]).long()])
    assert np.array_equal(got, want)
    del recv
    y_d = torch.randn(T * wl.K, wl.H, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(x_d)
    ep.moe_combine(y_d, L, w_d, out)
    toks = torch.randperm(T, generator=g)[:512]
    es = torch.from_numpy(o.expert_slot)[toks]                     # [n, K]
    sub_rows = es.clamp(min=0).reshape(-1)
    y_sub = y_d[sub_rows.cuda()].cpu()
    es_sub = torch.where(es >= 0, torch.arange(es.numel()).view(es.shape), torch.full_like(es, -1))
    ref, st = oracle.combine(bf16_bits(y_sub), es_sub.numpy().astype(np.int32), w[toks].numpy())
    assert st == 0
    assert bf16_ulp_diff(bf16_bits(out[toks.cuda()].cpu()), ref).max() <= 1
    assert ep.moe_layout_read_status(L) == (0, 0)
