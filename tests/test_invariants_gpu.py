"""Checks of the GPU path that do not go through the oracle's outputs.

1. Layout invariants, computed from the GPU layout alone, on all five
   workloads: every (token, rank) pair with an expert on the rank appears
   exactly once; recv_src_token is the inverse of recv_slot; the counts sum
   to T*K valid entries and to the number of pairs; every slot lies below
   the capacity; receive rows ascend by (primary expert, token) and expert
   rows by (expert, token, k).
2. The E4M3 encoding of every bf16 value in [-448, 448], through the FP8
   dispatch: a 1x128 block whose largest magnitude is exactly 448 has the
   scale RN(448 / 448) = 1, so its codes are E4M3(x) of its other values;
   compared with the oracle's encoder (written from the OCP definition).
   The same for MXFP8: a 1x32 block whose largest magnitude lies in
   [256, 512) has shared exponent 0, so its codes are E4M3(x) as well.
"""
import numpy as np
import pytest
import torch

import oracle
from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("name", ["tiny", "dsv3", "dsv3_fp8", "qwen_skew", "ds16_wide"])
def test_layout_invariants(name):
    from combine_moe_dispatch_02_gb300 import ep
    wl = WORKLOADS[name]
    inp = make_inputs(wl, with_y=False)
    T, K, E, R = wl.T, wl.K, wl.E, wl.R
    m = E // R
    L = ep.Layout(T, K, E, R)
    ep.moe_dispatch_layout(inp.topk_idx.cuda(), inp.topk_w.cuda(), E, R, L)
    assert ep.moe_layout_read_status(L) == (0, 0)
    idx = inp.topk_idx.numpy()
    rs = L.recv_slot.cpu().numpy()
    src = L.recv_src_token.cpu().numpy()
    es = L.expert_slot.cpu().numpy()
    tpe = L.tokens_per_expert.cpu().numpy()
    tpr = L.tokens_per_rank.cpu().numpy()
    eoff = L.expert_offset.cpu().numpy()
    roff = L.rank_offset.cpu().numpy()
    esr = L.expert_src_row.cpu().numpy()
    # which (t, r) pairs exist, straight from the routing
    valid = (idx >= 0) & (idx < E)
    reach = np.zeros((T, R), bool)
    tt, kk = np.nonzero(valid)
    reach[tt, idx[tt, kk] // m] = True
    assert np.array_equal(rs >= 0, reach)
    n_pairs = int(reach.sum())
    assert tpr.sum() == n_pairs == roff[R] and tpe.sum() == valid.sum() == eoff[E]
    used = rs[rs >= 0]
    assert used.max(initial=-1) < L.capacity and np.unique(used).size == used.size == n_pairs
    # recv_src_token inverts recv_slot; rows past the last pair are -1
    t_of, r_of = np.nonzero(rs >= 0)
    assert np.array_equal(src[rs[t_of, r_of]], t_of)
    assert np.all(src[n_pairs:] == -1)
    # receive rows ascend by (primary expert, token): primary = smallest id on the rank
    prim = np.full((T, R), E, np.int64)
    np.minimum.at(prim, (tt, idx[tt, kk] // m), idx[tt, kk])
    key = prim[t_of, r_of] * T + t_of
    order = np.argsort(rs[t_of, r_of])
    assert np.all(np.diff(key[order]) > 0)
    assert np.all(np.diff(roff) >= 0) and np.array_equal(np.diff(roff), tpr)
    # expert rows ascend by (expert, token, k) and point at their token's receive row
    ekey = (idx[tt, kk].astype(np.int64) * T + tt) * K + kk
    eorder = np.argsort(es[tt, kk])
    assert np.all(np.diff(ekey[eorder]) > 0)
    assert np.array_equal(np.sort(es[valid]), np.arange(valid.sum()))
    assert np.array_equal(esr[es[tt, kk]], rs[tt, idx[tt, kk] // m])


def _bf16_values_up_to(limit):
    """Every bf16 bit pattern whose value is finite and at most `limit` in
    magnitude (both signs, both zeros)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    keep = np.isfinite(v) & (np.abs(v) <= limit)
    return bits[keep]


def _dispatch_codes(x_bits, fmt):
    """FP8 / MXFP8 dispatch of the bf16 rows x_bits [T, H] to one rank."""
    from combine_moe_dispatch_02_gb300 import ep
    T, H = x_bits.shape
    x = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).cuda()
    idx = torch.zeros(T, 1, dtype=torch.int32).cuda()
    L = ep.Layout(T, 1, 1, 1)
    ep.moe_dispatch_layout(idx, None, 1, 1, L)
    recv, scales = ep.alloc_recv(L, H, fmt)
    ep.moe_dispatch(x, L, fmt, recv, scales)
    assert ep.moe_layout_read_status(L) == (0, 0)
    rows = L.recv_slot.cpu().numpy()[:, 0]
    return recv.cpu().numpy()[rows], scales.cpu().numpy()[rows]


def test_e4m3_every_bf16_value_through_fp8_dispatch():
    vals = _bf16_values_up_to(448.0)
    per = 127                                                  # slot 0 of each block holds 448
    nblk = (vals.size + per - 1) // per
    padded = np.concatenate([vals, np.zeros(nblk * per - vals.size, np.uint16)]).reshape(nblk, per)
    b448 = np.uint16(0x43E0)                                   # bf16 448.0
    blocks = np.concatenate([np.full((nblk, 1), b448, np.uint16), padded], axis=1)   # [nblk, 128]
    H = 1024                                                   # eight blocks per row
    rows = (nblk + 7) // 8
    blocks = np.concatenate([blocks, np.tile(blocks[:1], (rows * 8 - nblk, 1))])
    x_bits = blocks.reshape(rows, H)
    q, s = _dispatch_codes(x_bits, 1)
    assert np.all(s.view(np.float32) == 1.0)
    got = q.reshape(-1, 128)[:nblk, 1:].reshape(-1)[:vals.size]
    f = torch.from_numpy(vals.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    want = oracle.e4m3_encode_array(f)
    assert np.array_equal(got, want)


def test_mxfp8_e4m3_every_bf16_value_through_mxfp8_dispatch():
    vals = _bf16_values_up_to(448.0)
    per = 31                                                   # slot 0 of each 32-block holds 256
    nblk = (vals.size + per - 1) // per
    padded = np.concatenate([vals, np.zeros(nblk * per - vals.size, np.uint16)]).reshape(nblk, per)
    b256 = np.uint16(0x4380)                                   # bf16 256.0: amax in [256, 512) -> exponent 0
    # values of magnitude above 256 raise the block amax but keep floor(log2) = 8
    blocks = np.concatenate([np.full((nblk, 1), b256, np.uint16), padded], axis=1)    # [nblk, 32]
    H = 1024
    rows = (nblk + 31) // 32
    blocks = np.concatenate([blocks, np.tile(blocks[:1], (rows * 32 - nblk, 1))])
    x_bits = blocks.reshape(rows, H)
    q, s = _dispatch_codes(x_bits, 2)
    assert np.all(s == 127)                                    # E8M0 byte of 2^0
    got = q.reshape(-1, 32)[:nblk, 1:].reshape(-1)[:vals.size]
    f = torch.from_numpy(vals.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    want = oracle.e4m3_encode_array(f)
    assert np.array_equal(got, want)
