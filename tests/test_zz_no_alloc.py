"""The allocation-free layout entry point, moe_dispatch_layout_noalloc, is for
callers that cannot allocate device memory themselves (a plugin whose host
framework owns every device allocation, a serving loop whose memory is fixed
at start-up).  It must give exactly what moe_dispatch_layout gives.

The caller here owns only the layout's outputs (plain tensors); the struct's
workspace pointer is left NULL, so any use of caller scratch would show.  Two
calls in a row on different routings, each compared with the regular entry
point through the C ABI, bit for bit (the layout is integer work and the
weights are copied).  Collected last so that a failure here never hides
another test; it passes alone in a fresh process as well."""
import ctypes

import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import WORKLOADS, make_inputs, random_routing, random_weights

pytestmark = pytest.mark.gpu

FIELDS = ("tokens_per_expert", "expert_offset", "tokens_per_rank", "rank_offset", "recv_expert_offset",
          "recv_slot", "expert_slot", "recv_src_token", "expert_src_row", "expert_weight")


@pytest.fixture(scope="module")
def ep():
    assert torch.cuda.is_available()
    from combine_moe_dispatch_02_gb300 import build
    from combine_moe_dispatch_02_gb300 import ep as ep_mod
    build.build()
    ep_mod.lib()
    return ep_mod


def _caller_owned_layout(ep, T, K, E, R):
    """A moe_layout with caller-owned output tensors and no workspace."""
    cap = T * min(K, R)
    dev = "cuda"
    out = {
        "tokens_per_expert": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "expert_offset": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "tokens_per_rank": torch.full((R,), -7, dtype=torch.int32, device=dev),
        "rank_offset": torch.full((R + 1,), -7, dtype=torch.int32, device=dev),
        "recv_expert_offset": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "recv_slot": torch.full((T * R,), -7, dtype=torch.int32, device=dev),
        "expert_slot": torch.full((T * K,), -7, dtype=torch.int32, device=dev),
        "recv_src_token": torch.full((cap,), -7, dtype=torch.int32, device=dev),
        "expert_src_row": torch.full((T * K,), -7, dtype=torch.int32, device=dev),
        "expert_weight": torch.full((T * K,), -7.0, dtype=torch.float32, device=dev),
        "status": torch.zeros(1, dtype=torch.int32, device=dev),
    }
    L = ep.moe_layout()
    L.T, L.K, L.E, L.R, L.capacity = T, K, E, R, cap
    for name, t in out.items():
        setattr(L, name, t.data_ptr())
    L.workspace = None
    L.workspace_bytes = 0
    return L, out


def _regular(ep, idx, w, E, R):
    T, K = idx.shape
    Lr = ep.Layout(T, K, E, R)
    ep.moe_dispatch_layout(idx, w, E, R, Lr)
    return {f: getattr(Lr, f).flatten().cpu().numpy() for f in FIELDS}, ep.moe_layout_read_status(Lr)


def _cases():
    wl = WORKLOADS["dsv3"]
    a = make_inputs(wl, with_y=False)
    T, K, E = 1000, 6, 64
    b_idx = random_routing(T, K, E, 3, mask_frac=0.1, allow_duplicates=True)
    return [(a.topk_idx, a.topk_w, wl.E, wl.R), (b_idx, random_weights(T, K, 3), E, 8)]


def test_noalloc_layout_matches_regular_entry_point(ep):
    for idx_h, w_h, E, R in _cases():
        T, K = idx_h.shape
        idx, w = idx_h.cuda(), w_h.cuda()
        want, st = _regular(ep, idx, w, E, R)
        assert st == (0, 0)
        L, out = _caller_owned_layout(ep, T, K, E, R)
        for call in range(2):                                   # two calls in a row
            if call == 1:
                for t in out.values():
                    t.fill_(-7)
                out["status"].zero_()
            ep.moe_dispatch_layout_noalloc(idx, w, E, R, L)
            torch.cuda.synchronize()
            assert int(out["status"].item()) == 0
            for f in FIELDS:
                got = out[f].cpu().numpy()
                if f == "expert_weight":
                    assert np.array_equal(got.view(np.uint32), want[f].view(np.uint32)), (f, call)
                else:
                    assert np.array_equal(got, want[f]), (f, call)
        assert L.workspace is None                              # untouched


def test_noalloc_layout_rejects_sizes_beyond_its_scratch(ep):
    # 8 * T * K bytes of per-entry ranks alone exceed the fixed scratch array
    T, K, E, R = 1 << 18, 8, 64, 8
    L = ep.moe_layout()
    L.T, L.K, L.E, L.R, L.capacity = T, K, E, R, T * min(K, R)
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    for name in FIELDS + ("status",):
        setattr(L, name, dummy.data_ptr())
    st = ep.lib().moe_dispatch_layout_noalloc(ctypes.c_void_p(dummy.data_ptr()), None, E, R, ctypes.byref(L),
                                              None, None)
    assert st == ep.MOE_ERR_UNSUPPORTED


def test_noalloc_call_after_a_timed_out_one_on_another_stream(ep):
    """The shared array after a call whose scan waits ran out (a test hook
    makes the first tile never publish; 20 ms bound): a later call, on a
    second stream ordered after the first by an event, starts clean and
    matches the regular entry point bit for bit."""
    wl = WORKLOADS["dsv3"]
    T = 2048                                               # 32 scan tiles
    inp = make_inputs(wl.scaled(T), with_y=False)
    idx, w = inp.topk_idx.cuda(), inp.topk_w.cuda()
    want, st = _regular(ep, idx, w, wl.E, wl.R)
    assert st == (0, 0)
    L, out = _caller_owned_layout(ep, T, wl.K, wl.E, wl.R)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    ep.moe_dispatch_layout_noalloc(idx, w, wl.E, wl.R, L, stream=s1, wait_timeout_ns=20_000_000,
                                   debug_flags=ep.MOE_DEBUG_STALL_FIRST_TILE)
    done = torch.cuda.Event()
    done.record(s1)
    s2.wait_event(done)
    ep.moe_dispatch_layout_noalloc(idx, w, wl.E, wl.R, L, stream=s2)
    s2.synchronize()
    assert int(out["status"].item()) == 0
    for f in FIELDS:
        got = out[f].cpu().numpy()
        if f == "expert_weight":
            assert np.array_equal(got.view(np.uint32), want[f].view(np.uint32)), f
        else:
            assert np.array_equal(got, want[f]), f
    # and the timed-out call itself reported the timeout
    ep.moe_dispatch_layout_noalloc(idx, w, wl.E, wl.R, L, stream=s1, wait_timeout_ns=20_000_000,
                                   debug_flags=ep.MOE_DEBUG_STALL_FIRST_TILE)
    s1.synchronize()
    assert int(out["status"].item()) & ep.MOE_DEVERR_TIMEOUT
