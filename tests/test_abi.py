"""The C-ABI library builds, loads and exports every function declared in
include/moe_ep.h; host-only entry points validate their arguments.  No
GPU and no compute call: the calls below return before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from combine_moe_dispatch_02_gb300 import build, ep
    build.build()
    return ep.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_operator_calls():
    names = _declared_functions()
    for n in ("moe_dispatch_layout", "moe_dispatch", "moe_combine", "moe_layout_init", "moe_layout_bytes",
              "moe_layout_read_status", "moe_status_string"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_binding_names_match_header(lib):
    from combine_moe_dispatch_02_gb300 import ep
    assert sorted(ep.EXPORTED) == _declared_functions()


def test_layout_bytes_and_init_validation(lib):
    from combine_moe_dispatch_02_gb300 import ep
    n = ep.moe_layout_bytes(4096, 8, 256, 8, 4096 * 8)
    assert n > 4 * (4096 * 8 * 4)           # holds at least recv_slot + expert_slot + ...
    assert ep.moe_layout_bytes(16, 2, 6, 4, 32) == 0            # E % R != 0
    L = ep.moe_layout()
    fake = ctypes.c_void_p(1 << 20)                               # never dereferenced on the host
    init = lib.moe_layout_init
    assert init(ctypes.byref(L), 16, 2, 8, 4, 32, fake, n) == ep.MOE_OK
    assert L.T == 16 and L.num_tiles >= 1 and L.capacity == 32
    assert init(ctypes.byref(L), 16, 2, 8, 4, 31, fake, n) == ep.MOE_ERR_INVALID_ARG         # capacity < T*min(K,R)
    assert init(ctypes.byref(L), 16, 2, 8, 4, 32, ctypes.c_void_p((1 << 20) + 16), n) == ep.MOE_ERR_INVALID_ARG
    assert init(ctypes.byref(L), 16, 2, 8, 4, 32, fake, 10) == ep.MOE_ERR_INVALID_ARG        # too small
    assert init(ctypes.byref(L), 16, 33, 64, 4, 16 * 4, fake, 1 << 30) == ep.MOE_ERR_UNSUPPORTED  # K > 32
    assert init(ctypes.byref(L), 16, 2, 2048, 4, 32, fake, 1 << 30) == ep.MOE_ERR_UNSUPPORTED    # E > 1024


def test_operator_calls_reject_bad_arguments_on_the_host(lib):
    from combine_moe_dispatch_02_gb300 import ep
    L = ep.moe_layout()
    n = ep.moe_layout_bytes(16, 2, 8, 4, 32)
    assert lib.moe_layout_init(ctypes.byref(L), 16, 2, 8, 4, 32, ctypes.c_void_p(1 << 20), n) == ep.MOE_OK
    p = ctypes.c_void_p(1 << 21)
    # expert / rank counts that do not match the layout
    assert lib.moe_dispatch_layout(p, p, 16, 4, ctypes.byref(L), None, None) == ep.MOE_ERR_INVALID_ARG
    # hidden not a multiple of 8; misaligned rows; fp8 with hidden % 128 != 0
    assert lib.moe_dispatch(p, 12, ctypes.byref(L), 0, p, None, None, None) == ep.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(ctypes.c_void_p((1 << 21) + 2), 64, ctypes.byref(L), 0, p, None, None, None) \
        == ep.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(p, 64, ctypes.byref(L), 1, p, p, None, None) == ep.MOE_ERR_INVALID_ARG
    assert lib.moe_dispatch(p, 64, ctypes.byref(L), 2, p, p, None, None) == ep.MOE_ERR_INVALID_ARG   # MXFP8 needs hidden % 128
    assert lib.moe_dispatch(p, 128, ctypes.byref(L), 3, p, p, None, None) == ep.MOE_ERR_INVALID_ARG  # no such format
    assert lib.moe_dispatch(p, 128, ctypes.byref(L), 2, p, None, None, None) == ep.MOE_ERR_INVALID_ARG  # scales missing
    assert lib.moe_combine(p, 12, ctypes.byref(L), p, p, None, None) == ep.MOE_ERR_INVALID_ARG
    assert lib.moe_combine(None, 64, ctypes.byref(L), p, p, None, None) == ep.MOE_ERR_INVALID_ARG
    # layout + dispatch in one call: the checks of both (nothing is enqueued when either fails)
    with_layout = lib.moe_dispatch_with_layout
    assert with_layout(p, p, 16, 4, ctypes.byref(L), p, 64, 0, p, None, None, None) == ep.MOE_ERR_INVALID_ARG  # E
    assert with_layout(p, p, 8, 4, ctypes.byref(L), p, 12, 0, p, None, None, None) == ep.MOE_ERR_INVALID_ARG   # hidden
    assert with_layout(p, p, 8, 4, ctypes.byref(L), p, 64, 1, p, p, None, None) == ep.MOE_ERR_INVALID_ARG     # fp8 hidden
    assert with_layout(None, p, 8, 4, ctypes.byref(L), p, 64, 0, p, None, None, None) == ep.MOE_ERR_INVALID_ARG  # ids
    assert with_layout(p, p, 8, 4, ctypes.byref(L), p, 64, 0, p, None, None,
                       ctypes.byref(ep.moe_tuning(variant=5))) == ep.MOE_ERR_INVALID_ARG


def test_more_calls_reject_bad_arguments_on_the_host(lib):
    """Refusals that happen before anything is enqueued (no GPU needed): the
    scale buffer rules, tuning outside its ranges, the backward pair and the
    low-latency calls."""
    from combine_moe_dispatch_02_gb300 import ep
    INVALID, UNSUPPORTED = ep.MOE_ERR_INVALID_ARG, ep.MOE_ERR_UNSUPPORTED
    L = ep.moe_layout()
    n = ep.moe_layout_bytes(16, 2, 8, 4, 32)
    assert lib.moe_layout_init(ctypes.byref(L), 16, 2, 8, 4, 32, ctypes.c_void_p(1 << 20), n) == ep.MOE_OK
    Lp = ctypes.byref(L)
    p = ctypes.c_void_p(1 << 21)
    off4 = ctypes.c_void_p((1 << 21) + 4)        # 4-byte but not 16-byte aligned
    off2 = ctypes.c_void_p((1 << 21) + 2)        # not even 4-byte aligned
    # a bf16 dispatch takes no scale buffer; FP8 scale words must be 4-byte aligned
    assert lib.moe_dispatch(p, 128, Lp, 0, p, p, None, None) == INVALID
    assert lib.moe_dispatch(p, 128, Lp, 1, p, off2, None, None) == INVALID
    # tuning outside its ranges
    for t in (ep.moe_tuning(stages=1), ep.moe_tuning(stages=9), ep.moe_tuning(chunk_bytes=100),
              ep.moe_tuning(chunk_bytes=384), ep.moe_tuning(variant=5), ep.moe_tuning(num_channels=-1)):
        assert lib.moe_dispatch(p, 128, Lp, 0, p, None, None, ctypes.byref(t)) == INVALID
    assert lib.moe_combine(p, 64, Lp, p, p, None, ctypes.byref(ep.moe_tuning(variant=5))) == INVALID
    # backward pair
    assert lib.moe_dispatch_backward(p, 12, Lp, p, None, None) == INVALID              # hidden % 8
    assert lib.moe_dispatch_backward(off4, 64, Lp, p, None, None) == INVALID           # misaligned rows
    assert lib.moe_combine_backward(p, p, 64, Lp, p, p, None, None, None) == INVALID   # no grad_w
    assert lib.moe_combine_backward(p, p, 64, Lp, off2, p, p, None, None) == INVALID   # misaligned weights
    # low-latency layout
    assert lib.moe_ll_dispatch(p, p, 16, 33, 8, 64, 4, p, p, p, p, None, None) == UNSUPPORTED    # K > 32
    assert lib.moe_ll_dispatch(p, p, 1024, 8, 8, 64, 4, p, p, p, p, None, None) == UNSUPPORTED   # T*K > 4096
    assert lib.moe_ll_dispatch(p, p, 16, 2, 8, 12, 4, p, p, p, p, None, None) == INVALID         # hidden % 8
    assert lib.moe_ll_dispatch(p, p, 16, 2, 8, 64, 4, p, None, p, p, None, None) == INVALID      # no counts
    assert lib.moe_ll_combine(p, p, p, 16, 2, 8, 64, 4, p, None, None, None) == INVALID          # no status
    assert lib.moe_ll_combine(p, p, off2, 16, 2, 8, 64, 4, p, p, None, None) == INVALID         # misaligned w


def test_status_strings(lib):
    from combine_moe_dispatch_02_gb300 import ep
    for s in range(7):
        assert ep.moe_status_string(s) and ep.moe_status_string(s) != "unknown status"


def test_multi_source_layout_init_validation(lib):
    from combine_moe_dispatch_02_gb300 import ep
    S, Ts, K, E, R = 4, 100, 3, 8, 4
    n = ep.moe_layout_sources_bytes(S, Ts, K, E, R)
    assert n > 4 * (S * Ts * R)                                   # recv_src_token alone is R * T ints
    assert ep.moe_layout_sources_bytes(0, Ts, K, E, R) == 0
    assert ep.moe_layout_sources_bytes(ep.MOE_MAX_SOURCES + 1, 1, K, E, R) == 0
    assert ep.moe_layout_sources_bytes(S, Ts, K, 6, R) == 0          # E % R != 0
    assert ep.moe_layout_sources_bytes(1024, 1 << 20, 1, 256, 256) == 0   # R * T overflows int32
    L = ep.moe_layout()
    fake = ctypes.c_void_p(1 << 20)                               # never dereferenced on the host
    init = lib.moe_layout_init_sources
    assert init(ctypes.byref(L), S, Ts, K, E, R, fake, n) == ep.MOE_OK
    assert (L.T, L.capacity, L.num_sources, L.source_tokens) == (S * Ts, R * S * Ts, S, Ts)
    assert L.recv_expert_offset is None and L.recv_source_offset
    assert init(ctypes.byref(L), S, Ts, K, E, R, fake, n - 1) == ep.MOE_ERR_INVALID_ARG
    assert init(ctypes.byref(L), 0, Ts, K, E, R, fake, n) == ep.MOE_ERR_INVALID_ARG
    assert init(ctypes.byref(L), S, Ts, 33, 64, R, fake, 1 << 30) == ep.MOE_ERR_UNSUPPORTED
    # the single-source init records no sources
    M = ep.moe_layout()
    assert lib.moe_layout_init(ctypes.byref(M), 16, 2, 8, 4, 32, fake, ep.moe_layout_bytes(16, 2, 8, 4, 32)) == ep.MOE_OK
    assert M.num_sources == 0 and M.source_tokens == 16 and M.recv_source_offset is None


def test_layout_kind_fields_must_agree(lib):
    """moe_dispatch_layout rejects a struct whose layout-kind fields disagree
    before anything is enqueued."""
    from combine_moe_dispatch_02_gb300 import ep
    S, Ts, K, E, R = 2, 16, 2, 8, 4
    L = ep.moe_layout()
    fake = ctypes.c_void_p(1 << 20)
    assert lib.moe_layout_init_sources(ctypes.byref(L), S, Ts, K, E, R, fake,
                                       ep.moe_layout_sources_bytes(S, Ts, K, E, R)) == ep.MOE_OK
    p = ctypes.c_void_p(1 << 21)
    for field, value in (("recv_source_offset", None), ("source_tokens", Ts + 1), ("capacity", R * S * Ts - 1),
                         ("num_sources", -1)):
        bad = ep.moe_layout.from_buffer_copy(L)
        setattr(bad, field, value)
        assert lib.moe_dispatch_layout(p, p, E, R, ctypes.byref(bad), None, None) == ep.MOE_ERR_INVALID_ARG, field
        assert lib.moe_dispatch_layout_noalloc(p, p, E, R, ctypes.byref(bad), None, None) == ep.MOE_ERR_INVALID_ARG
    single = ep.moe_layout()
    assert lib.moe_layout_init(ctypes.byref(single), 16, 2, 8, 4, 32, fake, ep.moe_layout_bytes(16, 2, 8, 4, 32)) == 0
    single.recv_expert_offset = None
    assert lib.moe_dispatch_layout(p, p, 8, 4, ctypes.byref(single), None, None) == ep.MOE_ERR_INVALID_ARG
