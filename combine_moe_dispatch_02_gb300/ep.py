"""Thin ctypes binding of libmoe_ep.so (C ABI in include/moe_ep.h).

Argument marshalling only: every step of dispatch layout, dispatch and
combine runs in the library's CUDA kernels.  torch supplies device memory
(tensors) and streams.  There is no fallback: if the library is missing the
import of :func:`lib` raises.

The functions keep the C names (``moe_dispatch_layout``, ``moe_dispatch``,
``moe_combine`` ...) and take torch tensors where the C call takes device
pointers.  :class:`Layout` owns the device memory of one routing layout and
exposes its arrays as tensor views.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_ep.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_CAPACITY = 2
MOE_ERR_TIMEOUT = 3
MOE_ERR_CUDA = 4
MOE_ERR_UNSUPPORTED = 5
MOE_ERR_EXPERT_ID = 6

MOE_DEVERR_EXPERT_ID = 0x1
MOE_DEVERR_CAPACITY = 0x2
MOE_DEVERR_TIMEOUT = 0x4

MOE_DEBUG_STALL_FIRST_TILE = 0x1

MOE_FORMAT_BF16 = 0
MOE_FORMAT_FP8 = 1
MOE_FORMAT_MXFP8 = 2

EXPORTED = ["moe_layout_bytes", "moe_layout_init", "moe_layout_sources_bytes", "moe_layout_init_sources",
            "moe_dispatch_layout", "moe_dispatch_layout_noalloc",
            "moe_dispatch", "moe_dispatch_with_layout", "moe_combine", "moe_dispatch_backward", "moe_combine_backward",
            "moe_ll_dispatch", "moe_ll_combine",
            "moe_layout_read_status", "moe_status_string", "moe_device_sm_count"]

MOE_NOALLOC_SCRATCH_BYTES = 8 << 20
MOE_MAX_SOURCES = 1024


class moe_layout(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("K", ctypes.c_int32), ("E", ctypes.c_int32), ("R", ctypes.c_int32),
        ("capacity", ctypes.c_int64),
        ("tile_tokens", ctypes.c_int32), ("num_tiles", ctypes.c_int32),
        ("num_sources", ctypes.c_int32), ("source_tokens", ctypes.c_int32),
        ("tokens_per_expert", ctypes.c_void_p), ("expert_offset", ctypes.c_void_p),
        ("tokens_per_rank", ctypes.c_void_p), ("rank_offset", ctypes.c_void_p),
        ("recv_expert_offset", ctypes.c_void_p), ("recv_slot", ctypes.c_void_p),
        ("expert_slot", ctypes.c_void_p), ("recv_src_token", ctypes.c_void_p),
        ("expert_src_row", ctypes.c_void_p), ("expert_weight", ctypes.c_void_p),
        ("recv_source_offset", ctypes.c_void_p),
        ("status", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class moe_tuning(ctypes.Structure):
    _fields_ = [("num_channels", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("chunk_bytes", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("wait_timeout_ns", ctypes.c_uint64), ("debug_flags", ctypes.c_uint32),
                ("reserved2", ctypes.c_uint32)]


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {moe_status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_ep.so; raises if it has not been built (no fallback path)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with combine_moe_dispatch_02_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.moe_layout_bytes.restype = ctypes.c_size_t
        L.moe_layout_bytes.argtypes = [i32, i32, i32, i32, i64]
        L.moe_layout_init.restype = ctypes.c_int
        L.moe_layout_init.argtypes = [ctypes.POINTER(moe_layout), i32, i32, i32, i32, i64, P, ctypes.c_size_t]
        L.moe_layout_sources_bytes.restype = ctypes.c_size_t
        L.moe_layout_sources_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.moe_layout_init_sources.restype = ctypes.c_int
        L.moe_layout_init_sources.argtypes = [ctypes.POINTER(moe_layout), i32, i32, i32, i32, i32, P,
                                              ctypes.c_size_t]
        L.moe_dispatch_layout.restype = ctypes.c_int
        L.moe_dispatch_layout.argtypes = [P, P, i32, i32, ctypes.POINTER(moe_layout), P, ctypes.POINTER(moe_tuning)]
        L.moe_dispatch_layout_noalloc.restype = ctypes.c_int
        L.moe_dispatch_layout_noalloc.argtypes = [P, P, i32, i32, ctypes.POINTER(moe_layout), P,
                                                  ctypes.POINTER(moe_tuning)]
        L.moe_dispatch.restype = ctypes.c_int
        L.moe_dispatch.argtypes = [P, i32, ctypes.POINTER(moe_layout), i32, P, P, P,
                                   ctypes.POINTER(moe_tuning)]
        L.moe_dispatch_with_layout.restype = ctypes.c_int
        L.moe_dispatch_with_layout.argtypes = [P, P, i32, i32, ctypes.POINTER(moe_layout), P, i32, i32, P, P, P,
                                               ctypes.POINTER(moe_tuning)]
        L.moe_combine.restype = ctypes.c_int
        L.moe_combine.argtypes = [P, i32, ctypes.POINTER(moe_layout), P, P, P, ctypes.POINTER(moe_tuning)]
        L.moe_dispatch_backward.restype = ctypes.c_int
        L.moe_dispatch_backward.argtypes = [P, i32, ctypes.POINTER(moe_layout), P, P, ctypes.POINTER(moe_tuning)]
        L.moe_combine_backward.restype = ctypes.c_int
        L.moe_combine_backward.argtypes = [P, P, i32, ctypes.POINTER(moe_layout), P, P, P, P,
                                           ctypes.POINTER(moe_tuning)]
        L.moe_ll_dispatch.restype = ctypes.c_int
        L.moe_ll_dispatch.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P, P, ctypes.POINTER(moe_tuning)]
        L.moe_ll_combine.restype = ctypes.c_int
        L.moe_ll_combine.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, ctypes.POINTER(moe_tuning)]
        L.moe_layout_read_status.restype = ctypes.c_int
        L.moe_layout_read_status.argtypes = [ctypes.POINTER(moe_layout), P, ctypes.POINTER(ctypes.c_uint32)]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_device_sm_count.restype = ctypes.c_int32
        L.moe_device_sm_count.argtypes = []
        _lib = L
    return _lib


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoeError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: torch.cuda.Stream | None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _tuning(num_channels=0, stages=0, chunk_bytes=0, variant=0, wait_timeout_ns=0, debug_flags=0):
    if not (num_channels or stages or chunk_bytes or variant or wait_timeout_ns or debug_flags):
        return None
    return ctypes.pointer(moe_tuning(num_channels, stages, chunk_bytes, variant, wait_timeout_ns, debug_flags, 0))


def moe_layout_bytes(T: int, K: int, E: int, R: int, capacity: int) -> int:
    return int(lib().moe_layout_bytes(T, K, E, R, capacity))


def moe_layout_sources_bytes(S: int, source_tokens: int, K: int, E: int, R: int) -> int:
    return int(lib().moe_layout_sources_bytes(S, source_tokens, K, E, R))


class Layout:
    """Device memory and C struct of one routing layout.

    The arrays are views of one zero-initialised uint8 device buffer carved by
    ``moe_layout_init`` (or, with ``sources=S``, by ``moe_layout_init_sources``:
    T = S * Ts tokens from S source ranks, capacity R * T); the buffer stays
    alive as long as this object."""

    def __init__(self, T: int, K: int, E: int, R: int, capacity: int | None = None,
                 device: torch.device | str = "cuda", sources: int = 0):
        self.S = sources
        if sources:
            if capacity is not None or T % sources:
                raise MoeError(MOE_ERR_INVALID_ARG, "multi-source layout: T = S * Ts, capacity R * T")
            capacity = R * T
            nbytes = moe_layout_sources_bytes(sources, T // sources, K, E, R)
        else:
            if capacity is None:
                capacity = T * min(K, R)
            nbytes = moe_layout_bytes(T, K, E, R, capacity)
        if nbytes == 0:
            raise MoeError(MOE_ERR_INVALID_ARG, "moe_layout_bytes")
        self.buf = torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)
        base = self.buf.data_ptr()
        self._off0 = (-base) % 256                      # 256-byte aligned start
        self.c = moe_layout()
        if sources:
            _check(lib().moe_layout_init_sources(ctypes.byref(self.c), sources, T // sources, K, E, R,
                                                 ctypes.c_void_p(base + self._off0), nbytes),
                   "moe_layout_init_sources")
        else:
            _check(lib().moe_layout_init(ctypes.byref(self.c), T, K, E, R, capacity,
                                         ctypes.c_void_p(base + self._off0), nbytes), "moe_layout_init")
        self.T, self.K, self.E, self.R, self.capacity = T, K, E, R, capacity

    def _view(self, field: str, count: int, dtype=torch.int32) -> torch.Tensor:
        addr = getattr(self.c, field)
        off = addr - self.buf.data_ptr()
        esz = torch.empty(0, dtype=dtype).element_size()
        return self.buf[off:off + count * esz].view(dtype)

    @property
    def tokens_per_expert(self): return self._view("tokens_per_expert", self.E)
    @property
    def expert_offset(self): return self._view("expert_offset", self.E + 1)
    @property
    def tokens_per_rank(self): return self._view("tokens_per_rank", self.R)
    @property
    def rank_offset(self): return self._view("rank_offset", self.R + 1)
    @property
    def recv_expert_offset(self):
        return None if self.S else self._view("recv_expert_offset", self.E + 1)
    @property
    def recv_source_offset(self):
        return self._view("recv_source_offset", self.R * (self.S + 1)).view(self.R, self.S + 1) if self.S else None
    @property
    def recv_slot(self): return self._view("recv_slot", self.T * self.R).view(self.T, self.R)
    @property
    def expert_slot(self): return self._view("expert_slot", self.T * self.K).view(self.T, self.K)
    @property
    def recv_src_token(self): return self._view("recv_src_token", self.capacity)
    @property
    def expert_src_row(self): return self._view("expert_src_row", self.T * self.K)
    @property
    def expert_weight(self): return self._view("expert_weight", self.T * self.K, torch.float32)
    @property
    def status_word(self): return self._view("status", 1)


def moe_dispatch_layout(topk_idx: torch.Tensor, topk_w: torch.Tensor | None, num_experts: int, num_ranks: int,
                        L: Layout, stream=None, **tuning) -> None:
    assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous()
    assert topk_w is None or (topk_w.dtype == torch.float32 and topk_w.is_contiguous())
    _check(lib().moe_dispatch_layout(_ptr(topk_idx), _ptr(topk_w), num_experts, num_ranks, ctypes.byref(L.c),
                                     _stream(stream), _tuning(**tuning)), "moe_dispatch_layout")


def moe_dispatch_layout_noalloc(topk_idx: torch.Tensor, topk_w: torch.Tensor | None, num_experts: int,
                                num_ranks: int, L: moe_layout, stream=None, **tuning) -> None:
    """The allocation-free layout entry point.  `L` is a plain moe_layout whose
    sizes, output pointers and status pointer the caller has filled in; its
    workspace fields are not used."""
    assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous()
    assert topk_w is None or (topk_w.dtype == torch.float32 and topk_w.is_contiguous())
    _check(lib().moe_dispatch_layout_noalloc(_ptr(topk_idx), _ptr(topk_w), num_experts, num_ranks, ctypes.byref(L),
                                             _stream(stream), _tuning(**tuning)), "moe_dispatch_layout_noalloc")


def moe_dispatch(x: torch.Tensor, L: Layout, fmt, recv_x: torch.Tensor,
                 recv_scales: torch.Tensor | None = None, stream=None, **tuning) -> None:
    """fmt: MOE_FORMAT_BF16 / MOE_FORMAT_FP8 / MOE_FORMAT_MXFP8 (False / True
    stand for bf16 / FP8)."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    assert recv_x.is_contiguous() and (recv_scales is None or recv_scales.is_contiguous())
    _check(lib().moe_dispatch(_ptr(x), x.shape[-1], ctypes.byref(L.c), int(fmt), _ptr(recv_x),
                              _ptr(recv_scales), _stream(stream), _tuning(**tuning)), "moe_dispatch")


def moe_dispatch_with_layout(topk_idx: torch.Tensor, topk_w: torch.Tensor | None, num_experts: int,
                             num_ranks: int, L: Layout, x: torch.Tensor, fmt, recv_x: torch.Tensor,
                             recv_scales: torch.Tensor | None = None, stream=None, **tuning) -> None:
    """moe_dispatch_layout followed by moe_dispatch in one call (the dispatch
    may read x while the layout is computed)."""
    assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous()
    assert topk_w is None or (topk_w.dtype == torch.float32 and topk_w.is_contiguous())
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    assert recv_x.is_contiguous() and (recv_scales is None or recv_scales.is_contiguous())
    _check(lib().moe_dispatch_with_layout(_ptr(topk_idx), _ptr(topk_w), num_experts, num_ranks, ctypes.byref(L.c),
                                          _ptr(x), x.shape[-1], int(fmt), _ptr(recv_x), _ptr(recv_scales),
                                          _stream(stream), _tuning(**tuning)), "moe_dispatch_with_layout")


def moe_combine(y: torch.Tensor, L: Layout, topk_w: torch.Tensor, out: torch.Tensor, stream=None,
                **tuning) -> None:
    assert y.dtype == torch.bfloat16 and y.is_contiguous() and out.is_contiguous()
    assert topk_w.dtype == torch.float32 and topk_w.is_contiguous()
    _check(lib().moe_combine(_ptr(y), y.shape[-1], ctypes.byref(L.c), _ptr(topk_w), _ptr(out),
                             _stream(stream), _tuning(**tuning)), "moe_combine")


def moe_dispatch_backward(grad_recv: torch.Tensor, L: Layout, grad_x: torch.Tensor, stream=None, **tuning) -> None:
    assert grad_recv.dtype == torch.bfloat16 and grad_recv.is_contiguous() and grad_x.is_contiguous()
    _check(lib().moe_dispatch_backward(_ptr(grad_recv), grad_recv.shape[-1], ctypes.byref(L.c), _ptr(grad_x),
                                       _stream(stream), _tuning(**tuning)), "moe_dispatch_backward")


def moe_combine_backward(grad_out: torch.Tensor, y: torch.Tensor, L: Layout, topk_w: torch.Tensor,
                         grad_y: torch.Tensor, grad_w: torch.Tensor, stream=None, **tuning) -> None:
    assert grad_out.dtype == torch.bfloat16 and y.dtype == torch.bfloat16 and topk_w.dtype == torch.float32
    assert all(t.is_contiguous() for t in (grad_out, y, topk_w, grad_y, grad_w))
    _check(lib().moe_combine_backward(_ptr(grad_out), _ptr(y), y.shape[-1], ctypes.byref(L.c), _ptr(topk_w),
                                      _ptr(grad_y), _ptr(grad_w), _stream(stream), _tuning(**tuning)),
           "moe_combine_backward")


def moe_ll_dispatch(x: torch.Tensor, topk_idx: torch.Tensor, E: int, cap: int, recv: torch.Tensor,
                    tokens_per_expert: torch.Tensor, ll_slot: torch.Tensor, status: torch.Tensor, stream=None,
                    **tuning) -> None:
    T, H = x.shape
    K = topk_idx.shape[1]
    assert x.dtype == torch.bfloat16 and topk_idx.dtype == torch.int32
    assert all(t.is_contiguous() for t in (x, topk_idx, recv, tokens_per_expert, ll_slot, status))
    _check(lib().moe_ll_dispatch(_ptr(x), _ptr(topk_idx), T, K, E, H, cap, _ptr(recv), _ptr(tokens_per_expert),
                                 _ptr(ll_slot), _ptr(status), _stream(stream), _tuning(**tuning)), "moe_ll_dispatch")


def moe_ll_combine(y: torch.Tensor, ll_slot: torch.Tensor, topk_w: torch.Tensor, E: int, cap: int,
                   out: torch.Tensor, status: torch.Tensor, stream=None, **tuning) -> None:
    T, K = ll_slot.shape
    H = y.shape[-1]
    assert y.dtype == torch.bfloat16 and topk_w.dtype == torch.float32
    assert all(t.is_contiguous() for t in (y, ll_slot, topk_w, out, status))
    _check(lib().moe_ll_combine(_ptr(y), _ptr(ll_slot), _ptr(topk_w), T, K, E, H, cap, _ptr(out), _ptr(status),
                                _stream(stream), _tuning(**tuning)), "moe_ll_combine")


def moe_layout_read_status(L: Layout, stream=None) -> tuple[int, int]:
    """Synchronises the stream; returns (status, raw MOE_DEVERR_* flags)."""
    flags = ctypes.c_uint32(0)
    st = lib().moe_layout_read_status(ctypes.byref(L.c), _stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def moe_device_sm_count() -> int:
    return int(lib().moe_device_sm_count())


# ------------------------------------------------------------ conveniences

def alloc_recv(L: Layout, hidden: int, fmt, device="cuda"):
    """Receive buffers for moe_dispatch: (recv_x, recv_scales or None)."""
    fmt = int(fmt)
    if fmt == MOE_FORMAT_FP8:
        return (torch.empty(L.capacity, hidden, dtype=torch.uint8, device=device),
                torch.empty(L.capacity, hidden // 128, dtype=torch.float32, device=device))
    if fmt == MOE_FORMAT_MXFP8:
        return (torch.empty(L.capacity, hidden, dtype=torch.uint8, device=device),
                torch.empty(L.capacity, hidden // 32, dtype=torch.uint8, device=device))
    return torch.empty(L.capacity, hidden, dtype=torch.bfloat16, device=device), None
