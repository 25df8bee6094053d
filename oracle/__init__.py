"""CPU oracle for MoE token dispatch / combine -- TEST INFRASTRUCTURE ONLY.

A plain single-threaded C implementation (``moe_oracle.c``) of what the
dispatch-layout, dispatch (bf16 / FP8 E4M3 with 1x128 fp32 scales) and
combine operators compute, wrapped here with ctypes over numpy arrays.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The CUDA library never links or calls
it, and this package imports nothing from the product package.

The operators are the dispatch and combine of Hybrid-EP / DeepEP ("Inside the
Nebius + PyTorch DeepSeek V3 recipe", section "Mixture-of-experts and wide
expert parallelism"; Hybrid-EP news article, section "Technical Structure").
The orderings, the FP8 recipe and the combine arithmetic are readings of
those pages stated in ``moe_oracle.h``.  Every function is pinned by tests
that compute their expected values without calling it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

ERR_ARG = 1
ERR_EXPERT_ID = 2
ERR_CAPACITY = 4


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "moe_oracle.h"))):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def set_library(cdll: ctypes.CDLL | None) -> None:
    """Route every oracle call to another build of moe_oracle.c (the mutation
    tests use this to check that the pins catch planted mistakes); None
    restores the default library."""
    global _lib
    _lib = cdll


def load(path: str) -> ctypes.CDLL:
    """Load a build of moe_oracle.c and declare its signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    L.moe_ref_bf16_encode.restype = ctypes.c_uint16
    L.moe_ref_bf16_encode.argtypes = [ctypes.c_float]
    L.moe_ref_bf16_decode.restype = ctypes.c_float
    L.moe_ref_bf16_decode.argtypes = [ctypes.c_uint16]
    L.moe_ref_e4m3_encode.restype = ctypes.c_uint8
    L.moe_ref_e4m3_encode.argtypes = [ctypes.c_float]
    L.moe_ref_e4m3_decode.restype = ctypes.c_float
    L.moe_ref_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.moe_ref_layout.restype = ctypes.c_int
    L.moe_ref_layout.argtypes = [P, P, i32, i32, i32, i32, i64] + [P] * 10
    L.moe_ref_layout_sources.restype = ctypes.c_int
    L.moe_ref_layout_sources.argtypes = [P, P, i32, i32, i32, i32, i32] + [P] * 10
    L.moe_ref_dispatch_bf16.restype = ctypes.c_int
    L.moe_ref_dispatch_bf16.argtypes = [P, i32, i32, i32, P, i64, P]
    L.moe_ref_dispatch_fp8.restype = ctypes.c_int
    L.moe_ref_dispatch_fp8.argtypes = [P, i32, i32, i32, P, i64, P, P]
    L.moe_ref_dispatch_mxfp8.restype = ctypes.c_int
    L.moe_ref_dispatch_mxfp8.argtypes = [P, i32, i32, i32, P, i64, P, P]
    L.moe_ref_combine.restype = ctypes.c_int
    L.moe_ref_combine.argtypes = [P, i64, i32, i32, i32, P, P, P]
    L.moe_ref_ll_dispatch.restype = ctypes.c_int
    L.moe_ref_ll_dispatch.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P]
    L.moe_ref_dispatch_backward.restype = ctypes.c_int
    L.moe_ref_dispatch_backward.argtypes = [P, i64, i32, i32, i32, P, P]
    L.moe_ref_combine_backward.restype = ctypes.c_int
    L.moe_ref_combine_backward.argtypes = [P, P, i64, i32, i32, i32, P, P, P, P]
    return L


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


# ------------------------------------------------------------------ codecs

def bf16_encode(v: float) -> int:
    return int(lib().moe_ref_bf16_encode(float(v)))


def bf16_decode(b: int) -> float:
    return float(lib().moe_ref_bf16_decode(int(b)))


def e4m3_encode(v: float) -> int:
    return int(lib().moe_ref_e4m3_encode(float(v)))


def e4m3_decode(q: int) -> float:
    return float(lib().moe_ref_e4m3_decode(int(q)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    """Vector form of :func:`e4m3_encode` (a loop over the C scalar routine)."""
    f = lib().moe_ref_e4m3_encode
    flat = np.ascontiguousarray(v, dtype=np.float32).ravel()
    return np.fromiter((f(float(x)) for x in flat), dtype=np.uint8, count=flat.size).reshape(np.shape(v))


# ------------------------------------------------------------------ layout

@dataclass
class Layout:
    T: int
    K: int
    E: int
    R: int
    capacity: int
    tokens_per_expert: np.ndarray
    expert_offset: np.ndarray
    tokens_per_rank: np.ndarray
    rank_offset: np.ndarray
    recv_expert_offset: np.ndarray
    recv_slot: np.ndarray
    expert_slot: np.ndarray
    recv_src_token: np.ndarray
    expert_src_row: np.ndarray
    expert_weight: np.ndarray
    status: int
    num_sources: int = 0                           # 0: single-source packed layout
    recv_source_offset: np.ndarray | None = None   # [R, S+1], multi-source only

    @property
    def n_pairs(self) -> int:
        """Receive rows in use (summed over the destination ranks)."""
        return int(self.tokens_per_rank.sum())


def layout(topk_idx: np.ndarray, topk_w: np.ndarray | None, E: int, R: int,
           capacity: int | None = None) -> Layout:
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    if capacity is None:
        capacity = T * min(K, R)
    w = None if topk_w is None else np.ascontiguousarray(topk_w, dtype=np.float32)
    i32 = np.int32
    L = Layout(T, K, E, R, capacity,
               np.zeros(E, i32), np.zeros(E + 1, i32), np.zeros(R, i32), np.zeros(R + 1, i32),
               np.zeros(E + 1, i32), np.zeros((T, R), i32), np.zeros((T, K), i32),
               np.zeros(capacity, i32), np.zeros(T * K, i32), np.zeros(T * K, np.float32), 0)
    L.status = lib().moe_ref_layout(
        _ptr(topk_idx), _ptr(w), T, K, E, R, capacity,
        _ptr(L.tokens_per_expert), _ptr(L.expert_offset), _ptr(L.tokens_per_rank),
        _ptr(L.rank_offset), _ptr(L.recv_expert_offset), _ptr(L.recv_slot), _ptr(L.expert_slot),
        _ptr(L.recv_src_token), _ptr(L.expert_src_row), _ptr(L.expert_weight))
    return L


def layout_sources(topk_idx: np.ndarray, topk_w: np.ndarray | None, S: int, E: int, R: int) -> Layout:
    """Multi-source receive layout: topk_idx [S*Ts, K] holds the S sources'
    routing one after the other; capacity is R * T (one region of T rows per
    destination).  recv_expert_offset is None."""
    topk_idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, K = topk_idx.shape
    assert S >= 1 and T % S == 0, "every source holds the same number of tokens"
    Ts = T // S
    capacity = R * T
    w = None if topk_w is None else np.ascontiguousarray(topk_w, dtype=np.float32)
    i32 = np.int32
    L = Layout(T, K, E, R, capacity,
               np.zeros(E, i32), np.zeros(E + 1, i32), np.zeros(R, i32), np.zeros(R + 1, i32),
               None, np.zeros((T, R), i32), np.zeros((T, K), i32),
               np.zeros(capacity, i32), np.zeros(T * K, i32), np.zeros(T * K, np.float32), 0,
               num_sources=S, recv_source_offset=np.zeros((R, S + 1), i32))
    L.status = lib().moe_ref_layout_sources(
        _ptr(topk_idx), _ptr(w), S, Ts, K, E, R,
        _ptr(L.tokens_per_expert), _ptr(L.expert_offset), _ptr(L.tokens_per_rank),
        _ptr(L.rank_offset), _ptr(L.recv_source_offset), _ptr(L.recv_slot), _ptr(L.expert_slot),
        _ptr(L.recv_src_token), _ptr(L.expert_src_row), _ptr(L.expert_weight))
    return L


# ---------------------------------------------------------------- dispatch

def dispatch_bf16(x_bits: np.ndarray, L: Layout, recv_x: np.ndarray | None = None):
    """x_bits: uint16 [T,H] bf16 patterns.  Returns (recv_x uint16 [capacity,H], status);
    rows that receive no token keep their initial contents (zeros if recv_x is None)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    if recv_x is None:
        recv_x = np.zeros((L.capacity, H), np.uint16)
    st = lib().moe_ref_dispatch_bf16(_ptr(x_bits), T, H, L.R, _ptr(L.recv_slot), L.capacity, _ptr(recv_x))
    return recv_x, st


def dispatch_fp8(x_bits: np.ndarray, L: Layout):
    """Returns (recv_q uint8 [capacity,H], recv_scales float32 [capacity,H/128], status)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    recv_q = np.zeros((L.capacity, H), np.uint8)
    recv_s = np.zeros((L.capacity, max(H // 128, 1)), np.float32)
    st = lib().moe_ref_dispatch_fp8(_ptr(x_bits), T, H, L.R, _ptr(L.recv_slot), L.capacity,
                                    _ptr(recv_q), _ptr(recv_s))
    return recv_q, recv_s, st


def dispatch_mxfp8(x_bits: np.ndarray, L: Layout):
    """Returns (recv_q uint8 [capacity,H], recv_scales uint8 E8M0 [capacity,H/32], status)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H = x_bits.shape
    recv_q = np.zeros((L.capacity, H), np.uint8)
    recv_s = np.zeros((L.capacity, max(H // 32, 1)), np.uint8)
    st = lib().moe_ref_dispatch_mxfp8(_ptr(x_bits), T, H, L.R, _ptr(L.recv_slot), L.capacity,
                                      _ptr(recv_q), _ptr(recv_s))
    return recv_q, recv_s, st


# ----------------------------------------------------------------- combine

def combine(y_bits: np.ndarray, expert_slot: np.ndarray, topk_w: np.ndarray):
    """y_bits: uint16 [n_rows,H] expert-major bf16.  Returns (out uint16 [T,H], status)."""
    y_bits = np.ascontiguousarray(y_bits, dtype=np.uint16)
    expert_slot = np.ascontiguousarray(expert_slot, dtype=np.int32)
    topk_w = np.ascontiguousarray(topk_w, dtype=np.float32)
    n_rows, H = y_bits.shape
    T, K = expert_slot.shape
    out = np.zeros((T, H), np.uint16)
    st = lib().moe_ref_combine(_ptr(y_bits), n_rows, T, K, H, _ptr(expert_slot), _ptr(topk_w), _ptr(out))
    return out, st


# ---------------------------------------------------------------- backward

def dispatch_backward(grad_recv_bits: np.ndarray, recv_slot: np.ndarray):
    """grad_recv uint16 [n_rows,H] bf16.  Returns (grad_x uint16 [T,H], status)."""
    g = np.ascontiguousarray(grad_recv_bits, dtype=np.uint16)
    recv_slot = np.ascontiguousarray(recv_slot, dtype=np.int32)
    n_rows, H = g.shape
    T, R = recv_slot.shape
    out = np.zeros((T, H), np.uint16)
    st = lib().moe_ref_dispatch_backward(_ptr(g), n_rows, T, R, H, _ptr(recv_slot), _ptr(out))
    return out, st


def combine_backward(grad_out_bits: np.ndarray, y_bits: np.ndarray, expert_slot: np.ndarray, topk_w: np.ndarray,
                     grad_y: np.ndarray | None = None):
    """Returns (grad_y uint16 [n_rows,H], grad_w float64 [T,K], status); rows of
    grad_y no entry maps to keep their initial contents (zeros if None)."""
    go = np.ascontiguousarray(grad_out_bits, dtype=np.uint16)
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    es = np.ascontiguousarray(expert_slot, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float32)
    n_rows, H = y.shape
    T, K = es.shape
    if grad_y is None:
        grad_y = np.zeros((n_rows, H), np.uint16)
    gw = np.zeros((T, K), np.float64)
    st = lib().moe_ref_combine_backward(_ptr(go), _ptr(y), n_rows, T, K, H, _ptr(es), _ptr(w), _ptr(grad_y), _ptr(gw))
    return grad_y, gw, st


# ------------------------------------------------------------- low latency

def ll_dispatch(x_bits: np.ndarray, topk_idx: np.ndarray, E: int, cap: int, recv: np.ndarray | None = None):
    """Returns (recv uint16 [E*cap,H], tokens_per_expert int32 [E], ll_slot int32 [T,K], status)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, H = x_bits.shape
    K = idx.shape[1]
    if recv is None:
        recv = np.zeros((E * cap, H), np.uint16)
    tpe = np.zeros(E, np.int32)
    slot = np.zeros((T, K), np.int32)
    st = lib().moe_ref_ll_dispatch(_ptr(x_bits), _ptr(idx), T, K, E, H, cap, _ptr(recv), _ptr(tpe), _ptr(slot))
    return recv, tpe, slot, st
