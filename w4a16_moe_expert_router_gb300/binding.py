"""Thin ctypes binding of the C ABI in ``include/moe_w4a16.h``.

Functions keep the C names and only marshal arguments: device buffers are any
object with ``data_ptr()`` (torch tensors) or raw integer addresses, host
buffers are numpy arrays, and a stream is a ``torch.cuda.Stream``, a raw
``cudaStream_t`` integer, or ``None`` for torch's current stream.  Every step of
the layer runs in the library's CUDA kernels; if the shared library has not been
built, loading it raises (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe_w4a16.so")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE, ERR_TIMEOUT, ERR_VALUE = range(9)
GATE_UP, DOWN = 0, 1

EXPORTED = ("moe_w4a16_workspace_bytes", "moe_w4a16_workspace_init", "moe_w4a16_route", "moe_w4a16_forward",
            "moe_w4a16_experts",
            "moe_w4a16_gate_up", "moe_w4a16_down", "moe_w4a16_combine", "moe_w4a16_read_error", "moe_w4a16_pack", "moe_w4a16_unpack", "moe_w4a16_prepared_bytes",
            "moe_w4a16_prepare", "moe_w4a16_unprepare", "moe_w4a16_status_string", "moe_w4a16_forward_noalloc",
            "moe_w4a16_selftest_wait_timeout", "moe_w4a16_sampler_workspace_bytes", "moe_w4a16_sample",
            "moe_w4a16_block_front", "moe_w4a16_block", "moe_w4a16_noalloc_read_error")

NOALLOC_SCRATCH_BYTES = 40 << 20  # MOE_W4A16_NOALLOC_SCRATCH_BYTES


class MoeW4A16Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({moe_w4a16_status_string(status)})")


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("tokens", "hidden", "inter", "experts", "top_k", "group_gate_up",
                                              "group_down", "activation", "reduction", "format")]


class Sampler(ctypes.Structure):
    _fields_ = [("positions", ctypes.c_int32), ("vocab", ctypes.c_int32), ("inv_temperature", ctypes.c_float),
                ("rule", ctypes.c_int32), ("bound", ctypes.c_float), ("step", ctypes.c_uint32),
                ("noise", ctypes.c_int32), ("seed", ctypes.c_uint64)]


class Weights(ctypes.Structure):
    _fields_ = [("gate_up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


class Routing(ctypes.Structure):
    _fields_ = [("topk_idx", ctypes.c_void_p), ("topk_w", ctypes.c_void_p), ("expert_offsets", ctypes.c_void_p),
                ("pair_list", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
            P = ctypes.POINTER
            st = ctypes.c_int
            L.moe_w4a16_workspace_bytes.argtypes = [P(Shape)]
            L.moe_w4a16_workspace_bytes.restype = sz
            L.moe_w4a16_workspace_init.argtypes = [vp, sz, vp]
            L.moe_w4a16_workspace_init.restype = st
            L.moe_w4a16_route.argtypes = [P(Shape), vp, P(Routing), vp, sz, vp]
            L.moe_w4a16_route.restype = st
            L.moe_w4a16_forward.argtypes = [P(Shape), vp, P(Routing), P(Weights), vp, ctypes.c_float, vp, vp, sz, vp]
            L.moe_w4a16_forward.restype = st
            L.moe_w4a16_gate_up.argtypes = [P(Shape), vp, P(Routing), P(Weights), vp, sz, vp]
            L.moe_w4a16_experts.restype = st
            L.moe_w4a16_experts.argtypes = [P(Shape), vp, P(Routing), P(Weights), vp, sz, vp]
            L.moe_w4a16_gate_up.restype = st
            L.moe_w4a16_down.argtypes = [P(Shape), P(Routing), P(Weights), vp, sz, vp]
            L.moe_w4a16_down.restype = st
            L.moe_w4a16_combine.argtypes = [P(Shape), P(Routing), vp, ctypes.c_float, vp, vp, sz, vp]
            L.moe_w4a16_combine.restype = st
            L.moe_w4a16_forward_noalloc.argtypes = [P(Shape), vp, P(Routing), P(Weights), vp, ctypes.c_float, vp,
                                                    vp]
            L.moe_w4a16_forward_noalloc.restype = st
            L.moe_w4a16_block_front.argtypes = [P(Shape), vp, vp, ctypes.c_float, vp, vp, vp, vp]
            L.moe_w4a16_block_front.restype = st
            L.moe_w4a16_block.argtypes = [P(Shape), vp, vp, ctypes.c_float, vp, P(Routing), P(Weights), vp, vp, sz,
                                          vp]
            L.moe_w4a16_block.restype = st
            L.moe_w4a16_noalloc_read_error.argtypes = [vp, P(ctypes.c_int32)]
            L.moe_w4a16_noalloc_read_error.restype = st
            L.moe_w4a16_selftest_wait_timeout.argtypes = [vp, sz, ctypes.c_uint64, vp]
            L.moe_w4a16_selftest_wait_timeout.restype = st
            L.moe_w4a16_sampler_workspace_bytes.argtypes = [P(Sampler)]
            L.moe_w4a16_sampler_workspace_bytes.restype = sz
            L.moe_w4a16_sample.argtypes = [P(Sampler), vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.moe_w4a16_sample.restype = st
            L.moe_w4a16_read_error.argtypes = [vp, sz, vp, P(ctypes.c_int)]
            L.moe_w4a16_read_error.restype = st
            L.moe_w4a16_pack.argtypes = [vp, i64, i64, vp]
            L.moe_w4a16_pack.restype = st
            L.moe_w4a16_unpack.argtypes = [vp, i64, i64, vp]
            L.moe_w4a16_unpack.restype = st
            L.moe_w4a16_prepared_bytes.argtypes = [P(Shape), i32]
            L.moe_w4a16_prepared_bytes.restype = sz
            L.moe_w4a16_prepare.argtypes = [P(Shape), i32, vp, vp, vp, vp]
            L.moe_w4a16_prepare.restype = st
            L.moe_w4a16_unprepare.argtypes = [P(Shape), i32, vp, vp, vp, vp]
            L.moe_w4a16_unprepare.restype = st
            L.moe_w4a16_status_string.argtypes = [st]
            L.moe_w4a16_status_string.restype = ctypes.c_char_p
            _lib = L
    return _lib


# ----------------------------------------------------------------- marshalling

def make_shape(tokens, hidden, inter, experts, top_k, group_gate_up, group_down, activation=0,
               reduction=0, format=0) -> Shape:
    return Shape(tokens, hidden, inter, experts, top_k, group_gate_up, group_down, activation, reduction, format)


def _dptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _hptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != OK:
        raise MoeW4A16Error(status, where)


@dataclass
class RoutingBuffers:
    """Device buffers of one routing (allocated by the caller, e.g. with torch)."""
    topk_idx: object
    topk_w: object
    expert_offsets: object
    pair_list: object

    def c(self) -> Routing:
        return Routing(_dptr(self.topk_idx), _dptr(self.topk_w), _dptr(self.expert_offsets), _dptr(self.pair_list))


# ------------------------------------------------------------------- the C ABI

def moe_w4a16_status_string(status: int) -> str:
    return lib().moe_w4a16_status_string(int(status)).decode()


def moe_w4a16_workspace_bytes(shape: Shape) -> int:
    return int(lib().moe_w4a16_workspace_bytes(ctypes.byref(shape)))


def moe_w4a16_workspace_init(workspace, stream=None) -> None:
    _check(lib().moe_w4a16_workspace_init(_dptr(workspace), _nbytes(workspace), _stream(stream)),
           "moe_w4a16_workspace_init")


def moe_w4a16_route(shape: Shape, logits, routing: RoutingBuffers, workspace, stream=None) -> None:
    r = routing.c()
    _check(lib().moe_w4a16_route(ctypes.byref(shape), _dptr(logits), ctypes.byref(r), _dptr(workspace),
                                 _nbytes(workspace), _stream(stream)), "moe_w4a16_route")


def moe_w4a16_forward(shape: Shape, x, routing: RoutingBuffers, gate_up, down, norm_gamma, norm_eps: float, out,
                      workspace, stream=None) -> None:
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_forward(ctypes.byref(shape), _dptr(x), ctypes.byref(r), ctypes.byref(w),
                                   _dptr(norm_gamma), float(norm_eps), _dptr(out), _dptr(workspace),
                                   _nbytes(workspace), _stream(stream)), "moe_w4a16_forward")


def moe_w4a16_block_front(shape: Shape, x, norm_gamma, norm_eps: float, router_w, u, logits, stream=None) -> None:
    _check(lib().moe_w4a16_block_front(ctypes.byref(shape), _dptr(x), _dptr(norm_gamma), float(norm_eps),
                                       _dptr(router_w), _dptr(u), _dptr(logits), _stream(stream)),
           "moe_w4a16_block_front")


def moe_w4a16_block(shape: Shape, x, norm_gamma, norm_eps: float, router_w, routing: RoutingBuffers, gate_up, down,
                    out, workspace, stream=None) -> None:
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_block(ctypes.byref(shape), _dptr(x), _dptr(norm_gamma), float(norm_eps), _dptr(router_w),
                                 ctypes.byref(r), ctypes.byref(w), _dptr(out), _dptr(workspace), _nbytes(workspace),
                                 _stream(stream)), "moe_w4a16_block")


def moe_w4a16_forward_noalloc(shape: Shape, x, routing: RoutingBuffers, gate_up, down, norm_gamma,
                              norm_eps: float, out, stream=None) -> None:
    """The forward pass with the library's static scratch array instead of a
    workspace, for callers that cannot allocate device memory (see the header)."""
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_forward_noalloc(ctypes.byref(shape), _dptr(x), ctypes.byref(r), ctypes.byref(w),
                                           _dptr(norm_gamma), float(norm_eps), _dptr(out), _stream(stream)),
           "moe_w4a16_forward_noalloc")


def moe_w4a16_noalloc_read_error(stream=None) -> int:
    """The error word of the current device's static scratch (the last
    allocation-free call's device-side status)."""
    code = ctypes.c_int32(0)
    _check(lib().moe_w4a16_noalloc_read_error(_stream(stream), ctypes.byref(code)), "moe_w4a16_noalloc_read_error")
    return code.value


def moe_w4a16_experts(shape: Shape, x, routing: RoutingBuffers, gate_up, down, workspace, stream=None) -> None:
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_experts(ctypes.byref(shape), _dptr(x), ctypes.byref(r), ctypes.byref(w), _dptr(workspace),
                                   _nbytes(workspace), _stream(stream)), "moe_w4a16_experts")


def moe_w4a16_gate_up(shape: Shape, x, routing: RoutingBuffers, gate_up, down, workspace, stream=None) -> None:
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_gate_up(ctypes.byref(shape), _dptr(x), ctypes.byref(r), ctypes.byref(w), _dptr(workspace),
                                   _nbytes(workspace), _stream(stream)), "moe_w4a16_gate_up")


def moe_w4a16_down(shape: Shape, routing: RoutingBuffers, gate_up, down, workspace, stream=None) -> None:
    r = routing.c()
    w = Weights(_dptr(gate_up), _dptr(down))
    _check(lib().moe_w4a16_down(ctypes.byref(shape), ctypes.byref(r), ctypes.byref(w), _dptr(workspace),
                                _nbytes(workspace), _stream(stream)), "moe_w4a16_down")


def moe_w4a16_combine(shape: Shape, routing: RoutingBuffers, norm_gamma, norm_eps: float, out, workspace,
                      stream=None) -> None:
    r = routing.c()
    _check(lib().moe_w4a16_combine(ctypes.byref(shape), ctypes.byref(r), _dptr(norm_gamma), float(norm_eps),
                                   _dptr(out), _dptr(workspace), _nbytes(workspace), _stream(stream)),
           "moe_w4a16_combine")


def make_sampler(positions, vocab, inv_temperature=1.0, rule=0, bound=0.0, step=0, seed=0, noise=0) -> Sampler:
    return Sampler(positions, vocab, inv_temperature, rule, bound, step, noise, seed)


def moe_w4a16_sampler_workspace_bytes(cfg: Sampler) -> int:
    return int(lib().moe_w4a16_sampler_workspace_bytes(ctypes.byref(cfg)))


def moe_w4a16_sample(cfg: Sampler, logits, revealed, token, entropy, pmax, accept, workspace, stream=None) -> None:
    _check(lib().moe_w4a16_sample(ctypes.byref(cfg), _dptr(logits), _dptr(revealed), _dptr(token), _dptr(entropy),
                                  _dptr(pmax), _dptr(accept), _dptr(workspace), _nbytes(workspace), _stream(stream)),
           "moe_w4a16_sample")


def moe_w4a16_read_error(workspace, stream=None) -> int:
    code = ctypes.c_int(0)
    _check(lib().moe_w4a16_read_error(_dptr(workspace), _nbytes(workspace), _stream(stream), ctypes.byref(code)),
           "moe_w4a16_read_error")
    return code.value


def moe_w4a16_selftest_wait_timeout(workspace, limit_ns: int, stream=None) -> None:
    _check(lib().moe_w4a16_selftest_wait_timeout(_dptr(workspace), _nbytes(workspace), limit_ns, _stream(stream)),
           "moe_w4a16_selftest_wait_timeout")


def moe_w4a16_pack(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    K = c.shape[-1]
    rows = c.size // K if K else 0
    out = np.zeros(c.shape[:-1] + (K // 2,), np.uint8)
    _check(lib().moe_w4a16_pack(_hptr(c), rows, K, _hptr(out)), "moe_w4a16_pack")
    return out


def moe_w4a16_unpack(packed: np.ndarray) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    K = 2 * p.shape[-1]
    rows = p.size * 2 // K if K else 0
    out = np.zeros(p.shape[:-1] + (K,), np.uint8)
    _check(lib().moe_w4a16_unpack(_hptr(p), rows, K, _hptr(out)), "moe_w4a16_unpack")
    return out


def moe_w4a16_prepared_bytes(shape: Shape, which: int) -> int:
    return int(lib().moe_w4a16_prepared_bytes(ctypes.byref(shape), int(which)))


def moe_w4a16_prepare(shape: Shape, which: int, q: np.ndarray, scale: np.ndarray, zero) -> np.ndarray:
    """zero: the zero-points (format 0) or biases (format 1); None allowed for format 2."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(scale, dtype=np.uint16)
    z = None if zero is None else np.ascontiguousarray(zero, dtype=np.uint16)
    n = moe_w4a16_prepared_bytes(shape, which)
    if n == 0:
        raise MoeW4A16Error(ERR_SHAPE, "moe_w4a16_prepare")
    if q.nbytes + 2 * s.nbytes != n or (z is not None and z.nbytes != s.nbytes):
        raise MoeW4A16Error(ERR_SHAPE, "moe_w4a16_prepare: array sizes do not match the shape")
    out = np.empty(n, np.uint8)
    _check(lib().moe_w4a16_prepare(ctypes.byref(shape), int(which), _hptr(q), _hptr(s),
                                   None if z is None else _hptr(z), _hptr(out)), "moe_w4a16_prepare")
    return out


def moe_w4a16_unprepare(shape: Shape, which: int, prepared: np.ndarray, q_shape, sz_shape):
    p = np.ascontiguousarray(prepared, dtype=np.uint8)
    q = np.zeros(q_shape, np.uint8)
    s = np.zeros(sz_shape, np.uint16)
    z = np.zeros(sz_shape, np.uint16)
    if q.nbytes + s.nbytes + z.nbytes != p.nbytes or p.nbytes != moe_w4a16_prepared_bytes(shape, which):
        raise MoeW4A16Error(ERR_SHAPE, "moe_w4a16_unprepare: array sizes do not match the shape")
    _check(lib().moe_w4a16_unprepare(ctypes.byref(shape), int(which), _hptr(p), _hptr(q), _hptr(s), _hptr(z)),
           "moe_w4a16_unprepare")
    return q, s, z
