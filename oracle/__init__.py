"""ctypes loader for the CPU oracle: ``moe_oracle.c`` (the MoE expert layer, fp64)
and ``sampler_oracle.c`` (the per-step sampler: entropy, Gumbel-max, acceptance).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product path (the package
``w4a16_moe_expert_router_gb300``) never imports this module, and this module
never imports the product package.

Every function here is marshalling only; the arithmetic is in the two C files,
which cite the passages of the pages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "moe_oracle.c"), os.path.join(_HERE, "sampler_oracle.c")]
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_SHAPE, ERR_NONFINITE, ERR_ALLOC = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, no fp contraction, no fast-math)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-pthread", "-o", tmp, *_SRCS, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("tokens", "hidden", "inter", "experts", "top_k",
                                              "group_gate_up", "group_down", "activation", "format")]


class _Weights(ctypes.Structure):
    _fields_ = [("gate_up_q", ctypes.c_void_p), ("gate_up_scale", ctypes.c_void_p),
                ("gate_up_zero", ctypes.c_void_p), ("down_q", ctypes.c_void_p),
                ("down_scale", ctypes.c_void_p), ("down_zero", ctypes.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            L.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_half_to_double.restype = dbl
            L.oracle_double_to_half.argtypes = [dbl]
            L.oracle_double_to_half.restype = ctypes.c_uint16
            L.oracle_route.argtypes = [i32, i32, i32, vp, vp, vp]
            L.oracle_permute.argtypes = [i32, i32, i32, vp, vp, vp]
            L.oracle_code.argtypes = [vp, i64]
            L.oracle_dequant.argtypes = [ctypes.c_int, ctypes.c_uint16, ctypes.c_uint16]
            L.oracle_dequant.restype = dbl
            L.oracle_dequant_format.argtypes = [ctypes.c_int, ctypes.c_uint16, ctypes.c_uint16, ctypes.c_int]
            L.oracle_dequant_format.restype = dbl
            L.oracle_gelu.argtypes = [dbl, ctypes.c_int]
            L.oracle_gelu.restype = dbl
            L.oracle_rmsnorm.argtypes = [i64, vp, vp, dbl, vp]
            L.oracle_moe_forward.argtypes = [ctypes.POINTER(_Shape), vp, vp, vp, ctypes.POINTER(_Weights), vp,
                                             dbl, vp, ctypes.c_int, ctypes.c_int, vp]
            L.oracle_moe_forward_dense.argtypes = [ctypes.POINTER(_Shape), vp, vp, vp,
                                                   ctypes.POINTER(_Weights), vp]
            L.oracle_block_front.argtypes = [i32, i32, i32, vp, vp, ctypes.c_float, vp, vp, vp]
            L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
            L.oracle_log_f32.argtypes = [ctypes.c_float]
            L.oracle_log_f32.restype = ctypes.c_float
            L.oracle_gumbel_key.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_uint32]
            L.oracle_gumbel_key.restype = ctypes.c_float
            L.oracle_exp_f32.argtypes = [ctypes.c_float]
            L.oracle_exp_f32.restype = ctypes.c_float
            L.oracle_group_counter.argtypes = [ctypes.c_uint32]
            L.oracle_group_counter.restype = ctypes.c_uint32
            L.oracle_group_word.argtypes = [ctypes.c_uint32]
            L.oracle_group_word.restype = ctypes.c_int
            L.oracle_group_key.argtypes = [vp, ctypes.c_float, ctypes.c_uint32]
            L.oracle_group_key.restype = ctypes.c_float
            L.oracle_group_pick.argtypes = [vp, ctypes.c_float, ctypes.c_uint32]
            L.oracle_group_pick.restype = ctypes.c_int
            L.oracle_sample.argtypes = [i32, i64, vp, ctypes.c_float, ctypes.c_uint64, ctypes.c_uint32,
                                        ctypes.c_int, ctypes.c_int, vp, vp, vp]
            L.oracle_accept_entropy.argtypes = [i32, vp, vp, ctypes.c_float, vp]
            L.oracle_accept_confidence.argtypes = [i32, vp, vp, ctypes.c_float, vp]
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int) -> float:
    return lib().oracle_half_to_double(int(bits))


def double_to_half(v: float) -> int:
    return lib().oracle_double_to_half(float(v))


def code(packed_row: np.ndarray, kk: int) -> int:
    row = _c(packed_row, np.uint8)
    return lib().oracle_code(_ptr(row), int(kk))


def dequant(q: int, zero_bits: int, scale_bits: int) -> float:
    return lib().oracle_dequant(int(q), int(zero_bits), int(scale_bits))


def dequant_format(q: int, second_bits: int, scale_bits: int, fmt: int) -> float:
    """One weight of format 0 (asymmetric zero-point), 1 (affine bias) or 2 (symmetric)."""
    return lib().oracle_dequant_format(int(q), int(second_bits), int(scale_bits), int(fmt))


def gelu(a: float, act: int = 0) -> float:
    return lib().oracle_gelu(float(a), int(act))


def route(logits: np.ndarray, k: int):
    """Top-k expert ids (router-rank order) and fp64 softmax weights over them."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    st = lib().oracle_route(T, E, k, _ptr(lg), _ptr(idx), _ptr(w))
    if st != OK:
        raise ValueError(f"oracle_route status {st}")
    return idx, w


def permute(topk_idx: np.ndarray, E: int):
    """Per-expert pair lists: offsets [E+1] and pair ids p = t*k + r, grouped by expert."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    off = np.zeros(E + 1, np.int32)
    pl = np.zeros(T * k, np.int32)
    st = lib().oracle_permute(T, E, k, _ptr(idx), _ptr(off), _ptr(pl))
    if st != OK:
        raise ValueError(f"oracle_permute status {st}")
    return off, pl


def rmsnorm(u: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    u = _c(u, np.float64)
    g = _c(gamma, np.float32)
    out = np.zeros_like(u)
    lib().oracle_rmsnorm(u.shape[0], _ptr(u), _ptr(g), float(eps), _ptr(out))
    return out


def _shape(T, d, f, E, k, g1, g2, act, fmt=0):
    return _Shape(T, d, f, E, k, g1, g2, act, fmt)


def _weights(w: dict):
    arrs = {
        "gate_up_q": _c(w["gate_up_q"], np.uint8), "gate_up_scale": _c(w["gate_up_scale"], np.uint16),
        "gate_up_zero": _c(w["gate_up_zero"], np.uint16), "down_q": _c(w["down_q"], np.uint8),
        "down_scale": _c(w["down_scale"], np.uint16), "down_zero": _c(w["down_zero"], np.uint16),
    }
    return _Weights(*[_ptr(arrs[n]) for n, _ in _Weights._fields_]), arrs


def forward(x_bits: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, weights: dict, *,
            group_gate_up: int, group_down: int, activation: int = 0, gamma: np.ndarray | None = None,
            eps: float = 1e-6, token_sel: np.ndarray | None = None, nthreads: int = 1,
            round_fp16: bool = False, fmt: int = 0) -> np.ndarray:
    """The layer (sparse form).  Returns fp64 [T][d]; unselected tokens stay NaN.

    x_bits: fp16 bit patterns [T][d] (uint16); weights: canonical arrays
    gate_up_q [E][2f][d/2], gate_up_scale/zero [E][2f][d/g1], down_q [E][d][f/2],
    down_scale/zero [E][d][f/g2] (scale/zero as fp16 bit patterns).
    """
    x = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    wt = _c(topk_w, np.float64)
    T, d = x.shape
    k = idx.shape[1]
    E, two_f, _ = weights["gate_up_q"].shape
    f = two_f // 2
    sh = _shape(T, d, f, E, k, group_gate_up, group_down, activation, fmt)
    cw, keep = _weights(weights)
    g = None if gamma is None else _c(gamma, np.float32)
    sel = None if token_sel is None else _c(token_sel, np.uint8)
    out = np.full((T, d), np.nan, np.float64)
    st = lib().oracle_moe_forward(ctypes.byref(sh), _ptr(x), _ptr(idx), _ptr(wt), ctypes.byref(cw), _ptr(g),
                                  float(eps), _ptr(sel), int(nthreads), int(bool(round_fp16)), _ptr(out))
    del keep
    if st != OK:
        raise ValueError(f"oracle_moe_forward status {st}")
    return out


def forward_dense(x_bits: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, weights: dict, *,
                  group_gate_up: int, group_down: int, activation: int = 0, fmt: int = 0) -> np.ndarray:
    """The layer (dense form: every expert on every token, gated by G[t][e])."""
    x = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    wt = _c(topk_w, np.float64)
    T, d = x.shape
    k = idx.shape[1]
    E, two_f, _ = weights["gate_up_q"].shape
    sh = _shape(T, d, two_f // 2, E, k, group_gate_up, group_down, activation, fmt)
    cw, keep = _weights(weights)
    out = np.zeros((T, d), np.float64)
    st = lib().oracle_moe_forward_dense(ctypes.byref(sh), _ptr(x), _ptr(idx), _ptr(wt), ctypes.byref(cw), _ptr(out))
    del keep
    if st != OK:
        raise ValueError(f"oracle_moe_forward_dense status {st}")
    return out


def block_front(x_bits: np.ndarray, gamma: np.ndarray, eps: float, wr_bits: np.ndarray):
    """The MoE block's pre-norm and router projection in their fixed fp32 order:
    returns u (fp16 bit patterns [T][d]) and the router logits (fp32 [T][E])."""
    x = _c(x_bits, np.uint16)
    g = _c(gamma, np.float32)
    w = _c(wr_bits, np.uint16)
    T, d = x.shape
    E = w.shape[0]
    u = np.zeros((T, d), np.uint16)
    logits = np.zeros((T, E), np.float32)
    st = lib().oracle_block_front(int(T), int(d), int(E), _ptr(x), _ptr(g), float(eps), _ptr(w), _ptr(u),
                                  _ptr(logits))
    if st != OK:
        raise ValueError(f"oracle_block_front status {st}")
    return u, logits


# ------------------------------------------------------------------ sampler

def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 of one counter (4 words) under one key (2 words)."""
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def log_f32(x: float) -> float:
    """The fp32 natural log the Gumbel keys are defined with."""
    return float(lib().oracle_log_f32(ctypes.c_float(x)))


def gumbel_key(logit: float, inv_temp: float, word: int) -> float:
    return float(lib().oracle_gumbel_key(ctypes.c_float(logit), ctypes.c_float(inv_temp), ctypes.c_uint32(word)))


def exp_f32(x: float) -> float:
    """The fp32 exponential (of x <= 0) the group keys are defined with."""
    return float(lib().oracle_exp_f32(ctypes.c_float(x)))


def group_counter_word(g: int) -> tuple[int, int]:
    """The Philox counter (first word) and word index of group g (entries 4g .. 4g+3)."""
    return int(lib().oracle_group_counter(int(g))), int(lib().oracle_group_word(int(g)))


def group_key(l4, inv_temp: float, word: int) -> float:
    """Gumbel key of a group of four logits under one Philox word."""
    a = _c(l4, np.float32)
    return float(lib().oracle_group_key(_ptr(a), ctypes.c_float(inv_temp), ctypes.c_uint32(word)))


def group_pick(l4, inv_temp: float, word: int) -> int:
    """The token (0 .. 3) inside a group of four logits under one Philox word."""
    a = _c(l4, np.float32)
    return int(lib().oracle_group_pick(_ptr(a), ctypes.c_float(inv_temp), ctypes.c_uint32(word)))


def sample(logits: np.ndarray, inv_temp: float, seed: int, step: int, nthreads: int = 1, noise: int = 0):
    """Gumbel-max tokens (int32 [P]) and fp64 entropy and top-1 probability [P] of
    softmax(logits * inv_temp); noise 0 draws one Gumbel per group of four entries,
    1 one per entry."""
    lg = _c(logits, np.float32)
    P, V = lg.shape
    tok = np.zeros(P, np.int32)
    ent = np.zeros(P, np.float64)
    pm = np.zeros(P, np.float64)
    st = lib().oracle_sample(P, V, _ptr(lg), float(inv_temp), int(seed), int(step), int(noise), int(nthreads),
                             _ptr(tok), _ptr(ent), _ptr(pm))
    if st != OK:
        raise ValueError(f"oracle_sample status {st}")
    return tok, ent, pm


def accept_entropy(entropy: np.ndarray, revealed: np.ndarray, bound: float) -> np.ndarray:
    """Entropy-bound acceptance (uint8 [P]) decided on fp32 entropies."""
    h = _c(entropy, np.float32)
    rv = _c(revealed, np.uint8)
    acc = np.zeros(h.shape[0], np.uint8)
    st = lib().oracle_accept_entropy(h.shape[0], _ptr(h), _ptr(rv), float(bound), _ptr(acc))
    if st != OK:
        raise ValueError(f"oracle_accept_entropy status {st}")
    return acc


def accept_confidence(pmax: np.ndarray, revealed: np.ndarray, threshold: float) -> np.ndarray:
    """Confidence-threshold acceptance (uint8 [P]) decided on fp32 top-1 probabilities."""
    pm = _c(pmax, np.float32)
    rv = _c(revealed, np.uint8)
    acc = np.zeros(pm.shape[0], np.uint8)
    st = lib().oracle_accept_confidence(pm.shape[0], _ptr(pm), _ptr(rv), float(threshold), _ptr(acc))
    if st != OK:
        raise ValueError(f"oracle_accept_confidence status {st}")
    return acc
