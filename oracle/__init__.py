"""CPU oracle of the decode-time MoE layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``moe_oracle.c`` (plain C,
double precision) through ctypes and shares no code with the CUDA library.
Every array in and out is a numpy array on the host.

Parity pins for every function live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

FMT_FP8_B128 = 1
FMT_NVFP4_G16 = 2


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                           "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


class _Proj(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("rows", ctypes.c_int), ("cols", ctypes.c_int),
                ("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("global_", ctypes.c_void_p)]


class _Experts(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("gate", _Proj), ("up", _Proj), ("down", _Proj)]


_P = ctypes.c_void_p


def _declare(L: ctypes.CDLL) -> None:
    L.oracle_e4m3_value.restype = ctypes.c_double
    L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    L.oracle_e2m1_value.restype = ctypes.c_double
    L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
    L.oracle_bf16_rne.restype = ctypes.c_uint16
    L.oracle_bf16_rne.argtypes = [ctypes.c_double]
    L.oracle_bf16_value.restype = ctypes.c_double
    L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    L.oracle_router_logits.restype = None
    L.oracle_router_logits.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
    L.oracle_topk_softmax.restype = None
    L.oracle_topk_softmax.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P]
    L.oracle_align_sizes.restype = None
    L.oracle_align_sizes.argtypes = [ctypes.c_int] * 3 + [_P] * 3
    L.oracle_align.restype = ctypes.c_int
    L.oracle_align.argtypes = [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int] + [_P] * 8
    L.oracle_dequant_proj.restype = None
    L.oracle_dequant_proj.argtypes = [ctypes.POINTER(_Proj), ctypes.c_int, _P]
    ex = ctypes.POINTER(_Experts)
    L.oracle_grouped_gate_up.restype = None
    L.oracle_grouped_gate_up.argtypes = [ex, ex, _P, ctypes.c_int, ctypes.c_int,
                                         _P, _P, _P, ctypes.c_int, _P, _P]
    L.oracle_grouped_down.restype = None
    L.oracle_grouped_down.argtypes = [ex, ex, _P, _P, ctypes.c_int, ctypes.c_int,
                                      _P, _P, _P, ctypes.c_int, _P, _P]
    L.oracle_blend.restype = None
    L.oracle_shared_gate.restype = None
    L.oracle_shared_gate.argtypes = [_P, _P, ctypes.c_int, ctypes.c_int, _P]
    L.oracle_blend.argtypes = [_P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                               _P, _P]
    L.oracle_moe_layer.restype = ctypes.c_int
    L.oracle_moe_layer.argtypes = [ex, ex, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   _P, _P, _P, _P, _P]


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def e2m1_value(nibble: int) -> float:
    return lib().oracle_e2m1_value(nibble)


def bf16_rne(v: float) -> int:
    return lib().oracle_bf16_rne(float(v))


def bf16_round_array(a: np.ndarray) -> np.ndarray:
    """Round every element of a float64 array to bf16 bits (uint16)."""
    f = lib().oracle_bf16_rne
    flat = np.ascontiguousarray(a, dtype=np.float64).ravel()
    return np.array([f(float(v)) for v in flat], dtype=np.uint16).reshape(np.shape(a))


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# routing and alignment
# --------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """float64 [M, E] logits of bf16 rows x [M, H] against bf16 router weights [E, H]."""
    x = _c(x_bits, np.uint16)
    W = _c(w_bits, np.uint16)
    M, H = x.shape
    E = W.shape[0]
    assert W.shape[1] == H
    out = np.empty((M, E), np.float64)
    lib().oracle_router_logits(_ptr(x), _ptr(W), M, H, E, _ptr(out))
    return out


def shared_gate(x_bits: np.ndarray, gate_bits: np.ndarray) -> np.ndarray:
    """float64 [M] gates sigmoid(x[t] . gate_w) of bf16 rows x [M, H] and a
    bf16 gate weight [H]."""
    x = _c(x_bits, np.uint16)
    g = _c(gate_bits, np.uint16).ravel()
    M, H = x.shape
    assert g.shape == (H,)
    out = np.empty(M, np.float64)
    lib().oracle_shared_gate(_ptr(x), _ptr(g), M, H, _ptr(out))
    return out


def topk_softmax(logits: np.ndarray, k: int):
    """ids int32 [M, k] (descending logit, ties to the lower id), w float64 [M, k]."""
    lg = _c(logits, np.float32)
    M, E = lg.shape
    ids = np.empty((M, k), np.int32)
    w = np.empty((M, k), np.float64)
    lib().oracle_topk_softmax(_ptr(lg), M, E, k, _ptr(ids), _ptr(w))
    return ids, w


def align_sizes(n: int, E: int, BS: int):
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    lib().oracle_align_sizes(n, E, BS, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return a.value, b.value, c.value


def align(ids: np.ndarray, E: int, BS: int) -> dict:
    """Alignment tables of the flat slot ids (any integer dtype)."""
    ids64 = _c(np.asarray(ids).ravel(), np.int64)
    n = ids64.size
    max_total, max_blocks, cap = align_sizes(n, E, BS)
    out = dict(
        sorted_token_ids=np.empty(max_total, np.int32),
        sorted_expert_ids=np.empty(max_blocks, np.int32),
        expert_offsets=np.empty(E + 1, np.int32),
        token_to_perm=np.empty(n, np.int32),
        active_experts=np.empty(cap, np.int32),
        active_count=np.zeros(1, np.int32),
        num_tokens_post_padded=np.zeros(1, np.int32),
        counts=np.empty(E, np.int32),
    )
    bad = lib().oracle_align(
        _ptr(ids64), n, E, BS, _ptr(out["sorted_token_ids"]), _ptr(out["sorted_expert_ids"]),
        _ptr(out["expert_offsets"]), _ptr(out["token_to_perm"]), _ptr(out["active_experts"]),
        _ptr(out["active_count"]), _ptr(out["num_tokens_post_padded"]), _ptr(out["counts"]))
    out["bad"] = bad
    out["max_total"], out["max_blocks"], out["cap"] = max_total, max_blocks, cap
    return out


# --------------------------------------------------------------------------
# expert weights
# --------------------------------------------------------------------------

@dataclass
class Proj:
    """One projection of E experts (host numpy arrays).  FP8: codes uint8
    [E, rows, cols], scale float32 [E, rows/128, cols/128], glob None.
    NVFP4: codes uint8 [E, rows, cols/2], scale uint8 [E, rows, cols/16],
    glob float32 [E]."""
    fmt: int
    rows: int
    cols: int
    codes: np.ndarray
    scale: np.ndarray
    glob: Optional[np.ndarray] = None

    def _struct(self) -> _Proj:
        self.codes = _c(self.codes, np.uint8)
        self.scale = _c(self.scale, np.float32 if self.fmt == FMT_FP8_B128 else np.uint8)
        if self.glob is not None:
            self.glob = _c(self.glob, np.float32)
        return _Proj(self.fmt, self.rows, self.cols, self.codes.ctypes.data,
                     self.scale.ctypes.data,
                     None if self.glob is None else self.glob.ctypes.data)


@dataclass
class Experts:
    E: int
    H: int
    I: int
    gate: Proj
    up: Proj
    down: Proj

    def _struct(self) -> _Experts:
        return _Experts(self.E, self.H, self.I, self.gate._struct(), self.up._struct(),
                        self.down._struct())


def _exp_ptr(X: Optional[Experts]):
    if X is None:
        return None, None
    s = X._struct()
    return s, ctypes.pointer(s)


def dequant(P: Proj, e: int) -> np.ndarray:
    out = np.empty((P.rows, P.cols), np.float64)
    s = P._struct()
    lib().oracle_dequant_proj(ctypes.byref(s), e, _ptr(out))
    return out


def grouped_gate_up(X: Experts, S: Optional[Experts], x_bits: np.ndarray, M: int, top_k: int,
                    tables: dict):
    x = _c(x_bits, np.uint16)
    h = np.zeros((tables["max_total"], X.I), np.float64)
    h_sh = np.zeros((M, S.I), np.float64) if S is not None else None
    _xs, xp = _exp_ptr(X)
    _ss, sp = _exp_ptr(S)
    lib().oracle_grouped_gate_up(xp, sp, _ptr(x), M, top_k, _ptr(tables["sorted_token_ids"]),
                                 _ptr(tables["expert_offsets"]), _ptr(tables["active_experts"]),
                                 int(tables["active_count"][0]), _ptr(h), _ptr(h_sh))
    return h, h_sh


def grouped_down(X: Experts, S: Optional[Experts], h: np.ndarray, h_sh: Optional[np.ndarray],
                 M: int, top_k: int, tables: dict):
    h = _c(h, np.float64)
    h_sh = None if h_sh is None else _c(h_sh, np.float64)
    y = np.zeros((tables["max_total"], X.H), np.float64)
    y_sh = np.zeros((M, X.H), np.float64) if S is not None else None
    _xs, xp = _exp_ptr(X)
    _ss, sp = _exp_ptr(S)
    lib().oracle_grouped_down(xp, sp, _ptr(h), _ptr(h_sh), M, top_k,
                              _ptr(tables["sorted_token_ids"]), _ptr(tables["expert_offsets"]),
                              _ptr(tables["active_experts"]), int(tables["active_count"][0]),
                              _ptr(y), _ptr(y_sh))
    return y, y_sh


def blend(y: np.ndarray, w: np.ndarray, token_to_perm: np.ndarray, y_sh: Optional[np.ndarray],
          M: int, top_k: int, H: int, gate: Optional[np.ndarray] = None):
    """gate: float64 [M] shared-expert gates, or None (ungated)."""
    y = _c(y, np.float64)
    w = _c(w, np.float64)
    ttp = _c(token_to_perm, np.int32)
    y_sh = None if y_sh is None else _c(y_sh, np.float64)
    gate = None if gate is None else _c(gate, np.float64)
    out_d = np.empty((M, H), np.float64)
    out_b = np.empty((M, H), np.uint16)
    lib().oracle_blend(_ptr(y), _ptr(w), _ptr(ttp), _ptr(y_sh), _ptr(gate), M, top_k, H,
                       _ptr(out_d), _ptr(out_b))
    return out_d, out_b


def moe_layer(X: Experts, S: Optional[Experts], x_bits: np.ndarray, M: int, top_k: int, BS: int,
              logits: Optional[np.ndarray] = None, ids: Optional[np.ndarray] = None,
              w: Optional[np.ndarray] = None, shared_gate_bits: Optional[np.ndarray] = None):
    """The whole layer; returns (out float64 [M, H], out bf16 bits [M, H], bad ids).
    shared_gate_bits: bf16 [H] gate weight of the shared expert, or None."""
    x = _c(x_bits, np.uint16)
    lg = None if logits is None else _c(logits, np.float32)
    ids_c = None if ids is None else _c(ids, np.int32)
    w_c = None if w is None else _c(w, np.float64)
    out_d = np.empty((M, X.H), np.float64)
    out_b = np.empty((M, X.H), np.uint16)
    _xs, xp = _exp_ptr(X)
    _ss, sp = _exp_ptr(S)
    gw = None if shared_gate_bits is None else _c(shared_gate_bits, np.uint16).ravel()
    bad = lib().oracle_moe_layer(xp, sp, _ptr(gw), _ptr(x), M, top_k, BS, _ptr(lg), _ptr(ids_c), _ptr(w_c),
                                 _ptr(out_d), _ptr(out_b))
    return out_d, out_b, bad
