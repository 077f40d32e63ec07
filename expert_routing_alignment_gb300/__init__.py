"""Decode-time MoE layer for GB300 (sm_103a): Python binding of the C ABI.

Every function here marshals torch tensors into the C ABI of
``include/moe_gb300.h`` (``libmoe_gb300.so``) and returns; each step of the
layer runs in the library's CUDA kernels on the current torch stream (or the
stream passed in).  There is no fallback: if the library is missing or fails
to load, every call raises.

    import expert_routing_alignment_gb300 as moe
    ex = moe.Experts.from_tensors(moe.FMT_FP8_B128, E, H, I, gate, up, down)
    layer = moe.LayerDesc(top_k=8, block_size=16, routed=ex)
    ws = moe.alloc_workspace(layer, max_M=8)
    moe.moe_decode_layer(layer, x, out, ws, router_logits=logits)
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

from . import build as _build

MOE_OK = 0
MOE_EINVAL = 1
MOE_EUNSUPPORTED = 2
MOE_ECUDA = 3
MOE_ERR_BAD_ID = 0x1

FMT_FP8_B128 = 1
FMT_NVFP4_G16 = 2
FMT_NVFP4_GATE_UP = 3   # gate and up NVFP4_G16, down FP8_B128
PATH_AUTO = 0
PATH_SIMT = 1
PATH_TC = 2
PATH_SIMT_STAGED = 3
MOE_ERR_TIMEOUT = 0x2
MAX_EXPERTS = 1024
MAX_ROWS = 128
MAX_ROWS_TC = 4096   # M admitted on the tensor-core path (FP8 experts)
TOKEN_FORM_ROWS = 16   # tensor-core path: up to this M, x terms are kept by token
F4_TOKEN_COLUMNS_SMALL = 16   # NVFP4 tensor-core kernel: token columns for M <= 16
F4_TOKEN_COLUMNS = 32         # and for 16 < M <= 32 (its largest M)

LIB_PATH = _build.LIB


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        names = {1: "MOE_EINVAL", 2: "MOE_EUNSUPPORTED", 3: "MOE_ECUDA"}
        msg = f"{fn} failed: {names.get(status, status)}"
        if status == MOE_ECUDA:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


# --------------------------------------------------------------------------
# ctypes mirror of the header's structs
# --------------------------------------------------------------------------

class _Proj(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p)]


class _Experts(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("num_experts", ctypes.c_int), ("hidden", ctypes.c_int),
                ("inter", ctypes.c_int), ("gate", _Proj), ("up", _Proj), ("down", _Proj)]


class _LayerDesc(ctypes.Structure):
    _fields_ = [("top_k", ctypes.c_int), ("block_size", ctypes.c_int), ("path", ctypes.c_int),
                ("routed", _Experts), ("shared", ctypes.POINTER(_Experts)),
                ("shared_gate", ctypes.c_void_p), ("router_weight", ctypes.c_void_p)]


class _WsView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "topk_ids", "topk_w", "sorted_token_ids", "sorted_expert_ids", "expert_offsets",
        "token_to_perm", "active_experts", "active_count", "num_tokens_post_padded", "h",
        "h_shared", "y", "y_shared", "blend_counters", "router_logits", "shared_gate", "tc_x_terms", "tc_x_scale",
        "tc_h_terms", "tc_h_scale", "tc_done", "total_bytes")] + [
        ("max_total", ctypes.c_int), ("max_blocks", ctypes.c_int), ("cap", ctypes.c_int),
        ("tc_items", ctypes.c_size_t)]


_P = ctypes.c_void_p
_I = ctypes.c_int
EXPORTS = {
    "moe_version": (ctypes.c_char_p, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (_I, []),
    "moe_align_sizes": (_I, [_I, _I, _I, _P, _P, _P]),
    "moe_align": (_I, [_P, _I, _I, _I, _I] + [_P] * 9),
    "moe_topk_softmax": (_I, [_P, _I, _I, _I, _P, _P, _P]),
    "moe_router_logits": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_gate_up": (_I, [ctypes.POINTER(_Experts), ctypes.POINTER(_Experts), _P, _I, _I,
                                 _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_grouped_down": (_I, [ctypes.POINTER(_Experts), ctypes.POINTER(_Experts), _P, _P, _I, _I,
                              _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_blend": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "moe_decode_layer_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(_LayerDesc), _I]),
    "moe_decode_layer_workspace_view": (_I, [ctypes.POINTER(_LayerDesc), _I,
                                             ctypes.POINTER(_WsView)]),
    "moe_decode_layer": (_I, [ctypes.POINTER(_LayerDesc), _P, _I, _P, _P, _P, _P, _P,
                              ctypes.c_size_t, _P, _P]),
    "moe_decode_layer_launches": (_I, [ctypes.POINTER(_LayerDesc), _I, _I]),
    "moe_decode_layer_noalloc": (_I, [ctypes.POINTER(_LayerDesc), _P, _I, _P, _P, _P, _P, _P,
                                      _P]),
    "moe_decode_experts": (_I, [ctypes.POINTER(_LayerDesc), _P, _I, _P, _P, ctypes.c_size_t, _P,
                                _P]),
}

_lib: Optional[ctypes.CDLL] = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded library (built on first use when missing or stale)."""
    global _lib
    if _lib is None:
        if build_if_missing:
            _build.build()
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run expert_routing_alignment_gb300.build")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(fn: str, status: int) -> None:
    if status != MOE_OK:
        raise MoeError(fn, status, load().moe_last_cuda_error() if status == MOE_ECUDA else 0)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# --------------------------------------------------------------------------
# weight descriptors
# --------------------------------------------------------------------------

@dataclass
class Experts:
    """An expert set on the device (see moe_experts in the header).  Each
    projection is (codes, scale, global_scale or None)."""
    fmt: int
    num_experts: int
    hidden: int
    inter: int
    gate: Sequence
    up: Sequence
    down: Sequence
    _struct: _Experts = field(init=False, repr=False)

    def __post_init__(self):
        def proj(p):
            codes, scale, glob = (list(p) + [None])[:3]
            return _Proj(codes.data_ptr(), scale.data_ptr(),
                         None if glob is None else glob.data_ptr())
        self._struct = _Experts(self.fmt, self.num_experts, self.hidden, self.inter,
                                proj(self.gate), proj(self.up), proj(self.down))

    @staticmethod
    def from_synth(d) -> "Experts":
        """From a ``synth.ExpertData`` already on the device."""
        fmt = {"fp8": FMT_FP8_B128, "nvfp4": FMT_NVFP4_G16,
               "nvfp4_gate_up": FMT_NVFP4_GATE_UP}[d.fmt]
        t = lambda p: (p.codes, p.scale, p.glob)
        return Experts(fmt, d.E, d.H, d.I, t(d.gate), t(d.up), t(d.down))


@dataclass
class LayerDesc:
    top_k: int
    block_size: int
    routed: Experts
    shared: Optional[Experts] = None
    path: int = PATH_AUTO
    # bf16 [E, H] on the device: lets moe_decode_layer take x alone (hidden in)
    router_weight: Optional[torch.Tensor] = None
    # bf16 [H] on the device: gates the shared expert, sigmoid(x . shared_gate)
    shared_gate: Optional[torch.Tensor] = None
    _struct: _LayerDesc = field(init=False, repr=False)

    def __post_init__(self):
        sh = ctypes.pointer(self.shared._struct) if self.shared is not None else None
        self._struct = _LayerDesc(self.top_k, self.block_size, self.path, self.routed._struct, sh,
                                  _ptr(self.shared_gate), _ptr(self.router_weight))

    @property
    def num_experts(self) -> int:
        return self.routed.num_experts


# --------------------------------------------------------------------------
# entry points (same names as the C ABI)
# --------------------------------------------------------------------------

def moe_version() -> str:
    return load().moe_version().decode()


def moe_align_sizes(n: int, num_experts: int, block_size: int):
    a, b, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("moe_align_sizes", load().moe_align_sizes(n, num_experts, block_size, ctypes.byref(a),
                                                      ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def alloc_align_outputs(n: int, num_experts: int, block_size: int, device="cuda") -> dict:
    max_total, max_blocks, cap = moe_align_sizes(n, num_experts, block_size)
    i32 = dict(dtype=torch.int32, device=device)
    return dict(sorted_token_ids=torch.empty(max(max_total, 1), **i32),
                sorted_expert_ids=torch.empty(max(max_blocks, 1), **i32),
                expert_offsets=torch.empty(num_experts + 1, **i32),
                token_to_perm=torch.empty(max(n, 1), **i32),
                active_experts=torch.empty(max(cap, 1), **i32),
                active_count=torch.empty(1, **i32),
                num_tokens_post_padded=torch.empty(1, **i32),
                max_total=max_total, max_blocks=max_blocks, cap=cap)


def moe_align(topk_ids: torch.Tensor, num_experts: int, block_size: int,
              out: Optional[dict] = None, err_word: Optional[torch.Tensor] = None,
              stream=None) -> dict:
    """Alignment tables of the flat ids (int32 or int64, device)."""
    ids = topk_ids.contiguous().view(-1)
    n = ids.numel()
    if out is None:
        out = alloc_align_outputs(n, num_experts, block_size, ids.device)
    _check("moe_align", load().moe_align(
        _ptr(ids), int(ids.dtype == torch.int64), n, num_experts, block_size,
        _ptr(out["sorted_token_ids"]), _ptr(out["sorted_expert_ids"]),
        _ptr(out["expert_offsets"]), _ptr(out["token_to_perm"]), _ptr(out["active_experts"]),
        _ptr(out["active_count"]), _ptr(out["num_tokens_post_padded"]), _ptr(err_word),
        _stream(stream)))
    return out


def moe_topk_softmax(logits: torch.Tensor, top_k: int, ids: Optional[torch.Tensor] = None,
                     w: Optional[torch.Tensor] = None, stream=None):
    M, E = logits.shape
    if ids is None:
        ids = torch.empty(M, top_k, dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty(M, top_k, dtype=torch.float32, device=logits.device)
    _check("moe_topk_softmax", load().moe_topk_softmax(_ptr(logits), M, E, top_k, _ptr(ids),
                                                       _ptr(w), _stream(stream)))
    return ids, w


def _dense(name: str, t: torch.Tensor, dtype: torch.dtype, shape: tuple) -> None:
    """The C entry points read plain row-major buffers: refuse anything else."""
    if t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != shape:
        raise ValueError(f"{name}: want a contiguous {dtype} tensor of shape {shape}, "
                         f"got {t.dtype} {tuple(t.shape)}")


def moe_router_logits(x: torch.Tensor, router_weight: torch.Tensor,
                      logits: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """fp32 logits [M, E] = x [M, H] (bf16) times router_weight [E, H] (bf16) transposed."""
    M, H = x.shape
    E = router_weight.shape[0]
    _dense("x", x, torch.bfloat16, (M, H))
    _dense("router_weight", router_weight, torch.bfloat16, (E, H))
    if logits is None:
        logits = torch.empty(M, E, dtype=torch.float32, device=x.device)
    _dense("logits", logits, torch.float32, (M, E))
    _check("moe_router_logits", load().moe_router_logits(_ptr(x), _ptr(router_weight), M, H, E,
                                                         _ptr(logits), _stream(stream)))
    return logits


def _sp(x: Optional[Experts]):
    return None if x is None else ctypes.pointer(x._struct)


def moe_grouped_gate_up(routed: Experts, shared: Optional[Experts], x: torch.Tensor, top_k: int,
                        tables: dict, h: torch.Tensor, h_shared: Optional[torch.Tensor] = None,
                        path: int = PATH_AUTO, stream=None) -> None:
    M = x.shape[0]
    _check("moe_grouped_gate_up", load().moe_grouped_gate_up(
        _sp(routed), _sp(shared), _ptr(x), M, top_k, _ptr(tables["expert_offsets"]),
        _ptr(tables["sorted_token_ids"]), _ptr(tables["active_experts"]),
        _ptr(tables["active_count"]), _ptr(h), _ptr(h_shared), path, _stream(stream)))


def moe_grouped_down(routed: Experts, shared: Optional[Experts], h: torch.Tensor,
                     h_shared: Optional[torch.Tensor], M: int, top_k: int, tables: dict,
                     y: torch.Tensor, y_shared: Optional[torch.Tensor] = None,
                     path: int = PATH_AUTO, stream=None) -> None:
    _check("moe_grouped_down", load().moe_grouped_down(
        _sp(routed), _sp(shared), _ptr(h), _ptr(h_shared), M, top_k,
        _ptr(tables["expert_offsets"]), _ptr(tables["sorted_token_ids"]),
        _ptr(tables["active_experts"]), _ptr(tables["active_count"]), _ptr(y), _ptr(y_shared),
        path, _stream(stream)))


def moe_blend(y: torch.Tensor, topk_w: torch.Tensor, token_to_perm: torch.Tensor,
              y_shared: Optional[torch.Tensor], out: torch.Tensor, top_k: int,
              x: Optional[torch.Tensor] = None, shared_gate: Optional[torch.Tensor] = None,
              stream=None) -> None:
    """shared_gate (bf16 [H]) with x (bf16 [M, H]) gates the shared term by
    sigmoid(x[t] . shared_gate)."""
    M, H = out.shape
    if shared_gate is not None:
        if x is None:
            raise ValueError("shared_gate: x is required to compute the gate")
        _dense("x", x, torch.bfloat16, (M, H))
        _dense("shared_gate", shared_gate, torch.bfloat16, (H,))
    _check("moe_blend", load().moe_blend(_ptr(y), _ptr(topk_w), _ptr(token_to_perm),
                                         _ptr(y_shared), _ptr(x), _ptr(shared_gate), _ptr(out),
                                         M, top_k, H, _stream(stream)))


def workspace_bytes(layer: LayerDesc, max_M: int) -> int:
    nbytes = load().moe_decode_layer_workspace_bytes(ctypes.pointer(layer._struct), max_M)
    if nbytes == 0:
        raise MoeError("moe_decode_layer_workspace_bytes", MOE_EINVAL)
    return nbytes


def alloc_workspace(layer: LayerDesc, max_M: int, device="cuda") -> torch.Tensor:
    return torch.zeros(workspace_bytes(layer, max_M), dtype=torch.uint8, device=device)


def workspace_view(layer: LayerDesc, M: int, ws: torch.Tensor) -> dict:
    """Tensors aliasing the layer's intermediates inside the workspace."""
    v = _WsView()
    _check("moe_decode_layer_workspace_view",
           load().moe_decode_layer_workspace_view(ctypes.pointer(layer._struct), M,
                                                  ctypes.byref(v)))
    k, E = layer.top_k, layer.num_experts
    H, I = layer.routed.hidden, layer.routed.inter
    Is = layer.shared.inter if layer.shared is not None else 0

    def sl(off, count, dtype):
        nb = count * torch.tensor([], dtype=dtype).element_size()
        return ws[off: off + nb].view(dtype)

    tc = {}
    mt = v.max_total
    f4 = layer.routed.fmt in (FMT_NVFP4_G16, FMT_NVFP4_GATE_UP)
    if v.tc_h_terms and f4:
        # the NVFP4 tensor-core kernel: f16 h terms (hi, lo) [2][max_total][I],
        # the f16 x table [H/128][2][NT][64] of NT = 16 or 32 token columns
        nt = F4_TOKEN_COLUMNS_SMALL if M <= F4_TOKEN_COLUMNS_SMALL else F4_TOKEN_COLUMNS
        tc = dict(
            tc_h_terms=sl(v.tc_h_terms, 2 * mt * I, torch.float16).view(2, mt, I),
            tc_h_scale=sl(v.tc_h_scale, mt * (I // 128), torch.float32).view(mt, I // 128),
            tc_items=sl(v.tc_items, 4 * v.cap, torch.int32).view(v.cap, 4),
            tc_x_table=sl(v.tc_x_terms, nt * H, torch.float16).view(H // 128, 2, nt, 64),
            tc_x_scale=sl(v.tc_x_scale, nt, torch.float32))
    elif v.tc_h_terms:   # the FP8 tensor-core kernel's h terms and the active table
        tc = dict(
            tc_h_terms=sl(v.tc_h_terms, 3 * mt * I, torch.uint8).view(3, mt, I),
            tc_h_scale=sl(v.tc_h_scale, mt * (I // 128), torch.float32).view(mt, I // 128),
            tc_items=sl(v.tc_items, 4 * v.cap, torch.int32).view(v.cap, 4))
    if v.tc_x_terms and not f4 and M <= TOKEN_FORM_ROWS:   # x terms by token [H/128][2][16][128]
        tc.update(
            tc_x_table=sl(v.tc_x_terms, 2 * 16 * H, torch.uint8).view(H // 128, 2, 16, 128),
            tc_x_scale=sl(v.tc_x_scale, 16, torch.float32))
    elif v.tc_x_terms and not f4:   # x terms by sorted row [2][max_total][H]
        tc.update(
            tc_x_terms=sl(v.tc_x_terms, 2 * mt * H, torch.uint8).view(2, mt, H),
            tc_x_scale=sl(v.tc_x_scale, mt, torch.float32))

    return dict(
        topk_ids=sl(v.topk_ids, M * k, torch.int32), topk_w=sl(v.topk_w, M * k, torch.float32),
        sorted_token_ids=sl(v.sorted_token_ids, v.max_total, torch.int32),
        sorted_expert_ids=sl(v.sorted_expert_ids, v.max_blocks, torch.int32),
        expert_offsets=sl(v.expert_offsets, E + 1, torch.int32),
        token_to_perm=sl(v.token_to_perm, M * k, torch.int32),
        active_experts=sl(v.active_experts, v.cap, torch.int32),
        active_count=sl(v.active_count, 1, torch.int32),
        num_tokens_post_padded=sl(v.num_tokens_post_padded, 1, torch.int32),
        h=sl(v.h, v.max_total * I, torch.float32).view(v.max_total, I),
        h_shared=sl(v.h_shared, M * Is, torch.float32).view(M, Is),
        y=sl(v.y, v.max_total * H, torch.float32).view(v.max_total, H),
        y_shared=sl(v.y_shared, M * H, torch.float32).view(M, H),
        router_logits=sl(v.router_logits, M * E, torch.float32).view(M, E),
        shared_gate=sl(v.shared_gate, M, torch.float32),
        max_total=v.max_total, max_blocks=v.max_blocks, cap=v.cap, **tc)


def moe_decode_layer_launches(layer: LayerDesc, M: int, with_logits: int = 1) -> int:
    """Kernels one moe_decode_layer call enqueues (host only); with_logits 0:
    ids given, 1: logits given, 2: logits computed from x (hidden in)."""
    n = load().moe_decode_layer_launches(ctypes.pointer(layer._struct), M, int(with_logits))
    if n < 0:
        raise MoeError("moe_decode_layer_launches", MOE_EINVAL)
    return n


def moe_decode_layer(layer: LayerDesc, x: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                     router_logits: Optional[torch.Tensor] = None,
                     topk_ids: Optional[torch.Tensor] = None,
                     topk_w: Optional[torch.Tensor] = None,
                     err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    M = x.shape[0]
    _check("moe_decode_layer", load().moe_decode_layer(
        ctypes.pointer(layer._struct), _ptr(x), M, _ptr(router_logits), _ptr(topk_ids),
        _ptr(topk_w), _ptr(out), _ptr(workspace), workspace.numel(), _ptr(err_word),
        _stream(stream)))


def moe_decode_experts(layer: LayerDesc, x: torch.Tensor, out: torch.Tensor,
                       workspace: torch.Tensor, err_word: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """The expert half of moe_decode_layer (grouped gate+up, down, blend) on
    the routing and alignment tables that an earlier moe_decode_layer call
    with the same layer and M left in this workspace, with this x."""
    M = x.shape[0]
    _check("moe_decode_experts", load().moe_decode_experts(
        ctypes.pointer(layer._struct), _ptr(x), M, _ptr(out), _ptr(workspace),
        workspace.numel(), _ptr(err_word), _stream(stream)))


NOALLOC_SCRATCH_BYTES = 32 << 20


def moe_decode_layer_noalloc(layer: LayerDesc, x: torch.Tensor, out: torch.Tensor,
                             router_logits: Optional[torch.Tensor] = None,
                             topk_ids: Optional[torch.Tensor] = None,
                             topk_w: Optional[torch.Tensor] = None,
                             err_word: Optional[torch.Tensor] = None, stream=None) -> None:
    """moe_decode_layer without a caller workspace, for callers that cannot
    allocate device memory: the library's fixed device array (32 MiB, shared
    by every call on the device) serves as the workspace."""
    M = x.shape[0]
    _check("moe_decode_layer_noalloc", load().moe_decode_layer_noalloc(
        ctypes.pointer(layer._struct), _ptr(x), M, _ptr(router_logits), _ptr(topk_ids),
        _ptr(topk_w), _ptr(out), _ptr(err_word), _stream(stream)))
