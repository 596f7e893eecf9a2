"""Python binding of the qsmoe CUDA library (quantized sparse MoE FFN layer).

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels (``_build/libqsmoe.so``, built from ``csrc/`` for sm_103a).
torch supplies device memory and the stream; the functions here allocate
outputs and workspaces with torch when the caller does not pass them, call
the C entry point of the same name, and raise ``QSMError`` on a non-zero
status.  There is no fallback: if the library cannot be built or loaded,
importing the binding's functions fails.

Entry points (see include/qsmoe.h for the exact contracts):
  moe_route, moe_group_tokens, moe_ffn_forward, q8_gemv
plus ``MoEForward``, which owns the buffers of one layer call and issues the
three calls in order on one stream.
"""
from __future__ import annotations

import ctypes
import dataclasses
import threading

import torch

from . import build as _build

Q8_0 = 0
AFFINE4_G64 = 1

DEV_BAD_EXPERT_ID = 1
DEV_NONFINITE = 2
DEV_FP16_RANGE = 4
DEV_TIMEOUT = 8

_lock = threading.Lock()
_lib = None


class QSMError(RuntimeError):
    pass


class QWeightsC(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int32), ("experts", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("cols", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p)]


class MoELayerC(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("gate_up", QWeightsC), ("down", QWeightsC),
                ("shared_gate_up", QWeightsC), ("shared_down", QWeightsC),
                ("shared_gate", ctypes.c_void_p)]


class GroupingC(ctypes.Structure):
    _fields_ = [("counts", ctypes.c_void_p), ("offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("inv_perm", ctypes.c_void_p),
                ("tile_map", ctypes.c_void_p), ("n_tiles", ctypes.c_void_p),
                ("tile_rows", ctypes.c_int32), ("max_tiles", ctypes.c_int32)]


def lib() -> ctypes.CDLL:
    """The loaded C library (built in-tree on first use if stale)."""
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(_build.build())
            P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
            st = ctypes.c_int
            L.moe_route_workspace_bytes.argtypes = [i32, i32, i32]
            L.moe_route_workspace_bytes.restype = sz
            L.moe_route.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P,
                                    sz, P, P]
            L.moe_route.restype = st
            L.moe_group_max_tiles.argtypes = [i32, i32, i32, i32]
            L.moe_group_max_tiles.restype = i32
            L.moe_group_tokens.argtypes = [P, i32, i32, i32,
                                           ctypes.POINTER(GroupingC), P, P]
            L.moe_group_tokens.restype = st
            L.moe_route_group.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P,
                                          ctypes.POINTER(GroupingC), P, sz, P, P]
            L.moe_route_group.restype = st
            L.moe_ffn_tile_rows.argtypes = [i32]
            L.moe_ffn_tile_rows.restype = i32
            L.moe_ffn_workspace_bytes.argtypes = [ctypes.POINTER(MoELayerC),
                                                  i32]
            L.moe_ffn_workspace_bytes.restype = sz
            L.moe_ffn_forward.argtypes = [ctypes.POINTER(MoELayerC), P, i32, P,
                                          P, ctypes.POINTER(GroupingC), P, P,
                                          P, sz, P, P]
            L.moe_ffn_forward.restype = st
            L.moe_ffn_forward_noalloc.argtypes = [
                ctypes.POINTER(MoELayerC), P, i32, P, P,
                ctypes.POINTER(GroupingC), P, P, P, P]
            L.moe_ffn_forward_noalloc.restype = st
            L.q8_gemv.argtypes = [P, P, P, i32, i32, P, P, P]
            L.q8_gemv.restype = st
            L.q8_quantize_x.argtypes = [P, i32, P, P, P, P]
            L.q8_quantize_x.restype = st
            L.q8_gemv_i8.argtypes = [P, P, P, P, i32, i32, P, P, P]
            L.q8_gemv_i8.restype = st
            L.qsm_status_str.argtypes = [st]
            L.qsm_status_str.restype = ctypes.c_char_p
            L.qsm_abi_version.restype = i32
            L.qsm_debug_force_path.argtypes = [i32]
            L.qsm_debug_force_path.restype = st
            L.moe_layer_workspace_bytes.argtypes = [ctypes.POINTER(MoELayerC), i32, i32]
            L.moe_layer_workspace_bytes.restype = sz
            L.moe_layer_forward.argtypes = [ctypes.POINTER(MoELayerC), P, i32, i32, P,
                                            P, i32, P, P, P, P, P, sz, P, P]
            L.moe_layer_forward.restype = st
            L.moe_decode_layer_workspace_bytes.argtypes = [ctypes.POINTER(MoELayerC), i32]
            L.moe_decode_layer_workspace_bytes.restype = sz
            L.moe_decode_layer.argtypes = [ctypes.POINTER(MoELayerC), P, i32, P, P, i32,
                                           P, P, P, P, P, sz, P, P]
            L.moe_decode_layer.restype = st
            L.qsm_debug_barrier_skew.argtypes = [i32]
            L.qsm_debug_barrier_skew.restype = st
            L.qsm_debug_gu_dump.argtypes = [P, sz]
            L.qsm_debug_gu_dump.restype = st
            L.qsm_decode_layer_fits.argtypes = [ctypes.POINTER(MoELayerC), i32, i32, i32]
            L.qsm_decode_layer_fits.restype = i32
            L.qsm_launch_count.argtypes = []
            L.qsm_launch_count.restype = ctypes.c_uint64
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        msg = lib().qsm_status_str(status).decode()
        raise QSMError(f"{what}: {msg} (status {status})")


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _status(dev_status, device) -> torch.Tensor:
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=device)
    return dev_status


def _u16(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype in (torch.bfloat16, torch.float16) and t.is_contiguous()
    return t


# ------------------------------------------------------------------ weights

def qweights_c(qt) -> QWeightsC:
    """C view of a quantized tensor (any object with qtype, experts, rows,
    cols, codes, scales, biases as contiguous CUDA tensors)."""
    return QWeightsC(int(qt.qtype), int(qt.experts), int(qt.rows),
                     int(qt.cols), qt.codes.data_ptr(), qt.scales.data_ptr(),
                     None if qt.biases is None else qt.biases.data_ptr())


class Layer:
    """C view of one MoE layer; keeps the torch tensors alive."""

    def __init__(self, H, I, E, k, gate_up, down, shared_gate_up,
                 shared_down, w_router, logit_bias=None, shared_gate=None):
        self.H, self.I, self.E, self.k = H, I, E, k
        self.w_router = w_router
        self.logit_bias = logit_bias
        self.shared_gate = shared_gate  # [H] fp32 or None (ungated)
        self._keep = (gate_up, down, shared_gate_up, shared_down, shared_gate)
        self.qtype = int(gate_up.qtype)
        self.c = MoELayerC(H, I, E, k, qweights_c(gate_up), qweights_c(down),
                           qweights_c(shared_gate_up), qweights_c(shared_down),
                           _p(shared_gate))

    @classmethod
    def from_synth(cls, L, shared_gate=None) -> "Layer":
        s = L.shape
        return cls(s.H, s.I, s.E, s.k, L.gate_up, L.down, L.shared_gate_up,
                   L.shared_down, L.w_router, L.logit_bias, shared_gate)


ROUTE_RENORMALIZE = 1        # weights: softmax over the selected experts
ROUTE_BIAS_SELECT_ONLY = 2   # the logit bias selects, the weights ignore it


def route_flags(renormalize=True, bias_select_only=False) -> int:
    """The routing calls' flags word: renormalize is a bool, or already a
    flags word (the library rejects unknown bits)."""
    return int(renormalize) | (ROUTE_BIAS_SELECT_ONLY if bias_select_only else 0)


# ------------------------------------------------------------------ router

def route_workspace_bytes(T: int, H: int, E: int) -> int:
    return int(lib().moe_route_workspace_bytes(T, H, E))


def moe_route(x: torch.Tensor, w_router: torch.Tensor, k: int,
              logit_bias: torch.Tensor | None = None, renormalize=True,
              topk_idx=None, topk_w=None, workspace=None, dev_status=None,
              stream=None, *, bias_select_only=False):
    """Router logits, top-k and routing weights -> (topk_idx, topk_w)."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(route_workspace_bytes(T, H, E),
                                dtype=torch.uint8, device=dev)
    dev_status = _status(dev_status, dev)
    _check(lib().moe_route(_p(_u16(x)), _p(w_router), _p(logit_bias), T, H, E,
                           k, route_flags(renormalize, bias_select_only), _p(topk_idx),
                           _p(topk_w),
                           _p(workspace), workspace.numel(), _p(dev_status),
                           _stream(stream)), "moe_route")
    return topk_idx, topk_w


# ---------------------------------------------------------------- grouping

@dataclasses.dataclass
class Grouping:
    counts: torch.Tensor
    offsets: torch.Tensor
    perm: torch.Tensor
    inv_perm: torch.Tensor
    tile_map: torch.Tensor
    n_tiles: torch.Tensor
    tile_rows: int
    max_tiles: int

    @classmethod
    def empty(cls, T: int, k: int, E: int, tile_rows: int, device):
        mt = int(lib().moe_group_max_tiles(T, k, E, tile_rows))
        i32 = dict(dtype=torch.int32, device=device)
        A = T * k
        return cls(torch.empty(E, **i32), torch.empty(E + 1, **i32),
                   torch.empty(max(A, 1), **i32), torch.empty(max(A, 1), **i32),
                   torch.empty(max(2 * mt, 2), **i32), torch.empty(1, **i32),
                   tile_rows, mt)

    @property
    def c(self) -> GroupingC:
        return GroupingC(self.counts.data_ptr(), self.offsets.data_ptr(),
                         self.perm.data_ptr(), self.inv_perm.data_ptr(),
                         self.tile_map.data_ptr(), self.n_tiles.data_ptr(),
                         self.tile_rows, self.max_tiles)


def group_max_tiles(T: int, k: int, E: int, tile_rows: int) -> int:
    return int(lib().moe_group_max_tiles(T, k, E, tile_rows))


def moe_group_tokens(topk_idx: torch.Tensor, E: int, tile_rows: int,
                     out: Grouping | None = None, dev_status=None,
                     stream=None) -> Grouping:
    T, k = topk_idx.shape
    if out is None:
        out = Grouping.empty(T, k, E, tile_rows, topk_idx.device)
    dev_status = _status(dev_status, topk_idx.device)
    gc = out.c
    _check(lib().moe_group_tokens(_p(topk_idx), T, k, E, ctypes.byref(gc),
                                  _p(dev_status), _stream(stream)),
           "moe_group_tokens")
    return out


def moe_route_group(x: torch.Tensor, w_router: torch.Tensor, k: int,
                    grouping: Grouping, logit_bias=None, renormalize=True,
                    topk_idx=None, topk_w=None, workspace=None, dev_status=None,
                    stream=None, raise_unsupported=True, *,
                    bias_select_only=False):
    """Router + grouping in one launch (T <= 8).  Returns (topk_idx, topk_w),
    or None when the shape is not supported and raise_unsupported is False.
    The workspace is the router's (route_workspace_bytes, zero-initialised
    once)."""
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(route_workspace_bytes(T, H, E), 256),
                                dtype=torch.uint8, device=dev)
    dev_status = _status(dev_status, dev)
    gc = grouping.c
    st = lib().moe_route_group(_p(_u16(x)), _p(w_router), _p(logit_bias), T, H, E,
                               k, route_flags(renormalize, bias_select_only),
                               _p(topk_idx),
                               _p(topk_w), ctypes.byref(gc), _p(workspace),
                               workspace.numel(), _p(dev_status), _stream(stream))
    if st == 2 and not raise_unsupported:
        return None
    _check(st, "moe_route_group")
    return topk_idx, topk_w


# --------------------------------------------------------------------- FFN

def ffn_tile_rows(T: int) -> int:
    return int(lib().moe_ffn_tile_rows(T))


def ffn_workspace_bytes(layer: Layer, T: int) -> int:
    return int(lib().moe_ffn_workspace_bytes(ctypes.byref(layer.c), T))


def moe_ffn_forward(layer: Layer, x: torch.Tensor, topk_idx: torch.Tensor,
                    topk_w: torch.Tensor, grouping: Grouping, y=None,
                    y_f32=None, workspace=None, dev_status=None, stream=None):
    """Expert FFNs + combine -> y (bf16); y_f32=True also returns the fp32
    result before rounding."""
    T, H = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y_f32 is True:
        y_f32 = torch.empty((T, H), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(ffn_workspace_bytes(layer, T), 256),
                                dtype=torch.uint8, device=dev)
    dev_status = _status(dev_status, dev)
    gc = grouping.c
    _check(lib().moe_ffn_forward(ctypes.byref(layer.c), _p(_u16(x)), T,
                                 _p(topk_idx), _p(topk_w), ctypes.byref(gc),
                                 _p(y), _p(y_f32 if y_f32 is not False else None),
                                 _p(workspace), workspace.numel(),
                                 _p(dev_status), _stream(stream)),
           "moe_ffn_forward")
    return y, (y_f32 if isinstance(y_f32, torch.Tensor) else None)


def moe_ffn_forward_noalloc(layer: Layer, x: torch.Tensor,
                            topk_idx: torch.Tensor, topk_w: torch.Tensor,
                            grouping: Grouping, y=None, y_f32=None,
                            dev_status=None, stream=None):
    """moe_ffn_forward with the library's built-in scratch (T <= 64): for
    callers that cannot allocate device memory.  Outputs as moe_ffn_forward."""
    T, H = x.shape
    dev = x.device
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y_f32 is True:
        y_f32 = torch.empty((T, H), dtype=torch.float32, device=dev)
    dev_status = _status(dev_status, dev)
    gc = grouping.c
    _check(lib().moe_ffn_forward_noalloc(
        ctypes.byref(layer.c), _p(_u16(x)), T, _p(topk_idx), _p(topk_w),
        ctypes.byref(gc), _p(y), _p(y_f32 if y_f32 is not False else None),
        _p(dev_status), _stream(stream)), "moe_ffn_forward_noalloc")
    return y, (y_f32 if isinstance(y_f32, torch.Tensor) else None)


def layer_workspace_bytes(layer: Layer, T: int, chunk: int) -> int:
    return int(lib().moe_layer_workspace_bytes(ctypes.byref(layer.c), T, chunk))


def moe_layer_forward(layer: Layer, x: torch.Tensor, chunk: int, renormalize=True,
                      bias_select_only=False, *,
                      y=None, y_f32=None, topk_idx=None, topk_w=None,
                      workspace=None, dev_status=None, stream=None):
    """The whole layer (route -> group -> FFN) in chunks of at most `chunk`
    tokens on one workspace sized for a chunk (zero-initialised once).
    Returns (y, y_f32 or None, topk_idx, topk_w)."""
    T, H = x.shape
    dev = x.device
    k = layer.k
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y_f32 is True:
        y_f32 = torch.empty((T, H), dtype=torch.float32, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(layer_workspace_bytes(layer, T, chunk), 256),
                                dtype=torch.uint8, device=dev)
    dev_status = _status(dev_status, dev)
    _check(lib().moe_layer_forward(
        ctypes.byref(layer.c), _p(_u16(x)), T, chunk, _p(layer.w_router),
        _p(layer.logit_bias), route_flags(renormalize, bias_select_only), _p(topk_idx),
        _p(topk_w),
        _p(y), _p(y_f32 if y_f32 is not False else None), _p(workspace),
        workspace.numel(), _p(dev_status), _stream(stream)), "moe_layer_forward")
    return y, (y_f32 if isinstance(y_f32, torch.Tensor) else None), topk_idx, topk_w


def decode_layer_workspace_bytes(layer: Layer, T: int) -> int:
    """0 when the one-launch decode layer does not support the layer or T."""
    return int(lib().moe_decode_layer_workspace_bytes(ctypes.byref(layer.c), T))


def moe_decode_layer(layer: Layer, x: torch.Tensor, renormalize=True,
                     bias_select_only=False, *, y=None, y_f32=None, topk_idx=None,
                     topk_w=None, workspace=None, dev_status=None, stream=None,
                     raise_unsupported=True):
    """The layer for T <= 8 tokens in one launch (router, selection, gate_up,
    down, combine).  The workspace must start zeroed and serve layers of one
    hidden size.  Returns (y, y_f32 or None, topk_idx, topk_w), or None when
    unsupported and raise_unsupported is False."""
    T, H = x.shape
    dev = x.device
    k = layer.k
    need = decode_layer_workspace_bytes(layer, T)
    if need == 0:
        if raise_unsupported:
            raise QSMError("moe_decode_layer: unsupported layer or token count")
        return None
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if y_f32 is True:
        y_f32 = torch.empty((T, H), dtype=torch.float32, device=dev)
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=dev)
    dev_status = _status(dev_status, dev)
    _check(lib().moe_decode_layer(
        ctypes.byref(layer.c), _p(_u16(x)), T, _p(layer.w_router), _p(layer.logit_bias),
        route_flags(renormalize, bias_select_only), _p(topk_idx), _p(topk_w), _p(y),
        _p(y_f32 if y_f32 is not False else None), _p(workspace), workspace.numel(),
        _p(dev_status), _stream(stream)), "moe_decode_layer")
    return y, (y_f32 if isinstance(y_f32, torch.Tensor) else None), topk_idx, topk_w


def debug_barrier_skew(skew: int) -> None:
    """Test hook: the decode layer's logit exchange waits for a call tag
    `skew` ahead of its own, so that every wait runs out (0 = off)."""
    _check(lib().qsm_debug_barrier_skew(int(skew)), "qsm_debug_barrier_skew")


def debug_gu_dump(buf: torch.Tensor | None) -> None:
    """Test hook: the gate_up kernels also write their fp32 gate and up
    values to buf (a CUDA float32 tensor), or stop when buf is None."""
    if buf is None:
        _check(lib().qsm_debug_gu_dump(None, 0), "qsm_debug_gu_dump")
    else:
        assert buf.dtype == torch.float32 and buf.is_cuda and buf.is_contiguous()
        _check(lib().qsm_debug_gu_dump(_p(buf), buf.numel()), "qsm_debug_gu_dump")


def force_path(mode: str | int) -> None:
    """Test hook: "auto", "decode" or "prefill"."""
    m = {"auto": 0, "decode": 1, "prefill": 2}.get(mode, mode)
    _check(lib().qsm_debug_force_path(int(m)), "qsm_debug_force_path")


def launch_count() -> int:
    """Kernels the library has launched (or recorded into a graph) so far."""
    return int(lib().qsm_launch_count())


# -------------------------------------------------------------------- GEMV

def q8_gemv(x: torch.Tensor, q: torch.Tensor, d: torch.Tensor, y=None,
            dev_status=None, stream=None) -> torch.Tensor:
    N, K = q.shape
    if y is None:
        y = torch.empty(N, dtype=torch.bfloat16, device=x.device)
    dev_status = _status(dev_status, x.device)
    _check(lib().q8_gemv(_p(_u16(x)), _p(q), _p(d), N, K, _p(y),
                         _p(dev_status), _stream(stream)), "q8_gemv")
    return y


# ---------------------------------------------------------- whole layer

class MoEForward:
    """Buffers of one MoE layer call for T tokens, and the call sequence on
    one stream (nothing is read back).  When moe_decode_layer supports the
    layer and T (T <= 8), one launch (one_launch=True); otherwise route ->
    group -> FFN, with the fused moe_route_group launch for T <= 8."""

    def __init__(self, layer: Layer, T: int, device="cuda", renormalize=True,
                 want_f32=False, fuse_route_group=True, *, bias_select_only=False,
                 one_launch=True):
        self.layer, self.T = layer, T
        self.renormalize = route_flags(renormalize, bias_select_only)
        self.fuse_route_group = fuse_route_group
        dl = decode_layer_workspace_bytes(layer, T) if one_launch else 0
        self.decode_ws = (torch.zeros(dl, dtype=torch.uint8, device=device)
                          if dl else None)
        k, E, H = layer.k, layer.E, layer.H
        i32 = dict(dtype=torch.int32, device=device)
        self.topk_idx = torch.empty((T, k), **i32)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.route_ws = torch.zeros(max(route_workspace_bytes(T, H, E), 256),
                                    dtype=torch.uint8, device=device)
        self.grouping = Grouping.empty(T, k, E, ffn_tile_rows(T), device)
        self.ffn_ws = torch.empty(max(ffn_workspace_bytes(layer, T), 256),
                                  dtype=torch.uint8, device=device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.y_f32 = (torch.empty((T, H), dtype=torch.float32, device=device)
                      if want_f32 else None)
        self.dev_status = torch.zeros(1, **i32)
        if self.decode_ws is not None:
            # the one-launch call's arguments, marshalled once (per call only x,
            # y and the stream change)
            self._dl_fn = lib().moe_decode_layer
            self._dl_head = (ctypes.byref(layer.c),)
            self._dl_mid = (T, _p(layer.w_router), _p(layer.logit_bias), self.renormalize,
                            _p(self.topk_idx), _p(self.topk_w))
            self._dl_tail = (_p(self.y_f32), _p(self.decode_ws), self.decode_ws.numel(),
                             _p(self.dev_status))

    def __call__(self, x: torch.Tensor, stream=None, out=None) -> torch.Tensor:
        """Run the layer on x [T, H] bf16; the result goes to out (a [T, H]
        bf16 tensor, contiguous) when given, else to self.y.  Returns it."""
        L = self.layer
        y = self.y if out is None else out
        if out is not None and (out.dtype != torch.bfloat16 or out.shape != self.y.shape
                                or not out.is_contiguous()):
            raise QSMError("MoEForward: out must be a contiguous [T, H] bf16 tensor")
        if self.decode_ws is not None:
            if x.dtype != torch.bfloat16 or not x.is_contiguous():
                raise QSMError("MoEForward: x must be a contiguous bf16 tensor")
            st = (torch.cuda.current_stream() if stream is None else stream).cuda_stream
            rc = self._dl_fn(*self._dl_head, ctypes.c_void_p(x.data_ptr()), *self._dl_mid,
                             ctypes.c_void_p(y.data_ptr()), *self._dl_tail,
                             ctypes.c_void_p(st))
            if rc:
                _check(rc, "moe_decode_layer")
            return y
        fused = None
        if self.fuse_route_group and self.T <= 8:
            fused = moe_route_group(x, L.w_router, L.k, self.grouping,
                                    L.logit_bias, self.renormalize,
                                    self.topk_idx, self.topk_w, self.route_ws,
                                    self.dev_status, stream,
                                    raise_unsupported=False)
        if fused is None:
            moe_route(x, L.w_router, L.k, L.logit_bias, self.renormalize,
                      self.topk_idx, self.topk_w, self.route_ws,
                      self.dev_status, stream)
            moe_group_tokens(self.topk_idx, L.E, self.grouping.tile_rows,
                             self.grouping, self.dev_status, stream)
        moe_ffn_forward(L, x, self.topk_idx, self.topk_w, self.grouping,
                        y, self.y_f32 if self.y_f32 is not None else False,
                        self.ffn_ws, self.dev_status, stream)
        return y


def q8_quantize_x(x: torch.Tensor, qx=None, dx=None, dev_status=None, stream=None):
    """x [K] bf16 -> (qx [K] int8, dx [K/32] fp32): the activation quantized
    once for the int8-activation GEMV."""
    K = x.numel()
    dev = x.device
    if qx is None:
        qx = torch.empty(K, dtype=torch.int8, device=dev)
    if dx is None:
        dx = torch.empty(K // 32, dtype=torch.float32, device=dev)
    dev_status = _status(dev_status, dev)
    _check(lib().q8_quantize_x(_p(_u16(x)), K, _p(qx), _p(dx), _p(dev_status),
                               _stream(stream)), "q8_quantize_x")
    return qx, dx


def q8_gemv_i8(qx: torch.Tensor, dx: torch.Tensor, q: torch.Tensor, d: torch.Tensor,
               y=None, dev_status=None, stream=None) -> torch.Tensor:
    N, K = q.shape
    if y is None:
        y = torch.empty(N, dtype=torch.bfloat16, device=q.device)
    dev_status = _status(dev_status, q.device)
    _check(lib().q8_gemv_i8(_p(qx), _p(dx), _p(q), _p(_u16(d)), N, K, _p(y),
                            _p(dev_status), _stream(stream)), "q8_gemv_i8")
    return y
