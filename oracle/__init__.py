"""fp64 CPU oracle for the quantized sparse MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` call it; the CUDA library does not, and the
two share no code.  The arithmetic lives in ``oracle.c`` (plain loops in
double, each function citing the passage it follows); this module compiles
it with gcc on first use and marshals numpy arrays through ctypes.

All bf16 / fp16 inputs are passed as their uint16 bit patterns.

Parity status of every function: pinned (see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

Q8_0 = 0
AFFINE4_G64 = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _QMat(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int32), ("experts", ctypes.c_int32),
                ("rows", ctypes.c_int32), ("cols", ctypes.c_int32),
                ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("biases", ctypes.c_void_p)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = ctypes.c_double
            lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_f16_to_f64.restype = ctypes.c_double
            lib.orc_weight.argtypes = [ctypes.POINTER(_QMat), ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int]
            lib.orc_weight.restype = ctypes.c_double
            lib.orc_row_bytes.argtypes = [i32, i32]
            lib.orc_row_bytes.restype = ctypes.c_int64
            lib.orc_qmatvec.argtypes = [ctypes.POINTER(_QMat), ctypes.c_int,
                                        P, P]
            lib.orc_router_logits.argtypes = [P, P, P, i32, i32, i32, P]
            lib.orc_topk.argtypes = [P, i32, i32, i32, i32, P, P]
            lib.orc_topk_sel.argtypes = [P, P, i32, i32, i32, i32, P, P]
            lib.orc_shared_gate.argtypes = [P, P, i32, i32, P]
            lib.orc_group.argtypes = [P, i32, i32, i32, i32, P, P, P, P, P, P]
            lib.orc_group.restype = ctypes.c_int
            lib.orc_silu.argtypes = [ctypes.c_double]
            lib.orc_silu.restype = ctypes.c_double
            lib.orc_expert_ffn.argtypes = [ctypes.POINTER(_QMat),
                                           ctypes.POINTER(_QMat), ctypes.c_int,
                                           P, P, P, P]
            lib.orc_moe_layer.argtypes = [P, i32, P, P, i32,
                                          ctypes.POINTER(_QMat),
                                          ctypes.POINTER(_QMat),
                                          ctypes.POINTER(_QMat),
                                          ctypes.POINTER(_QMat), P, i32, P]
            lib.orc_moe_layer_ex.argtypes = [P, i32, P, P, i32,
                                             ctypes.POINTER(_QMat),
                                             ctypes.POINTER(_QMat),
                                             ctypes.POINTER(_QMat),
                                             ctypes.POINTER(_QMat), P, P, i32, P]
            lib.orc_q8_gemv.argtypes = [P, P, P, i32, i32, P]
            lib.orc_q8_quantize_x.argtypes = [P, i32, P, P]
            lib.orc_q8_gemv_i8.argtypes = [P, P, P, P, i32, i32, P]
            lib.orc_max_threads.restype = ctypes.c_int
            lib.orc_set_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        a = a.view(np.uint16) if a.dtype.itemsize == 2 else a.astype(np.uint16)
    return a


class QWeights:
    """A quantized weight tensor [experts, rows, cols] as numpy arrays.

    Q8_0:        codes int8 [E, rows, cols], scales fp16-bits [E, rows, cols/32]
    AFFINE4_G64: codes uint32 [E, rows, cols/8] (input c in bits 4*(c%8)..),
                 scales / biases fp16-bits [E, rows, cols/64]
    """

    def __init__(self, qtype, codes, scales, biases=None):
        self.qtype = int(qtype)
        self.codes = np.ascontiguousarray(codes)
        self.scales = _u16(scales)
        self.biases = None if biases is None else _u16(biases)
        self.experts, self.rows = self.codes.shape[0], self.codes.shape[1]
        if self.qtype == Q8_0:
            assert self.codes.dtype == np.int8
            self.cols = self.codes.shape[2]
        else:
            assert self.codes.dtype == np.uint32 and self.biases is not None
            self.cols = self.codes.shape[2] * 8
        self._s = _QMat(self.qtype, self.experts, self.rows, self.cols,
                        self.codes.ctypes.data, self.scales.ctypes.data,
                        None if self.biases is None else self.biases.ctypes.data)

    @property
    def struct(self):
        return ctypes.byref(self._s)


def bf16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = _u16(bits)
    return np.array([lib.orc_bf16_to_f64(int(v)) for v in b.ravel()],
                    dtype=np.float64).reshape(b.shape)


def f16_to_f64(bits) -> np.ndarray:
    lib = _load()
    b = _u16(bits)
    return np.array([lib.orc_f16_to_f64(int(v)) for v in b.ravel()],
                    dtype=np.float64).reshape(b.shape)


def weight(w: QWeights, e: int, n: int, c: int) -> float:
    return _load().orc_weight(w.struct, e, n, c)


def row_bytes(qtype: int, cols: int) -> int:
    return int(_load().orc_row_bytes(qtype, cols))


def dequant_expert(w: QWeights, e: int) -> np.ndarray:
    """W[e] as a dense float64 [rows, cols] matrix (weight by weight)."""
    lib = _load()
    out = np.empty((w.rows, w.cols), np.float64)
    for n in range(w.rows):
        for c in range(w.cols):
            out[n, c] = lib.orc_weight(w.struct, e, n, c)
    return out


def qmatvec(w: QWeights, e: int, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(w.rows, np.float64)
    _load().orc_qmatvec(w.struct, e, _ptr(x), _ptr(y))
    return y


def router_logits(x_bf16, w_router, bias=None) -> np.ndarray:
    x = _u16(x_bf16)
    wr = np.ascontiguousarray(w_router, dtype=np.float32)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, E), np.float64)
    _load().orc_router_logits(_ptr(x), _ptr(wr), _ptr(b), T, H, E, _ptr(out))
    return out


def topk(logits, k: int, renormalize: bool = True):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = l.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().orc_topk(_ptr(l), T, E, k, int(bool(renormalize)), _ptr(idx),
                     _ptr(w))
    return idx, w


def topk_sel(sel_logits, weight_logits, k: int, renormalize: bool = True):
    """Top k by sel_logits, routing weights from weight_logits."""
    s = np.ascontiguousarray(sel_logits, dtype=np.float64)
    w = np.ascontiguousarray(weight_logits, dtype=np.float64)
    T, E = s.shape
    assert w.shape == (T, E)
    idx = np.empty((T, k), np.int32)
    out = np.empty((T, k), np.float64)
    _load().orc_topk_sel(_ptr(s), _ptr(w), T, E, k, int(bool(renormalize)), _ptr(idx),
                         _ptr(out))
    return idx, out


def route(x_bf16, w_router, k: int, bias=None, renormalize: bool = True,
          bias_select_only: bool = False):
    """Router: logits + bias select the experts; the weights come from the
    same logits, or from the logits without the bias (bias_select_only)."""
    sel = router_logits(x_bf16, w_router, bias)
    if bias is None or not bias_select_only:
        return topk(sel, k, renormalize)
    return topk_sel(sel, router_logits(x_bf16, w_router, None), k, renormalize)


def shared_gate(x_bf16, w_sg) -> np.ndarray:
    """g[t] = sigmoid(x[t] . w_sg) in fp64."""
    x = _u16(x_bf16)
    T, H = x.shape
    w = np.ascontiguousarray(w_sg, dtype=np.float32)
    assert w.shape == (H,)
    g = np.empty(T, np.float64)
    _load().orc_shared_gate(_ptr(x), _ptr(w), T, H, _ptr(g))
    return g


def group(topk_idx, E: int, tile_rows: int):
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    T, k = idx.shape
    A = T * k
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(A, np.int32)
    inv_perm = np.empty(A, np.int32)
    max_tiles = A // tile_rows + E + 1
    tile_map = np.empty(2 * max_tiles, np.int32)
    n_tiles = np.zeros(1, np.int32)
    rc = _load().orc_group(_ptr(idx), T, k, E, tile_rows, _ptr(counts),
                           _ptr(offsets), _ptr(perm), _ptr(inv_perm),
                           _ptr(tile_map), _ptr(n_tiles))
    if rc != 0:
        raise ValueError("expert id out of range")
    nt = int(n_tiles[0])
    return dict(counts=counts, offsets=offsets, perm=perm, inv_perm=inv_perm,
                tile_map=tile_map[:2 * nt].reshape(nt, 2), n_tiles=nt)


def silu(g: float) -> float:
    return _load().orc_silu(float(g))


def expert_ffn(gate_up: QWeights, down: QWeights, e: int, x: np.ndarray):
    """Returns (o [H], gu [2I], h [I]) for one expert and one token."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    H, I = down.rows, down.cols
    o = np.empty(H, np.float64)
    gu = np.empty(2 * I, np.float64)
    h = np.empty(I, np.float64)
    _load().orc_expert_ffn(gate_up.struct, down.struct, e, _ptr(x), _ptr(o),
                           _ptr(gu), _ptr(h))
    return o, gu, h


def moe_layer(x_bf16, topk_idx, topk_w, gate_up: QWeights, down: QWeights,
              shared_gate_up: QWeights, shared_down: QWeights,
              tokens=None, shared_w=None) -> np.ndarray:
    """fp64 layer output for `tokens` (default: all), shape [len(tokens), H];
    shared_w [T] scales the shared expert per token (default 1)."""
    x = _u16(x_bf16)
    T, H = x.shape
    idx = np.ascontiguousarray(topk_idx, dtype=np.int32)
    w = np.ascontiguousarray(topk_w, dtype=np.float64)
    k = idx.shape[1]
    toks = np.arange(T, dtype=np.int32) if tokens is None else \
        np.ascontiguousarray(tokens, dtype=np.int32)
    y = np.empty((len(toks), H), np.float64)
    if shared_w is None:
        _load().orc_moe_layer(_ptr(x), H, _ptr(idx), _ptr(w), k, gate_up.struct,
                              down.struct, shared_gate_up.struct,
                              shared_down.struct, _ptr(toks), len(toks), _ptr(y))
    else:
        sw = np.ascontiguousarray(shared_w, dtype=np.float64)
        assert sw.shape == (T,)
        _load().orc_moe_layer_ex(_ptr(x), H, _ptr(idx), _ptr(w), k, gate_up.struct,
                                 down.struct, shared_gate_up.struct,
                                 shared_down.struct, _ptr(sw), _ptr(toks), len(toks),
                                 _ptr(y))
    return y


def q8_gemv(x_bf16, q, d) -> np.ndarray:
    x = _u16(x_bf16).ravel()
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = _u16(d)
    N, K = q.shape
    y = np.empty(N, np.float64)
    _load().orc_q8_gemv(_ptr(x), _ptr(q), _ptr(d), N, K, _ptr(y))
    return y


def q8_quantize_x(x_bf16):
    """Activation x [K] -> (int8 codes [K], fp32 block scales [K/32])."""
    x = _u16(x_bf16).ravel()
    K = x.size
    q = np.empty(K, np.int8)
    d = np.empty(K // 32, np.float32)
    _load().orc_q8_quantize_x(_ptr(x), K, _ptr(q), _ptr(d))
    return q, d


def q8_gemv_i8(qx, dx, q, d) -> np.ndarray:
    """Q8_0 GEMV on a quantized activation (q8_quantize_x), fp64."""
    qx = np.ascontiguousarray(qx, dtype=np.int8)
    dx = np.ascontiguousarray(dx, dtype=np.float32)
    q = np.ascontiguousarray(q, dtype=np.int8)
    d = _u16(d)
    N, K = q.shape
    y = np.empty(N, np.float64)
    _load().orc_q8_gemv_i8(_ptr(qx), _ptr(dx), _ptr(q), _ptr(d), N, K, _ptr(y))
    return y


def max_threads() -> int:
    return int(_load().orc_max_threads())


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))
