"""moe_ffn_forward_noalloc: the FFN entry point for callers that cannot
allocate device memory (it takes its scratch from an array built into the
library instead of a caller-provided workspace).

Called through the C ABI and compared with moe_ffn_forward, which gets a
workspace from the caller, on two calls in a row: the second call reuses the
built-in scratch that the first call left behind.  Both entry points run the
same kernels on the same inputs, so on the decode path (a fixed summation
order) the fp32 output is bit-equal too.  This file is named to be collected
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _helpers import tol_metric

pytestmark = pytest.mark.gpu

QSM_OK = 0
QSM_ERR_INVALID_ARGUMENT = 1
QSM_ERR_UNSUPPORTED = 2


def _call_noalloc(qsm, layer, x, fwd, y, y32, status, T=None):
    gc = fwd.grouping.c
    s = torch.cuda.current_stream()
    return qsm.lib().moe_ffn_forward_noalloc(
        ctypes.byref(layer.c), ctypes.c_void_p(x.data_ptr()),
        x.shape[0] if T is None else T,
        ctypes.c_void_p(fwd.topk_idx.data_ptr()),
        ctypes.c_void_p(fwd.topk_w.data_ptr()), ctypes.byref(gc),
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(y32.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(s.cuda_stream))


def _compare(qsm, shape, seed, Ts):
    L = synth.draw_layer(shape, "cuda", seed=seed)
    layer = qsm.Layer.from_synth(L)
    for call, T in enumerate(Ts):                # calls in a row
        x = synth.draw_x(T, shape.H, "cuda", seed, call)
        fwd = qsm.MoEForward(layer, T, want_f32=True, one_launch=False)
        fwd(x)                                   # route, group, FFN (workspace)
        y = torch.full_like(fwd.y, float("nan"))
        y32 = torch.full_like(fwd.y_f32, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _call_noalloc(qsm, layer, x, fwd, y, y32, status)
        assert rc == QSM_OK, qsm.lib().qsm_status_str(rc)
        torch.cuda.synchronize()
        assert status.item() == 0 and fwd.dev_status.item() == 0
        assert torch.equal(y32.view(torch.int32), fwd.y_f32.view(torch.int32))
        assert torch.equal(y.view(torch.int16), fwd.y.view(torch.int16))


def test_noalloc_matches_workspace_entry_point(qsm):
    _compare(qsm, synth.QWEN, 21, (16, 64))


def test_noalloc_affine4_matches_workspace_entry_point(qsm):
    _compare(qsm, synth.QWEN_A4, 23, (64, 8))


def test_noalloc_forced_prefill_path(qsm):
    """With the prefill kernels forced (test hook), a 16-token call still fits
    the built-in scratch; the fp32 reduce-add order of that path may differ
    between calls, so the outputs agree within 1e-5 of max |y|."""
    shape = synth.QWEN
    L = synth.draw_layer(shape, "cuda", seed=24)
    layer = qsm.Layer.from_synth(L)
    T = 16
    x = synth.draw_x(T, shape.H, "cuda", 24)
    qsm.force_path("prefill")
    try:
        fwd = qsm.MoEForward(layer, T, want_f32=True, one_launch=False)
        fwd(x)
        y = torch.full_like(fwd.y, float("nan"))
        y32 = torch.full_like(fwd.y_f32, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _call_noalloc(qsm, layer, x, fwd, y, y32, status)
        torch.cuda.synchronize()
    finally:
        qsm.force_path("auto")
    assert rc == QSM_OK, qsm.lib().qsm_status_str(rc)
    assert status.item() == 0 and fwd.dev_status.item() == 0
    ref = fwd.y_f32.cpu().numpy().astype(np.float64)
    assert tol_metric(y32.cpu().numpy(), ref) <= 1e-5


def test_noalloc_rejects_sizes_beyond_its_scratch(qsm):
    shape = synth.QWEN
    L = synth.draw_layer(shape, "cuda", seed=22)
    layer = qsm.Layer.from_synth(L)
    T = 65
    x = synth.draw_x(T, shape.H, "cuda", 22)
    fwd = qsm.MoEForward(layer, T)
    y = torch.zeros((T, shape.H), dtype=torch.bfloat16, device="cuda")
    y32 = torch.zeros((T, shape.H), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _call_noalloc(qsm, layer, x, fwd, y, y32, status)
    assert rc == QSM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert int(y32.abs().sum().item()) == 0      # nothing was enqueued


def test_noalloc_zero_and_negative_token_counts(qsm):
    shape = synth.QWEN
    L = synth.draw_layer(shape, "cuda", seed=25)
    layer = qsm.Layer.from_synth(L)
    x = synth.draw_x(4, shape.H, "cuda", 25)
    fwd = qsm.MoEForward(layer, 4, one_launch=False)
    y = torch.zeros((4, shape.H), dtype=torch.bfloat16, device="cuda")
    y32 = torch.zeros((4, shape.H), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(qsm, layer, x, fwd, y, y32, status, T=0) == QSM_OK
    assert _call_noalloc(qsm, layer, x, fwd, y, y32, status, T=-1) == \
        QSM_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    assert status.item() == 0
    assert int(y32.abs().sum().item()) == 0      # nothing was written
