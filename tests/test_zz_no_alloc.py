"""moe_ffn_forward_noalloc: the FFN entry point for callers that cannot
allocate device memory (it takes its scratch from an array built into the
library instead of a caller-provided workspace).

Called through the C ABI and compared with moe_ffn_forward, which gets a
workspace from the caller, on two calls in a row: the second call reuses the
built-in scratch that the first call left behind.  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from _helpers import tol_metric

pytestmark = pytest.mark.gpu

TOL = 2e-3
QSM_ERR_UNSUPPORTED = 2


def _call_noalloc(qsm, layer, x, fwd, y, y32, status):
    gc = fwd.grouping.c
    s = torch.cuda.current_stream()
    return qsm.lib().moe_ffn_forward_noalloc(
        ctypes.byref(layer.c), ctypes.c_void_p(x.data_ptr()), x.shape[0],
        ctypes.c_void_p(fwd.topk_idx.data_ptr()),
        ctypes.c_void_p(fwd.topk_w.data_ptr()), ctypes.byref(gc),
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(y32.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(s.cuda_stream))


def test_noalloc_matches_workspace_entry_point(qsm):
    shape = synth.QWEN
    L = synth.draw_layer(shape, "cuda", seed=21)
    layer = qsm.Layer.from_synth(L)
    for call, T in enumerate((16, 64)):          # two calls in a row
        x = synth.draw_x(T, shape.H, "cuda", 21, call)
        fwd = qsm.MoEForward(layer, T, want_f32=True)
        fwd(x)                                   # route, group, FFN (workspace)
        y = torch.full_like(fwd.y, float("nan"))
        y32 = torch.full_like(fwd.y_f32, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _call_noalloc(qsm, layer, x, fwd, y, y32, status)
        assert rc == 0, qsm.lib().qsm_status_str(rc)
        torch.cuda.synchronize()
        assert status.item() == 0 and fwd.dev_status.item() == 0
        ref32 = fwd.y_f32.cpu().numpy().astype(np.float64)
        assert tol_metric(y32.cpu().numpy(), ref32) <= TOL
        assert torch.equal(y.view(torch.int16), fwd.y.view(torch.int16))


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
