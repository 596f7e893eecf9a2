"""The whole layer in chunks (moe_layer_forward) against the oracle and
across chunk sizes: routing bit-exact for every chunking, outputs within
the tolerance, workspace bounded by the chunk size."""
import numpy as np
import pytest
import torch

import synth
from _gpu_cases import (TOL, TOPK_W_ATOL, check_against, check_layer_output, layer,
                        oracle_route, x_for)

pytestmark = pytest.mark.gpu


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


@pytest.mark.parametrize("shape", [synth.QWEN, synth.QWEN_A4], ids=["q8", "a4"])
def test_chunked_layer_matches_oracle_and_unchunked(qsm, shape):
    """Every token and every output of a 1000-token layer (Zipf-offset
    routing), for each chunking, against one oracle run of all tokens."""
    import oracle
    from _helpers import bits16
    T = 1000
    Lg, q, wr, bias = layer(shape, 8, "noise")
    x = x_for(shape, T, 800, Lg, wr, bias)
    L = qsm.Layer.from_synth(Lg)
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    ref = oracle.moe_layer(bits16(x), idx_o, w_o, *q)
    outs = {}
    for chunk in (T, 512, 300, 64, 7):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        y, y32, ti, tw = qsm.moe_layer_forward(L, x.cuda(), chunk, y_f32=True,
                                               dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, chunk
        assert np.array_equal(ti.cpu().numpy(), idx_o), chunk
        np.testing.assert_allclose(tw.cpu().numpy(), w_o, atol=TOPK_W_ATOL)
        err = check_against(y, y32, ref)
        assert err <= TOL, (chunk, err)
        outs[chunk] = y32.cpu().numpy().astype(np.float64)
    # prefill-sized chunkings differ only in the fp32 combine order
    for chunk in (512, 300):
        assert _rel(outs[chunk], outs[T]) < 1e-5, chunk
    # decode-sized chunks run the decode kernels: within the tolerance
    for chunk in (64, 7):
        assert _rel(outs[chunk], outs[T]) <= TOL, chunk


def test_chunked_workspace_is_bounded(qsm):
    Lg, _, _, _ = layer(synth.QWEN, 0, None)
    L = qsm.Layer.from_synth(Lg)
    full = qsm.layer_workspace_bytes(L, 4096, 4096)
    half = qsm.layer_workspace_bytes(L, 4096, 2048)
    assert 0 < half < 0.6 * full
    # the bound depends on the chunk, not on T
    assert qsm.layer_workspace_bytes(L, 65536, 2048) == half


def test_chunked_layer_repeat_and_tail(qsm):
    """Two calls in a row on one workspace (router counters re-armed) give
    the same routing and outputs within one fp32 reduce-add reordering; a
    tail chunk of one token runs on the decode kernels."""
    shape = synth.QWEN
    T = 257
    Lg, q, wr, bias = layer(shape, 9, None)
    x = x_for(shape, T, 900, Lg, wr, bias).cuda()
    L = qsm.Layer.from_synth(Lg)
    ws = torch.zeros(qsm.layer_workspace_bytes(L, T, 128), dtype=torch.uint8,
                     device="cuda")
    a = qsm.moe_layer_forward(L, x, 128, y_f32=True, workspace=ws)
    a = [t.clone() for t in a]
    b = qsm.moe_layer_forward(L, x, 128, y_f32=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    assert _rel(b[1].cpu().numpy(), a[1].cpu().numpy()) < 1e-5
    idx_o, w_o = oracle_route(x.cpu(), wr, bias, shape.k)
    err, _ = check_layer_output(b[0], b[1], x.cpu(), idx_o, w_o, q,
                                np.array([0, 1, 127, 128, 255, 256], np.int32))
    assert err <= TOL


def test_chunked_layer_rejects_bad_chunk(qsm):
    Lg, _, _, _ = layer(synth.TINY, 0, None)
    L = qsm.Layer.from_synth(Lg)
    x = synth.draw_x(4, synth.TINY.H, "cuda", 3)
    assert qsm.layer_workspace_bytes(L, 4, 0) == 0
    with pytest.raises(qsm.QSMError):
        qsm.moe_layer_forward(L, x, 0)
