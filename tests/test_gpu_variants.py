"""Router and shared-expert variants against the oracle: a logit bias that
selects experts without entering the weights (QSM_ROUTE_BIAS_SELECT_ONLY),
and a sigmoid-gated shared expert (qsm_moe_layer.shared_gate), on the
decode, prefill, fused-router and chunked paths."""
import numpy as np
import pytest
import torch

import synth
from _gpu_cases import (TOL, TOPK_W_ATOL, check_layer_output, layer, oracle_route,
                        x_for)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,renorm", [(1, True), (5, True), (40, False), (300, True),
                                      (300, False), (1000, True)])
def test_route_bias_select_only(qsm, T, renorm):
    shape = synth.QWEN
    Lg, _, wr, bias = layer(shape, 10, "noise")
    x = x_for(shape, T, 1000 + T, Lg, wr, bias)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w = qsm.moe_route(x.cuda(), wr.cuda(), shape.k, bias.cuda(), renorm,
                           dev_status=st, bias_select_only=True)
    torch.cuda.synchronize()
    assert st.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, renorm, bias_select_only=True)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=0, atol=TOPK_W_ATOL)
    # the selection matches the plain router's; only the weights differ
    idx_p, w_p = oracle_route(x, wr, bias, shape.k, renorm)
    assert np.array_equal(idx_p, idx_o)
    assert np.abs(w_p - w_o).max() > 1e-3


@pytest.mark.parametrize("shape,T,gated,sel_only", [
    (synth.QWEN, 1, True, False), (synth.QWEN, 3, True, True),
    (synth.QWEN, 16, True, False), (synth.QWEN, 64, True, True),
    (synth.QWEN_A4, 16, True, False), (synth.QWEN, 8, False, True)])
def test_decode_variants(qsm, shape, T, gated, sel_only):
    Lg, q, wr, bias = layer(shape, 11, "noise")
    sg = synth.draw_shared_gate(shape.H, "cuda", 11) if gated else None
    x = x_for(shape, T, 1100 + T, Lg, wr, bias)
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg, sg), T, want_f32=True,
                         bias_select_only=sel_only)
    fwd(x.cuda())
    torch.cuda.synchronize()
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, True, sel_only)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(fwd.topk_w.cpu().numpy(), w_o, atol=TOPK_W_ATOL)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q, shared_gate=sg)
    assert err <= TOL


@pytest.mark.parametrize("shape,T", [(synth.QWEN, 100), (synth.QWEN, 1000),
                                     (synth.QWEN_A4, 300)])
def test_prefill_gated_shared_expert(qsm, shape, T):
    Lg, q, wr, bias = layer(shape, 12, "noise")
    sg = synth.draw_shared_gate(shape.H, "cuda", 12)
    x = x_for(shape, T, 1200 + T, Lg, wr, bias)
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg, sg), T, want_f32=True,
                         bias_select_only=True)
    fwd(x.cuda())
    torch.cuda.synchronize()
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, True, True)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    toks = np.sort(np.random.default_rng(T).choice(T, 40, replace=False)).astype(np.int32)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q, toks, shared_gate=sg)
    assert err <= TOL


def test_gate_changes_the_output(qsm):
    """The gate is applied: a gate vector of zeros gives sigmoid(0) = 1/2
    for every token, so the shared expert enters at half weight, far from
    the ungated layer."""
    import oracle
    from _helpers import bits16, tol_metric
    shape = synth.QWEN
    Lg, q, wr, bias = layer(shape, 13, None)
    T = 16
    x = x_for(shape, T, 1300, Lg, wr, bias).cuda()
    outs = {}
    for name, sg in (("plain", None), ("zero", torch.zeros(shape.H, device="cuda"))):
        fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg, sg), T, want_f32=True)
        fwd(x)
        torch.cuda.synchronize()
        outs[name] = fwd.y_f32.cpu().numpy().astype(np.float64)
    idx_o, w_o = oracle_route(x.cpu(), wr, bias, shape.k)
    ref_half = oracle.moe_layer(bits16(x.cpu()), idx_o, w_o, *q, shared_w=np.full(T, 0.5))
    assert tol_metric(outs["zero"], ref_half) <= TOL
    assert tol_metric(outs["plain"], ref_half) > 10 * TOL


def test_chunked_layer_with_variants(qsm):
    shape = synth.QWEN
    Lg, q, wr, bias = layer(shape, 14, "noise")
    sg = synth.draw_shared_gate(shape.H, "cuda", 14)
    T = 600
    x = x_for(shape, T, 1400, Lg, wr, bias)
    L = qsm.Layer.from_synth(Lg, sg)
    y, y32, ti, tw = qsm.moe_layer_forward(L, x.cuda(), 256, True, True, y_f32=True)
    torch.cuda.synchronize()
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, True, True)
    assert np.array_equal(ti.cpu().numpy(), idx_o)
    np.testing.assert_allclose(tw.cpu().numpy(), w_o, atol=TOPK_W_ATOL)
    toks = np.array([0, 255, 256, 511, 512, 599], np.int32)
    err, _ = check_layer_output(y, y32, x, idx_o, w_o, q, toks, shared_gate=sg)
    assert err <= TOL
