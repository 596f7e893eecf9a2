"""The whole layer (route -> group -> FFN) through the C ABI against the
fp64 oracle: routing bit-exact, fp32 output within 2e-3 of max |y|, bf16
output = round-to-nearest-even of the fp32 output."""
import numpy as np
import pytest
import torch

import synth
from _gpu_cases import (TOL, TOPK_W_ATOL, check_layer_output, layer,
                        oracle_route, x_for)

pytestmark = pytest.mark.gpu

Q8_CASES = [1, 2, 3, 16, 40, 63, 64]
A4_CASES = [1, 16, 64]


def run(qsm, Lg, x, renorm=True):
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg), x.shape[0], renormalize=renorm,
                         want_f32=True)
    fwd(x.cuda())
    torch.cuda.synchronize()
    return fwd


def _check(qsm, shape, T, seed, zipf=None, renorm=True, tokens=None):
    Lg, q, wr, bias = layer(shape, seed, zipf)
    x = x_for(shape, T, seed + T, Lg, wr, bias)
    fwd = run(qsm, Lg, x, renorm)
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, renorm)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(fwd.topk_w.cpu().numpy(), w_o, atol=TOPK_W_ATOL)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q, tokens)
    assert err <= TOL, f"max-normalised error {err:.3e} > {TOL}"
    return err


def test_tiny_layer(qsm):
    _check(qsm, synth.TINY, 4, seed=0)


@pytest.mark.parametrize("T", Q8_CASES)
def test_qwen_q8_decode(qsm, T):
    _check(qsm, synth.QWEN, T, seed=0)


@pytest.mark.parametrize("T", A4_CASES)
def test_qwen_affine4_decode(qsm, T):
    _check(qsm, synth.QWEN_A4, T, seed=1)


def test_full_softmax_weights(qsm):
    _check(qsm, synth.QWEN, 5, seed=0, renorm=False)


def test_all_tokens_on_same_experts(qsm):
    """A logit bias that sends every token to experts 0..7: eight groups of
    T rows, each split over several 8-row blocks."""
    shape = synth.QWEN
    Lg, q, wr, _ = layer(shape, 0, None)
    bias = torch.zeros(shape.E)
    bias[:8] = 100.0 + torch.arange(8, dtype=torch.float32)  # distinct, no ties
    Lb = synth.MoELayer(shape, Lg.w_router, bias.cuda(), Lg.gate_up, Lg.down,
                        Lg.shared_gate_up, Lg.shared_down)
    x = synth.draw_x(40, shape.H, "cpu", 5)
    fwd = run(qsm, Lb, x)
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    assert set(idx_o.ravel().tolist()) == set(range(8))
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q)
    assert err <= TOL


def test_zero_tokens_is_a_noop(qsm):
    Lg, _, _, _ = layer(synth.TINY, 0, None)
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg), 0)
    fwd(torch.empty((0, synth.TINY.H), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert fwd.dev_status.item() == 0


def test_repeat_calls_are_deterministic(qsm):
    Lg, _, wr, bias = layer(synth.QWEN, 0, None)
    x = x_for(synth.QWEN, 16, 9, Lg, wr, bias).cuda()
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg), 16, want_f32=True)
    fwd(x)
    a = fwd.y_f32.clone()
    fwd(x)
    torch.cuda.synchronize()
    assert torch.equal(a, fwd.y_f32)


def test_bad_expert_id_is_flagged_not_fatal(qsm):
    """An out-of-range expert id injected between route and FFN sets the
    status bit; the kernels skip it and the context stays usable."""
    shape = synth.TINY
    Lg, _, _, _ = layer(shape, 0, None)
    x = synth.draw_x(4, shape.H, "cuda", 3)
    L = qsm.Layer.from_synth(Lg)
    fwd = qsm.MoEForward(L, 4)
    qsm.moe_route(x, L.w_router, L.k, None, True, fwd.topk_idx, fwd.topk_w,
                  fwd.route_ws, fwd.dev_status)
    fwd.topk_idx[1, 0] = 12345
    qsm.moe_group_tokens(fwd.topk_idx, L.E, fwd.grouping.tile_rows,
                         fwd.grouping, fwd.dev_status)
    qsm.moe_ffn_forward(L, x, fwd.topk_idx, fwd.topk_w, fwd.grouping, fwd.y,
                        False, fwd.ffn_ws, fwd.dev_status)
    torch.cuda.synchronize()
    assert fwd.dev_status.item() & qsm.DEV_BAD_EXPERT_ID
    assert torch.isfinite(fwd.y.float()).all()


def test_invalid_arguments_rejected(qsm):
    Lg, _, _, _ = layer(synth.TINY, 0, None)
    L = qsm.Layer.from_synth(Lg)
    x = synth.draw_x(4, synth.TINY.H, "cuda", 3)
    with pytest.raises(qsm.QSMError):
        qsm.moe_route(x, L.w_router, 0)                 # k = 0
    with pytest.raises(qsm.QSMError):
        qsm.moe_route(x, L.w_router, 17)                # k > E
    fwd = qsm.MoEForward(L, 4)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qsm.QSMError):
        qsm.moe_ffn_forward(L, x, fwd.topk_idx, fwd.topk_w, fwd.grouping,
                            workspace=small)
