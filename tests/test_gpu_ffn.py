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


def run(qsm, Lg, x, renorm=True, one_launch=True):
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg), x.shape[0], renormalize=renorm,
                         want_f32=True, one_launch=one_launch)
    fwd(x.cuda())
    torch.cuda.synchronize()
    return fwd


def _check(qsm, shape, T, seed, zipf=None, renorm=True, tokens=None, one_launch=True):
    Lg, q, wr, bias = layer(shape, seed, zipf)
    x = x_for(shape, T, seed + T, Lg, wr, bias)
    fwd = run(qsm, Lg, x, renorm, one_launch)
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, renorm)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(fwd.topk_w.cpu().numpy(), w_o, atol=TOPK_W_ATOL)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q, tokens)
    assert err <= TOL, f"max-normalised error {err:.3e} > {TOL}"
    return err


# one_launch: T <= 8 goes through moe_decode_layer (one launch) or through
# route + group + FFN launches; larger T always takes the launches.
@pytest.mark.parametrize("one_launch", [True, False])
def test_tiny_layer(qsm, one_launch):
    _check(qsm, synth.TINY, 4, seed=0, one_launch=one_launch)


@pytest.mark.parametrize("one_launch", [True, False])
@pytest.mark.parametrize("T", Q8_CASES)
def test_qwen_q8_decode(qsm, T, one_launch):
    if T > 8 and not one_launch:
        pytest.skip("the launches path is the only path for T > 8")
    _check(qsm, synth.QWEN, T, seed=0, one_launch=one_launch)


@pytest.mark.parametrize("one_launch", [True, False])
@pytest.mark.parametrize("T", A4_CASES)
def test_qwen_affine4_decode(qsm, T, one_launch):
    if T > 8 and not one_launch:
        pytest.skip("the launches path is the only path for T > 8")
    _check(qsm, synth.QWEN_A4, T, seed=1, one_launch=one_launch)


# Past 8 tokens the decode path streams gate_up with one persistent CTA per
# SM over (slot, 16-row tile) items: a slot of one token after full ones
# (T = 9, 17), the small layer's shapes (H = 256: the chunk loop's generic
# form; I = 128: 16 tiles per slot), and the largest T the decode path takes
# when forced (128: every expert holds several slots).
@pytest.mark.parametrize("shape,T", [(synth.QWEN, 9), (synth.QWEN_A4, 17), (synth.TINY, 9),
                                     (synth.TINY, 64)])
def test_decode_stream_edges(qsm, shape, T):
    _check(qsm, shape, T, seed=2, one_launch=False)


def test_decode_path_forced_at_128_tokens(qsm):
    qsm.force_path("decode")
    try:
        _check(qsm, synth.QWEN, 128, seed=3, one_launch=False)
    finally:
        qsm.force_path("auto")


@pytest.mark.parametrize("one_launch", [True, False])
def test_full_softmax_weights(qsm, one_launch):
    _check(qsm, synth.QWEN, 5, seed=0, renorm=False, one_launch=one_launch)


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


# ------------------------------------------------------------------ prefill

PREFILL_CASES = [65, 128, 200, 1000]


@pytest.mark.parametrize("T", PREFILL_CASES)
def test_qwen_q8_prefill(qsm, T):
    # full-layer oracle on a token sample (every output of those tokens)
    rng = np.random.default_rng(T)
    toks = np.sort(rng.choice(T, min(T, 48), replace=False)).astype(np.int32)
    _check(qsm, synth.QWEN, T, seed=2, tokens=toks)


def test_tiny_layer_forced_prefill(qsm):
    qsm.force_path("prefill")
    try:
        _check(qsm, synth.TINY, 4, seed=0)
        _check(qsm, synth.TINY, 37, seed=1)
    finally:
        qsm.force_path("auto")


@pytest.mark.parametrize("T", [1, 16, 64, 100])
def test_cross_path_same_tokens(qsm, T):
    """The decode kernels and the prefill kernels both meet the tolerance on
    the same tokens, and agree with each other within it."""
    Lg, q, wr, bias = layer(synth.QWEN, 0, None)
    x = x_for(synth.QWEN, T, 77 + T, Lg, wr, bias)
    outs = {}
    for path in ("decode", "prefill"):
        qsm.force_path(path)
        try:
            fwd = run(qsm, Lg, x)
        finally:
            qsm.force_path("auto")
        assert fwd.dev_status.item() == 0
        outs[path] = fwd.y_f32.cpu().numpy().astype(np.float64)
    idx_o, w_o = oracle_route(x, wr, bias, synth.QWEN.k)
    from _helpers import tol_metric
    import oracle as orc
    from _helpers import bits16
    ref = orc.moe_layer(bits16(x), idx_o, w_o, *q)
    for path, y32 in outs.items():
        assert tol_metric(y32, ref) <= TOL, path
    assert tol_metric(outs["decode"], outs["prefill"]) <= TOL


def test_prefill_zipf_t4096_all_tokens(qsm):
    """The prefill workload at full size: T=4096, Zipf-offset routing (many
    empty experts, a few very large groups); all routing bit-exact, and every
    output of every token against the oracle (447 blocks: every row position
    of every 128-row block, short blocks of every 16-row size)."""
    shape = synth.QWEN
    Lg, q, wr, bias = layer(shape, 3, "noise")
    x = x_for(shape, 4096, 4096, Lg, wr, bias)
    fwd = run(qsm, Lg, x)
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    counts = np.bincount(idx_o.ravel(), minlength=shape.E)
    assert (counts == 0).sum() > 0          # some experts are empty
    assert counts.max() > 128               # some experts span several blocks
    assert np.array_equal(fwd.grouping.counts.cpu().numpy(), counts)
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q)
    assert err <= TOL


def test_prefill_repeat_is_stable(qsm):
    """Two prefill calls in a row give results within one bf16 ulp (the
    fp32 reduce-add order may differ)."""
    Lg, _, wr, bias = layer(synth.QWEN, 0, None)
    x = x_for(synth.QWEN, 300, 5, Lg, wr, bias).cuda()
    fwd = qsm.MoEForward(qsm.Layer.from_synth(Lg), 300, want_f32=True)
    fwd(x)
    a = fwd.y_f32.clone()
    fwd(x)
    torch.cuda.synchronize()
    rel = (a - fwd.y_f32).abs().max().item() / a.abs().max().item()
    assert rel < 1e-5


# ------------------------------------------------- affine-4 prefill (NEXT-1)

@pytest.mark.parametrize("T", [65, 300, 1000])
def test_qwen_affine4_prefill(qsm, T):
    """The grouped tcgen05 GEMMs with affine-4 weights (fp16(s*q + b) tiles
    expanded on chip) against the fp64 oracle on sampled tokens."""
    rng = np.random.default_rng(T + 7)
    toks = np.sort(rng.choice(T, min(T, 48), replace=False)).astype(np.int32)
    _check(qsm, synth.QWEN_A4, T, seed=4, tokens=toks)


@pytest.mark.parametrize("T", [16, 100])
def test_affine4_cross_path(qsm, T):
    """Affine-4: the decode and the prefill kernels both meet the tolerance
    on the same tokens and agree with each other within it."""
    from _helpers import bits16, tol_metric
    import oracle as orc
    shape = synth.QWEN_A4
    Lg, q, wr, bias = layer(shape, 5, None)
    x = x_for(shape, T, 91 + T, Lg, wr, bias)
    outs = {}
    for path in ("decode", "prefill"):
        qsm.force_path(path)
        try:
            fwd = run(qsm, Lg, x)
        finally:
            qsm.force_path("auto")
        assert fwd.dev_status.item() == 0
        outs[path] = fwd.y_f32.cpu().numpy().astype(np.float64)
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    ref = orc.moe_layer(bits16(x), idx_o, w_o, *q)
    for path, y32 in outs.items():
        assert tol_metric(y32, ref) <= TOL, path
    assert tol_metric(outs["decode"], outs["prefill"]) <= TOL


def test_affine4_prefill_zipf_t2048_all_tokens(qsm):
    """Affine-4 prefill with uneven groups (Zipf offset): routing bit-exact,
    every output of every token against the oracle."""
    shape = synth.QWEN_A4
    Lg, q, wr, bias = layer(shape, 6, "noise")
    T = 2048
    x = x_for(shape, T, 2048, Lg, wr, bias)
    fwd = run(qsm, Lg, x)
    assert fwd.dev_status.item() == 0
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    assert np.array_equal(fwd.topk_idx.cpu().numpy(), idx_o)
    counts = np.bincount(idx_o.ravel(), minlength=shape.E)
    assert (counts == 0).sum() > 0 and counts.max() > 128
    err, _ = check_layer_output(fwd.y, fwd.y_f32, x, idx_o, w_o, q)
    assert err <= TOL
