"""The one-launch decode layer (moe_decode_layer) against the fp64 oracle
and against moe_route: ids and weights bit-identical to moe_route, fp32
output within 2e-3 of max |y|, bf16 output = RNE(fp32 output)."""
import numpy as np
import pytest
import torch

import synth
from _gpu_cases import TOL, TOPK_W_ATOL, check_layer_output, layer, oracle_route, x_for

pytestmark = pytest.mark.gpu


CASES = [
    # (shape, T, seed, zipf, renormalize)
    (synth.QWEN, 1, 0, None, True),
    (synth.QWEN, 2, 1, None, True),
    (synth.QWEN, 3, 2, "noise", True),
    (synth.QWEN, 8, 3, None, True),       # up to 64 distinct experts: 17 C items
    (synth.QWEN, 5, 4, None, False),      # full softmax weights
    (synth.QWEN_A4, 1, 5, None, True),
    (synth.QWEN_A4, 8, 6, None, True),
    (synth.TINY, 1, 7, None, True),       # H = 256: 16 CTAs, E = 16, k = 2
    (synth.TINY, 8, 8, None, False),
    # E > 256: 32 candidates per lane and 8 consumer warps; 32 experts per CTA
    (synth.LayerShape(H=256, E=512, k=8, I=128), 2, 9, None, True),
    (synth.LayerShape(H=256, E=512, k=8, I=128), 5, 10, None, False),
]


@pytest.mark.parametrize("shape,T,seed,zipf,renorm", CASES)
def test_decode_layer_matches_oracle(qsm, shape, T, seed, zipf, renorm):
    Lg, q, wr, bias = layer(shape, seed, zipf)
    x = x_for(shape, T, seed + 50, Lg, wr, bias).cuda()
    L = qsm.Layer.from_synth(Lg)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, y32, idx, w = qsm.moe_decode_layer(L, x, renorm, y_f32=True, dev_status=st)
    i2, w2 = qsm.moe_route(x, L.w_router, L.k, L.logit_bias, renorm, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(idx, i2)
    assert torch.equal(w, w2)
    idx_o, w_o = oracle_route(x.cpu(), wr, bias, shape.k, renorm)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=0, atol=TOPK_W_ATOL)
    err, _ = check_layer_output(y, y32, x.cpu(), idx_o, w_o, q)
    assert err <= TOL, f"max-normalised error {err:.3e} > {TOL}"


def test_decode_layer_repeat_on_one_workspace(qsm):
    """Calls on one workspace give the same bits; each call adds one arrival
    per CTA to the call ticket and writes its tag (the number of calls so
    far) into every logit word and into the h words of every slot it uses
    (the shared expert and the distinct selected experts, all T tokens)."""
    shape = synth.QWEN
    T = 4
    Lg, _, wr, bias = layer(shape, 0, None)
    L = qsm.Layer.from_synth(Lg)
    x = x_for(shape, T, 77, Lg, wr, bias).cuda()
    ws = torch.zeros(qsm.decode_layer_workspace_bytes(L, T), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        y, y32, idx, w = qsm.moe_decode_layer(L, x, y_f32=True, workspace=ws)
        outs.append((y32.clone(), idx.clone(), w.clone()))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(outs[0], o))
    # one arrival per CTA: a CTA per SM, at least H / 16, at most the tiles
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (min(8 * shape.k, shape.E) + 1) * (shape.I // 8)  # of up to 8 tokens
    G = max(shape.H // 16, min(sms, tiles))
    assert int(ws[:8].view(torch.int64).item()) == 3 * G
    # the tagged logits [8, E] after the 256-byte ticket, then h [slots, T, I / 2]
    lw = ws[256:256 + 8 * shape.E * 8].view(torch.int64).cpu().numpy()
    assert ((lw >> 32) == 3).all()
    hb = 256 + (8 * shape.E * 8 + 255) // 256 * 256
    slots = 1 + len(set(idx.cpu().numpy().ravel().tolist()))
    n = slots * T * (shape.I // 2)
    hw = ws[hb:hb + 8 * n].view(torch.int64).cpu().numpy()
    assert ((hw >> 32) == 3).all()


def test_decode_layer_workspace_shared_across_T(qsm):
    """One workspace (sized for the largest T) serves calls of different T in
    any order, with the bits of a fresh workspace per call.  (Leftover h of
    a smaller call once sat where a larger call's tagged logits go: a stale
    word that looked like the current call's tag changed one CTA's
    selection.)"""
    shape = synth.QWEN
    Lg, _, wr, bias = layer(shape, 1, None)
    L = qsm.Layer.from_synth(Lg)
    ws = torch.zeros(qsm.decode_layer_workspace_bytes(L, 8), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for T in (8, 1, 5, 1, 8, 3, 8, 2, 8):
        x = x_for(shape, T, 200 + T, Lg, wr, bias).cuda()
        a = qsm.moe_decode_layer(L, x, y_f32=True, workspace=ws, dev_status=st)
        b = qsm.moe_decode_layer(L, x, y_f32=True, dev_status=st)
        torch.cuda.synchronize()
        assert st.item() == 0, T
        assert all(torch.equal(u, v) for u, v in zip(a, b)), T


def test_decode_layer_all_tokens_on_same_experts(qsm):
    """A bias that sends every token to experts 0..7: 8 distinct experts, each
    routed for all T tokens."""
    shape = synth.QWEN
    Lg, q, wr, _ = layer(shape, 0, None)
    bias = torch.zeros(shape.E)
    bias[:8] = 100.0 + torch.arange(8, dtype=torch.float32)
    Lb = synth.MoELayer(shape, Lg.w_router, bias.cuda(), Lg.gate_up, Lg.down,
                        Lg.shared_gate_up, Lg.shared_down)
    x = synth.draw_x(8, shape.H, "cpu", 5)
    y, y32, idx, w = qsm.moe_decode_layer(qsm.Layer.from_synth(Lb), x.cuda(), y_f32=True)
    torch.cuda.synchronize()
    idx_o, w_o = oracle_route(x, wr, bias, shape.k)
    assert set(idx_o.ravel().tolist()) == set(range(8))
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    err, _ = check_layer_output(y, y32, x, idx_o, w_o, q)
    assert err <= TOL


def test_decode_layer_agrees_with_launches_path(qsm):
    """One launch and route + group + FFN launches: same routing bits, outputs
    within the combine's reordering of fp32 additions."""
    shape = synth.QWEN
    Lg, _, wr, bias = layer(shape, 0, None)
    L = qsm.Layer.from_synth(Lg)
    x = x_for(shape, 6, 91, Lg, wr, bias).cuda()
    a = qsm.MoEForward(L, 6, want_f32=True, one_launch=True)
    b = qsm.MoEForward(L, 6, want_f32=True, one_launch=False)
    a(x)
    b(x)
    torch.cuda.synchronize()
    assert a.decode_ws is not None and b.decode_ws is None
    assert torch.equal(a.topk_idx, b.topk_idx) and torch.equal(a.topk_w, b.topk_w)
    scale = b.y_f32.abs().max().item()
    assert (a.y_f32 - b.y_f32).abs().max().item() <= 1e-4 * scale


def test_decode_layer_unsupported(qsm):
    Lg, _, _, _ = layer(synth.QWEN, 0, None)
    L = qsm.Layer.from_synth(Lg)
    assert qsm.decode_layer_workspace_bytes(L, 9) == 0
    x = synth.draw_x(9, synth.QWEN.H, "cuda", 1)
    assert qsm.moe_decode_layer(L, x, raise_unsupported=False) is None
    with pytest.raises(qsm.QSMError):
        qsm.moe_decode_layer(L, x)


def test_decode_layer_barrier_timeout_is_reported(qsm):
    """A logit exchange that cannot complete (test hook: the awaited call tag
    raised by one) makes every bounded wait run out: the call sets QSM_DEV_TIMEOUT and
    returns; the context stays usable.  The timed-out call's results are
    invalid and, as the header requires, its workspace is zeroed before the
    next call, which is exact."""
    shape = synth.TINY
    Lg, q, wr, bias = layer(shape, 7, None)
    L = qsm.Layer.from_synth(Lg)
    x = x_for(shape, 1, 57, Lg, wr, bias).cuda()
    ws = torch.zeros(qsm.decode_layer_workspace_bytes(L, 1), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    qsm.debug_barrier_skew(1)
    try:
        qsm.moe_decode_layer(L, x, workspace=ws, dev_status=st)
        torch.cuda.synchronize()
    finally:
        qsm.debug_barrier_skew(0)
    assert st.item() & qsm.DEV_TIMEOUT
    st.zero_()
    ws.zero_()
    y, y32, idx, w = qsm.moe_decode_layer(L, x, y_f32=True, workspace=ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    idx_o, w_o = oracle_route(x.cpu(), wr, bias, shape.k, True)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    err, _ = check_layer_output(y, y32, x.cpu(), idx_o, w_o, q)
    assert err <= TOL


@pytest.mark.parametrize("one_launch", [True, False])
def test_moe_forward_out_argument(qsm, one_launch):
    """MoEForward writes into a caller's tensor when given out= (both paths),
    with the same bits as into its own buffer."""
    shape = synth.QWEN
    Lg, _, wr, bias = layer(shape, 0, None)
    L = qsm.Layer.from_synth(Lg)
    x = x_for(shape, 3, 31, Lg, wr, bias).cuda()
    f = qsm.MoEForward(L, 3, one_launch=one_launch)
    own = f(x).clone()
    out = torch.empty((2, 3, shape.H), dtype=torch.bfloat16, device="cuda")
    r = f(x, out=out[1])
    torch.cuda.synchronize()
    assert r.data_ptr() == out[1].data_ptr()
    assert torch.equal(out[1], own)
    with pytest.raises(qsm.QSMError):
        f(x, out=torch.empty((3, shape.H), dtype=torch.float32, device="cuda"))
