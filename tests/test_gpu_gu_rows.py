"""Per-row identity of the fused gate_up projection on the MoE kernels.

"oMLX MoE gate/up 融合优化", section "融合原理": gate and up are concatenated
along the output axis and computed by one quantized matmul whose rows come
out bit-identical to the separate gate and up projections.  For the kernels
here that means every gate_up output row depends only on its own weight row
and its token, never on the other half of the concatenation.  A test hook
(qsm_debug_gu_dump) makes the kernels write their fp32 gate and up values
before SwiGLU.  Replacing only the up half of every expert's [gate; up]
weight must leave every gate value bit-identical, and replacing only the
gate half every up value, on each path: the one-launch decode layer, the
decode FFN kernels and the prefill grouped GEMM (Q8_0 and affine-4)."""
import numpy as np
import pytest
import torch

import synth
from _gpu_cases import layer, x_for

pytestmark = pytest.mark.gpu


def _swap_half(qt, half, I, seed):
    """qt with rows [half*I, (half+1)*I) of every expert (codes and block
    constants) taken from an independent draw."""
    o = synth.draw_qtensor(qt.qtype, qt.experts, qt.rows, qt.cols, "cuda", seed, 0,
                           f"swap{half}")
    sl = slice(half * I, (half + 1) * I)
    codes, scales = qt.codes.clone(), qt.scales.clone()
    codes[:, sl] = o.codes[:, sl]
    scales[:, sl] = o.scales[:, sl]
    biases = None
    if qt.biases is not None:
        biases = qt.biases.clone()
        biases[:, sl] = o.biases[:, sl]
    return synth.QTensor(qt.qtype, qt.experts, qt.rows, qt.cols, codes, scales, biases)


def _variant(Lg, half):
    I = Lg.shape.I
    return synth.MoELayer(Lg.shape, Lg.w_router, Lg.logit_bias,
                          _swap_half(Lg.gate_up, half, I, 31),
                          Lg.down, _swap_half(Lg.shared_gate_up, half, I, 32),
                          Lg.shared_down)


def _dump(qsm, Lg, x, path):
    T, k, E, I = x.shape[0], Lg.shape.k, Lg.shape.E, Lg.shape.I
    rows = (min(E, T * k) + 1) * T if path == "one_launch" else T * k + T
    buf = torch.full((rows * 2 * I,), float("nan"), dtype=torch.float32, device="cuda")
    L = qsm.Layer.from_synth(Lg)
    qsm.debug_gu_dump(buf)
    try:
        if path == "prefill":
            qsm.force_path("prefill")
        fwd = qsm.MoEForward(L, T, one_launch=(path == "one_launch"))
        if path == "one_launch":
            assert fwd.decode_ws is not None
        fwd(x.cuda())
        torch.cuda.synchronize()
    finally:
        qsm.debug_gu_dump(None)
        qsm.force_path("auto")
    assert fwd.dev_status.item() == 0
    return buf.view(rows, 2 * I).view(torch.int32).cpu().numpy(), fwd.topk_idx.cpu().numpy()


CASES = [("one_launch", synth.QWEN, 3, None), ("one_launch", synth.QWEN_A4, 1, None),
         ("decode", synth.QWEN, 16, None), ("decode", synth.QWEN_A4, 40, None),
         ("prefill", synth.QWEN, 40, None), ("prefill", synth.QWEN, 1024, "noise"),
         ("prefill", synth.QWEN_A4, 300, None)]


@pytest.mark.parametrize("path,shape,T,zipf", CASES,
                         ids=[f"{c[0]}-{'a4' if c[1].qtype else 'q8'}-T{c[2]}" for c in CASES])
def test_gate_up_rows_depend_only_on_their_weight_row(qsm, path, shape, T, zipf):
    Lg, _, wr, bias = layer(shape, 11, zipf)
    x = x_for(shape, T, 1300 + T, Lg, wr, bias)
    I = shape.I
    d0, idx0 = _dump(qsm, Lg, x, path)
    d_up, idx1 = _dump(qsm, _variant(Lg, 1), x, path)     # up half replaced
    d_gate, idx2 = _dump(qsm, _variant(Lg, 0), x, path)   # gate half replaced
    assert np.array_equal(idx0, idx1) and np.array_equal(idx0, idx2)
    written = ~np.isnan(d0.view(np.float32)).all(axis=1)
    assert written.sum() >= T * (shape.k + 1) if path != "one_launch" else written.sum() > T
    assert np.array_equal(d0[:, :I], d_up[:, :I]), "gate values changed with the up rows"
    assert np.array_equal(d0[:, I:], d_gate[:, I:]), "up values changed with the gate rows"
    # the replacement did change the half it replaced
    assert not np.array_equal(d0[written][:, I:], d_up[written][:, I:])
    assert not np.array_equal(d0[written][:, :I], d_gate[written][:, :I])
