"""Dense Q8_0 GEMV against the oracle on the Llama-3.2-1B projection shapes."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import bits16, tol_metric

pytestmark = pytest.mark.gpu


def assert_faithful_bf16(y, ref):
    """The bf16 output is within one bf16 ulp of the correctly rounded fp64
    result (plus 1e-6 of max |ref| for fp32 accumulation near zero).  The
    max-normalised 2e-3 bound cannot apply to a bf16-only output: rounding
    alone reaches 2^-8 of a value."""
    ref_b = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).float().numpy()
    _, e = np.frexp(np.abs(ref_b))
    ulp = np.ldexp(1.0, e - 8)
    slack = 1e-6 * np.max(np.abs(ref))
    bad = np.abs(y - ref_b) > ulp + slack
    assert not bad.any(), f"{bad.sum()} outputs off by more than one bf16 ulp"
    assert tol_metric(y, ref) <= 2.0 ** -8


# the config's five shapes and the stacked ones of a layer (QKV, gate_up)
_SHAPES = dict(synth.GEMV_SHAPES)
_SHAPES.update({"layer_" + k: v for k, v in synth.GEMV_LAYER_SHAPES.items()
                if v not in synth.GEMV_SHAPES.values()})


@pytest.mark.parametrize("name", sorted(_SHAPES))
def test_gemv_shapes(qsm, name):
    N, K = _SHAPES[name]
    x, q, d = synth.draw_gemv(N, K, "cuda", seed=3, name=name)
    y = qsm.q8_gemv(x, q, d)
    torch.cuda.synchronize()
    rows = np.arange(N) if N <= 8192 else np.random.default_rng(0).choice(N, 4096, replace=False)
    qn = q[rows].cpu().numpy()
    ref = oracle.q8_gemv(bits16(x), qn, bits16(d[rows]))
    yc = y.float().cpu().numpy()[rows]
    assert_faithful_bf16(yc, ref)


def test_gemv_one_hot_bit_exact(qsm):
    N, K = 300, 1024
    _, q, d = synth.draw_gemv(N, K, "cuda", seed=4)
    for i in (0, 31, 32, 517, 1023):
        x = torch.zeros(K, dtype=torch.bfloat16, device="cuda")
        x[i] = 1.0
        y = qsm.q8_gemv(x, q, d)
        ref = oracle.q8_gemv(bits16(x), q.cpu().numpy(), bits16(d))
        ref_b = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)
        assert torch.equal(y.cpu().view(torch.int16), ref_b.view(torch.int16))


def test_fused_gate_up_rows_bit_identical(qsm):
    """oMLX gate/up fusion: the concatenated [gate; up] projection gives, per
    row, the same bits as the two projections run separately."""
    N, K = 8192, 2048
    x, gq, gd = synth.draw_gemv(N, K, "cuda", seed=5, name="gate")
    _, uq, ud = synth.draw_gemv(N, K, "cuda", seed=6, name="up")
    fused = qsm.q8_gemv(x, torch.cat([gq, uq]), torch.cat([gd, ud]))
    g = qsm.q8_gemv(x, gq, gd)
    u = qsm.q8_gemv(x, uq, ud)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), torch.cat([g, u]).view(torch.int16))


def test_stacked_qkv_rows_bit_identical(qsm):
    """Projections that read the same activation, stacked into one matrix
    (Q 2048, K 512 and V 512 rows of a Llama-3.2-1B layer), give per row the
    bits of the separate calls."""
    K = 2048
    x, qq, qd = synth.draw_gemv(2048, K, "cuda", seed=7, name="q")
    _, kq, kd = synth.draw_gemv(512, K, "cuda", seed=8, name="k")
    _, vq, vd = synth.draw_gemv(512, K, "cuda", seed=9, name="v")
    fused = qsm.q8_gemv(x, torch.cat([qq, kq, vq]), torch.cat([qd, kd, vd]))
    parts = [qsm.q8_gemv(x, a, b) for a, b in ((qq, qd), (kq, kd), (vq, vd))]
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), torch.cat(parts).view(torch.int16))


def test_gemv_ragged_rows(qsm):
    for N in (1, 15, 17, 1000):
        x, q, d = synth.draw_gemv(N, 512, "cuda", seed=N)
        y = qsm.q8_gemv(x, q, d)
        ref = oracle.q8_gemv(bits16(x), q.cpu().numpy(), bits16(d))
        assert_faithful_bf16(y.float().cpu().numpy(), ref)


# K % 256 == 0 takes the TMA-fed tiles (one cluster per tile when the
# segments are split over CTAs: K = 768 with a partial last segment, K =
# 16384 with 8 CTAs per tile); the other K take the register-fed kernels.
GEMV_EDGE = [(33, 768), (7, 16384), (100, 832), (64, 64), (3000, 2304), (129, 256)]


@pytest.mark.parametrize("N,K", GEMV_EDGE)
def test_gemv_edge_shapes(qsm, N, K):
    x, q, d = synth.draw_gemv(N, K, "cuda", seed=N + K)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = qsm.q8_gemv(x, q, d, dev_status=st)
    qx, dx = qsm.q8_quantize_x(x)
    y8 = qsm.q8_gemv_i8(qx, dx, q, d, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert_faithful_bf16(y.float().cpu().numpy(),
                         oracle.q8_gemv(bits16(x), q.cpu().numpy(), bits16(d)))
    q_o, d_o = oracle.q8_quantize_x(bits16(x))
    assert_faithful_bf16(y8.float().cpu().numpy(),
                         oracle.q8_gemv_i8(q_o, d_o, q.cpu().numpy(), bits16(d)))


@pytest.mark.parametrize("N,K", [(4096, 8192), (20000, 2048), (20000, 8192), (20000, 768)])
def test_gemv_rows_independent_of_n(qsm, N, K):
    """A row's bits do not depend on how many rows the call has: the split
    of K over CTAs changes with N, and 20000 rows (>= 8 tiles per SM) take
    the persistent streaming kernel, but the summation order is the same."""
    x, q, d = synth.draw_gemv(N, K, "cuda", seed=12)
    qx, dx = qsm.q8_quantize_x(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    full = qsm.q8_gemv(x, q, d, dev_status=st)
    full8 = qsm.q8_gemv_i8(qx, dx, q, d, dev_status=st)
    part = qsm.q8_gemv(x, q[:48].contiguous(), d[:48].contiguous())
    part8 = qsm.q8_gemv_i8(qx, dx, q[:48].contiguous(), d[:48].contiguous())
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(full[:48].view(torch.int16), part.view(torch.int16))
    assert torch.equal(full8[:48].view(torch.int16), part8.view(torch.int16))
    rows = np.random.default_rng(N + K).choice(N, 512, replace=False)
    ref = oracle.q8_gemv(bits16(x), q[rows].cpu().numpy(), bits16(d[rows]))
    assert_faithful_bf16(full.float().cpu().numpy()[rows], ref)
    assert int(rows.max()) < N


# ------------------------------------------------ int8-activation mode

@pytest.mark.parametrize("K", [64, 2048, 8192])
def test_quantize_x_bit_exact(qsm, K):
    """The activation codes and block scales equal the oracle's bit for bit
    (both decide in fp32), including an all-zero block and exact halves."""
    x = synth.draw_x(1, K, "cuda", seed=50 + K)[0]
    x[32:64] = 0.0
    qx, dx = qsm.q8_quantize_x(x)
    torch.cuda.synchronize()
    q_o, d_o = oracle.q8_quantize_x(bits16(x))
    assert np.array_equal(qx.cpu().numpy(), q_o)
    assert np.array_equal(dx.cpu().numpy().view(np.uint32), d_o.view(np.uint32))


@pytest.mark.parametrize("name", sorted(synth.GEMV_SHAPES))
def test_gemv_i8_shapes(qsm, name):
    """On the Llama-3.2-1B shapes the int8-activation GEMV is within one
    bf16 ulp of its fp64 oracle (exact block dot products, the same codes)."""
    N, K = synth.GEMV_SHAPES[name]
    x, q, d = synth.draw_gemv(N, K, "cuda", seed=7, name=name)
    qx, dx = qsm.q8_quantize_x(x)
    y = qsm.q8_gemv_i8(qx, dx, q, d)
    torch.cuda.synchronize()
    rows = np.arange(N) if N <= 8192 else np.random.default_rng(1).choice(N, 4096, replace=False)
    q_o, d_o = oracle.q8_quantize_x(bits16(x))
    ref = oracle.q8_gemv_i8(q_o, d_o, q[rows].cpu().numpy(), bits16(d[rows]))
    assert_faithful_bf16(y.float().cpu().numpy()[rows], ref)


def test_gemv_i8_ragged_and_fused_rows(qsm):
    """Ragged N, and rows of a [gate; up] concatenation bit-identical to the
    separate projections (the summation order depends on K only)."""
    N, K = 1000, 2048
    x, gq, gd = synth.draw_gemv(N, K, "cuda", seed=8, name="gate")
    _, uq, ud = synth.draw_gemv(N, K, "cuda", seed=9, name="up")
    qx, dx = qsm.q8_quantize_x(x)
    fused = qsm.q8_gemv_i8(qx, dx, torch.cat([gq, uq]), torch.cat([gd, ud]))
    g = qsm.q8_gemv_i8(qx, dx, gq, gd)
    u = qsm.q8_gemv_i8(qx, dx, uq, ud)
    torch.cuda.synchronize()
    assert torch.equal(fused[:N].view(torch.int16), g.view(torch.int16))
    assert torch.equal(fused[N:].view(torch.int16), u.view(torch.int16))
    q_o, d_o = oracle.q8_quantize_x(bits16(x))
    assert_faithful_bf16(g.float().cpu().numpy(),
                         oracle.q8_gemv_i8(q_o, d_o, gq.cpu().numpy(), bits16(gd)))


def test_gemv_i8_close_to_exact_gemv(qsm):
    """The activation's rounding moves the result by at most the analytic
    bound sum_b |d| * sum|q| * dx / 2 from the exact Q8_0 GEMV."""
    N, K = 512, 2048
    x, q, d = synth.draw_gemv(N, K, "cuda", seed=10)
    qx, dx = qsm.q8_quantize_x(x)
    y8 = qsm.q8_gemv_i8(qx, dx, q, d).float().cpu().numpy()
    y = oracle.q8_gemv(bits16(x), q.cpu().numpy(), bits16(d))
    dw = d.cpu().to(torch.float64).numpy().reshape(N, K // 32)
    qa = np.abs(q.cpu().numpy().astype(np.float64)).reshape(N, K // 32, 32).sum(2)
    bound = (dw * qa * dx.cpu().numpy().astype(np.float64)[None, :] / 2).sum(1)
    ulp = np.abs(y) * 2.0 ** -8  # the bf16 output rounding
    assert np.all(np.abs(y8 - y) <= bound + ulp + 1e-6)
