"""Seeded layer cases shared by the GPU parity tests (cached per process)."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth
from _helpers import bits16, oracle_q, tie_free_x, tol_metric

TOL = 2e-3          # max |y32 - y_ref| / max |y_ref|, per output tensor
TOPK_W_ATOL = 1e-5  # routing weights (fp32 vs fp64)


@functools.lru_cache(maxsize=4)
def layer(shape: synth.LayerShape, seed: int = 0, zipf: str | None = None):
    """(gpu MoELayer, oracle weights (4), router weight / bias on cpu)."""
    Lg = synth.draw_layer(shape, "cuda", seed=seed, zipf=zipf)
    q = tuple(oracle_q(t) for t in (Lg.gate_up, Lg.down, Lg.shared_gate_up,
                                    Lg.shared_down))
    wr = Lg.w_router.cpu()
    bias = None if Lg.logit_bias is None else Lg.logit_bias.cpu()
    return Lg, q, wr, bias


def cpu_view(Lg, wr, bias):
    """A CPU MoELayer with only the router (for tie-free draws)."""
    return synth.MoELayer(Lg.shape, wr, bias, None, None, None, None)


def x_for(shape, T, seed, Lg, wr, bias, layer_id=0):
    return tie_free_x(cpu_view(Lg, wr, bias), T, seed=seed, layer=layer_id)


def oracle_route(x, wr, bias, k, renormalize=True, bias_select_only=False):
    return oracle.route(bits16(x), wr.numpy(),
                        k, None if bias is None else bias.numpy(), renormalize,
                        bias_select_only)


def check_layer_output(y, y32, x, idx_o, w_o, q, tokens=None, shared_gate=None):
    """fp32 output within TOL of the oracle, bf16 output = RNE(fp32).
    shared_gate: the gate vector [H] of a gated shared expert, or None."""
    sw = None if shared_gate is None else \
        oracle.shared_gate(bits16(x), shared_gate.cpu().numpy())
    ref = oracle.moe_layer(bits16(x), idx_o, w_o, *q, tokens=tokens, shared_w=sw)
    y32n = y32.cpu().numpy().astype(np.float64)
    yb = y.cpu()
    if tokens is not None:
        y32n = y32n[tokens]
        yb = yb[tokens]
    err = tol_metric(y32n, ref)
    rne = torch.from_numpy(y32n.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(yb.view(torch.int16), rne.view(torch.int16)), \
        "bf16 output is not the round-to-nearest-even of the fp32 output"
    return err, ref


def check_against(y, y32, ref):
    """check_layer_output against a precomputed oracle output of all tokens
    (one oracle run serving several GPU runs of the same inputs)."""
    y32n = y32.cpu().numpy().astype(np.float64)
    err = tol_metric(y32n, ref)
    rne = torch.from_numpy(y32n.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(y.cpu().view(torch.int16), rne.view(torch.int16)), \
        "bf16 output is not the round-to-nearest-even of the fp32 output"
    return err
