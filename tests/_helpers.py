"""Shared helpers for the tests: tensor conversion and tie-free inputs.

Nothing here computes any part of the layer; the near-tie check asks the
oracle for router logits.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Adjacent sorted logits among a token's top k+1 must differ by this much so
# that the selected expert set does not depend on the accumulation order.
TIE_GAP = 1e-4


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 / fp16 tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(
        np.uint16)


def oracle_q(qt: synth.QTensor) -> oracle.QWeights:
    codes = qt.codes.detach().cpu().contiguous().numpy()
    if qt.qtype == synth.AFFINE4_G64:
        codes = codes.view(np.uint32)
    return oracle.QWeights(qt.qtype, codes, bits16(qt.scales),
                           None if qt.biases is None else bits16(qt.biases))


def oracle_layer(L: synth.MoELayer):
    return (oracle_q(L.gate_up), oracle_q(L.down), oracle_q(L.shared_gate_up),
            oracle_q(L.shared_down))


def near_tie_tokens(logits: np.ndarray, k: int, gap: float = TIE_GAP):
    """Tokens whose top k+1 sorted logits hold two values closer than gap."""
    E = logits.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-logits, axis=1)[:, :m]
    d = top[:, :-1] - top[:, 1:]
    return np.nonzero((d < gap).any(axis=1))[0].tolist()


def tie_free_x(L: synth.MoELayer, T: int, seed: int = 0, layer: int = 0,
               max_attempts: int = 50) -> torch.Tensor:
    """x [T, H] bf16 (cpu) whose routing has no near-ties, redrawing the
    offending token rows from the same seeded stream."""
    H, k = L.shape.H, L.shape.k
    x = synth.draw_x(T, H, "cpu", seed, layer)
    wr = L.w_router.detach().cpu().numpy()
    bias = None if L.logit_bias is None else L.logit_bias.cpu().numpy()
    for attempt in range(1, max_attempts + 1):
        logits = oracle.router_logits(bits16(x), wr, bias)
        bad = near_tie_tokens(logits, k)
        if not bad:
            return x
        x = synth.redraw_x_rows(x, bad, seed, layer, attempt)
    raise RuntimeError("could not draw tie-free tokens")


def tol_metric(y32: np.ndarray, ref: np.ndarray) -> float:
    """max |y - ref| / max |ref|: the FFN output error measure."""
    return float(np.max(np.abs(y32.astype(np.float64) - ref)) /
                 max(np.max(np.abs(ref)), 1e-300))
