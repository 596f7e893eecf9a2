"""Seeded synthetic inputs for the quantized sparse MoE FFN layer.

This module only draws random tensors with the shapes and distributions of
the workloads; it holds none of the layer's arithmetic.  It is shared by the
tests (which hand the same tensors to the CUDA library and to the CPU oracle)
and by ``bench.py``.

Workloads (shapes of a Qwen3.6-35B-A3B-style MoE layer):
  tiny      T=4, H=256, E=16, k=2 + shared, I=128, Q8_0
  decode    T=1, 40 independent layers, H=2048, E=256, k=8 + shared, I=512, Q8_0
  prefill   T=4096, one layer of the decode shapes, router logits offset by a
            Zipf(s=1) per-expert bias so that group sizes are uneven
  batched   T in {1, 16, 64}, 40 layers, affine 4-bit weights (group 64)
  gemv      batch-1 Q8_0 projections of Llama-3.2-1B shapes (N x K)

Distributions: Q8_0 codes uniform integers in [-127, 127], fp16 scales
U(0.002, 0.02); affine-4 codes uniform in [0, 15], fp16 scales U(0.005, 0.05)
and fp16 biases U(-0.4, 0.4); router weight fp32 N(0, 0.05); x bf16 N(0, 1)
(an fp32 normal draw rounded to bf16).

Every tensor is drawn from its own torch.Generator seeded by
(seed, layer, tensor name), so a tensor does not depend on which others were
drawn first.  Values drawn on "cpu" and on "cuda" differ; a test hands the
same tensors to both sides.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch

Q8_0 = 0
AFFINE4_G64 = 1


@dataclasses.dataclass(frozen=True)
class LayerShape:
    H: int
    E: int
    k: int
    I: int
    qtype: int = Q8_0


TINY = LayerShape(H=256, E=16, k=2, I=128)
QWEN = LayerShape(H=2048, E=256, k=8, I=512)
QWEN_A4 = LayerShape(H=2048, E=256, k=8, I=512, qtype=AFFINE4_G64)

# Llama-3.2-1B batch-1 projections, (N, K) = (outputs, inputs).
GEMV_SHAPES = {
    "q_o": (2048, 2048),
    "k_v": (512, 2048),
    "gate_up": (8192, 2048),
    "down": (2048, 8192),
    "lm_head": (128256, 2048),
}

# The same projections as one layer's calls, those that read the same
# activation stacked into one matrix: Q, K and V (2048 + 512 + 512 rows) and
# gate and up (8192 + 8192 rows); then O, down and the LM head.
GEMV_LAYER_SHAPES = {
    "qkv": (3072, 2048),
    "o": (2048, 2048),
    "gate_up": (16384, 2048),
    "down": (2048, 8192),
    "lm_head": (128256, 2048),
}


def sub_seed(seed: int, *parts) -> int:
    """A stable 63-bit seed for one named tensor."""
    h = hashlib.sha256(repr((seed,) + tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, seed: int, *parts) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(sub_seed(seed, *parts))
    return g


def _uniform(shape, lo, hi, device, g) -> torch.Tensor:
    return torch.empty(shape, dtype=torch.float32, device=device).uniform_(
        lo, hi, generator=g)


def draw_x(T: int, H: int, device="cpu", seed: int = 0, layer: int = 0,
           attempt: int = 0) -> torch.Tensor:
    """Hidden states [T, H] bf16 ~ N(0, 1)."""
    g = _gen(device, seed, layer, "x", attempt)
    return torch.randn((T, H), generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def redraw_x_rows(x: torch.Tensor, rows, seed: int, layer: int,
                  attempt: int) -> torch.Tensor:
    """Replace the listed token rows of x by fresh N(0,1) draws (attempt>0)."""
    rows = list(rows)
    if not rows:
        return x
    fresh = draw_x(len(rows), x.shape[1], x.device, seed, layer,
                   ("redraw", attempt, tuple(rows)))
    x = x.clone()
    x[torch.tensor(rows, device=x.device)] = fresh
    return x


def draw_router(E: int, H: int, device="cpu", seed: int = 0,
                layer: int = 0) -> torch.Tensor:
    """Router weight [E, H] fp32 ~ N(0, 0.05)."""
    g = _gen(device, seed, layer, "w_router")
    return torch.randn((E, H), generator=g, device=device,
                       dtype=torch.float32) * 0.05


def draw_shared_gate(H: int, device="cpu", seed: int = 0, layer: int = 0) -> torch.Tensor:
    """Shared-expert gate vector [H] fp32 ~ N(0, 0.05), like a router row
    (the gate sigmoid(x . w) then spreads over (0, 1) for x ~ N(0, 1))."""
    g = _gen(device, seed, layer, "shared_gate")
    return torch.randn((H,), generator=g, device=device, dtype=torch.float32) * 0.05


def zipf_logit_bias(E: int, H: int, seed: int = 0, layer: int = 0,
                    s: float = 1.0, in_noise_units: bool = True,
                    device="cpu") -> torch.Tensor:
    """Per-expert router offset that makes expert popularity Zipf-like.

    Ranks 1..E are a seeded random permutation; the offset of the expert of
    rank r is -s * ln(r), times the logit noise scale sigma_L = 0.05*sqrt(H)
    (the standard deviation of a router logit for N(0,1) inputs) when
    `in_noise_units` is set.  In noise units the skew leaves many experts
    empty; in raw units every expert still gets tokens.
    """
    g = _gen("cpu", seed, layer, "zipf_rank")
    ranks = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    scale = 0.05 * math.sqrt(H) if in_noise_units else 1.0
    return (-s * scale * torch.log(ranks)).to(torch.float32).to(device)


@dataclasses.dataclass
class QTensor:
    """Quantized weights [experts, rows, cols] on some device.

    Q8_0:        codes int8  [E, rows, cols]; scales fp16 [E, rows, cols/32]
    AFFINE4_G64: codes int32 [E, rows, cols/8] (input c in bits 4*(c%8)..);
                 scales, biases fp16 [E, rows, cols/64]
    """
    qtype: int
    experts: int
    rows: int
    cols: int
    codes: torch.Tensor
    scales: torch.Tensor
    biases: torch.Tensor | None = None

    def to(self, device) -> "QTensor":
        return QTensor(self.qtype, self.experts, self.rows, self.cols,
                       self.codes.to(device), self.scales.to(device),
                       None if self.biases is None else self.biases.to(device))

    def expert(self, e: int) -> "QTensor":
        return QTensor(self.qtype, 1, self.rows, self.cols,
                       self.codes[e:e + 1], self.scales[e:e + 1],
                       None if self.biases is None else self.biases[e:e + 1])

    def nbytes(self) -> int:
        n = self.codes.numel() * self.codes.element_size()
        n += self.scales.numel() * 2
        if self.biases is not None:
            n += self.biases.numel() * 2
        return n


def draw_qtensor(qtype: int, experts: int, rows: int, cols: int,
                 device="cpu", seed: int = 0, layer: int = 0,
                 name: str = "w") -> QTensor:
    if qtype == Q8_0:
        assert cols % 32 == 0
        g = _gen(device, seed, layer, name, "codes")
        codes = torch.randint(-127, 128, (experts, rows, cols), generator=g,
                              device=device, dtype=torch.int8)
        g = _gen(device, seed, layer, name, "scales")
        scales = _uniform((experts, rows, cols // 32), 0.002, 0.02, device,
                          g).to(torch.float16)
        return QTensor(qtype, experts, rows, cols, codes, scales)
    assert qtype == AFFINE4_G64 and cols % 64 == 0
    g = _gen(device, seed, layer, name, "codes")
    packed = torch.randint(0, 256, (experts, rows, cols // 2), generator=g,
                           device=device, dtype=torch.uint8)
    codes = packed.view(torch.int32)
    g = _gen(device, seed, layer, name, "scales")
    scales = _uniform((experts, rows, cols // 64), 0.005, 0.05, device,
                      g).to(torch.float16)
    g = _gen(device, seed, layer, name, "biases")
    biases = _uniform((experts, rows, cols // 64), -0.4, 0.4, device,
                      g).to(torch.float16)
    return QTensor(qtype, experts, rows, cols, codes, scales, biases)


@dataclasses.dataclass
class MoELayer:
    shape: LayerShape
    w_router: torch.Tensor          # [E, H] fp32
    logit_bias: torch.Tensor | None  # [E] fp32 or None
    gate_up: QTensor                # [E, 2I, H]
    down: QTensor                   # [E, H, I]
    shared_gate_up: QTensor         # [1, 2I, H]
    shared_down: QTensor            # [1, H, I]

    def to(self, device) -> "MoELayer":
        return MoELayer(self.shape, self.w_router.to(device),
                        None if self.logit_bias is None
                        else self.logit_bias.to(device),
                        self.gate_up.to(device), self.down.to(device),
                        self.shared_gate_up.to(device),
                        self.shared_down.to(device))


def draw_layer(shape: LayerShape, device="cpu", seed: int = 0, layer: int = 0,
               zipf: str | None = None) -> MoELayer:
    """One MoE layer's weights.  zipf: None, "noise" (offset in logit-noise
    units, many empty experts) or "raw" (plain -ln(rank) offset)."""
    H, E, I, q = shape.H, shape.E, shape.I, shape.qtype
    bias = None
    if zipf is not None:
        bias = zipf_logit_bias(E, H, seed, layer,
                               in_noise_units=(zipf == "noise"), device=device)
    return MoELayer(
        shape,
        draw_router(E, H, device, seed, layer),
        bias,
        draw_qtensor(q, E, 2 * I, H, device, seed, layer, "gate_up"),
        draw_qtensor(q, E, H, I, device, seed, layer, "down"),
        draw_qtensor(q, 1, 2 * I, H, device, seed, layer, "shared_gate_up"),
        draw_qtensor(q, 1, H, I, device, seed, layer, "shared_down"),
    )


def draw_gemv(N: int, K: int, device="cpu", seed: int = 0, name="gemv"):
    """A batch-1 Q8_0 projection: (x [K] bf16, codes [N, K] int8,
    scales [N, K/32] fp16)."""
    w = draw_qtensor(Q8_0, 1, N, K, device, seed, 0, name)
    x = draw_x(1, K, device, seed, 0, name)[0]
    return x, w.codes[0], w.scales[0]
