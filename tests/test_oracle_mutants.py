"""The oracle's pins must catch plausible slips.

Each case plants one mistake in a copy of oracle.c (on the CPU), builds it,
swaps it in for the real oracle library and runs every pin in
test_oracle_pins.py: at least one pin has to fail.  Mutations are chosen to
stay in bounds so a mutant cannot crash the test process.
"""
import os
import shutil
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "bf16 exponent bias": ("exp - 127);", "exp - 126);"),
    "f16 subnormal scale": ("-14 - 10", "-15 - 10"),
    "q8 block index": ("m->scales[row * (m->cols / 32) + c / 32]",
                       "m->scales[row * (m->cols / 32)]"),
    "affine bias dropped": ("return scale * code + bias;", "return scale * code;"),
    "nibble order": ("(word >> (4 * (c % 8)))", "(word >> (4 * (7 - c % 8)))"),
    "router operand transposed": ("(double)w_router[(size_t)e * H + h]",
                                  "(double)w_router[(size_t)h * E + e]"),
    "router bias dropped": ("if (bias) acc += (double)bias[e];", "(void)bias;"),
    "tie break": ("return (a->e < b->e) ? -1 : (a->e > b->e);",
                  "return (a->e > b->e) ? -1 : (a->e < b->e);"),
    "softmax denominator": ("for (int j = 0; j < k; ++j) denom += exp(w[s[j].e] - top);",
                            "for (int j = 0; j < k && j < 1; ++j) denom += exp(w[s[j].e] - top);"),
    "full softmax over the selection": ("for (int e = 0; e < E; ++e) denom += exp(w[e] - top);",
                                        "for (int e = 0; e < k; ++e) denom += exp(w[e] - top);"),
    "softmax sign": ("topk_w[(size_t)t * k + j] = exp(w[s[j].e] - top) / denom;",
                     "topk_w[(size_t)t * k + j] = exp(top - w[s[j].e]) / denom;"),
    "weights from the selection logits": ("const double* w = wl + (size_t)t * E;",
                                          "const double* w = sel + (size_t)t * E;"),
    "shared gate sign": ("gate[t] = 1.0 / (1.0 + exp(-z));",
                         "gate[t] = 1.0 / (1.0 + exp(z));"),
    "shared gate index": ("(double)w_sg[h]", "(double)w_sg[H - 1 - h]"),
    "shared gate ignored": ("(shared_w ? shared_w[t] : 1.0)", "1.0"),
    "unstable scatter": ("for (int64_t a = 0; a < A; ++a)\n      if (topk_idx[a] == e) perm[pos++] = (int32_t)a;",
                         "for (int64_t a = A - 1; a >= 0; --a)\n      if (topk_idx[a] == e) perm[pos++] = (int32_t)a;"),
    "tile row step": ("tile_map[2 * nt + 1] = offsets[e] + m * BM;",
                      "tile_map[2 * nt + 1] = offsets[e] + m;"),
    "silu sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "gate/up swapped": ("h[i] = orc_silu(gu[i]) * gu[I + i];",
                        "h[i] = orc_silu(gu[I + i]) * gu[i];"),
    "shared expert dropped": ("acc += (shared_w ? shared_w[t] : 1.0) * o[(i * (k + 1) + k) * H + n];",
                              "(void)shared_w;"),
    "routing weight pairing": ("acc += topk_w[(size_t)t * k + j] * o[(i * (k + 1) + j) * H + n];",
                               "acc += topk_w[(size_t)t * k + (k - 1 - j)] * o[(i * (k + 1) + j) * H + n];"),
    "gemv block index": ("orc_f16_to_f64(d[(size_t)n * (K / 32) + c / 32])",
                         "orc_f16_to_f64(d[(size_t)n * (K / 32)])"),
    "activation scale 128": ("const float db = amax / 127.0f;", "const float db = amax / 128.0f;"),
    "truncating activation codes": ("r = roundf(v / db);", "r = truncf(v / db);"),
    "activation block scale index": ("* (double)dx[b] *", "* (double)dx[0] *"),
    "int8 dot input index": ("(long long)qx[32 * b + i]", "(long long)qx[i]"),
    "matvec input index": ("acc += orc_weight(m, e, n, c) * x[c];",
                           "acc += orc_weight(m, e, n, c) * x[m->cols - 1 - c];"),
}


def _pin_functions():
    return [getattr(pins, n) for n in sorted(dir(pins))
            if n.startswith("test_") and callable(getattr(pins, n))]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique/found: {old!r}"
    mut = tmp_path / "oracle_mut.c"
    mut.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-o", str(so), str(mut), "-lm"], check=True)
    real = oracle._load()
    try:
        oracle._lib = None
        saved_path = oracle._LIB_PATH
        oracle._LIB_PATH = str(so)
        oracle._SRC_SAVED = oracle._SRC
        oracle._SRC = str(mut)
        oracle._load()
        failed = []
        for fn in _pin_functions():
            try:
                fn()
            except Exception as exc:  # noqa: BLE001 - any failure counts
                failed.append((fn.__name__, type(exc).__name__))
    finally:
        oracle._lib = real
        oracle._LIB_PATH = saved_path
        oracle._SRC = oracle._SRC_SAVED
    assert failed, f"mutant '{name}' survived every pin"
