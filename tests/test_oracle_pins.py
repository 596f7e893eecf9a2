"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compare the oracle with itself: each checks a value the pages
print, a closed form, an invariant, a brute-force result on a tiny input, or
a library routine (numpy / scipy / torch dtype conversion) on a special case.
Together they are meant to fail on a plausible slip anywhere in the oracle:
a dropped term, a wrong sign or index, a transposed operand, swapped
gate/up halves, a wrong block or group index.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth
from _helpers import bits16, oracle_layer, oracle_q, tie_free_x

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------- numbers

def test_bf16_decode_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(
        torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_decode_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------------ Q8_0 format

def test_q8_0_sizes_from_page():
    g = gold("q8_0_block.json")
    assert oracle.row_bytes(oracle.Q8_0, g["block_weights"]) == g["block_bytes"]
    assert g["tile_rows"] * oracle.row_bytes(oracle.Q8_0, 32) == g["tile_bytes"]


def test_q8_0_dequant_golden_row():
    g = gold("q8_0_block.json")["row"]
    codes = np.array(g["codes"], np.int8).reshape(1, 1, 64)
    scales = np.array([int(s, 16) for s in g["scale_f16_bits"]],
                      np.uint16).reshape(1, 1, 2)
    w = oracle.QWeights(oracle.Q8_0, codes, scales)
    got = [oracle.weight(w, 0, 0, c) for c in range(64)]
    assert got == g["values"]


def test_q8_0_indexing_multi_expert():
    # Distinct codes/scales per (expert, row, block): a wrong stride fails.
    E, R, C = 3, 4, 96
    codes = ((np.arange(E * R * C) * 7) % 255 - 127).astype(np.int8).reshape(E, R, C)
    sc = np.arange(E * R * (C // 32), dtype=np.float64).reshape(E, R, C // 32)
    scales = (0.01 + 0.001 * sc).astype(np.float16)
    w = oracle.QWeights(oracle.Q8_0, codes, scales.view(np.uint16))
    for e, n, c in [(0, 0, 0), (1, 2, 33), (2, 3, 95), (2, 0, 64), (1, 3, 31)]:
        ref = float(codes[e, n, c]) * float(scales[e, n, c // 32])
        assert oracle.weight(w, e, n, c) == ref


# --------------------------------------------------------- affine 4-bit

def test_affine4_sizes_from_page():
    g = gold("affine4_group.json")
    per_w = oracle.row_bytes(oracle.AFFINE4_G64, g["group"]) / g["group"]
    assert per_w == 0.5625
    # 2 bytes per bf16 weight -> 70 GB; the 4-bit checkpoint ~19.4 GB (the
    # page's total includes tensors we do not model, so only loosely).
    assert abs(g["params"] * 2 / 1e9 - g["bf16_gb"]) < 1e-9
    assert abs(g["params"] * per_w / 1e9 - g["checkpoint_gb"]) / g["checkpoint_gb"] < 0.02


def test_affine4_dequant_golden_row():
    g = gold("affine4_group.json")["row"]
    words = np.array([int(s, 16) for s in g["words"]], np.uint32).reshape(1, 1, 16)
    scales = np.array([int(s, 16) for s in g["scale_f16_bits"]], np.uint16).reshape(1, 1, 2)
    biases = np.array([int(s, 16) for s in g["bias_f16_bits"]], np.uint16).reshape(1, 1, 2)
    w = oracle.QWeights(oracle.AFFINE4_G64, words, scales, biases)
    assert [oracle.weight(w, 0, 0, c) for c in range(16)] == g["values_first_16"]
    assert [oracle.weight(w, 0, 0, c) for c in range(64, 73)] == g["values_group1_first_9"]
    # code 0 gives the bias, code 15 gives 15*scale + bias (closed form)
    assert oracle.weight(w, 0, 0, 0) == -1.0
    assert oracle.weight(w, 0, 0, 15) == 15 * 0.25 - 1.0


# ------------------------------------------------------------------ router

def test_router_logits_one_hot_rows():
    rng = np.random.default_rng(1)
    E, H = 6, 64
    wr = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    bias = rng.normal(0, 1, E).astype(np.float32)
    x = np.zeros((3, H), np.float32)
    x[0, 5] = 1.0
    x[1, 63] = 2.0
    x[2, 0] = -0.5
    xb = bits16(torch.from_numpy(x).to(torch.bfloat16))
    l = oracle.router_logits(xb, wr, None)
    assert np.array_equal(l[0], wr[:, 5].astype(np.float64))
    assert np.array_equal(l[1], 2.0 * wr[:, 63].astype(np.float64))
    assert np.array_equal(l[2], -0.5 * wr[:, 0].astype(np.float64))
    lb = oracle.router_logits(xb, wr, bias)
    assert np.array_equal(lb[0], wr[:, 5].astype(np.float64) + bias.astype(np.float64))


def test_router_logits_random_matches_blas():
    rng = np.random.default_rng(2)
    T, E, H = 5, 16, 256
    x = torch.randn(T, H, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    wr = rng.normal(0, 0.05, (E, H)).astype(np.float32)
    l = oracle.router_logits(bits16(x), wr, None)
    ref = x.to(torch.float64).numpy() @ wr.astype(np.float64).T
    np.testing.assert_allclose(l, ref, rtol=0, atol=1e-12)


def _brute_topk(row, k):
    order = sorted(range(len(row)), key=lambda e: (-row[e], e))
    return order[:k]


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(4)
    for trial in range(200):
        E = int(rng.integers(1, 17))
        k = int(rng.integers(1, E + 1))
        T = int(rng.integers(1, 5))
        # few distinct values -> many exact ties
        logits = rng.integers(-3, 4, (T, E)).astype(np.float64) * 0.5
        idx, w = oracle.topk(logits, k, True)
        for t in range(T):
            assert idx[t].tolist() == _brute_topk(logits[t].tolist(), k)


def test_topk_weights_softmax_identities():
    rng = np.random.default_rng(5)
    T, E, k = 7, 32, 8
    logits = rng.normal(0, 3, (T, E))
    idx, w = oracle.topk(logits, k, True)
    full = scipy.special.softmax(logits, axis=1)
    for t in range(T):
        sel = full[t, idx[t]]
        np.testing.assert_allclose(w[t], sel / sel.sum(), rtol=1e-13)
        assert abs(w[t].sum() - 1.0) < 1e-14 and (w[t] > 0).all()
        assert (np.diff(w[t]) <= 0).all()           # sorted by logit
    idx0, w0 = oracle.topk(logits, k, False)
    assert np.array_equal(idx0, idx)
    for t in range(T):
        np.testing.assert_allclose(w0[t], full[t, idx[t]], rtol=1e-13)


def test_topk_k_equals_one_and_e():
    logits = np.array([[0.1, 2.0, -1.0, 2.0]])
    idx, w = oracle.topk(logits, 1, True)
    assert idx.tolist() == [[1]] and w.tolist() == [[1.0]]
    idx, w = oracle.topk(logits, 4, True)
    assert idx.tolist() == [[1, 3, 0, 2]]


# ---------------------------------------------------------------- grouping

def test_grouping_brute_force():
    rng = np.random.default_rng(6)
    for trial in range(50):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, min(E, 8) + 1))
        T = int(rng.integers(0, 60))
        BM = int(rng.choice([1, 3, 16, 128]))
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        g = oracle.group(idx, E, BM)
        flat = idx.ravel()
        assert np.array_equal(g["counts"], np.bincount(flat, minlength=E))
        assert g["offsets"][0] == 0 and g["offsets"][-1] == T * k
        assert np.array_equal(np.diff(g["offsets"]), g["counts"])
        assert np.array_equal(g["perm"], np.argsort(flat, kind="stable"))
        assert np.array_equal(g["inv_perm"][g["perm"]], np.arange(T * k))
        # the block map covers every expert group exactly once, in order
        covered = []
        for e, r0 in g["tile_map"]:
            end = min(r0 + BM, g["offsets"][e + 1])
            assert g["offsets"][e] <= r0 < end
            covered.extend(range(r0, end))
        assert covered == list(range(T * k))
        assert g["n_tiles"] == sum(-(-int(c) // BM) for c in g["counts"])


def test_grouping_counts_from_page():
    g = gold("routing_counts.json")
    rng = np.random.default_rng(7)
    idx = np.stack([rng.permutation(g["E"])[:g["k"]] for _ in range(g["T"])]).astype(np.int32)
    r = oracle.group(idx, g["E"], 128)
    assert int(r["counts"].sum()) == g["assignments"]
    assert r["counts"].mean() == g["mean_rows_per_expert"]


def test_grouping_rejects_bad_expert_id():
    with pytest.raises(ValueError):
        oracle.group(np.array([[0, 5]], np.int32), 4, 16)


# -------------------------------------------------------------- activation

def test_silu_matches_library():
    for g in [-30.0, -2.5, -1e-3, 0.0, 1e-3, 0.7, 3.0, 40.0]:
        ref = g * scipy.special.expit(g)
        assert abs(oracle.silu(g) - ref) <= 1e-15 * max(1.0, abs(ref))
    assert oracle.silu(0.0) == 0.0


# -------------------------------------------------------------- expert FFN

def _const_q8(E, R, C, code_of_row, scale_of_row):
    codes = np.empty((E, R, C), np.int8)
    scales = np.empty((E, R, C // 32), np.float16)
    for e in range(E):
        for n in range(R):
            codes[e, n, :] = code_of_row(e, n)
            scales[e, n, :] = scale_of_row(e, n)
    return oracle.QWeights(oracle.Q8_0, codes, scales.view(np.uint16))


def test_expert_closed_form_constant_weights():
    # gate rows code 3 scale 1/64, up rows code -5 scale 1/32, x = 0.5 everywhere
    # -> g = 3/64 * 0.5 * H, u = -5/32 * 0.5 * H, h = silu(g) * u for all i;
    # down row n: code n - 7, scale 1/8 -> o[n] = (n-7)/8 * I * h.
    H, I = 64, 32
    gu = _const_q8(1, 2 * I, H, lambda e, n: 3 if n < I else -5,
                   lambda e, n: 1 / 64 if n < I else 1 / 32)
    dn = _const_q8(1, H, I, lambda e, n: n - 7, lambda e, n: 1 / 8)
    x = np.full(H, 0.5)
    o, g_u, h = oracle.expert_ffn(gu, dn, 0, x)
    g = 3 / 64 * 0.5 * H
    u = -5 / 32 * 0.5 * H
    hv = g / (1 + math.exp(-g)) * u
    assert np.all(g_u[:I] == g) and np.all(g_u[I:] == u)
    np.testing.assert_allclose(h, hv, rtol=1e-15)
    np.testing.assert_allclose(o, [(n - 7) / 8 * I * hv for n in range(H)], rtol=1e-14)


def test_expert_one_hot_and_dense_library():
    L = synth.draw_layer(synth.TINY, "cpu", seed=11)
    gu_q, dn_q, _, _ = oracle_layer(L)
    e = 5
    Wgu = oracle.dequant_expert(gu_q, e)
    Wdn = oracle.dequant_expert(dn_q, e)
    H, I = synth.TINY.H, synth.TINY.I
    # one-hot x: gu = the column of Wgu
    x = np.zeros(H)
    x[17] = 1.0
    _, g_u, _ = oracle.expert_ffn(gu_q, dn_q, e, x)
    assert np.array_equal(g_u, Wgu[:, 17])
    # random x: dense fp64 SwiGLU MLP through numpy matmul
    x = np.random.default_rng(12).normal(size=H)
    o, g_u, h = oracle.expert_ffn(gu_q, dn_q, e, x)
    gd, ud = Wgu[:I] @ x, Wgu[I:] @ x
    hd = gd * scipy.special.expit(gd) * ud
    np.testing.assert_allclose(g_u, np.concatenate([gd, ud]), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h, hd, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(o, Wdn @ hd, rtol=1e-10, atol=1e-10)


def test_fused_gate_up_equals_separate_rowwise():
    # oMLX gate/up fusion: concatenating gate and up along the output axis
    # gives, per row, the same bits as the two separate matmuls.
    assert gold("gate_up_fusion.json")["order"] == ["gate", "up"]
    L = synth.draw_layer(synth.TINY, "cpu", seed=13)
    I = synth.TINY.I
    fused = oracle_q(L.gate_up)
    gate = oracle.QWeights(fused.qtype, fused.codes[:, :I].copy(), fused.scales[:, :I].copy())
    up = oracle.QWeights(fused.qtype, fused.codes[:, I:].copy(), fused.scales[:, I:].copy())
    x = np.random.default_rng(14).normal(size=synth.TINY.H)
    for e in (0, 9):
        f = oracle.qmatvec(fused, e, x)
        assert np.array_equal(f[:I], oracle.qmatvec(gate, e, x))
        assert np.array_equal(f[I:], oracle.qmatvec(up, e, x))


def test_affine4_expert_against_dense_library():
    shape = synth.LayerShape(H=128, E=3, k=1, I=64, qtype=synth.AFFINE4_G64)
    L = synth.draw_layer(shape, "cpu", seed=15)
    gu_q, dn_q, _, _ = oracle_layer(L)
    x = np.random.default_rng(16).normal(size=128)
    o, g_u, _ = oracle.expert_ffn(gu_q, dn_q, 2, x)
    # independent dequant in numpy from the bit layout
    codes = L.gate_up.codes[2].numpy().view(np.uint32)
    nib = np.stack([(codes >> (4 * j)) & 15 for j in range(8)], axis=-1).reshape(128, 128)
    sc = L.gate_up.scales[2].to(torch.float64).numpy().repeat(64, axis=1)
    bi = L.gate_up.biases[2].to(torch.float64).numpy().repeat(64, axis=1)
    W = sc * nib + bi
    np.testing.assert_allclose(g_u, W @ x, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ layer

def test_layer_combine_closed_form():
    # Each routed expert e is constant (code e+1 in every gate/up/down row,
    # scale 1/16); the shared expert has all-zero codes.  Then
    # o_e[n] = (e+1)/16 * I * h_e with h_e = silu(g_e) * g_e,
    # g_e = (e+1)/16 * sum(x), and y = sum_j w_j o_{e_j}: a swapped
    # weight/expert pairing or a dropped term changes the result.
    H, I, E, k = 64, 32, 4, 2
    gu = _const_q8(E, 2 * I, H, lambda e, n: e + 1, lambda e, n: 1 / 16)
    dn = _const_q8(E, H, I, lambda e, n: e + 1, lambda e, n: 1 / 16)
    z_gu = _const_q8(1, 2 * I, H, lambda e, n: 0, lambda e, n: 1.0)
    z_dn = _const_q8(1, H, I, lambda e, n: 0, lambda e, n: 1.0)
    x = torch.full((1, H), 0.25).to(torch.bfloat16)
    idx = np.array([[2, 0]], np.int32)
    w = np.array([[0.7, 0.3]])
    y = oracle.moe_layer(bits16(x), idx, w, gu, dn, z_gu, z_dn)

    def o(e):
        g = (e + 1) / 16 * 0.25 * H
        h = g / (1 + math.exp(-g)) * g
        return (e + 1) / 16 * I * h
    np.testing.assert_allclose(y[0], 0.7 * o(2) + 0.3 * o(0), rtol=1e-14)


def test_layer_single_expert_is_dense_mlp():
    # E = 1, k = 1: the layer is the dense SwiGLU MLP of the one expert plus
    # the shared expert's MLP (routing weight 1).
    shape = synth.LayerShape(H=128, E=1, k=1, I=64)
    L = synth.draw_layer(shape, "cpu", seed=17)
    x = synth.draw_x(3, 128, "cpu", seed=17)
    idx, w = oracle.route(bits16(x), L.w_router.numpy(), 1)
    assert idx.tolist() == [[0]] * 3 and np.all(w == 1.0)
    gu_q, dn_q, sgu_q, sdn_q = oracle_layer(L)
    y = oracle.moe_layer(bits16(x), idx, w, gu_q, dn_q, sgu_q, sdn_q)
    X = x.to(torch.float64).numpy()

    def mlp(guq, dnq):
        Wg = oracle.dequant_expert(guq, 0)
        Wd = oracle.dequant_expert(dnq, 0)
        G, U = X @ Wg[:64].T, X @ Wg[64:].T
        return (G * scipy.special.expit(G) * U) @ Wd.T
    np.testing.assert_allclose(y, mlp(gu_q, dn_q) + mlp(sgu_q, sdn_q), rtol=1e-10, atol=1e-9)


def test_layer_token_subset_and_order():
    L = synth.draw_layer(synth.TINY, "cpu", seed=18)
    x = tie_free_x(L, 4, seed=18)
    idx, w = oracle.route(bits16(x), L.w_router.numpy(), 2)
    q = oracle_layer(L)
    full = oracle.moe_layer(bits16(x), idx, w, *q)
    sub = oracle.moe_layer(bits16(x), idx, w, *q, tokens=[3, 1])
    assert np.array_equal(sub[0], full[3]) and np.array_equal(sub[1], full[1])


# ------------------------------------------- router / shared-expert variants

def test_topk_selection_only_bias_hand_example():
    # E = 4, k = 2, logits l and a bias that moves experts 0 and 2 to the top:
    # selection by l + b = [4, 2, 3, 1.5] -> experts (0, 2); the weights use
    # the unbiased logits (1.0, 0.5): w0 = 1 / (1 + e^-0.5); the plain router
    # weights the biased logits (4, 3) instead: w0 = 1 / (1 + e^-1).
    l = np.array([[1.0, 2.0, 0.5, 1.5]])
    b = np.array([3.0, 0.0, 2.5, 0.0])
    idx, w = oracle.topk_sel(l + b, l, 2, True)
    assert idx.tolist() == [[0, 2]]
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-0.5)), 1 / (1 + math.exp(0.5))],
                               rtol=1e-15)
    idx2, w2 = oracle.topk(l + b, 2, True)
    assert idx2.tolist() == [[0, 2]]
    np.testing.assert_allclose(w2[0], [1 / (1 + math.exp(-1.0)), 1 / (1 + math.exp(1.0))],
                               rtol=1e-15)
    # full softmax at the selected experts: e^l_j / sum_e e^l_e (unbiased)
    _, w3 = oracle.topk_sel(l + b, l, 2, False)
    den = sum(math.exp(v) for v in l[0])
    np.testing.assert_allclose(w3[0], [math.exp(1.0) / den, math.exp(0.5) / den], rtol=1e-15)


def test_route_selection_only_bias_reduces_to_plain():
    # a zero bias, or one equal for every expert, selects and weights exactly
    # like the plain router; a real bias changes the selection only through
    # l + b and leaves the weights those of the unbiased logits
    L = synth.draw_layer(synth.TINY, "cpu", seed=30, zipf="noise")
    x = tie_free_x(L, 6, seed=30)
    xb, wr = bits16(x), L.w_router.numpy()
    i0, w0 = oracle.route(xb, wr, 2)
    i1, w1 = oracle.route(xb, wr, 2, np.zeros(16, np.float32), True, True)
    assert np.array_equal(i0, i1) and np.array_equal(w0, w1)
    bias = L.logit_bias.numpy()
    i2, w2 = oracle.route(xb, wr, 2, bias, True, True)
    lb = oracle.router_logits(xb, wr, bias)
    lu = oracle.router_logits(xb, wr, None)
    ref_i = np.argsort(-lb, axis=1, kind="stable")[:, :2]
    assert np.array_equal(i2, ref_i)
    sel = np.take_along_axis(lu, ref_i, axis=1)
    ref_w = np.exp(sel - sel.max(1, keepdims=True))
    ref_w /= ref_w.sum(1, keepdims=True)
    np.testing.assert_allclose(w2, ref_w, rtol=1e-13)


def test_shared_gate_closed_forms():
    H = 64
    x = torch.zeros((3, H))
    x[0, 5] = 1.0          # one-hot: z = w_sg[5]
    x[1, :] = 0.5          # constant: z = 0.5 * sum(w_sg)
    xb = bits16(x.to(torch.bfloat16))
    w = np.zeros(H, np.float32)
    g0 = oracle.shared_gate(xb, w)
    assert np.array_equal(g0, [0.5, 0.5, 0.5])   # sigmoid(0) exactly
    w[5] = math.log(3.0)
    g = oracle.shared_gate(xb, w)
    # sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4; w_sg[5] is ln 3 rounded to fp32,
    # which moves the gate by less than 1e-8
    assert abs(g[0] - 0.75) < 1e-8
    # constant row: z = 0.5 * w_sg[5]
    z = 0.5 * float(np.float32(math.log(3.0)))
    np.testing.assert_allclose(g[1], 1 / (1 + math.exp(-z)), rtol=1e-14)
    assert g[2] == 0.5


def test_layer_gated_shared_expert_is_linear_in_the_gate():
    # y(g) = y(0) + g * o_shared: with g = 1 the gated layer equals the plain
    # layer bit for bit, and any g interpolates linearly
    L = synth.draw_layer(synth.TINY, "cpu", seed=31)
    x = tie_free_x(L, 3, seed=31)
    xb = bits16(x)
    idx, w = oracle.route(xb, L.w_router.numpy(), 2)
    q = oracle_layer(L)
    plain = oracle.moe_layer(xb, idx, w, *q)
    y1 = oracle.moe_layer(xb, idx, w, *q, shared_w=np.ones(3))
    assert np.array_equal(plain, y1)
    y0 = oracle.moe_layer(xb, idx, w, *q, shared_w=np.zeros(3))
    g = np.array([0.25, 0.5, 0.9])
    yg = oracle.moe_layer(xb, idx, w, *q, shared_w=g)
    np.testing.assert_allclose(yg, y0 + g[:, None] * (y1 - y0), rtol=1e-12, atol=1e-12)
    # y(1) - y(0) is the shared expert's own output (one-expert FFN)
    X = x.to(torch.float64).numpy()
    for t in range(3):
        o_sh, _, _ = oracle.expert_ffn(q[2], q[3], 0, X[t])
        np.testing.assert_allclose(y1[t] - y0[t], o_sh, rtol=1e-9, atol=1e-9)


# ------------------------------------------------------------------ GEMV

def test_q8_gemv_one_hot_and_library():
    x, q, d = synth.draw_gemv(48, 96, "cpu", seed=19)
    qn, dn = q.numpy(), bits16(d)
    oh = torch.zeros(96).to(torch.bfloat16)
    oh[70] = 1.0
    y = oracle.q8_gemv(bits16(oh), qn, dn)
    dd = d.to(torch.float64).numpy()
    assert np.array_equal(y, qn[:, 70].astype(np.float64) * dd[:, 70 // 32])
    y = oracle.q8_gemv(bits16(x), qn, dn)
    W = qn.astype(np.float64) * dd.repeat(32, axis=1)
    np.testing.assert_allclose(y, W @ x.to(torch.float64).numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------- input recipe

def test_zipf_offset_leaves_empty_experts():
    # Recipe check (not the method): the noise-unit Zipf offset skews routing
    # enough that some experts get no token at T=4096.
    E, H = 256, 2048
    b = synth.zipf_logit_bias(E, H, seed=0)
    assert b.max().item() == 0.0 and sorted(b.tolist())[0] < -10


# --------------------------------------------- int8-activation GEMV mode

def _exact_blocks(K, seed):
    """x whose blocks are integers j * 2^-7 with max |j| = 127 per block
    (then d = 2^-7 exactly and the codes are the integers j), with a
    different power-of-two scale per block so block indices matter."""
    rng = np.random.default_rng(seed)
    j = rng.integers(-127, 128, size=K)
    j[::32] = 127 * np.where(rng.random(K // 32) < 0.5, 1, -1)
    scale = 2.0 ** (-7 - (np.arange(K) // 32) % 3)
    return torch.from_numpy(j * scale).to(torch.bfloat16), j


def test_quantize_x_exact_codes_and_special_blocks():
    x, j = _exact_blocks(256, 40)
    q, d = oracle.q8_quantize_x(bits16(x))
    assert np.array_equal(q.astype(np.int64), j)
    np.testing.assert_array_equal(d, (2.0 ** (-7 - np.arange(8) % 3)).astype(np.float32))
    z = torch.zeros(64, dtype=torch.bfloat16)
    z[40] = -3.0
    qz, dz = oracle.q8_quantize_x(bits16(z))
    assert dz[0] == 0.0 and not qz[:32].any()          # all-zero block
    assert qz[40] == -127 and np.count_nonzero(qz[32:]) == 1
    assert dz[1] == np.float32(3.0) / np.float32(127.0)


def test_quantize_x_reconstruction_bound():
    x = synth.draw_x(1, 4096, "cpu", seed=41).reshape(-1)
    q, d = oracle.q8_quantize_x(bits16(x))
    X = x.to(torch.float64).numpy()
    err = np.abs(X - np.repeat(d.astype(np.float64), 32) * q)
    # half a step, plus the fp32 rounding of x / d (|x / d| <= 127)
    assert np.all(err <= np.repeat(d.astype(np.float64), 32) * (0.5 + 127 * 2.0 ** -22))
    assert np.abs(q).max() == 127


def test_gemv_i8_equals_exact_gemv_on_quantizable_x():
    N, K = 40, 256
    _, q, d = synth.draw_gemv(N, K, "cpu", seed=42)
    x, _ = _exact_blocks(K, 43)
    qx, dx = oracle.q8_quantize_x(bits16(x))
    y8 = oracle.q8_gemv_i8(qx, dx, q.numpy(), bits16(d))
    y = oracle.q8_gemv(bits16(x), q.numpy(), bits16(d))
    np.testing.assert_allclose(y8, y, rtol=1e-12, atol=1e-12)


def test_gemv_i8_within_quantization_bound():
    N, K = 32, 512
    x, q, d = synth.draw_gemv(N, K, "cpu", seed=44)
    qx, dx = oracle.q8_quantize_x(bits16(x))
    y8 = oracle.q8_gemv_i8(qx, dx, q.numpy(), bits16(d))
    y = oracle.q8_gemv(bits16(x), q.numpy(), bits16(d))
    dw = d.to(torch.float64).numpy().reshape(N, K // 32)
    qa = np.abs(q.numpy().astype(np.float64)).reshape(N, K // 32, 32).sum(2)
    bound = (np.abs(dw) * qa * dx.astype(np.float64)[None, :] / 2).sum(1)
    assert np.all(np.abs(y8 - y) <= bound * (1 + 1e-6) + 1e-12)
    assert np.abs(y8 - y).max() > 0   # it is an approximation
