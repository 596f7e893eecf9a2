"""Router and grouping kernels against the oracle: bit-exact ids, counts,
permutations and block maps; routing weights within 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _gpu_cases import TOPK_W_ATOL, layer, oracle_route, x_for

pytestmark = pytest.mark.gpu

ROUTE_CASES = [
    # (shape, T, zipf, renormalize)
    (synth.TINY, 4, None, True),
    (synth.TINY, 1, None, False),
    (synth.QWEN, 1, None, True),
    (synth.QWEN, 3, None, True),
    (synth.QWEN, 16, None, True),
    (synth.QWEN, 40, None, True),
    (synth.QWEN, 64, None, False),
    (synth.QWEN, 65, None, True),
    (synth.TINY, 100, None, False),          # tensor-core router, E = 16
    (synth.QWEN, 300, None, False),          # tensor-core router, full softmax
    (synth.QWEN, 1000, "noise", True),
    (synth.QWEN, 4096, "noise", True),
    # tensor-core router with 2 slices of H per tile (H % 256 != 0), a
    # ragged last tile, and the full softmax
    (synth.LayerShape(H=384, E=64, k=4, I=128), 200, None, True),
    (synth.LayerShape(H=384, E=64, k=4, I=128), 129, None, False),
]


def _router_only(shape, seed, zipf):
    wr = synth.draw_router(shape.E, shape.H, "cpu", seed, 0)
    bias = None
    if zipf:
        bias = synth.zipf_logit_bias(shape.E, shape.H, seed, 0,
                                     in_noise_units=(zipf == "noise"))
    return wr, bias


@pytest.mark.parametrize("shape,T,zipf,renorm", ROUTE_CASES)
def test_route_matches_oracle(qsm, shape, T, zipf, renorm):
    seed = 100 + T
    wr, bias = _router_only(shape, seed, zipf)
    L = synth.MoELayer(shape, wr, bias, None, None, None, None)
    from _helpers import tie_free_x
    x = tie_free_x(L, T, seed=seed)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w = qsm.moe_route(x.cuda(), wr.cuda(), shape.k,
                           None if bias is None else bias.cuda(), renorm,
                           dev_status=st)
    torch.cuda.synchronize()
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, renorm)
    assert st.item() == 0
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=0, atol=TOPK_W_ATOL)


def test_route_workspace_is_rearmed(qsm):
    """Two calls in a row on one workspace give the same result."""
    shape = synth.QWEN
    wr, bias = _router_only(shape, 7, None)
    x = synth.draw_x(24, shape.H, "cuda", 7)
    ws = torch.zeros(qsm.route_workspace_bytes(24, shape.H, shape.E),
                     dtype=torch.uint8, device="cuda")
    a = qsm.moe_route(x, wr.cuda(), 8, workspace=ws)
    a = (a[0].clone(), a[1].clone())
    b = qsm.moe_route(x, wr.cuda(), 8, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    counters = ws[:256]                     # the arrival counters come first
    assert int(counters.sum().item()) == 0


def _check_grouping(g, idx, E, BM):
    ref = oracle.group(idx, E, BM)
    assert np.array_equal(g.counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(g.offsets.cpu().numpy(), ref["offsets"])
    A = idx.size
    assert np.array_equal(g.perm.cpu().numpy()[:A], ref["perm"])
    assert np.array_equal(g.inv_perm.cpu().numpy()[:A], ref["inv_perm"])
    nt = int(g.n_tiles.item())
    assert nt == ref["n_tiles"]
    assert np.array_equal(g.tile_map.cpu().numpy()[:2 * nt].reshape(nt, 2),
                          ref["tile_map"])


@pytest.mark.parametrize("T,k,E,BM", [
    (0, 8, 256, 8), (1, 8, 256, 8), (3, 2, 16, 8), (64, 8, 256, 8),
    (65, 8, 256, 128), (4096, 8, 256, 128), (4096, 8, 256, 8),
    (777, 4, 1024, 16), (2048, 8, 256, 32)])
def test_group_matches_oracle(qsm, T, k, E, BM):
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
        if T else np.zeros((0, k), np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = qsm.moe_group_tokens(torch.from_numpy(idx).cuda(), E, BM, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    _check_grouping(g, idx, E, BM)


def test_group_skewed_all_to_one_expert_block(qsm):
    """Every token routed to the same k experts (one huge group each)."""
    T, k, E, BM = 3000, 8, 256, 128
    idx = np.tile(np.arange(100, 100 + k, dtype=np.int32), (T, 1))
    g = qsm.moe_group_tokens(torch.from_numpy(idx).cuda(), E, BM)
    torch.cuda.synchronize()
    _check_grouping(g, idx, E, BM)


def test_group_flags_bad_expert_id(qsm):
    T, k, E = 5, 2, 16
    idx = np.array([[0, 1], [2, 99], [3, 4], [-1, 5], [6, 7]], np.int32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = qsm.moe_group_tokens(torch.from_numpy(idx).cuda(), E, 8, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & qsm.DEV_BAD_EXPERT_ID
    inv = g.inv_perm.cpu().numpy()
    assert inv[3] == -1 and inv[6] == -1
    assert int(g.offsets[E].item()) == T * k - 2
    valid = idx.ravel().copy()
    ok = (valid >= 0) & (valid < E)
    assert int(g.counts.sum().item()) == ok.sum()


@pytest.mark.parametrize("shape,T,zipf,renorm", [
    (synth.QWEN, 1, None, True), (synth.QWEN, 2, None, True),
    (synth.QWEN, 3, "noise", True), (synth.QWEN, 8, None, False),
    (synth.TINY, 4, None, True), (synth.TINY, 8, None, False)])
def test_fused_route_group_matches_separate_calls(qsm, shape, T, zipf, renorm):
    """moe_route_group gives the routing and grouping of moe_route +
    moe_group_tokens bit for bit, and the oracle's routing and grouping."""
    seed = 300 + T
    wr, bias = _router_only(shape, seed, zipf)
    L = synth.MoELayer(shape, wr, bias, None, None, None, None)
    from _helpers import tie_free_x
    x = tie_free_x(L, T, seed=seed).cuda()
    wrc, bc = wr.cuda(), None if bias is None else bias.cuda()
    BM = 8
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g1 = qsm.Grouping.empty(T, shape.k, shape.E, BM, "cuda")
    i1, w1 = qsm.moe_route_group(x, wrc, shape.k, g1, bc, renorm, dev_status=st)
    i2, w2 = qsm.moe_route(x, wrc, shape.k, bc, renorm, dev_status=st)
    g2 = qsm.moe_group_tokens(i2, shape.E, BM, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(i1, i2)
    assert torch.equal(w1, w2)
    for name in ("counts", "offsets", "perm", "inv_perm", "n_tiles"):
        assert torch.equal(getattr(g1, name), getattr(g2, name)), name
    nt = int(g1.n_tiles.item())
    assert torch.equal(g1.tile_map[:2 * nt], g2.tile_map[:2 * nt])
    idx_o, w_o = oracle_route(x.cpu(), wr, bias, shape.k, renorm)
    assert np.array_equal(i1.cpu().numpy(), idx_o)
    np.testing.assert_allclose(w1.cpu().numpy(), w_o, rtol=0, atol=TOPK_W_ATOL)
    _check_grouping(g1, idx_o, shape.E, BM)


def test_fused_route_group_rejects_unsupported(qsm):
    shape = synth.QWEN
    x = synth.draw_x(9, shape.H, "cuda", 1)
    g = qsm.Grouping.empty(9, shape.k, shape.E, 8, "cuda")
    assert qsm.moe_route_group(x, synth.draw_router(shape.E, shape.H, "cuda", 1),
                               shape.k, g, raise_unsupported=False) is None
    x = synth.draw_x(2, shape.H, "cuda", 1)            # E > 256
    g = qsm.Grouping.empty(2, shape.k, 512, 8, "cuda")
    assert qsm.moe_route_group(x, synth.draw_router(512, shape.H, "cuda", 1),
                               shape.k, g, raise_unsupported=False) is None


def test_fused_route_group_repeat_and_bias(qsm):
    """Back-to-back calls on one workspace (the arrival counter re-arms) with
    a logit bias that sends several tokens to the same experts, so groups
    hold more than one row and span blocks of 2 rows."""
    shape = synth.QWEN
    T, BM = 8, 2
    wr = synth.draw_router(shape.E, shape.H, "cpu", 11)
    bias = torch.zeros(shape.E)
    bias[[3, 17, 200]] = torch.tensor([40.0, 60.0, 80.0])
    from _helpers import tie_free_x
    x = tie_free_x(synth.MoELayer(shape, wr, bias, None, None, None, None), T, seed=11)
    ws = torch.zeros(max(qsm.route_workspace_bytes(T, shape.H, shape.E), 256),
                     dtype=torch.uint8, device="cuda")
    g = qsm.Grouping.empty(T, shape.k, shape.E, BM, "cuda")
    for _ in range(2):
        i1, w1 = qsm.moe_route_group(x.cuda(), wr.cuda(), shape.k, g, bias.cuda(),
                                     True, workspace=ws)
    torch.cuda.synchronize()
    idx_o, w_o = oracle_route(x, wr, bias, shape.k, True)
    assert (idx_o[:, :3] == np.array([200, 17, 3])).all()
    assert np.array_equal(i1.cpu().numpy(), idx_o)
    np.testing.assert_allclose(w1.cpu().numpy(), w_o, rtol=0, atol=TOPK_W_ATOL)
    _check_grouping(g, idx_o, shape.E, BM)
    assert int(ws[:256].sum().item()) == 0
