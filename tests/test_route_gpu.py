"""Parity of routing (smoe_route_topk_bf16) and the weighted combine
(smoe_combine) with the f64 oracle, through the C ABI.

Logits are held to the matvec tolerance.  The selection is an integer
decision taken on the GPU's f32 logits, so it is compared bit for bit with
the oracle's selection applied to those same logits (values, ties to the
lower index, NaN last), and the weights with the oracle's weights of those
logits.  A full layer (route, the selected experts' FFN, combine) is checked
against the oracle's FFN of the same experts combined with the same weights.
"""
import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


@pytest.fixture(scope="module")
def smoe(dev):
    import moe_expert_ffn_smoe_gb300 as m
    return m


def _route(smoe, dev, g, x, n, d, k):
    logits = torch.full((n,), float("nan"), device=dev)
    idx = torch.full((k,), -1, dtype=torch.int32, device=dev)
    w = torch.full((k,), float("nan"), device=dev)
    smoe.smoe_route_topk_bf16(to_dev(g, dev), to_dev(x, dev), n, d, k, logits, idx, w)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("n,d,k,seed", [
    (128, 4096, 8, 1),      # the page's router shape, top-8
    (1, 8, 1, 2),           # one expert
    (3, 16, 3, 3),          # every expert selected
    (8192, 512, 64, 4),     # the largest n and k accepted
    (130, 2048, 7, 5),      # a ragged expert count
    (256, 1024, 64, 11),    # the largest n of the rank-counting selection
    (257, 1024, 8, 12),     # the smallest n of the round-by-round selection
])
def test_route(smoe, dev, n, d, k, seed):
    g = inp.bf16_rows(n, d, seed, 1)
    x = inp.activations(d, seed)
    logits, idx, w = _route(smoe, dev, g, x, n, d, k)
    ref, a = oracle.matvec_bf16(g, n, d, x.astype(np.float64))
    check(logits, ref, a, f"router logits {n}x{d}")
    oi, ow = oracle.topk(logits.astype(np.float64), k)
    np.testing.assert_array_equal(idx, oi)
    np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("n", [16, 600])
def test_route_ties_go_to_the_lower_index(smoe, dev, n):
    """Three equal rows holding the largest logit: all three are selected,
    in ascending index order, ahead of every other expert."""
    d, k = 64, 6
    g = inp.bf16_rows(n, d, 6, 1)
    x = inp.activations(d, 6)
    ref, _ = oracle.matvec_bf16(g, n, d, x.astype(np.float64))
    m = int(np.argmax(ref))
    tied = sorted({m, (m + 7) % n, (m + n // 2) % n})
    for e in tied:
        g[e] = g[m]
    logits, idx, w = _route(smoe, dev, g, x, n, d, k)
    assert logits[tied[0]] == logits[tied[1]] == logits[tied[2]]
    oi, ow = oracle.topk(logits.astype(np.float64), k)
    np.testing.assert_array_equal(idx, oi)
    np.testing.assert_array_equal(idx[:3], tied)
    assert w[0] == w[1] == w[2]


@pytest.mark.parametrize("n", [32, 300])
def test_route_nan_token_selects_by_index(smoe, dev, n):
    d, k = 64, 4
    g = inp.bf16_rows(n, d, 7, 1)
    x = inp.activations(d, 7)
    x[5] = np.nan
    logits, idx, w = _route(smoe, dev, g, x, n, d, k)
    assert np.isnan(logits).all()
    np.testing.assert_array_equal(idx, np.arange(k))
    assert np.isnan(w).all()


@pytest.mark.parametrize("k,d", [(8, 4096), (1, 100), (64, 1024), (0, 256)])
def test_combine(smoe, dev, k, d):
    rng = np.random.default_rng(8 + k)
    eo = rng.normal(size=(max(k, 1), d)).astype(np.float32)[:k]
    w = rng.dirichlet(np.ones(max(k, 1))).astype(np.float32)[:k]
    out = torch.full((d,), float("nan"), device=dev)
    smoe.smoe_combine(k, to_dev(eo, dev) if k else None, to_dev(w, dev) if k else None, out, d)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    if k == 0:
        assert (got == 0).all()
        return
    ref, a = oracle.combine(eo.astype(np.float64), w.astype(np.float64))
    # k f32 products and sums: well inside 1e-6 of sum |w y|
    assert (np.abs(got - ref) <= 1e-6 * a + 1e-7).all()


def test_moe_layer_route_experts_combine(smoe, dev):
    """Router over 16 experts, top-4, the selected experts' FFN in one call,
    then the combine: against the oracle on the GPU's selection and weights."""
    n, k, d_model, d_ff, group = 16, 4, 1024, 512, 64
    experts = [inp.expert(4, d_model, d_ff, group, 9, e) for e in range(n)]
    tens = [{kk: to_dev(v, dev) for kk, v in ex.items()} for ex in experts]
    g = inp.bf16_rows(n, d_model, 9, 2)
    x = inp.activations(d_model, 9)
    xd = to_dev(x, dev)
    logits, idx, w = _route(smoe, dev, g, x, n, d_model, k)
    sel = [int(e) for e in idx]
    nb = smoe.smoe_experts_ffn_workspace_bytes(k, d_ff)
    ws = torch.zeros(nb // 4, dtype=torch.int32, device=dev)
    eo = torch.empty((k, d_model), device=dev)
    L = lambda key: [tens[e][key] for e in sel]
    smoe.smoe_experts_ffn_q4(L("gate_codes"), L("gate_scales"), L("up_codes"), L("up_scales"),
                             L("down_codes"), L("down_scales"), xd, eo, d_model, d_ff, group, ws, nb)
    out = torch.empty(d_model, device=dev)
    smoe.smoe_combine(k, eo, to_dev(w, dev), out, d_model)
    torch.cuda.synchronize()
    ys, mags = [], []
    for e in sel:
        ex = experts[e]
        _, y, a = oracle.ffn(4, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
                             ex["down_codes"], ex["down_scales"], d_model, d_ff, group, x.astype(np.float64))
        ys.append(y)
        mags.append(a)
    ref, _ = oracle.combine(np.array(ys), w.astype(np.float64))
    # each expert output is within 1e-4 of its own sum |w x| (+1e-6); the
    # combine adds at most w_r times that per expert, plus its own rounding
    bound = sum(wr * (1e-4 * m + 1e-6) for wr, m in zip(w.astype(np.float64), mags)) + 1e-6
    got = out.cpu().numpy()
    assert (np.abs(got - ref) <= bound).all(), float(np.max(np.abs(got - ref) / bound))
