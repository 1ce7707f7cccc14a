"""Parity of the multi-expert token batch (smoe_experts_ffn_batch_q4/q2)
with the f64 oracle, through the C ABI.

Every expert with routed tokens gets its own token matrix; the call runs
all of them in one launch set (per 32 experts) when the shape takes the
tensor cores, else expert after expert.  Each expert's Y is checked
against the oracle's FFN of that expert over its own tokens.
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


def _run(smoe, dev, bits, Ts, d_model, d_ff, group, seed):
    n = len(Ts)
    experts = [inp.expert(bits, d_model, d_ff, group, seed, e) for e in range(n)]
    Xs = [inp.activations((max(T, 1), d_model), seed + 10 * e)[:T] for e, T in enumerate(Ts)]
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in experts]
    Xd = [to_dev(X, dev) if T else None for X, T in zip(Xs, Ts)]
    Yd = [torch.full((max(T, 1), d_model), float("nan"), device=dev) for T in Ts]
    need = smoe.smoe_experts_ffn_batch_workspace_bytes(Ts, d_model, d_ff, group)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    fn = smoe.smoe_experts_ffn_batch_q4 if bits == 4 else smoe.smoe_experts_ffn_batch_q2
    fn([t["gate_codes"] for t in tens], [t["gate_scales"] for t in tens], [t["up_codes"] for t in tens],
       [t["up_scales"] for t in tens], [t["down_codes"] for t in tens], [t["down_scales"] for t in tens],
       Xd, Yd, Ts, d_model, d_ff, group, ws, need)
    torch.cuda.synchronize()
    assert smoe.smoe_last_device_status() == 0
    return experts, Xs, [Y.cpu().numpy() for Y in Yd]


def _check_expert(bits, ex, X, Y, T, d_model, d_ff, group, tag, sample=None):
    if T == 0:
        assert np.isnan(Y).all(), f"{tag}: an expert without tokens was written"
        return
    args = (bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
            ex["down_codes"], ex["down_scales"])
    toks = range(T) if sample is None or T <= sample else sorted(set(
        [0, T - 1] + list(np.random.default_rng(T).integers(0, T, sample))))
    for tok in toks:
        _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64), tok, 1)
        check(Y[tok], ref[0], a[0], f"{tag} token {tok}")


@pytest.mark.parametrize("bits,Ts", [
    (4, [1, 16, 0, 37, 130, 2, 64, 5]),   # ragged counts, an empty expert, one over a 128-token tile
    (2, [3, 0, 20]),
])
def test_experts_batch_ragged(smoe, dev, bits, Ts):
    d_model, d_ff, group = 4096, 1536, 64
    experts, Xs, Ys = _run(smoe, dev, bits, Ts, d_model, d_ff, group, 50 + bits)
    for e, T in enumerate(Ts):
        _check_expert(bits, experts[e], Xs[e], Ys[e][:T] if T else Ys[e], T, d_model, d_ff, group,
                      f"Q{bits} expert {e} T={T}", sample=4)


def test_experts_batch_35_experts_two_launch_sets(smoe, dev):
    """More than 32 experts: two groups of launches over one workspace."""
    d_model, d_ff, group = 512, 256, 64
    Ts = [1 + (7 * e) % 11 for e in range(35)]
    experts, Xs, Ys = _run(smoe, dev, 4, Ts, d_model, d_ff, group, 60)
    for e in (0, 17, 31, 32, 34):
        _check_expert(4, experts[e], Xs[e], Ys[e][:Ts[e]], Ts[e], d_model, d_ff, group, f"expert {e}")


def test_experts_batch_small_shape_falls_back(smoe, dev):
    """A shape off the tensor-core grid (160 / 96, groups of 32): expert by expert."""
    d_model, d_ff, group = 160, 96, 32
    Ts = [4, 1, 9]
    experts, Xs, Ys = _run(smoe, dev, 4, Ts, d_model, d_ff, group, 61)
    for e, T in enumerate(Ts):
        _check_expert(4, experts[e], Xs[e], Ys[e][:T], T, d_model, d_ff, group, f"expert {e}")


def test_experts_batch_matches_single_expert_calls(smoe, dev):
    """An expert computed in a shared grid and the same expert through the
    single-expert call: both held to the oracle tolerance (the K splits of
    the two grids may differ, so the partial sums can be grouped
    differently)."""
    d_model, d_ff, group = 4096, 1536, 64
    Ts = [16, 16, 16]
    experts, Xs, Ys = _run(smoe, dev, 4, Ts, d_model, d_ff, group, 62)
    t = {k: to_dev(v, dev) for k, v in experts[1].items()}
    Y1 = torch.full((16, d_model), float("nan"), device=dev)
    need = smoe.smoe_ffn_batch_workspace_bytes(16, d_model, d_ff, group)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    smoe.ffn_batch_q4(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], t["down_codes"],
                      t["down_scales"], to_dev(Xs[1], dev), Y1, 16, d_model, d_ff, group, ws, need)
    torch.cuda.synchronize()
    _check_expert(4, experts[1], Xs[1], Y1.cpu().numpy(), 16, d_model, d_ff, group, "single call", sample=4)
    _check_expert(4, experts[1], Xs[1], Ys[1][:16], 16, d_model, d_ff, group, "grouped call", sample=4)


@pytest.mark.parametrize("bits,d_model,d_ff,Ts", [
    (4, 4096, 1536, [16] * 7 + [9]),            # 192 gate/up and 256 down tiles
    (2, 4096, 1536, [16] * 7 + [9]),
    (4, 2048, 2048, [16] * 5 + [12]),           # 192 gate/up tiles, 96 down tiles
])
def test_experts_batch_more_tiles_than_sms(smoe, dev, bits, d_model, d_ff, Ts):
    """16-token tiles outnumbering the SMs: those kernels run two CTAs per SM
    on half the tensor memory each (the last case only for gate/up, so the
    two layouts follow each other)."""
    group = 64
    experts, Xs, Ys = _run(smoe, dev, bits, Ts, d_model, d_ff, group, 70 + bits)
    for e, T in enumerate(Ts):
        _check_expert(bits, experts[e], Xs[e], Ys[e][:T], T, d_model, d_ff, group,
                      f"Q{bits} expert {e} T={T}", sample=3)
