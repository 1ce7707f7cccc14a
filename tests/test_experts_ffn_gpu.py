"""Parity of the one-launch routed-expert FFN (smoe_experts_ffn_q4/q2)
with the f64 oracle, through the C ABI.

The call computes hidden_e = SiLU(gate_e x) * (up_e x) and
out_e = down_e hidden_e for every expert in one launch (per 64 experts);
shapes the one-launch kernel does not take run as the two grouped calls.
The one-launch result and the grouped two-call result are both held to the
oracle tolerance (they may sum a row's parts in different orders: the
grouped gate/up splits rows over more warps when a CTA has few of them),
repeated calls must reproduce their own result bit for bit, and the
hand-off counters must be zero again after every call.
"""
import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, hidden_bound_absdot, to_dev

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


SYNC_WORDS = 128  # SMOE_FFN_SYNC_BYTES / 4


def _workspace(smoe, dev, n, d_ff):
    nb = smoe.smoe_experts_ffn_workspace_bytes(n, d_ff)
    assert nb % 256 == 0 and nb >= smoe.SMOE_FFN_SYNC_BYTES + min(n, 64) * d_ff * 4
    return torch.zeros(nb // 4, dtype=torch.int32, device=dev), nb


def _hidden(ws, n, d_ff):
    return ws.view(torch.float32)[SYNC_WORDS:SYNC_WORDS + n * d_ff].view(n, d_ff)


def _call(smoe, bits, tens, xd, out, d_model, d_ff, group, ws, nb, stream=None):
    fn = smoe.smoe_experts_ffn_q4 if bits == 4 else smoe.smoe_experts_ffn_q2
    fn([t["gate_codes"] for t in tens], [t["gate_scales"] for t in tens], [t["up_codes"] for t in tens],
       [t["up_scales"] for t in tens], [t["down_codes"] for t in tens], [t["down_scales"] for t in tens],
       xd, out, d_model, d_ff, group, ws, nb, stream=stream)


def _grouped(smoe, bits, tens, xd, d_model, d_ff, group, dev):
    gu, dn = ((smoe.smoe_experts_gate_up_q4, smoe.smoe_experts_down_q4) if bits == 4 else
              (smoe.smoe_experts_gate_up_q2, smoe.smoe_experts_down_q2))
    n = len(tens)
    hidden = torch.full((n, d_ff), float("nan"), device=dev)
    out = torch.full((n, d_model), float("nan"), device=dev)
    gu([t["gate_codes"] for t in tens], [t["gate_scales"] for t in tens], [t["up_codes"] for t in tens],
       [t["up_scales"] for t in tens], xd, hidden, d_ff, d_model, group)
    dn([t["down_codes"] for t in tens], [t["down_scales"] for t in tens], hidden, out, d_model, d_ff, group)
    return hidden, out


def _check_against_oracle(bits, ex, x, hiddens, outs, d_model, d_ff, group, tag):
    """hiddens / outs: lists of (result, label) for this expert."""
    r = oracle.gate_up(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
                       d_ff, d_model, group, x.astype(np.float64))
    for h, lab in hiddens:
        check(h, r["hidden"], hidden_bound_absdot(r), f"{tag} {lab} hidden")
    y, a = oracle.qgemv(bits, ex["down_codes"], ex["down_scales"], d_model, d_ff, group, r["hidden"])
    for o, lab in outs:
        check(o, y, a, f"{tag} {lab} out")


def _setup(bits, n, d_model, d_ff, group, seed, dev):
    experts = [inp.expert(bits, d_model, d_ff, group, seed, e) for e in range(n)]
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in experts]
    x = inp.activations(d_model, seed)
    return experts, tens, x, to_dev(x, dev)


@pytest.mark.parametrize("bits,seed", [(4, 5), (2, 6)])
def test_experts_ffn_8_expert_decode(smoe, dev, bits, seed):
    d_model, d_ff, group, n = 4096, 1536, 64, 8
    experts, tens, x, xd = _setup(bits, n, d_model, d_ff, group, seed, dev)
    ws, nb = _workspace(smoe, dev, n, d_ff)
    out = torch.full((n, d_model), float("nan"), device=dev)
    _call(smoe, bits, tens, xd, out, d_model, d_ff, group, ws, nb)
    torch.cuda.synchronize()
    assert smoe.smoe_last_device_status() == 0
    assert int(ws[:SYNC_WORDS].abs().sum()) == 0, "hand-off counters not reset"
    h, o = _hidden(ws, n, d_ff).cpu().numpy(), out.cpu().numpy()
    gh, go = _grouped(smoe, bits, tens, xd, d_model, d_ff, group, dev)
    torch.cuda.synchronize()
    gh, go = gh.cpu().numpy(), go.cpu().numpy()
    for i, ex in enumerate(experts):
        _check_against_oracle(bits, ex, x, [(h[i], "one call"), (gh[i], "grouped")],
                              [(o[i], "one call"), (go[i], "grouped")], d_model, d_ff, group,
                              f"ffn Q{bits} expert {i}")


def test_experts_ffn_repeated_calls_and_graph(smoe, dev):
    """Back-to-back calls on one workspace (the counters must come back to
    zero every time) and the same calls captured in a CUDA graph."""
    d_model, d_ff, group, n = 4096, 1536, 64, 8
    _, tens, _, xd = _setup(4, n, d_model, d_ff, group, 5, dev)
    ws, nb = _workspace(smoe, dev, n, d_ff)
    ref = torch.empty((n, d_model), device=dev)
    _call(smoe, 4, tens, xd, ref, d_model, d_ff, group, ws, nb)
    outs = [torch.full((n, d_model), float("nan"), device=dev) for _ in range(4)]
    for o in outs:
        _call(smoe, 4, tens, xd, o, d_model, d_ff, group, ws, nb)
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, ref)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    gouts = [torch.full((n, d_model), float("nan"), device=dev) for _ in range(3)]
    with torch.cuda.graph(g, stream=s):
        for o in gouts:
            _call(smoe, 4, tens, xd, o, d_model, d_ff, group, ws, nb, stream=s)
    for _ in range(3):
        for o in gouts:
            o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for o in gouts:
            assert torch.equal(o, ref)
    assert int(ws[:SYNC_WORDS].abs().sum()) == 0
    assert smoe.smoe_last_device_status() == 0


@pytest.mark.parametrize("bits,n,d_model,d_ff,group", [
    (4, 5, 4096, 1536, 64),    # 30 CTAs per expert: ragged row ranges
    (4, 1, 4096, 1536, 64),    # one expert over every SM
    (2, 2, 4096, 4096, 64),    # Q2 through the one-launch kernel
    (4, 3, 3072, 2048, 64),    # 3 and 2 chunks per lane
    (4, 70, 2048, 2048, 64),   # two launches: 64 experts, then 6
    (4, 3, 256, 512, 64),      # shapes the one-launch kernel does not take
    (4, 2, 160, 96, 32),
    (2, 4, 512, 256, 64),
])
def test_experts_ffn_shapes(smoe, dev, bits, n, d_model, d_ff, group):
    experts, tens, x, xd = _setup(bits, n, d_model, d_ff, group, 80 + n, dev)
    ws, nb = _workspace(smoe, dev, n, d_ff)
    out = torch.full((n, d_model), float("nan"), device=dev)
    _call(smoe, bits, tens, xd, out, d_model, d_ff, group, ws, nb)
    torch.cuda.synchronize()
    assert smoe.smoe_last_device_status() == 0
    assert int(ws[:SYNC_WORDS].abs().sum()) == 0
    o = out.cpu().numpy()
    _, go = _grouped(smoe, bits, tens, xd, d_model, d_ff, group, dev)
    torch.cuda.synchronize()
    go = go.cpu().numpy()
    for i in sorted({0, n // 2, n - 1}):
        _check_against_oracle(bits, experts[i], x, [], [(o[i], "one call"), (go[i], "grouped")], d_model, d_ff,
                              group, f"ffn n={n} expert {i}")


def test_experts_ffn_empty_hidden_writes_zeros(smoe, dev):
    d_model, d_ff, group, n = 256, 0, 64, 2
    _, tens, _, xd = _setup(4, n, d_model, 64, group, 90, dev)
    ws, nb = _workspace(smoe, dev, n, d_ff)
    ws = torch.zeros(64, dtype=torch.int32, device=dev) if nb == 0 else ws
    out = torch.full((n, d_model), float("nan"), device=dev)
    _call(smoe, 4, tens, xd, out, d_model, d_ff, group, ws, max(nb, 256))
    torch.cuda.synchronize()
    assert torch.equal(out, torch.zeros_like(out))


def test_experts_ffn_nan_token_gives_nan(smoe, dev):
    d_model, d_ff, group, n = 4096, 1536, 64, 2
    _, tens, x, _ = _setup(4, n, d_model, d_ff, group, 91, dev)
    x[5] = np.nan
    ws, nb = _workspace(smoe, dev, n, d_ff)
    out = torch.zeros((n, d_model), device=dev)
    _call(smoe, 4, tens, to_dev(x, dev), out, d_model, d_ff, group, ws, nb)
    torch.cuda.synchronize()
    assert np.isnan(out.cpu().numpy()).all()
    assert int(ws[:SYNC_WORDS].abs().sum()) == 0
