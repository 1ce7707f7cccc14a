"""Wide-dynamic-range parity of every decode entry point with the f64 oracle.

The tolerance |gpu - oracle| <= 1e-4 * sum|w_i x_i| + 1e-6 is relative to
the dot's own absolute sum, so it must hold when x spans many orders of
magnitude inside one group: a large entry over a weight next to the zero
point (|w| = s/15 for Q4, s/3 for Q2) and many tiny entries under extreme
weights, all of whose rounding errors point the same way
(smoe_inputs.wide_range_x / aligned_codes).  The tiny entries sit just under
half a rounding step (or a full step) at several resolutions, so that a
kernel which rounded x on a grid coarser than about 2^-20 of the block
maximum, or rounded some columns more coarsely than others, fails here.
Also: tokens with outlier channels (x1000) and vectors that are mostly
near zero.

Entries covered: the single-expert gate/up (rows split over warp classes)
and down calls, the grouped 8-expert calls, rows too long for register
digits (shared-memory digits), rows that are not a multiple of 8 chunks
(the f32 kernels), the one-launch FFN, and the token batch on the tensor
cores and on the CUDA cores.
"""
import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, hidden_bound_absdot, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# small-entry multipliers: just under a step at 2^-18 and half a step at
# 2^-21 / 2^-22, one and a half steps at 2^-22; None mixes all of them
RELS = [0.999 * 2.0 ** -18, 0.49999 * 2.0 ** -21, 0.49999 * 2.0 ** -22, 1.49999 * 2.0 ** -22, None]
KINDS = [("blocks", r) for r in RELS] + [("outliers", None), ("near_zero", None)]
KIND_IDS = ["rel18", "rel21", "rel22", "rel22x3", "mixed", "outliers", "near_zero"]


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


def _x(n, seed, kind, rel, tid=inp.X_ID + 1):
    return inp.wide_range_x(n, seed, kind, tid=tid, rel=rel)


def _expert(bits, d_model, d_ff, group, x, seed, e=0):
    ex, _ = inp.wide_range_expert(bits, d_model, d_ff, group, x, seed, e)
    return ex


def _check_hidden(bits, ex, x, hidden, d_ff, d_model, group, tag):
    r = oracle.gate_up(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
                       d_ff, d_model, group, x.astype(np.float64))
    return check(hidden, r["hidden"], hidden_bound_absdot(r), tag)


def _check_down(bits, codes, scales, h, out, rows, cols, group, tag):
    y, a = oracle.qgemv(bits, codes, scales, rows, cols, group, np.asarray(h, dtype=np.float64))
    return check(out, y, a, tag)


def _gate_up(smoe, bits):
    return smoe.smoe_gate_up_q4 if bits == 4 else smoe.smoe_gate_up_q2


def _down(smoe, bits):
    return smoe.smoe_down_q4 if bits == 4 else smoe.smoe_down_q2


def _single(smoe, dev, bits, d_model, d_ff, group, kind, rel, seed, tag):
    """gate/up on a wide-range token, down on a wide-range hidden vector."""
    x = _x(d_model, seed, kind, rel)
    h_in = _x(d_ff, seed + 1000, kind, rel)
    ex = _expert(bits, d_model, d_ff, group, x, seed)
    # down codes aligned against the vector it is given
    ex["down_codes"] = inp.pack_codes(inp.aligned_codes(d_model, d_ff, bits, h_in, seed, 77), bits)
    t = {k: to_dev(v, dev) for k, v in ex.items()}
    hidden = torch.full((d_ff,), float("nan"), device=dev)
    out = torch.full((d_model,), float("nan"), device=dev)
    _gate_up(smoe, bits)(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], to_dev(x, dev),
                         hidden, d_ff, d_model, group)
    _down(smoe, bits)(t["down_codes"], t["down_scales"], to_dev(h_in, dev), out, d_model, d_ff, group)
    torch.cuda.synchronize()
    w1 = _check_hidden(bits, ex, x, hidden.cpu().numpy(), d_ff, d_model, group, f"{tag} hidden")
    w2 = _check_down(bits, ex["down_codes"], ex["down_scales"], h_in, out.cpu().numpy(), d_model, d_ff, group,
                     f"{tag} out")
    return max(w1, w2)


@pytest.mark.parametrize("kind,rel", KINDS, ids=KIND_IDS)
@pytest.mark.parametrize("bits", [4, 2])
def test_single_expert_4096_1536(smoe, dev, bits, kind, rel):
    """One expert over every SM: gate/up splits rows over warp classes;
    down is the register-digit kernel (Q4) or the shared-memory one (Q2)."""
    _single(smoe, dev, bits, 4096, 1536, 64, kind, rel, 11, f"single Q{bits} {kind}")


@pytest.mark.parametrize("bits,d_model,d_ff,group", [
    (4, 8192, 256, 64),   # rows of 256 chunks: shared-memory digits
    (2, 8192, 512, 128),
    (4, 160, 96, 32),     # 5 / 3 chunks per row: the f32 kernels
    (2, 256, 192, 64),    # 4 / 3 chunks per row
    (4, 256, 256, 64),    # the small workload's shape
])
@pytest.mark.parametrize("kind,rel", [KINDS[0], KINDS[2], KINDS[4], KINDS[5]],
                         ids=["rel18", "rel22", "mixed", "outliers"])
def test_other_shapes(smoe, dev, bits, d_model, d_ff, group, kind, rel):
    _single(smoe, dev, bits, d_model, d_ff, group, kind, rel, 12, f"Q{bits} {d_model}/{d_ff} {kind}")


@pytest.mark.parametrize("kind,rel", [KINDS[0], KINDS[1], KINDS[2], KINDS[5], KINDS[6]],
                         ids=["rel18", "rel21", "rel22", "outliers", "near_zero"])
@pytest.mark.parametrize("bits", [4, 2])
def test_grouped_8_experts(smoe, dev, bits, kind, rel):
    """The grouped calls: one launch for 8 gate/ups, one for 8 downs, each
    down fed its own wide-range vector."""
    d_model, d_ff, group, n = 4096, 1536, 64, 8
    x = _x(d_model, 21, kind, rel)
    exs, hs = [], []
    for e in range(n):
        ex, _ = inp.wide_range_expert(bits, d_model, d_ff, group, x, 21, e)
        h = _x(d_ff, 300 + e, kind, rel)
        ex["down_codes"] = inp.pack_codes(inp.aligned_codes(d_model, d_ff, bits, h, 21, 90 + e), bits)
        exs.append(ex)
        hs.append(h)
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in exs]
    hidden = torch.full((n, d_ff), float("nan"), device=dev)
    out = torch.full((n, d_model), float("nan"), device=dev)
    gu = smoe.smoe_experts_gate_up_q4 if bits == 4 else smoe.smoe_experts_gate_up_q2
    dn = smoe.smoe_experts_down_q4 if bits == 4 else smoe.smoe_experts_down_q2
    gu([t["gate_codes"] for t in tens], [t["gate_scales"] for t in tens], [t["up_codes"] for t in tens],
       [t["up_scales"] for t in tens], to_dev(x, dev), hidden, d_ff, d_model, group)
    dn([t["down_codes"] for t in tens], [t["down_scales"] for t in tens], to_dev(np.stack(hs), dev), out,
       d_model, d_ff, group)
    torch.cuda.synchronize()
    h, o = hidden.cpu().numpy(), out.cpu().numpy()
    for e in (0, 3, 7):
        _check_hidden(bits, exs[e], x, h[e], d_ff, d_model, group, f"grouped Q{bits} {kind} hidden {e}")
        _check_down(bits, exs[e]["down_codes"], exs[e]["down_scales"], hs[e], o[e], d_model, d_ff, group,
                    f"grouped Q{bits} {kind} out {e}")


@pytest.mark.parametrize("kind,rel", [KINDS[0], KINDS[2], KINDS[5]], ids=["rel18", "rel22", "outliers"])
@pytest.mark.parametrize("bits", [4, 2])
def test_one_launch_ffn(smoe, dev, bits, kind, rel):
    """smoe_experts_ffn_q4/q2: gate/up on a wide-range token, then down on
    the hidden vectors the launch itself produced."""
    d_model, d_ff, group, n = 4096, 1536, 64, 4
    x = _x(d_model, 31, kind, rel)
    exs = [inp.wide_range_expert(bits, d_model, d_ff, group, x, 31, e)[0] for e in range(n)]
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in exs]
    need = smoe.smoe_experts_ffn_workspace_bytes(n, d_ff)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    out = torch.full((n, d_model), float("nan"), device=dev)
    fn = smoe.smoe_experts_ffn_q4 if bits == 4 else smoe.smoe_experts_ffn_q2
    fn(*([t[k] for t in tens] for k in ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes",
                                        "down_scales")), to_dev(x, dev), out, d_model, d_ff, group, ws, need)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    for e in (0, n - 1):
        ex = exs[e]
        _, y, a = oracle.ffn(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
                             ex["down_codes"], ex["down_scales"], d_model, d_ff, group, x.astype(np.float64))
        # out's bound: the oracle's sum |w h| plus the propagated error of
        # hidden (each hidden element within its own bound, times |w|)
        r = oracle.gate_up(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"], d_ff,
                           d_model, group, x.astype(np.float64))
        hb = 1e-4 * hidden_bound_absdot(r) + 1e-6
        wabs = _abs_down(bits, ex, d_model, d_ff, group, hb)
        err = np.abs(o[e].astype(np.float64) - y)
        bound = 1e-4 * a + 1e-6 + wabs
        assert np.isfinite(o[e]).all()
        i = int(np.argmax(err / bound))
        assert err[i] <= bound[i], f"one-launch Q{bits} {kind} expert {e} row {i}: {err[i]:.3g} > {bound[i]:.3g}"


def _abs_down(bits, ex, d_model, d_ff, group, v):
    """sum_k |w_jk| v_k for every row j of down (v >= 0): the oracle's
    sum |w x| with x = v, since every v_k is non-negative."""
    _, a = oracle.qgemv(bits, ex["down_codes"], ex["down_scales"], d_model, d_ff, group, v)
    return a


@pytest.mark.parametrize("bits,d_model,d_ff,group,T", [
    (4, 4096, 1536, 64, 4),   # tensor cores
    (2, 4096, 1536, 64, 3),
    (4, 160, 96, 32, 3),      # CUDA-core multi-token kernel
    (2, 256, 192, 64, 2),
])
def test_token_batch(smoe, dev, bits, d_model, d_ff, group, T):
    """Every token row wide-range (one kind per row); Y within the bound
    of the oracle's batch, with hidden's propagated error added for Y."""
    kinds = [KINDS[0], KINDS[2], KINDS[5], KINDS[6]]
    X = np.stack([_x(d_model, 41 + t, *kinds[t % len(kinds)]) for t in range(T)])
    ex = inp.wide_range_expert(bits, d_model, d_ff, group, X[0], 41)[0]
    t = {k: to_dev(v, dev) for k, v in ex.items()}
    need = smoe.smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    Y = torch.full((T, d_model), float("nan"), device=dev)
    fn = smoe.ffn_batch_q4 if bits == 4 else smoe.ffn_batch_q2
    fn(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], t["down_codes"], t["down_scales"],
       to_dev(X, dev), Y, T, d_model, d_ff, group, ws, need)
    torch.cuda.synchronize()
    got = Y.cpu().numpy().astype(np.float64)
    for i in range(T):
        xi = X[i].astype(np.float64)
        _, y, a = oracle.ffn(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"],
                             ex["down_codes"], ex["down_scales"], d_model, d_ff, group, xi)
        r = oracle.gate_up(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"], d_ff,
                           d_model, group, xi)
        hb = 1e-4 * hidden_bound_absdot(r) + 1e-6
        bound = 1e-4 * a + 1e-6 + _abs_down(bits, ex, d_model, d_ff, group, hb)
        err = np.abs(got[i] - y)
        assert np.isfinite(got[i]).all()
        j = int(np.argmax(err / bound))
        assert err[j] <= bound[j], f"batch Q{bits} T={T} token {i} row {j}: {err[j]:.3g} > {bound[j]:.3g}"
