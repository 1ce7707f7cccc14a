"""Parity of the CUDA path (through the C ABI) with the f64 oracle.

Every input is seeded and synthetic (smoe_inputs).  Floating-point outputs
must satisfy |gpu - oracle| <= 1e-4 * sum|w x| + 1e-6 per element; integer
unpacking is checked bit-exactly through one-hot probes.
"""
import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, hidden_bound_absdot, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Z = {4: 7.5, 2: 1.5}


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


def _fns(smoe, bits):
    return ((smoe.smoe_gate_up_q4, smoe.smoe_down_q4) if bits == 4 else
            (smoe.smoe_gate_up_q2, smoe.smoe_down_q2))


def _run_expert(smoe, dev, bits, e, x, d_model, d_ff, group):
    gate_up, down = _fns(smoe, bits)
    t = {k: to_dev(v, dev) for k, v in e.items()}
    xd = to_dev(x, dev)
    hidden = torch.full((d_ff,), float("nan"), device=dev)
    out = torch.full((d_model,), float("nan"), device=dev)
    gate_up(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], xd, hidden, d_ff,
            d_model, group)
    down(t["down_codes"], t["down_scales"], hidden, out, d_model, d_ff, group)
    torch.cuda.synchronize()
    return hidden.cpu().numpy(), out.cpu().numpy(), t


def _check_expert(bits, e, x, hidden, out, d_model, d_ff, group, tag):
    x64 = x.astype(np.float64)
    r = oracle.gate_up(bits, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                       d_ff, d_model, group, x64)
    w1 = check(hidden, r["hidden"], hidden_bound_absdot(r), f"{tag} hidden")
    y, a = oracle.qgemv(bits, e["down_codes"], e["down_scales"], d_model, d_ff, group, r["hidden"])
    w2 = check(out, y, a, f"{tag} out")
    return max(w1, w2)


# ---------------------------------------------------------------- one expert

@pytest.mark.parametrize("bits", [4, 2])
def test_ffn_256_full(smoe, dev, bits):
    d_model = d_ff = 256
    e = inp.expert(bits, d_model, d_ff, 64, seed=0)
    x = inp.activations(d_model, 0)
    hidden, out, t = _run_expert(smoe, dev, bits, e, x, d_model, d_ff, 64)
    _check_expert(bits, e, x, hidden, out, d_model, d_ff, 64, f"Q{bits} 256")
    # down alone on the f32-rounded oracle hidden: the tight check of one GEMV
    r = oracle.gate_up(bits, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                       d_ff, d_model, 64, x.astype(np.float64))
    h32 = r["hidden"].astype(np.float32)
    o = torch.empty(d_model, device=dev)
    _fns(smoe, bits)[1](t["down_codes"], t["down_scales"], to_dev(h32, dev), o, d_model, d_ff, 64)
    y, a = oracle.qgemv(bits, e["down_codes"], e["down_scales"], d_model, d_ff, 64,
                        h32.astype(np.float64))
    check(o.cpu().numpy(), y, a, f"Q{bits} down alone")


@pytest.mark.parametrize("bits,seed", [(4, 5), (2, 6)])
def test_8_expert_decode_full(smoe, dev, bits, seed):
    """The 8-expert decode workload at full size: gate/up [1536,4096] and down
    [4096,1536] per expert, one token, per-expert outputs [8,4096]."""
    d_model, d_ff, group = 4096, 1536, 64
    x = inp.activations(d_model, seed)
    xd = to_dev(x, dev)
    gate_up, down = _fns(smoe, bits)
    experts = [inp.expert(bits, d_model, d_ff, group, seed, e) for e in range(8)]
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in experts]
    hidden = torch.full((8, d_ff), float("nan"), device=dev)
    out = torch.full((8, d_model), float("nan"), device=dev)
    for i, t in enumerate(tens):
        gate_up(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], xd, hidden[i],
                d_ff, d_model, group)
        down(t["down_codes"], t["down_scales"], hidden[i], out[i], d_model, d_ff, group)
    torch.cuda.synchronize()
    h, o = hidden.cpu().numpy(), out.cpu().numpy()
    worst = 0.0
    for i, ex in enumerate(experts):
        worst = max(worst, _check_expert(bits, ex, x, h[i], o[i], d_model, d_ff, group,
                                         f"Q{bits} expert {i}"))
    print(f"Q{bits} 8-expert decode: max err/bound {worst:.3g}")


# ------------------------------------------------ bit-exact unpacking probes

def _probe_down_codes(smoe, dev, bits, codes, scales, rows, cols, group, ks):
    """Recovers code[r, k] for every row r and each k in ks from one-hot
    inputs: down(e_k)[r] = s[r, k/group] * (code[r,k]/Z - 1)."""
    down = _fns(smoe, bits)[1]
    cd, sd = to_dev(codes, dev), to_dev(scales, dev)
    got = np.empty((rows, len(ks)), dtype=np.int64)
    hid = torch.zeros(cols, device=dev)
    out = torch.empty((len(ks), rows), device=dev)
    for j, k in enumerate(ks):
        hid.zero_()
        hid[k] = 1.0
        down(cd, sd, hid, out[j], rows, cols, group)
    torch.cuda.synchronize()
    o = out.cpu().numpy().astype(np.float64).T
    s = scales.astype(np.float64)[:, [k // group for k in ks]]
    got[:] = np.rint(Z[bits] * (o / s + 1.0)).astype(np.int64)
    return got


@pytest.mark.parametrize("bits,rows,cols", [(4, 256, 256), (2, 256, 256), (4, 4096, 1536),
                                            (2, 4096, 1536), (4, 64, 4096), (2, 64, 4096)])
def test_unpack_probes_down(smoe, dev, bits, rows, cols):
    group = 64
    codes = inp.packed_codes(rows, cols, bits, 21, 1)
    scales = inp.scales(rows, cols // group, 21, 2)
    if cols <= 256:
        ks = list(range(cols))
    else:
        per = 32 if bits == 4 else 64
        ks = sorted(set([0, 1, 2, 3, per - 1, per, 63, 64, cols - 1, cols - 2]
                        + list(np.random.default_rng(3).integers(0, cols, 40))))
    got = _probe_down_codes(smoe, dev, bits, codes, scales, rows, cols, group, ks)
    want = oracle.unpack(codes, bits, rows * cols).reshape(rows, cols)[:, ks].astype(np.int64)
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"first mismatch (row, k-index) {bad[0]}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


@pytest.mark.parametrize("bits", [4, 2])
def test_unpack_probes_gate_up(smoe, dev, bits):
    """Gate codes and up codes recovered bit-exactly through the fused pass:
    with one matrix at the top code (w = +s) the other is decoded by the
    nearest of its 2^bits candidate hidden values."""
    d_ff, d_model, group = 1536, 4096, 64
    gate_up = _fns(smoe, bits)[0]
    codes = inp.packed_codes(d_ff, d_model, bits, 22, 1)
    sc = inp.scales(d_ff, d_model // group, 22, 2)
    top = np.full_like(codes, 0xFF)
    sc_top = inp.scales(d_ff, d_model // group, 22, 3)
    nvals = 1 << bits
    want = oracle.unpack(codes, bits, d_ff * d_model).reshape(d_ff, d_model)
    ks = [0, 1, 31, 32, 63, 64, 4095] + list(np.random.default_rng(4).integers(0, d_model, 9))
    v = 8.0
    for role in ("gate", "up"):
        if role == "gate":
            args = (codes, sc, top, sc_top)
        else:
            args = (top, sc_top, codes, sc)
        t = [to_dev(a, dev) for a in args]
        hid = torch.empty((len(ks), d_ff), device=dev)
        xd = torch.zeros(d_model, device=dev)
        for j, k in enumerate(ks):
            xd.zero_()
            xd[k] = v
            gate_up(*t, xd, hid[j], d_ff, d_model, group)
        torch.cuda.synchronize()
        h = hid.cpu().numpy().astype(np.float64)
        for j, k in enumerate(ks):
            s_test = sc.astype(np.float64)[:, k // group]
            s_top = sc_top.astype(np.float64)[:, k // group]
            c = np.arange(nvals, dtype=np.float64)
            w_test = s_test[:, None] * (c[None, :] / Z[bits] - 1.0) * v   # [d_ff, nvals]
            w_top = (s_top * v)[:, None]
            if role == "gate":
                cand = w_test / (1.0 + np.exp(-w_test)) * w_top
            else:
                cand = w_top / (1.0 + np.exp(-w_top)) * w_test
            dec = np.argmin(np.abs(cand - h[j][:, None]), axis=1)
            assert (dec == want[:, k]).all(), f"{role} k={k}: {np.count_nonzero(dec != want[:, k])} codes differ"


# ---------------------------------------------------------------- bf16

@pytest.mark.parametrize("rows,cols,seed", [
    (8192, 4096, 1), (4096, 8192, 2), (512, 4096, 3),
    (3, 8, 11),          # one 16-byte chunk per row, fewer rows than SMs
    (200, 32768, 12),    # the widest rows: 8 chunks per thread, x read from shared memory
    (777, 4104, 13),     # a ragged last chunk round (513 chunks per row)
    (100, 12288, 14),    # 3 chunks per thread
    (1024, 8192, 15),    # 2 chunks per thread, fewer rows than 8 per CTA
    (9, 2056, 17),       # a ragged last chunk round with few rows
])
def test_bf16_full(smoe, dev, rows, cols, seed):
    w = inp.bf16_rows(rows, cols, seed, 1)
    x = inp.activations(cols, seed)
    y = torch.full((rows,), float("nan"), device=dev)
    smoe.matvec_bf16(to_dev(w, dev), to_dev(x, dev), y, rows, cols)
    torch.cuda.synchronize()
    ref, a = oracle.matvec_bf16(w, rows, cols, x.astype(np.float64))
    check(y.cpu().numpy(), ref, a, f"bf16 {rows}x{cols}")


def test_bf16_lm_head_sampled_rows(smoe, dev):
    rows, cols, seed = 151936, 4096, 4
    w = inp.bf16_rows(rows, cols, seed, 1)
    x = inp.activations(cols, seed)
    y = torch.full((rows,), float("nan"), device=dev)
    smoe.matvec_bf16(to_dev(w, dev), to_dev(x, dev), y, rows, cols)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    assert np.isfinite(got).all()
    sample = sorted(set([0, 1, rows - 1, rows - 2, 4095, 4096]
                        + list(np.random.default_rng(5).integers(0, rows, 2000))))
    ref = np.empty(len(sample))
    a = np.empty(len(sample))
    for i, r in enumerate(sample):
        ref[i:i + 1], a[i:i + 1] = oracle.matvec_bf16(w, rows, cols, x.astype(np.float64), r, 1)
    check(got[sample], ref, a, "bf16 LM head (sampled rows)")


def test_bf16_single_nonzero_is_exact(smoe, dev):
    rows, cols = 64, 256
    w = np.zeros((rows, cols), np.uint16)
    w[17, 200] = 0x4040   # 3.0
    x = inp.activations(cols, 9)
    y = torch.empty(rows, device=dev)
    smoe.matvec_bf16(to_dev(w, dev), to_dev(x, dev), y, rows, cols)
    torch.cuda.synchronize()
    g = y.cpu().numpy()
    assert g[17] == np.float32(3.0) * x[200] and np.count_nonzero(g) == 1


def _bf16_batch_case(smoe, dev, shapes, seed):
    ws, xs, ys, host = [], [], [], []
    for i, (rows, cols) in enumerate(shapes):
        w = inp.bf16_rows(rows, cols, seed, 1 + i)
        x = inp.activations(cols, seed + 100 * i)
        host.append((w, x))
        ws.append(to_dev(w, dev) if rows * cols else None)
        xs.append(to_dev(x, dev) if cols else None)
        ys.append(torch.full((max(rows, 1),), float("nan"), device=dev))
    smoe.matvec_bf16_batch(ws, xs, ys, [r for r, _ in shapes], [c for _, c in shapes])
    torch.cuda.synchronize()
    for i, ((rows, cols), (w, x)) in enumerate(zip(shapes, host)):
        if rows == 0:
            assert torch.isnan(ys[i]).all(), "an entry with no rows was written"
            continue
        got = ys[i].cpu().numpy()[:rows]
        if cols == 0:
            assert (got == 0).all()
            continue
        ref, a = oracle.matvec_bf16(w, rows, cols, x.astype(np.float64))
        check(got, ref, a, f"bf16 batch entry {i} {rows}x{cols}")


@pytest.mark.parametrize("shapes", [
    [(512, 4096)] * 8,                                   # the small-matvec case: one launch
    [(8192, 4096), (3, 8), (777, 4104), (1, 64), (4096, 1536)],  # mixed sizes, one chunk class
    [(100, 12288), (512, 4096), (200, 32768), (64, 2048)],      # three chunk classes: three launches
    [(0, 4096), (16, 0), (37, 520)],                     # an empty entry and a zero-width one
])
def test_bf16_batch(smoe, dev, shapes):
    _bf16_batch_case(smoe, dev, shapes, 21)


def test_bf16_batch_70_entries(smoe, dev):
    """More than 64 entries: two launches of one class."""
    rng = np.random.default_rng(22)
    shapes = [(int(rng.integers(1, 300)), 8 * int(rng.integers(1, 600))) for _ in range(70)]
    _bf16_batch_case(smoe, dev, shapes, 22)


# ---------------------------------------------------------------- token batch

def _batch(smoe, dev, T, e, X, d_model, d_ff, group, bits=4):
    t = {k: to_dev(v, dev) for k, v in e.items()}
    Y = torch.full((max(T, 1), d_model), float("nan"), device=dev)
    need = smoe.smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    fn = smoe.ffn_batch_q4 if bits == 4 else smoe.ffn_batch_q2
    fn(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"],
       t["down_codes"], t["down_scales"], to_dev(X, dev), Y, T, d_model, d_ff, group, ws, need)
    torch.cuda.synchronize()
    return Y.cpu().numpy()[:T]


@pytest.mark.parametrize("T", [1, 3, 16, 32, 64, 100, 200, 256])
def test_token_batch(smoe, dev, T):
    """Token tiles of 16, 32, 64 and 128 tokens; 100 and 200 leave a
    partly padded last tile."""
    d_model, d_ff, group = 4096, 1536, 64
    e = inp.expert(4, d_model, d_ff, group, seed=7)
    X = inp.activations((T, d_model), 7)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group)
    toks = list(range(T)) if T <= 16 else sorted(set([0, 1, T - 1, T // 2] + list(
        np.random.default_rng(T).integers(0, T, 6))))
    args = (4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    for tok in toks:
        _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64), tok, 1)
        check(Y[tok], ref[0], a[0], f"batch T={T} token {tok}")


def test_token_batch_small_shape_all_tokens(smoe, dev):
    d_model, d_ff, group, T = 256, 512, 64, 13
    e = inp.expert(4, d_model, d_ff, group, seed=30)
    X = inp.activations((T, d_model), 30)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group)
    args = (4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64))
    check(Y, ref, a, "batch 256/512 T=13")


@pytest.mark.parametrize("d_model,d_ff,group,T", [
    (320, 192, 64, 20),    # code chunks and the last down row tile run past the matrix
    (512, 256, 128, 70),   # groups of 128 columns: one scale per two K tiles
    (768, 384, 192, 40),   # groups of 192: three K tiles per scale, K splits starting mid-group
    (768, 384, 192, 16),   # the same with 16-token tiles (A in tensor memory)
    (512, 256, 32, 8),     # groups of 32: no tensor-core path, 8 tokens stay on the decode slots
])
def test_token_batch_ragged_shapes(smoe, dev, d_model, d_ff, group, T):
    e = inp.expert(4, d_model, d_ff, group, seed=31)
    X = inp.activations((T, d_model), 31)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group)
    args = (4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64))
    check(Y, ref, a, f"batch {d_model}/{d_ff} g{group} T={T}")


@pytest.mark.parametrize("bits,T", [(4, 2), (4, 5), (4, 6), (4, 7), (4, 8), (2, 4), (2, 6), (2, 7)])
def test_token_batch_slots(smoe, dev, bits, T):
    """2 to 6 tokens run as one decode slot per token (the grouped decode
    kernels sharing the expert's weights); 7 and more go to the tensor cores."""
    d_model, d_ff, group = 4096, 1536, 64
    e = inp.expert(bits, d_model, d_ff, group, 17, 0)
    X = inp.activations((T, d_model), 17)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group, bits=bits)
    _, y_ref, y_abs = oracle.ffn_batch(bits, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                                       e["down_codes"], e["down_scales"], T, d_model, d_ff, group,
                                       X.astype(np.float64))
    check(Y, y_ref, y_abs, f"Q{bits} batch of {T} tokens")


@pytest.mark.parametrize("T", [1, 2, 16, 64, 100, 256])
def test_token_batch_q2(smoe, dev, T):
    """Q2 codes through the same tiles: eight K tiles per code chunk, and the
    Q2 order of columns inside a tile on both operands."""
    d_model, d_ff, group = 4096, 1536, 64
    e = inp.expert(2, d_model, d_ff, group, seed=8)
    X = inp.activations((T, d_model), 8)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group, bits=2)
    toks = list(range(T)) if T <= 16 else sorted(set([0, 1, T - 1, T // 2] + list(
        np.random.default_rng(T).integers(0, T, 6))))
    args = (2, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    for tok in toks:
        _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64), tok, 1)
        check(Y[tok], ref[0], a[0], f"Q2 batch T={T} token {tok}")


@pytest.mark.parametrize("d_model,d_ff,group,T", [
    (320, 192, 64, 20),    # a chunk of 8 K tiles longer than the row: zero fill past the matrix
    (512, 256, 128, 70),   # groups of 128 columns
    (768, 384, 192, 40),   # groups of 192: three K tiles per scale
    (256, 0, 64, 5),       # no hidden columns: Y = 0
])
def test_token_batch_q2_ragged(smoe, dev, d_model, d_ff, group, T):
    e = inp.expert(2, d_model, max(d_ff, 64), group, seed=32)
    if d_ff == 0:
        X = inp.activations((T, d_model), 32)
        Y = _batch(smoe, dev, T, e, X, d_model, 0, group, bits=2)
        assert (Y == 0).all()
        return
    X = inp.activations((T, d_model), 32)
    Y = _batch(smoe, dev, T, e, X, d_model, d_ff, group, bits=2)
    args = (2, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
            e["down_codes"], e["down_scales"])
    _, ref, a = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64))
    check(Y, ref, a, f"Q2 batch {d_model}/{d_ff} g{group} T={T}")


# ------------------------------------------------------ ragged and edge cases

@pytest.mark.parametrize("bits,rows,cols,group", [
    (4, 37, 160, 32),      # 5 chunks per row: generic kernel, odd row count
    (2, 45, 320, 64),      # Q2, 5 chunks per row
    (4, 1, 64, 64),        # one row, one group
    (4, 300, 4096, 4096),  # one group spanning the row
    (4, 129, 8192, 64),    # wide row (generic kernel)
    (2, 77, 1536, 192),    # Q2 down width, group 192
    (4, 1000, 3072, 96),   # 96 chunks: L=32, 3 per lane
    (4, 33, 32768, 64),    # the widest input the ABI accepts
    (2, 17, 32768, 64),
])
def test_ragged_gemv(smoe, dev, bits, rows, cols, group):
    codes = inp.packed_codes(rows, cols, bits, 40, 1)
    sc = inp.scales(rows, cols // group, 40, 2)
    x = inp.activations(cols, 40)
    y = torch.full((rows,), float("nan"), device=dev)
    _fns(smoe, bits)[1](to_dev(codes, dev), to_dev(sc, dev), to_dev(x, dev), y, rows, cols, group)
    torch.cuda.synchronize()
    ref, a = oracle.qgemv(bits, codes, sc, rows, cols, group, x.astype(np.float64))
    check(y.cpu().numpy(), ref, a, f"Q{bits} {rows}x{cols} g{group}")


@pytest.mark.parametrize("bits,d_ff,d_model", [
    (4, 5, 160), (2, 3, 320), (4, 1, 32768),
    # under 24 rows per CTA: rows split in two over 16 warps
    (4, 1000, 4096),   # 2 chunks per lane, ragged rows per CTA
    (4, 2000, 2048),   # 1 chunk per lane
    (2, 1500, 4096),   # Q2, 1 chunk per lane
    (4, 3496, 4096),   # 23 rows per CTA: still split
    (4, 3648, 4096),   # 24 rows per CTA: not split
])
def test_ragged_gate_up(smoe, dev, bits, d_ff, d_model):
    group = 32 if bits == 4 else 64
    e = inp.expert(bits, d_model, d_ff, group, seed=41)
    x = inp.activations(d_model, 41)
    gate_up = _fns(smoe, bits)[0]
    t = {k: to_dev(v, dev) for k, v in e.items()}
    h = torch.full((d_ff,), float("nan"), device=dev)
    gate_up(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], to_dev(x, dev), h,
            d_ff, d_model, group)
    torch.cuda.synchronize()
    r = oracle.gate_up(bits, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"],
                       d_ff, d_model, group, x.astype(np.float64))
    check(h.cpu().numpy(), r["hidden"], hidden_bound_absdot(r), f"gate_up Q{bits} {d_ff}x{d_model}")


def test_zero_columns_write_zeros(smoe, dev):
    out = torch.full((10,), float("nan"), device=dev)
    smoe.smoe_down_q4(None, None, None, out, 10, 0, 64)
    h = torch.full((7,), float("nan"), device=dev)
    smoe.smoe_gate_up_q2(None, None, None, None, None, h, 7, 0, 64)
    y = torch.full((5,), float("nan"), device=dev)
    smoe.matvec_bf16(None, None, y, 5, 0)
    torch.cuda.synchronize()
    assert (out.cpu() == 0).all() and (h.cpu() == 0).all() and (y.cpu() == 0).all()


def test_constant_code_and_zero_input(smoe, dev):
    rows, cols, group = 64, 4096, 64
    sc = inp.scales(rows, cols // group, 42, 2)
    x = inp.activations(cols, 42)
    y = torch.empty(rows, device=dev)
    for code in (0, 7, 8, 15):
        codes = np.full((rows, cols // 2), code | (code << 4), np.uint8)
        smoe.smoe_down_q4(to_dev(codes, dev), to_dev(sc, dev), to_dev(x, dev), y, rows, cols, group)
        torch.cuda.synchronize()
        ref, a = oracle.qgemv(4, codes, sc, rows, cols, group, x.astype(np.float64))
        check(y.cpu().numpy(), ref, a, f"constant code {code}")
    codes = inp.packed_codes(rows, cols, 4, 42, 1)
    smoe.smoe_down_q4(to_dev(codes, dev), to_dev(sc, dev), torch.zeros(cols, device=dev), y, rows,
                      cols, group)
    torch.cuda.synchronize()
    assert (y.cpu() == 0).all()


# ------------------------------------------------ streams and graph capture

def test_graph_capture_of_8_expert_sequence_matches_eager(smoe, dev):
    d_model, d_ff, group = 4096, 1536, 64
    x = to_dev(inp.activations(d_model, 5), dev)
    tens = [{k: to_dev(v, dev) for k, v in inp.expert(4, d_model, d_ff, group, 5, e).items()}
            for e in range(8)]
    hid = torch.empty((8, d_ff), device=dev)
    out = torch.empty((8, d_model), device=dev)

    def step(stream):
        for i, t in enumerate(tens):
            smoe.smoe_gate_up_q4(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], x,
                                 hid[i], d_ff, d_model, group, stream=stream)
            smoe.smoe_down_q4(t["down_codes"], t["down_scales"], hid[i], out[i], d_model, d_ff,
                              group, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    s.synchronize()
    eager = out.clone()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


# ------------------------------------------------------ grouped expert calls

def _grouped(smoe, bits):
    return ((smoe.smoe_experts_gate_up_q4, smoe.smoe_experts_down_q4) if bits == 4 else
            (smoe.smoe_experts_gate_up_q2, smoe.smoe_experts_down_q2))


def _run_grouped(smoe, dev, bits, experts, x, d_model, d_ff, group):
    gu, dn = _grouped(smoe, bits)
    tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in experts]
    n = len(experts)
    hidden = torch.full((n, d_ff), float("nan"), device=dev)
    out = torch.full((n, d_model), float("nan"), device=dev)
    gu([t["gate_codes"] for t in tens], [t["gate_scales"] for t in tens], [t["up_codes"] for t in tens],
       [t["up_scales"] for t in tens], to_dev(x, dev), hidden, d_ff, d_model, group)
    dn([t["down_codes"] for t in tens], [t["down_scales"] for t in tens], hidden, out, d_model, d_ff, group)
    torch.cuda.synchronize()
    return hidden, out, tens


@pytest.mark.parametrize("bits,seed", [(4, 5), (2, 6)])
def test_grouped_8_expert_decode(smoe, dev, bits, seed):
    """One launch for the gate/up of all 8 experts, one for their downs."""
    d_model, d_ff, group = 4096, 1536, 64
    experts = [inp.expert(bits, d_model, d_ff, group, seed, e) for e in range(8)]
    x = inp.activations(d_model, seed)
    hidden, out, tens = _run_grouped(smoe, dev, bits, experts, x, d_model, d_ff, group)
    h, o = hidden.cpu().numpy(), out.cpu().numpy()
    for i, ex in enumerate(experts):
        _check_expert(bits, ex, x, h[i], o[i], d_model, d_ff, group, f"grouped Q{bits} expert {i}")
    # the single-expert calls of the same experts (one expert over every SM:
    # gate/up splits its rows over more warps, so the row parts are summed in
    # another order) are held to the same oracle tolerance
    gate_up, down = _fns(smoe, bits)
    h1 = torch.empty(d_ff, device=dev)
    o1 = torch.empty(d_model, device=dev)
    xd = to_dev(x, dev)
    for i in (0, 7):
        t = tens[i]
        gate_up(t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], xd, h1, d_ff, d_model, group)
        down(t["down_codes"], t["down_scales"], hidden[i], o1, d_model, d_ff, group)
        torch.cuda.synchronize()
        _check_expert(bits, experts[i], x, h1.cpu().numpy(), o1.cpu().numpy(), d_model, d_ff, group,
                      f"single-expert Q{bits} expert {i}")


@pytest.mark.parametrize("bits,n,d_model,d_ff,group", [(4, 3, 256, 512, 64), (2, 5, 512, 256, 64),
                                                      (4, 8, 4096, 128, 64),  # split gate/up, 7 rows per CTA
                                                      (4, 70, 256, 64, 64), (4, 2, 160, 96, 32)])
def test_grouped_ragged(smoe, dev, bits, n, d_model, d_ff, group):
    experts = [inp.expert(bits, d_model, d_ff, group, 60 + n, e) for e in range(n)]
    x = inp.activations(d_model, 60 + n)
    hidden, out, _ = _run_grouped(smoe, dev, bits, experts, x, d_model, d_ff, group)
    h, o = hidden.cpu().numpy(), out.cpu().numpy()
    for i in sorted(set([0, n // 2, n - 1])):
        _check_expert(bits, experts[i], x, h[i], o[i], d_model, d_ff, group, f"grouped n={n} expert {i}")


def test_grouped_zero_experts_is_a_no_op(smoe, dev):
    smoe.smoe_experts_gate_up_q4([], [], [], [], None, None, 1536, 4096, 64)
    smoe.smoe_experts_down_q2([], [], None, None, 4096, 1536, 64)


def test_nan_input_gives_nan_rows(smoe, dev):
    rows, cols, group = 64, 4096, 64
    codes = inp.packed_codes(rows, cols, 4, 43, 1)
    sc = inp.scales(rows, cols // group, 43, 2)
    x = inp.activations(cols, 43)
    x[100] = np.nan
    y = torch.zeros(rows, device=dev)
    smoe.smoe_down_q4(to_dev(codes, dev), to_dev(sc, dev), to_dev(x, dev), y, rows, cols, group)
    torch.cuda.synchronize()
    assert np.isnan(y.cpu().numpy()).all()
