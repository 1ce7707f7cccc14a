"""Device-side routed dispatch (smoe_experts_ffn_routed_q4/q2) through the C ABI.

A whole MoE layer for one token runs on the GPU with no host round trip:
smoe_route_topk_bf16 writes the top-k expert indices and weights, the routed
call reads the indices on the device and runs the selected experts' FFN out
of device tables of expert pointers, and smoe_combine adds the outputs with
the weights (S-MoE "Metal Compute Kernels": "Grouped Expert Dispatch" and the
exact-routing gate matvec of "Batched Scout Matvec").  Checked against the
oracle's route, FFN and combine on the GPU's selection; the layer captured
in one CUDA graph must equal the eager layer and follow a new token's
selection on replay.  Invalid device indices and table entries are caught
on the device (before any load through them) and reported as SMOE_ERR_ROUTE.
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


KEYS = ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes", "down_scales")


class Layer:
    """n experts on the device, their pointer tables, a bf16 router."""

    def __init__(self, smoe, dev, bits, n, d_model, d_ff, group, seed):
        self.smoe, self.dev, self.bits = smoe, dev, bits
        self.n, self.d_model, self.d_ff, self.group = n, d_model, d_ff, group
        self.experts = [inp.expert(bits, d_model, d_ff, group, seed, e) for e in range(n)]
        self.tens = [{k: to_dev(v, dev) for k, v in ex.items()} for ex in self.experts]
        self.tabs = [smoe.pointer_table([t[k] for t in self.tens], dev) for k in KEYS]
        self.gate = inp.bf16_rows(n, d_model, seed, 3)
        self.gate_d = to_dev(self.gate, dev)

    def buffers(self, k):
        d = self.dev
        self.k = k
        self.logits = torch.empty(self.n, device=d)
        self.idx = torch.empty(k, dtype=torch.int32, device=d)
        self.w = torch.empty(k, device=d)
        self.wsb = self.smoe.smoe_experts_ffn_routed_workspace_bytes(k, self.d_ff)
        self.ws = torch.empty(self.wsb, dtype=torch.uint8, device=d)
        self.eo = torch.full((k, self.d_model), float("nan"), device=d)
        self.out = torch.full((self.d_model,), float("nan"), device=d)
        self.x = torch.empty(self.d_model, device=d)

    def routed(self, stream=None):
        f = self.smoe.smoe_experts_ffn_routed_q4 if self.bits == 4 else self.smoe.smoe_experts_ffn_routed_q2
        f(self.n, self.k, *self.tabs, self.idx, self.x, self.eo, self.d_model, self.d_ff, self.group, self.ws,
          self.wsb, stream=stream)

    def layer(self, stream=None):
        s = self.smoe
        s.smoe_route_topk_bf16(self.gate_d, self.x, self.n, self.d_model, self.k, self.logits, self.idx, self.w,
                               stream=stream)
        self.routed(stream)
        s.smoe_combine(self.k, self.eo, self.w, self.out, self.d_model, stream=stream)

    def check(self, x, tag):
        """The GPU's logits within the bound of the oracle's, its selection
        the oracle's selection of those logits, each expert output and the
        combined output within their bounds."""
        torch.cuda.synchronize()
        x64 = x.astype(np.float64)
        l_ref, l_abs, _, _ = oracle.route(self.gate, self.n, self.d_model, x64, self.k)
        gl = self.logits.cpu().numpy().astype(np.float64)
        check(gl, l_ref, l_abs, f"{tag} logits")
        oi, ow = oracle.topk(gl, self.k)
        idx = self.idx.cpu().numpy()
        assert (idx == oi).all(), f"{tag}: selection {idx} vs oracle {oi}"
        w = self.w.cpu().numpy().astype(np.float64)
        eo = self.eo.cpu().numpy()
        ys, mags = [], []
        for r, e in enumerate(idx):
            ex = self.experts[int(e)]
            _, y, a = oracle.ffn(self.bits, *(ex[k] for k in KEYS), self.d_model, self.d_ff, self.group, x64)
            check(eo[r], y, a, f"{tag} expert output {r} (expert {int(e)})")
            ys.append(y)
            mags.append(a)
        ref, _ = oracle.combine(np.array(ys), w)
        bound = sum(wr * (1e-4 * m + 1e-6) for wr, m in zip(w, mags)) + 1e-6
        got = self.out.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) <= bound).all(), f"{tag} combined: {float(np.max(np.abs(got - ref) / bound))}"
        return idx


@pytest.mark.parametrize("bits,n,k", [(4, 16, 8), (2, 16, 8), (4, 24, 1)])
def test_moe_layer_on_device(smoe, dev, bits, n, k):
    """route -> routed FFN -> combine, no host round trip between them; k = 1
    runs one slot over every SM (gate/up rows split over warp classes)."""
    L = Layer(smoe, dev, bits, n, 4096, 1536, 64, 70 + bits)
    L.buffers(k)
    x = inp.activations(4096, 71)
    L.x.copy_(torch.from_numpy(x))
    L.layer()
    L.check(x, f"Q{bits} n={n} k={k}")
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK


def test_layer_in_one_graph_follows_each_token(smoe, dev):
    """The four calls captured in one CUDA graph: a replay equals the eager
    layer bit for bit, and replays on new tokens (copied into the same
    buffer) select other experts and still match the oracle."""
    L = Layer(smoe, dev, 4, 32, 4096, 1536, 64, 80)
    L.buffers(8)
    x0 = inp.activations(4096, 81)
    L.x.copy_(torch.from_numpy(x0))
    L.layer()
    torch.cuda.synchronize()
    eager = L.out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        L.layer(stream=s)  # warm up on the capture stream
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        L.layer(stream=s)
    L.out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(L.out, eager)
    sels = [tuple(L.check(x0, "graph token 0"))]
    for t in (1, 2, 3):
        x = inp.activations(4096, 81 + 10 * t)
        L.x.copy_(torch.from_numpy(x))
        g.replay()
        sels.append(tuple(L.check(x, f"graph token {t}")))
    assert len(set(sels)) > 1, "the replays never changed the selection"


@pytest.mark.parametrize("bits,d_model,d_ff,group", [(4, 8192, 512, 64), (2, 1024, 512, 128), (4, 256, 256, 64)])
def test_routed_other_shapes(smoe, dev, bits, d_model, d_ff, group):
    """Rows of 256 chunks (shared-memory digits), Q2 groups of 128, and the
    small workload's shape, with indices written directly."""
    n, k = 5, 3
    L = Layer(smoe, dev, bits, n, d_model, d_ff, group, 90)
    L.buffers(k)
    x = inp.activations(d_model, 91)
    L.x.copy_(torch.from_numpy(x))
    sel = [4, 0, 4]  # an expert may appear twice
    L.idx.copy_(torch.tensor(sel, dtype=torch.int32))
    L.routed()
    torch.cuda.synchronize()
    eo = L.eo.cpu().numpy()
    for r, e in enumerate(sel):
        ex = L.experts[e]
        r_gu = oracle.gate_up(bits, ex["gate_codes"], ex["gate_scales"], ex["up_codes"], ex["up_scales"], d_ff,
                              d_model, group, x.astype(np.float64))
        y, a = oracle.qgemv(bits, ex["down_codes"], ex["down_scales"], d_model, d_ff, group, r_gu["hidden"])
        check(eo[r], y, a, f"Q{bits} {d_model}/{d_ff} slot {r}")


def test_invalid_device_index_and_table_entry(smoe, dev):
    """An index outside the table, and a table entry that is not 16-byte
    aligned, are caught on the device before any load through them: those
    slots' outputs are NaN, the status is SMOE_ERR_ROUTE, the other slots
    are right and the context stays usable."""
    n, k, d_model, d_ff, group = 4, 3, 1024, 512, 64
    L = Layer(smoe, dev, 4, n, d_model, d_ff, group, 95)
    L.buffers(k)
    x = inp.activations(d_model, 96)
    L.x.copy_(torch.from_numpy(x))
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK
    L.idx.copy_(torch.tensor([2, n, 1], dtype=torch.int32))  # slot 1: one past the table
    L.routed()
    assert smoe.smoe_last_device_status() == smoe.SMOE_ERR_ROUTE
    eo = L.eo.cpu().numpy()
    assert np.isnan(eo[1]).all()
    for r, e in ((0, 2), (2, 1)):
        ex = L.experts[e]
        _, y, a = oracle.ffn(4, *(ex[kk] for kk in KEYS), d_model, d_ff, group, x.astype(np.float64))
        check(eo[r], y, a, f"valid slot {r}")
    L.idx.copy_(torch.tensor([-1, 0, 3], dtype=torch.int32))
    L.routed()
    assert smoe.smoe_last_device_status() == smoe.SMOE_ERR_ROUTE
    assert np.isnan(L.eo.cpu().numpy()[0]).all()
    # a misaligned down-codes entry for expert 3 (the pointer plus 4 bytes)
    L.tabs[4][3] += 4
    L.idx.copy_(torch.tensor([0, 3, 1], dtype=torch.int32))
    L.routed()
    assert smoe.smoe_last_device_status() == smoe.SMOE_ERR_ROUTE
    eo = L.eo.cpu().numpy()
    assert np.isnan(eo[1]).all() and np.isfinite(eo[0]).all() and np.isfinite(eo[2]).all()
    L.tabs[4][3] -= 4
    # the context is still usable
    L.routed()
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK
    assert np.isfinite(L.eo.cpu().numpy()).all()
