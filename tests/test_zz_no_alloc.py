"""ffn_batch_q4_noalloc: the token-batch FFN for callers that must not
allocate device memory (a host program that owns all device memory through
its own pools, a plugin inside such a program, or a caller that cannot
afford cudaMalloc's device-wide synchronisation).  Its workspace is a
static device array inside the library instead of a caller buffer.

The test calls it through the C ABI twice in a row, with different inputs,
and checks each result against the ordinary ffn_batch_q4 (which takes a
caller workspace) within the tolerance of the other parity tests,
1e-4 * sum|w x| + 1e-6 per element (sum|w x| from the oracle).  This file
is collected last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    import moe_expert_ffn_smoe_gb300 as smoe

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    d_model, d_ff, group, T = 4096, 1536, 64, 16
    e = inp.expert(4, d_model, d_ff, group, seed=50)
    t = {k: to_dev(v, dev) for k, v in e.items()}
    w = (t["gate_codes"], t["gate_scales"], t["up_codes"], t["up_scales"], t["down_codes"],
         t["down_scales"])
    need = smoe.smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group)
    assert 0 < need <= smoe.SMOE_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    args = (4, e["gate_codes"], e["gate_scales"], e["up_codes"], e["up_scales"], e["down_codes"],
            e["down_scales"])

    for seed in (51, 52):
        X = inp.activations((T, d_model), seed)
        Xd = to_dev(X, dev)
        Y_ws = torch.full((T, d_model), float("nan"), device=dev)
        Y_na = torch.full((T, d_model), float("nan"), device=dev)
        smoe.ffn_batch_q4(*w, Xd, Y_ws, T, d_model, d_ff, group, ws, need)
        smoe.ffn_batch_q4_noalloc(*w, Xd, Y_na, T, d_model, d_ff, group)
        torch.cuda.synchronize()
        _, ref, absdot = oracle.ffn_batch(*args, T, d_model, d_ff, group, X.astype(np.float64))
        check(Y_na.cpu().numpy(), Y_ws.cpu().numpy().astype(np.float64), absdot,
              f"noalloc vs workspace entry point, seed {seed}")
        check(Y_na.cpu().numpy(), ref, absdot, f"noalloc vs oracle, seed {seed}")

    # a batch whose hidden activations exceed the static array is refused
    # before anything is launched
    T_big = smoe.SMOE_NOALLOC_SCRATCH_BYTES // (4 * d_ff) + 1
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.ffn_batch_q4_noalloc(*w, 1 << 20, 2 << 20, T_big, d_model, d_ff, group)
    assert ei.value.status == smoe.SMOE_ERR_SHAPE
