"""Device-side failure detection without a fault: a bounded wait that can
never succeed gives up, the host reads SMOE_ERR_TIMEOUT from the status
word, and the context still runs a kernel correctly afterwards."""
import time

import numpy as np
import pytest

import oracle
import smoe_inputs as inp
from tests.gpu_util import check, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def smoe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build_library()
    torch.cuda.set_device(torch.device("cuda:0"))
    import moe_expert_ffn_smoe_gb300 as m
    return m


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "device_counter"])
def test_wait_gives_up_and_the_context_stays_usable(smoe, kind):
    dev = torch.device("cuda:0")
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK
    t0 = time.monotonic()
    smoe.smoe_selftest_bounded_wait(kind)
    status = smoe.smoe_last_device_status()
    waited = time.monotonic() - t0
    assert status == smoe.SMOE_ERR_TIMEOUT
    assert waited < 60.0
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK  # read and cleared

    # the context is intact: a bf16 matvec still matches the oracle
    rows, cols = 96, 512
    w = inp.bf16_rows(rows, cols, 3, 1)
    x = inp.activations(cols, 3)
    y = torch.full((rows,), float("nan"), device=dev)
    smoe.matvec_bf16(to_dev(w, dev), to_dev(x, dev), y, rows, cols)
    torch.cuda.synchronize()
    ref, a = oracle.matvec_bf16(w, rows, cols, x.astype(np.float64))
    check(y.cpu().numpy(), ref, a, "matvec after a timed-out wait")
    assert smoe.smoe_last_device_status() == smoe.SMOE_OK


def test_selftest_refuses_an_unknown_kind(smoe):
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_selftest_bounded_wait(2)
    assert e.value.status == smoe.SMOE_ERR_SHAPE
