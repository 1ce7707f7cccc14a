"""smoe_copy: SM-driven copies between device memory and pinned host
memory, bit for bit, and the refusal of pageable host memory."""
import numpy as np
import pytest

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


def _bits(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 2**31, n, dtype=np.int64).astype(np.int32))


@pytest.mark.parametrize("nbytes", [16, 4096, 16384, 131072, 16 * 100003])
def test_copy_device_and_pinned_host(smoe, nbytes):
    dev = torch.device("cuda:0")
    n = nbytes // 4
    src_host = _bits(n, nbytes).pin_memory()
    mid = torch.full((n,), -1, dtype=torch.int32, device=dev)
    dst_dev = torch.full((n,), -1, dtype=torch.int32, device=dev)
    back = torch.full((n,), -1, dtype=torch.int32).pin_memory()
    smoe.smoe_copy(mid, src_host, nbytes)       # pinned host -> device
    smoe.smoe_copy(dst_dev, mid, nbytes)        # device -> device
    smoe.smoe_copy(back, dst_dev, nbytes)       # device -> pinned host
    torch.cuda.synchronize()
    assert torch.equal(back, src_host)
    assert torch.equal(dst_dev.cpu(), src_host)


def test_copy_refuses_pageable_host_memory(smoe):
    dev = torch.device("cuda:0")
    pageable = torch.zeros(1024, dtype=torch.int32)
    d = torch.zeros(1024, dtype=torch.int32, device=dev)
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_copy(d, pageable, 4096)
    assert e.value.status == smoe.SMOE_ERR_MEMORY
    with pytest.raises(smoe.SmoeError) as e:
        smoe.smoe_copy(pageable, d, 4096)
    assert e.value.status == smoe.SMOE_ERR_MEMORY


def test_copy_tail_is_untouched(smoe):
    """Exactly `nbytes` are written: the words after them keep their value."""
    dev = torch.device("cuda:0")
    src = _bits(1024, 3).to(dev)
    dst = torch.full((1024,), 7, dtype=torch.int32, device=dev)
    smoe.smoe_copy(dst, src, 4 * 1000)
    torch.cuda.synchronize()
    assert torch.equal(dst[:1000], src[:1000])
    assert (dst[1000:] == 7).all()
