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


def test_outputs_written_straight_into_pinned_host_memory(smoe):
    """Outputs may be page-locked host memory the device addresses: the
    kernels write them over the host link, bit for bit what they write into
    device memory (grouped down, single down, combine, bf16 matvec)."""
    import smoe_inputs as inp
    dev = torch.device("cuda:0")
    d_model, d_ff, group, n = 1024, 512, 64, 3
    ex = [{k: torch.from_numpy(v).to(dev) for k, v in inp.expert(4, d_model, d_ff, group, 51, e).items()}
          for e in range(n)]
    h = torch.from_numpy(inp.activations((n, d_ff), 52)).to(dev)
    out_dev = torch.empty((n, d_model), device=dev)
    out_host = torch.full((n, d_model), float("nan")).pin_memory()
    args = ([t["down_codes"] for t in ex], [t["down_scales"] for t in ex], h)
    smoe.smoe_experts_down_q4(*args, out_dev, d_model, d_ff, group)
    smoe.smoe_experts_down_q4(*args, out_host, d_model, d_ff, group)
    one_dev = torch.empty(d_model, device=dev)
    one_host = torch.full((d_model,), float("nan")).pin_memory()
    smoe.smoe_down_q4(ex[0]["down_codes"], ex[0]["down_scales"], h[0], one_dev, d_model, d_ff, group)
    smoe.smoe_down_q4(ex[0]["down_codes"], ex[0]["down_scales"], h[0], one_host, d_model, d_ff, group)
    w = torch.tensor([0.5, 0.3, 0.2], device=dev)
    comb_dev = torch.empty(d_model, device=dev)
    comb_host = torch.full((d_model,), float("nan")).pin_memory()
    smoe.smoe_combine(n, out_dev, w, comb_dev, d_model)
    smoe.smoe_combine(n, out_dev, w, comb_host, d_model)
    wb = torch.from_numpy(inp.bf16_rows(64, 512, 53, 1).view(np.int16)).to(dev)
    xb = torch.from_numpy(inp.activations(512, 53)).to(dev)
    mv_dev = torch.empty(64, device=dev)
    mv_host = torch.full((64,), float("nan")).pin_memory()
    smoe.matvec_bf16(wb, xb, mv_dev, 64, 512)
    smoe.matvec_bf16(wb, xb, mv_host, 64, 512)
    torch.cuda.synchronize()
    assert torch.equal(out_host, out_dev.cpu())
    assert torch.equal(one_host, one_dev.cpu())
    assert torch.equal(comb_host, comb_dev.cpu())
    assert torch.equal(mv_host, mv_dev.cpu())
