"""Host-side checks of the C ABI that need no GPU.

The library validates every argument on the host before touching CUDA, so
calls that break the contract return their status here without a device.
Pointer arguments in these tests are plain integers that are never
dereferenced: every call below is refused before any launch (a call that
passed the checks would launch, so none is made here).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "smoe.h")


@pytest.fixture(scope="module")
def smoe():
    import __graft_entry__
    __graft_entry__.build_library()
    import moe_expert_ffn_smoe_gb300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\**\s*([a-z_][a-z_0-9]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(smoe):
    names = _declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(smoe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in smoe.h but not exported"
    assert set(names) == set(smoe.EXPORTED)


def test_abi_version_and_status_strings(smoe):
    assert smoe.smoe_abi_version() == 2
    for s in range(10):
        assert smoe.smoe_status_string(s) != "unknown status"
    assert smoe.smoe_status_string(99) == "unknown status"


A = 1 << 20  # an aligned fake device address (never dereferenced)


def _gu(smoe, fn, d_ff=256, d_model=256, group=64, ptrs=None, stream=0):
    p = ptrs or [A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x400000, A + 0x500000]
    return fn(*p, d_ff, d_model, group, stream)


@pytest.mark.parametrize("bits", [4, 2])
def test_gate_up_refuses_bad_shapes(smoe, bits):
    f = smoe._lib.smoe_gate_up_q4 if bits == 4 else smoe._lib.smoe_gate_up_q2
    unit = 32 if bits == 4 else 64
    assert _gu(smoe, f, d_model=unit + 16) == smoe.SMOE_ERR_SHAPE        # cols not a multiple
    assert _gu(smoe, f, group=unit // 2) == smoe.SMOE_ERR_SHAPE           # group not a multiple
    assert _gu(smoe, f, d_model=3 * unit, group=2 * unit) == smoe.SMOE_ERR_SHAPE  # group !| cols
    assert _gu(smoe, f, group=0) == smoe.SMOE_ERR_SHAPE
    assert _gu(smoe, f, d_ff=-1) == smoe.SMOE_ERR_SHAPE
    assert _gu(smoe, f, d_model=smoe.SMOE_MAX_COLS + 64 * 16) == smoe.SMOE_ERR_SHAPE


def test_gate_up_refuses_null_misaligned_alias(smoe):
    f = smoe._lib.smoe_gate_up_q4
    base = [A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x400000, A + 0x500000]
    for i in range(6):
        p = list(base)
        p[i] = None
        assert _gu(smoe, f, ptrs=p) == smoe.SMOE_ERR_NULL
        p = list(base)
        p[i] += 4
        assert _gu(smoe, f, ptrs=p) == smoe.SMOE_ERR_ALIGN
    p = list(base)
    p[5] = p[4] + 512          # hidden overlaps x (x is 1 KB)
    assert _gu(smoe, f, ptrs=p) == smoe.SMOE_ERR_ALIAS
    p = list(base)
    p[5] = p[0] + 16           # hidden inside the gate codes
    assert _gu(smoe, f, ptrs=p) == smoe.SMOE_ERR_ALIAS


def test_empty_output_is_a_no_op_without_pointers(smoe):
    L = smoe._lib
    assert L.smoe_gate_up_q4(None, None, None, None, None, None, 0, 256, 64, None) == 0
    assert L.smoe_down_q2(None, None, None, None, 0, 256, 64, None) == 0
    assert L.matvec_bf16(None, None, None, 0, 64, None) == 0
    assert L.ffn_batch_q4(None, None, None, None, None, None, None, None, 0, 256, 256, 64, None, 0,
                          None) == 0


def test_down_refusals(smoe):
    L = smoe._lib
    ok = [A, A + 0x100000, A + 0x200000, A + 0x300000]
    assert L.smoe_down_q4(*ok, 256, 96, 64, None) == smoe.SMOE_ERR_SHAPE     # 96 % 64 != 0
    assert L.smoe_down_q2(*ok, 256, 96, 64, None) == smoe.SMOE_ERR_SHAPE     # Q2 wants % 64
    assert L.smoe_down_q4(ok[0], ok[1], ok[2], None, 256, 256, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_down_q4(ok[0], ok[1] + 8, ok[2], ok[3], 256, 256, 64, None) == smoe.SMOE_ERR_ALIGN
    assert L.smoe_down_q4(ok[0], ok[1], ok[2], ok[2] + 64, 256, 256, 64, None) == smoe.SMOE_ERR_ALIAS


def test_bf16_refusals(smoe):
    L = smoe._lib
    assert L.matvec_bf16(A, A + 0x100000, A + 0x200000, 16, 12, None) == smoe.SMOE_ERR_SHAPE
    assert L.matvec_bf16(A, A + 0x100000, A + 0x200000, 16, smoe.SMOE_MAX_COLS + 8, None) == \
        smoe.SMOE_ERR_SHAPE
    assert L.matvec_bf16(A + 2, A + 0x100000, A + 0x200000, 16, 64, None) == smoe.SMOE_ERR_ALIGN
    assert L.matvec_bf16(A, None, A + 0x200000, 16, 64, None) == smoe.SMOE_ERR_NULL
    assert L.matvec_bf16(A, A + 0x100000, A + 16, 16, 64, None) == smoe.SMOE_ERR_ALIAS


def test_batch_workspace_size_and_refusals(smoe):
    L = smoe._lib
    need = L.smoe_ffn_batch_workspace_bytes(16, 4096, 1536, 64)
    assert need >= 16 * 1536 * 4 and need % 256 == 0
    assert L.smoe_ffn_batch_workspace_bytes(0, 4096, 1536, 64) == 0
    assert L.smoe_ffn_batch_workspace_bytes(4, 4096, 1536, 48) == ctypes.c_size_t(-1).value
    w = [A + i * 0x1000000 for i in range(6)]
    X, Y, ws = A + 0x8000000, A + 0x9000000, A + 0xA000000
    args = lambda T, wsp, wsb: (*w, X, Y, T, 4096, 1536, 64, wsp, wsb, None)
    assert L.ffn_batch_q4(*args(16, ws, need - 256)) == smoe.SMOE_ERR_WORKSPACE
    assert L.ffn_batch_q4(*args(16, None, need)) == smoe.SMOE_ERR_WORKSPACE
    assert L.ffn_batch_q4(*args(16, ws + 8, need)) == smoe.SMOE_ERR_ALIGN
    assert L.ffn_batch_q4(*args(-1, ws, need)) == smoe.SMOE_ERR_SHAPE
    assert L.ffn_batch_q4(*args(16, X + 1024, need)) == smoe.SMOE_ERR_ALIAS   # workspace inside X


def test_binding_raises_with_status(smoe):
    with pytest.raises(smoe.SmoeError) as ei:
        smoe.smoe_gate_up_q4(A, A, A, A, A, A, 256, 100, 64, stream=0)
    assert ei.value.status == smoe.SMOE_ERR_SHAPE


def test_grouped_refusals(smoe):
    L = smoe._lib
    P = lambda vals: (ctypes.c_void_p * len(vals))(*vals)
    g = P([A, A + 0x100000])
    gs = P([A + 0x200000, A + 0x300000])
    x, h = A + 0x400000, A + 0x500000
    assert L.smoe_experts_gate_up_q4(-1, g, gs, g, gs, x, h, 256, 256, 64, None) == smoe.SMOE_ERR_SHAPE
    assert L.smoe_experts_gate_up_q4(2, g, gs, g, gs, x, h, 256, 100, 64, None) == smoe.SMOE_ERR_SHAPE
    assert L.smoe_experts_gate_up_q4(2, None, gs, g, gs, x, h, 256, 256, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_experts_gate_up_q4(2, P([A, 0]), gs, g, gs, x, h, 256, 256, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_experts_gate_up_q4(2, P([A, A + 8]), gs, g, gs, x, h, 256, 256, 64, None) == smoe.SMOE_ERR_ALIGN
    assert L.smoe_experts_gate_up_q4(2, g, gs, g, gs, x, x + 256, 256, 256, 64, None) == smoe.SMOE_ERR_ALIAS
    assert L.smoe_experts_gate_up_q4(2, g, gs, g, gs, x, A + 0x100000 + 1024, 256, 256, 64, None) == \
        smoe.SMOE_ERR_ALIAS
    assert L.smoe_experts_down_q2(2, g, gs, x, A + 0x200000, 256, 256, 64, None) == smoe.SMOE_ERR_ALIAS
    assert L.smoe_experts_down_q4(0, None, None, None, None, 256, 256, 64, None) == smoe.SMOE_OK


def test_experts_ffn_workspace_and_refusals(smoe):
    L = smoe._lib
    assert L.smoe_experts_ffn_workspace_bytes(0, 1536) == 0
    assert L.smoe_experts_ffn_workspace_bytes(8, 1536) == 512 + 8 * 1536 * 4
    assert L.smoe_experts_ffn_workspace_bytes(100, 1536) == 512 + 64 * 1536 * 4
    assert L.smoe_experts_ffn_workspace_bytes(3, 100) % 256 == 0
    assert L.smoe_experts_ffn_workspace_bytes(3, -1) == ctypes.c_size_t(-1).value
    P = lambda vals: (ctypes.c_void_p * len(vals))(*vals)
    w = [P([A + 0x1000000 * (6 * e + k) for e in range(2)]) for k in range(6)]
    x, out = A + 0x40000000, A + 0x41000000
    ws = A + 0x42000000
    need = L.smoe_experts_ffn_workspace_bytes(2, 1536)
    f = L.smoe_experts_ffn_q4
    args = lambda n=2, wsp=ws, wsb=need, o=out, dm=4096, df=1536, g=64: (n, *w, x, o, dm, df, g, wsp, wsb, None)
    assert f(*args(wsb=need - 4)) == smoe.SMOE_ERR_WORKSPACE
    assert f(*args(wsp=None)) == smoe.SMOE_ERR_WORKSPACE
    assert f(*args(wsp=ws + 8)) == smoe.SMOE_ERR_ALIGN
    assert f(*args(n=-1)) == smoe.SMOE_ERR_SHAPE
    assert f(*args(df=1000)) == smoe.SMOE_ERR_SHAPE          # d_ff not a multiple of the group
    assert f(*args(o=ws + 1024)) == smoe.SMOE_ERR_ALIAS      # out inside the workspace
    assert f(*args(wsp=x - 256)) == smoe.SMOE_ERR_ALIAS      # workspace over x
    assert f(*args(o=A + 0x1000000 * 4 + 64)) == smoe.SMOE_ERR_ALIAS  # out over expert 0's down codes
    assert f(*args(n=0)) == smoe.SMOE_OK
    bad = [P([A, A + 8])] + w[1:]
    assert f(2, *bad, x, out, 4096, 1536, 64, ws, need, None) == smoe.SMOE_ERR_ALIGN


def test_bf16_batch_refusals(smoe):
    L = smoe._lib
    P = lambda v: (ctypes.c_void_p * len(v))(*v)
    I = lambda v: (ctypes.c_int * len(v))(*v)
    w = [A, A + 0x1000000, A + 0x2000000]
    x = [A + 0x3000000, A + 0x3100000, A + 0x3200000]
    y = [A + 0x4000000, A + 0x4100000, A + 0x4200000]
    rows, cols = [16, 32, 8], [64, 128, 4096]

    def call(n=3, w=w, x=x, y=y, rows=rows, cols=cols):
        return L.matvec_bf16_batch(n, P(w), P(x), P(y), I(rows), I(cols), None)

    assert L.matvec_bf16_batch(0, None, None, None, None, None, None) == smoe.SMOE_OK
    assert L.matvec_bf16_batch(-1, None, None, None, None, None, None) == smoe.SMOE_ERR_SHAPE
    assert L.matvec_bf16_batch(2, None, P(x), P(y), I(rows), I(cols), None) == smoe.SMOE_ERR_NULL
    assert call(cols=[64, 12, 4096]) == smoe.SMOE_ERR_SHAPE                        # cols % 8
    assert call(cols=[64, 128, smoe.SMOE_MAX_COLS + 8]) == smoe.SMOE_ERR_SHAPE
    assert call(rows=[16, -1, 8]) == smoe.SMOE_ERR_SHAPE
    assert call(w=[A, 0, A + 0x2000000]) == smoe.SMOE_ERR_NULL
    assert call(y=[A + 0x4000000, A + 0x4100000, A + 0x4200004]) == smoe.SMOE_ERR_ALIGN
    assert call(y=[A + 0x4000000, A + 0x4000000 + 32, A + 0x4200000]) == smoe.SMOE_ERR_ALIAS  # two outputs
    assert call(y=[A + 0x4000000, A + 0x1000000 + 256, A + 0x4200000]) == smoe.SMOE_ERR_ALIAS  # y1 over w1
    assert call(y=[A + 0x3200000, A + 0x4100000, A + 0x4200000]) == smoe.SMOE_ERR_ALIAS   # y0 over x2


def test_experts_batch_workspace_and_refusals(smoe):
    L = smoe._lib
    I = lambda v: (ctypes.c_int * len(v))(*v)
    P = lambda v: (ctypes.c_void_p * len(v))(*v)
    T = [16, 0, 3]
    need = L.smoe_experts_ffn_batch_workspace_bytes(3, I(T), 4096, 1536, 64)
    assert need > 0 and need % 256 == 0
    assert need >= L.smoe_ffn_batch_workspace_bytes(16, 4096, 1536, 64)
    assert L.smoe_experts_ffn_batch_workspace_bytes(0, None, 4096, 1536, 64) == 0
    assert L.smoe_experts_ffn_batch_workspace_bytes(2, I([4, -1]), 4096, 1536, 64) == ctypes.c_size_t(-1).value
    assert L.smoe_experts_ffn_batch_workspace_bytes(2, I([4, 4]), 4096, 1536, 48) == ctypes.c_size_t(-1).value
    w = [[A + 0x1000000 * (3 * k + e) for e in range(3)] for k in range(6)]
    X = [A + 0x20000000 + 0x1000000 * e for e in range(3)]
    Y = [A + 0x30000000 + 0x1000000 * e for e in range(3)]
    ws = A + 0x40000000
    f = L.smoe_experts_ffn_batch_q4

    def args(T=T, X=X, Y=Y, wsp=ws, wsb=need, group=64, n=3):
        return (n, *[P(v) for v in w], P(X), P(Y), I(T), 4096, 1536, group, wsp, wsb, None)

    assert f(*args(n=-1)) == smoe.SMOE_ERR_SHAPE
    assert f(*args(T=[16, -2, 3])) == smoe.SMOE_ERR_SHAPE
    assert f(*args(group=48)) == smoe.SMOE_ERR_SHAPE
    assert f(*args(T=[0, 0, 0])) == smoe.SMOE_OK                               # nothing to do
    assert f(*args(wsb=need - 256)) == smoe.SMOE_ERR_WORKSPACE
    assert f(*args(wsp=ws + 8)) == smoe.SMOE_ERR_ALIGN
    need3 = L.smoe_experts_ffn_batch_workspace_bytes(3, I([16, 5, 3]), 4096, 1536, 64)
    assert f(*args(X=[X[0], 0, X[2]], T=[16, 5, 3], wsb=need3)) == smoe.SMOE_ERR_NULL
    assert f(*args(Y=[Y[0], Y[0] + 64, Y[2]], T=[16, 5, 3], wsb=need3)) == smoe.SMOE_ERR_ALIAS   # two outputs
    assert f(*args(Y=[X[2] + 256, Y[1], Y[2]])) == smoe.SMOE_ERR_ALIAS                # Y0 over X2
    assert f(*args(wsp=w[4][2] + 1024)) == smoe.SMOE_ERR_ALIAS                         # workspace over down codes
    # an expert with no tokens may hold null pointers
    X2 = [X[0], 0, X[2]]
    Y2 = [Y[0], 0, Y[2]]
    assert f(*args(X=X2, Y=Y2, wsp=0)) == smoe.SMOE_ERR_WORKSPACE                       # still needs the workspace
    assert smoe._lib.smoe_experts_ffn_batch_q2(*args(group=32)) == smoe.SMOE_ERR_SHAPE  # Q2 groups of 64


def test_route_and_combine_refusals(smoe):
    L = smoe._lib
    g, x = A, A + 0x1000000
    lg, ix, w = A + 0x2000000, A + 0x2100000, A + 0x2200000
    r = lambda n=128, d=4096, k=8, g=g, x=x, lg=lg, ix=ix, w=w: L.smoe_route_topk_bf16(g, x, n, d, k, lg, ix, w, None)
    assert r(k=0) == smoe.SMOE_ERR_SHAPE
    assert r(k=129) == smoe.SMOE_ERR_SHAPE
    assert r(n=200, k=smoe.SMOE_MAX_TOP_K + 1) == smoe.SMOE_ERR_SHAPE
    assert r(n=smoe.SMOE_MAX_ROUTE_EXPERTS + 1) == smoe.SMOE_ERR_SHAPE
    assert r(d=4100) == smoe.SMOE_ERR_SHAPE
    assert r(n=0) == smoe.SMOE_ERR_SHAPE
    assert r(lg=0) == smoe.SMOE_ERR_NULL
    assert r(g=0) == smoe.SMOE_ERR_NULL
    assert r(lg=lg + 4) == smoe.SMOE_ERR_ALIGN
    assert r(ix=ix + 2) == smoe.SMOE_ERR_ALIGN
    assert r(lg=g + 1024) == smoe.SMOE_ERR_ALIAS          # logits inside the gate matrix
    assert r(w=ix + 16) == smoe.SMOE_ERR_ALIAS            # weights over the indices
    c = lambda k=8, eo=A, tw=A + 0x100000, out=A + 0x200000, d=4096: L.smoe_combine(k, eo, tw, out, d, None)
    assert c(k=-1) == smoe.SMOE_ERR_SHAPE
    assert c(d=0) == smoe.SMOE_OK
    assert c(eo=0) == smoe.SMOE_ERR_NULL
    assert c(out=A + 0x200002) == smoe.SMOE_ERR_ALIGN
    assert c(out=A + 4096) == smoe.SMOE_ERR_ALIAS          # out inside the expert outputs


def test_selftest_refuses_unknown_kind(smoe):
    for kind in (-1, 2, 7):
        assert smoe._lib.smoe_selftest_bounded_wait(kind, None) == smoe.SMOE_ERR_SHAPE


def test_copy_refusals(smoe):
    L = smoe._lib
    A = 0x7f0000000000
    assert L.smoe_copy(None, None, 0, None) == smoe.SMOE_OK                # nothing to copy
    assert L.smoe_copy(None, A, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_copy(A, None, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_copy(A + 8, A + 4096, 64, None) == smoe.SMOE_ERR_ALIGN   # dst
    assert L.smoe_copy(A, A + 4104, 64, None) == smoe.SMOE_ERR_ALIGN       # src
    assert L.smoe_copy(A, A + 4096, 40, None) == smoe.SMOE_ERR_ALIGN       # size
    assert L.smoe_copy(A, A + 48, 64, None) == smoe.SMOE_ERR_ALIAS         # overlapping ranges
    assert smoe.smoe_status_string(smoe.SMOE_ERR_MEMORY) != "unknown status"


def test_q2_grouped_and_one_launch_refusals(smoe):
    """The Q2 grouped and one-launch entries apply the Q2 layout rules
    (cols a multiple of 64, groups a multiple of 64) before any launch."""
    L = smoe._lib
    P = lambda vals: (ctypes.c_void_p * len(vals))(*vals)
    g = P([A, A + 0x100000])
    gs = P([A + 0x200000, A + 0x300000])
    x, h = A + 0x400000, A + 0x500000
    assert L.smoe_experts_gate_up_q2(2, g, gs, g, gs, x, h, 256, 256, 32, None) == smoe.SMOE_ERR_SHAPE
    assert L.smoe_experts_gate_up_q2(2, g, gs, g, gs, x, h, 256, 96, 64, None) == smoe.SMOE_ERR_SHAPE
    assert L.smoe_experts_gate_up_q2(2, None, gs, g, gs, x, h, 256, 256, 64, None) == smoe.SMOE_ERR_NULL
    assert L.smoe_experts_gate_up_q2(0, None, None, None, None, None, None, 256, 256, 64, None) == smoe.SMOE_OK
    w = [P([A + 0x1000000 * (6 * e + k) for e in range(2)]) for k in range(6)]
    x, out, ws = A + 0x40000000, A + 0x41000000, A + 0x42000000
    need = L.smoe_experts_ffn_workspace_bytes(2, 1536)
    f = L.smoe_experts_ffn_q2
    assert f(2, *w, x, out, 4096, 1536, 32, ws, need, None) == smoe.SMOE_ERR_SHAPE     # Q2 groups of 64
    assert f(2, *w, x, out, 4096, 1536, 64, ws, need - 4, None) == smoe.SMOE_ERR_WORKSPACE


def test_noalloc_refusals_before_any_launch(smoe):
    L = smoe._lib
    ptrs = [A + 0x1000000 * i for i in range(8)]
    # a workspace beyond the fixed device array
    big = 100000
    assert L.smoe_ffn_batch_workspace_bytes(big, 4096, 1536, 64) > smoe.SMOE_NOALLOC_SCRATCH_BYTES
    assert L.ffn_batch_q4_noalloc(*ptrs, big, 4096, 1536, 64, None) == smoe.SMOE_ERR_SHAPE
    assert L.ffn_batch_q4_noalloc(*ptrs, -1, 4096, 1536, 64, None) == smoe.SMOE_ERR_SHAPE
    assert L.ffn_batch_q4_noalloc(*ptrs, 0, 4096, 1536, 64, None) == smoe.SMOE_OK
    # the shape is checked before the empty batch returns, as in ffn_batch_q4
    assert L.ffn_batch_q4_noalloc(*ptrs, 0, 4096, 1536, 48, None) == smoe.SMOE_ERR_SHAPE
    assert L.ffn_batch_q4(*ptrs[:8], 0, 4096, 1536, 48, None, 0, None) == smoe.SMOE_ERR_SHAPE
    assert L.smoe_ffn_batch_workspace_bytes(0, 4096, 1536, 48) == ctypes.c_size_t(-1).value


@pytest.mark.parametrize("bits", [4, 2])
def test_routed_refusals_before_any_launch(smoe, bits):
    """smoe_experts_ffn_routed_q4/q2: every host-side check returns its
    status without launching (fake, aligned device addresses)."""
    L = smoe._lib
    f = L.smoe_experts_ffn_routed_q4 if bits == 4 else L.smoe_experts_ffn_routed_q2
    tabs = [A + 0x100000 * i for i in range(6)]
    idx, x, out, ws = A + 0x1000000, A + 0x2000000, A + 0x3000000, A + 0x4000000
    need = L.smoe_experts_ffn_routed_workspace_bytes(8, 1536)
    assert need == 8 * 1536 * 4
    assert L.smoe_experts_ffn_routed_workspace_bytes(65, 1536) == ctypes.c_size_t(-1).value
    assert L.smoe_experts_ffn_routed_workspace_bytes(-1, 1536) == ctypes.c_size_t(-1).value

    def call(n=128, k=8, tabs=tabs, idx=idx, x=x, out=out, d_model=4096, d_ff=1536, group=64, ws=ws,
             wsb=need):
        return f(n, k, *tabs, idx, x, out, d_model, d_ff, group, ws, wsb, None)

    assert call(k=0) == smoe.SMOE_OK                       # nothing selected: no-op
    assert call(k=65) == smoe.SMOE_ERR_SHAPE               # beyond SMOE_MAX_ROUTED_SLOTS
    assert call(k=-1) == smoe.SMOE_ERR_SHAPE
    assert call(n=0) == smoe.SMOE_ERR_SHAPE                # no index could be valid
    assert call(group=48) == smoe.SMOE_ERR_SHAPE
    assert call(d_model=4096 + 16) == smoe.SMOE_ERR_SHAPE
    assert call(idx=None) == smoe.SMOE_ERR_NULL
    assert call(out=None) == smoe.SMOE_ERR_NULL
    assert call(tabs=[None] + tabs[1:]) == smoe.SMOE_ERR_NULL
    assert call(tabs=[A + 4] + tabs[1:]) == smoe.SMOE_ERR_ALIGN   # tables are pointer arrays
    assert call(idx=idx + 2) == smoe.SMOE_ERR_ALIGN
    assert call(out=out + 8) == smoe.SMOE_ERR_ALIGN
    assert call(ws=None) == smoe.SMOE_ERR_WORKSPACE
    assert call(wsb=need - 4) == smoe.SMOE_ERR_WORKSPACE
    assert call(out=ws) == smoe.SMOE_ERR_ALIAS             # out over the workspace
    assert call(out=x) == smoe.SMOE_ERR_ALIAS              # out over the token
    assert call(idx=out + 64) == smoe.SMOE_ERR_ALIAS       # out over the indices
    # rows the bulk-copy decode kernels do not take: not whole multiples of
    # 8 chunks, or longer than 8192 columns
    assert call(d_model=256, d_ff=96 if bits == 4 else 192, group=32 if bits == 4 else 64) == smoe.SMOE_ERR_SHAPE
    assert call(d_model=16384) == smoe.SMOE_ERR_SHAPE
    assert call(d_ff=1536 + (128 if bits == 4 else 256)) == smoe.SMOE_ERR_SHAPE
