"""Python binding of libsmoe.so (include/smoe.h): group-quantized routed-expert
GEMVs for GB300.

Argument marshalling only: each function below has the name of the C entry
point it calls, turns tensors into device pointers and a stream into a
cudaStream_t, and raises SmoeError when the call returns a non-zero status.
Every step of the computation runs in the library's CUDA kernels; there is no
Python or CPU implementation here and no fallback.  If the library has not
been built, importing this package raises ImportError.

Pointer arguments accept a torch.Tensor (its data_ptr()), an int device
address, or None (NULL).  `stream` accepts a torch.cuda.Stream, an int
cudaStream_t, or None for torch's current stream on the current device.

One MoE layer for one token, every step on the GPU and no host round trip
(the four calls can be captured in one CUDA graph)::

    import moe_expert_ffn_smoe_gb300 as smoe
    # once, when the weights are loaded: device tables of expert pointers
    tabs = [smoe.pointer_table(ts, dev) for ts in (gc, gs, uc, us, dc, ds)]
    # per token; gate: bf16 bits [n_experts, d_model] as int16; x: f32 [d_model]
    smoe.smoe_route_topk_bf16(gate, x, n_experts, d_model, k, logits, idx, w)
    smoe.smoe_experts_ffn_routed_q4(n_experts, k, *tabs, idx, x, expert_out,
                                    d_model, d_ff, group, ws, ws_bytes)
    smoe.smoe_combine(k, expert_out, w, out, d_model)

(`ws`: smoe_experts_ffn_routed_workspace_bytes(k, d_ff) bytes.)  With the
selection on the host, smoe_experts_ffn_q4 takes host lists of the selected
experts' tensors instead.  Several tokens per expert go through
smoe_experts_ffn_batch_q4/q2; a dense bf16 matvec is matvec_bf16, many of
them in one submission matvec_bf16_batch.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsmoe.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
        "(the library has no CPU fallback)")

_lib = ctypes.CDLL(LIB_PATH)

SMOE_OK = 0
SMOE_ERR_NULL = 1
SMOE_ERR_ALIGN = 2
SMOE_ERR_SHAPE = 3
SMOE_ERR_WORKSPACE = 4
SMOE_ERR_LAUNCH = 5
SMOE_ERR_TIMEOUT = 6
SMOE_ERR_ALIAS = 7
SMOE_ERR_MEMORY = 8
SMOE_ERR_ROUTE = 9
SMOE_MAX_ROUTED_SLOTS = 64
SMOE_MAX_COLS = 32768
SMOE_NOALLOC_SCRATCH_BYTES = 32 << 20
SMOE_FFN_SYNC_BYTES = 512

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t

_SIGS = {
    "smoe_abi_version": ([], _I),
    "smoe_status_string": ([_I], ctypes.c_char_p),
    "smoe_gate_up_q4": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_gate_up_q2": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_down_q4": ([_P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_down_q2": ([_P, _P, _P, _P, _I, _I, _I, _P], _I),
    "matvec_bf16": ([_P, _P, _P, _I, _I, _P], _I),
    "matvec_bf16_batch": ([_I, _P, _P, _P, _P, _P, _P], _I),
    "smoe_experts_gate_up_q4": ([_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_experts_gate_up_q2": ([_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_experts_down_q4": ([_I, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_experts_down_q2": ([_I, _P, _P, _P, _P, _I, _I, _I, _P], _I),
    "smoe_experts_ffn_workspace_bytes": ([_I, _I], _SZ),
    "smoe_experts_ffn_q4": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_experts_ffn_q2": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_ffn_batch_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "ffn_batch_q4": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "ffn_batch_q2": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_experts_ffn_routed_workspace_bytes": ([_I, _I], _SZ),
    "smoe_experts_ffn_routed_q4": ([_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_experts_ffn_routed_q2": ([_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_route_topk_bf16": ([_P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "smoe_combine": ([_I, _P, _P, _P, _I, _P], _I),
    "smoe_experts_ffn_batch_workspace_bytes": ([_I, _P, _I, _I, _I], _SZ),
    "smoe_experts_ffn_batch_q4": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "smoe_experts_ffn_batch_q2": ([_I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _SZ, _P], _I),
    "ffn_batch_q4_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "smoe_last_device_status": ([_P], _I),
    "smoe_selftest_bounded_wait": ([_I, _P], _I),
    "smoe_copy": ([_P, _P, ctypes.c_size_t, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class SmoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: status {status} ({smoe_status_string(status)})")


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        import torch
        if not torch.cuda.is_available():
            return None
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status, where):
    if status != SMOE_OK:
        raise SmoeError(status, where)


def smoe_abi_version():
    return _lib.smoe_abi_version()


def smoe_status_string(status):
    return _lib.smoe_status_string(int(status)).decode()


def smoe_gate_up_q4(gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model, group,
                    stream=None):
    _check(_lib.smoe_gate_up_q4(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes), _ptr(up_scales),
                                _ptr(x), _ptr(hidden), d_ff, d_model, group, _stream(stream)),
           "smoe_gate_up_q4")


def smoe_gate_up_q2(gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model, group,
                    stream=None):
    _check(_lib.smoe_gate_up_q2(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes), _ptr(up_scales),
                                _ptr(x), _ptr(hidden), d_ff, d_model, group, _stream(stream)),
           "smoe_gate_up_q2")


def smoe_down_q4(down_codes, down_scales, hidden, out, d_model, d_ff, group, stream=None):
    _check(_lib.smoe_down_q4(_ptr(down_codes), _ptr(down_scales), _ptr(hidden), _ptr(out), d_model,
                             d_ff, group, _stream(stream)), "smoe_down_q4")


def smoe_down_q2(down_codes, down_scales, hidden, out, d_model, d_ff, group, stream=None):
    _check(_lib.smoe_down_q2(_ptr(down_codes), _ptr(down_scales), _ptr(hidden), _ptr(out), d_model,
                             d_ff, group, _stream(stream)), "smoe_down_q2")


def _ptr_array(items):
    """A host array of device pointers (ctypes), kept alive by the caller."""
    arr = (ctypes.c_void_p * max(1, len(items)))()
    for i, t in enumerate(items):
        arr[i] = _ptr(t)
    return arr


def _experts_gate_up(fn, name, gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model,
                     group, stream):
    n = len(gate_codes)
    if not (len(gate_scales) == len(up_codes) == len(up_scales) == n):
        raise ValueError(f"{name}: per-expert lists differ in length")
    arrs = [_ptr_array(a) for a in (gate_codes, gate_scales, up_codes, up_scales)]
    _check(fn(n, *arrs, _ptr(x), _ptr(hidden), d_ff, d_model, group, _stream(stream)), name)


def smoe_experts_gate_up_q4(gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model,
                            group, stream=None):
    """Per-expert lists of tensors; hidden is [n_experts, d_ff]."""
    _experts_gate_up(_lib.smoe_experts_gate_up_q4, "smoe_experts_gate_up_q4", gate_codes, gate_scales,
                     up_codes, up_scales, x, hidden, d_ff, d_model, group, stream)


def smoe_experts_gate_up_q2(gate_codes, gate_scales, up_codes, up_scales, x, hidden, d_ff, d_model,
                            group, stream=None):
    _experts_gate_up(_lib.smoe_experts_gate_up_q2, "smoe_experts_gate_up_q2", gate_codes, gate_scales,
                     up_codes, up_scales, x, hidden, d_ff, d_model, group, stream)


def _experts_down(fn, name, down_codes, down_scales, hidden, out, d_model, d_ff, group, stream):
    n = len(down_codes)
    if len(down_scales) != n:
        raise ValueError(f"{name}: per-expert lists differ in length")
    arrs = [_ptr_array(a) for a in (down_codes, down_scales)]
    _check(fn(n, *arrs, _ptr(hidden), _ptr(out), d_model, d_ff, group, _stream(stream)), name)


def smoe_experts_down_q4(down_codes, down_scales, hidden, out, d_model, d_ff, group, stream=None):
    """Per-expert lists of tensors; hidden [n_experts, d_ff], out [n_experts, d_model]."""
    _experts_down(_lib.smoe_experts_down_q4, "smoe_experts_down_q4", down_codes, down_scales, hidden, out,
                  d_model, d_ff, group, stream)


def smoe_experts_down_q2(down_codes, down_scales, hidden, out, d_model, d_ff, group, stream=None):
    _experts_down(_lib.smoe_experts_down_q2, "smoe_experts_down_q2", down_codes, down_scales, hidden, out,
                  d_model, d_ff, group, stream)


def smoe_experts_ffn_workspace_bytes(n_experts, d_ff):
    return _lib.smoe_experts_ffn_workspace_bytes(n_experts, d_ff)


def _experts_ffn(fn, name, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, x, out,
                 d_model, d_ff, group, workspace, workspace_bytes, stream):
    lists = (gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales)
    n = len(gate_codes)
    if any(len(a) != n for a in lists):
        raise ValueError(f"{name}: per-expert lists differ in length")
    arrs = [_ptr_array(a) for a in lists]
    _check(fn(n, *arrs, _ptr(x), _ptr(out), d_model, d_ff, group, _ptr(workspace), workspace_bytes,
              _stream(stream)), name)


def smoe_experts_ffn_q4(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, x, out,
                        d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    """Per-expert lists of tensors; out [n_experts, d_model]; workspace of
    smoe_experts_ffn_workspace_bytes(n_experts, d_ff) bytes whose first
    SMOE_FFN_SYNC_BYTES are zero before the first call."""
    _experts_ffn(_lib.smoe_experts_ffn_q4, "smoe_experts_ffn_q4", gate_codes, gate_scales, up_codes, up_scales,
                 down_codes, down_scales, x, out, d_model, d_ff, group, workspace, workspace_bytes, stream)


def smoe_experts_ffn_q2(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, x, out,
                        d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    _experts_ffn(_lib.smoe_experts_ffn_q2, "smoe_experts_ffn_q2", gate_codes, gate_scales, up_codes, up_scales,
                 down_codes, down_scales, x, out, d_model, d_ff, group, workspace, workspace_bytes, stream)


def matvec_bf16(w, x, y, rows, cols, stream=None):
    _check(_lib.matvec_bf16(_ptr(w), _ptr(x), _ptr(y), rows, cols, _stream(stream)), "matvec_bf16")


def matvec_bf16_batch(ws, xs, ys, rows, cols, stream=None):
    """Lists of n tensors (or device addresses) and n sizes; one submission."""
    n = len(ws)
    if not (len(xs) == len(ys) == len(rows) == len(cols) == n):
        raise ValueError("matvec_bf16_batch: lists differ in length")
    arrs = [_ptr_array(a) for a in (ws, xs, ys)]
    r = (ctypes.c_int * max(1, n))(*rows)
    c = (ctypes.c_int * max(1, n))(*cols)
    _check(_lib.matvec_bf16_batch(n, *arrs, r, c, _stream(stream)), "matvec_bf16_batch")


def smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group):
    return _lib.smoe_ffn_batch_workspace_bytes(T, d_model, d_ff, group)


def ffn_batch_q4(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                 d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    _check(_lib.ffn_batch_q4(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes), _ptr(up_scales),
                             _ptr(down_codes), _ptr(down_scales), _ptr(X), _ptr(Y), T, d_model,
                             d_ff, group, _ptr(workspace), workspace_bytes, _stream(stream)),
           "ffn_batch_q4")


def ffn_batch_q2(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                 d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    _check(_lib.ffn_batch_q2(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes), _ptr(up_scales),
                             _ptr(down_codes), _ptr(down_scales), _ptr(X), _ptr(Y), T, d_model,
                             d_ff, group, _ptr(workspace), workspace_bytes, _stream(stream)),
           "ffn_batch_q2")


SMOE_MAX_TOP_K = 64
SMOE_MAX_ROUTE_EXPERTS = 8192


def pointer_table(tensors, device):
    """A device array (torch int64 [n]) of the tensors' data pointers: the
    table argument of smoe_experts_ffn_routed_q4/q2, built once."""
    import torch
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def smoe_experts_ffn_routed_workspace_bytes(k, d_ff):
    return _lib.smoe_experts_ffn_routed_workspace_bytes(k, d_ff)


def smoe_experts_ffn_routed_q4(n_experts, k, gate_codes, gate_scales, up_codes, up_scales, down_codes,
                               down_scales, top_idx, x, out, d_model, d_ff, group, workspace, workspace_bytes,
                               stream=None):
    """Tables: device arrays of n_experts pointers (pointer_table); top_idx:
    int32 [k] on the device; out [k, d_model]."""
    _check(_lib.smoe_experts_ffn_routed_q4(n_experts, k, _ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes),
                                           _ptr(up_scales), _ptr(down_codes), _ptr(down_scales), _ptr(top_idx),
                                           _ptr(x), _ptr(out), d_model, d_ff, group, _ptr(workspace),
                                           workspace_bytes, _stream(stream)),
           "smoe_experts_ffn_routed_q4")


def smoe_experts_ffn_routed_q2(n_experts, k, gate_codes, gate_scales, up_codes, up_scales, down_codes,
                               down_scales, top_idx, x, out, d_model, d_ff, group, workspace, workspace_bytes,
                               stream=None):
    _check(_lib.smoe_experts_ffn_routed_q2(n_experts, k, _ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes),
                                           _ptr(up_scales), _ptr(down_codes), _ptr(down_scales), _ptr(top_idx),
                                           _ptr(x), _ptr(out), d_model, d_ff, group, _ptr(workspace),
                                           workspace_bytes, _stream(stream)),
           "smoe_experts_ffn_routed_q2")


def smoe_route_topk_bf16(gate_w, x, n_experts, d_model, k, logits, top_idx, top_w, stream=None):
    _check(_lib.smoe_route_topk_bf16(_ptr(gate_w), _ptr(x), n_experts, d_model, k, _ptr(logits), _ptr(top_idx),
                                     _ptr(top_w), _stream(stream)), "smoe_route_topk_bf16")


def smoe_combine(k, expert_out, top_w, out, d_model, stream=None):
    _check(_lib.smoe_combine(k, _ptr(expert_out), _ptr(top_w), _ptr(out), d_model, _stream(stream)),
           "smoe_combine")


def smoe_experts_ffn_batch_workspace_bytes(T, d_model, d_ff, group):
    """T: list of per-expert token counts."""
    t = (ctypes.c_int * max(1, len(T)))(*T)
    return _lib.smoe_experts_ffn_batch_workspace_bytes(len(T), t, d_model, d_ff, group)


def _experts_batch(fn, name, gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                   d_model, d_ff, group, workspace, workspace_bytes, stream):
    n = len(T)
    lists = (gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y)
    if any(len(v) != n for v in lists):
        raise ValueError(f"{name}: per-expert lists differ in length")
    arrs = [_ptr_array(v) for v in lists]
    t = (ctypes.c_int * max(1, n))(*T)
    _check(fn(n, *arrs, t, d_model, d_ff, group, _ptr(workspace), workspace_bytes, _stream(stream)), name)


def smoe_experts_ffn_batch_q4(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                              d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    """Per-expert lists of tensors (X[e], Y[e]: [T[e], d_model]) and token counts T."""
    _experts_batch(_lib.smoe_experts_ffn_batch_q4, "smoe_experts_ffn_batch_q4", gate_codes, gate_scales,
                   up_codes, up_scales, down_codes, down_scales, X, Y, T, d_model, d_ff, group, workspace,
                   workspace_bytes, stream)


def smoe_experts_ffn_batch_q2(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X, Y, T,
                              d_model, d_ff, group, workspace, workspace_bytes, stream=None):
    _experts_batch(_lib.smoe_experts_ffn_batch_q2, "smoe_experts_ffn_batch_q2", gate_codes, gate_scales,
                   up_codes, up_scales, down_codes, down_scales, X, Y, T, d_model, d_ff, group, workspace,
                   workspace_bytes, stream)


def ffn_batch_q4_noalloc(gate_codes, gate_scales, up_codes, up_scales, down_codes, down_scales, X,
                         Y, T, d_model, d_ff, group, stream=None):
    """ffn_batch_q4 with the library's static device workspace, for callers
    that must not allocate device memory (see include/smoe.h)."""
    _check(_lib.ffn_batch_q4_noalloc(_ptr(gate_codes), _ptr(gate_scales), _ptr(up_codes),
                                     _ptr(up_scales), _ptr(down_codes), _ptr(down_scales), _ptr(X),
                                     _ptr(Y), T, d_model, d_ff, group, _stream(stream)),
           "ffn_batch_q4_noalloc")


def smoe_last_device_status(stream=None):
    return _lib.smoe_last_device_status(_stream(stream))


def smoe_copy(dst, src, nbytes, stream=None):
    """dst <- src (nbytes) by the SMs; tensors or addresses of device memory or
    pinned host memory."""
    _check(_lib.smoe_copy(_ptr(dst), _ptr(src), nbytes, _stream(stream)), "smoe_copy")


def smoe_selftest_bounded_wait(kind, stream=None):
    """One warp whose bounded wait never succeeds (kind 0: mbarrier, 1: device
    counter); smoe_last_device_status then reports SMOE_ERR_TIMEOUT."""
    _check(_lib.smoe_selftest_bounded_wait(kind, _stream(stream)), "smoe_selftest_bounded_wait")
