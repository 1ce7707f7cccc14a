"""Helpers of the GPU parity tests: uploads and the tolerance checks.

Tolerance (per output element): |gpu - oracle| <= 1e-4 * sum_i |w_i x_i| + 1e-6,
with sum_i |w_i x_i| returned by the oracle.  For the hidden activations of
the gate/up pass, which are not a single dot product, the same bound is
carried through hidden = SiLU(g) * u to first order (|SiLU'| <= 1.1):
    1e-4 * (1.1 * |u| * sum|w_g x| + |SiLU(g)| * sum|w_u x|) + 1e-6.
"""
import numpy as np

EPS = 1e-4
FLOOR = 1e-6


def to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(dev)


def check(got, ref, absdot, what, eps=EPS, floor=FLOOR):
    got = np.asarray(got, dtype=np.float64).reshape(-1)
    ref = np.asarray(ref, dtype=np.float64).reshape(-1)
    bound = eps * np.asarray(absdot, dtype=np.float64).reshape(-1) + floor
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    ratio = np.abs(got - ref) / bound
    i = int(np.argmax(ratio))
    assert ratio[i] <= 1.0, (f"{what}: element {i}: gpu {got[i]!r} oracle {ref[i]!r} "
                             f"bound {bound[i]:.3g} (err/bound {ratio[i]:.3g})")
    return float(ratio[i])


def hidden_bound_absdot(r):
    """The first-order absdot of hidden for oracle.gate_up() output r."""
    with np.errstate(over="ignore"):  # exp(-g) = inf for g << 0 gives SiLU(g) = -0, as it should
        silu_g = r["g"] / (1.0 + np.exp(-r["g"]))
    return 1.1 * np.abs(r["u"]) * r["g_abs"] + np.abs(silu_g) * r["u_abs"]
