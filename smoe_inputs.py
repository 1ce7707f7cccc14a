"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds random-number generation only: none of the method's
arithmetic (no unpacking, dequantisation, dot products or SiLU).  Every array
comes from numpy's ``default_rng([seed, tensor_id, block])``, so the same
(seed, tensor id) gives the same bytes on every host.

Recipes (shapes and distributions of the workloads the S-MoE page
"Metal Compute Kernels" measures; its "real vault blobs" are not available,
so these synthetic tensors stand in for them):

* packed codes: independent uniform bytes.  A uniform byte is exactly two
  independent uniform Q4 codes (0..15) or four uniform Q2 codes (0..3), so
  the generator needs no knowledge of the packing order.
* scales: f32 uniform in [0.01, 0.05], one per (row, group of columns).
* activations x / X: f32 standard normal.
* bf16 weights: f32 normal with standard deviation 0.02, rounded to the
  nearest bf16 (ties to even) and stored as uint16 bit patterns; generated in
  blocks of 4096 rows so that any row range can be regenerated on its own.
"""
import numpy as np

BF16_ROW_BLOCK = 4096

# tensor ids inside one expert (expert e uses 16*e + id)
GATE_CODES, GATE_SCALES, UP_CODES, UP_SCALES, DOWN_CODES, DOWN_SCALES = range(6)
X_ID = 100000


def _rng(seed, tid, block=0):
    return np.random.default_rng([int(seed), int(tid), int(block)])


def packed_codes(rows, cols, bits, seed, tid):
    """uint8 [rows, cols*bits/8] of uniform random bytes."""
    nbytes = cols * bits // 8
    return _rng(seed, tid).integers(0, 256, size=(rows, nbytes), dtype=np.uint8)


def scales(rows, ngroups, seed, tid, lo=0.01, hi=0.05):
    """f32 [rows, ngroups] uniform in [lo, hi)."""
    return _rng(seed, tid).uniform(lo, hi, size=(rows, ngroups)).astype(np.float32)


def activations(shape, seed, tid=X_ID):
    """f32 standard normal of the given shape."""
    return _rng(seed, tid).standard_normal(size=shape, dtype=np.float32)


def _f32_to_bf16_bits(a):
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_rows(rows, cols, seed, tid, r0=0, r1=None, std=0.02):
    """uint16 bf16 bit patterns for rows [r0, r1) of a [rows, cols] matrix."""
    r1 = rows if r1 is None else r1
    out = np.empty((r1 - r0, cols), dtype=np.uint16)
    b0, b1 = r0 // BF16_ROW_BLOCK, (r1 + BF16_ROW_BLOCK - 1) // BF16_ROW_BLOCK
    for b in range(b0, b1):
        lo, hi = b * BF16_ROW_BLOCK, min(rows, (b + 1) * BF16_ROW_BLOCK)
        blk = _rng(seed, tid, b).standard_normal(size=(hi - lo, cols), dtype=np.float32)
        blk *= np.float32(std)
        s0, s1 = max(lo, r0), min(hi, r1)
        out[s0 - r0:s1 - r0] = _f32_to_bf16_bits(blk[s0 - lo:s1 - lo])
    return out


def expert(bits, d_model, d_ff, group, seed, e=0):
    """The six tensors of one expert: gate/up [d_ff, d_model], down [d_model, d_ff]."""
    base = 16 * e
    return {
        "gate_codes": packed_codes(d_ff, d_model, bits, seed, base + GATE_CODES),
        "gate_scales": scales(d_ff, d_model // group, seed, base + GATE_SCALES),
        "up_codes": packed_codes(d_ff, d_model, bits, seed, base + UP_CODES),
        "up_scales": scales(d_ff, d_model // group, seed, base + UP_SCALES),
        "down_codes": packed_codes(d_model, d_ff, bits, seed, base + DOWN_CODES),
        "down_scales": scales(d_model, d_ff // group, seed, base + DOWN_SCALES),
    }


# The five workloads: (name, description) -> parameters.
CONFIGS = {
    "q4_ffn_256": dict(bits=4, d_model=256, d_ff=256, group=64, experts=1, seed=0),
    "bf16_matvec": dict(shapes=[(8192, 4096), (4096, 8192), (512, 4096), (151936, 4096)],
                        seeds=[1, 2, 3, 4]),
    "q4_8expert_decode": dict(bits=4, d_model=4096, d_ff=1536, group=64, experts=8, seed=5),
    "q2_8expert_decode": dict(bits=2, d_model=4096, d_ff=1536, group=64, experts=8, seed=6),
    "q4_token_batch": dict(bits=4, d_model=4096, d_ff=1536, group=64, experts=1,
                           tokens=[1, 16, 64, 256], seed=7),
}
