"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds random-number generation and the packing of hand-chosen
codes into the stated byte layout only: none of the method's arithmetic (no
unpacking, dequantisation, dot products or SiLU).  Every array
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
* wide-range cases (edge cases, not a workload): activations spanning many
  orders of magnitude inside one group, outlier channels, or mostly
  near-zero entries, against codes chosen so that rounding errors add up.
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


# ------------------------------------------------------------------ layout
# The packed layout the workloads state: Q4 byte j of a row holds column 2j
# in its low nibble and 2j+1 in its high nibble; Q2 byte j holds columns
# 4j..4j+3 from the lowest bit pair up.  Used only to build hand-designed
# inputs; the oracle unpacks with its own code.

def pack_codes(codes, bits):
    """uint8 [rows, cols*bits/8] from one code per column, uint8 [rows, cols]."""
    codes = np.asarray(codes, dtype=np.uint8)
    per = 8 // bits
    rows, cols = codes.shape
    c = codes.reshape(rows, cols // per, per).astype(np.uint32)
    out = np.zeros((rows, cols // per), dtype=np.uint32)
    for i in range(per):
        out |= c[:, :, i] << np.uint32(bits * i)
    return out.astype(np.uint8)


# ------------------------------------------------------- wide-range inputs
# Activations whose magnitudes span many orders inside one group, with
# weights chosen so that rounding errors of small entries add up instead of
# cancelling.  They stand in for heavy-tailed residual streams and for
# hidden vectors SiLU(g) * u with g far below zero.

# magnitudes of the small entries of a 32-column block, relative to the
# block's largest |x|: just under half (or one and a half) of a rounding
# step at several resolutions, and just under a full step
SMALL_REL = (0.999 * 2.0 ** -18, 0.49999 * 2.0 ** -21, 0.49999 * 2.0 ** -22, 0.49999 * 2.0 ** -23,
             1.49999 * 2.0 ** -22, 0.9999 * 2.0 ** -22, 0.49999 * 2.0 ** -24, 0.3 * 2.0 ** -20)


def wide_range_x(n, seed, kind="blocks", tid=X_ID + 1, rel=None):
    """f32 [n] with a wide dynamic range.

    kind "blocks": in every block of 32 entries the first is +-2^k (k in
    -6..6, sometimes one unit of 2^-10 below a power of two) and the other
    31 are +-rel times it (rel=None: one of SMALL_REL per block).
    kind "outliers": standard normal with a few channels (0.2 %, at least
    4) multiplied by 1000.
    kind "near_zero": 95 % of the entries about 1e-6 (normal), the rest
    standard normal.
    """
    r = _rng(seed, tid)
    if kind == "blocks":
        x = np.empty(n, dtype=np.float64)
        for b0 in range(0, n, 32):
            k = int(r.integers(-6, 7))
            big = 2.0 ** k * (1.0 - 2.0 ** -10 if r.random() < 0.25 else 1.0)
            big *= 1.0 if r.random() < 0.5 else -1.0
            rb = SMALL_REL[(b0 // 32 + int(r.integers(0, 2))) % len(SMALL_REL)] if rel is None else rel
            m = min(32, n - b0)
            sgn = np.where(r.random(m) < 0.5, -1.0, 1.0)
            x[b0:b0 + m] = sgn * abs(big) * rb
            x[b0] = big
        return x.astype(np.float32)
    if kind == "outliers":
        x = r.standard_normal(n).astype(np.float32)
        k = max(4, n // 500)
        idx = r.choice(n, size=k, replace=False)
        x[idx] *= np.float32(1000.0)
        return x
    if kind == "near_zero":
        x = (r.standard_normal(n) * 1e-6).astype(np.float32)
        big = r.random(n) < 0.05
        x[big] = r.standard_normal(int(big.sum())).astype(np.float32)
        return x
    raise ValueError(kind)


def aligned_codes(rows, cols, bits, x, seed, tid):
    """uint8 [rows, cols] codes (one per column) against the activation x.

    The first column of every 32-column block (where wide_range_x puts the
    block's largest entry) gets a code next to the zero point (Q4: 7 or 8,
    Q2: 1 or 2: the smallest weight magnitude); every other column gets an
    extreme code (Q4: 0 or 15, Q2: 0 or 3).  Half of the rows take the
    extreme code whose weight has the sign of x there, so the rounding
    errors of the small entries all point the same way; a quarter take the
    opposite sign, a quarter a random one.
    """
    r = _rng(seed, tid)
    top = (1 << bits) - 1
    mid = (top - 1) // 2  # 7 (Q4) or 1 (Q2); mid + 1 is the other code next to Z
    pos = np.asarray(x, dtype=np.float64) >= 0
    codes = np.empty((rows, cols), dtype=np.uint8)
    for i in range(rows):
        mode = r.random()
        if mode < 0.5:
            hi = pos
        elif mode < 0.75:
            hi = ~pos
        else:
            hi = r.random(cols) < 0.5
        row = np.where(hi, top, 0).astype(np.uint8)
        row[0::32] = mid + r.integers(0, 2, size=row[0::32].shape[0])
        codes[i] = row
    return codes


def scales_mixed(rows, ngroups, seed, tid):
    """f32 [rows, ngroups]: each row's scales all 0.05 or all 1.0."""
    r = _rng(seed, tid)
    pick = np.where(r.random(rows) < 0.5, 0.05, 1.0).astype(np.float32)
    return np.repeat(pick[:, None], ngroups, axis=1)


def wide_range_expert(bits, d_model, d_ff, group, x, seed, e=0):
    """An expert whose gate/up codes are aligned against x and whose down
    codes are aligned against a wide-range vector of length d_ff drawn from
    the same seed (for calls that feed down a chosen input)."""
    base = 16 * e
    h = wide_range_x(d_ff, seed, "blocks", tid=X_ID + 7 + base)
    return {
        "gate_codes": pack_codes(aligned_codes(d_ff, d_model, bits, x, seed, base + GATE_CODES), bits),
        "gate_scales": scales_mixed(d_ff, d_model // group, seed, base + GATE_SCALES),
        "up_codes": pack_codes(aligned_codes(d_ff, d_model, bits, x, seed, base + UP_CODES), bits),
        "up_scales": scales_mixed(d_ff, d_model // group, seed, base + UP_SCALES),
        "down_codes": pack_codes(aligned_codes(d_model, d_ff, bits, h, seed, base + DOWN_CODES), bits),
        "down_scales": scales_mixed(d_model, d_ff // group, seed, base + DOWN_SCALES),
    }, h
