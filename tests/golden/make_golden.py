"""Writes q4_ffn_256_seed0.txt: the oracle's output for the one-token Q4
expert FFN with d_model = d_ff = 256, group 64, seed 0 (the small workload of
the S-MoE page "Metal Compute Kernels", section "Fused FFN Kernels -- One
Simdgroup Per Output Row", with synthetic inputs).

The stored values come from the oracle alone; the test that reads them
checks that later changes to the oracle leave this output as it was.
Run:  python -m tests.golden.make_golden
"""
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
PATH = os.path.join(HERE, "q4_ffn_256_seed0.txt")


def compute():
    import oracle
    import smoe_inputs as inp
    e = inp.expert(4, 256, 256, 64, seed=0)
    x = inp.activations(256, 0).astype(np.float64)
    hidden, out, out_abs = oracle.ffn(4, e["gate_codes"], e["gate_scales"], e["up_codes"],
                                      e["up_scales"], e["down_codes"], e["down_scales"],
                                      256, 256, 64, x)
    return {"hidden": hidden, "out": out, "out_abs": out_abs}


def write(path=PATH):
    vals = compute()
    with open(path, "w") as f:
        f.write("# oracle output, Q4 expert FFN d_model=256 d_ff=256 group=64 seed=0\n")
        f.write("# written by tests/golden/make_golden.py (calls only the oracle)\n")
        for key, arr in vals.items():
            f.write(f"{key} {arr.size}\n")
            f.write("\n".join(f"{v:.17g}" for v in arr) + "\n")


def read(path=PATH):
    out, key, n, buf = {}, None, 0, []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if key is None:
                key, n = line.split()[0], int(line.split()[1])
                buf = []
                continue
            buf.append(float(line))
            if len(buf) == n:
                out[key] = np.array(buf)
                key = None
    return out


if __name__ == "__main__":
    write()
    print(PATH)
