"""Writes tests/golden/tiny_siso_chain.txt: the oracle's output for the tiny
SISO workload (B1 L64 H2 G1 P16 N16 A8; packed projection ~N(0,1), dt_bias
~U(-4,-2), scan biases ~N(0, 0.1^2), D = 1, seeded as in
selective_state_space_mamba3_gb300.inputs), the preprocess chained into the
scan, in FP64.

The source pages print no worked numeric example of the scan (their tests
check shapes only), so this fixture is a regression pin: it freezes the
oracle's result for the tiny workload in text form, and
tests/test_oracle_pins.py checks that the oracle still reproduces it. It is
written from the oracle alone (and the seeded input generators), never from
the CUDA path:

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
FIXTURE = os.path.join(HERE, "tiny_siso_chain.txt")


def tiny_chain_output():
    """Oracle preprocess -> oracle SISO scan of the tiny workload, out [1, 64, 2, 16]."""
    sys.path.insert(0, ROOT)
    import oracle
    from selective_state_space_mamba3_gb300 import inputs as gen
    w = gen.TINY_SISO
    p = gen.tiny_projection(w)
    kw = dict(inner_size=32, state_size=16, num_heads=2, num_rope_angles=8, num_groups=1,
              mimo_rank=1, **gen.TINY_PRE)
    pre = oracle.preprocess(p["projected"], p["dt_bias"], **kw)
    shape = dict(x=(1, 64, 2, 16), z=(1, 64, 2, 16), bh=(1, 64, 1, 16), ch=(1, 64, 1, 16),
                 dt=(1, 64, 2), adt=(1, 64, 2), trap=(1, 64, 2), angle=(1, 64, 8))
    ins = {k: pre[k].astype(np.float32).reshape(shape[k]) for k in shape}
    return oracle.scan(w.cfg(), ins["ch"], ins["bh"], ins["x"], ins["z"], ins["adt"], ins["dt"],
                       ins["trap"], ins["angle"], p["c_bias"], p["b_bias"], p["d"])


def main():
    out = np.asarray(tiny_chain_output(), dtype=np.float64)
    with open(FIXTURE, "w") as f:
        f.write("# Oracle output of the tiny SISO workload (B1 L64 H2 G1 P16 N16 A8), preprocess\n")
        f.write("# chained into the scan, FP64; out[0, t, h, p] in row-major order, one value per\n")
        f.write("# line. Written by tests/golden/make_golden.py (oracle only).\n")
        for v in out.ravel():
            f.write("%.17g\n" % v)
    print(FIXTURE, out.size)


if __name__ == "__main__":
    main()
