"""Write the stored expected values under tests/golden/ from the oracle alone.

The pages print no worked numeric example for the attention, so the stored
fixture is the oracle's own output on the tiny fp32 workload (seeded inputs
from transformer_xl_relative_rel_gb300.inputs).  It guards the oracle against
unnoticed changes; the oracle itself is pinned by tests/test_oracle_pins.py.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from transformer_xl_relative_rel_gb300 import inputs  # noqa: E402

SHAPE = inputs.LayerShape(batch=1, heads=2, d_head=16, seg_len=16, mem_len=16)
SEED = 1


def tiny_inputs():
    return inputs.unit_layer(SHAPE, SEED)


def main():
    p = tiny_inputs()
    out = oracle.rel_attn(p["q"], p["k"], p["v"], p["r"], p["u"], p["w"], mem_len=SHAPE.mem_len)
    path = os.path.join(HERE, "tiny_f32_out.txt")
    with open(path, "w") as f:
        f.write("# oracle output of the tiny fp32 workload: B1 H2 D16 L16 M16, seed 1,\n")
        f.write("# float32 unit-variance inputs (transformer_xl_relative_rel_gb300.inputs.unit_layer)\n")
        f.write("# written by tests/golden/make_golden.py; layout [L][B][H][D] flattened\n")
        for x in out.reshape(-1):
            f.write(f"{x:.17g}\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
