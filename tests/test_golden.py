"""The oracle still reproduces its stored output on the tiny fp32 workload."""
import os

import numpy as np

import oracle
from tests.golden.make_golden import SHAPE, tiny_inputs

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_golden(oracle_lib):
    ref = np.loadtxt(os.path.join(HERE, "golden", "tiny_f32_out.txt"))
    p = tiny_inputs()
    out = oracle.rel_attn(p["q"], p["k"], p["v"], p["r"], p["u"], p["w"], mem_len=SHAPE.mem_len)
    np.testing.assert_allclose(out.reshape(-1), ref, rtol=0, atol=1e-13)
