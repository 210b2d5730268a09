"""Calls on different streams run concurrently and stay correct.

txl_rel_attn_fwd keeps one library scratch buffer per (device, stream) for
its key-split partials and for 64-wide copies of odd head sizes.  Two
streams issue interleaved split-path calls with no synchronisation between
them; every result must match the oracle.  A stream that grows its buffer
(a larger shape after a smaller one) must not disturb the other stream's
calls in flight either.
"""
import numpy as np
import pytest
import torch

from tests.helpers import TOL_BF16, device_layer, oracle_full, record_error, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def test_two_streams_split_calls_concurrently():
    import transformer_xl_relative_rel_gb300 as txl
    # per stream: a small split shape first, then a larger one (the buffer
    # grows in that stream's order while the other stream is busy)
    shapes = {0: [(1, 2, 64, 128, 900), (1, 4, 64, 128, 1600)],
              1: [(2, 1, 41, 128, 700), (1, 3, 41, 130, 1500)]}
    for sid, lst in shapes.items():
        for (B, H, D, L, M) in lst:
            sp, _ = txl.rel_attn_fwd_plan(B, M, L, H, D, txl.TXL_BF16)
            assert sp > 1 or D != 64, f"{(B, H, D, L, M)} must take the split path"
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    cases = []
    for rep in range(3):
        for k in range(2):
            for sid in (0, 1):
                B, H, D, L, M = shapes[sid][k]
                p = inputs.unit_layer(unit_shape(B, H, D, L, M), 4000 + 10 * rep + 2 * k + sid)
                dev, host = device_layer(p, torch.bfloat16)
                cases.append((sid, dev, host, M))
    torch.cuda.synchronize()
    outs = []
    for sid, dev, host, M in cases:
        s = streams[sid]
        with torch.cuda.stream(s):
            out = torch.full_like(dev["q"], float("nan"))
            txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M,
                             out=out, stream=s)
        outs.append(out)
    torch.cuda.synchronize()
    txl.check()
    for (sid, dev, host, M), out in zip(cases, outs):
        want = oracle_full(host, M)
        err = np.abs(out.double().cpu().numpy() - want).max()
        record_error("two_streams", tuple(dev["q"].shape) + (M,), err, TOL_BF16)
        assert np.isfinite(err) and err <= TOL_BF16, f"stream {sid}: max abs err {err:.3e}"
