"""Parity of the CUDA backward (txl_rel_attn_bwd) against the oracle's
float64 gradients.

Element by element on small seeded problems (ragged lengths, odd head size,
no memory, absent biases); at the char_train training shape on one head's
slice over the whole batch (which also covers the batch sums of dr, du, dv
bias) plus the value-gradient identity on every head.

Tolerance: each gradient tensor is compared as max|gpu - ref| / max(1,
max|ref|).  fp32 path: 1e-4.  bf16 path: 2e-2 — the contractions take q+u,
q+v, P and dA rounded once to bf16 (relative error 2^-9 each) with fp32
accumulation, the same rounding budget as the forward's 2e-2 bound on
unit-variance inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import device_layer, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
NAMES = ("dq", "dk", "dv", "dr", "du", "dw")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _dout(shape, seed, dtype):
    g = inputs.rng(seed)
    d = g.standard_normal(shape, dtype=np.float32)
    t = torch.from_numpy(d).to(dtype)
    return t.cuda(), t.double().numpy()


def _rel_err(got, ref):
    return float(np.abs(got - ref).max() / max(1.0, np.abs(ref).max()))


def _run(B, H, D, L, M, dtype, seed, biases=True):
    import transformer_xl_relative_rel_gb300 as txl
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), seed)
    if not biases:
        p["u"][:] = 0.0
        p["w"][:] = 0.0
    dev, host = device_layer(p, dtype)
    dout, dout_h = _dout((L, B, H, D), seed + 1, dtype)
    g = txl.rel_attn_bwd(dev["q"], dev["k"], dev["v"], dev["r"],
                         dev["u"] if biases else None, dev["w"] if biases else None, dout, mem_len=M)
    torch.cuda.synchronize()
    got = {n: g[n].double().cpu().numpy() for n in NAMES}
    return got, host, dout_h


@pytest.mark.parametrize("B,H,D,L,M,dtype", [
    (1, 2, 16, 16, 16, torch.float32),        # the tiny configuration
    (2, 2, 41, 37, 50, torch.float32),        # odd head size, ragged lengths
    (2, 3, 64, 150, 150, torch.bfloat16),
    (2, 2, 41, 150, 150, torch.bfloat16),     # base-LM head size
    (1, 2, 64, 130, 0, torch.bfloat16),       # no memory
    (3, 2, 32, 20, 300, torch.bfloat16),      # memory much longer than the segment
])
def test_bwd_matches_oracle(B, H, D, L, M, dtype):
    got, host, dout = _run(B, H, D, L, M, dtype, seed=1000 + B * 7 + D)
    ref = oracle.rel_attn_bwd(**host, dout=dout, mem_len=M)
    errs = {n: _rel_err(got[n], ref[n]) for n in NAMES}
    for n in NAMES:
        assert np.isfinite(got[n]).all(), n
        assert errs[n] <= TOL[dtype], f"{n}: {errs[n]:.3e} > {TOL[dtype]} ({errs})"


def test_bwd_absent_biases_are_zero_biases():
    B, H, D, L, M = 2, 2, 64, 70, 90
    got, host, dout = _run(B, H, D, L, M, torch.bfloat16, seed=77, biases=False)
    ref = oracle.rel_attn_bwd(**host, dout=dout, mem_len=M)   # host biases are zero
    for n in NAMES:
        assert _rel_err(got[n], ref[n]) <= TOL[torch.bfloat16], n


def test_bwd_char_train_shape_one_head_slice():
    """B22 H8 D64 L768 M768 (the training shape, the launch the benchmark
    times): head 5 over the whole batch against the oracle, and on every
    head the identity sum_j dv_j = sum_i dout_i (the weights of a row sum to
    one)."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, L, M = 22, 8, 64, 768, 768
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 5)
    dev, host = device_layer(p, torch.bfloat16)
    dout, dout_h = _dout((L, B, H, D), 6, torch.bfloat16)
    g = txl.rel_attn_bwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], dout, mem_len=M)
    torch.cuda.synchronize()
    h = 5
    sl = {n: host[n][:, :, h:h + 1] for n in ("q", "k", "v")}
    sl["r"] = host["r"][:, h:h + 1]
    sl["u"] = host["u"][h:h + 1]
    sl["w"] = host["w"][h:h + 1]
    ref = oracle.rel_attn_bwd(**sl, dout=dout_h[:, :, h:h + 1], mem_len=M)
    got = {n: g[n].double().cpu().numpy() for n in NAMES}
    pick = dict(dq=got["dq"][:, :, h:h + 1], dk=got["dk"][:, :, h:h + 1], dv=got["dv"][:, :, h:h + 1],
                dr=got["dr"][:, h:h + 1], du=got["du"][h:h + 1], dw=got["dw"][h:h + 1])
    for n in NAMES:
        assert np.isfinite(got[n]).all(), n
        assert _rel_err(pick[n], ref[n]) <= TOL[torch.bfloat16], n
    colsum = got["dv"].sum(axis=0)
    assert _rel_err(colsum, dout_h.sum(axis=0)) <= TOL[torch.bfloat16]


def _random_shapes(seed, n):
    g = np.random.Generator(np.random.PCG64(seed))
    return [(int(g.integers(1, 3)), int(g.integers(1, 3)), int(g.choice([8, 16, 41, 64])),
             int(g.integers(1, 160)), int(g.choice([0, int(g.integers(1, 220))])),
             [torch.float32, torch.bfloat16][int(g.integers(0, 2))]) for _ in range(n)]


@pytest.mark.parametrize("B,H,D,L,M,dtype", _random_shapes(41, 6))
def test_bwd_random_shapes(B, H, D, L, M, dtype):
    got, host, dout = _run(B, H, D, L, M, dtype, seed=5000 + B * 13 + H * 7 + D + L + M)
    ref = oracle.rel_attn_bwd(**host, dout=dout, mem_len=M)
    for n in NAMES:
        assert np.isfinite(got[n]).all(), n
        assert _rel_err(got[n], ref[n]) <= TOL[dtype], n
