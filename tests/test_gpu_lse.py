"""The forward's row log-sum-exp (txl_rel_attn_fwd_lse) and the backward that
takes it back with the saved output (txl_rel_attn_bwd with out and lse).

* lse against the oracle's float64 log of each row's softmax denominator, on
  ragged shapes, a head size that goes through the padded path, no memory, a
  single query row, and a memory long enough that the keys are split across
  CTAs (the partial results' combine writes lse there);
* the output of the lse call is bit-identical to the plain forward's;
* the backward fed the saved output and lse matches the oracle's gradients
  and the backward that runs its own forward.

Tolerance: lse compared as max|gpu - ref| / max(1, max|ref|) <= 2e-2, the
bf16 forward's bound (the scores are sums of bf16 products with fp32
accumulation; the log of the fp32 row sum adds a relative 1e-6).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import device_layer, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2
NAMES = ("dq", "dk", "dv", "dr", "du", "dw")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _rel_err(got, ref):
    return float(np.abs(got - ref).max() / max(1.0, np.abs(ref).max()))


def _fwd_lse(dev, B, H, L, M):
    import transformer_xl_relative_rel_gb300 as txl
    lse = torch.full((B, H, L), float("nan"), dtype=torch.float32, device="cuda")
    out = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M, lse=lse)
    return out, lse


@pytest.mark.parametrize("B,H,D,L,M", [
    (2, 3, 64, 150, 150),
    (1, 2, 41, 37, 50),        # head size 41: the zero-padded 64-wide copies
    (2, 2, 64, 130, 0),        # no memory
    (3, 2, 64, 1, 0),          # one query, one key: lse is that score
    (1, 2, 64, 64, 3000),      # long memory: keys split across CTAs
])
def test_lse_matches_oracle(B, H, D, L, M):
    import transformer_xl_relative_rel_gb300 as txl
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 900 + L + M)
    dev, host = device_layer(p, torch.bfloat16)
    out, lse = _fwd_lse(dev, B, H, L, M)
    plain = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    ref_out, ref_lse = oracle.rel_attn(**host, mem_len=M, return_lse=True)
    got = lse.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert _rel_err(got, ref_lse) <= TOL
    assert _rel_err(out.double().cpu().numpy(), ref_out) <= TOL


def _dout(shape, seed):
    g = inputs.rng(seed)
    t = torch.from_numpy(g.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
    return t.cuda(), t.double().numpy()


@pytest.mark.parametrize("B,H,D,L,M", [
    (2, 3, 64, 150, 150),
    (1, 2, 64, 64, 3000),
    (1, 2, 41, 40, 30),        # another head size: the saved pair is accepted and not needed
])
def test_bwd_with_saved_forward_matches_oracle(B, H, D, L, M):
    import transformer_xl_relative_rel_gb300 as txl
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 950 + L)
    dev, host = device_layer(p, torch.bfloat16)
    dout, dout_h = _dout((L, B, H, D), 951 + L)
    out, lse = _fwd_lse(dev, B, H, L, M)
    args = (dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], dout)
    saved = txl.rel_attn_bwd(*args, mem_len=M, out=out, lse=lse)
    again = txl.rel_attn_bwd(*args, mem_len=M)
    torch.cuda.synchronize()
    ref = oracle.rel_attn_bwd(**host, dout=dout_h, mem_len=M)
    for n in NAMES:
        a = saved[n].double().cpu().numpy()
        b = again[n].double().cpu().numpy()
        assert np.isfinite(a).all(), n
        assert _rel_err(a, ref[n]) <= TOL, n
        assert _rel_err(a, b) <= 1e-3, n


def test_bwd_with_saved_forward_char_train_shape():
    """B22 H8 D64 L768 M768: the saved pair gives the gradients of the
    recomputing backward."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, L, M = 22, 8, 64, 768, 768
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 15)
    dev, _ = device_layer(p, torch.bfloat16)
    dout, _ = _dout((L, B, H, D), 16)
    out, lse = _fwd_lse(dev, B, H, L, M)
    args = (dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], dout)
    saved = txl.rel_attn_bwd(*args, mem_len=M, out=out, lse=lse)
    again = txl.rel_attn_bwd(*args, mem_len=M)
    torch.cuda.synchronize()
    for n in NAMES:
        a = saved[n].double().cpu().numpy()
        assert np.isfinite(a).all(), n
        assert _rel_err(a, again[n].double().cpu().numpy()) <= 1e-3, n
