"""Parity of the CUDA relative attention against the oracle (float64).

Element by element on small seeded problems that span several tiles and a
ragged tail; on sampled rows at the full workload sizes, in the same launch
configuration the benchmark uses.  Tolerances: max |err| <= 1e-4 on the fp32
path, <= 2e-2 on the bf16 path with unit-variance inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import (TOL_BF16, TOL_F32, device_layer, gather_rows, oracle_full,
                           oracle_rows, record_error, run_library, unit_shape)
from transformer_xl_relative_rel_gb300 import inputs
from transformer_xl_relative_rel_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _check_full(B, H, D, L, M, dtype, seed, tol):
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), seed)
    dev, host = device_layer(p, dtype)
    out = run_library(dev, M)
    torch.cuda.synchronize()
    ref = oracle_full(host, M)
    got = out.double().cpu().numpy()
    err = np.abs(got - ref).max()
    record_error("full_" + ("f32" if dtype == torch.float32 else "bf16"), (B, H, D, L, M), err, tol)
    assert np.isfinite(got).all()
    assert err <= tol, f"max abs err {err:.3e} > {tol} for B{B} H{H} D{D} L{L} M{M} {dtype}"
    return err


# ------------------------------------------------------------------ fp32 path
@pytest.mark.parametrize("B,H,D,L,M", [
    (1, 2, 16, 16, 16),        # the tiny workload
    (2, 3, 24, 70, 45),        # several query blocks and key tiles, ragged tails
    (1, 2, 41, 37, 0),         # no memory
    (1, 1, 8, 1, 50),          # a single query sees all memory
    (1, 1, 128, 40, 30),       # widest head
    (1, 1, 1, 5, 3),           # d_head = 1
    (3, 1, 64, 33, 97),
])
def test_f32_parity(B, H, D, L, M):
    _check_full(B, H, D, L, M, torch.float32, seed=1000 + L + M, tol=TOL_F32)


def test_f32_tiny_workload_exact_inputs():
    w = WORKLOADS["tiny_f32"]
    s = w.shape
    p = inputs.unit_layer(s, w.seed)
    dev, host = device_layer(p, torch.float32)
    out = run_library(dev, s.mem_len)
    ref = oracle_full(host, s.mem_len)
    assert np.abs(out.double().cpu().numpy() - ref).max() <= TOL_F32


# ------------------------------------------------------------------ bf16 path
@pytest.mark.parametrize("B,H,D,L,M", [
    (1, 2, 64, 16, 16),
    (2, 2, 64, 200, 150),      # two query tiles (ragged), several key tiles
    (1, 3, 64, 300, 0),        # no memory: pure causal
    (1, 1, 64, 1, 300),        # one query over long memory
    (2, 2, 41, 150, 150),      # d_head 41: padded to 48, loaded without TMA
    (1, 2, 48, 130, 70),
    (1, 2, 40, 129, 127),      # d_head % 16 == 8: zero padding slice with TMA
    (1, 2, 32, 257, 31),
    (1, 2, 16, 64, 64),
    (1, 1, 24, 100, 20),
    (1, 2, 64, 128, 1600),     # long memory: keys split across CTAs + combine
    (2, 1, 41, 128, 900),      # split path without TMA
])
def test_bf16_parity(B, H, D, L, M):
    _check_full(B, H, D, L, M, torch.bfloat16, seed=2000 + L + M + D, tol=TOL_BF16)


def test_bf16_repeatable():
    """Same inputs, same bits: no races between the CTA's roles."""
    p = inputs.unit_layer(unit_shape(2, 2, 64, 200, 150), 7)
    dev, _ = device_layer(p, torch.bfloat16)
    a = run_library(dev, 150).clone()
    for _ in range(3):
        b = run_library(dev, 150)
        assert torch.equal(a, b)


# -------------------------------------------- full workload sizes, sampled rows
FULL = ["base_lm", "large_lm", "long_mem_b1", "long_mem_b16", "char_train", "char_eval"]


@pytest.mark.parametrize("name", FULL)
def test_bf16_full_size_unit_variance(name):
    w = WORKLOADS[name]
    s = w.shape
    p = inputs.unit_layer(s, w.seed)
    dev, host = device_layer(p, torch.bfloat16)
    out = run_library(dev, s.mem_len)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(s, w.seed, n_random=256, all_heads_of_b0=(s.heads * s.seg_len <= 4096))
    ref = oracle_rows(host, s.mem_len, rows)
    got = gather_rows(out, rows)
    err = np.abs(got - ref).max()
    record_error("full_size_unit_" + name, (s.batch, s.heads, s.d_head, s.seg_len, s.mem_len), err, TOL_BF16)
    assert err <= TOL_BF16, f"{name}: max abs err {err:.3e}"
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("B,H,L,M", [
    (2, 2, 3800, 0),     # the sliding-window recompute of bench.py --recompute-vs-reuse
    (2, 2, 128, 3800),   # its memory-reuse counterpart
])
def test_bf16_recompute_vs_reuse_shapes(B, H, L, M):
    """The two call shapes the recompute-vs-reuse measurement times, on
    unit-variance inputs, checked on sampled rows."""
    s = inputs.LayerShape(batch=B, heads=H, d_head=64, seg_len=L, mem_len=M)
    p = inputs.unit_layer(s, 900 + L)
    dev, host = device_layer(p, torch.bfloat16)
    out = run_library(dev, M)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(s, 900 + L, n_random=128, all_heads_of_b0=False)
    ref = oracle_rows(host, M, rows)
    err = np.abs(gather_rows(out, rows) - ref).max()
    record_error("recompute_vs_reuse", (B, H, 64, L, M), err, TOL_BF16)
    assert err <= TOL_BF16, f"max abs err {err:.3e}"


# ------------------------------------ absent biases: the Shaw et al. form
@pytest.mark.parametrize("dtype,tol,D", [(torch.float32, TOL_F32, 24), (torch.bfloat16, TOL_BF16, 64),
                                         (torch.bfloat16, TOL_BF16, 41)])
def test_absent_biases_are_the_shaw_form(dtype, tol, D):
    """u_bias = v_bias = None: terms (a) + (b) only.  Same bits as explicit
    zero biases, and the oracle with u = v = 0; one absent bias drops one term."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, L, M = 2, 2, 150, 140
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 4100 + D)
    dev, host = device_layer(p, dtype)
    zero = torch.zeros_like(dev["u"])
    got = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], None, None, mem_len=M).clone()
    same = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], zero, zero, mem_len=M)
    assert torch.equal(got, same)
    z = np.zeros_like(host["u"])
    ref = oracle.rel_attn(host["q"], host["k"], host["v"], host["r"], z, z, mem_len=M)
    assert np.abs(got.double().cpu().numpy() - ref).max() <= tol
    # only u absent: the global content bias (c) goes, (d) stays
    got_u = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], None, dev["w"], mem_len=M).clone()
    same_u = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], zero, dev["w"], mem_len=M)
    assert torch.equal(got_u, same_u)


# ------------------------------------------------ seeded random shape sweep
def _random_shapes(seed, n, dmax):
    g = np.random.Generator(np.random.PCG64(seed))
    ds = [d for d in (1, 5, 8, 16, 24, 32, 40, 41, 48, 56, 64, 96, 128) if d <= dmax]
    out = []
    for _ in range(n):
        out.append((int(g.integers(1, 4)), int(g.integers(1, 4)), int(g.choice(ds)),
                    int(g.integers(1, 301)), int(g.choice([0, int(g.integers(1, 450))]))))
    return out


@pytest.mark.parametrize("B,H,D,L,M", _random_shapes(31, 16, 64))
def test_bf16_random_shapes(B, H, D, L, M):
    """Shapes drawn from one seed (any head size up to 64, ragged lengths,
    with and without memory), element by element against the oracle."""
    _check_full(B, H, D, L, M, torch.bfloat16, seed=3000 + B * 131 + H * 17 + D * 7 + L + M, tol=TOL_BF16)


@pytest.mark.parametrize("B,H,D,L,M", _random_shapes(37, 6, 128))
def test_f32_random_shapes(B, H, D, L, M):
    _check_full(B, H, D, L, M, torch.float32, seed=4000 + B * 131 + H * 17 + D * 7 + L + M, tol=TOL_F32)


# ----------------------------------------------------- near the call's limits
@pytest.mark.parametrize("B,H,D,L,M,dtype", [
    (1, 2, 64, 128, 65536, torch.bfloat16),    # a 64K memory: the most key splits (16)
    (1, 64, 64, 256, 256, torch.bfloat16),     # many heads
    (1, 2, 128, 100, 60, torch.float32),       # the largest head size (fp32 path)
])
def test_near_limits_sampled_rows(B, H, D, L, M, dtype):
    import transformer_xl_relative_rel_gb300 as txl
    s = inputs.LayerShape(batch=B, heads=H, d_head=D, seg_len=L, mem_len=M)
    if dtype == torch.bfloat16:
        assert txl.rel_attn_fwd_plan(B, M, L, H, D, txl.TXL_BF16)[0] >= 1
    p = inputs.unit_layer(s, 1234 + H)
    dev, host = device_layer(p, dtype)
    out = run_library(dev, M)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    rows = inputs.sample_rows(s, 1234 + H, n_random=96, all_heads_of_b0=False)
    ref = oracle_rows(host, M, rows)
    err = np.abs(gather_rows(out, rows) - ref).max()
    record_error("near_limits", (B, H, D, L, M), err, TOL_BF16 if dtype == torch.bfloat16 else TOL_F32)
    assert err <= (TOL_BF16 if dtype == torch.bfloat16 else TOL_F32), f"max abs err {err:.3e}"


# ------------------------------------------------------------------ diagonal tiles
def _memory_below_segment(shape, seed):
    """Inputs whose memory keys point away from every query (logits near -8
    in the kernel's log2 units) and whose segment keys point along it (logits
    near +4): each row meets its first large logits on its diagonal tile,
    about 2^12 above the reference max its earlier tiles set.  The
    dominant logits stay small, so the bf16 roundings of the inputs keep the
    usual error scale."""
    L, B, H, D, M = shape.seg_len, shape.batch, shape.heads, shape.d_head, shape.mem_len
    T = M + L
    g = inputs.rng(seed)
    e = g.standard_normal((B, H, D)).astype(np.float32)
    e /= np.linalg.norm(e, axis=-1, keepdims=True)
    p = inputs.unit_layer(shape, seed)
    p["q"] = (4.0 * e[None] + 0.1 * g.standard_normal((L, B, H, D))).astype(np.float32)
    sign = np.where(np.arange(T) < M, -11.0, 5.5).astype(np.float32)[:, None, None, None]
    p["k"] = (sign * e[None] + 0.1 * g.standard_normal((T, B, H, D))).astype(np.float32)
    p["u"] = (0.1 * g.standard_normal((H, D))).astype(np.float32)
    p["w"] = (0.1 * g.standard_normal((H, D))).astype(np.float32)
    return p


@pytest.mark.parametrize("B,H,D,L,M", [
    (1, 2, 64, 128, 512),      # one query block, four memory tiles before its diagonal
    (2, 1, 64, 100, 300),      # ragged query block and key tail
    (1, 2, 64, 128, 2048),     # long memory: the planner splits the keys
])
def test_bf16_diagonal_raises_the_row_max(B, H, D, L, M):
    """Diagonal tiles run the straight exponential path once a row has a
    finite reference max; when their logits lie far above it the row-sum
    check must raise the reference (and rescale the accumulated output)."""
    shape = unit_shape(B, H, D, L, M)
    p = _memory_below_segment(shape, 4242 + L + M)
    dev, host = device_layer(p, torch.bfloat16)
    out = run_library(dev, M)
    torch.cuda.synchronize()
    ref = oracle_full(host, M)
    got = out.double().cpu().numpy()
    err = np.abs(got - ref).max()
    record_error("diag_raise_bf16", (B, H, D, L, M), err, TOL_BF16)
    assert np.isfinite(got).all()
    assert err <= TOL_BF16, f"max abs err {err:.3e} for B{B} H{H} D{D} L{L} M{M}"
