"""Projections into the attention layout, the device-built relative table and
attention on padded heads (CUDA, `-m gpu`).  References: the oracle's float64
projections and table on exactly the values the device read, and its
attention."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, TOL_F32
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu


def _rel_err(got, ref):
    return np.abs(got - ref).max() / max(1e-12, np.abs(ref).max())


def _bf16_close(got, ref, d_in):
    """bf16 output of an fp32-accumulated product: one bf16 unit in the last
    place of the reference plus the fp32 accumulation error of d_in terms."""
    return np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6 * np.sqrt(d_in) * (1 + np.abs(ref))


@pytest.mark.parametrize("dtype,rtol", [(torch.float32, 1e-5), (torch.bfloat16, 1e-2)])
@pytest.mark.parametrize("rows,d_in,heads,d_head,d_pad", [(300, 410, 10, 41, 64), (96, 64, 2, 32, 32),
                                                          (7, 24, 3, 5, 8)])
def test_project_heads(dtype, rtol, rows, d_in, heads, d_head, d_pad):
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(rows + d_in)
    x = torch.randn(rows, d_in, generator=g, device="cuda").to(dtype)
    w = (0.05 * torch.randn(heads * d_head, d_in, generator=g, device="cuda")).to(dtype)
    y = txl.project_heads(x, w, heads, d_head, d_pad)
    ref = oracle.project_heads(x.double().cpu().numpy(), w.double().cpu().numpy(), heads, d_head, d_pad)
    got = y.double().cpu().numpy()
    assert _rel_err(got[..., :d_head], ref[..., :d_head]) <= rtol
    assert (got[..., d_head:] == 0).all()


# the tensor-core GEMM: several 128-row tiles with a ragged last one, K tails
# (d_in not a multiple of 64), one and several 256-column tiles, padded heads,
# TMA operand loads (d_in % 8 == 0) and the cp.async loaders (d_in % 8 != 0)
@pytest.mark.parametrize("rows,d_in,heads,d_head,d_pad", [
    (1000, 512, 8, 64, 64),       # char-LM head shape, two 256-column tiles
    (777, 1024, 16, 64, 64),      # large-LM, four column tiles, ragged rows
    (300, 410, 10, 41, 64),       # base-LM: cp.async loaders (row pitch 820 bytes), padded heads
    (129, 96, 3, 32, 32),         # one 96-column tile, K tail
    (50, 200, 5, 48, 48),         # 240 columns, 48-wide heads (TMA box of 5 heads)
    (130, 66, 4, 20, 24),         # cp.async, heads padded 20 -> 24, output rows 192 bytes
    (5, 16, 1, 16, 16),           # a single small tile
])
def test_project_heads_tensor_core(rows, d_in, heads, d_head, d_pad):
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(7 * rows + d_in)
    x = torch.randn(rows, d_in, generator=g, device="cuda").bfloat16()
    w = (0.02 * torch.randn(heads * d_head, d_in, generator=g, device="cuda")).bfloat16()
    y = torch.full((rows, heads, d_pad), float("nan"), dtype=torch.bfloat16, device="cuda")
    txl.project_heads(x, w, heads, d_head, d_pad, out=y)
    ref = oracle.project_heads(x.double().cpu().numpy(), w.double().cpu().numpy(), heads, d_head, d_pad)
    got = y.double().cpu().numpy()
    assert np.isfinite(got).all()
    assert _bf16_close(got, ref, d_in).all(), f"max abs err {np.abs(got - ref).max():.3e}"
    assert (got[..., d_head:] == 0).all()
    # the same product again (the pipeline's barriers restart cleanly)
    y2 = txl.project_heads(x, w, heads, d_head, d_pad)
    assert torch.equal(y, y2)


# the layer's three projections from one extended context [M+L, B, d_in]:
# the fused launch (x read once; q's rows start a 128-row block), the fused
# launch with q's rows as a band of their own (q's first row inside a
# block), and shapes that take one launch per product (cp.async rows, fp32);
# every case against the oracle and bit for bit against three project_heads
# calls
@pytest.mark.parametrize("dtype,T,B,M,d_in,heads,d_head,d_pad", [
    (torch.bfloat16, 384, 2, 256, 512, 8, 64, 64),    # q from row 512: fused q, k, v
    (torch.bfloat16, 200, 3, 72, 256, 4, 64, 64),     # q from row 216 (inside a block): q's own band
    (torch.bfloat16, 150, 3, 50, 256, 16, 64, 64),    # q's own band from row 150, four column tiles
    (torch.bfloat16, 97, 3, 32, 512, 8, 64, 64),      # ragged last block (291 rows), q from row 96
    (torch.bfloat16, 160, 2, 64, 1024, 16, 64, 64),   # four column tiles per product
    (torch.bfloat16, 150, 2, 100, 410, 10, 41, 64),   # cp.async rows: three launches
    (torch.bfloat16, 64, 2, 0, 128, 2, 48, 48),       # no memory: q over all rows
    (torch.bfloat16, 200, 1, 128, 64, 1, 16, 16),     # q fused: one partial row block, a 16-wide output
    (torch.float32, 40, 2, 24, 64, 2, 16, 16),        # fp32: the CUDA-core kernel three times
])
def test_project_qkv(dtype, T, B, M, d_in, heads, d_head, d_pad):
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(T * 31 + d_in)
    x = torch.randn(T, B, d_in, generator=g, device="cuda").to(dtype)
    ws = [(0.02 * torch.randn(heads * d_head, d_in, generator=g, device="cuda")).to(dtype) for _ in range(3)]
    nan = float("nan")
    q = torch.full((T - M, B, heads, d_pad), nan, dtype=dtype, device="cuda")
    k = torch.full((T, B, heads, d_pad), nan, dtype=dtype, device="cuda")
    v = torch.full((T, B, heads, d_pad), nan, dtype=dtype, device="cuda")
    txl.project_qkv(x, ws[0], ws[1], ws[2], heads, d_head, d_pad, q_from=M, q=q, k=k, v=v)
    xd = x.double().cpu().numpy().reshape(T * B, d_in)
    for name, got, xr, w in (("q", q, xd[M * B:], ws[0]), ("k", k, xd, ws[1]), ("v", v, xd, ws[2])):
        ref = oracle.project_heads(xr, w.double().cpu().numpy(), heads, d_head, d_pad)
        gn = got.double().cpu().numpy().reshape(ref.shape)
        assert np.isfinite(gn).all(), name
        if dtype == torch.bfloat16:
            assert _bf16_close(gn, ref, d_in).all(), f"{name}: max abs err {np.abs(gn - ref).max():.3e}"
        else:
            assert _rel_err(gn, ref) <= 1e-5, name
        assert (gn[..., d_head:] == 0).all(), name
    assert torch.equal(q, txl.project_heads(x[M:], ws[0], heads, d_head, d_pad))
    assert torch.equal(k, txl.project_heads(x, ws[1], heads, d_head, d_pad))
    assert torch.equal(v, txl.project_heads(x, ws[2], heads, d_head, d_pad))
    # without q, and with no q rows
    q2, k2, v2 = txl.project_qkv(x, None, ws[1], ws[2], heads, d_head, d_pad)
    assert q2 is None and torch.equal(k2, k) and torch.equal(v2, v)
    q3, k3, v3 = txl.project_qkv(x, ws[0], ws[1], ws[2], heads, d_head, d_pad, q_from=T)
    assert q3.shape[0] == 0 and torch.equal(k3, k) and torch.equal(v3, v)


def test_project_qkv_full_size_sampled_rows():
    """char-LM training's layer inputs as the recurrence runs them (T = 1536,
    B = 22, q from the memory's end, row 16,896): one fused launch; sampled
    rows of each product against the oracle."""
    import transformer_xl_relative_rel_gb300 as txl
    T, B, M, dm, H, D = 1536, 22, 768, 512, 8, 64
    g = torch.Generator(device="cuda").manual_seed(1536)
    x = torch.randn(T, B, dm, generator=g, device="cuda").bfloat16()
    ws = [(0.02 * torch.randn(H * D, dm, generator=g, device="cuda")).bfloat16() for _ in range(3)]
    q, k, v = txl.project_qkv(x, ws[0], ws[1], ws[2], H, D, D, q_from=M)
    rng = np.random.Generator(np.random.PCG64(2))
    xf = x.reshape(T * B, dm)
    for got, lo, w in ((q, M * B, ws[0]), (k, 0, ws[1]), (v, 0, ws[2])):
        sel = rng.choice(T * B - lo, 128, replace=False)
        idx = torch.tensor(sel, device="cuda")
        ref = oracle.project_heads(xf[lo:][idx].double().cpu().numpy(), w.double().cpu().numpy(), H, D)
        gn = got.reshape(-1, H, D)[idx].double().cpu().numpy()
        assert _bf16_close(gn, ref, dm).all(), f"max abs err {np.abs(gn - ref).max():.3e}"


def test_project_heads_padding_stays_zero_with_inf_inputs():
    """Padding columns are written as zeros, not as products with zero
    weights (an infinite input would make those NaN)."""
    import transformer_xl_relative_rel_gb300 as txl
    x = torch.randn(256, 128, device="cuda").bfloat16()
    x[3, 5] = float("inf")
    w = (0.02 * torch.randn(4 * 24, 128, device="cuda")).bfloat16()
    y = txl.project_heads(x, w, 4, 24, 32)
    assert (y[..., 24:] == 0).all()


def test_project_heads_full_size_sampled_rows():
    """char-LM evaluation's k projection: [M+L]*B = 86,416 rows of 512, as the
    chain runs it; sampled rows against the oracle."""
    import transformer_xl_relative_rel_gb300 as txl
    T, B, dm, H, D = 3928, 22, 512, 8, 64
    g = torch.Generator(device="cuda").manual_seed(3928)
    x = torch.randn(T, B, dm, generator=g, device="cuda").bfloat16()
    w = (0.02 * torch.randn(H * D, dm, generator=g, device="cuda")).bfloat16()
    y = txl.project_heads(x, w, H, D, D)
    sel = np.random.Generator(np.random.PCG64(1)).choice(T * B, 256, replace=False)
    xs = x.reshape(T * B, dm)[torch.tensor(sel, device="cuda")].double().cpu().numpy()
    ref = oracle.project_heads(xs, w.double().cpu().numpy(), H, D)
    got = y.reshape(T * B, H, D)[torch.tensor(sel, device="cuda")].double().cpu().numpy()
    assert _bf16_close(got, ref, dm).all(), f"max abs err {np.abs(got - ref).max():.3e}"


@pytest.mark.parametrize("dtype,rtol", [(torch.float32, 2e-4), (torch.bfloat16, 1e-2)])
@pytest.mark.parametrize("klen,d_model,heads,d_head,d_pad", [(300, 410, 10, 41, 64), (1536, 512, 8, 64, 64),
                                                             (33, 20, 2, 10, 16)])
def test_rel_table(dtype, rtol, klen, d_model, heads, d_head, d_pad):
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(klen + d_model)
    w_r = (0.02 * torch.randn(heads * d_head, d_model, generator=g, device="cuda")).to(dtype)
    r = txl.rel_table(w_r, klen, heads, d_head, d_pad)
    ref = oracle.rel_table(w_r.double().cpu().numpy(), klen, heads, d_head, d_pad)   # row t: distance klen-1-t
    got = r.double().cpu().numpy()
    assert _rel_err(got[..., :d_head], ref[..., :d_head]) <= rtol
    assert (got[..., d_head:] == 0).all()


@pytest.mark.parametrize("dtype,tol,B,H,D,Dp,L,M", [
    (torch.bfloat16, TOL_BF16, 2, 3, 41, 64, 150, 150),   # base-LM head size, TMA on the padded rows
    (torch.bfloat16, TOL_BF16, 2, 2, 41, 48, 130, 70),    # padded to 48: thread loads
    (torch.bfloat16, TOL_BF16, 1, 2, 20, 32, 64, 200),
    (torch.float32, TOL_F32, 1, 2, 13, 16, 40, 24),
])
def test_padded_attention_matches_unpadded(dtype, tol, B, H, D, Dp, L, M):
    import transformer_xl_relative_rel_gb300 as txl
    p = inputs.unit_layer(inputs.LayerShape(B, H, D, L, M), 6000 + D + Dp)

    def padded(a):
        z = np.zeros(a.shape[:-1] + (Dp,), dtype=np.float32)
        z[..., :D] = a
        return torch.from_numpy(z)
    dev = {n: padded(p[n]).to(dtype).cuda() for n in ("q", "k", "v", "r")}
    for n in ("u", "w"):
        dev[n] = padded(p[n]).float().cuda()
    out = txl.rel_attn_fwd_padded(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M,
                                  d_head=D)
    host = {n: dev[n][..., :D].double().cpu().numpy() for n in ("q", "k", "v", "r", "u", "w")}
    ref = oracle.rel_attn(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"], mem_len=M)
    got = out.double().cpu().numpy()
    assert np.abs(got[..., :D] - ref).max() <= tol
    assert (got[..., D:] == 0).all()


def test_layer_from_hidden_states():
    """Hidden states -> projections + table (d_head 41 padded to 64) -> padded
    attention, against the oracle on the projected values."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, Dp, L, M = 2, 10, 41, 64, 150, 150
    T, dm = M + L, H * D
    g = torch.Generator(device="cuda").manual_seed(41)
    h_ext = torch.randn(T, B, dm, generator=g, device="cuda").bfloat16()
    wq, wk, wv, wr = ((0.05 * torch.randn(dm, dm, generator=g, device="cuda")).bfloat16() for _ in range(4))
    u = 0.02 * torch.randn(H, Dp, generator=g, device="cuda")
    w = 0.02 * torch.randn(H, Dp, generator=g, device="cuda")
    u[:, D:] = 0
    w[:, D:] = 0
    q = txl.project_heads(h_ext[M:].contiguous(), wq, H, D, Dp)
    k = txl.project_heads(h_ext, wk, H, D, Dp)
    v = txl.project_heads(h_ext, wv, H, D, Dp)
    r = txl.rel_table(wr, T, H, D, Dp)
    out = txl.rel_attn_fwd_padded(q, k, v, r, u, w, mem_len=M, d_head=D)
    host = {n: t[..., :D].double().cpu().numpy() for n, t in (("q", q), ("k", k), ("v", v), ("r", r),
                                                               ("u", u), ("w", w))}
    ref = oracle.rel_attn(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"], mem_len=M)
    assert np.abs(out[..., :D].double().cpu().numpy() - ref).max() <= TOL_BF16


@pytest.mark.parametrize("cells,T,B,M,d_in,heads,with_q", [
    (3, 384, 2, 256, 512, 8, True),      # one grouped launch, q fused
    (10, 200, 3, 128, 256, 4, True),     # two launches (8 + 2 cells)
    (4, 160, 2, 64, 1024, 16, False),    # k and v only
    (3, 200, 3, 72, 256, 4, True),       # q's first row inside a block: q's own band in each cell
])
def test_project_qkv_cells_equals_per_cell(cells, T, B, M, d_in, heads, with_q):
    """Several layer calls' projections in grouped launches: every output bit
    for bit what project_qkv gives cell by cell (the oracle checks of
    project_qkv above cover the values)."""
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(cells * 101 + T)
    xs = [torch.randn(T, B, d_in, generator=g, device="cuda").bfloat16() for _ in range(cells)]
    mk = lambda: [(0.02 * torch.randn(heads * 64, d_in, generator=g, device="cuda")).bfloat16() for _ in range(cells)]
    wqs, wks, wvs = (mk() if with_q else None), mk(), mk()
    qs, ks, vs = txl.project_qkv_cells(xs, wqs, wks, wvs, heads, 64, 64, q_from=M)
    for c in range(cells):
        q1, k1, v1 = txl.project_qkv(xs[c], wqs[c] if with_q else None, wks[c], wvs[c], heads, 64, 64, q_from=M)
        assert torch.equal(ks[c], k1) and torch.equal(vs[c], v1), c
        if with_q:
            assert torch.equal(qs[c], q1), c
    if not with_q:
        assert qs is None
