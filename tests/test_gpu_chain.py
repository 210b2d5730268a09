"""The configured chains as the pages run them: layers over segments, with the
memory rollover feeding the next segment's keys and values (CUDA, `-m gpu`).

Transformer-XL Section 3.2: the extended context of layer n in segment tau+1
is [SG(memory); h], where the memory is the newest M hidden states that layer
n saw in segment tau.  Section 3.3's procedure projects q from the segment's
states and k, v from the whole extended context, builds the relative table
from W_kR and the sinusoid, and attends.  Here every step of that per-layer
procedure runs in the library (txl_project_qkv, txl_project_heads, txl_rel_table, the
attention entry point, txl_rel_attn_fwd_mem or txl_mem_update, txl_ring_append); the glue between
layers, h^n = LayerNorm(a^{n-1} W_o + h^{n-1}), runs in torch and is not
checked.  Language-model initialisation: hidden states N(0, 1), weights and
biases N(0, 0.02^2).

Every layer call is checked against the oracle on sampled rows, fed that
call's exact device inputs (so errors do not compound across layers); the
projections of the rolled memory against the oracle's projections; each
rollover bit for bit against the oracle's rollover.  A second chain keeps
the memory as a ring and attends through txl_rel_attn_fwd_ring; it is
checked the same way.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, record_error
from transformer_xl_relative_rel_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

LAYERS, SEGMENTS = 2, 3
N_ROWS = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _bf16_close(got, ref):
    """A bf16 result of an fp32-accumulated float64 reference: within one
    bf16 unit in the last place of the reference, plus 1e-4 for the fp32
    accumulation of up to 1024 products of size ~0.02 (results near zero)."""
    return np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-4


def _sample(B, H, L, g):
    """Sampled (b, h, i) rows on two batch entries (first and last), so the
    oracle needs only those two sequences' keys and values."""
    bsel = sorted({0, B - 1})
    rows = np.stack([g.integers(0, len(bsel), N_ROWS), g.integers(0, H, N_ROWS), g.integers(0, L, N_ROWS)], 1)
    return bsel, rows.astype(np.int64)


def _check_attention(tag, q, k, v, r, u, w, out, D, M, g, kv_start=0):
    """Oracle rows for sampled (b, h, i) of one layer call on exactly the
    device values (first D columns of padded heads; k, v unrolled from a ring
    when kv_start is given)."""
    L, B, H, _ = q.shape
    T = k.shape[0]
    bsel, rows = _sample(B, H, L, g)
    idx = torch.tensor(bsel, device=q.device)
    order = (torch.arange(T, device=q.device) + kv_start) % T          # key j at ring row (start + j) mod T
    host = dict(q=q.index_select(1, idx)[..., :D], k=k.index_select(1, idx)[order][..., :D],
                v=v.index_select(1, idx)[order][..., :D], r=r[..., :D], u=u[..., :D], w=w[..., :D])
    host = {n: t.double().cpu().numpy() for n, t in host.items()}
    ref = oracle.rel_attn_rows(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"], mem_len=M,
                               rows=rows)
    o = out.index_select(1, idx)[..., :D].double().cpu().numpy()
    got = np.stack([o[i, b, h] for b, h, i in rows])
    err = np.abs(got - ref).max()
    record_error(tag, (B, H, D, L, M), err, TOL_BF16)
    assert np.isfinite(got).all() and err <= TOL_BF16, f"{tag}: max abs err {err:.3e}"
    return err


def _check_projection(tag, x, w, y, H, D, g):
    """Sampled rows of a projection against the oracle's float64 projection
    of the same bf16 inputs."""
    xf = x.reshape(-1, x.shape[-1])
    yf = y.reshape(xf.shape[0], H, -1)
    sel = torch.tensor(np.sort(g.choice(xf.shape[0], size=min(64, xf.shape[0]), replace=False)),
                       device=x.device)
    ref = oracle.project_heads(xf.index_select(0, sel).double().cpu().numpy(), w.double().cpu().numpy(), H, D,
                               yf.shape[-1])
    got = yf.index_select(0, sel).double().cpu().numpy()
    assert _bf16_close(got, ref).all(), f"{tag}: projection off by {np.abs(got - ref).max():.3e}"


class _Layer:
    def __init__(self, s, dp, gen, dev):
        H, D, dm = s.heads, s.d_head, s.d_model

        def wt(*shape):
            return (0.02 * torch.randn(*shape, generator=gen, device=dev)).bfloat16()
        self.wq, self.wk, self.wv, self.wr, self.wo = (wt(dm, dm) for _ in range(5))
        self.u = torch.zeros(H, dp, device=dev)
        self.w = torch.zeros(H, dp, device=dev)
        self.u[:, :D] = 0.02 * torch.randn(H, D, generator=gen, device=dev)
        self.w[:, :D] = 0.02 * torch.randn(H, D, generator=gen, device=dev)


def _glue(a, lay, h, s):
    """h^n = LayerNorm(a W_o + h^{n-1}) (the paper's Linear + residual +
    LayerNorm; no feed-forward), in torch: not part of the checked path."""
    L, B = h.shape[:2]
    a2 = a[..., :s.d_head].reshape(L, B, s.d_model).float()
    x = a2 @ lay.wo.float() + h.float()
    return torch.nn.functional.layer_norm(x, (s.d_model,)).bfloat16().contiguous()


@pytest.mark.parametrize("name", ["base_lm", "large_lm", "char_train", "char_eval"])
def test_chain_matches_oracle_every_call(name):
    import transformer_xl_relative_rel_gb300 as txl
    wl = WORKLOADS[name]
    s = wl.shape
    B, H, D, L, M, T, dm = s.batch, s.heads, s.d_head, s.seg_len, s.mem_len, s.klen, s.d_model
    dp = 64 if D != 64 else D                 # head vectors stored 64 wide (zeros past D)
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(wl.seed)
    g = np.random.Generator(np.random.PCG64(wl.seed + 17))
    layers = [_Layer(s, dp, gen, dev) for _ in range(LAYERS)]
    tables = [txl.rel_table(lay.wr, T, H, D, dp) for lay in layers]
    # initial memory (first segment): seeded N(0, 1) hidden states per layer
    ext = [torch.randn(T, B, dm, generator=gen, device=dev).bfloat16() for _ in range(LAYERS)]
    spare = [torch.empty_like(x) for x in ext]
    # the same chain with the memory as a ring of T rows (starts at row 0)
    ring = [x.clone() for x in ext]
    start = [0] * LAYERS

    def attend(q, k, v, r, lay, kv_start=None):
        if kv_start is None:
            if dp != D:
                return txl.rel_attn_fwd_padded(q, k, v, r, lay.u, lay.w, mem_len=M, d_head=D)
            return txl.rel_attn_fwd(q, k, v, r, lay.u, lay.w, mem_len=M)
        assert dp == D
        return txl.rel_attn_fwd_ring(q, k, v, r, lay.u, lay.w, mem_len=M, kv_start=kv_start)

    worst = 0.0
    for seg in range(SEGMENTS):
        h = torch.randn(L, B, dm, generator=gen, device=dev).bfloat16()   # the segment's input states
        h_ring = h
        for n, lay in enumerate(layers):
            # extended context [SG(memory); h]: the memory rows came from the
            # previous segment's rollover of this layer
            ext[n][M:].copy_(h)
            # q of the segment's rows M.., k and v of all rows: one call, as
            # the benchmark's recurrence makes it
            q, k, v = txl.project_qkv(ext[n], lay.wq, lay.wk, lay.wv, H, D, dp, q_from=M)
            if dp == D:
                # attention and the next segment's memory (newest M rows of
                # [memory; h]) in one call, as the benchmark's recurrence runs it
                a = txl.rel_attn_fwd_mem(q, k, v, tables[n], lay.u, lay.w, mem_len=M, mem_next=spare[n],
                                         ext_ctx=ext[n])
            else:
                a = attend(q, k, v, tables[n], lay)
            if seg > 0 and M > 0:
                # keys and values of the rolled memory
                _check_projection(f"{name} k(mem)", ext[n][:M], lay.wk, k[:M], H, D, g)
                _check_projection(f"{name} v(mem)", ext[n][:M], lay.wv, v[:M], H, D, g)
            worst = max(worst, _check_attention(f"chain_{name}", q, k, v, tables[n], lay.u, lay.w, a, D, M, g))
            # the memory for the next segment: newest M rows of [memory; h]
            if dp != D:
                txl.mem_update(spare[n], ext[n], mem_len=M)
            torch.cuda.synchronize()
            want = oracle.mem_update(ext[n].view(torch.int16).cpu().numpy(), M)
            assert np.array_equal(spare[n][:M].view(torch.int16).cpu().numpy(), want), f"{name}: rollover bits"
            ext[n], spare[n] = spare[n], ext[n]

            if dp == D:
                # ring: the segment's L rows replace the oldest L, in place
                st = start[n]
                txl.ring_append(ring[n], h_ring, (st + M) % T)
                kr = txl.project_heads(ring[n], lay.wk, H, D, dp)
                vr = txl.project_heads(ring[n], lay.wv, H, D, dp)
                qr = txl.project_heads(h_ring, lay.wq, H, D, dp)
                ar = attend(qr, kr, vr, tables[n], lay, kv_start=st)
                _check_attention(f"chain_ring_{name}", qr, kr, vr, tables[n], lay.u, lay.w, ar, D, M, g,
                                 kv_start=st)
                start[n] = (st + L) % T
                h_ring = _glue(ar, lay, h_ring, s)
            h = _glue(a, lay, h, s)
    assert worst <= TOL_BF16
