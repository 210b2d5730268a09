"""The Python binding's argument checks, on the host: wrong shapes, dtypes,
devices and pairings are refused with an exception before the library is
called (these checks are what stands between a caller's tensors and the raw
pointers the C ABI receives).  Host tensors stand in for device tensors: the
shape and dtype checks come before the device check, and the device check
itself is one of the refusals tested.  No compute call is made."""
import pytest
import torch

import transformer_xl_relative_rel_gb300 as txl
from transformer_xl_relative_rel_gb300 import abi

L, B, H, D, M = 8, 2, 2, 16, 8
T = L + M
ON_DEVICE = "contiguous CUDA tensors"


def _layer(dtype=torch.bfloat16):
    return dict(q=torch.zeros(L, B, H, D, dtype=dtype), k=torch.zeros(T, B, H, D, dtype=dtype),
                v=torch.zeros(T, B, H, D, dtype=dtype), r=torch.zeros(T, H, D, dtype=dtype),
                u=torch.zeros(H, D), w=torch.zeros(H, D))


def test_attention_shape_dtype_and_device_checks():
    p = _layer()
    q, k, v, r, u, w = (p[n] for n in ("q", "k", "v", "r", "u", "w"))
    with pytest.raises(ValueError, match="k must be"):
        txl.rel_attn_fwd(q, k[:-1], v, r, u, w, mem_len=M)          # k one row short
    with pytest.raises(ValueError, match="r must be"):
        txl.rel_attn_fwd(q, k, v, r[:, :1], u, w, mem_len=M)         # table heads
    with pytest.raises(ValueError, match="k must be"):
        txl.rel_attn_fwd(q, k, v, r, u, w, mem_len=M + 1)            # memory length against k
    with pytest.raises(TypeError, match="dtype"):
        txl.rel_attn_fwd(q, k.float(), v, r, u, w, mem_len=M)        # mixed dtypes
    with pytest.raises(ValueError, match="u_bias"):
        txl.rel_attn_fwd(q, k, v, r, u.double(), w, mem_len=M)       # bias dtype
    with pytest.raises(ValueError, match="v_bias"):
        txl.rel_attn_fwd(q, k, v, r, u, w[:1], mem_len=M)            # bias shape
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.rel_attn_fwd(q, k, v, r, u, w, mem_len=M)                # host tensors
    for fn, extra in ((txl.rel_attn_fwd_mem, dict(mem_next=torch.zeros(T, B, 32, dtype=torch.bfloat16),
                                                  ext_ctx=torch.zeros(T, B, 32, dtype=torch.bfloat16))),
                      (txl.rel_attn_bwd, dict(dout=torch.zeros(L, B, H, D, dtype=torch.bfloat16)))):
        with pytest.raises(ValueError, match="k must be"):          # the attention's checks come first
            fn(q, k[:-1], v, r, u, w, mem_len=M, **extra)
        with pytest.raises(ValueError, match=ON_DEVICE):
            fn(q, k, v, r, u, w, mem_len=M, **extra)
    with pytest.raises(TypeError, match="unsupported dtype"):
        abi._dtype_code(torch.zeros(1, dtype=torch.float16))         # no fp16 path


def test_rollover_checks():
    ext = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="larger than the extended context"):
        txl.mem_update(torch.zeros(T, B, 32, dtype=torch.bfloat16), ext, mem_len=T + 1)
    with pytest.raises(ValueError, match="mem_next must be"):
        txl.mem_update(torch.zeros(M, B, 31, dtype=torch.bfloat16), ext, mem_len=M)
    with pytest.raises(ValueError, match="mem_next must be"):
        txl.mem_update(torch.zeros(M - 1, B, 32, dtype=torch.bfloat16), ext, mem_len=M)
    with pytest.raises(TypeError, match="dtypes differ"):
        txl.mem_update(torch.zeros(M, B, 32, dtype=torch.float32), ext, mem_len=M)
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.mem_update(torch.zeros(M, B, 32, dtype=torch.bfloat16), ext, mem_len=M)


def test_plan_query_rejects_bad_shapes():
    from transformer_xl_relative_rel_gb300 import _build
    _build.build()                      # the query runs in the library (no GPU needed)
    txl.load_library()
    with pytest.raises(txl.TxlError, match="invalid"):
        txl.rel_attn_fwd_plan(1, -1, 16, 2, 64, txl.TXL_BF16)
    with pytest.raises(txl.TxlError, match="unsupported"):
        txl.rel_attn_fwd_plan(1, 16, 16, 2, 65, txl.TXL_BF16)        # bf16 head size past 64


def test_noalloc_binding_checks_like_the_default_entry():
    # the no-alloc entry point refuses what rel_attn_fwd refuses, and also a
    # missing output (it would have to allocate one)
    p = _layer()
    q, k, v, r, u, w = (p[n] for n in ("q", "k", "v", "r", "u", "w"))
    out = torch.zeros_like(q)
    with pytest.raises(ValueError, match="out must be given"):
        txl.rel_attn_fwd_noalloc(q, k, v, r, u, w, mem_len=M, out=None)
    with pytest.raises(ValueError, match="k must be"):
        txl.rel_attn_fwd_noalloc(q, k[:-1], v, r, u, w, mem_len=M, out=out)
    with pytest.raises(ValueError, match="k must be"):
        txl.rel_attn_fwd_noalloc(q, k, v, r, u, w, mem_len=M + 1, out=out)
    with pytest.raises(TypeError, match="dtype"):
        txl.rel_attn_fwd_noalloc(q, k, v.float(), r, u, w, mem_len=M, out=out)
    with pytest.raises(ValueError, match="u_bias"):
        txl.rel_attn_fwd_noalloc(q, k, v, r, u[:, :1], w, mem_len=M, out=out)
    with pytest.raises(ValueError, match="out must be"):
        txl.rel_attn_fwd_noalloc(q, k, v, r, u, w, mem_len=M, out=out[:1])
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.rel_attn_fwd_noalloc(q, k, v, r, u, w, mem_len=M, out=out)
    r_strided = torch.zeros(T, D, H, dtype=r.dtype).transpose(1, 2)     # right shape, not contiguous
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.rel_attn_fwd_noalloc(q, k, v, r_strided, u, w, mem_len=M, out=out)


def test_project_qkv_checks():
    d_in, heads, d_head, d_pad = 32, 2, 16, 16
    x = torch.zeros(T, B, d_in, dtype=torch.bfloat16)
    w = [torch.zeros(heads * d_head, d_in, dtype=torch.bfloat16) for _ in range(3)]
    with pytest.raises(ValueError, match="q_from"):
        txl.project_qkv(x, w[0], w[1], w[2], heads, d_head, d_pad, q_from=T + 1)
    with pytest.raises(ValueError, match="w_k must be"):
        txl.project_qkv(x, w[0], w[1][:, :-1], w[2], heads, d_head, d_pad, q_from=M)   # contraction length
    with pytest.raises(ValueError, match="w_v is required"):
        txl.project_qkv(x, w[0], w[1], None, heads, d_head, d_pad, q_from=M)
    with pytest.raises(ValueError, match="w_q must be"):
        txl.project_qkv(x, w[0].float(), w[1], w[2], heads, d_head, d_pad, q_from=M)  # weight dtype
    with pytest.raises(ValueError, match="q is given without w_q"):
        txl.project_qkv(x, None, w[1], w[2], heads, d_head, d_pad, q=torch.zeros(L, B, heads, d_pad))
    with pytest.raises(ValueError, match="q must be"):                                # q spans L rows, not T
        txl.project_qkv(x, w[0], w[1], w[2], heads, d_head, d_pad, q_from=M,
                        q=torch.zeros(T, B, heads, d_pad, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="k must be"):                                # padded width
        txl.project_qkv(x, w[0], w[1], w[2], heads, d_head, d_pad, q_from=M,
                        k=torch.zeros(T, B, heads, d_pad + 8, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.project_qkv(x, w[0], w[1], w[2], heads, d_head, d_pad, q_from=M)          # host tensors


def test_project_qkv_cells_checks():
    d_in, heads, d_head, d_pad = 32, 2, 16, 16
    xs = [torch.zeros(T, B, d_in, dtype=torch.bfloat16) for _ in range(2)]
    ws = [torch.zeros(heads * d_head, d_in, dtype=torch.bfloat16) for _ in range(2)]
    with pytest.raises(ValueError, match="same length"):
        txl.project_qkv_cells(xs, ws, ws[:1], ws, heads, d_head, d_pad, q_from=M)
    with pytest.raises(ValueError, match="first cell's shape"):
        txl.project_qkv_cells([xs[0], xs[1][:, :1]], ws, ws, ws, heads, d_head, d_pad, q_from=M)
    with pytest.raises(ValueError, match="w_k must be"):                                # a cell's weight
        txl.project_qkv_cells(xs, ws, [ws[0][:, :-1], ws[1]], ws, heads, d_head, d_pad, q_from=M)
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.project_qkv_cells(xs, ws, ws, ws, heads, d_head, d_pad, q_from=M)
    assert txl.project_qkv_cells([], None, [], [], heads, d_head, d_pad) == ([], [], [])


def test_rel_attn_fwd_mem_cells_checks():
    t = _layer()
    ext = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    nxt = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    one = lambda key: [t[key], t[key]]
    with pytest.raises(ValueError, match="same length"):
        txl.rel_attn_fwd_mem_cells(one("q"), one("k"), one("v"), one("r"), one("u"), [t["w"]], M, [nxt, nxt],
                                   [ext, ext])
    with pytest.raises(ValueError, match="first call's shape"):
        txl.rel_attn_fwd_mem_cells([t["q"], t["q"][:1]], one("k"), one("v"), one("r"), one("u"), one("w"), M,
                                   [nxt, nxt], [ext, ext])
    with pytest.raises(ValueError, match="ext_ctx must be"):
        txl.rel_attn_fwd_mem_cells(one("q"), one("k"), one("v"), one("r"), one("u"), one("w"), M, [nxt, nxt],
                                   [ext, ext[:, :1]])
    with pytest.raises(ValueError, match=ON_DEVICE):
        txl.rel_attn_fwd_mem_cells(one("q"), one("k"), one("v"), one("r"), one("u"), one("w"), M, [nxt, nxt],
                                   [ext, ext])
    assert txl.rel_attn_fwd_mem_cells([], [], [], [], None, None, M, [], []) == []
