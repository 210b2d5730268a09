"""The Python binding's argument checks, on the host: wrong shapes, dtypes,
devices and pairings are refused with an exception before the library is
called (these checks are what stands between a caller's tensors and the raw
pointers the C ABI receives).  CPU tensors stand in for device tensors where
the check under test comes first; no compute call is made."""
import pytest
import torch

import transformer_xl_relative_rel_gb300 as txl

L, B, H, D, M = 8, 2, 2, 16, 8
T = L + M


def _layer(dtype=torch.bfloat16):
    return dict(q=torch.zeros(L, B, H, D, dtype=dtype), k=torch.zeros(T, B, H, D, dtype=dtype),
                v=torch.zeros(T, B, H, D, dtype=dtype), r=torch.zeros(T, H, D, dtype=dtype),
                u=torch.zeros(H, D), w=torch.zeros(H, D))


def _fwd(p, **kw):
    return txl.rel_attn_fwd(p["q"], p["k"], p["v"], p["r"], p["u"], p["w"], mem_len=M, **kw)


def test_attention_shapes_and_dtypes():
    p = _layer()
    with pytest.raises(ValueError):
        txl.rel_attn_fwd(p["q"], p["k"][:-1], p["v"], p["r"], p["u"], p["w"], mem_len=M)   # k one row short
    with pytest.raises(ValueError):
        txl.rel_attn_fwd(p["q"], p["k"], p["v"], p["r"][:, :1], p["u"], p["w"], mem_len=M)   # table heads
    with pytest.raises(TypeError):
        txl.rel_attn_fwd(p["q"], p["k"].float(), p["v"], p["r"], p["u"], p["w"], mem_len=M)   # mixed dtypes
    with pytest.raises(ValueError):
        txl.rel_attn_fwd(p["q"], p["k"], p["v"], p["r"], p["u"].double(), p["w"], mem_len=M)  # bias dtype
    with pytest.raises(ValueError):
        txl.rel_attn_fwd(p["q"], p["k"], p["v"], p["r"], p["u"][:1], p["w"], mem_len=M)       # bias shape
    with pytest.raises(ValueError):
        _fwd(p)                                   # host tensors: refused before any pointer is taken
    from transformer_xl_relative_rel_gb300 import abi
    with pytest.raises(TypeError):
        abi._dtype_code(torch.zeros(1, dtype=torch.float16))   # no fp16 path


def test_attention_output_and_lse_checks():
    p = _layer()
    with pytest.raises(ValueError):
        _fwd(p, out=torch.zeros(L, B, H, D + 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        _fwd(p, out=torch.zeros(L, B, H, D, dtype=torch.float32))


def test_backward_pairing_and_shapes():
    p = _layer()
    dout = torch.zeros(L, B, H, D, dtype=torch.bfloat16)
    args = (p["q"], p["k"], p["v"], p["r"], p["u"], p["w"])
    with pytest.raises(ValueError):
        txl.rel_attn_bwd(*args, dout[:-1], mem_len=M)                 # dout shaped unlike q
    with pytest.raises(ValueError):
        txl.rel_attn_bwd(*args, dout, mem_len=M)                      # host tensors


def test_fused_rollover_checks():
    p = _layer()
    ext = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    nxt = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    args = (p["q"], p["k"], p["v"], p["r"], p["u"], p["w"])
    with pytest.raises(ValueError):
        txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=nxt, ext_ctx=ext[:-1])     # context rows
    with pytest.raises(ValueError):
        txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=nxt[:1], ext_ctx=ext)      # too small
    with pytest.raises(ValueError):
        txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=nxt, ext_ctx=ext)          # host tensors


def test_rollover_and_ring_checks():
    ext = torch.zeros(T, B, 32, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        txl.mem_update(torch.zeros(T, B, 32, dtype=torch.bfloat16), ext, mem_len=T + 1)
    with pytest.raises(ValueError):
        txl.mem_update(torch.zeros(M, B, 31, dtype=torch.bfloat16), ext, mem_len=M)
    with pytest.raises(TypeError):
        txl.mem_update(torch.zeros(M, B, 32, dtype=torch.float32), ext, mem_len=M)
    with pytest.raises(ValueError):
        txl.mem_update(torch.zeros(M, B, 32, dtype=torch.bfloat16), ext, mem_len=M)   # host tensors
