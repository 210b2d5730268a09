"""The memory rollover kernel against the oracle's definition, bit for bit."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T_L,B,dm", [((32, 16), 3, 64), ((150 + 150, 150), 60, 410),
                                      ((128 + 1600, 128), 2, 1024), ((13, 5), 3, 7),
                                      ((9, 9), 2, 8), ((40, 7), 1, 33)])
def test_rollover_bit_exact(dtype, T_L, B, dm):
    import transformer_xl_relative_rel_gb300 as txl
    T, L = T_L
    M = T - L
    g = torch.Generator().manual_seed(T * 7 + dm)
    ext = torch.randn(T, B, dm, generator=g).to(dtype)
    nxt = torch.full((T, B, dm), -7.0).to(dtype)
    d_ext, d_nxt = ext.cuda(), nxt.cuda()
    txl.mem_update(d_nxt, d_ext, mem_len=M)
    torch.cuda.synchronize()
    got = d_nxt.cpu()
    want = oracle.mem_update(ext.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy(), M)
    got_bits = got.view(torch.int16 if dtype == torch.bfloat16 else torch.int32).numpy()
    assert np.array_equal(got_bits[:M], want)
    # rows past M are the caller's (the next segment's current rows): untouched
    assert torch.equal(got[M:], nxt[M:])


def test_rollover_zero_memory_is_noop():
    import transformer_xl_relative_rel_gb300 as txl
    ext = torch.randn(8, 2, 16, device="cuda").bfloat16()
    nxt = torch.zeros(8, 2, 16, device="cuda").bfloat16()
    txl.mem_update(nxt, ext, mem_len=0)
    torch.cuda.synchronize()
    assert (nxt == 0).all()


@pytest.mark.parametrize("B,H,D,L,M,dm,dtype", [
    (22, 8, 64, 768, 768, 512, torch.bfloat16),    # the training shape: the attention launch takes the copy
    (22, 8, 64, 128, 3800, 512, torch.bfloat16),   # a copy too large to hide: its own launch
    (2, 3, 64, 150, 130, 41, torch.bfloat16),      # rows not 16-byte aligned: its own launch
    (2, 2, 41, 37, 50, 82, torch.bfloat16),        # padded head size
    (2, 2, 24, 40, 30, 48, torch.float32),         # fp32 path
])
def test_attn_with_rollover_equals_the_two_calls(B, H, D, L, M, dm, dtype):
    """txl_rel_attn_fwd_mem: the attention output bit-identical to
    txl_rel_attn_fwd's, the new memory bit-identical to the oracle's
    rollover, rows past M of mem_next untouched."""
    import transformer_xl_relative_rel_gb300 as txl
    from tests.helpers import device_layer, unit_shape
    from transformer_xl_relative_rel_gb300 import inputs
    T = M + L
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 300 + L + dm)
    dev, _ = device_layer(p, dtype)
    g = torch.Generator().manual_seed(dm + M)
    ext = torch.randn(T, B, dm, generator=g).to(dtype)
    nxt = torch.full((T, B, dm), -7.0).to(dtype)
    d_ext, d_nxt = ext.cuda(), nxt.cuda()
    args = (dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"])
    out = txl.rel_attn_fwd_mem(*args, mem_len=M, mem_next=d_nxt, ext_ctx=d_ext)
    plain = txl.rel_attn_fwd(*args, mem_len=M)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    ibits = torch.int16 if dtype == torch.bfloat16 else torch.int32
    want = oracle.mem_update(ext.view(ibits).numpy(), M)
    got = d_nxt.cpu()
    assert np.array_equal(got.view(ibits).numpy()[:M], want)
    assert torch.equal(got[M:], nxt[M:])
