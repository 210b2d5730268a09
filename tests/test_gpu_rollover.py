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
