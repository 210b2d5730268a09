"""Ring-stored extended context (k, v rows rotated by kv_start) and the ring
append: the same results as the unrolled layout, checked against the oracle
on the unrolled values (CUDA, `-m gpu`)."""
import numpy as np
import pytest
import torch

from tests.helpers import TOL_BF16, TOL_F32, device_layer, oracle_full, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu


def _ring(x, start):
    """Store the unrolled rows x[j] at ring row (start + j) mod len."""
    return torch.roll(x, shifts=start, dims=0).contiguous()


@pytest.mark.parametrize("dtype,tol,B,H,D,L,M,start", [
    (torch.bfloat16, TOL_BF16, 2, 2, 64, 200, 184, 0),      # ring == plain layout
    (torch.bfloat16, TOL_BF16, 2, 2, 64, 200, 184, 8),      # wraps inside a key tile (TMA 8-row boxes)
    (torch.bfloat16, TOL_BF16, 1, 2, 64, 130, 1030, 640),   # long memory: key splits + wrap
    (torch.bfloat16, TOL_BF16, 2, 2, 64, 150, 150, 37),     # start not a multiple of 8: thread loads
    (torch.bfloat16, TOL_BF16, 2, 2, 64, 100, 27, 64),      # M+L not a multiple of 8
    (torch.bfloat16, TOL_BF16, 2, 2, 41, 150, 150, 299),    # d_head 41 (thread loads), start = T-1
    (torch.float32, TOL_F32, 1, 2, 24, 60, 50, 77),         # fp32 path
])
def test_ring_attention_matches_unrolled(dtype, tol, B, H, D, L, M, start):
    import transformer_xl_relative_rel_gb300 as txl
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 5000 + start + D)
    dev, host = device_layer(p, dtype)
    k_ring, v_ring = _ring(dev["k"], start), _ring(dev["v"], start)
    got = txl.rel_attn_fwd_ring(dev["q"], k_ring, v_ring, dev["r"], dev["u"], dev["w"], mem_len=M,
                                kv_start=start)
    plain = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M)
    if start == 0:
        assert torch.equal(got, plain)
    ref = oracle_full(host, M)
    err = np.abs(got.double().cpu().numpy() - ref).max()
    assert err <= tol, f"max abs err {err:.3e}"


@pytest.mark.parametrize("ring_len,n,start", [(10, 3, 0), (10, 3, 8), (10, 10, 4), (257, 128, 200),
                                              (7, 0, 3)])
def test_ring_append_is_a_rotated_copy(ring_len, n, start):
    import transformer_xl_relative_rel_gb300 as txl
    g = torch.Generator(device="cuda").manual_seed(ring_len + n + start)
    ring = torch.randn(ring_len, 3, 40, generator=g, device="cuda").bfloat16()
    rows = torch.randn(n, 3, 40, generator=g, device="cuda").bfloat16()
    want = ring.clone()
    for i in range(n):
        want[(start + i) % ring_len] = rows[i]
    nxt = txl.ring_append(ring, rows, start)
    torch.cuda.synchronize()
    assert torch.equal(ring, want)
    assert nxt == (start + n) % ring_len


def test_ring_segments_match_rollover_chain():
    """Three segments with a ring (append L rows) give the same memory as the
    copy rollover (txl_mem_update into the other buffer)."""
    import transformer_xl_relative_rel_gb300 as txl
    B, dm, L, M = 2, 64, 24, 40
    T = M + L
    g = torch.Generator(device="cuda").manual_seed(11)
    mem0 = torch.randn(M, B, dm, generator=g, device="cuda").bfloat16()
    segs = [torch.randn(L, B, dm, generator=g, device="cuda").bfloat16() for _ in range(3)]
    # copy rollover: ext = [mem; h], next mem = newest M rows
    ext = torch.empty(T, B, dm, dtype=torch.bfloat16, device="cuda")
    nxt = torch.empty_like(ext)
    ext[:M] = mem0
    # ring of T rows holding [mem; h] from row `start`
    ring = torch.zeros(T, B, dm, dtype=torch.bfloat16, device="cuda")
    ring[:M] = mem0
    start = 0          # oldest row of the context
    for h in segs:
        ext[M:] = h
        txl.ring_append(ring, h, (start + M) % T)     # the segment's rows after the memory
        unrolled = torch.roll(ring, shifts=-start, dims=0)
        assert torch.equal(unrolled, ext)             # same extended context
        txl.mem_update(nxt, ext, mem_len=M)
        ext, nxt = nxt, ext
        start = (start + L) % T                       # the oldest L rows drop out
    torch.cuda.synchronize()
