"""Several independent layer calls in shared launches
(txl_rel_attn_fwd_mem_cells, CUDA, `-m gpu`).

Each call is Section 3.3's attention of one layer plus Section 3.2's cache
update of that layer, as txl_rel_attn_fwd_mem makes it; the grouped entry
point only changes which launch (and which CTA) computes a work item, never
its arithmetic, so every output and every rolled memory must equal, bit for
bit, what the calls give one by one.  The one-by-one call is itself checked
against the oracle in test_gpu_attention.py and test_gpu_chain.py; one
grouped case here is also checked against the oracle directly.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, record_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _calls(n, B, H, D, L, M, dm, seed, no_bias=()):
    g = torch.Generator(device="cuda").manual_seed(seed)
    T = M + L
    bf = lambda *shape: torch.randn(*shape, generator=g, device="cuda").bfloat16()
    calls = []
    for c in range(n):
        calls.append(dict(q=bf(L, B, H, D), k=bf(T, B, H, D), v=bf(T, B, H, D), r=bf(T, H, D),
                          u=None if c in no_bias else 0.1 * torch.randn(H, D, generator=g, device="cuda"),
                          w=None if c in no_bias else 0.1 * torch.randn(H, D, generator=g, device="cuda"),
                          ext=bf(T, B, dm)))
    return calls


def _bits(t):
    return t.view(torch.int16)


@pytest.mark.parametrize("n,B,H,D,L,M,dm,no_bias", [
    (3, 3, 2, 64, 256, 256, 128, ()),          # one grouped launch, whole tiles
    (9, 2, 2, 64, 128, 128, 64, ()),           # 8 calls + 1 call
    (10, 2, 3, 64, 200, 72, 96, (4,)),         # ragged query tiles, memory not a tile multiple, no biases in call 4
    (2, 1, 1, 64, 1, 0, 32, ()),               # a single query row, no memory (nothing to roll)
    (4, 2, 2, 64, 128, 1600, 64, ()),          # long memory: each call splits its keys, so call by call
    (3, 2, 2, 32, 96, 64, 64, ()),             # 32-wide heads: call by call
])
def test_cells_equal_calls_one_by_one(n, B, H, D, L, M, dm, no_bias):
    import transformer_xl_relative_rel_gb300 as txl
    calls = _calls(n, B, H, D, L, M, dm, seed=n * 1000 + L, no_bias=no_bias)
    T = M + L
    nxt = [torch.full((T, B, dm), float("nan"), device="cuda").bfloat16() for _ in range(n)]
    outs = txl.rel_attn_fwd_mem_cells([c["q"] for c in calls], [c["k"] for c in calls], [c["v"] for c in calls],
                                      [c["r"] for c in calls], [c["u"] for c in calls], [c["w"] for c in calls], M,
                                      nxt, [c["ext"] for c in calls])
    torch.cuda.synchronize()
    txl.check()
    for c, call in enumerate(calls):
        nxt1 = torch.full((T, B, dm), float("nan"), device="cuda").bfloat16()
        out1 = txl.rel_attn_fwd_mem(call["q"], call["k"], call["v"], call["r"], call["u"], call["w"], M,
                                    mem_next=nxt1, ext_ctx=call["ext"])
        torch.cuda.synchronize()
        assert torch.equal(_bits(outs[c]), _bits(out1)), f"call {c}: output"
        assert torch.equal(_bits(nxt[c][:M]), _bits(nxt1[:M])), f"call {c}: rolled memory"
        assert torch.equal(_bits(nxt[c][:M]), _bits(call["ext"][L:])), f"call {c}: newest M rows"


def test_cells_against_oracle():
    """A grouped launch's outputs on sampled rows of every call against the
    oracle, fed each call's device inputs."""
    import transformer_xl_relative_rel_gb300 as txl
    n, B, H, D, L, M, dm = 5, 2, 2, 64, 256, 128, 64
    calls = _calls(n, B, H, D, L, M, dm, seed=7)
    nxt = [torch.empty(M, B, dm, device="cuda").bfloat16() for _ in range(n)]
    outs = txl.rel_attn_fwd_mem_cells([c["q"] for c in calls], [c["k"] for c in calls], [c["v"] for c in calls],
                                      [c["r"] for c in calls], [c["u"] for c in calls], [c["w"] for c in calls], M,
                                      nxt, [c["ext"] for c in calls])
    torch.cuda.synchronize()
    txl.check()
    g = np.random.default_rng(11)
    for c, call in enumerate(calls):
        rows = np.stack([g.integers(0, B, 24), g.integers(0, H, 24), g.integers(0, L, 24)], 1).astype(np.int64)
        host = {k: call[k].double().cpu().numpy() for k in ("q", "k", "v", "r", "u", "w")}
        ref = oracle.rel_attn_rows(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"], mem_len=M,
                                   rows=rows)
        o = outs[c].double().cpu().numpy()
        got = np.stack([o[i, b, h] for b, h, i in rows])
        err = np.abs(got - ref).max()
        record_error("attention_cells", (B, H, D, L, M), err, TOL_BF16)
        assert np.isfinite(got).all() and err <= TOL_BF16, f"call {c}: max abs err {err:.3e}"
        assert torch.equal(_bits(nxt[c]), _bits(call["ext"][L:]))
