"""The stream-K schedule of the bf16 kernel (CUDA, `-m gpu`).

With one query tile per (b, h) (L <= 128) and at least as many (b, h) as
SMs, the key tiles of all items are cut into equal contiguous ranges, one per
CTA: items inside a range are computed whole, items cut by a range boundary in
two parts that a merge launch combines.  Every output row, whole or merged,
must match the oracle element by element; the log-sum-exp output too.
"""
import numpy as np
import pytest
import torch

from tests.helpers import TOL_BF16, device_layer, oracle_full, record_error, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _candidates():
    """(B, H, D, L, M) with B*H at least the SM count and not a multiple of
    it, and memories long enough that the split model divides the keys (so
    the stream-K schedule runs; key tiles per item from 24 to 32), or B*H
    just above the SM count."""
    n = _sms()
    return [(n + 8, 1, 64, 128, 3000),       # a full query block
            (n + 8, 1, 64, 64, 3000),        # a ragged query block
            (n + 18, 1, 64, 33, 2600),       # ragged keys in the last tile
            (n + 9, 1, 56, 100, 3000),       # head size 56: thread loads
            (n + 9, 1, 64, 1, 3000),         # one query per item
            (n + 3, 1, 64, 128, 4000),
            # the long-memory evaluation shape with just over one (b, h) per
            # SM: the model keeps its keys whole, but whole items would
            # leave most CTAs idle in the second round, so stream-K runs
            (-(-(n + 1) // 16), 16, 64, 128, 1600)]


def _streamk(B, H, D, L, M):
    import transformer_xl_relative_rel_gb300 as txl
    splits, _ = txl.rel_attn_fwd_plan(B, M, L, H, D, txl.TXL_BF16)
    return splits == 2


def test_candidates_take_the_schedule():
    assert sum(_streamk(*c) for c in _candidates()) >= 4


@pytest.mark.parametrize("idx", range(7))
def test_streamk_matches_oracle(idx):
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, L, M = _candidates()[idx]
    if not _streamk(B, H, D, L, M):
        pytest.skip("the split model keeps this shape whole on this device")
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 7000 + idx)
    dev, host = device_layer(p, torch.bfloat16)
    out = torch.full_like(dev["q"], float("nan"))
    txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M, out=out)
    txl.check()
    ref = oracle_full(host, M)
    got = out.double().cpu().numpy()
    err = np.abs(got - ref).max()
    record_error("streamk", (B, H, D, L, M), err, TOL_BF16)
    assert np.isfinite(got).all() and err <= TOL_BF16, f"max abs err {err:.3e}"


def test_streamk_lse_and_repeatable():
    """The row log-sum-exp of whole and merged items, and the same bits on
    a second call."""
    import oracle
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, L, M = _candidates()[0]
    assert _streamk(B, H, D, L, M)
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 7100)
    dev, host = device_layer(p, torch.bfloat16)
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")
    out = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M, lse=lse)
    again = txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"], mem_len=M)
    assert torch.equal(out, again)
    ref_out, ref_lse = oracle.rel_attn(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"],
                                       mem_len=M, return_lse=True)
    assert np.abs(out.double().cpu().numpy() - ref_out).max() <= TOL_BF16
    # the log-sum-exp as the other tests bound it: relative to max(1, |lse|)
    lse_err = np.abs(lse.double().cpu().numpy() - ref_lse).max() / max(1.0, np.abs(ref_lse).max())
    assert lse_err <= 2e-2


def test_streamk_ring():
    """The schedule with keys and values stored as a ring."""
    import transformer_xl_relative_rel_gb300 as txl
    B, H, D, L, M = _candidates()[0]
    start = 200
    assert _streamk(B, H, D, L, M)
    p = inputs.unit_layer(unit_shape(B, H, D, L, M), 7200)
    dev, host = device_layer(p, torch.bfloat16)
    k_ring = torch.roll(dev["k"], shifts=start, dims=0).contiguous()
    v_ring = torch.roll(dev["v"], shifts=start, dims=0).contiguous()
    out = txl.rel_attn_fwd_ring(dev["q"], k_ring, v_ring, dev["r"], dev["u"], dev["w"], mem_len=M, kv_start=start)
    assert np.abs(out.double().cpu().numpy() - oracle_full(host, M)).max() <= TOL_BF16
