"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait in the library's kernels is bounded; when one runs out the
kernel records a device error word and winds down, and txl_check reports
TXL_ERR_TIMEOUT.  txl_selftest_wait runs that same wait, limited to a few
milliseconds, on an mbarrier nothing completes (no copy or MMA in flight), so
the path from an expired wait to the host's status is exercised with no
GPU fault; the context stays usable and the next call is correct.
"""
import numpy as np
import pytest
import torch

from tests.helpers import TOL_BF16, device_layer, oracle_full, run_library, unit_shape
from transformer_xl_relative_rel_gb300 import inputs

pytestmark = pytest.mark.gpu

TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from transformer_xl_relative_rel_gb300 import _build, abi
    _build.build()
    abi.load_library()


def test_expired_wait_reports_timeout_then_recovers():
    import transformer_xl_relative_rel_gb300 as txl
    txl.check()                                   # nothing pending
    txl.selftest_wait(2000)                       # a 2 ms wait that runs out
    with pytest.raises(txl.TxlError) as err:
        txl.check()
    assert err.value.status == TIMEOUT
    txl.check()                                   # reported once, then cleared
    # the context is intact: an attention call right after is correct
    p = inputs.unit_layer(unit_shape(1, 2, 64, 130, 70), 77)
    dev, host = device_layer(p, torch.bfloat16)
    out = run_library(dev, 70)
    txl.check()
    assert np.abs(out.double().cpu().numpy() - oracle_full(host, 70)).max() <= TOL_BF16


def test_selftest_on_a_side_stream():
    import transformer_xl_relative_rel_gb300 as txl
    s = torch.cuda.Stream()
    txl.selftest_wait(500, stream=s)
    with pytest.raises(txl.TxlError) as err:
        txl.check(stream=s)
    assert err.value.status == TIMEOUT
    txl.check(stream=s)
