"""The benchmark's recurrence runs its (layer, segment) cells as a wavefront:
cell (n, tau) needs layer n-1's output of segment tau and layer n's memory
from segment tau-1, so the cells of one diagonal n + tau are independent.
Here the wavefront step and the segment-by-segment order start from the same
state and must leave every buffer the calls write bit-identical (CUDA,
`-m gpu`).  The per-call results themselves are checked against the oracle
in test_gpu_chain.py."""
import dataclasses

import pytest
import torch

pytestmark = pytest.mark.gpu


def _state(chain):
    return [[x.clone() for x in lay["ext"]] + [lay[k].clone() for k in ("q", "k", "v")] for lay in chain.layers]


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("name,layers,segments,fused", [("char_train", 3, 4, True), ("large_lm", 3, 3, False),
                                                         ("base_lm", 2, 3, False)])
def test_wavefront_step_equals_segment_order(name, layers, segments, fused):
    import bench
    import transformer_xl_relative_rel_gb300 as txl
    from transformer_xl_relative_rel_gb300.workloads import WORKLOADS
    w = dataclasses.replace(WORKLOADS[name], layers=layers, segments=segments)
    chain = bench.LayerChain(w, torch.device("cuda", 0), txl, fused=fused and w.shape.d_head == 64)
    start, cur0 = _state(chain), chain.cur
    last_out = chain.layers[-1]["out"]
    for tau in range(segments):
        chain.segment(txl, tau)
        chain.cur ^= 1
    torch.cuda.synchronize()
    seq, seq_out, seq_cur = _state(chain), last_out.clone(), chain.cur
    for lay, saved in zip(chain.layers, start):
        for dst, src in zip(lay["ext"] + [lay[k] for k in ("q", "k", "v")], saved):
            dst.copy_(src)
    chain.cur = cur0
    chain.step(txl)
    torch.cuda.synchronize()
    txl.check()
    assert chain.cur == seq_cur
    for lay, want in zip(chain.layers, seq):
        for got, ref in zip(lay["ext"] + [lay[k] for k in ("q", "k", "v")], want):
            assert torch.equal(_bits(got), _bits(ref))
    assert torch.equal(_bits(last_out), _bits(seq_out))
