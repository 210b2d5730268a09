"""Shared helpers for the GPU parity tests: seeded inputs -> device tensors,
the oracle on exactly the values the device saw, and error measures."""
import json
import os

import numpy as np
import torch

import oracle
from transformer_xl_relative_rel_gb300 import inputs

# tolerances stated for this method: fp32 path max |err| <= 1e-4; bf16 inputs
# with fp32 accumulation <= 2e-2 on unit-variance inputs
TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def device_layer(p, dtype):
    """numpy float32 layer inputs -> CUDA tensors (q,k,v,r in `dtype`, biases fp32)
    plus float64 numpy copies of exactly the values the GPU sees."""
    dev = {}
    host = {}
    for name in ("q", "k", "v", "r"):
        t = torch.from_numpy(np.ascontiguousarray(p[name])).to(dtype)
        dev[name] = t.cuda()
        host[name] = t.double().numpy()
    for name in ("u", "w"):
        t = torch.from_numpy(np.ascontiguousarray(p[name])).float()
        dev[name] = t.cuda()
        host[name] = t.double().numpy()
    return dev, host


def run_library(dev, mem_len, out=None):
    import transformer_xl_relative_rel_gb300 as txl
    return txl.rel_attn_fwd(dev["q"], dev["k"], dev["v"], dev["r"], dev["u"], dev["w"],
                            mem_len=mem_len, out=out)


def oracle_full(host, mem_len):
    return oracle.rel_attn(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"],
                           mem_len=mem_len)


def oracle_rows(host, mem_len, rows):
    return oracle.rel_attn_rows(host["q"], host["k"], host["v"], host["r"], host["u"], host["w"],
                                mem_len=mem_len, rows=rows)


def gather_rows(out, rows):
    o = out.double().cpu().numpy()
    return np.stack([o[i, b, h] for b, h, i in rows]) if len(rows) else np.zeros((0, o.shape[-1]))


def unit_shape(B, H, D, L, M):
    return inputs.LayerShape(B, H, D, L, M)


def record_error(case, shape, err, tol):
    """Append one parity result (the case, its shape, the max abs error and
    the tolerance) to the JSON-lines file named by TXL_PARITY_LOG, if set, so
    a run reports how much of each tolerance the kernels use."""
    path = os.environ.get("TXL_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": case, "shape": [int(x) for x in shape], "max_abs_err": float(err),
                            "tol": float(tol)}) + "\n")
