"""Pins for the oracle's backward (``oracle.rel_attn_bwd``).

The gradients are checked against things that do not share its loop:

* central finite differences of the forward oracle (itself pinned in
  test_oracle_pins.py) for every element of every input, on two small
  problems, one with B = 2 and M != L so that the batch sums of the table and
  bias gradients and the reversed-table index are exercised;
* the value-gradient identity: the softmax weights of a row sum to one, so
  the column sums of dv equal the row sums of dout;
* translation invariance of the softmax: when every key (or every table row)
  of a head is the same vector, shifting the logits of a row by a constant
  changes nothing, so the bias gradient du (or dv-bias dw) and the part of dq
  along that vector vanish;
* with r, u and v set to zero the method is textbook attention: dq, dk, dv
  equal torch autograd through scaled_dot_product_attention in float64.

A final test plants mistakes in copies of the backward's C source and checks
that the finite-difference pin catches each one.
"""
import os
import shutil

import numpy as np
import pytest
import torch

import oracle


def _problem(B, H, D, L, M, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    T = M + L
    p = dict(q=g.standard_normal((L, B, H, D)), k=g.standard_normal((T, B, H, D)),
             v=g.standard_normal((T, B, H, D)), r=g.standard_normal((T, H, D)),
             u=g.standard_normal((H, D)), w=g.standard_normal((H, D)))
    dout = g.standard_normal((L, B, H, D))
    return p, dout


def _fd_grads(mod, p, dout, M, eps=1e-6):
    """Central differences of sum(dout * out) for every input element."""
    grads = {}
    for name in ("q", "k", "v", "r", "u", "w"):
        x = p[name]
        gx = np.zeros_like(x)
        flat = x.reshape(-1)
        gflat = gx.reshape(-1)
        for e in range(flat.size):
            keep = flat[e]
            flat[e] = keep + eps
            lp = float((mod.rel_attn(**p, mem_len=M) * dout).sum())
            flat[e] = keep - eps
            lm = float((mod.rel_attn(**p, mem_len=M) * dout).sum())
            flat[e] = keep
            gflat[e] = (lp - lm) / (2 * eps)
        grads["d" + name] = gx
    return grads


def _max_rel(a, b):
    return float(np.abs(a - b).max() / max(1.0, np.abs(b).max()))


FD_CASES = [(1, 2, 4, 5, 3), (2, 2, 3, 4, 6)]


@pytest.mark.parametrize("B,H,D,L,M", FD_CASES)
def test_bwd_matches_finite_differences(oracle_lib, B, H, D, L, M):
    p, dout = _problem(B, H, D, L, M, seed=100 + B)
    got = oracle.rel_attn_bwd(**p, dout=dout, mem_len=M)
    fd = _fd_grads(oracle, p, dout, M)
    for name in ("dq", "dk", "dv", "dr", "du", "dw"):
        assert got[name].shape == fd[name].shape
        # central differences at eps 1e-6: truncation ~1e-12, rounding ~1e-10
        assert _max_rel(got[name], fd[name]) < 1e-7, name


def test_bwd_dv_column_sums(oracle_lib):
    B, H, D, L, M = 2, 3, 5, 6, 4
    p, dout = _problem(B, H, D, L, M, seed=7)
    g = oracle.rel_attn_bwd(**p, dout=dout, mem_len=M)
    np.testing.assert_allclose(g["dv"].sum(axis=0), dout.sum(axis=0), rtol=0, atol=1e-12)


def test_bwd_translation_invariance(oracle_lib):
    B, H, D, L, M = 2, 2, 4, 5, 4
    p, dout = _problem(B, H, D, L, M, seed=11)
    T = M + L
    kap = np.random.Generator(np.random.PCG64(12)).standard_normal((H, D))
    rho = np.random.Generator(np.random.PCG64(13)).standard_normal((H, D))
    # every key of a head the same vector: the content logit is constant per row
    pk = dict(p, k=np.broadcast_to(kap[None, None], (T, B, H, D)).copy())
    g = oracle.rel_attn_bwd(**pk, dout=dout, mem_len=M)
    np.testing.assert_allclose(g["du"], 0.0, rtol=0, atol=1e-12)
    # every table row the same vector: the position logit is constant per row
    pr = dict(p, r=np.broadcast_to(rho[None], (T, H, D)).copy())
    g = oracle.rel_attn_bwd(**pr, dout=dout, mem_len=M)
    np.testing.assert_allclose(g["dw"], 0.0, rtol=0, atol=1e-12)
    # both: every logit of a row is the same, so dq = (kappa + rho) * sum_j dA_ij = 0
    pb = dict(p, k=pk["k"], r=pr["r"])
    g = oracle.rel_attn_bwd(**pb, dout=dout, mem_len=M)
    np.testing.assert_allclose(g["dq"], 0.0, rtol=0, atol=1e-12)


def _visible(L, M):
    i = np.arange(L)[:, None]
    j = np.arange(M + L)[None, :]
    return j <= M + i


def test_bwd_textbook_attention_autograd(oracle_lib):
    B, H, D, L, M = 2, 3, 8, 7, 5
    p, dout = _problem(B, H, D, L, M, seed=17)
    p["r"][:] = 0.0
    p["u"][:] = 0.0
    p["w"][:] = 0.0
    got = oracle.rel_attn_bwd(**p, dout=dout, mem_len=M)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a.transpose(1, 2, 0, 3))).requires_grad_(True)
    qt, kt, vt = to(p["q"]), to(p["k"]), to(p["v"])
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(_visible(L, M)))
    o.backward(torch.from_numpy(np.ascontiguousarray(dout.transpose(1, 2, 0, 3))))
    back = lambda t: t.grad.numpy().transpose(2, 0, 1, 3)
    np.testing.assert_allclose(got["dq"], back(qt), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dk"], back(kt), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dv"], back(vt), rtol=0, atol=1e-12)


# plausible mistakes in the backward, each planted in a copy of the C source
MUTANTS = {
    "no_softmax_centering": ("const double da = s[j] * (dp[j] - delta) * scale;",
                             "const double da = s[j] * dp[j] * scale;"),
    "unscaled_score_gradient": ("const double da = s[j] * (dp[j] - delta) * scale;",
                                "const double da = s[j] * (dp[j] - delta);"),
    "table_row_not_reversed": ("drp[t * D + d] += da * (qi[d] + wh[d]);",
                               "drp[off * D + d] += da * (qi[d] + wh[d]);"),
    "table_grad_with_u_bias": ("drp[t * D + d] += da * (qi[d] + wh[d]);",
                               "drp[t * D + d] += da * (qi[d] + uh[d]);"),
    "value_grad_from_dp": ("dvj[d] += s[j] * gi[d];", "dvj[d] += dp[j] * gi[d];"),
    "query_grad_content_only": ("dqi[d] += da * (kj[d] + rr[d]);", "dqi[d] += da * kj[d];"),
    "bias_grads_swapped": ("dup[d] += da * kj[d];", "dup[d] += da * rr[d];"),
}


def _bwd_pins_pass(mod):
    B, H, D, L, M = 2, 1, 3, 3, 4
    p, dout = _problem(B, H, D, L, M, seed=3)
    got = mod.rel_attn_bwd(**p, dout=dout, mem_len=M)
    fd = _fd_grads(mod, p, dout, M)
    return all(_max_rel(got[n], fd[n]) < 1e-7 for n in got)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_bwd_pins_catch_planted_mistake(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    assert _bwd_pins_pass(oracle), "pins must pass on the real oracle"
    src = open(os.path.join(os.path.dirname(oracle.__file__), "txl_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    mdir = tmp_path / name
    mdir.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "__init__.py"), mdir / "__init__.py")
    (mdir / "txl_oracle.c").write_text(src.replace(old, new))
    import importlib.util
    spec = importlib.util.spec_from_file_location(f"oracle_bwd_mutant_{name}", mdir / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)
    assert not _bwd_pins_pass(mod), f"planted mistake {name!r} went unnoticed"
