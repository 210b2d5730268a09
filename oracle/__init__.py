"""Plain CPU reference (the oracle) for Transformer-XL relative attention.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only code that may import this package.
The product library (``transformer_xl_relative_rel_gb300``) never imports it,
and this package imports nothing from the product.

Contents
  * ``txl_oracle.c`` -- the float64 triple loop over (i, j, d) with direct
    ``r_{i-j}`` indexing (Transformer-XL, Section 3.3 procedure and Appendix B
    table order), built here with gcc into ``liboracle.so``.
  * ``rel_attn_bwd`` (same C file) -- the gradients of one layer call for a
    given output gradient, the chain rule written out per query row.
  * ``mem_update`` -- the memory rollover of Section 3.2 written as its plain
    definition in numpy: the new memory is the newest M rows of
    [old memory; current hidden states].
  * ``project_heads`` -- the projections of Section 3.3's procedure
    (q = h W_q, k = h~ W_kE, v = h~ W_v) in float64, laid out per head.
  * ``sinusoid`` / ``rel_table`` -- the relative encoding R (the sinusoid of
    Vaswani et al. that Section 3.3 re-uses) and Appendix B's reversed
    projected table Q_t = W_kR R_{T-1-t}, in float64.

All functions take numpy arrays in the T-major layouts of the library:
``q, out: [L, B, H, D]``, ``k, v: [T, B, H, D]`` with ``T = M + L``,
``r: [T, H, D]`` (row t is ``W_kR R_{T-1-t}``), ``u, w: [H, D]``.
Any float dtype is accepted and converted exactly to float64.

Status: parity pinned (tests/test_oracle_pins.py); no function here is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "txl_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib: Optional[ctypes.CDLL] = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``txl_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, -O2).

    Plain portable C: no architecture flags, so the same source builds on the
    x86 development host and on the Arm GPU host.
    """
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.txl_oracle_rel_attn.argtypes = [
            _dp, _dp, _dp, _dp, _dp, _dp,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            _dp, _dp, _dp, ctypes.c_int]
        lib.txl_oracle_rel_attn.restype = None
        lib.txl_oracle_rel_attn_rows.argtypes = [
            _dp, _dp, _dp, _dp, _dp, _dp,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            ctypes.POINTER(ctypes.c_int64), ctypes.c_long, _dp, ctypes.c_int]
        lib.txl_oracle_rel_attn_rows.restype = None
        lib.txl_oracle_rel_attn_bwd.argtypes = [
            _dp, _dp, _dp, _dp, _dp, _dp, _dp,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
            _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp, ctypes.c_int]
        lib.txl_oracle_rel_attn_bwd.restype = None
        lib.txl_oracle_max_threads.argtypes = []
        lib.txl_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the OpenMP runtime would give the oracle on this host."""
    return int(_load().txl_oracle_max_threads())


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _shapes(q, k, v, r, u, w, mem_len):
    L, B, H, D = q.shape
    T = mem_len + L
    if k.shape != (T, B, H, D) or v.shape != (T, B, H, D):
        raise ValueError(f"k/v must be [{T},{B},{H},{D}], got {k.shape}, {v.shape}")
    if r.shape != (T, H, D):
        raise ValueError(f"r must be [{T},{H},{D}], got {r.shape}")
    if u.shape != (H, D) or w.shape != (H, D):
        raise ValueError(f"u/v biases must be [{H},{D}]")
    return B, H, D, L, T


def rel_attn(q, k, v, r, u, w, mem_len: int, return_prob: bool = False,
             nthreads: int = 0, return_lse: bool = False):
    """Relative attention of one layer over [memory; segment], float64.

    Returns ``out`` of shape [L, B, H, D]; then, when ``return_prob``, the
    attention weights ``P`` of shape [B, H, L, M+L] (exact zeros where
    masked); then, when ``return_lse``, each row's log-sum-exp of its scaled
    scores, [B, H, L].
    """
    q, k, v, r, u, w = (_f64(x) for x in (q, k, v, r, u, w))
    B, H, D, L, T = _shapes(q, k, v, r, u, w, mem_len)
    out = np.zeros((L, B, H, D), dtype=np.float64)
    prob = np.zeros((B, H, L, T), dtype=np.float64) if return_prob else None
    lse = np.zeros((B, H, L), dtype=np.float64) if return_lse else None
    null = ctypes.cast(None, _dp)
    _load().txl_oracle_rel_attn(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u), _ptr(w),
        B, H, D, L, mem_len, _ptr(out),
        _ptr(prob) if prob is not None else null, _ptr(lse) if lse is not None else null,
        int(nthreads))
    res = (out,) + ((prob,) if return_prob else ()) + ((lse,) if return_lse else ())
    return res if len(res) > 1 else out


def rel_attn_rows(q, k, v, r, u, w, mem_len: int, rows, nthreads: int = 0):
    """The same computation for selected query rows only.

    ``rows`` is an int array of shape [n, 3] holding (b, h, i) triples; the
    result is [n, D] float64.
    """
    q, k, v, r, u, w = (_f64(x) for x in (q, k, v, r, u, w))
    B, H, D, L, T = _shapes(q, k, v, r, u, w, mem_len)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    if rows.size and ((rows < 0).any() or (rows[:, 0] >= B).any()
                      or (rows[:, 1] >= H).any() or (rows[:, 2] >= L).any()):
        raise ValueError("row index out of range")
    out = np.zeros((rows.shape[0], D), dtype=np.float64)
    _load().txl_oracle_rel_attn_rows(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u), _ptr(w),
        B, H, D, L, mem_len,
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), rows.shape[0],
        _ptr(out), int(nthreads))
    return out


def rel_attn_bwd(q, k, v, r, u, w, dout, mem_len: int, nthreads: int = 0):
    """Gradients of ``rel_attn`` for the output gradient ``dout`` [L, B, H, D],
    float64: the chain rule through the masked softmax and the four-term
    score, written out per query row (Section 3.3 procedure; every input,
    the memory rows of k and v included, gets its gradient).

    Returns a dict with ``dq`` [L,B,H,D], ``dk``, ``dv`` [T,B,H,D], ``dr``
    [T,H,D] (summed over the batch), ``du``, ``dw`` [H,D] (the u and v bias
    gradients, summed over batch and query rows).
    """
    q, k, v, r, u, w, dout = (_f64(x) for x in (q, k, v, r, u, w, dout))
    B, H, D, L, T = _shapes(q, k, v, r, u, w, mem_len)
    if dout.shape != q.shape:
        raise ValueError(f"dout must be {q.shape}, got {dout.shape}")
    g = dict(dq=np.zeros((L, B, H, D)), dk=np.zeros((T, B, H, D)), dv=np.zeros((T, B, H, D)),
             dr=np.zeros((T, H, D)), du=np.zeros((H, D)), dw=np.zeros((H, D)))
    dr_part = np.zeros((B * H, T, D))
    du_part = np.zeros((B * H, D))
    dw_part = np.zeros((B * H, D))
    _load().txl_oracle_rel_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u), _ptr(w), _ptr(dout),
        B, H, D, L, mem_len,
        _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dr"]), _ptr(g["du"]), _ptr(g["dw"]),
        _ptr(dr_part), _ptr(du_part), _ptr(dw_part), int(nthreads))
    return g


def mem_update(ext_ctx, mem_len: int) -> np.ndarray:
    """New memory after one segment (Section 3.2: a cache of length M).

    ``ext_ctx`` is the layer's extended context [M+L, ...] = [old memory;
    current hidden states].  The new memory is its newest ``mem_len`` rows,
    oldest first.  Works on any dtype, bit for bit.
    """
    ext = np.asarray(ext_ctx)
    if mem_len == 0:
        return ext[:0].copy()
    return ext[ext.shape[0] - mem_len:].copy()


def project_heads(x, w, heads: int, d_head: int, d_pad: Optional[int] = None) -> np.ndarray:
    """One projection of Section 3.3's procedure, per head, in float64.

    ``x`` [..., d_in] (hidden states, e.g. the extended context
    [SG(memory); h] for k and v, the segment h for q) times ``w``^T, with
    ``w`` the paper's projection matrix [heads*d_head, d_in] (q = h W_q^T):
    element (..., h, d) is sum_c x[..., c] w[h*d_head + d, c].  The result is
    [..., heads, d_pad] with zeros in columns d_head..d_pad-1 (``d_pad``
    defaults to ``d_head``).
    """
    x = _f64(x)
    w = _f64(w)
    d_pad = d_head if d_pad is None else d_pad
    if w.shape != (heads * d_head, x.shape[-1]):
        raise ValueError(f"w must be [{heads * d_head}, {x.shape[-1]}], got {w.shape}")
    if d_pad < d_head:
        raise ValueError("d_pad < d_head")
    y = np.matmul(x, w.T).reshape(x.shape[:-1] + (heads, d_head))
    out = np.zeros(x.shape[:-1] + (heads, d_pad))
    out[..., :d_head] = y
    return out


def sinusoid(n_pos: int, d_model: int) -> np.ndarray:
    """The relative encoding R as a [n_pos, d_model] float64 table, row p for
    distance p: frequencies w_c = 10000^(-2c/d_model) for column pairs
    (2c, 2c+1), column 2c = sin(p w_c), column 2c+1 = cos(p w_c) (a last odd
    column is a sine)."""
    out = np.zeros((n_pos, d_model))
    for c2 in range(0, d_model, 2):
        freq = 10000.0 ** (-c2 / d_model)
        ang = np.arange(n_pos, dtype=np.float64) * freq
        out[:, c2] = np.sin(ang)
        if c2 + 1 < d_model:
            out[:, c2 + 1] = np.cos(ang)
    return out


def rel_table(w_r, klen: int, heads: int, d_head: int, d_pad: Optional[int] = None) -> np.ndarray:
    """Appendix B's table in the library's row order, float64 [klen, heads, d_pad]:
    row t holds W_kR R_{klen-1-t} (the projection of distance klen-1-t), split
    into heads, zeros past d_head.  ``w_r`` is W_kR in the paper's layout,
    [heads*d_head, d_model]."""
    w_r = _f64(w_r)
    R = sinusoid(klen, w_r.shape[1])
    by_distance = project_heads(R, w_r, heads, d_head, d_pad)      # row p: distance p
    return np.ascontiguousarray(by_distance[::-1])
