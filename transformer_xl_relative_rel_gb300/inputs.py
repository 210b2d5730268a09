"""Seeded synthetic inputs shared by the CUDA path's tests and the oracle.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both sides of every parity check receive the same arrays
from here (numpy PCG64, float32, later rounded to bf16 by the caller where the
workload is bf16).

The one piece of structure it builds is the relative position table ``r`` that
the library takes as an input: a sinusoid encoding of the offsets (Transformer-XL
Section 3.3 re-uses the sinusoid of Vaswani et al. for ``R``) projected by a
random ``W_kR`` and stored in the reversed row order of Appendix B, so that row
``t`` holds the projection of offset ``T-1-t``.  Which sinusoid convention is
used does not affect parity, because ``r`` is an input to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def sinusoid(n_pos: int, d_model: int) -> np.ndarray:
    """[n_pos, d_model] table: row p is the encoding of offset p.

    Column 2c holds sin(p * 10000^(-2c/d_model)) and column 2c+1 the matching
    cosine (for odd d_model the last column is a sine).
    """
    p = np.arange(n_pos, dtype=np.float64)[:, None]
    c = np.arange(0, d_model, 2, dtype=np.float64)[None, :]
    ang = p * np.power(10000.0, -c / d_model)
    out = np.zeros((n_pos, d_model), dtype=np.float64)
    out[:, 0::2] = np.sin(ang)
    out[:, 1::2] = np.cos(ang)[:, : d_model // 2]
    return out


def reversed_rel_table(w_r: np.ndarray, T: int, heads: int, d_head: int) -> np.ndarray:
    """Projected relative table in the library's row order, [T, H, D] float32.

    ``w_r`` is [d_model, H*D]; row t of the result is sinusoid(T-1-t) @ w_r.
    """
    d_model = w_r.shape[0]
    proj = sinusoid(T, d_model) @ w_r.astype(np.float64)      # row p = offset p
    return np.ascontiguousarray(proj[::-1].reshape(T, heads, d_head).astype(np.float32))


@dataclass(frozen=True)
class LayerShape:
    batch: int
    heads: int
    d_head: int
    seg_len: int
    mem_len: int

    @property
    def klen(self) -> int:
        return self.mem_len + self.seg_len

    @property
    def d_model(self) -> int:
        return self.heads * self.d_head


def unit_layer(shape: LayerShape, seed: int) -> Dict[str, np.ndarray]:
    """One layer's inputs with unit-variance q, k, v, u, v-bias and r.

    q, k, v, u, w ~ N(0, 1); r = sinusoid @ W_r with W_r ~ N(0, 2/d_model), so
    that each entry of r also has unit variance.
    """
    g = rng(seed)
    L, B, H, D, T = shape.seg_len, shape.batch, shape.heads, shape.d_head, shape.klen
    q = g.standard_normal((L, B, H, D), dtype=np.float32)
    k = g.standard_normal((T, B, H, D), dtype=np.float32)
    v = g.standard_normal((T, B, H, D), dtype=np.float32)
    u = g.standard_normal((H, D), dtype=np.float32)
    w = g.standard_normal((H, D), dtype=np.float32)
    w_r = g.standard_normal((H * D, H * D)) * np.sqrt(2.0 / (H * D))
    r = reversed_rel_table(w_r, T, H, D)
    return dict(q=q, k=k, v=v, r=r, u=u, w=w)


def lm_weights(shape: LayerShape, seed: int, layers: int, std: float = 0.02
               ) -> Dict[str, np.ndarray]:
    """Per-layer projection weights of the language-model-shaped chains.

    W_q, W_kE, W_v, W_kR, W_o ~ N(0, std^2) of shape [layers, d_model, d_model]
    (W_o maps the attention output back to d_model), u, v ~ N(0, std^2) of
    shape [layers, H, D].
    """
    g = rng(seed)
    dm, H, D = shape.d_model, shape.heads, shape.d_head
    out = {}
    for name in ("w_q", "w_k", "w_v", "w_r", "w_o"):
        out[name] = (g.standard_normal((layers, dm, dm)) * std).astype(np.float32)
    out["u"] = (g.standard_normal((layers, H, D)) * std).astype(np.float32)
    out["w"] = (g.standard_normal((layers, H, D)) * std).astype(np.float32)
    return out


def hidden_states(shape: LayerShape, seed: int, rows: int) -> np.ndarray:
    """[rows, B, d_model] float32 hidden states ~ N(0, 1)."""
    return rng(seed).standard_normal((rows, shape.batch, shape.d_model), dtype=np.float32)


def sample_rows(shape: LayerShape, seed: int, n_random: int, all_heads_of_b0: bool = True
                ) -> np.ndarray:
    """(b, h, i) triples to check at full size: every head and position of
    batch 0 (when asked) plus ``n_random`` uniform picks."""
    g = rng(seed + 7919)
    rows = []
    if all_heads_of_b0:
        hh, ii = np.meshgrid(np.arange(shape.heads), np.arange(shape.seg_len), indexing="ij")
        rows.append(np.stack([np.zeros(hh.size, dtype=np.int64), hh.ravel(), ii.ravel()], 1))
    if n_random:
        rows.append(np.stack([g.integers(0, shape.batch, n_random),
                              g.integers(0, shape.heads, n_random),
                              g.integers(0, shape.seg_len, n_random)], 1).astype(np.int64))
    return np.concatenate(rows, 0) if rows else np.zeros((0, 3), dtype=np.int64)
