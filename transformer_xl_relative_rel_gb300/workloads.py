"""The synthetic workloads, shaped like the pages' language-modelling settings.

Transformer-XL's experiments (Section 4.1) train with memory equal to the
segment length and evaluate with much longer memories: attention lengths of 384
(training) and 1,600 (evaluation) on WikiText-103-sized models, and longer
memories (3,800 at evaluation) for character-level models.  No text from those
corpora is used; the inputs below stand in for them (seeded, synthetic).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Tuple

from .inputs import LayerShape


@dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    layers: int
    segments: int
    dtype: str          # "f32" or "bf16"
    seed: int
    init: str          # "unit": q,k,v,r ~ N(0,1); "lm": hidden N(0,1), weights N(0, 0.02^2)
    note: str = ""

    def flops_per_call(self) -> float:
        """Algorithmic FLOPs of one layer call: 2*D each for the content term,
        the position term and the value product, over the visible pairs."""
        s = self.shape
        pairs = s.seg_len * s.mem_len + s.seg_len * (s.seg_len + 1) // 2
        return 6.0 * s.d_head * s.batch * s.heads * pairs

    def issued_flops_per_call(self, splits: int = 1) -> float:
        """FLOPs the bf16 kernel issues to the tensor cores for one call: per
        128-key tile of a 128-row query tile, the content tile (2*128*128*DP,
        DP = D padded to 16), the tile's whole 256-column band window
        (2*128*256*DP: rows need columns 127-i .. 254-i) and the P.V tile
        (2*128*128*DP).  Tiles past a query tile's causal limit are not
        issued; key splits only partition the tiles."""
        s = self.shape
        dp = (s.d_head + 15) // 16 * 16
        per = 2.0 * 128 * 128 * dp
        nqt = (s.seg_len + 127) // 128
        total = 0.0
        for qt in range(nqt):
            kend = min(s.klen, s.mem_len + min(s.seg_len, (qt + 1) * 128))
            ntile = (kend + 127) // 128
            total += 4 * per * ntile
        return total * s.batch * s.heads

    def bytes_per_call(self) -> float:
        """Minimum HBM bytes of one layer call: q and out once, k and v once,
        r once (element size of the workload's dtype; u, v biases are tiny)."""
        s = self.shape
        e = 4 if self.dtype == "f32" else 2
        dm = s.d_model
        return e * (2 * s.batch * s.seg_len * dm + 2 * s.batch * s.klen * dm + s.klen * dm)

    def rollover_bytes(self) -> float:
        """HBM bytes of one memory rollover (read M rows, write M rows)."""
        s = self.shape
        e = 4 if self.dtype == "f32" else 2
        return 2.0 * e * s.mem_len * s.batch * s.d_model


def _w(name, B, H, D, L, M, layers, segments, dtype, seed, init, note=""):
    return Workload(name, LayerShape(B, H, D, L, M), layers, segments, dtype, seed, init, note)


WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    _w("tiny_f32", 1, 2, 16, 16, 16, 1, 1, "f32", 1, "unit",
       "tiny fp32 check, single layer forward"),
    _w("base_lm", 60, 10, 41, 150, 150, 16, 4, "bf16", 2, "lm",
       "base-LM shape (d_model 410), 16 layers x 4 segments"),
    _w("large_lm", 16, 16, 64, 384, 384, 18, 4, "bf16", 3, "lm",
       "large-LM shape (d_model 1024), 18 layers x 4 segments"),
    _w("long_mem_b1", 1, 16, 64, 128, 1600, 1, 1, "bf16", 4, "lm", "long-memory evaluation"),
    _w("long_mem_b2", 2, 16, 64, 128, 1600, 1, 1, "bf16", 4, "lm", "long-memory evaluation"),
    _w("long_mem_b4", 4, 16, 64, 128, 1600, 1, 1, "bf16", 4, "lm", "long-memory evaluation"),
    _w("long_mem_b8", 8, 16, 64, 128, 1600, 1, 1, "bf16", 4, "lm", "long-memory evaluation"),
    _w("long_mem_b16", 16, 16, 64, 128, 1600, 1, 1, "bf16", 4, "lm", "long-memory evaluation"),
    _w("char_train", 22, 8, 64, 768, 768, 24, 8, "bf16", 5, "lm",
       "char-LM training shape (d_model 512), 24 layers x 8 segments"),
    _w("char_eval", 22, 8, 64, 128, 3800, 24, 8, "bf16", 5, "lm",
       "char-LM evaluation shape (d_model 512), 24 layers x 8 segments"),
]}

#: the benchmark's default workload: the largest per-call work, the only
#: clearly tensor-bound shape, where the tensor-roofline fraction is quoted.
DEFAULT_BENCH = "char_train"


def as_tuple(w: Workload) -> Tuple[int, int, int, int, int]:
    s = w.shape
    return s.batch, s.heads, s.d_head, s.seg_len, s.mem_len
