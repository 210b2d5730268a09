"""ctypes binding of libtxl (the C ABI in include/txl.h).

Argument marshalling only: the functions take torch tensors that already live
on the GPU, check their shapes, dtypes and layouts, and pass raw device
pointers and sizes to the library.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU path.  If ``libtxl.so`` is missing the
first call raises ``TxlError``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

TXL_F32 = 0
TXL_BF16 = 1

_STATUS = {0: "TXL_OK", 1: "TXL_ERR_INVALID", 2: "TXL_ERR_UNSUPPORTED", 3: "TXL_ERR_CUDA",
           4: "TXL_ERR_TIMEOUT"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libtxl.so"
_lib: Optional[ctypes.CDLL] = None

#: every symbol include/txl.h declares (checked by the host-side tests)
EXPORTS = ("txl_rel_attn_fwd", "txl_mem_update", "txl_check", "txl_status_string",
           "txl_last_cuda_error", "txl_version", "txl_shutdown", "txl_rel_attn_fwd_noalloc",
           "txl_rel_attn_fwd_ring", "txl_ring_append", "txl_rel_attn_fwd_padded", "txl_project_heads",
           "txl_project_qkv", "txl_project_qkv_cells", "txl_rel_table", "txl_rel_attn_bwd", "txl_rel_attn_bwd_workspace", "txl_rel_attn_fwd_lse", "txl_rel_attn_fwd_mem", "txl_rel_attn_fwd_mem_cells", "txl_rel_attn_fwd_plan", "txl_selftest_wait")


class TxlError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_STATUS.get(status, status)}")


def library_path() -> str:
    return os.path.join(_HERE, _LIB_NAME)


def load_library() -> ctypes.CDLL:
    """Load libtxl.so from the package directory (built by ``_build.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise TxlError(3, f"{path} not built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.txl_rel_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.txl_rel_attn_fwd.restype = i
    lib.txl_rel_attn_fwd_lse.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp]
    lib.txl_rel_attn_fwd_lse.restype = i
    ip = ctypes.POINTER(ctypes.c_int)
    lib.txl_rel_attn_fwd_plan.argtypes = [i, i, i, i, i, i, ip, ip]
    lib.txl_rel_attn_fwd_plan.restype = i
    lib.txl_rel_attn_fwd_mem.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp, i, vp]
    lib.txl_rel_attn_fwd_mem.restype = i
    pp = ctypes.POINTER(vp)
    lib.txl_rel_attn_fwd_mem_cells.argtypes = [i, pp, pp, pp, pp, pp, pp, i, i, i, i, i, i, pp, pp, pp, i, vp]
    lib.txl_rel_attn_fwd_mem_cells.restype = i
    lib.txl_rel_attn_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp]
    lib.txl_rel_attn_fwd_noalloc.restype = i
    lib.txl_rel_attn_fwd_ring.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp]
    lib.txl_rel_attn_fwd_ring.restype = i
    lib.txl_ring_append.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.txl_ring_append.restype = i
    lib.txl_rel_attn_fwd_padded.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp]
    lib.txl_rel_attn_fwd_padded.restype = i
    lib.txl_project_heads.argtypes = [vp, vp, vp, i, i, i, i, i, i, vp]
    lib.txl_project_heads.restype = i
    lib.txl_project_qkv.argtypes = [vp, i, i, vp, vp, vp, vp, vp, vp, i, i, i, i, i, vp]
    lib.txl_project_qkv.restype = i
    pp = ctypes.POINTER(ctypes.c_void_p)
    lib.txl_project_qkv_cells.argtypes = [i, pp, pp, pp, pp, pp, pp, pp, i, i, i, i, i, i, i, vp]
    lib.txl_project_qkv_cells.restype = i
    lib.txl_rel_table.argtypes = [vp, vp, i, i, i, i, i, i, vp]
    lib.txl_rel_table.restype = i
    lib.txl_rel_attn_bwd_workspace.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
    lib.txl_rel_attn_bwd_workspace.restype = i
    lib.txl_rel_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                     vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.txl_rel_attn_bwd.restype = i
    lib.txl_mem_update.argtypes = [vp, vp, i, i, i, i, i, vp]
    lib.txl_mem_update.restype = i
    lib.txl_selftest_wait.argtypes = [ctypes.c_uint, vp]
    lib.txl_selftest_wait.restype = i
    lib.txl_check.argtypes = [vp]
    lib.txl_check.restype = i
    lib.txl_status_string.argtypes = [i]
    lib.txl_status_string.restype = ctypes.c_char_p
    lib.txl_last_cuda_error.argtypes = []
    lib.txl_last_cuda_error.restype = i
    lib.txl_version.argtypes = []
    lib.txl_version.restype = i
    lib.txl_shutdown.argtypes = []
    lib.txl_shutdown.restype = None
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().txl_status_string(int(status)).decode()


def _raise(st: int, what: str):
    if st != 0:
        lib = load_library()
        msg = f"{what} ({lib.txl_status_string(st).decode()}"
        if st == 3:
            msg += f", cuda error {lib.txl_last_cuda_error()}"
        raise TxlError(st, msg + ")")


def _stream_ptr(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return TXL_F32
    if t.dtype == torch.bfloat16:
        return TXL_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t) -> Optional[int]:
    return t.data_ptr() if t is not None and t.numel() > 0 else None


def _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out):
    import torch
    L, B, H, D = q.shape
    T = mem_len + L
    for name, t, shp in (("k", k, (T, B, H, D)), ("v", v, (T, B, H, D)), ("r", r, (T, H, D))):
        if tuple(t.shape) != shp:
            raise ValueError(f"{name} must be {list(shp)}, got {list(t.shape)}")
        if t.dtype != q.dtype:
            raise TypeError(f"{name} dtype {t.dtype} != q dtype {q.dtype}")
    for name, t in (("u_bias", u_bias), ("v_bias", v_bias)):
        if t is not None and (tuple(t.shape) != (H, D) or t.dtype != torch.float32):
            raise ValueError(f"{name} must be float32 [{H}, {D}] or None")
    if out is not None and (tuple(out.shape) != (L, B, H, D) or out.dtype != q.dtype):
        raise ValueError("out must be a contiguous tensor shaped and typed like q")
    for t in (q, k, v, r, u_bias, v_bias, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty_like(q)
    return out


def rel_attn_fwd(q, k, v, r, u_bias, v_bias, mem_len: int, out=None, stream=None, lse=None):
    """Relative attention of one layer (Transformer-XL Section 3.3).

    q: [L, B, H, D]; k, v: [M+L, B, H, D]; r: [M+L, H, D] (reversed table);
    u_bias, v_bias: [H, D] float32, or None to drop that bias term (both
    None: Shaw et al.'s form, terms (a) + (b) only); all CUDA, contiguous,
    same dtype (float32 or bfloat16) except the biases.  Returns ``out``
    [L, B, H, D].  ``lse`` (bfloat16 inputs only): a contiguous float32 CUDA
    tensor [B, H, L] that receives each query row's log-sum-exp of its
    scaled scores (txl_rel_attn_fwd_lse), to hand to ``rel_attn_bwd``.
    """
    import torch
    L, B, H, D = q.shape
    out = _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out)
    if lse is None:
        st = load_library().txl_rel_attn_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
            B, mem_len, L, H, D, _dtype_code(q), _ptr(out), _stream_ptr(stream))
        _raise(st, "txl_rel_attn_fwd")
        return out
    if tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32 or not lse.is_cuda \
            or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous float32 CUDA tensor [{B}, {H}, {L}]")
    st = load_library().txl_rel_attn_fwd_lse(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
        B, mem_len, L, H, D, _dtype_code(q), _ptr(out), _ptr(lse), _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_lse")
    return out


def rel_attn_fwd_plan(batch: int, mem_len: int, seg_len: int, heads: int, d_head: int,
                      dtype_code: int) -> tuple:
    """(key splits, kernel launches) of a txl_rel_attn_fwd call of this shape."""
    sp, nl = ctypes.c_int(0), ctypes.c_int(0)
    st = load_library().txl_rel_attn_fwd_plan(batch, mem_len, seg_len, heads, d_head, dtype_code,
                                              ctypes.byref(sp), ctypes.byref(nl))
    _raise(st, "txl_rel_attn_fwd_plan")
    return int(sp.value), int(nl.value)


def rel_attn_fwd_mem(q, k, v, r, u_bias, v_bias, mem_len: int, mem_next, ext_ctx, out=None, stream=None):
    """``rel_attn_fwd`` and ``mem_update`` of one layer in one call
    (txl_rel_attn_fwd_mem): returns ``out``; ``mem_next`` receives the newest
    ``mem_len`` rows of ``ext_ctx`` [M+L, B, d_model] (same dtype as q)."""
    L, B, H, D = q.shape
    out = _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out)
    if ext_ctx.dim() != 3 or ext_ctx.shape[0] != mem_len + L or ext_ctx.shape[1] != B:
        raise ValueError(f"ext_ctx must be [{mem_len + L}, {B}, d_model]")
    dm = ext_ctx.shape[2]
    for name, t in (("ext_ctx", ext_ctx), ("mem_next", mem_next)):
        if t.dtype != q.dtype or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor typed like q")
    if mem_next.numel() < mem_len * B * dm:
        raise ValueError(f"mem_next must hold at least [{mem_len}, {B}, {dm}]")
    st = load_library().txl_rel_attn_fwd_mem(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
        B, mem_len, L, H, D, _dtype_code(q), _ptr(out), _ptr(mem_next), _ptr(ext_ctx), dm, _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_mem")
    return out


def rel_attn_fwd_mem_cells(qs, ks, vs, rs, us, ws, mem_len: int, mem_nexts, ext_ctxs, outs=None, stream=None):
    """Several independent ``rel_attn_fwd_mem`` calls of one shape
    (txl_rel_attn_fwd_mem_cells): lists of equal length, call c taking
    qs[c] .. ext_ctxs[c] (``us``/``ws`` may be None, or hold None entries).
    Returns the list of outputs."""
    n = len(qs)
    lists = [ks, vs, rs, mem_nexts, ext_ctxs] + [x for x in (us, ws, outs) if x is not None]
    if any(len(x) != n for x in lists):
        raise ValueError("the calls' lists must have the same length")
    if n == 0:
        return []
    L, B, H, D = qs[0].shape
    dm = ext_ctxs[0].shape[2] if ext_ctxs[0].dim() == 3 else -1
    for c in range(n):
        if tuple(qs[c].shape) != (L, B, H, D) or qs[c].dtype != qs[0].dtype:
            raise ValueError("every call's q must have the first call's shape and dtype")
        if tuple(ext_ctxs[c].shape) != (mem_len + L, B, dm):
            raise ValueError(f"ext_ctx must be [{mem_len + L}, {B}, {dm}] in every call")
    res = []
    for c in range(n):
        u = None if us is None else us[c]
        w = None if ws is None else ws[c]
        out = _check_attn(qs[c], ks[c], vs[c], rs[c], u, w, mem_len, None if outs is None else outs[c])
        ext, nxt = ext_ctxs[c], mem_nexts[c]
        for name, t in (("ext_ctx", ext), ("mem_next", nxt)):
            if t.dtype != qs[0].dtype or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous CUDA tensor typed like q")
        if nxt.numel() < mem_len * B * dm:
            raise ValueError(f"mem_next must hold at least [{mem_len}, {B}, {dm}]")
        res.append(out)
    arr = lambda ts: (ctypes.c_void_p * n)(*[_ptr(t) for t in ts])
    st = load_library().txl_rel_attn_fwd_mem_cells(
        n, arr(qs), arr(ks), arr(vs), arr(rs), None if us is None else arr(us), None if ws is None else arr(ws),
        B, mem_len, L, H, D, _dtype_code(qs[0]), arr(res), arr(mem_nexts), arr(ext_ctxs), dm, _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_mem_cells")
    return res


def rel_attn_bwd_workspace_bytes(batch: int, mem_len: int, seg_len: int, heads: int, d_head: int,
                                 dtype_code: int) -> int:
    """Workspace bytes txl_rel_attn_bwd needs for this shape."""
    n = ctypes.c_size_t(0)
    st = load_library().txl_rel_attn_bwd_workspace(batch, mem_len, seg_len, heads, d_head, dtype_code,
                                                   ctypes.byref(n))
    _raise(st, "txl_rel_attn_bwd_workspace")
    return int(n.value)


def rel_attn_bwd(q, k, v, r, u_bias, v_bias, dout, mem_len: int, workspace=None, grads=None,
                 bias_grads: bool = True, stream=None, out=None, lse=None):
    """Gradients of ``rel_attn_fwd`` for the output gradient ``dout`` (shaped
    like q).  Returns a dict ``dq, dk, dv, dr`` (shaped and typed like q, k,
    v, r) and ``du, dw`` (float32 [H, D]; None when ``bias_grads`` is False).
    ``workspace``: a CUDA uint8 tensor of at least
    ``rel_attn_bwd_workspace_bytes`` bytes (allocated when None); ``grads``:
    preallocated outputs with the same keys.  ``out``, ``lse``: the forward's
    output and row log-sum-exp from ``rel_attn_fwd(..., lse=...)`` on the
    same inputs (both or neither); given, the backward skips its own
    forward."""
    import torch
    L, B, H, D = q.shape
    _check_attn(q, k, v, r, u_bias, v_bias, mem_len, q)
    if tuple(dout.shape) != (L, B, H, D) or dout.dtype != q.dtype or not dout.is_cuda \
            or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous CUDA tensor shaped and typed like q")
    if grads is None:
        grads = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                     dr=torch.empty_like(r))
        if bias_grads:
            grads["du"] = torch.empty((H, D), dtype=torch.float32, device=q.device)
            grads["dw"] = torch.empty((H, D), dtype=torch.float32, device=q.device)
    grads.setdefault("du", None)
    grads.setdefault("dw", None)
    if (out is None) != (lse is None):
        raise ValueError("out and lse come together or not at all")
    if out is not None:
        if tuple(out.shape) != (L, B, H, D) or out.dtype != q.dtype or not out.is_cuda \
                or not out.is_contiguous():
            raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
        if tuple(lse.shape) != (B, H, L) or lse.dtype != torch.float32 or not lse.is_cuda \
                or not lse.is_contiguous():
            raise ValueError(f"lse must be a contiguous float32 CUDA tensor [{B}, {H}, {L}]")
    nbytes = rel_attn_bwd_workspace_bytes(B, mem_len, L, H, D, _dtype_code(q))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    elif workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace must hold {nbytes} bytes")
    st = load_library().txl_rel_attn_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias), _ptr(dout), _ptr(out), _ptr(lse),
        B, mem_len, L, H, D, _dtype_code(q),
        _ptr(grads["dq"]), _ptr(grads["dk"]), _ptr(grads["dv"]), _ptr(grads["dr"]),
        _ptr(grads["du"]), _ptr(grads["dw"]), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _raise(st, "txl_rel_attn_bwd")
    return grads


def rel_attn_fwd_ring(q, k, v, r, u_bias, v_bias, mem_len: int, kv_start: int, out=None, stream=None):
    """rel_attn_fwd with k, v stored as a ring of M+L rows: the context's key j
    (0 = oldest memory row) is at row (kv_start + j) mod (M+L)."""
    L, B, H, D = q.shape
    out = _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out)
    st = load_library().txl_rel_attn_fwd_ring(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
        B, mem_len, L, H, D, int(kv_start), _dtype_code(q), _ptr(out), _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_ring")
    return out


def rel_attn_fwd_padded(q, k, v, r, u_bias, v_bias, mem_len: int, d_head: int, out=None, stream=None):
    """rel_attn_fwd on head vectors padded to q.shape[-1] elements (zeros past
    ``d_head``), as project_heads / rel_table write them."""
    L, B, H, Dp = q.shape
    out = _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out)
    st = load_library().txl_rel_attn_fwd_padded(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
        B, mem_len, L, H, int(d_head), Dp, _dtype_code(q), _ptr(out), _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_padded")
    return out


def project_heads(x, w, heads: int, d_head: int, d_pad: int, out=None, stream=None):
    """y[..., heads, d_pad] = x[..., d_in] @ w.T with ``w`` the paper's
    [heads*d_head, d_in] projection (torch.nn.Linear's weight layout);
    padding columns d_head.. are zero.  x: [*lead, d_in]; returns
    [*lead, heads, d_pad]."""
    import torch
    lead = tuple(x.shape[:-1])
    d_in = x.shape[-1]
    rows = 1
    for n in lead:
        rows *= n
    if tuple(w.shape) != (heads * d_head, d_in) or w.dtype != x.dtype:
        raise ValueError(f"w must be [{heads * d_head}, {d_in}] of x's dtype")
    if out is not None and (tuple(out.shape) != lead + (heads, d_pad) or out.dtype != x.dtype):
        raise ValueError(f"out must be {list(lead + (heads, d_pad))} of x's dtype")
    for t in (x, w, out):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    if out is None:
        out = torch.empty(*lead, heads, d_pad, dtype=x.dtype, device=x.device)
    st = load_library().txl_project_heads(_ptr(x), _ptr(w), _ptr(out), rows, d_in, heads, d_head, d_pad,
                                          _dtype_code(x), _stream_ptr(stream))
    _raise(st, "txl_project_heads")
    return out


def _qkv_prepare(x, w_q, w_k, w_v, heads, d_head, d_pad, q_from, q, k, v):
    """project_qkv's argument checks; returns its (q, k, v) outputs, allocated where not given."""
    import torch
    T = x.shape[0]
    rest = tuple(x.shape[1:-1])
    d_in = x.shape[-1]
    per = 1
    for n in rest:
        per *= n
    if not 0 <= q_from <= T:
        raise ValueError(f"q_from must lie in [0, {T}]")
    for name, w in (("w_q", w_q), ("w_k", w_k), ("w_v", w_v)):
        if w is None and name != "w_q":
            raise ValueError(f"{name} is required")
        if w is not None and (tuple(w.shape) != (heads * d_head, d_in) or w.dtype != x.dtype):
            raise ValueError(f"{name} must be [{heads * d_head}, {d_in}] of x's dtype")
    if w_q is None and q is not None:
        raise ValueError("q is given without w_q")
    shapes = {"q": (T - q_from,) + rest + (heads, d_pad), "k": (T,) + rest + (heads, d_pad),
              "v": (T,) + rest + (heads, d_pad)}
    outs = {"q": q, "k": k, "v": v}
    for name, t in outs.items():
        if t is not None and (tuple(t.shape) != shapes[name] or t.dtype != x.dtype):
            raise ValueError(f"{name} must be {list(shapes[name])} of x's dtype")
    for t in (x, w_q, w_k, w_v, q, k, v):
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")
    for name in ("k", "v") + (("q",) if w_q is not None else ()):
        if outs[name] is None:
            outs[name] = torch.empty(*shapes[name], dtype=x.dtype, device=x.device)
    return outs["q"], outs["k"], outs["v"]


def project_qkv(x, w_q, w_k, w_v, heads: int, d_head: int, d_pad: int, q_from: int = 0,
                q=None, k=None, v=None, stream=None):
    """A layer's q, k, v projections of one extended context: k = x @ w_k.T
    and v = x @ w_v.T over all of x's leading positions, q = x[q_from:] @
    w_q.T (the segment's own positions; ``w_q=None`` skips q).  x: [T, *rest,
    d_in]; outputs [T or T - q_from, *rest, heads, d_pad], as project_heads
    writes them.  Returns (q, k, v)."""
    T = x.shape[0]
    d_in = x.shape[-1]
    per = 1
    for n in x.shape[1:-1]:
        per *= n
    q, k, v = _qkv_prepare(x, w_q, w_k, w_v, heads, d_head, d_pad, q_from, q, k, v)
    outs = {"q": q, "k": k, "v": v}
    # no q rows (q_from == T): the library is asked for k and v only
    wq_arg = w_q if (w_q is not None and q_from < T) else None
    st = load_library().txl_project_qkv(
        _ptr(x), T * per, d_in, _ptr(wq_arg), _ptr(w_k), _ptr(w_v), _ptr(outs["q"]) if wq_arg is not None else None,
        _ptr(outs["k"]), _ptr(outs["v"]), q_from * per, heads, d_head, d_pad, _dtype_code(x), _stream_ptr(stream))
    _raise(st, "txl_project_qkv")
    return outs["q"], outs["k"], outs["v"]


def project_qkv_cells(xs, wqs, wks, wvs, heads: int, d_head: int, d_pad: int, q_from: int = 0,
                      qs=None, ks=None, vs=None, stream=None):
    """project_qkv for several layer calls of one shape at once (lists of
    equal length: the cells' extended contexts, their weights and, if given,
    their outputs); ``wqs=None`` skips q.  Returns (qs, ks, vs) lists."""
    n = len(xs)
    if not (len(wks) == len(wvs) == n and (wqs is None or len(wqs) == n)):
        raise ValueError("the cells' lists must have the same length")
    if n == 0:
        return [], [], []
    T = xs[0].shape[0]
    shape = tuple(xs[0].shape)
    for x in xs:
        if tuple(x.shape) != shape or x.dtype != xs[0].dtype:
            raise ValueError("every cell's x must have the first cell's shape and dtype")
    res = {"q": [], "k": [], "v": []}
    for c in range(n):
        # per cell, the single-cell binding's checks and allocations (no call)
        q1, k1, v1 = _qkv_prepare(xs[c], None if wqs is None else wqs[c], wks[c], wvs[c], heads, d_head, d_pad,
                                  q_from, None if qs is None else qs[c], None if ks is None else ks[c],
                                  None if vs is None else vs[c])
        res["q"].append(q1)
        res["k"].append(k1)
        res["v"].append(v1)
    per = 1
    for d in shape[1:-1]:
        per *= d
    with_q = wqs is not None and q_from < T
    arr = lambda ts: (ctypes.c_void_p * n)(*[_ptr(t) for t in ts])
    st = load_library().txl_project_qkv_cells(
        n, arr(xs), arr(wqs) if with_q else None, arr(wks), arr(wvs), arr(res["q"]) if with_q else None,
        arr(res["k"]), arr(res["v"]), T * per, shape[-1], q_from * per, heads, d_head, d_pad, _dtype_code(xs[0]),
        _stream_ptr(stream))
    _raise(st, "txl_project_qkv_cells")
    return (res["q"] if wqs is not None else None), res["k"], res["v"]


def rel_table(w_r, klen: int, heads: int, d_head: int, d_pad: int, out=None, stream=None):
    """Appendix B's reversed projected table [klen, heads, d_pad] from W_kR in
    the paper's layout [heads*d_head, d_model] and the sinusoid of the
    relative distance."""
    import torch
    if w_r.dim() != 2 or w_r.shape[0] != heads * d_head or not w_r.is_cuda or not w_r.is_contiguous():
        raise ValueError(f"w_r must be a contiguous CUDA [{heads * d_head}, d_model] tensor")
    d_model = w_r.shape[1]
    if out is None:
        out = torch.empty(klen, heads, d_pad, dtype=w_r.dtype, device=w_r.device)
    st = load_library().txl_rel_table(_ptr(w_r), _ptr(out), klen, d_model, heads, d_head, d_pad,
                                      _dtype_code(w_r), _stream_ptr(stream))
    _raise(st, "txl_rel_table")
    return out


def ring_append(ring, rows, start: int, stream=None):
    """Write ``rows`` [n, ...] into ``ring`` [ring_len, ...] at rows
    (start + i) mod ring_len; returns the next start, (start + n) mod ring_len."""
    n = rows.shape[0]
    ring_len = ring.shape[0]
    if tuple(rows.shape[1:]) != tuple(ring.shape[1:]) or rows.dtype != ring.dtype:
        raise ValueError("rows must match the ring's row shape and dtype")
    for t in (ring, rows):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    row_elems = ring[0].numel() if ring_len else 0
    st = load_library().txl_ring_append(_ptr(ring), _ptr(rows), ring_len, n, row_elems, int(start),
                                        _dtype_code(ring), _stream_ptr(stream))
    _raise(st, "txl_ring_append")
    return (start + n) % ring_len if ring_len else 0


def rel_attn_fwd_noalloc(q, k, v, r, u_bias, v_bias, mem_len: int, out, stream=None):
    """The same call through txl_rel_attn_fwd_noalloc, for callers that may not
    allocate device memory: ``out`` must be given, and the library allocates
    nothing (its split-key scratch is a fixed array in the library).  The
    arguments are checked exactly as ``rel_attn_fwd`` checks them."""
    if out is None:
        raise ValueError("out must be given: this entry point allocates nothing")
    L, B, H, D = q.shape
    _check_attn(q, k, v, r, u_bias, v_bias, mem_len, out)
    code = _dtype_code(q)
    st = load_library().txl_rel_attn_fwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(r), _ptr(u_bias), _ptr(v_bias),
        B, mem_len, L, H, D, code, _ptr(out), _stream_ptr(stream))
    _raise(st, "txl_rel_attn_fwd_noalloc")
    return out


def rel_attn_fwd_raw(q_ptr, k_ptr, v_ptr, r_ptr, u_ptr, w_ptr, batch, mem_len, seg_len,
                     heads, d_head, dtype_code, out_ptr, stream_ptr) -> int:
    """The C entry point with raw integers (for host-side argument tests)."""
    return load_library().txl_rel_attn_fwd(q_ptr, k_ptr, v_ptr, r_ptr, u_ptr, w_ptr, batch,
                                           mem_len, seg_len, heads, d_head, dtype_code,
                                           out_ptr, stream_ptr)


def mem_update(mem_next, ext_ctx, mem_len: int, stream=None):
    """Memory rollover (Section 3.2): mem_next[:M] = newest M rows of ext_ctx.

    ext_ctx: [M+L, B, d_model]; mem_next: [>= M, B, d_model]; same dtype.
    """
    T, B, dm = ext_ctx.shape
    L = T - mem_len
    if L < 0:
        raise ValueError("mem_len larger than the extended context")
    if mem_next.dim() != 3 or mem_next.shape[0] < mem_len or tuple(mem_next.shape[1:]) != (B, dm):
        raise ValueError(f"mem_next must be [>= {mem_len}, {B}, {dm}]")
    if mem_next.dtype != ext_ctx.dtype:
        raise TypeError("mem_next and ext_ctx dtypes differ")
    for t in (mem_next, ext_ctx):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    st = load_library().txl_mem_update(_ptr(mem_next), _ptr(ext_ctx), B, mem_len, L, dm,
                                       _dtype_code(ext_ctx), _stream_ptr(stream))
    _raise(st, "txl_mem_update")
    return mem_next


def mem_update_raw(dst_ptr, src_ptr, batch, mem_len, seg_len, d_model, dtype_code,
                   stream_ptr) -> int:
    return load_library().txl_mem_update(dst_ptr, src_ptr, batch, mem_len, seg_len, d_model,
                                         dtype_code, stream_ptr)


def selftest_wait(limit_us: int, stream=None) -> None:
    """Launch the bounded-wait self test (txl_selftest_wait): a wait that runs
    out after ``limit_us`` microseconds; the next ``check`` raises
    TXL_ERR_TIMEOUT."""
    _raise(load_library().txl_selftest_wait(int(limit_us), _stream_ptr(stream)), "txl_selftest_wait")


def check(stream=None) -> None:
    """Synchronise the stream and raise if a kernel reported an error."""
    _raise(load_library().txl_check(_stream_ptr(stream)), "txl_check")
