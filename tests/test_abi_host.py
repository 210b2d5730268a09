"""Host-side checks of the C ABI: the library builds and loads, exports every
symbol include/txl.h declares, and rejects bad arguments before launching
anything.  No compute call is made here (these run without a GPU)."""
import ctypes
import os
import re

import pytest

import transformer_xl_relative_rel_gb300 as txl
from transformer_xl_relative_rel_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT = 0, 1, 2, 3, 4
FAKE = 0x10000   # 16-byte aligned, never dereferenced: every call below fails validation first


@pytest.fixture(scope="module")
def lib():
    from transformer_xl_relative_rel_gb300 import _build
    _build.build()
    return abi.load_library()


def test_header_declares_exactly_the_exports(lib):
    hdr = open(os.path.join(ROOT, "include", "txl.h")).read()
    declared = set(re.findall(r"\b(txl_[a-z_0-9]+)\s*\(", hdr))
    assert declared == set(abi.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for st in (OK, INVALID, UNSUPPORTED, CUDA, TIMEOUT):
        assert txl.status_string(st)
    assert txl.status_string(99) == "unknown status"
    assert lib.txl_version() >= 100


def _attn(**kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, r=FAKE * 4, u=FAKE * 5, w=FAKE * 6, B=2, M=8, L=8, H=2,
             D=16, dt=1, out=FAKE * 7, stream=None)
    a.update(kw)
    return abi.rel_attn_fwd_raw(a["q"], a["k"], a["v"], a["r"], a["u"], a["w"], a["B"], a["M"],
                                a["L"], a["H"], a["D"], a["dt"], a["out"], a["stream"])


def test_attn_rejects_bad_arguments(lib):
    assert _attn(dt=7) == UNSUPPORTED
    assert _attn(B=-1) == INVALID
    assert _attn(M=-1) == INVALID
    assert _attn(L=-3) == INVALID
    assert _attn(D=0) == INVALID
    assert _attn(D=129, dt=0) == UNSUPPORTED
    assert _attn(D=65, dt=1) == UNSUPPORTED
    assert _attn(q=None) == INVALID
    assert _attn(out=None) == INVALID
    assert _attn(q=FAKE + 2) == INVALID            # misaligned
    assert _attn(u=FAKE + 2) == INVALID
    assert _attn(out=FAKE) == INVALID              # out overlaps q
    assert _attn(out=FAKE * 2 + 64) == INVALID     # out overlaps k


def test_attn_accepts_absent_biases(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the call would launch on the fake pointers")
    # a NULL bias drops its term (Shaw et al.'s form): the arguments pass and
    # the call fails only at the device, which this machine does not have
    assert _attn(u=None) == CUDA
    assert _attn(u=None, w=None) == CUDA


def test_attn_empty_is_a_no_op(lib):
    # nothing to compute: OK without touching any pointer (NULLs allowed)
    assert _attn(B=0, q=None, k=None, v=None, r=None, u=None, w=None, out=None) == OK
    assert _attn(L=0, q=None, k=None, v=None, r=None, u=None, w=None, out=None) == OK
    assert _attn(H=0, q=None, k=None, v=None, r=None, u=None, w=None, out=None) == OK


def _attn_mem(**kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, r=FAKE * 4, u=FAKE * 5, w=FAKE * 6, B=2, M=8, L=8, H=2,
             D=16, dt=1, out=FAKE * 7, mem_next=FAKE * 8, ext=FAKE * 9, dm=32, stream=None)
    a.update(kw)
    return abi.load_library().txl_rel_attn_fwd_mem(
        a["q"], a["k"], a["v"], a["r"], a["u"], a["w"], a["B"], a["M"], a["L"], a["H"], a["D"], a["dt"],
        a["out"], a["mem_next"], a["ext"], a["dm"], a["stream"])


def test_attn_mem_rejects_bad_arguments(lib):
    assert _attn_mem(dt=7) == UNSUPPORTED
    assert _attn_mem(dm=-1) == INVALID
    assert _attn_mem(mem_next=None) == INVALID
    assert _attn_mem(ext=None) == INVALID
    assert _attn_mem(mem_next=FAKE * 8 + 1) == INVALID          # misaligned
    assert _attn_mem(mem_next=FAKE * 9 + 64) == INVALID         # mem_next overlaps ext_ctx
    assert _attn_mem(mem_next=FAKE * 2 + 32) == INVALID         # mem_next overlaps k
    assert _attn_mem(mem_next=FAKE * 7) == INVALID              # mem_next overlaps out
    assert _attn_mem(ext=FAKE * 7 - 64) == INVALID              # ext_ctx overlaps out
    assert _attn_mem(q=None) == INVALID                         # the attention's own checks
    assert _attn_mem(D=65) == UNSUPPORTED
    # nothing to do at all: OK without touching a pointer
    assert _attn_mem(B=0, M=0, q=None, k=None, v=None, r=None, u=None, w=None, out=None, mem_next=None,
                     ext=None) == OK
    # nothing to roll: the attention alone (its pointers are still checked)
    assert _attn_mem(M=0, mem_next=None, ext=None, q=None) == INVALID


def test_attn_mem_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the call would launch on the fake pointers")
    assert _attn_mem() == CUDA
    assert _attn_mem(H=0) == CUDA             # no heads: the rollover alone still launches
    assert _attn_mem(B=0) == OK               # no batch: nothing to attend and no rows to roll


def test_attn_plan(lib):
    import torch
    # the training shape runs unsplit in one launch; a head size other than 64
    # adds the padding copies; fp32 is one launch; nothing to do is no launch
    if not torch.cuda.is_available():
        assert txl.rel_attn_fwd_plan(22, 768, 768, 8, 64, txl.TXL_BF16) == (1, 1)
        sp, nl = txl.rel_attn_fwd_plan(60, 150, 150, 10, 41, txl.TXL_BF16)
        assert nl == 3 + (1 if sp > 1 else 0)
    assert txl.rel_attn_fwd_plan(1, 16, 16, 2, 16, txl.TXL_F32) == (1, 1)
    assert txl.rel_attn_fwd_plan(0, 16, 16, 2, 16, txl.TXL_BF16) == (1, 0)
    n = ctypes.c_int(0)
    f = lib.txl_rel_attn_fwd_plan
    assert f(1, 16, 16, 2, 16, 7, ctypes.byref(n), ctypes.byref(n)) == UNSUPPORTED
    assert f(1, 16, 16, 2, 16, 1, None, ctypes.byref(n)) == INVALID
    assert f(1, -1, 16, 2, 16, 1, ctypes.byref(n), ctypes.byref(n)) == INVALID
    assert f(1, 16, 16, 2, 65, 1, ctypes.byref(n), ctypes.byref(n)) == UNSUPPORTED


def test_mem_update_rejects_bad_arguments(lib):
    f = abi.mem_update_raw
    assert f(FAKE, FAKE * 4, 2, 4, 4, 8, 9, None) == UNSUPPORTED
    assert f(FAKE, FAKE * 4, -1, 4, 4, 8, 1, None) == INVALID
    assert f(None, FAKE * 4, 2, 4, 4, 8, 1, None) == INVALID
    assert f(FAKE + 1, FAKE * 4, 2, 4, 4, 8, 1, None) == INVALID     # misaligned
    assert f(FAKE * 4 + 16, FAKE * 4, 2, 4, 4, 8, 1, None) == INVALID  # overlapping buffers
    assert f(None, None, 2, 0, 4, 8, 1, None) == OK                   # M = 0: nothing to copy
    assert f(None, None, 0, 4, 4, 8, 1, None) == OK


def test_no_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.txl_check(None) == CUDA


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(abi, "_lib", None)
    monkeypatch.setattr(abi, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(txl.TxlError):
        abi.load_library()


def test_ring_calls_reject_bad_arguments(lib):
    f = lib.txl_rel_attn_fwd_ring
    args = [FAKE, FAKE * 2, FAKE * 3, FAKE * 4, FAKE * 5, FAKE * 6, 2, 8, 8, 2, 16]
    assert f(*args, -1, 1, FAKE * 7, None) == INVALID      # kv_start < 0
    assert f(*args, 16, 1, FAKE * 7, None) == INVALID      # kv_start >= M+L
    g = lib.txl_ring_append
    assert g(FAKE, FAKE * 4, 10, 11, 8, 0, 1, None) == INVALID   # more rows than the ring
    assert g(FAKE, FAKE * 4, 10, 3, 8, 10, 1, None) == INVALID   # start outside the ring
    assert g(FAKE, FAKE * 4, 10, 3, 8, -1, 1, None) == INVALID
    assert g(FAKE, FAKE + 8, 10, 3, 8, 0, 1, None) == INVALID    # rows overlap the ring
    assert g(None, FAKE * 4, 10, 3, 8, 0, 1, None) == INVALID
    assert g(FAKE, FAKE * 4, 10, 3, 8, 0, 9, None) == UNSUPPORTED
    assert g(None, None, 10, 0, 8, 0, 1, None) == OK              # nothing to copy


def _bwd_ws(B=2, M=8, L=8, H=2, D=16, dt=1):
    n = ctypes.c_size_t(0)
    st = abi.load_library().txl_rel_attn_bwd_workspace(B, M, L, H, D, dt, ctypes.byref(n))
    return st, n.value


def test_bwd_workspace_query(lib):
    st, n = _bwd_ws()
    assert st == OK
    B, M, L, H, D = 2, 8, 8, 2, 16
    # at least the score, P, dP and dA of every (b, h, i, j) (two fp32, three bf16)
    assert n >= B * H * L * (M + L) * (2 * 4 + 3 * 2)
    assert _bwd_ws(dt=0)[1] > n                      # fp32 operands take more
    assert _bwd_ws(B=4)[1] > n
    assert _bwd_ws(dt=7)[0] == UNSUPPORTED
    assert _bwd_ws(D=129)[0] == UNSUPPORTED
    assert _bwd_ws(B=0)[0] == INVALID
    assert _bwd_ws(L=0)[0] == INVALID
    assert _bwd_ws(M=-1)[0] == INVALID
    assert abi.load_library().txl_rel_attn_bwd_workspace(2, 8, 8, 2, 16, 1, None) == INVALID


def _bwd(**kw):
    st, need = _bwd_ws()
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, r=FAKE * 4, u=FAKE * 5, w=FAKE * 6, dout=FAKE * 7,
             out=None, lse=None, B=2, M=8, L=8, H=2, D=16, dt=1, dq=FAKE * 8, dk=FAKE * 9, dv=FAKE * 10,
             dr=FAKE * 11, du=FAKE * 12, dw=FAKE * 13, ws=FAKE * 14, nws=need, stream=None)
    a.update(kw)
    return abi.load_library().txl_rel_attn_bwd(
        a["q"], a["k"], a["v"], a["r"], a["u"], a["w"], a["dout"], a["out"], a["lse"], a["B"], a["M"],
        a["L"], a["H"], a["D"], a["dt"], a["dq"], a["dk"], a["dv"], a["dr"], a["du"], a["dw"], a["ws"],
        a["nws"], a["stream"])


def test_bwd_rejects_bad_arguments(lib):
    assert _bwd(dt=7) == UNSUPPORTED
    assert _bwd(D=129) == UNSUPPORTED
    assert _bwd(B=0) == INVALID
    assert _bwd(L=0) == INVALID
    assert _bwd(M=-2) == INVALID
    for name in ("q", "k", "v", "r", "dout", "dq", "dk", "dv", "dr", "ws"):
        assert _bwd(**{name: None}) == INVALID, name
    assert _bwd(nws=1024) == INVALID                  # workspace too small
    assert _bwd(ws=FAKE * 14 + 16) == INVALID         # workspace not 256-byte aligned
    assert _bwd(q=FAKE + 1) == INVALID                # misaligned bf16 operand
    assert _bwd(du=FAKE * 12 + 2) == INVALID          # misaligned fp32 output
    assert _bwd(dq=FAKE) == INVALID                   # dq overlaps q
    assert _bwd(dv=FAKE * 9 + 64) == INVALID          # dv overlaps dk
    assert _bwd(dr=FAKE * 14 + 4096) == INVALID       # dr inside the workspace
    # the saved forward output and log-sum-exp come together
    assert _bwd(out=FAKE * 15) == INVALID
    assert _bwd(lse=FAKE * 16) == INVALID
    assert _bwd(out=FAKE * 15 + 2, lse=FAKE * 16) == INVALID   # out not 16-byte aligned
    assert _bwd(out=FAKE * 15, lse=FAKE * 16 + 2) == INVALID   # lse not 4-byte aligned
    assert _bwd(out=FAKE * 15, lse=FAKE * 16, dq=FAKE * 15) == INVALID   # dq overlaps out
    assert _bwd(out=FAKE * 15, lse=FAKE * 16, ws=FAKE * 16) == INVALID   # lse inside the workspace


def _attn_lse(**kw):
    a = dict(q=FAKE, k=FAKE * 2, v=FAKE * 3, r=FAKE * 4, u=FAKE * 5, w=FAKE * 6, B=2, M=8, L=8, H=2,
             D=16, dt=1, out=FAKE * 7, lse=FAKE * 8, stream=None)
    a.update(kw)
    return abi.load_library().txl_rel_attn_fwd_lse(
        a["q"], a["k"], a["v"], a["r"], a["u"], a["w"], a["B"], a["M"], a["L"], a["H"], a["D"], a["dt"],
        a["out"], a["lse"], a["stream"])


def test_attn_lse_rejects_bad_arguments(lib):
    assert _attn_lse(lse=None) == INVALID
    assert _attn_lse(dt=0) == UNSUPPORTED             # the log-sum-exp comes from the bf16 kernels
    assert _attn_lse(lse=FAKE * 8 + 2) == INVALID     # misaligned
    assert _attn_lse(lse=FAKE * 7 + 64) == INVALID    # inside out
    assert _attn_lse(lse=FAKE * 2 + 16) == INVALID    # inside k
    assert _attn_lse(B=0, q=None, k=None, v=None, r=None, u=None, w=None, out=None, lse=None) == OK


def test_bwd_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the call would launch on the fake pointers")
    assert _bwd() == CUDA
    assert _bwd(out=FAKE * 15, lse=FAKE * 16) == CUDA
    assert _attn_lse() == CUDA
    assert _bwd(u=None, w=None, du=None, dw=None) == CUDA


def test_selftest_wait_rejects_bad_limits(lib):
    # the limit is checked on the host before anything is launched
    assert lib.txl_selftest_wait(0, None) == INVALID
    assert lib.txl_selftest_wait(1000001, None) == INVALID


def _attn_mem_cells(n=2, dt=1, B=2, M=8, L=8, H=2, D=16, dm=32, swap=None, cells=None):
    """n calls of _attn_mem's shape, call c's buffers FAKE * (16 c + 1 ..)
    (none overlapping); ``swap`` = (name, c, value) replaces one pointer."""
    names = ("q", "k", "v", "r", "u", "w", "out", "mem_next", "ext")
    ptrs = {nm: [FAKE * (16 * c + 1 + x) for c in range(n)] for x, nm in enumerate(names)}
    if swap:
        ptrs[swap[0]][swap[1]] = swap[2]
    arr = lambda xs: (ctypes.c_void_p * n)(*xs)
    return abi.load_library().txl_rel_attn_fwd_mem_cells(
        n if cells is None else cells, *(arr(ptrs[nm]) for nm in names[:6]), B, M, L, H, D, dt,
        arr(ptrs["out"]), arr(ptrs["mem_next"]), arr(ptrs["ext"]), dm, None)


def test_attn_mem_cells_rejects_bad_arguments(lib):
    assert _attn_mem_cells(dt=7) == UNSUPPORTED
    assert _attn_mem_cells(cells=-1) == INVALID
    assert _attn_mem_cells(cells=0) == OK                          # no calls: nothing looked at
    assert _attn_mem_cells(dm=-1) == INVALID
    assert _attn_mem_cells(D=65) == UNSUPPORTED                    # every call's own checks
    assert _attn_mem_cells(swap=("q", 1, FAKE * 17 + 2)) == INVALID            # call 1 misaligned
    assert _attn_mem_cells(swap=("mem_next", 1, FAKE * 8)) == INVALID          # call 1's mem_next is call 0's
    assert _attn_mem_cells(swap=("out", 1, FAKE * 2 + 64)) == INVALID          # call 1 writes call 0's k
    assert _attn_mem_cells(swap=("mem_next", 1, FAKE * 9 + 32)) == INVALID     # ... call 0's ext_ctx
    # reads may be shared: both calls on one table and one q
    assert _attn_mem_cells(swap=("r", 1, FAKE * 4)) == CUDA
    assert _attn_mem_cells(swap=("q", 1, FAKE * 1)) == CUDA
    # valid arguments reach the device (none here)
    assert _attn_mem_cells(n=3) == CUDA
