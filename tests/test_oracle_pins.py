"""Pins for the oracle: checks against what the method and the mathematics fix.

Nothing here re-types the oracle's loop.  Each pin reaches the same numbers by
another route the pages give, or by a special case that reduces to a library
routine or to a closed form:

* the four-term expansion of Transformer-XL Section 3.3 from hidden states and
  weights, with the naive per-pair projection W_kR R_{i-j};
* the Appendix B route: B~ = q Q^T followed by a per-row left shift, and the
  same shift read as a flat array with row pitch T-1;
* an absolute-position route (sinusoids at absolute positions combined by the
  angle-difference identities), which pins the sign of i-j and the table order;
* the segment-recurrence identity (Section 3.2): the memory path equals the
  last L rows of the same attention over the whole concatenated context;
* reductions to torch's scaled-dot-product attention and to a plain softmax;
* for the row log-sum-exp: a closed form (all scores zero: log of the count of
  visible keys), torch's logsumexp on textbook attention, and exp(s - lse)
  against the row's weights.

A final test plants mistakes in copies of the oracle's C source and checks that
these pins catch every one of them.
"""
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
from transformer_xl_relative_rel_gb300 import inputs

TOL = 1e-12


def _rand(shape, g):
    return g.standard_normal(shape)


def _problem(B, H, D, L, M, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    T = M + L
    return dict(q=_rand((L, B, H, D), g), k=_rand((T, B, H, D), g), v=_rand((T, B, H, D), g),
                r=_rand((T, H, D), g), u=_rand((H, D), g), w=_rand((H, D), g)), g


def _softmax_rows(s):
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def _attend(scores, mask, v):
    """scores, mask: [L, T]; v: [T, D] -> [L, D] (masked entries excluded)."""
    s = np.where(mask, scores, -np.inf)
    return _softmax_rows(s) @ v


def _visible(L, M):
    i = np.arange(L)[:, None]
    j = np.arange(M + L)[None, :]
    return j <= M + i


# ---------------------------------------------------------------------------
# 1. Four-term expansion from hidden states (Section 3.3), naive per-pair route
# ---------------------------------------------------------------------------
def _four_term_bruteforce(h_ext, Wq, Wk, Wv, Wr, R, u, w, B, H, D, L, M):
    """Scores from the four named terms with W_kR R_{i-j} projected per pair.

    h_ext: [T, B, d_model] extended context [memory; segment]; R: [T, d_model]
    relative encodings indexed by the distance i-j (row p = distance p).
    """
    T = M + L
    out = np.zeros((L, B, H, D))
    for b in range(B):
        for hd in range(H):
            sl = slice(hd * D, (hd + 1) * D)
            for i in range(L):
                xi = h_ext[M + i, b]                    # the query token's state
                qi = xi @ Wq[:, sl]
                scores = np.full(T, -np.inf)
                for j in range(T):
                    if j > M + i:
                        continue                        # future position
                    kj = h_ext[j, b] @ Wk[:, sl]        # W_kE E_xj
                    rij = R[M + i - j] @ Wr[:, sl]      # W_kR R_{i-j}, per pair
                    a = qi @ kj                         # (a) content addressing
                    bb = qi @ rij                       # (b) content-dependent position bias
                    c = u[hd] @ kj                      # (c) global content bias
                    d = w[hd] @ rij                     # (d) global position bias
                    scores[j] = (a + bb + c + d) / np.sqrt(D)
                p = _softmax_rows(scores[None, :])[0]
                vals = h_ext[:, b] @ Wv[:, sl]
                out[i, b, hd] = p @ vals
    return out


@pytest.mark.parametrize("B,H,D,L,M", [(2, 2, 4, 5, 3), (1, 3, 2, 4, 0), (1, 1, 3, 1, 6),
                                       (2, 1, 5, 6, 6)])
def test_four_term_bruteforce(oracle_lib, B, H, D, L, M):
    g = np.random.Generator(np.random.PCG64(100 + L + M))
    T, dm = M + L, H * D
    h_ext = _rand((T, B, dm), g)
    Wq, Wk, Wv, Wr = (_rand((dm, dm), g) * 0.5 for _ in range(4))
    R = _rand((T, dm), g)            # any table works; rows indexed by distance
    u, w = _rand((H, D), g), _rand((H, D), g)
    ref = _four_term_bruteforce(h_ext, Wq, Wk, Wv, Wr, R, u, w, B, H, D, L, M)

    # the library's inputs: projected q, k, v and the reversed table of Appendix B
    q = (h_ext[M:] @ Wq).reshape(L, B, H, D)
    k = (h_ext @ Wk).reshape(T, B, H, D)
    v = (h_ext @ Wv).reshape(T, B, H, D)
    Q = np.stack([R[T - 1 - t] @ Wr for t in range(T)]).reshape(T, H, D)   # Q_t = W_kR R_{T-1-t}
    got = oracle.rel_attn(q, k, v, Q, u, w, mem_len=M)
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL * max(1.0, np.abs(ref).max()))


def _shaw_bruteforce(h_ext, Wq, Wk, Wv, Rhat, B, H, D, L, M):
    """Shaw et al.'s form as Section 3.3 describes it: terms (a) and (b) only,
    with one free relative-position table Rhat [distance][H*D] in place of
    W_kR R (no global biases)."""
    T = M + L
    out = np.zeros((L, B, H, D))
    for b in range(B):
        for hd in range(H):
            sl = slice(hd * D, (hd + 1) * D)
            for i in range(L):
                qi = h_ext[M + i, b] @ Wq[:, sl]
                scores = np.full(T, -np.inf)
                for j in range(M + i + 1):
                    kj = h_ext[j, b] @ Wk[:, sl]
                    scores[j] = (qi @ kj + qi @ Rhat[M + i - j, sl]) / np.sqrt(D)
                p = _softmax_rows(scores[None, :])[0]
                out[i, b, hd] = p @ (h_ext[:, b] @ Wv[:, sl])
    return out


@pytest.mark.parametrize("B,H,D,L,M", [(2, 2, 4, 5, 3), (1, 2, 3, 6, 0)])
def test_shaw_form_is_zero_bias_case(oracle_lib, B, H, D, L, M):
    """Terms (a) + (b) with a free table == the oracle with u = v = 0 and the
    table reversed as in Appendix B."""
    g = np.random.Generator(np.random.PCG64(300 + L + M))
    T, dm = M + L, H * D
    h_ext = _rand((T, B, dm), g)
    Wq, Wk, Wv = (_rand((dm, dm), g) * 0.5 for _ in range(3))
    Rhat = _rand((T, dm), g)
    ref = _shaw_bruteforce(h_ext, Wq, Wk, Wv, Rhat, B, H, D, L, M)
    q = (h_ext[M:] @ Wq).reshape(L, B, H, D)
    k = (h_ext @ Wk).reshape(T, B, H, D)
    v = (h_ext @ Wv).reshape(T, B, H, D)
    r = np.stack([Rhat[T - 1 - t] for t in range(T)]).reshape(T, H, D)
    zero = np.zeros((H, D))
    got = oracle.rel_attn(q, k, v, r, zero, zero, mem_len=M)
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL * max(1.0, np.abs(ref).max()))


# ---------------------------------------------------------------------------
# 2. Appendix B: B~ = (q+v) Q^T, then row i left-shifted by L-1-i
# ---------------------------------------------------------------------------
def _appendix_b(q, k, v, r, u, w, M, strided):
    L, B, H, D = q.shape
    T = M + L
    out = np.zeros_like(q)
    vis = _visible(L, M)
    for b in range(B):
        for hd in range(H):
            qu = q[:, b, hd] + u[hd]
            qv = q[:, b, hd] + w[hd]
            ac = qu @ k[:, b, hd].T                      # terms (a)+(c), [L, T]
            bt = qv @ r[:, hd].T                         # B~ = qv Q^T, [L, T]
            if strided:
                # the left shift as a read of the flat B~ with row pitch T-1
                flat = bt.reshape(-1)
                bd = np.zeros((L, T))
                for i in range(L):
                    for j in range(M + i + 1):
                        bd[i, j] = flat[(L - 1) + i * (T - 1) + j]
            else:
                bd = np.zeros((L, T))
                for i in range(L):
                    s = L - 1 - i                        # row i shifts left by L-1-i
                    bd[i, : T - s] = bt[i, s:]
            out[:, b, hd] = _attend((ac + bd) / np.sqrt(D), vis, v[:, b, hd])
    return out


@pytest.mark.parametrize("strided", [False, True])
@pytest.mark.parametrize("B,H,D,L,M", [(2, 2, 8, 7, 5), (1, 2, 3, 9, 0), (1, 1, 4, 3, 11)])
def test_appendix_b_left_shift(oracle_lib, strided, B, H, D, L, M):
    p, _ = _problem(B, H, D, L, M, seed=7 + L)
    ref = _appendix_b(**p, M=M, strided=strided)
    got = oracle.rel_attn(**p, mem_len=M)
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL * 10)


def test_left_shift_equals_strided_read():
    """The two readings of the shift agree entry by entry on the visible part."""
    g = np.random.Generator(np.random.PCG64(3))
    L, M = 6, 4
    T = L + M
    bt = g.standard_normal((L, T))
    flat = bt.reshape(-1)
    for i in range(L):
        for j in range(M + i + 1):
            assert bt[i, j + L - 1 - i] == flat[(L - 1) + i * (T - 1) + j]


# ---------------------------------------------------------------------------
# 3. Masked softmax: rows sum to one, future keys get exactly zero weight
# ---------------------------------------------------------------------------
def test_softmax_rows_and_mask(oracle_lib):
    p, _ = _problem(2, 3, 8, 10, 6, seed=11)
    out, prob = oracle.rel_attn(**p, mem_len=6, return_prob=True)
    L, T = 10, 16
    vis = _visible(L, 6)
    np.testing.assert_allclose(prob.sum(-1), 1.0, rtol=0, atol=TOL)
    assert (prob[..., ~vis] == 0.0).all()                    # exact zeros when masked
    assert (prob[:, :, vis] > 0).all()
    # out is the probability-weighted sum of the values
    v = p["v"]
    recon = np.einsum("bhlt,tbhd->lbhd", prob, v)
    np.testing.assert_allclose(out, recon, rtol=0, atol=TOL)


# ---------------------------------------------------------------------------
# 4. Only the distance matters: an absolute-position route
# ---------------------------------------------------------------------------
def _abs_route(q, k, v, u, w, Wr, M, c, dm):
    """BD from sinusoids at absolute positions pos_q = c+M+i, pos_k = c+j,
    combined with sin(a-b) = sin a cos b - cos a sin b and
    cos(a-b) = cos a cos b + sin a sin b."""
    L, B, H, D = q.shape
    T = M + L
    freq = np.power(10000.0, -np.arange(0, dm, 2) / dm)
    out = np.zeros_like(q)
    vis = _visible(L, M)
    for b in range(B):
        for hd in range(H):
            sl = slice(hd * D, (hd + 1) * D)
            sc = np.zeros((L, T))
            for i in range(L):
                a = (c + M + i) * freq
                for j in range(T):
                    bb = (c + j) * freq
                    enc = np.zeros(dm)
                    enc[0::2] = np.sin(a) * np.cos(bb) - np.cos(a) * np.sin(bb)
                    enc[1::2] = np.cos(a) * np.cos(bb) + np.sin(a) * np.sin(bb)
                    rr = enc @ Wr[:, sl]
                    sc[i, j] = ((q[i, b, hd] + u[hd]) @ k[j, b, hd]
                                + (q[i, b, hd] + w[hd]) @ rr)
            out[:, b, hd] = _attend(sc / np.sqrt(D), vis, v[:, b, hd])
    return out


@pytest.mark.parametrize("c", [0, 7, 1000])
def test_shift_invariance_absolute_positions(oracle_lib, c):
    B, H, D, L, M = 1, 2, 4, 5, 4
    T, dm = M + L, H * D
    p, g = _problem(B, H, D, L, M, seed=21)
    Wr = g.standard_normal((dm, dm)) * 0.5
    # the relative table in float64: row t holds W_kR R_{T-1-t}
    r = (inputs.sinusoid(T, dm) @ Wr)[::-1].reshape(T, H, D)
    got = oracle.rel_attn(p["q"], p["k"], p["v"], r, p["u"], p["w"], mem_len=M)
    ref = _abs_route(p["q"], p["k"], p["v"], p["u"], p["w"], Wr, M, c, dm)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-9)


# ---------------------------------------------------------------------------
# 5. Segment recurrence: memory path == last L rows over the whole context
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,M", [(4, 6), (8, 8), (5, 1)])
def test_recurrence_equivalence(oracle_lib, L, M):
    B, H, D = 2, 2, 6
    p, g = _problem(B, H, D, L, M, seed=31 + M)
    T = M + L
    q_mem = g.standard_normal((M, B, H, D))
    q_full = np.concatenate([q_mem, p["q"]], 0)       # queries for all T positions
    full = oracle.rel_attn(q_full, p["k"], p["v"], p["r"], p["u"], p["w"], mem_len=0)
    mem_path = oracle.rel_attn(**p, mem_len=M)
    assert full.shape[0] == T
    np.testing.assert_allclose(mem_path, full[M:], rtol=0, atol=TOL)


# ---------------------------------------------------------------------------
# 6. Special cases: library softmax attention, constant position term, L = 1
# ---------------------------------------------------------------------------
def _sdpa(qq, k, v, L, M):
    """torch scaled-dot-product attention, float64, explicit boolean mask."""
    qt = torch.from_numpy(np.ascontiguousarray(qq.transpose(1, 2, 0, 3)))      # B,H,L,D
    kt = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 2, 0, 3)))       # B,H,T,D
    vt = torch.from_numpy(np.ascontiguousarray(v.transpose(1, 2, 0, 3)))
    mask = torch.from_numpy(_visible(L, M))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return o.numpy().transpose(2, 0, 1, 3)


def test_no_position_term_is_textbook_attention(oracle_lib):
    B, H, D, L, M = 2, 3, 8, 9, 7
    p, _ = _problem(B, H, D, L, M, seed=41)
    p["r"][:] = 0.0
    p["u"][:] = 0.0
    p["w"][:] = 0.0
    got = oracle.rel_attn(**p, mem_len=M)
    np.testing.assert_allclose(got, _sdpa(p["q"], p["k"], p["v"], L, M), rtol=0, atol=TOL)


def test_constant_position_term_cancels(oracle_lib):
    B, H, D, L, M = 1, 2, 8, 6, 5
    p, g = _problem(B, H, D, L, M, seed=43)
    p["r"][:] = g.standard_normal((1, H, D))        # every distance encodes the same
    got = oracle.rel_attn(**p, mem_len=M)
    ref = _sdpa(p["q"] + p["u"][None, None], p["k"], p["v"], L, M)
    np.testing.assert_allclose(got, ref, rtol=0, atol=TOL)


def test_single_query_sees_all_keys(oracle_lib):
    B, H, D, L, M = 2, 2, 5, 1, 9
    p, _ = _problem(B, H, D, L, M, seed=47)
    got = oracle.rel_attn(**p, mem_len=M)
    T = M + L
    for b in range(B):
        for hd in range(H):
            s = np.array([((p["q"][0, b, hd] + p["u"][hd]) @ p["k"][j, b, hd]
                           + (p["q"][0, b, hd] + p["w"][hd]) @ p["r"][T - 1 - (M - j), hd])
                          for j in range(T)]) / np.sqrt(D)
            ref = _softmax_rows(s[None])[0] @ p["v"][:, b, hd]
            np.testing.assert_allclose(got[0, b, hd], ref, rtol=0, atol=TOL)


def test_rows_variant_matches_full(oracle_lib):
    B, H, D, L, M = 3, 2, 6, 7, 5
    p, _ = _problem(B, H, D, L, M, seed=53)
    full = oracle.rel_attn(**p, mem_len=M)
    rows = np.array([[0, 0, 0], [2, 1, 6], [1, 0, 3], [2, 1, 0]])
    got = oracle.rel_attn_rows(**p, mem_len=M, rows=rows)
    for x, (b, h, i) in enumerate(rows):
        assert np.array_equal(got[x], full[i, b, h])


def _lse_textbook(q, k, L, M):
    """torch log-sum-exp of the masked scaled dot products, float64."""
    qt = torch.from_numpy(np.ascontiguousarray(q.transpose(1, 2, 0, 3)))
    kt = torch.from_numpy(np.ascontiguousarray(k.transpose(1, 2, 0, 3)))
    s = qt @ kt.transpose(-1, -2) / np.sqrt(q.shape[-1])
    s = s.masked_fill(~torch.from_numpy(_visible(L, M)), float("-inf"))
    return torch.logsumexp(s, dim=-1).numpy()


def _lse_pins_pass(mod):
    # no key and no table content: every visible score is 0, so row i's
    # denominator is its count of visible keys, M + i + 1
    B, H, D, L, M = 2, 2, 4, 5, 3
    p, _ = _problem(B, H, D, L, M, seed=61)
    p["k"][:] = 0.0
    p["r"][:] = 0.0
    _, lse = mod.rel_attn(**p, mem_len=M, return_lse=True)
    if not np.allclose(lse, np.log(M + 1 + np.arange(L))[None, None], rtol=0, atol=1e-12):
        return False
    # no position term and no biases: the log-sum-exp of textbook attention
    p, _ = _problem(B, H, D, L, M, seed=62)
    p["q"] *= 3.0                                        # rows with a clear maximum
    p["r"][:] = 0.0
    p["u"][:] = 0.0
    p["w"][:] = 0.0
    _, lse = mod.rel_attn(**p, mem_len=M, return_lse=True)
    return np.allclose(lse, _lse_textbook(p["q"], p["k"], L, M), rtol=0, atol=1e-12)


def test_lse_pins(oracle_lib):
    assert _lse_pins_pass(oracle)


def test_lse_matches_its_probabilities(oracle_lib):
    """P_ij = exp(s_ij - lse_i) on the full four-term score of a single query
    row written out by hand."""
    B, H, D, L, M = 2, 2, 5, 1, 9
    p, _ = _problem(B, H, D, L, M, seed=63)
    _, prob, lse = oracle.rel_attn(**p, mem_len=M, return_prob=True, return_lse=True)
    T = M + L
    for b in range(B):
        for hd in range(H):
            s = np.array([((p["q"][0, b, hd] + p["u"][hd]) @ p["k"][j, b, hd]
                           + (p["q"][0, b, hd] + p["w"][hd]) @ p["r"][T - 1 - (M - j), hd])
                          for j in range(T)]) / np.sqrt(D)
            np.testing.assert_allclose(np.exp(s - lse[b, hd, 0]), prob[b, hd, 0], rtol=0, atol=TOL)


LSE_MUTANTS = {
    "lse_without_max": ("*lse_out = mx + log(z);", "*lse_out = log(z);"),
    "lse_of_max_only": ("*lse_out = mx + log(z);", "*lse_out = mx;"),
}


@pytest.mark.parametrize("name", sorted(LSE_MUTANTS))
def test_lse_pins_catch_planted_mistake(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    mod = _build_mutant(tmp_path, name)
    assert not _lse_pins_pass(mod), f"planted mistake {name!r} went unnoticed"


# ---------------------------------------------------------------------------
# 7. Memory rollover (Section 3.2): newest M rows of [memory; segment]
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("L,M", [(4, 4), (6, 2), (2, 7), (5, 0)])
def test_mem_update_closed_forms(L, M):
    g = np.random.Generator(np.random.PCG64(61))
    mem = g.standard_normal((M, 3, 4)).astype(np.float32)
    h = g.standard_normal((L, 3, 4)).astype(np.float32)
    new = oracle.mem_update(np.concatenate([mem, h], 0), M)
    assert new.shape == (M, 3, 4)
    if M <= L:
        assert np.array_equal(new, h[L - M:])             # only current states survive
    else:
        assert np.array_equal(new[: M - L], mem[L:])      # the newest old memory first
        assert np.array_equal(new[M - L:], h)
    # two rollovers: memory spans the last two segments when M = 2L
    if M == 2 * L and M > 0:
        h2 = g.standard_normal((L, 3, 4)).astype(np.float32)
        new2 = oracle.mem_update(np.concatenate([new, h2], 0), M)
        assert np.array_equal(new2, np.concatenate([h, h2], 0))


# ---------------------------------------------------------------------------
# 8. The pins catch planted mistakes (mutants of the oracle's C source)
# ---------------------------------------------------------------------------
MUTANTS = {
    "table_not_reversed": ("(T - 1 - off) * H", "(off) * H"),
    # a reversed distance that still stays inside the table
    "distance_reversed": ("const long off = M + i - j;", "const long off = j - i + L - 1;"),
    "self_masked": ("const long last = M + i;", "const long last = M + i - 1;"),
    "dropped_u_term": ("(qi[d] + uh[d]) * kj[d]", "(qi[d]) * kj[d]"),
    "dropped_d_term": ("(qi[d] + wh[d]) * rr[d]", "(qi[d]) * rr[d]"),
    "no_scale": ("s[j] = a * scale;", "s[j] = a;"),
    "key_index_transposed": ("k + ((j * B + b) * H + h) * D", "k + ((b * B + j) * H + h) * D"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "txl_oracle.c")).read()
    old, new = {**MUTANTS, **LSE_MUTANTS}[name]
    assert old in src, f"mutation anchor for {name} no longer in the oracle source"
    mdir = tmp_path / name
    mdir.mkdir()
    shutil.copy(os.path.join(os.path.dirname(oracle.__file__), "__init__.py"), mdir / "__init__.py")
    (mdir / "txl_oracle.c").write_text(src.replace(old, new))
    import importlib.util
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}", mdir / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build(force=True)          # a mutant that does not compile is a test error
    return mod


def _pins_pass(mod):
    """Run a compact set of the pins above against an oracle module."""
    B, H, D, L, M = 1, 2, 4, 5, 3
    g = np.random.Generator(np.random.PCG64(5))
    T, dm = M + L, H * D
    h_ext = _rand((T, B, dm), g)
    Wq, Wk, Wv, Wr = (_rand((dm, dm), g) * 0.5 for _ in range(4))
    R = _rand((T, dm), g)
    u, w = _rand((H, D), g), _rand((H, D), g)
    ref = _four_term_bruteforce(h_ext, Wq, Wk, Wv, Wr, R, u, w, B, H, D, L, M)
    q = (h_ext[M:] @ Wq).reshape(L, B, H, D)
    k = (h_ext @ Wk).reshape(T, B, H, D)
    v = (h_ext @ Wv).reshape(T, B, H, D)
    Q = np.stack([R[T - 1 - t] @ Wr for t in range(T)]).reshape(T, H, D)
    if not np.allclose(mod.rel_attn(q, k, v, Q, u, w, mem_len=M), ref, rtol=0, atol=1e-10):
        return False
    p, _ = _problem(2, 2, 4, 5, 3, seed=9)
    if not np.allclose(mod.rel_attn(**p, mem_len=3),
                       _appendix_b(**p, M=3, strided=False), rtol=0, atol=1e-10):
        return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc missing")
    assert _pins_pass(oracle), "pins must pass on the real oracle"
    mod = _build_mutant(tmp_path, name)
    assert not _pins_pass(mod), f"planted mistake {name!r} went unnoticed"


# ---------------------------------------------------------------------------
# Projections and the relative table (Section 3.3 procedure, Appendix B)
# ---------------------------------------------------------------------------
def _pin_projections_end_to_end(project_heads, rel_table, sinusoid):
    """q, k, v from the oracle's projections of [memory; segment] states and
    Q from its table, through the oracle's attention, equal the four-term
    expansion with W_kR R_{i-j} projected per pair (R by distance)."""
    g = np.random.Generator(np.random.PCG64(77))
    B, H, D, L, M = 2, 2, 3, 5, 4
    T, dm = M + L, H * D
    h_ext = g.standard_normal((T, B, dm))
    Wq, Wk, Wv, Wr = (g.standard_normal((dm, dm)) * 0.5 for _ in range(4))
    u, w = g.standard_normal((H, D)), g.standard_normal((H, D))
    R = sinusoid(T, dm)
    ref = _four_term_bruteforce(h_ext, Wq, Wk, Wv, Wr, R, u, w, B, H, D, L, M)
    # the paper's projection matrices are [out, in]: q = h W_q^T
    q = project_heads(h_ext[M:], Wq.T, H, D)
    k = project_heads(h_ext, Wk.T, H, D)
    v = project_heads(h_ext, Wv.T, H, D)
    Q = rel_table(Wr.T, T, H, D)
    got = oracle.rel_attn(q, k, v, Q, u, w, mem_len=M)
    return np.abs(got - ref).max() <= TOL * max(1.0, np.abs(ref).max())


def _pin_sinusoid(sinusoid):
    """The sinusoid of Vaswani et al. by its stated properties, not its
    formula: distance 0 encodes as [0, 1, 0, 1, ...]; each column pair is a
    (sin, cos) of one angle; the angles per unit distance, read back with
    atan2, form a geometric progression from 1 down to 1/10000 over the
    pairs (wavelengths 2 pi .. 10000 * 2 pi); and the encoding of p + k is a
    fixed rotation (depending on k only) of the encoding of p."""
    dm, n = 16, 40
    R = sinusoid(n, dm)
    ok = R.shape == (n, dm)
    ok &= np.array_equal(R[0], np.tile([0.0, 1.0], dm // 2))
    ok &= np.abs(R[:, 0::2] ** 2 + R[:, 1::2] ** 2 - 1.0).max() < 1e-12
    omega = np.arctan2(R[1, 0::2], R[1, 1::2])
    ratio = 10000.0 ** (-2.0 / dm)
    ok &= abs(omega[0] - 1.0) < 1e-12
    ok &= np.abs(omega[1:] / omega[:-1] - ratio).max() < 1e-9
    for kk in (1, 3, 17):
        for c in range(dm // 2):
            s, co = np.sin(kk * omega[c]), np.cos(kk * omega[c])
            rot = np.array([[co, s], [-s, co]])          # [sin(a+b), cos(a+b)] from [sin a, cos a]
            pair = R[:n - kk, 2 * c:2 * c + 2]
            ok &= np.abs(pair @ rot.T - R[kk:, 2 * c:2 * c + 2]).max() < 1e-9
    return bool(ok)


def _pin_padding(project_heads, rel_table):
    """Zero columns past d_head; the first d_head columns are the unpadded result."""
    g = np.random.Generator(np.random.PCG64(5))
    x, w = g.standard_normal((3, 4, 10)), g.standard_normal((2 * 3, 10))
    a, b = project_heads(x, w, 2, 3), project_heads(x, w, 2, 3, 8)
    t, tp = rel_table(w, 6, 2, 3), rel_table(w, 6, 2, 3, 8)
    return (b.shape == (3, 4, 2, 8) and np.array_equal(b[..., 3:], np.zeros((3, 4, 2, 5)))
            and np.array_equal(b[..., :3], a) and np.array_equal(tp[..., :3], t)
            and not tp[..., 3:].any())


def test_projection_and_table_pins():
    assert _pin_projections_end_to_end(oracle.project_heads, oracle.rel_table, oracle.sinusoid)
    assert _pin_sinusoid(oracle.sinusoid)
    assert _pin_padding(oracle.project_heads, oracle.rel_table)


def _mutant_project_transposed_heads(x, w, heads, d_head, d_pad=None):
    # heads and head columns interleaved the wrong way round
    y = np.matmul(np.asarray(x, float), np.asarray(w, float).T)
    y = y.reshape(y.shape[:-1] + (d_head, heads)).swapaxes(-1, -2)
    return oracle.project_heads(x, w, heads, d_head, d_pad) * 0 + np.pad(
        y, [(0, 0)] * (y.ndim - 1) + [(0, (d_pad or d_head) - d_head)])


def _mutant_table_not_reversed(w_r, klen, heads, d_head, d_pad=None):
    return oracle.rel_table(w_r, klen, heads, d_head, d_pad)[::-1]


def _mutant_table_off_by_one(w_r, klen, heads, d_head, d_pad=None):
    R = oracle.sinusoid(klen + 1, np.asarray(w_r).shape[1])[1:]       # distances 1..klen
    return oracle.project_heads(R, w_r, heads, d_head, d_pad)[::-1]


def _mutant_sin_cos_swapped(n_pos, d_model):
    R = oracle.sinusoid(n_pos, d_model)
    out = R.copy()
    out[:, 0::2], out[:, 1::2] = R[:, 1::2], R[:, 0::2]
    return out


def _mutant_frequency_exponent(n_pos, d_model):
    out = np.zeros((n_pos, d_model))
    for c2 in range(0, d_model, 2):
        f = 10000.0 ** (-c2 / (2 * d_model))          # half the exponent
        out[:, c2] = np.sin(np.arange(n_pos) * f)
        out[:, c2 + 1] = np.cos(np.arange(n_pos) * f)
    return out


def _mutant_cos_frequency(n_pos, d_model):
    out = oracle.sinusoid(n_pos, d_model)
    for c2 in range(0, d_model, 2):                     # cos column uses the next pair's frequency
        f = 10000.0 ** (-min(c2 + 2, d_model - 2) / d_model)
        out[:, c2 + 1] = np.cos(np.arange(n_pos) * f)
    return out


def _mutant_padding_garbage(x, w, heads, d_head, d_pad=None):
    y = oracle.project_heads(x, w, heads, d_head, d_pad)
    if d_pad and d_pad > d_head:
        y[..., d_head:] = 1.0
    return y


@pytest.mark.parametrize("name", ["project_heads_transposed", "table_not_reversed", "table_off_by_one",
                                  "sin_cos_swapped", "frequency_exponent", "cos_frequency",
                                  "padding_garbage"])
def test_projection_pins_catch_planted_mistakes(name):
    ph, rt, sn = oracle.project_heads, oracle.rel_table, oracle.sinusoid
    if name == "project_heads_transposed":
        ph = _mutant_project_transposed_heads
    elif name == "table_not_reversed":
        rt = _mutant_table_not_reversed
    elif name == "table_off_by_one":
        rt = _mutant_table_off_by_one
    elif name == "sin_cos_swapped":
        sn = _mutant_sin_cos_swapped
    elif name == "frequency_exponent":
        sn = _mutant_frequency_exponent
    elif name == "cos_frequency":
        sn = _mutant_cos_frequency
    elif name == "padding_garbage":
        ph = _mutant_padding_garbage
    caught = (not _pin_projections_end_to_end(ph, rt, sn)) or (not _pin_sinusoid(sn)) or \
        (not _pin_padding(ph, rt))
    assert caught, f"planted mistake {name} passed every pin"
