"""The CPU oracle on shapes drawn by hypothesis.

* prefill against brute force (the dense masked softmax of tests/pins.py:
  library softmax and logsumexp over the full score matrix), over batch,
  length, group size, head size, window (from 1 to beyond T), output-row sets
  (empty or any positions) and the optional raw queries of the output stream;
* a prefill followed by decoding steps against one longer prefill, over page
  sizes and windows;
* continuous-batching steps (every sequence appends its own chunk) against a
  prefill of each sequence over all its tokens;
* every gradient of the backward against torch.autograd through the dense
  masked forward, output rows at repeated positions included;
* the projection against a dense float64 product with the stream affines.
"""
import math

import numpy as np
import pytest
import torch

from tests import pins

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@pytest.fixture(scope="module")
def orc(oracle_mod):
    return oracle_mod.Oracle()


@st.composite
def prefill_case(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 24))
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 3))
    d = draw(st.sampled_from([4, 8]))
    window = draw(st.integers(1, T + 3))
    lists = [sorted(draw(st.sets(st.integers(0, T - 1), max_size=T))) for _ in range(B)]
    with_q_out = draw(st.booleans())
    seed = draw(st.integers(0, 2**16))
    return B, T, Hkv * g, Hkv, d, window, lists, with_q_out, seed


@hypothesis.settings(max_examples=60, deadline=None)
@hypothesis.given(prefill_case())
def test_prefill_matches_brute_force(orc, case):
    B, T, Hq, Hkv, d, window, lists, with_q_out, seed = case
    q, k, v, ab, bb, ao, bo = pins.rng_inputs(seed, B, T, Hq, Hkv, d)
    indptr, pos = pins.csr(lists)
    n_out = int(indptr[-1])
    q_out = torch.randn((n_out, Hq, d), generator=torch.Generator().manual_seed(seed)).numpy() if with_q_out else None
    scale = 1.0 / math.sqrt(d)
    got = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, window, scale, q_out=q_out)
    ref = pins.brute_prefill(q, k, v, ab, bb, ao, bo, indptr, pos, window, scale, q_out=q_out)
    for name, a, b in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref):
        a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
        assert a.shape == b.shape, name
        if a.size:
            assert float(np.max(np.abs(a - b))) <= 1e-9, name


@st.composite
def consistency_case(draw):
    B = draw(st.integers(1, 2))
    T0 = draw(st.integers(1, 12))
    N = draw(st.integers(1, 5))
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 3))
    window = draw(st.integers(1, T0 + N + 2))
    page = draw(st.sampled_from([1, 2, 4, 8]))
    seed = draw(st.integers(0, 2**16))
    return B, T0, N, Hkv * g, Hkv, 8, window, page, seed


@hypothesis.settings(max_examples=40, deadline=None)
@hypothesis.given(consistency_case())
def test_prefill_then_decode_equals_longer_prefill(orc, case):
    """Orthros paper, Sec. 3.2: a prefill of T0 tokens followed by N decoding
    steps gives, at every appended position, the base row and the output row
    of one prefill over T0 + N tokens (pages of any size, any window)."""
    B, T0, N, Hq, Hkv, d, window, page, seed = case
    T = T0 + N
    q, k, v, ab, bb, ao, bo = pins.rng_inputs(seed, B, T, Hq, Hkv, d)
    indptr, pos = pins.csr([list(range(T0, T))] * B)
    full = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, window, 0.3)
    rng = np.random.default_rng(seed)
    lens = np.full(B, T0, np.int32)
    kc, vc, bt = pins._paged_from_seq([k[b, :T0] for b in range(B)], [v[b, :T0] for b in range(B)], lens, page, N, rng)
    for s in range(N):
        t = T0 + s
        ob, lb, oo, lo = orc.decode(q[:, t], k[:, t], v[:, t], kc, vc, bt, lens, ab, bb, ao, bo, window, 0.3)
        rows = indptr[:-1] + s
        for a, b_ in ((ob, full[0][:, t]), (lb, full[1][:, :, t]), (oo, full[2][rows]), (lo, full[3][rows])):
            assert float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b_, np.float64)))) <= 1e-12
        lens = lens + 1


@st.composite
def batching_case(draw):
    B = draw(st.integers(1, 3))
    t0 = [draw(st.integers(1, 8)) for _ in range(B)]
    steps = draw(st.integers(1, 4))
    chunks = [[draw(st.integers(0, 4)) for _ in range(B)] for _ in range(steps)]
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 2))
    window = draw(st.integers(1, 12))
    page = draw(st.sampled_from([1, 2, 4]))
    seed = draw(st.integers(0, 2**16))
    return t0, chunks, Hkv * g, Hkv, 8, window, page, seed


@hypothesis.settings(max_examples=40, deadline=None)
@hypothesis.given(batching_case())
def test_continuous_batching_equals_per_sequence_prefill(orc, case):
    """Continuous batching: steps in which every sequence appends its own chunk
    (0 to 4 tokens) give each new token the base row, and each chunk's last
    token the output row, of one prefill of that sequence over all its tokens."""
    t0, chunks, Hq, Hkv, d, window, page, seed = case
    B = len(t0)
    total = [t0[b] + sum(c[b] for c in chunks) for b in range(B)]
    seqs = [pins.rng_inputs(seed + b, 1, total[b], Hq, Hkv, d) for b in range(B)]
    ab, bb, ao, bo = seqs[0][3:]
    ends = []
    for b in range(B):
        at, e = t0[b], []
        for c in chunks:
            at += c[b]
            if c[b]:
                e.append(at - 1)
        ends.append(e)
    full = []
    for b in range(B):
        q, k, v = seqs[b][:3]
        ip, ps = pins.csr([ends[b]])
        full.append(orc.prefill(q, k, v, ab, bb, ao, bo, ip, ps, window, 0.3))
    rng = np.random.default_rng(seed)
    lens = np.array(t0, np.int32)
    kc, vc, bt = pins._paged_from_seq([seqs[b][1][0, :t0[b]] for b in range(B)],
                                      [seqs[b][2][0, :t0[b]] for b in range(B)], lens, page,
                                      max(total[b] - t0[b] for b in range(B)), rng)
    for c in chunks:
        new_indptr = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
        pick = lambda x, b: x[0, lens[b]:lens[b] + c[b]]  # noqa: E731
        qn = np.concatenate([pick(seqs[b][0], b) for b in range(B)], 0).reshape(-1, Hq, d)
        kn = np.concatenate([pick(seqs[b][1], b) for b in range(B)], 0).reshape(-1, Hkv, d)
        vn = np.concatenate([pick(seqs[b][2], b) for b in range(B)], 0).reshape(-1, Hkv, d)
        oi, op = pins.csr([[int(lens[b]) + c[b] - 1] if c[b] else [] for b in range(B)])
        ob, lb, oo, lo = orc.extend(qn, kn, vn, kc, vc, bt, lens, new_indptr, oi, op, ab, bb, ao, bo, window, 0.3)
        for b in range(B):
            r0, r1 = int(new_indptr[b]), int(new_indptr[b + 1])
            L = int(lens[b])
            assert np.max(np.abs(ob[r0:r1] - full[b][0][0, L:L + c[b]]), initial=0.0) <= 1e-12
            assert np.max(np.abs(lb[r0:r1].T - full[b][1][0, :, L:L + c[b]]), initial=0.0) <= 1e-12
            if c[b]:
                r = ends[b].index(L + c[b] - 1)
                o_row = int(oi[b])
                assert np.max(np.abs(oo[o_row] - full[b][2][r])) <= 1e-12
                assert np.max(np.abs(lo[o_row] - full[b][3][r])) <= 1e-12
        lens = lens + np.asarray(c, np.int32)


@st.composite
def backward_case(draw):
    B = draw(st.integers(1, 2))
    T = draw(st.integers(1, 14))
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 3))
    d = draw(st.sampled_from([4, 8]))
    window = draw(st.integers(1, T + 2))
    # output rows may repeat a position (their query and gradient add up)
    lists = [sorted(draw(st.lists(st.integers(0, T - 1), max_size=T + 2))) for _ in range(B)]
    with_q_out = draw(st.booleans())
    seed = draw(st.integers(0, 2**16))
    return B, T, Hkv * g, Hkv, d, window, lists, with_q_out, seed


@hypothesis.settings(max_examples=30, deadline=None)
@hypothesis.given(backward_case())
def test_backward_matches_autograd(orc, case):
    """Every gradient of the oracle's backward equals torch.autograd (float64)
    through the dense masked forward of tests/pins.py."""
    B, T, Hq, Hkv, d, window, lists, with_q_out, seed = case
    q, k, v, ab, bb, ao, bo = pins.rng_inputs(seed, B, T, Hq, Hkv, d)
    indptr, pos = pins.csr(lists)
    n_out = int(indptr[-1])
    r = np.random.default_rng(seed)
    q_out = r.standard_normal((n_out, Hq, d)).astype(np.float32) if with_q_out else None
    do_b = r.standard_normal((B, T, Hq, d)).astype(np.float32)
    do_o = r.standard_normal((n_out, Hq, d)).astype(np.float32)
    scale = 0.9 / math.sqrt(d)
    got = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, window, scale, do_b, do_o, q_out=q_out)
    leaves = {n: torch.tensor(x, dtype=torch.float64, requires_grad=True)
              for n, x in (("q", q), ("k", k), ("v", v), ("ab", ab), ("bb", bb), ("ao", ao), ("bo", bo))}
    qo_t = torch.tensor(q_out, dtype=torch.float64, requires_grad=True) if q_out is not None else None
    ob, oo = pins.torch_forward(leaves["q"], leaves["k"], leaves["v"], leaves["ab"], leaves["bb"], leaves["ao"],
                                leaves["bo"], indptr, pos, window, scale, qo_t)
    loss = (ob * torch.from_numpy(do_b).double()).sum() + (oo * torch.from_numpy(do_o).double()).sum()
    loss.backward()
    for name, leaf in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("d_alpha_base", "ab"), ("d_beta_base", "bb"),
                       ("d_alpha_out", "ao"), ("d_beta_out", "bo")):
        grad = leaves[leaf].grad
        ref = grad.numpy() if grad is not None else np.zeros_like(np.asarray(got[name]))
        assert float(np.max(np.abs(np.asarray(got[name], np.float64) - ref), initial=0.0)) <= 1e-9, name
    if q_out is not None:
        ref = qo_t.grad.numpy() if qo_t.grad is not None else np.zeros((0, Hq, d))
        assert float(np.max(np.abs(np.asarray(got["dq_out"], np.float64) - ref), initial=0.0)) <= 1e-9


@st.composite
def projection_case(draw):
    n_base = draw(st.integers(0, 6))
    n_out = draw(st.integers(0, 6))
    d_model = draw(st.integers(1, 24))
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 3))
    d = draw(st.sampled_from([2, 4, 8]))
    seed = draw(st.integers(0, 2**16))
    return n_base, n_out, d_model, Hkv * g, Hkv, d, seed


@hypothesis.settings(max_examples=40, deadline=None)
@hypothesis.given(projection_case())
def test_projection_matches_a_dense_product(orc, case):
    """The projection (Orthros paper, Alg. 1 lines 4-5) equals x W^T in float64
    with each stream's affine on the query columns and K/V from base rows only."""
    n_base, n_out, d_model, Hq, Hkv, d, seed = case
    r = np.random.default_rng(seed)
    N = (Hq + 2 * Hkv) * d
    x = r.standard_normal((n_base + n_out, d_model)).astype(np.float32)
    w_t = r.standard_normal((N, d_model)).astype(np.float32)
    ab, bb, ao, bo = (r.standard_normal((Hq, d)).astype(np.float32) for _ in range(4))
    qb, qo, k, v = orc.qkv_project(x, n_base, w_t, Hq, Hkv, d, ab, bb, ao, bo)
    y = x.astype(np.float64) @ w_t.astype(np.float64).T
    Nq, Nkv = Hq * d, Hkv * d
    want_qb = y[:n_base, :Nq].reshape(n_base, Hq, d) * ab + bb
    want_qo = y[n_base:, :Nq].reshape(n_out, Hq, d) * ao + bo
    for got, want in ((qb, want_qb), (qo, want_qo), (k, y[:n_base, Nq:Nq + Nkv].reshape(n_base, Hkv, d)),
                      (v, y[:n_base, Nq + Nkv:].reshape(n_base, Hkv, d))):
        assert np.asarray(got).shape == want.shape
        assert float(np.max(np.abs(np.asarray(got, np.float64) - want), initial=0.0)) <= 1e-9
