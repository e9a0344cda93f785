"""The CPU oracle on shapes drawn by hypothesis.

* prefill against brute force (the dense masked softmax of tests/pins.py:
  library softmax and logsumexp over the full score matrix), over batch,
  length, group size, head size, window (from 1 to beyond T), output-row sets
  (empty or any positions) and the optional raw queries of the output stream;
* a prefill followed by decoding steps against one longer prefill, over page
  sizes and windows.
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
