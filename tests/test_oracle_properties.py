"""The CPU oracle against brute force on shapes drawn by hypothesis: batch,
length, group size, head size, window (from 1 to beyond T), output-row sets
(empty, repeated-free, any positions) and the optional raw queries of the
output stream. The brute force is the dense masked softmax of tests/pins.py
(library softmax and logsumexp over the full score matrix)."""
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
