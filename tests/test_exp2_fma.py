"""The prefill softmax's exponential on the FMA pipe (`exp2_fma_x2` in
csrc/ptx.cuh), checked on the CPU against 2^x itself.

The helper's constants and steps are read from the header and replayed in
float32 with numpy, one PTX instruction at a time (fused multiply-adds done
in float64 and rounded once, which is exact for float32 operands; NaN results
made canonical as the GPU makes them). The pins: the cubic's relative error on
[-1/2, 1/2] stays below 7.5e-5 (far below the 2^-9 rounding that P takes to
bf16), the assembled 2^x keeps that error for every x from -125.5 up (results
in the normal range), and the special inputs behave as a softmax needs: -inf
and anything at or below -127 give exactly +0, inputs between -127 and -126
give a subnormal below 2^-126, 0 gives the cubic's value at 0, NaN stays NaN.
"""
import os
import re

import numpy as np
import pytest

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "efficient_long_context_gb300",
                   "csrc", "ptx.cuh")


def _helper_source():
    src = open(HDR).read()
    i = src.index("void exp2_fma_x2(")
    return src[i:src.index("\n}\n", i)]


def _f32(hexword):
    return np.array([int(hexword, 16)], dtype=np.uint32).view(np.float32)[0]


def _constants():
    body = _helper_source()
    lo = [_f32(h) for h in re.findall(r"max\.NaN\.f32 x\d, %\d, 0f([0-9A-F]{8})", body)]
    movs = [_f32(h) for h in re.findall(r"mov\.b32 k, 0f([0-9A-F]{8})", body)]
    assert len(lo) == 2 and lo[0] == lo[1], lo
    assert len(movs) == 5, movs  # 1.5 * 2^23, then c3, c2, c1, c0 in Horner order
    scale = re.findall(r"mad\.lo\.u32 x\d, t\d, (\d+), q\d", body)
    assert scale == ["8388608", "8388608"], scale  # bits << 23
    return lo[0], movs[0], movs[1:]


def _canon(x):
    b = x.view(np.uint32).copy()
    b[np.isnan(x)] = 0x7FFFFFFF
    return b.view(np.float32)


def _fma(a, b, c):
    return _canon((a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32))


def exp2_fma(a):
    """The helper's instruction sequence replayed in float32."""
    floor_, magic, (c3, c2, c1, c0) = _constants()
    a = np.asarray(a, dtype=np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        x = np.where(np.isnan(a), a, np.maximum(a, floor_)).astype(np.float32)
        t = _canon((x + magic).astype(np.float32))
        r = _canon((t - magic).astype(np.float32))
        f = _canon((x - r).astype(np.float32))
        p = np.full_like(f, c3)
        for c in (c2, c1, c0):
            p = _fma(p, f, np.full_like(f, c))
    bits = (t.view(np.uint32).astype(np.uint64) * 8388608 + p.view(np.uint32).astype(np.uint64)) & 0xFFFFFFFF
    bits = bits.astype(np.uint32).view(np.int32)
    bits = np.maximum(bits, 0).view(np.uint32)
    bits = np.where(np.isnan(a), np.uint32(0x7FFFFFFF), bits)
    return bits.view(np.float32)


def test_cubic_relative_error_on_the_reduced_interval():
    _, _, (c3, c2, c1, c0) = _constants()
    f = np.linspace(-0.5, 0.5, 200001)
    p = ((c3 * f + c2) * f + c1) * f + c0
    rel = np.abs(p / np.exp2(f) - 1)
    assert rel.max() < 7.5e-5, rel.max()
    assert rel.max() < 2.0 ** -9 / 25  # well inside the bf16 rounding of P


def test_assembled_exp2_over_the_softmax_range():
    a = np.concatenate([np.linspace(-125.5, 0, 1000001), np.linspace(0, 8, 10001)]).astype(np.float32)
    got = exp2_fma(a).astype(np.float64)
    ref = np.exp2(a.astype(np.float64))
    rel = np.abs(got / ref - 1)
    assert rel.max() < 7.6e-5, (rel.max(), a[np.argmax(rel)])
    # monotone apart from the cubic's ripple: never off by a binade at an integer boundary
    ints = np.arange(-120, 8, dtype=np.float32)
    assert np.all(np.abs(exp2_fma(ints).astype(np.float64) / np.exp2(ints.astype(np.float64)) - 1) < 7.6e-5)


def test_special_inputs():
    a = np.array([-np.inf, -1e30, -200.0, -127.0, -126.6, 0.0, np.nan], dtype=np.float32)
    got = exp2_fma(a)
    assert np.all(got[:4] == 0.0) and not np.signbit(got[:5]).any()  # exactly +0: masked keys add nothing
    assert 0.0 < got[4] < 2.0 ** -126  # a subnormal (the hardware exponential flushes these to zero)
    assert got[5] == pytest.approx(1.0, rel=7.5e-5)
    assert np.isnan(got[6])


def test_an_erroneous_constant_is_caught(monkeypatch):
    """A transposed pair of coefficients must fail the error bound."""
    floor_, magic, (c3, c2, c1, c0) = _constants()
    import tests.test_exp2_fma as me
    monkeypatch.setattr(me, "_constants", lambda: (floor_, magic, (c2, c3, c1, c0)))
    a = np.linspace(-10, 0, 10001).astype(np.float32)
    rel = np.abs(me.exp2_fma(a).astype(np.float64) / np.exp2(a.astype(np.float64)) - 1)
    assert rel.max() > 1e-3
