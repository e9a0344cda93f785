"""The C-ABI library builds, loads and exports every symbol the header declares;
host-side argument checks return their error codes without touching a GPU."""
import ctypes
import os
import re

import pytest
import torch

import efficient_long_context_gb300 as ola
from efficient_long_context_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ola.load_library()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"ORTHROS_API\s+[\w\s\*]*?\b(orthros_\w+)\s*\(", src))
    return names


def test_header_declares_the_abi():
    names = declared_symbols()
    assert {"orthros_prefill", "orthros_decode", "orthros_check"} <= names
    assert names == set(ola._binding.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert ola.orthros_status_string(0) == "ok"
    assert "workspace" in ola.orthros_status_string(4)


def test_workspace_size_rejects_bad_shapes(lib):
    assert ola.orthros_prefill_workspace_size(1, 16, 4, 2, 128, 1, 8) > 0
    assert ola.orthros_prefill_workspace_size(1, 16, 3, 2, 128, 1, 8) == 0  # Hq % Hkv
    assert ola.orthros_prefill_workspace_size(1, 16, 4, 2, 96, 1, 8) == 0  # d
    assert ola.orthros_prefill_workspace_size(1, 16, 4, 2, 128, 1, 0) == 0  # window
    assert ola.orthros_decode_workspace_size(2, 4, 2, 64, 8, 64) > 0
    assert ola.orthros_decode_workspace_size(2, 4, 2, 64, 0, 64) == 0


def _call_prefill(lib, **over):
    args = dict(q=1 << 12, k=1 << 12, v=1 << 12, ab=1 << 12, bb=1 << 12, ao=1 << 12, bo=1 << 12,
                indptr=(ctypes.c_int32 * 2)(0, 1), pos=1 << 12, n_out=1, q_out=None,
                B=1, T=16, Hq=4, Hkv=2, d=128, window=8, scale=0.1, dtype=0,
                o_base=1 << 12, lse_base=1 << 12, o_out=1 << 12, lse_out=1 << 12,
                k_cache=None, v_cache=None, bt=None, max_pages=0, page_size=0, num_pages=0,
                ws=1 << 12, ws_bytes=1 << 30, stream=None)
    args.update(over)
    a = args
    return lib.orthros_prefill(a["q"], a["k"], a["v"], a["ab"], a["bb"], a["ao"], a["bo"],
                               a["indptr"], a["pos"], a["n_out"], a["q_out"], a["B"], a["T"], a["Hq"],
                               a["Hkv"], a["d"], a["window"], a["scale"], a["dtype"], a["o_base"],
                               a["lse_base"], a["o_out"], a["lse_out"], a["k_cache"], a["v_cache"],
                               a["bt"], a["max_pages"], a["page_size"], a["num_pages"], a["ws"],
                               a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Hq=3), 1),
    (dict(d=96), 2),
    (dict(window=0), 1),
    (dict(scale=float("inf")), 1),
    (dict(q=None), 1),
    (dict(q=(1 << 12) + 2), 1),  # misaligned
    (dict(indptr=(ctypes.c_int32 * 2)(0, 2)), 1),  # indptr[B] != n_out
    (dict(indptr=(ctypes.c_int32 * 2)(1, 1)), 1),  # indptr[0] != 0
    (dict(pos=None), 1),
    (dict(ws=None), 4),
    (dict(ws_bytes=8), 4),
    (dict(ws=(1 << 12) + 16), 1),  # workspace alignment
    (dict(k_cache=1 << 12), 1),  # partial cache arguments
    (dict(k_cache=1 << 12, v_cache=1 << 12, bt=1 << 12, max_pages=1, page_size=8, num_pages=4), 1),  # pages < T
    (dict(dtype=7), 1),
])
def test_prefill_host_checks(lib, over, code):
    assert _call_prefill(lib, **over) == code
    assert ola.orthros_last_error() != ""


def _call_shard(lib, **over):
    args = dict(q=1 << 12, k=1 << 12, v=1 << 12, ab=1 << 12, bb=1 << 12, ao=1 << 12, bo=1 << 12,
                indptr=(ctypes.c_int32 * 2)(0, 1), pos=1 << 12, n_rows=1, q_rows=1 << 12,
                B=1, Tq=16, Tkv=40, Hq=4, Hkv=2, d=128, window=8, scale=0.1, dtype=0,
                o_base=1 << 12, lse_base=1 << 12, o_part=1 << 12, lse_part=1 << 12,
                ws=1 << 12, ws_bytes=1 << 30, stream=None)
    args.update(over)
    a = args
    return lib.orthros_prefill_shard(a["q"], a["k"], a["v"], a["ab"], a["bb"], a["ao"], a["bo"], a["indptr"],
                                     a["pos"], a["n_rows"], a["q_rows"], a["B"], a["Tq"], a["Tkv"], a["Hq"],
                                     a["Hkv"], a["d"], a["window"], a["scale"], a["dtype"], a["o_base"],
                                     a["lse_base"], a["o_part"], a["lse_part"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Tq=0), 1),             # a shard holds at least one query row
    (dict(Tq=41), 1),            # more queries than keys
    (dict(dtype=1), 2),          # bf16 only
    (dict(q_rows=None), 1),      # output rows need their queries
    (dict(o_part=None), 1),
    (dict(o_part=(1 << 12) + 4), 1),  # misaligned
    (dict(indptr=(ctypes.c_int32 * 2)(0, 2)), 1),
    (dict(ws_bytes=8), 4),
    (dict(Hq=3), 1),
])
def test_shard_host_checks(lib, over, code):
    assert _call_shard(lib, **over) == code
    assert ola.orthros_last_error() != ""


def test_shard_workspace_size(lib):
    assert ola.orthros_prefill_shard_workspace_size(1, 16, 40, 4, 2, 128, 1, 8) > 0
    assert ola.orthros_prefill_shard_workspace_size(1, 41, 40, 4, 2, 128, 1, 8) == 0  # Tq > Tkv
    assert ola.orthros_prefill_shard_workspace_size(1, 16, 40, 4, 2, 128, 1, 8, torch.float32) == 0


@pytest.mark.parametrize("args,code", [
    ((0, 4, 8, 128, 0), 1),   # no partials
    ((2, -1, 8, 128, 0), 1),  # negative row count
    ((2, 4, 8, 96, 0), 2),    # head size
    ((2, 4, 8, 128, 5), 1),   # dtype
])
def test_merge_host_checks(lib, args, code):
    n_parts, n_rows, Hq, d, dtype = args
    rc = lib.orthros_merge_partials(1 << 12, 1 << 12, n_parts, n_rows, Hq, d, dtype, 1 << 12, 1 << 12, None)
    assert rc == code
    assert ola.orthros_last_error() != ""


def test_selftest_host_checks(lib):
    assert lib.orthros_selftest_wait_timeout(0, 1 << 12, 256, None) == 1  # limit must be >= 1
    assert lib.orthros_selftest_wait_timeout(1000, None, 256, None) == 4  # no workspace
    assert lib.orthros_selftest_wait_timeout(1000, (1 << 12) + 16, 256, None) == 1  # alignment


def test_decode_host_checks(lib):
    rc = lib.orthros_decode(1 << 12, None, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 0, 64, 4, 1 << 12,
                            1 << 12, 1 << 12, 1 << 12, 1 << 12, 2, 4, 2, 128, 16, 0.1, 0,
                            1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 20, None)
    assert rc == 1  # max_pages = 0
    rc = lib.orthros_decode(1 << 12, None, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 1 << 12, 4, 64, 4, 1 << 12,
                            1 << 12, 1 << 12, 1 << 12, 1 << 12, 2, 4, 2, 128, 16, 0.1, 0,
                            1 << 12, 1 << 12, 1 << 12, 1 << 12, None, 0, None)
    assert rc == 4  # no workspace


def _call_backward(lib, **over):
    P = 1 << 12
    a = dict(q=P, k=P, v=P, ab=P, bb=P, ao=P, bo=P, indptr=(ctypes.c_int32 * 2)(0, 1), pos=P, n_out=1,
             q_out=None, B=1, T=16, Hq=4, Hkv=2, d=128, window=8, scale=0.1, dtype=0,
             o_base=P, lse_base=P, o_out=P, lse_out=P, do_base=P, do_out=P,
             dq=P, dk=P, dv=P, dq_out=None, dab=P, dbb=P, dao=P, dbo=P, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(over)
    return lib.orthros_prefill_backward(
        a["q"], a["k"], a["v"], a["ab"], a["bb"], a["ao"], a["bo"], a["indptr"], a["pos"], a["n_out"], a["q_out"],
        a["B"], a["T"], a["Hq"], a["Hkv"], a["d"], a["window"], a["scale"], a["dtype"],
        a["o_base"], a["lse_base"], a["o_out"], a["lse_out"], a["do_base"], a["do_out"],
        a["dq"], a["dk"], a["dv"], a["dq_out"], a["dab"], a["dbb"], a["dao"], a["dbo"],
        a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("over,code", [
    (dict(Hq=3), 1),
    (dict(d=96), 2),
    (dict(window=0), 1),
    (dict(do_base=None), 1),
    (dict(dk=None), 1),
    (dict(dab=None), 1),
    (dict(q_out=1 << 12), 1),  # q_out without dq_out
    (dict(dq=(1 << 12) + 4), 1),  # misaligned
    (dict(indptr=(ctypes.c_int32 * 2)(0, 2)), 1),
    (dict(do_out=None), 1),
    (dict(ws=None), 4),
    (dict(ws_bytes=8), 4),
    (dict(ws=(1 << 12) + 16), 1),
])
def test_backward_host_checks(lib, over, code):
    assert _call_backward(lib, **over) == code
    assert ola.orthros_last_error() != ""


def test_backward_workspace_size(lib):
    assert ola.orthros_prefill_backward_workspace_size(2, 64, 4, 2, 128, 10, 16) > 0
    assert ola.orthros_prefill_backward_workspace_size(2, 64, 4, 2, 96, 10, 16) == 0
    assert ola.orthros_prefill_backward_workspace_size(2, 64, 4, 2, 128, -1, 16) == 0


def test_extend_host_checks(lib):
    P = 1 << 12
    ni = (ctypes.c_int32 * 3)(0, 2, 3)
    oi = (ctypes.c_int32 * 3)(0, 1, 1)

    def call(**over):
        a = dict(q=P, q_out=None, kn=P, vn=P, kc=P, vc=P, bt=P, max_pages=4, page_size=64, num_pages=8, lens=P,
                 ni=ni, oi=oi, pos=P, ab=P, bb=P, ao=P, bo=P, B=2, Hq=4, Hkv=2, d=128, w=16, scale=0.1, dtype=0,
                 ob=P, lb=P, oo=P, lo=P, ws=P, ws_bytes=1 << 30, stream=None)
        a.update(over)
        return lib.orthros_extend(a["q"], a["q_out"], a["kn"], a["vn"], a["kc"], a["vc"], a["bt"], a["max_pages"],
                                  a["page_size"], a["num_pages"], a["lens"], a["ni"], a["oi"], a["pos"], a["ab"],
                                  a["bb"], a["ao"], a["bo"], a["B"], a["Hq"], a["Hkv"], a["d"], a["w"], a["scale"],
                                  a["dtype"], a["ob"], a["lb"], a["oo"], a["lo"], a["ws"], a["ws_bytes"], a["stream"])

    assert call(Hq=3) == 1
    assert call(d=96) == 2
    assert call(max_pages=0) == 1
    assert call(ni=(ctypes.c_int32 * 3)(1, 2, 3)) == 1  # indptr[0] != 0
    assert call(oi=(ctypes.c_int32 * 3)(0, 2, 1)) == 1  # decreasing
    assert call(kn=None) == 1
    assert call(pos=None) == 1
    assert call(q=(1 << 12) + 2) == 1
    assert call(ws=None) == 4
    assert call(ws_bytes=8) == 4
    assert ola.orthros_extend_workspace_size(2, 3, 1, 4, 2, 128, 4, 64) > 0
    assert ola.orthros_extend_workspace_size(2, 3, 1, 4, 2, 96, 4, 64) == 0


def test_projection_host_checks(lib):
    P = 1 << 12

    def call(**over):
        a = dict(x=P, nb=2, no=1, dm=128, w=P, Hq=4, Hkv=2, d=64, ab=P, bb=P, ao=P, bo=P, qb=P, qo=P, ko=None,
                 vo=None, kc=None, vc=None, bt=None, B=0, mp=0, ps=0, np_=0, ts=None, tp=None, dtype=0, ws=P,
                 wsb=256, stream=None)
        a.update(over)
        return lib.orthros_qkv_project(a["x"], a["nb"], a["no"], a["dm"], a["w"], a["Hq"], a["Hkv"], a["d"], a["ab"],
                                       a["bb"], a["ao"], a["bo"], a["qb"], a["qo"], a["ko"], a["vo"], a["kc"], a["vc"],
                                       a["bt"], a["B"], a["mp"], a["ps"], a["np_"], a["ts"], a["tp"], a["dtype"],
                                       a["ws"], a["wsb"], a["stream"])

    assert call(dtype=1) == 2  # bf16 only
    assert call(d=96) == 2
    assert call(dm=100) == 2
    assert call(x=None) == 1
    assert call(ko=P) == 1  # k_out without v_out
    assert call(kc=P, vc=P, bt=P) == 1  # cache writes without token positions
    assert call(qo=None) == 1
    assert call(qb=P + 8) == 1
    assert call(ws=None) == 4


def test_product_path_fails_loudly_without_library(tmp_path):
    with pytest.raises(ola.OrthrosError):
        ola.load_library(str(tmp_path / "missing.so"))


def test_binding_does_not_import_oracle():
    import sys

    import efficient_long_context_gb300._binding  # noqa: F401
    src = open(os.path.join(ROOT, "efficient_long_context_gb300", "_binding.py")).read()
    assert "oracle" not in src
    for fn in os.listdir(os.path.join(ROOT, "efficient_long_context_gb300", "csrc")):
        assert "orthros_ref" not in open(os.path.join(ROOT, "efficient_long_context_gb300", "csrc", fn)).read()
    assert torch is not None and sys is not None


def test_host_tensors_are_refused_before_any_call():
    """A host tensor's address must never reach a kernel: the marshalling
    helper refuses it (checked on the helper itself, so no call is made)."""
    from efficient_long_context_gb300 import _binding

    with pytest.raises(_binding.OrthrosError, match="current CUDA device"):
        _binding._ptr(torch.zeros(4))
    assert _binding._ptr(None) is None
