"""orthros_prefill_from_host: the prefill with host-memory inputs and outputs.

Sequences longer than one chunk (16384 tokens here) run as chunked shards with
copies overlapping the compute; the results are checked against the oracle
(sampled base rows around every chunk boundary, every output row) and against
orthros_prefill on the device copies of the same inputs; the cache fill
against orthros_prefill's, byte for byte. Sequences of one chunk take the plain
copy / compute / copy path, which must give orthros_prefill's results exactly.
The argument checks made on the host run without a GPU.
"""
import ctypes

import numpy as np
import pytest
import torch

from efficient_long_context_gb300 import workloads as W
from tests.parity_util import TOL, compare_prefill, max_err


def _workload(B, T, window, positions_per_seq, seed):
    wdef = W.PrefillWorkload("from_host", B, T, 8, 2, 128, window, torch.bfloat16, "last", seed=seed)
    w = W.make_prefill(wdef)
    counts = [len(p) for p in positions_per_seq]
    w["out_indptr"] = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32)
    w["out_positions"] = torch.tensor(np.concatenate(positions_per_seq), dtype=torch.int32)
    return w


def _from_host(w, cache=None, workspace=None):
    import efficient_long_context_gb300 as ola

    aff = [w[n].cuda() for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    kw = {}
    if cache is not None:
        kw = dict(k_cache=cache[0], v_cache=cache[1], block_table=cache[2], page_size=cache[0].shape[1])
    if w.get("q_out") is not None:
        kw["q_out"] = w["q_out"].pin_memory()
    out = ola.orthros_prefill_from_host(w["q"].pin_memory(), w["k"].pin_memory(), w["v"].pin_memory(), *aff,
                                        w["out_indptr"], w["out_positions"], w["window"], w["scale"],
                                        workspace=workspace, **kw)
    torch.cuda.synchronize()
    return out


def _device(w, cache=None):
    import efficient_long_context_gb300 as ola

    q, k, v = (w[n].cuda() for n in ("q", "k", "v"))
    aff = [w[n].cuda() for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    kw = {}
    if cache is not None:
        kw = dict(k_cache=cache[0], v_cache=cache[1], block_table=cache[2], page_size=cache[0].shape[1])
    if w.get("q_out") is not None:
        kw["q_out"] = w["q_out"].cuda()
    out = ola.orthros_prefill(q, k, v, *aff, w["out_indptr"], w["out_positions"].cuda(), w["window"], w["scale"],
                              **kw)
    torch.cuda.synchronize()
    return [t.cpu() for t in out]


def _chunk_starts(T, chunk=16384):
    """The chunk boundaries the library uses for a sequence of T tokens (a
    quarter chunk, full chunks, the remainder ending in a quarter chunk)."""
    if T <= chunk:
        return [0, T]
    q = max(128, (chunk // 4) & ~127)
    st, t = [0], q
    while T - t > chunk + q:
        st.append(t)
        t += chunk
    if T - t > q:
        st.append(t)
        t = T - q
    return st + [t, T]


def _cache(B, T, Hkv, d, page_size=64, seed=0):
    pages = B * ((T + page_size - 1) // page_size)
    perm = torch.randperm(pages, generator=torch.Generator().manual_seed(seed)).to(torch.int32)
    kc = torch.zeros((pages, page_size, Hkv, d), dtype=torch.bfloat16, device="cuda")
    return kc, torch.zeros_like(kc), perm.view(B, -1).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("B,T,window", [(1, 40000, 1024), (2, 33000, 4096), (1, 20000, 1)])
def test_chunked_from_host_matches_oracle_and_device_call(B, T, window):
    import efficient_long_context_gb300 as ola

    rng = np.random.default_rng(T + window)
    per_seq = []
    for b in range(B):
        run = np.arange(T - 700, T - 688)  # a run of consecutive positions (one copy for the run)
        pts = [0, 5, 16383, 16384, 16385, T // 2, T - 1, T - 1] + list(rng.integers(0, T, 4))
        per_seq.append(np.array(sorted(pts)[:6] + list(run) + sorted(pts)[6:], np.int32))
    w = _workload(B, T, window, per_seq, seed=7 + B)
    cache_h, cache_d = _cache(B, T, 2, 128, seed=1), _cache(B, T, 2, 128, seed=1)
    ws = torch.empty(ola.orthros_prefill_from_host_workspace_size(B, T, 8, 2, 128, int(w["out_indptr"][-1]), window),
                     dtype=torch.uint8, device="cuda")
    got = _from_host(w, cache_h, ws)
    assert all(not t.is_cuda for t in got)
    rc, bits = ola.orthros_check(ws)
    assert rc == 0 and bits == 0, (rc, bits)
    # every output row and the base rows around each chunk boundary, against the oracle
    edges = {0, 1, 127, 128, T - 1, T - 2}
    for b0 in _chunk_starts(T)[1:-1]:
        edges |= {b0 + e for e in (-2, -1, 0, 1, 127, 128, window - 1, window)}
    base_rows = np.array(sorted(x for x in edges if 0 <= x < T), np.int32)
    compare_prefill(w, got, base_rows=base_rows, what=f"from_host B={B} T={T} w={window}")
    # the device call on the same inputs: both are within the oracle's
    # tolerance of the exact values, so within twice it of each other (the
    # chunks' key tiles start at other offsets, so P is rounded in other groups;
    # a row with a single key, window 1, keeps bf16(P) / l != 1 in its output)
    ref = _device(w, cache_d)
    tol_o, tol_l = TOL[torch.bfloat16]
    for name, a, r, tol in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref, (tol_o, tol_l, tol_o, tol_l)):
        err = max_err(a, r.float())
        assert err <= 2 * tol, (name, err)
    # the cache fill, byte for byte
    assert torch.equal(cache_h[0], cache_d[0]) and torch.equal(cache_h[1], cache_d[1])


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["q_out", "no_output_rows"])
def test_chunked_from_host_variants(variant):
    """Chunked path with the output rows' own raw queries (q_out, copied in
    once) and with no output rows at all, against orthros_prefill."""
    T = 36000
    if variant == "q_out":
        pos = [np.array([3, 4100, 4101, 20000, 35999], np.int32)]
    else:
        pos = [np.zeros(0, np.int32)]
    w = _workload(1, T, 2048, pos, seed=21)
    if variant == "q_out":
        w["q_out"] = torch.randn((len(pos[0]), 8, 128), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    got = _from_host(w)
    ref = _device(w)
    tol_o, tol_l = TOL[torch.bfloat16]
    for name, a, r, tol in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref, (tol_o, tol_l, tol_o, tol_l)):
        assert a.shape == r.shape, name
        err = max_err(a, r.float())
        assert err <= 2 * tol, (name, err)
    if variant == "q_out":
        compare_prefill(w, got, base_rows=np.array([0, 4095, 4096, 20479, 20480, T - 1], np.int32), what="q_out")


@pytest.mark.gpu
def test_single_chunk_from_host_f32_equals_device_call():
    """f32 takes the copy / compute / copy path (no chunks)."""
    T = 300
    wdef = W.PrefillWorkload("from_host_f32", 1, T, 4, 2, 64, 50, torch.float32, "last", seed=4)
    w = W.make_prefill(wdef)
    w["out_indptr"] = torch.tensor([0, 3], dtype=torch.int32)
    w["out_positions"] = torch.tensor([0, 150, 299], dtype=torch.int32)
    got = _from_host(w)
    ref = _device(w)
    for name, a, r in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref):
        assert torch.equal(a, r), name


@pytest.mark.gpu
def test_single_chunk_from_host_equals_device_call():
    T = 3000
    w = _workload(2, T, 512, [np.array([0, 999, 2999], np.int32), np.arange(2000, 2100, dtype=np.int32)], seed=3)
    got = _from_host(w)
    ref = _device(w)
    for name, a, r in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref):
        assert torch.equal(a, r), name


def test_host_checks_without_gpu():
    """Positions outside [0, T) and a missing workspace are refused before
    anything reaches the GPU (ctypes call with NULL device pointers)."""
    import efficient_long_context_gb300 as ola

    lib = ola.load_library()
    B, T, Hq, Hkv, d = 1, 100, 2, 1, 64
    host = lambda n, dt: np.zeros(n, dt)
    q = host(B * T * Hq * d, np.uint16)
    k = host(B * T * Hkv * d, np.uint16)
    o = host(B * T * Hq * d, np.uint16)
    lse = host(B * Hq * T, np.float32)
    oo, lo = host(Hq * d, np.uint16), host(Hq, np.float32)
    indptr = np.array([0, 1], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    i32p = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def call(pos, ws_bytes):
        return lib.orthros_prefill_from_host(p(q), p(k), p(k), None, None, None, None, i32p(indptr), i32p(pos), 1,
                                             None, B, T, Hq, Hkv, d, 16, 0.125, 0, p(o), p(lse), p(oo), p(lo),
                                             None, None, None, 0, 0, 0, None, ws_bytes, None)

    assert call(np.array([T], np.int32), 0) == 1  # ORTHROS_EINVAL: position past the sequence
    assert "outside" in ola.orthros_last_error()
    assert call(np.array([-1], np.int32), 0) == 1
    assert call(np.array([T - 1], np.int32), 0) == 4  # ORTHROS_EWORKSPACE: no workspace
    assert lib.orthros_prefill_from_host_workspace_size(B, T, Hq, Hkv, d, 1, 16, 0) > 0
    assert lib.orthros_prefill_from_host_workspace_size(B, T, Hq, Hkv, 96, 1, 16, 0) == 0  # unsupported d
