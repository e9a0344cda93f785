"""ctypes front end of the plain-C oracle ``orthros_ref.c``.

TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the
benchmark's CPU-baseline leg. The CUDA library neither imports nor links it.

Inputs are numpy float32 arrays (bf16 data is widened to float32 exactly by
the caller); outputs are float64. The functions here only marshal arguments:
all arithmetic is in the C file, which follows Sec. 3.1 (Eq. 4, Eq. 5, the
query affines) and Sec. 3.2 (the decoding pair) of the Orthros paper.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "orthros_ref.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liborthros_ref.so")
_lock = threading.Lock()
_lib = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into oracle/_build/."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.orthros_ref_prefill.restype = ctypes.c_int
    lib.orthros_ref_prefill.argtypes = [
        _f32p, _f32p, _f32p,  # q k v
        _f32p, _f32p, _f32p, _f32p,  # alpha/beta base, alpha/beta out
        _i32p, _i32p, _f32p,  # out_indptr out_positions q_out
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double,  # B T Hq Hkv d window scale
        _i32p, ctypes.c_int,  # base_rows n_base_rows
        _f64p, _f64p, _f64p, _f64p,  # o_base lse_base o_out lse_out
        ctypes.c_int,  # nthreads
    ]
    lib.orthros_ref_decode.restype = ctypes.c_int
    lib.orthros_ref_decode.argtypes = [
        _f32p, _f32p, _f32p, _f32p,  # q q_out k_new v_new
        _f32p, _f32p,  # k_cache v_cache
        _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,  # block_table max_pages page_size num_pages
        _i32p,  # cache_lens
        _f32p, _f32p, _f32p, _f32p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double,  # B Hq Hkv d window scale
        _f64p, _f64p, _f64p, _f64p,
        ctypes.c_int,
    ]
    lib.orthros_ref_qkv_project.restype = ctypes.c_int
    lib.orthros_ref_qkv_project.argtypes = [
        _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _f32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        _f32p, _f32p, _f32p, _f32p,
        _f64p, _f64p, _f64p, _f64p,
        _f32p, _f32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, _i32p, _i32p,
        ctypes.c_int,
    ]
    lib.orthros_ref_extend.restype = ctypes.c_int
    lib.orthros_ref_extend.argtypes = [
        _f32p, _f32p, _f32p, _f32p,  # q q_out k_new v_new
        _f32p, _f32p,  # caches
        _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,  # block_table max_pages page_size num_pages
        _i32p, _i32p, _i32p, _i32p,  # cache_lens new_indptr out_indptr out_positions
        _f32p, _f32p, _f32p, _f32p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
        _f64p, _f64p, _f64p, _f64p,
        ctypes.c_int,
    ]
    lib.orthros_ref_prefill_backward.restype = ctypes.c_int
    lib.orthros_ref_prefill_backward.argtypes = [
        _f32p, _f32p, _f32p,  # q k v
        _f32p, _f32p, _f32p, _f32p,  # affines
        _i32p, _i32p, _f32p,  # out_indptr out_positions q_out
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_double,  # B T Hq Hkv d window scale
        _f32p, _f32p, ctypes.c_int, ctypes.c_int,  # do_base do_out row_lo row_hi
        _f64p, _f64p, _f64p, _f64p,  # dq dk dv dq_out
        _f64p, _f64p, _f64p, _f64p,  # d alpha/beta base, d alpha/beta out
        ctypes.c_int,
    ]
    lib.orthros_ref_max_threads.restype = ctypes.c_int
    lib.orthros_ref_max_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


class Oracle:
    """The oracle bound to one compiled library (the default build, or another
    build of the same C source, e.g. one a test compiled with a planted mistake)."""

    def __init__(self, path=None):
        self._lib = _bind(path) if path else _load()

    def prefill(self, *args, **kwargs):
        return prefill(*args, _lib=self._lib, **kwargs)

    def decode(self, *args, **kwargs):
        return decode(*args, _lib=self._lib, **kwargs)

    def prefill_backward(self, *args, **kwargs):
        return prefill_backward(*args, _lib=self._lib, **kwargs)

    def extend(self, *args, **kwargs):
        return extend(*args, _lib=self._lib, **kwargs)

    def qkv_project(self, *args, **kwargs):
        return qkv_project(*args, _lib=self._lib, **kwargs)


def max_threads() -> int:
    return int(_load().orthros_ref_max_threads())


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a, t):
    if a is None:
        return ctypes.cast(None, t)
    return a.ctypes.data_as(t)


def prefill(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr,
            out_positions, window, scale, q_out=None, base_rows=None, nthreads=0, _lib=None):
    """Eq. 4 (every listed base row) and Eq. 5 (every output row) in float64.

    q [B,T,Hq,d], k/v [B,T,Hkv,d], affines [Hq,d], out_indptr [B+1] and
    out_positions [n_out] (CSR over sequences), q_out [n_out,Hq,d] or None.
    base_rows: None for all T positions, else an int array of positions.
    Returns (o_base, lse_base, o_out, lse_out) with shapes
    [B,R,Hq,d], [B,Hq,R], [n_out,Hq,d], [n_out,Hq] (R = T or len(base_rows)).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, d) and v.shape == k.shape
    ab, bb, ao, bo = (_f32(x) for x in (alpha_base, beta_base, alpha_out, beta_out))
    for x in (ab, bb, ao, bo):
        assert x.shape == (Hq, d)
    out_indptr = _i32(out_indptr)
    out_positions = _i32(out_positions if out_positions is not None else np.zeros(0, np.int32))
    assert out_indptr.shape == (B + 1,)
    n_out = int(out_indptr[-1])
    assert out_positions.shape == (n_out,)
    q_out = _f32(q_out)
    if q_out is not None:
        assert q_out.shape == (n_out, Hq, d)
    rows = _i32(base_rows)
    R = T if rows is None else rows.shape[0]
    o_base = np.zeros((B, R, Hq, d), np.float64)
    lse_base = np.zeros((B, Hq, R), np.float64)
    o_out = np.zeros((max(n_out, 0), Hq, d), np.float64)
    lse_out = np.zeros((max(n_out, 0), Hq), np.float64)
    # a zero-length row list still needs a valid pointer
    rows_arg = rows if rows is None or rows.size else np.zeros(1, np.int32)
    rc = (_lib or _load()).orthros_ref_prefill(
        _ptr(q, _f32p), _ptr(k, _f32p), _ptr(v, _f32p),
        _ptr(ab, _f32p), _ptr(bb, _f32p), _ptr(ao, _f32p), _ptr(bo, _f32p),
        _ptr(out_indptr, _i32p), _ptr(out_positions, _i32p), _ptr(q_out, _f32p),
        B, T, Hq, Hkv, d, int(window), float(scale),
        _ptr(rows_arg, _i32p), R,
        _ptr(o_base, _f64p), _ptr(lse_base, _f64p), _ptr(o_out, _f64p), _ptr(lse_out, _f64p),
        int(nthreads),
    )
    if rc != 0:
        raise ValueError(f"orthros_ref_prefill failed with code {rc}")
    return o_base, lse_base, o_out, lse_out


def decode(q, k_new, v_new, k_cache, v_cache, block_table, cache_lens,
           alpha_base, beta_base, alpha_out, beta_out, window, scale,
           q_out=None, nthreads=0, _lib=None):
    """One decoding step (Sec. 3.2): append, then Eq. 4 and Eq. 5 rows.

    k_cache / v_cache [num_pages, page_size, Hkv, d] float32 arrays are
    MODIFIED in place (the new K/V lands at position cache_lens[b]).
    Returns (o_base, lse_base, o_out, lse_out): [B,Hq,d], [B,Hq] twice.
    """
    q, k_new, v_new = _f32(q), _f32(k_new), _f32(v_new)
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float32 and v_cache.flags.c_contiguous
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    assert k_cache.shape == (num_pages, page_size, Hkv, d) and v_cache.shape == k_cache.shape
    block_table = _i32(block_table)
    max_pages = block_table.shape[1]
    cache_lens = _i32(cache_lens)
    ab, bb, ao, bo = (_f32(x) for x in (alpha_base, beta_base, alpha_out, beta_out))
    q_out = _f32(q_out)
    o_base = np.zeros((B, Hq, d), np.float64)
    o_out = np.zeros((B, Hq, d), np.float64)
    lse_base = np.zeros((B, Hq), np.float64)
    lse_out = np.zeros((B, Hq), np.float64)
    rc = (_lib or _load()).orthros_ref_decode(
        _ptr(q, _f32p), _ptr(q_out, _f32p), _ptr(k_new, _f32p), _ptr(v_new, _f32p),
        _ptr(k_cache, _f32p), _ptr(v_cache, _f32p),
        _ptr(block_table, _i32p), max_pages, page_size, num_pages, _ptr(cache_lens, _i32p),
        _ptr(ab, _f32p), _ptr(bb, _f32p), _ptr(ao, _f32p), _ptr(bo, _f32p),
        B, Hq, Hkv, d, int(window), float(scale),
        _ptr(o_base, _f64p), _ptr(lse_base, _f64p), _ptr(o_out, _f64p), _ptr(lse_out, _f64p),
        int(nthreads),
    )
    if rc != 0:
        raise ValueError(f"orthros_ref_decode failed with code {rc}")
    return o_base, lse_base, o_out, lse_out


def prefill_backward(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr,
                     out_positions, window, scale, do_base, do_out, q_out=None,
                     row_range=None, nthreads=0, _lib=None):
    """Gradients of Eq. 4 (all T base rows) and Eq. 5 (the output rows) in float64.

    do_base [B,T,Hq,d] and do_out [n_out,Hq,d] are dL/do of the two streams.
    row_range (lo, hi): only rows at positions in [lo, hi) contribute (default
    all); [t0, T) still gives exact dk/dv for keys >= t0 and exact dq in range.
    Returns a dict with dq [B,T,Hq,d], dk, dv [B,T,Hkv,d], dq_out [n_out,Hq,d]
    (None when q_out is None: the output rows' gradient then lands in dq),
    d_alpha_base, d_beta_base, d_alpha_out, d_beta_out [Hq,d].
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, T, Hkv, d) and v.shape == k.shape
    ab, bb, ao, bo = (_f32(x) for x in (alpha_base, beta_base, alpha_out, beta_out))
    out_indptr = _i32(out_indptr)
    out_positions = _i32(out_positions if out_positions is not None else np.zeros(0, np.int32))
    n_out = int(out_indptr[-1])
    assert out_positions.shape == (n_out,)
    q_out = _f32(q_out)
    if q_out is not None:
        assert q_out.shape == (n_out, Hq, d)
    do_base = _f32(do_base)
    assert do_base.shape == (B, T, Hq, d)
    do_out = _f32(do_out if do_out is not None else np.zeros((n_out, Hq, d), np.float32))
    assert do_out.shape == (n_out, Hq, d)
    dq = np.zeros((B, T, Hq, d), np.float64)
    dk = np.zeros((B, T, Hkv, d), np.float64)
    dv = np.zeros((B, T, Hkv, d), np.float64)
    dq_out = np.zeros((n_out, Hq, d), np.float64) if q_out is not None else None
    grads = [np.zeros((Hq, d), np.float64) for _ in range(4)]
    # zero-length arrays still need valid pointers
    pos_arg = out_positions if out_positions.size else np.zeros(1, np.int32)
    do_out_arg = do_out if do_out.size else np.zeros(1, np.float32)
    rc = (_lib or _load()).orthros_ref_prefill_backward(
        _ptr(q, _f32p), _ptr(k, _f32p), _ptr(v, _f32p),
        _ptr(ab, _f32p), _ptr(bb, _f32p), _ptr(ao, _f32p), _ptr(bo, _f32p),
        _ptr(out_indptr, _i32p), _ptr(pos_arg, _i32p), _ptr(q_out, _f32p),
        B, T, Hq, Hkv, d, int(window), float(scale),
        _ptr(do_base, _f32p), _ptr(do_out_arg, _f32p),
        int(row_range[0]) if row_range else 0, int(row_range[1]) if row_range else T,
        _ptr(dq, _f64p), _ptr(dk, _f64p), _ptr(dv, _f64p), _ptr(dq_out, _f64p),
        *(_ptr(g, _f64p) for g in grads),
        int(nthreads),
    )
    if rc != 0:
        raise ValueError(f"orthros_ref_prefill_backward failed with code {rc}")
    return {"dq": dq, "dk": dk, "dv": dv, "dq_out": dq_out,
            "d_alpha_base": grads[0], "d_beta_base": grads[1],
            "d_alpha_out": grads[2], "d_beta_out": grads[3]}


def extend(q, k_new, v_new, k_cache, v_cache, block_table, cache_lens, new_indptr, out_indptr, out_positions,
           alpha_base, beta_base, alpha_out, beta_out, window, scale, q_out=None, nthreads=0, _lib=None):
    """One continuous-batching step (appends, then Eq. 4 rows of the new tokens
    and Eq. 5 output rows) in float64; k_cache / v_cache are MODIFIED in place.
    q [n_new,Hq,d], k_new/v_new [n_new,Hkv,d], new_indptr/out_indptr [B+1],
    out_positions [n_out] absolute positions. Returns (o_base [n_new,Hq,d],
    lse_base [n_new,Hq], o_out [n_out,Hq,d], lse_out [n_out,Hq])."""
    q, k_new, v_new = _f32(q), _f32(k_new), _f32(v_new)
    n_new, Hq, d = q.shape
    Hkv = k_new.shape[1]
    assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.float32 and v_cache.flags.c_contiguous
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    block_table = _i32(block_table)
    max_pages = block_table.shape[1]
    new_indptr, out_indptr = _i32(new_indptr), _i32(out_indptr)
    B = new_indptr.shape[0] - 1
    assert out_indptr.shape == (B + 1,) and int(new_indptr[-1]) == n_new
    n_out = int(out_indptr[-1])
    out_positions = _i32(out_positions if out_positions is not None else np.zeros(0, np.int32))
    cache_lens = _i32(cache_lens)
    ab, bb, ao, bo = (_f32(x) for x in (alpha_base, beta_base, alpha_out, beta_out))
    q_out = _f32(q_out)
    o_base = np.zeros((n_new, Hq, d), np.float64)
    lse_base = np.zeros((n_new, Hq), np.float64)
    o_out = np.zeros((n_out, Hq, d), np.float64)
    lse_out = np.zeros((n_out, Hq), np.float64)
    dummy_f = np.zeros(1, np.float32)
    dummy_i = np.zeros(1, np.int32)
    rc = (_lib or _load()).orthros_ref_extend(
        _ptr(q if n_new else dummy_f, _f32p), _ptr(q_out, _f32p), _ptr(k_new if n_new else dummy_f, _f32p),
        _ptr(v_new if n_new else dummy_f, _f32p), _ptr(k_cache, _f32p), _ptr(v_cache, _f32p),
        _ptr(block_table, _i32p), max_pages, page_size, num_pages,
        _ptr(cache_lens, _i32p), _ptr(new_indptr, _i32p), _ptr(out_indptr, _i32p),
        _ptr(out_positions if n_out else dummy_i, _i32p),
        _ptr(ab, _f32p), _ptr(bb, _f32p), _ptr(ao, _f32p), _ptr(bo, _f32p),
        B, Hq, Hkv, d, int(window), float(scale),
        _ptr(o_base, _f64p), _ptr(lse_base, _f64p), _ptr(o_out, _f64p), _ptr(lse_out, _f64p), int(nthreads))
    if rc != 0:
        raise ValueError(f"orthros_ref_extend failed with code {rc}")
    return o_base, lse_base, o_out, lse_out


def qkv_project(x, n_base, w_t, Hq, Hkv, d, alpha_base, beta_base, alpha_out, beta_out,
                k_cache=None, v_cache=None, block_table=None, token_seq=None, token_pos=None,
                nthreads=0, _lib=None):
    """Shared Q/K/V projection of base rows x[:n_base] and output rows
    x[n_base:] with the stream affines on the query part (float64). The
    caches (float32, [num_pages, page_size, Hkv, d]) are MODIFIED when given.
    Returns (q_base [n_base,Hq,d], q_out [n_out,Hq,d], k, v [n_base,Hkv,d])."""
    x, w_t = _f32(x), _f32(w_t)
    rows, d_model = x.shape
    n_out = rows - n_base
    Nq, Nkv = Hq * d, Hkv * d
    assert w_t.shape == (Nq + 2 * Nkv, d_model)
    ab, bb, ao, bo = (_f32(a).reshape(-1) for a in (alpha_base, beta_base, alpha_out, beta_out))
    qb = np.zeros((n_base, Hq, d), np.float64)
    qo = np.zeros((n_out, Hq, d), np.float64)
    k = np.zeros((n_base, Hkv, d), np.float64)
    v = np.zeros((n_base, Hkv, d), np.float64)
    if k_cache is not None:
        assert k_cache.dtype == np.float32 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        bt = _i32(block_table)
        max_pages, page_size, num_pages = bt.shape[1], k_cache.shape[1], k_cache.shape[0]
        ts, tp = _i32(token_seq), _i32(token_pos)
    else:
        bt = ts = tp = None
        max_pages = page_size = num_pages = 1
    rc = (_lib or _load()).orthros_ref_qkv_project(
        _ptr(x, _f32p), int(n_base), int(n_out), int(d_model), _ptr(w_t, _f32p), Hq, Hkv, d,
        _ptr(ab, _f32p), _ptr(bb, _f32p), _ptr(ao, _f32p), _ptr(bo, _f32p),
        _ptr(qb, _f64p), _ptr(qo, _f64p), _ptr(k, _f64p), _ptr(v, _f64p),
        _ptr(k_cache, _f32p), _ptr(v_cache, _f32p), _ptr(bt, _i32p), max_pages, page_size, num_pages,
        _ptr(ts, _i32p), _ptr(tp, _i32p), int(nthreads))
    if rc != 0:
        raise ValueError(f"orthros_ref_qkv_project failed with code {rc}")
    return qb, qo, k, v
