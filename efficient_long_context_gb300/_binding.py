"""ctypes binding of include/orthros_attn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

ORTHROS_BF16 = 0
ORTHROS_F32 = 1
_DTYPES = {torch.bfloat16: ORTHROS_BF16, torch.float32: ORTHROS_F32}

STATUS_NAMES = {0: "ORTHROS_OK", 1: "ORTHROS_EINVAL", 2: "ORTHROS_EUNSUPPORTED", 3: "ORTHROS_ECUDA",
                4: "ORTHROS_EWORKSPACE", 5: "ORTHROS_EDEVICE", 6: "ORTHROS_ETIMEOUT"}

# the public symbols of include/orthros_attn.h
EXPORTS = ("orthros_prefill_workspace_size", "orthros_prefill", "orthros_prefill_from_host_workspace_size",
           "orthros_prefill_from_host", "orthros_prefill_shard_workspace_size",
           "orthros_prefill_shard", "orthros_merge_partials", "orthros_prefill_backward_workspace_size",
           "orthros_prefill_backward", "orthros_extend_workspace_size", "orthros_extend", "orthros_qkv_project",
           "orthros_decode_workspace_size",
           "orthros_decode", "orthros_decode_static", "orthros_check", "orthros_profile_begin", "orthros_profile_end",
           "orthros_selftest_wait_timeout", "orthros_status_string", "orthros_last_error")


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int), ("total_ms", ctypes.c_double)]


class OrthrosError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load_library(path: str | None = None):
    """Load liborthros_attn.so (built by efficient_long_context_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            raise OrthrosError(-1, f"{p} is missing: run efficient_long_context_gb300.build.build() first "
                                   "(there is no fallback path)")
        lib = ctypes.CDLL(p)
        vp, i32, f32p, i32p, sz = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_float), \
            ctypes.POINTER(ctypes.c_int32), ctypes.c_size_t
        lib.orthros_prefill_workspace_size.restype = sz
        lib.orthros_prefill_workspace_size.argtypes = [i32] * 7 + [i32]
        lib.orthros_prefill.restype = i32
        lib.orthros_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32p, vp, i32, vp,
                                        i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                        vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]
        lib.orthros_prefill_from_host_workspace_size.restype = sz
        lib.orthros_prefill_from_host_workspace_size.argtypes = [i32] * 8
        lib.orthros_prefill_from_host.restype = i32
        lib.orthros_prefill_from_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32p, i32p, i32, vp,
                                                  i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                                  vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, sz, vp]
        lib.orthros_prefill_shard_workspace_size.restype = sz
        lib.orthros_prefill_shard_workspace_size.argtypes = [i32] * 9
        lib.orthros_prefill_shard.restype = i32
        lib.orthros_prefill_shard.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32p, vp, i32, vp,
                                              i32, i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                              vp, vp, vp, vp, vp, sz, vp]
        lib.orthros_merge_partials.restype = i32
        lib.orthros_merge_partials.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]
        lib.orthros_prefill_backward_workspace_size.restype = sz
        lib.orthros_prefill_backward_workspace_size.argtypes = [i32] * 8
        lib.orthros_prefill_backward.restype = i32
        lib.orthros_prefill_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32p, vp, i32, vp,
                                                 i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                 vp, sz, vp]
        lib.orthros_extend_workspace_size.restype = sz
        lib.orthros_extend_workspace_size.argtypes = [i32] * 9
        lib.orthros_extend.restype = i32
        lib.orthros_extend.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp, i32p, i32p, vp,
                                       vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                       vp, vp, vp, vp, vp, sz, vp]
        lib.orthros_qkv_project.restype = i32
        lib.orthros_qkv_project.argtypes = [vp, i32, i32, i32, vp, i32, i32, i32, vp, vp, vp, vp,
                                            vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, i32,
                                            vp, sz, vp]
        lib.orthros_decode_workspace_size.restype = sz
        lib.orthros_decode_workspace_size.argtypes = [i32] * 7
        lib.orthros_decode.restype = i32
        lib.orthros_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp,
                                       vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                       vp, vp, vp, vp, vp, sz, vp]
        lib.orthros_decode_static.restype = i32
        lib.orthros_decode_static.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, vp,
                                              vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                                              vp, vp, vp, vp, vp]
        lib.orthros_selftest_wait_timeout.restype = i32
        lib.orthros_selftest_wait_timeout.argtypes = [ctypes.c_longlong, vp, sz, vp]
        lib.orthros_check.restype = i32
        lib.orthros_check.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
        lib.orthros_profile_begin.restype = i32
        lib.orthros_profile_begin.argtypes = []
        lib.orthros_profile_end.restype = i32
        lib.orthros_profile_end.argtypes = [ctypes.POINTER(KernelTime), i32]
        lib.orthros_status_string.restype = ctypes.c_char_p
        lib.orthros_status_string.argtypes = [i32]
        lib.orthros_last_error.restype = ctypes.c_char_p
        lib.orthros_last_error.argtypes = []
        del f32p
        if path is None:
            _lib = lib
        return lib


def orthros_status_string(status: int) -> str:
    return load_library().orthros_status_string(int(status)).decode()


def orthros_last_error() -> str:
    return load_library().orthros_last_error().decode()


def _raise_if(rc: int, lib):
    if rc != 0:
        raise OrthrosError(rc, lib.orthros_last_error().decode())


def _ptr(t):
    """Device address of a tensor argument. Every tensor the library reads or
    writes must live on the current CUDA device: a host tensor's address
    handed to a kernel would make it read host memory. Raised here, while the
    call's arguments are marshalled, so nothing is launched."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_cuda or t.device.index != torch.cuda.current_device():
            raise OrthrosError(1, f"tensor on {t.device}: every tensor argument must be on the current CUDA device")
        return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)
    return t


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise OrthrosError(1, f"unsupported element type {t.dtype}")
    return _DTYPES[t.dtype]


def _contig(name, t):
    if t is not None and not t.is_contiguous():
        raise OrthrosError(1, f"{name} must be contiguous")
    return t


def orthros_prefill_workspace_size(B, T, Hq, Hkv, d, n_out, window, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_prefill_workspace_size(B, T, Hq, Hkv, d, n_out, window, _DTYPES[dtype]))


def orthros_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, _DTYPES[dtype]))


def orthros_prefill(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions,
                    window, scale=None, *, q_out=None, out=None, k_cache=None, v_cache=None,
                    block_table=None, page_size=0, workspace=None, stream=None):
    """orthros_prefill of include/orthros_attn.h on torch CUDA tensors.

    out_indptr is a HOST int32 array-like [B+1]; every other tensor lives on
    the GPU. Returns (o_base [B,T,Hq,d], lse_base [B,Hq,T], o_out [n_out,Hq,d],
    lse_out [n_out,Hq]), allocated here unless `out` gives all four.
    """
    lib = load_library()
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    indptr = np.ascontiguousarray(np.asarray(out_indptr.cpu() if isinstance(out_indptr, torch.Tensor)
                                             else out_indptr, dtype=np.int32))
    n_out = int(indptr[-1]) if indptr.size else 0
    if scale is None:
        scale = d ** -0.5
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out), ("out_positions", out_positions)):
        _contig(name, t)
    if out is None:
        o_base = torch.empty_like(q)
        lse_base = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
        o_out = torch.empty((n_out, Hq, d), dtype=q.dtype, device=q.device)
        lse_out = torch.empty((n_out, Hq), dtype=torch.float32, device=q.device)
    else:
        o_base, lse_base, o_out, lse_out = out
    if workspace is None:
        ws = orthros_prefill_workspace_size(B, T, Hq, Hkv, d, n_out, window, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    max_pages = block_table.shape[1] if block_table is not None else 0
    num_pages = k_cache.shape[0] if k_cache is not None else 0
    rc = lib.orthros_prefill(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        indptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(out_positions), n_out, _ptr(q_out),
        B, T, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_out), _ptr(lse_out),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_pages, int(page_size), num_pages,
        _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_out, lse_out


def _host_ptr(t):
    """Host address of a CPU tensor argument of orthros_prefill_from_host."""
    if t is None:
        return None
    if t.is_cuda:
        raise OrthrosError(1, "orthros_prefill_from_host takes its inputs and outputs in host memory")
    _contig("host tensor", t)
    return ctypes.c_void_p(t.data_ptr())


def orthros_prefill_from_host_workspace_size(B, T, Hq, Hkv, d, n_out, window, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_prefill_from_host_workspace_size(B, T, Hq, Hkv, d, n_out, window,
                                                                       _DTYPES[dtype]))


def orthros_prefill_from_host(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions,
                              window, scale=None, *, q_out=None, out=None, k_cache=None, v_cache=None,
                              block_table=None, page_size=0, workspace=None, stream=None):
    """orthros_prefill_from_host of include/orthros_attn.h.

    q, k, v, out_positions, q_out and the outputs are CPU tensors (pinned, for
    copies that overlap the compute); the affines, the optional cache and the
    workspace are CUDA tensors. Returns (o_base, lse_base, o_out, lse_out) as
    CPU tensors, allocated here (pinned) unless `out` gives all four. The
    outputs are complete once `stream` has passed this call.
    """
    lib = load_library()
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    indptr = np.ascontiguousarray(np.asarray(out_indptr.cpu() if isinstance(out_indptr, torch.Tensor)
                                             else out_indptr, dtype=np.int32))
    n_out = int(indptr[-1]) if indptr.size else 0
    pos = np.ascontiguousarray(np.asarray(out_positions.cpu() if isinstance(out_positions, torch.Tensor)
                                          else out_positions, dtype=np.int32))
    if scale is None:
        scale = d ** -0.5
    if out is None:
        pin = torch.cuda.is_available()
        o_base = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
        lse_base = torch.empty((B, Hq, T), dtype=torch.float32, pin_memory=pin)
        o_out = torch.empty((n_out, Hq, d), dtype=q.dtype, pin_memory=pin)
        lse_out = torch.empty((n_out, Hq), dtype=torch.float32, pin_memory=pin)
    else:
        o_base, lse_base, o_out, lse_out = out
    dev = alpha_base.device
    if workspace is None:
        ws = orthros_prefill_from_host_workspace_size(B, T, Hq, Hkv, d, n_out, window, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=dev)
    max_pages = block_table.shape[1] if block_table is not None else 0
    num_pages = k_cache.shape[0] if k_cache is not None else 0
    rc = lib.orthros_prefill_from_host(
        _host_ptr(q), _host_ptr(k), _host_ptr(v), _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out),
        _ptr(beta_out), indptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if n_out else None, n_out, _host_ptr(q_out),
        B, T, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _host_ptr(o_base), _host_ptr(lse_base), _host_ptr(o_out) if n_out else None,
        _host_ptr(lse_out) if n_out else None,
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table), max_pages, int(page_size), num_pages,
        _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_out, lse_out


def orthros_prefill_shard_workspace_size(B, Tq, Tkv, Hq, Hkv, d, n_rows, window, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_prefill_shard_workspace_size(B, Tq, Tkv, Hq, Hkv, d, n_rows, window,
                                                                   _DTYPES[dtype]))


def orthros_prefill_shard(q, k, v, alpha_base, beta_base, alpha_out, beta_out, row_indptr, row_positions,
                          window, scale=None, *, q_rows=None, out=None, workspace=None, stream=None):
    """orthros_prefill_shard of include/orthros_attn.h on torch CUDA tensors.

    q [B, Tq, Hq, d] (the chunk's queries), k, v [B, Tkv, Hkv, d] (halo then
    chunk); row_indptr is a HOST int32 array-like [B+1], row_positions [n_rows]
    int32 in the K/V buffer's coordinates, q_rows [n_rows, Hq, d]. Returns
    (o_base [B,Tq,Hq,d], lse_base [B,Hq,Tq], o_part [n_rows,Hq,d] float,
    lse_part [n_rows,Hq] float), allocated here unless `out` gives all four.
    """
    lib = load_library()
    B, Tq, Hq, d = q.shape
    Tkv, Hkv = k.shape[1], k.shape[2]
    indptr = np.ascontiguousarray(np.asarray(row_indptr.cpu() if isinstance(row_indptr, torch.Tensor)
                                             else row_indptr, dtype=np.int32))
    n_rows = int(indptr[-1]) if indptr.size else 0
    if scale is None:
        scale = d ** -0.5
    for name, t in (("q", q), ("k", k), ("v", v), ("q_rows", q_rows), ("row_positions", row_positions)):
        _contig(name, t)
    if out is None:
        out = (torch.empty_like(q), torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device),
               torch.empty((n_rows, Hq, d), dtype=torch.float32, device=q.device),
               torch.empty((n_rows, Hq), dtype=torch.float32, device=q.device))
    o_base, lse_base, o_part, lse_part = out
    if workspace is None:
        ws = orthros_prefill_shard_workspace_size(B, Tq, Tkv, Hq, Hkv, d, n_rows, window, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    rc = lib.orthros_prefill_shard(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        indptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(row_positions), n_rows, _ptr(q_rows),
        B, Tq, Tkv, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_part), _ptr(lse_part), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_part, lse_part


def orthros_merge_partials(o_parts, lse_parts, dtype=torch.bfloat16, *, out=None, stream=None):
    """orthros_merge_partials of include/orthros_attn.h: o_parts [P, n, Hq, d]
    float, lse_parts [P, n, Hq] float -> (o [n, Hq, d] of `dtype`, lse [n, Hq])."""
    lib = load_library()
    P, n, Hq, d = o_parts.shape
    for name, t in (("o_parts", o_parts), ("lse_parts", lse_parts)):
        _contig(name, t)
    if out is None:
        out = (torch.empty((n, Hq, d), dtype=dtype, device=o_parts.device),
               torch.empty((n, Hq), dtype=torch.float32, device=o_parts.device))
    o, lse = out
    rc = lib.orthros_merge_partials(_ptr(o_parts), _ptr(lse_parts), P, n, Hq, d, _DTYPES[o.dtype], _ptr(o), _ptr(lse),
                                    _stream(stream))
    _raise_if(rc, lib)
    return o, lse


def orthros_prefill_backward_workspace_size(B, T, Hq, Hkv, d, n_out, window, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_prefill_backward_workspace_size(B, T, Hq, Hkv, d, n_out, window,
                                                                      _DTYPES[dtype]))


def orthros_prefill_backward(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions,
                             window, scale, o_base, lse_base, o_out, lse_out, do_base, do_out, *, q_out=None,
                             out=None, workspace=None, stream=None):
    """orthros_prefill_backward of include/orthros_attn.h on torch CUDA tensors.

    Returns a dict with dq, dk, dv, dq_out (None without q_out), d_alpha_base,
    d_beta_base, d_alpha_out, d_beta_out; allocated here unless `out` (a dict
    with the same keys) gives them.
    """
    lib = load_library()
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    indptr = np.ascontiguousarray(np.asarray(out_indptr.cpu() if isinstance(out_indptr, torch.Tensor)
                                             else out_indptr, dtype=np.int32))
    n_out = int(indptr[-1]) if indptr.size else 0
    if scale is None:
        scale = d ** -0.5
    for name, t in (("q", q), ("k", k), ("v", v), ("q_out", q_out), ("out_positions", out_positions),
                    ("o_base", o_base), ("o_out", o_out), ("do_base", do_base), ("do_out", do_out)):
        _contig(name, t)
    if out is None:
        dev = q.device
        out = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
               "dq_out": torch.empty_like(q_out) if q_out is not None else None}
        for n in ("d_alpha_base", "d_beta_base", "d_alpha_out", "d_beta_out"):
            out[n] = torch.empty((Hq, d), dtype=torch.float32, device=dev)
    if workspace is None:
        ws = orthros_prefill_backward_workspace_size(B, T, Hq, Hkv, d, n_out, window, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    rc = lib.orthros_prefill_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        indptr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _ptr(out_positions), n_out, _ptr(q_out),
        B, T, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_out), _ptr(lse_out), _ptr(do_base), _ptr(do_out),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dq_out"]),
        _ptr(out["d_alpha_base"]), _ptr(out["d_beta_base"]), _ptr(out["d_alpha_out"]), _ptr(out["d_beta_out"]),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return out


def orthros_extend_workspace_size(B, n_new, n_out, Hq, Hkv, d, max_pages, page_size, dtype=torch.bfloat16) -> int:
    return int(load_library().orthros_extend_workspace_size(B, n_new, n_out, Hq, Hkv, d, max_pages, page_size,
                                                            _DTYPES[dtype]))


def orthros_extend(q, k_new, v_new, k_cache, v_cache, block_table, cache_lens, new_indptr, out_indptr,
                   out_positions, alpha_base, beta_base, alpha_out, beta_out, window, scale=None, *, q_out=None,
                   out=None, workspace=None, stream=None):
    """orthros_extend of include/orthros_attn.h on torch CUDA tensors.

    new_indptr / out_indptr are HOST int32 array-likes [B+1]; k_cache /
    v_cache are updated in place. Returns (o_base [n_new,Hq,d], lse_base
    [n_new,Hq], o_out [n_out,Hq,d], lse_out [n_out,Hq]).
    """
    lib = load_library()
    n_new, Hq, d = q.shape
    Hkv = k_new.shape[1]
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    ni = np.ascontiguousarray(np.asarray(new_indptr, dtype=np.int32))
    oi = np.ascontiguousarray(np.asarray(out_indptr, dtype=np.int32))
    B = ni.shape[0] - 1
    n_out = int(oi[-1]) if oi.size else 0
    if scale is None:
        scale = d ** -0.5
    for name, t in (("q", q), ("q_out", q_out), ("k_new", k_new), ("v_new", v_new), ("out_positions", out_positions)):
        _contig(name, t)
    if out is None:
        out = (torch.empty_like(q), torch.empty((n_new, Hq), dtype=torch.float32, device=q.device),
               torch.empty((n_out, Hq, d), dtype=q.dtype, device=q.device),
               torch.empty((n_out, Hq), dtype=torch.float32, device=q.device))
    o_base, lse_base, o_out, lse_out = out
    if workspace is None:
        ws = orthros_extend_workspace_size(B, n_new, n_out, Hq, Hkv, d, max_pages, page_size, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    i32p = ctypes.POINTER(ctypes.c_int32)
    rc = lib.orthros_extend(
        _ptr(q), _ptr(q_out), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        max_pages, page_size, num_pages, _ptr(cache_lens), ni.ctypes.data_as(i32p), oi.ctypes.data_as(i32p),
        _ptr(out_positions), _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        B, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_out), _ptr(lse_out), _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_out, lse_out


def orthros_qkv_project(x, n_base, w_qkv, Hq, Hkv, d, alpha_base, beta_base, alpha_out, beta_out, *,
                        kv_out=False, k_cache=None, v_cache=None, block_table=None, token_seq=None,
                        token_pos=None, out=None, workspace=None, stream=None):
    """orthros_qkv_project of include/orthros_attn.h on torch CUDA tensors.

    x [n_base + n_out, d_model] (base rows first), w_qkv [(Hq+2Hkv) d, d_model].
    Returns (q_base [n_base,Hq,d], q_out [n_out,Hq,d], k [n_base,Hkv,d] or None,
    v or None); the caches are written in place when given.
    """
    lib = load_library()
    rows, d_model = x.shape
    n_out = rows - int(n_base)
    for name, t in (("x", x), ("w_qkv", w_qkv)):
        _contig(name, t)
    if out is None:
        dev = x.device
        out = (torch.empty((n_base, Hq, d), dtype=x.dtype, device=dev),
               torch.empty((n_out, Hq, d), dtype=x.dtype, device=dev),
               torch.empty((n_base, Hkv, d), dtype=x.dtype, device=dev) if kv_out else None,
               torch.empty((n_base, Hkv, d), dtype=x.dtype, device=dev) if kv_out else None)
    q_b, q_o, k_o, v_o = out
    if workspace is None:
        workspace = torch.empty(256, dtype=torch.uint8, device=x.device)
    max_pages = block_table.shape[1] if block_table is not None else 0
    B = block_table.shape[0] if block_table is not None else 0
    page_size = k_cache.shape[1] if k_cache is not None else 0
    num_pages = k_cache.shape[0] if k_cache is not None else 0
    rc = lib.orthros_qkv_project(
        _ptr(x), int(n_base), n_out, d_model, _ptr(w_qkv), Hq, Hkv, d,
        _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        _ptr(q_b), _ptr(q_o), _ptr(k_o), _ptr(v_o), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), B,
        max_pages, page_size, num_pages, _ptr(token_seq), _ptr(token_pos), _dtype(x),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return out


def orthros_decode(q, k_new, v_new, k_cache, v_cache, block_table, cache_lens, alpha_base, beta_base,
                   alpha_out, beta_out, window, scale=None, *, q_out=None, out=None, workspace=None,
                   stream=None):
    """orthros_decode of include/orthros_attn.h on torch CUDA tensors.

    k_cache / v_cache [num_pages, page_size, Hkv, d] are updated in place.
    Returns (o_base [B,Hq,d], lse_base [B,Hq], o_out [B,Hq,d], lse_out [B,Hq]).
    """
    lib = load_library()
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        o_base = torch.empty_like(q)
        o_out = torch.empty_like(q)
        lse_base = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
        lse_out = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    else:
        o_base, lse_base, o_out, lse_out = out
    if workspace is None:
        ws = orthros_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size, q.dtype)
        workspace = torch.empty(max(ws, 256), dtype=torch.uint8, device=q.device)
    rc = lib.orthros_decode(
        _ptr(q), _ptr(q_out), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        max_pages, page_size, num_pages, _ptr(cache_lens),
        _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        B, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_out), _ptr(lse_out),
        _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_out, lse_out


def orthros_decode_static(q, k_new, v_new, k_cache, v_cache, block_table, cache_lens, alpha_base, beta_base,
                          alpha_out, beta_out, window, scale=None, *, q_out=None, out=None, stream=None):
    """orthros_decode_static of include/orthros_attn.h: orthros_decode with the
    library's built-in scratch array instead of a caller workspace."""
    lib = load_library()
    B, Hq, d = q.shape
    Hkv = k_new.shape[1]
    num_pages, page_size = k_cache.shape[0], k_cache.shape[1]
    max_pages = block_table.shape[1]
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = (torch.empty_like(q), torch.empty((B, Hq), dtype=torch.float32, device=q.device),
               torch.empty_like(q), torch.empty((B, Hq), dtype=torch.float32, device=q.device))
    o_base, lse_base, o_out, lse_out = out
    rc = lib.orthros_decode_static(
        _ptr(q), _ptr(q_out), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        max_pages, page_size, num_pages, _ptr(cache_lens),
        _ptr(alpha_base), _ptr(beta_base), _ptr(alpha_out), _ptr(beta_out),
        B, Hq, Hkv, d, int(window), float(scale), _dtype(q),
        _ptr(o_base), _ptr(lse_base), _ptr(o_out), _ptr(lse_out), _stream(stream))
    _raise_if(rc, lib)
    return o_base, lse_base, o_out, lse_out


def orthros_selftest_wait_timeout(limit_cycles, workspace, stream=None):
    """orthros_selftest_wait_timeout of include/orthros_attn.h: one kernel whose
    bounded wait on a barrier nothing arms runs out after limit_cycles."""
    lib = load_library()
    rc = lib.orthros_selftest_wait_timeout(int(limit_cycles), _ptr(workspace), workspace.numel(), _stream(stream))
    _raise_if(rc, lib)


def orthros_check(workspace, stream=None):
    """Synchronise and read the device status word. Returns (status, bits)."""
    lib = load_library()
    bits = ctypes.c_uint32(0)
    rc = lib.orthros_check(_ptr(workspace), _stream(stream), ctypes.byref(bits))
    return int(rc), int(bits.value)


def orthros_profile_begin():
    """Start recording per-kernel CUDA-event times of the library's launches."""
    _raise_if(load_library().orthros_profile_begin(), load_library())


def orthros_profile_end():
    """Stop recording; returns {kernel name: (launches, total_ms)} in first-launch order."""
    lib = load_library()
    buf = (KernelTime * 64)()
    n = lib.orthros_profile_end(buf, 64)
    if n < 0:
        raise OrthrosError(3, "orthros_profile_end: CUDA error while reading events")
    return {buf[i].name.decode(): (buf[i].launches, buf[i].total_ms) for i in range(min(n, 64))}
