"""Helpers of the GPU parity tests: run the CUDA path through the binding and
the oracle on the same seeded inputs, then compare element by element."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances of the parity contract: bf16 outputs 2e-2 (o) / 2e-3 (lse) max
# abs; the fp32 path 1e-3 on both.
TOL = {torch.bfloat16: (2e-2, 2e-3), torch.float32: (1e-3, 1e-3)}

# Largest errors seen per named workload and output in this test session
# (written out at the end of the session when ORTHROS_PARITY_JSON is set).
MARGINS: dict = {}


def record_margin(workload: str, errs: dict, tol: dict, what: str = "max abs error vs the oracle"):
    ent = MARGINS.setdefault(workload, {"measure": what, "errors": {}, "tolerance": {}})
    for k, v in errs.items():
        ent["errors"][k] = max(float(v), ent["errors"].get(k, 0.0))
        ent["tolerance"][k] = float(tol[k])


def f32(t: torch.Tensor) -> np.ndarray:
    """Exact widening of bf16 / fp32 CPU tensors for the oracle."""
    return t.float().numpy()


def max_err(gpu, ref) -> float:
    g = gpu.detach().float().cpu().numpy().astype(np.float64) if isinstance(gpu, torch.Tensor) else gpu
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if g.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite GPU output"
    return float(np.max(np.abs(g - r)))


def run_gpu_prefill(w, dev="cuda", fill_cache=None, page_size=64, workspace=None):
    import efficient_long_context_gb300 as ola

    q, k, v = (w[n].to(dev) for n in ("q", "k", "v"))
    aff = [w[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    pos = w["out_positions"].to(dev)
    q_out = w["q_out"].to(dev) if w.get("q_out") is not None else None
    kw = {}
    if fill_cache is not None:
        kw = dict(k_cache=fill_cache[0], v_cache=fill_cache[1], block_table=fill_cache[2],
                  page_size=fill_cache[0].shape[1])
    out = ola.orthros_prefill(q, k, v, *aff, w["out_indptr"], pos, w["window"], w["scale"], q_out=q_out,
                              workspace=workspace, **kw)
    torch.cuda.synchronize()
    return out


def run_oracle_prefill(w, base_rows=None, out_rows=None, nthreads=0):
    """Oracle on the same inputs; out_rows optionally restricts output rows
    (indices into out_positions), base_rows the base positions."""
    import oracle

    indptr = w["out_indptr"].numpy()
    pos = w["out_positions"].numpy()
    q_out = f32(w["q_out"]) if w.get("q_out") is not None else None
    if out_rows is not None:
        out_rows = np.asarray(out_rows)
        B = len(indptr) - 1
        seq = np.searchsorted(indptr, out_rows, side="right") - 1
        counts = np.bincount(seq, minlength=B)
        indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        order = np.argsort(seq, kind="stable")
        out_rows = out_rows[order]
        pos = pos[out_rows]
        if q_out is not None:
            q_out = q_out[out_rows]
    res = oracle.prefill(f32(w["q"]), f32(w["k"]), f32(w["v"]), f32(w["alpha_base"]), f32(w["beta_base"]),
                         f32(w["alpha_out"]), f32(w["beta_out"]), indptr, pos, w["window"], w["scale"],
                         q_out=q_out, base_rows=base_rows, nthreads=nthreads)
    return res, out_rows


def compare_prefill(w, gpu, base_rows=None, out_rows=None, what=""):
    (ob, lb, oo, lo), out_rows = run_oracle_prefill(w, base_rows, out_rows)
    g_ob, g_lb, g_oo, g_lo = gpu
    if base_rows is not None:
        idx = torch.as_tensor(np.asarray(base_rows), dtype=torch.long, device=g_ob.device)
        g_ob = g_ob.index_select(1, idx)
        g_lb = g_lb.index_select(2, idx)
    if out_rows is not None:
        idx = torch.as_tensor(out_rows, dtype=torch.long, device=g_oo.device)
        g_oo = g_oo.index_select(0, idx)
        g_lo = g_lo.index_select(0, idx)
    tol_o, tol_l = TOL[w["dtype"]]
    errs = dict(o_base=max_err(g_ob, ob), lse_base=max_err(g_lb, lb), o_out=max_err(g_oo, oo),
                lse_out=max_err(g_lo, lo))
    assert errs["o_base"] <= tol_o and errs["o_out"] <= tol_o, f"{what} {errs}"
    assert errs["lse_base"] <= tol_l and errs["lse_out"] <= tol_l, f"{what} {errs}"
    return errs


def prefill_tolerances(dtype):
    tol_o, tol_l = TOL[dtype]
    return {"o_base": tol_o, "lse_base": tol_l, "o_out": tol_o, "lse_out": tol_l}


def sample_positions(T, window, n_random, seed):
    """Positions that exercise tile and window edges plus random ones."""
    r = np.random.default_rng(seed)
    edges = {0, 1, 2, 63, 64, 65, 127, 128, 129, 255, 256, window - 2, window - 1, window, window + 1,
             window + 127, window + 128, T // 2, T - 129, T - 128, T - 2, T - 1}
    pts = sorted(p for p in edges if 0 <= p < T)
    extra = r.choice(T, size=min(n_random, T), replace=False)
    return np.array(sorted(set(pts) | set(int(x) for x in extra)), np.int32)
