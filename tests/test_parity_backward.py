"""GPU parity of orthros_prefill_backward against the CPU oracle.

The GPU backward consumes the GPU forward's o and lse (as a training step
would); the oracle recomputes everything in float64 from the same inputs.
Small shapes are compared in full. The named training workloads run at full
size; the oracle then takes one sequence and the rows at positions [T-n, T),
which gives exact dk/dv for those keys and exact dq for those rows, and the
first rows, which gives their exact dq.

Tolerance (per element, per gradient tensor):
    |gpu - ref| <= tol * (rms(ref) + |ref| + rms(dO))
rms(dO), the size of the incoming gradient, is the floor for entries whose
exact value cancels to (near) zero. tol = 1e-3 for the fp32 path. For bf16,
tol = 5e-2, derived from the dominant error: D = dO . o reads the forward's
bf16 o, which is off by up to 2^-9 relative from storage plus the forward's
own rounding, so every ds of a row moves by p * dD with dD about
2^-8 * sqrt(d) * rms(dO) * rms(o); on rows whose exact ds cancel (a window of
one key) all of it shows against the floor, 2-4% at d = 64..128 and rms(o) ~ 1.
The affine gradients sum one such term per row, so their floor is
rms(dO) * sqrt(rows summed): B*T base rows, n_out output rows.
"""
import numpy as np
import pytest
import torch

from efficient_long_context_gb300 import workloads as W
from tests.parity_util import f32, record_margin, run_gpu_prefill

pytestmark = pytest.mark.gpu

GRAD_TOL = {torch.bfloat16: 5e-2, torch.float32: 1e-3}
NAMES = ("dq", "dk", "dv", "dq_out", "d_alpha_base", "d_beta_base", "d_alpha_out", "d_beta_out")


def run_gpu_backward(wl, do_base, do_out, fwd=None):
    import efficient_long_context_gb300 as ola

    dev = "cuda"
    if fwd is None:
        fwd = run_gpu_prefill(wl)
    o_b, l_b, o_o, l_o = fwd
    q, k, v = (wl[n].to(dev) for n in ("q", "k", "v"))
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    q_out = wl["q_out"].to(dev) if wl.get("q_out") is not None else None
    g = ola.orthros_prefill_backward(q, k, v, *aff, wl["out_indptr"], wl["out_positions"].to(dev), wl["window"],
                                     wl["scale"], o_b, l_b, o_o, l_o, do_base.to(dev), do_out.to(dev), q_out=q_out)
    torch.cuda.synchronize()
    return g


def run_oracle_backward(wl, do_base, do_out, row_range=None):
    import oracle

    q_out = f32(wl["q_out"]) if wl.get("q_out") is not None else None
    return oracle.prefill_backward(
        f32(wl["q"]), f32(wl["k"]), f32(wl["v"]), f32(wl["alpha_base"]), f32(wl["beta_base"]),
        f32(wl["alpha_out"]), f32(wl["beta_out"]), wl["out_indptr"].numpy(), wl["out_positions"].numpy(),
        wl["window"], wl["scale"], f32(do_base), f32(do_out), q_out=q_out, row_range=row_range)


def grad_err(gpu, ref, floor):
    """Largest |gpu - ref| / (rms(ref) + |ref| + floor) over the elements."""
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0
    assert np.all(np.isfinite(g)), "non-finite GPU gradient"
    rms = float(np.sqrt(np.mean(r * r)))
    return float(np.max(np.abs(g - r) / (rms + np.abs(r) + floor + 1e-30)))


def compare_backward(wl, gpu, ref, do_base, what="", select=None):
    """select: optional {name: index} restricting each compared tensor."""
    tol = GRAD_TOL[wl["dtype"]]
    floor = float(do_base.float().pow(2).mean().sqrt()) if do_base.numel() else 1.0
    n_out = int(wl["out_indptr"][-1])
    floors = {"d_alpha_base": floor * max(1, wl["B"] * wl["T"]) ** 0.5,
              "d_beta_base": floor * max(1, wl["B"] * wl["T"]) ** 0.5,
              "d_alpha_out": floor * max(1, n_out) ** 0.5,
              "d_beta_out": floor * max(1, n_out) ** 0.5}
    errs = {}
    for n in NAMES:
        if ref.get(n) is None:
            assert n != "dq_out" or gpu.get("dq_out") is None or wl.get("q_out") is None
            continue
        g, r = gpu[n], ref[n]
        if select and n in select:
            g, r = g[select[n]], r[select[n]]
        errs[n] = grad_err(g, r, floors.get(n, floor))
    bad = {n: e for n, e in errs.items() if e > tol}
    assert not bad, f"{what}: {errs}"
    print(f"[backward parity] {what}: " + ", ".join(f"{n} {e:.2e}" for n, e in errs.items()))
    return errs


SMALL = [
    # (B, T, Hq, Hkv, d, window, out_mode, dtype)
    (1, 1, 1, 1, 128, 1, "last", torch.bfloat16),
    (1, 100, 2, 1, 128, 64, "all", torch.bfloat16),
    (2, 333, 4, 4, 128, 63, ("span", 70), torch.bfloat16),
    (1, 333, 8, 2, 128, 65, "last", torch.bfloat16),
    (1, 300, 4, 1, 128, 128, ("list", [[0, 5, 127, 128, 128, 129, 299, 5]]), torch.bfloat16),
    (2, 257, 4, 2, 64, 256, "all", torch.bfloat16),
    (1, 300, 2, 2, 64, 1, "last", torch.bfloat16),
    (2, 333, 8, 2, 64, 65, ("span", 70), torch.bfloat16),
    (1, 300, 4, 1, 64, 128, ("list", [[0, 5, 127, 128, 128, 129, 299, 5]]), torch.bfloat16),
    (1, 300, 4, 2, 128, 307, ("list", [[]]), torch.bfloat16),
    (3, 129, 32, 8, 128, 64, ("list", [[128], [], [0, 64, 128]]), torch.bfloat16),
    (1, 200, 4, 2, 64, 50, "all", torch.float32),
    (2, 150, 2, 1, 128, 17, ("list", [[3, 3, 149], [0, 77]]), torch.float32),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}T{c[1]}h{c[2]}x{c[3]}d{c[4]}w{c[5]}{str(c[7])[6:]}")
@pytest.mark.parametrize("with_q_out", [False, True])
def test_backward_small(case, with_q_out):
    B, T, Hq, Hkv, d, w, mode, dt = case
    wl = W.small_prefill(B, T, Hq, Hkv, d, w, dtype=dt, out_mode=mode, seed=T + 3 * w, with_q_out=with_q_out)
    do_b, do_o = W.make_grad_outputs(wl, seed=T + w)
    gpu = run_gpu_backward(wl, do_b, do_o)
    ref = run_oracle_backward(wl, do_b, do_o)
    compare_backward(wl, gpu, ref, do_b, what=str(case))


@pytest.mark.parametrize("d", [128, 64])
def test_backward_many_tiles_per_key_block(d):
    """GQA 16/1 with every position an output row: the first key block visits
    16 x (3 band + 64 output-row) = 1072 query tiles on the tensor-core path
    (the tile list is generated while the tiles stream, with no cap)."""
    wl = W.small_prefill(1, 4096, 16, 1, d, 64, out_mode="all", seed=21)
    do_b, do_o = W.make_grad_outputs(wl, seed=22)
    compare_backward(wl, run_gpu_backward(wl, do_b, do_o), run_oracle_backward(wl, do_b, do_o), do_b,
                     what="1072 tiles per key block")


@pytest.mark.parametrize("d", [128, 64])
def test_backward_key_offsets(d):
    wl = W.small_prefill(1, 400, 8, 2, d, 100, out_mode=("span", 150), seed=9, k_offset_std=0.5)
    do_b, do_o = W.make_grad_outputs(wl, seed=4)
    compare_backward(wl, run_gpu_backward(wl, do_b, do_o), run_oracle_backward(wl, do_b, do_o), do_b,
                     what="offsets")


def _one_sequence(wl, b):
    """The workload restricted to sequence b (sequences are independent)."""
    ip = wl["out_indptr"]
    r0, r1 = int(ip[b]), int(ip[b + 1])
    one = dict(wl)
    for n in ("q", "k", "v"):
        one[n] = wl[n][b:b + 1].contiguous()
    one["out_indptr"] = torch.tensor([0, r1 - r0], dtype=torch.int32)
    one["out_positions"] = wl["out_positions"][r0:r1].contiguous()
    if wl.get("q_out") is not None:
        one["q_out"] = wl["q_out"][r0:r1].contiguous()
    one["B"] = 1
    return one, r0, r1


@pytest.mark.parametrize("work", [W.PT_2K, W.SFT_8K], ids=lambda x: x.name)
def test_backward_named_workload_sampled(work):
    """Full-size GPU backward (the benchmark's launch), checked on the last
    sequence: the last n_tail positions (their dq, and dk/dv of their keys)
    and the first 64 positions (their dq)."""
    wl = W.make_prefill(work)
    do_b, do_o = W.make_grad_outputs(wl, seed=work.seed + 7)
    gpu = run_gpu_backward(wl, do_b, do_o)
    b = wl["B"] - 1
    one, r0, r1 = _one_sequence(wl, b)
    do_b1 = do_b[b:b + 1].contiguous()
    do_o1 = do_o[r0:r1].contiguous()
    g1 = {n: (gpu[n][b:b + 1] if n in ("dq", "dk", "dv") else gpu[n]) for n in ("dq", "dk", "dv")}
    T = work.T
    n_tail = 96
    tail = run_oracle_backward(one, do_b1, do_o1, row_range=(T - n_tail, T))
    sl = (slice(None), slice(T - n_tail, T))
    errs = compare_backward(one, g1, {n: tail[n] for n in ("dq", "dk", "dv")}, do_b1, what=f"{work.name} tail",
                            select={"dq": sl, "dk": sl, "dv": sl})
    head = run_oracle_backward(one, do_b1, do_o1, row_range=(0, 64))
    errs.update(compare_backward(one, {"dq": g1["dq"]}, {"dq": head["dq"]}, do_b1, what=f"{work.name} head",
                                 select={"dq": (slice(None), slice(0, 64))}))
    assert errs
    record_margin(f"{work.name} backward", errs, {n: GRAD_TOL[work.dtype] for n in errs},
                  "largest |gpu - ref| / (rms(ref) + |ref| + floor) on the last sequence's last 96 and first 64 rows")


@pytest.mark.parametrize("work", [W.PT_2K, W.SFT_8K], ids=lambda x: x.name)
def test_backward_one_full_sequence_every_gradient(work):
    """One whole sequence of a training workload (its full length, all of its
    output rows) through the GPU backward, against the oracle's full backward
    of it: every gradient, the affine gradients summed over all its rows
    included."""
    wl = W.make_prefill(work)
    do_b, do_o = W.make_grad_outputs(wl, seed=work.seed + 7)
    one, r0, r1 = _one_sequence(wl, wl["B"] - 1)
    do_b1 = do_b[wl["B"] - 1:].contiguous()
    do_o1 = do_o[r0:r1].contiguous()
    gpu = run_gpu_backward(one, do_b1, do_o1)
    ref = run_oracle_backward(one, do_b1, do_o1)
    errs = compare_backward(one, gpu, ref, do_b1, what=f"{work.name} one sequence")
    record_margin(f"{work.name} backward, one full sequence", errs, {n: GRAD_TOL[work.dtype] for n in errs},
                  "largest |gpu - ref| / (rms(ref) + |ref| + floor), every row of one sequence")
