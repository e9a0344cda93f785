"""GPU parity of orthros_decode against the CPU oracle over several steps.

Each step appends one token per sequence and runs the base (windowed) and
output (full-history) queries; the cache state carries over between steps,
so later steps also check the earlier appends.
"""
import os

import numpy as np
import pytest
import torch

import efficient_long_context_gb300 as ola
from efficient_long_context_gb300 import workloads as W
from tests.parity_util import TOL, f32, max_err, record_margin

pytestmark = pytest.mark.gpu


def _sub_state(st, seqs):
    """The sampled sequences' pages as a compact float32 pool for the oracle."""
    bt = st.block_table[seqs].numpy()
    used = np.unique(bt[bt >= 0])
    remap = np.full(st.k_cache.shape[0], -1, np.int64)
    remap[used] = np.arange(len(used))
    bt_c = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    kc = f32(st.k_cache[torch.as_tensor(used)])
    vc = f32(st.v_cache[torch.as_tensor(used)])
    return kc, vc, bt_c


def run_and_compare(st, steps, seqs=None, what=""):
    import oracle

    m = st.meta
    dev = "cuda"
    kc = st.k_cache.to(dev)
    vc = st.v_cache.to(dev)
    bt = st.block_table.to(dev)
    lens = st.cache_lens.to(dev)
    B = m["B"]
    seqs = np.arange(B) if seqs is None else np.asarray(seqs)
    okc, ovc, obt = _sub_state(st, seqs)
    olens = st.cache_lens.numpy()[seqs].copy()
    aff = [st.alpha_base, st.beta_base, st.alpha_out, st.beta_out]
    aff_d = [a.to(dev) for a in aff]
    ws = torch.empty(ola.orthros_decode_workspace_size(B, m["Hq"], m["Hkv"], m["d"], m["max_pages"],
                                                       m["page_size"], m["dtype"]), dtype=torch.uint8,
                     device=dev)
    tol_o, tol_l = TOL[m["dtype"]]
    worst = {}
    for s in range(steps):
        q = st.q[s].to(dev)
        qo = st.q_out[s].to(dev) if st.q_out is not None else None
        out = ola.orthros_decode(q, st.k_new[s].to(dev), st.v_new[s].to(dev), kc, vc, bt, lens, *aff_d,
                                 m["window"], m["scale"], q_out=qo, workspace=ws)
        rc, bits = ola.orthros_check(ws)
        assert rc == 0 and bits == 0, (rc, bits)
        lens += 1
        ref = oracle.decode(f32(st.q[s][seqs]), f32(st.k_new[s][seqs]), f32(st.v_new[s][seqs]), okc, ovc,
                            obt, olens, *(f32(a) for a in aff), m["window"], m["scale"],
                            q_out=None if st.q_out is None else f32(st.q_out[s][seqs]))
        olens += 1
        idx = torch.as_tensor(seqs, device=dev)
        errs = [max_err(g.index_select(0, idx), r) for g, r in zip(out, ref)]
        for name, e in zip(("o_base", "lse_base", "o_out", "lse_out"), errs):
            worst[name] = max(worst.get(name, 0.0), e)
        assert errs[0] <= tol_o and errs[2] <= tol_o, f"{what} step {s} {errs}"
        assert errs[1] <= tol_l and errs[3] <= tol_l, f"{what} step {s} {errs}"
    # the appended keys landed in the right slots
    torch.cuda.synchronize()
    return worst


SMALL = [
    # (B, Hq, Hkv, d, window, page_size, lens, dtype, steps, q_out)
    (3, 4, 2, 128, 16, 16, [0, 5, 100], torch.bfloat16, 4, False),
    (4, 32, 8, 128, 64, 64, [1, 63, 64, 1000], torch.bfloat16, 3, True),
    (2, 8, 8, 64, 1, 64, [10, 300], torch.bfloat16, 2, False),
    (2, 4, 1, 128, 5000, 64, [2000, 4500], torch.bfloat16, 2, True),
    (5, 8, 2, 128, 128, 32, [0, 127, 128, 129, 3000], torch.bfloat16, 3, False),
    (2, 4, 2, 64, 30, 16, [7, 400], torch.float32, 3, True),
    # GQA groups of 9-16 query heads (e.g. 64/4): base and output rows in separate groups on the TMA path
    (3, 32, 2, 128, 300, 64, [5, 700, 5000], torch.bfloat16, 3, True),
    (2, 24, 2, 128, 64, 128, [129, 2000], torch.bfloat16, 2, False),
    (2, 64, 4, 128, 4096, 64, [10000, 20000], torch.bfloat16, 2, False),
    (1, 2, 2, 128, 100, 64, [0], torch.float32, 2, False),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}h{c[1]}x{c[2]}d{c[3]}w{c[4]}p{c[5]}{str(c[7])[6:]}")
def test_small_decode(case):
    B, Hq, Hkv, d, w, P, lens, dt, steps, with_qo = case
    wl = W.DecodeWorkload("small", B, Hq, Hkv, d, w, P, 0, 0, steps, dtype=dt, seed=sum(lens) + w)
    st = W.make_decode(wl, lens=lens, with_q_out=with_qo)
    run_and_compare(st, steps, what=str(case))


def test_decode_workload_sampled():
    """The 32-sequence paged decoding workload at full size over all of its
    128 steps (every append, including those that open fresh pages), checked
    on a sample of sequences (shortest, longest and two random)."""
    steps = W.DECODE_32.steps
    st = W.make_decode(W.DECODE_32, steps=steps)
    lens = st.cache_lens.numpy()
    r = np.random.default_rng(1)
    seqs = sorted({int(np.argmin(lens)), int(np.argmax(lens)), *map(int, r.choice(len(lens), 2, replace=False))})
    worst = run_and_compare(st, steps, seqs=seqs, what="decode workload")
    tol_o, tol_l = TOL[torch.bfloat16]
    record_margin(W.DECODE_32.name, worst, {"o_base": tol_o, "lse_base": tol_l, "o_out": tol_o, "lse_out": tol_l},
                  f"max abs error vs the oracle over {steps} steps of {len(seqs)} sampled sequences")


@pytest.mark.skipif(os.environ.get("ORTHROS_FULL_PARITY") != "1",
                    reason="about a minute of oracle time; set ORTHROS_FULL_PARITY=1")
def test_decode_workload_every_sequence():
    """The 32-sequence decoding workload over all 128 steps, every sequence
    compared with the oracle (413 GB of cache reads in the oracle)."""
    steps = W.DECODE_32.steps
    st = W.make_decode(W.DECODE_32, steps=steps)
    worst = run_and_compare(st, steps, what="decode workload, every sequence")
    tol_o, tol_l = TOL[torch.bfloat16]
    record_margin(W.DECODE_32.name + ", every sequence", worst,
                  {"o_base": tol_o, "lse_base": tol_l, "o_out": tol_o, "lse_out": tol_l},
                  f"max abs error vs the oracle over {steps} steps of all 32 sequences")


def test_decode_steps_replayed_from_a_cuda_graph():
    """Several decoding steps captured once in a CUDA graph (a serving loop's
    form: no host work per step) and replayed give the oracle's results; the
    call does nothing on the host that capture forbids."""
    import oracle

    wl = W.DecodeWorkload("graph", 3, 8, 2, 128, 64, 64, 0, 0, 3, seed=12)
    st = W.make_decode(wl, lens=[5, 70, 300])
    m = st.meta
    dev = "cuda"
    kc0, vc0 = st.k_cache.to(dev), st.v_cache.to(dev)
    kc, vc = kc0.clone(), vc0.clone()
    bt = st.block_table.to(dev)
    steps = 3
    lens = (st.cache_lens[None, :].long() + torch.arange(steps)[:, None]).to(torch.int32).to(dev)
    aff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    q, kn, vn = st.q.to(dev), st.k_new.to(dev), st.v_new.to(dev)
    ws = torch.empty(ola.orthros_decode_workspace_size(3, 8, 2, 128, m["max_pages"], m["page_size"]),
                     dtype=torch.uint8, device=dev)
    outs = [(torch.empty_like(q[0]), torch.empty((3, 8), dtype=torch.float32, device=dev), torch.empty_like(q[0]),
             torch.empty((3, 8), dtype=torch.float32, device=dev)) for _ in range(steps)]
    # warm up outside capture (first calls set kernel attributes), then restore the cache
    ola.orthros_decode(q[0], kn[0], vn[0], kc, vc, bt, lens[0], *aff, wl.window, wl.scale, out=outs[0], workspace=ws)
    torch.cuda.synchronize()
    kc.copy_(kc0)
    vc.copy_(vc0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for s in range(steps):
            ola.orthros_decode(q[s], kn[s], vn[s], kc, vc, bt, lens[s], *aff, wl.window, wl.scale, out=outs[s],
                               workspace=ws)
    kc.copy_(kc0)  # capture ran nothing; start from the initial cache anyway
    vc.copy_(vc0)
    g.replay()
    torch.cuda.synchronize()
    assert ola.orthros_check(ws) == (0, 0)
    okc, ovc = f32(st.k_cache).copy(), f32(st.v_cache).copy()
    olens = st.cache_lens.numpy().copy()
    tol_o, tol_l = TOL[torch.bfloat16]
    for s in range(steps):
        ref = oracle.decode(f32(st.q[s]), f32(st.k_new[s]), f32(st.v_new[s]), okc, ovc, st.block_table.numpy(),
                            olens, *(f32(a) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)),
                            wl.window, wl.scale)
        olens += 1
        errs = [max_err(gg, r) for gg, r in zip(outs[s], ref)]
        assert errs[0] <= tol_o and errs[2] <= tol_o and errs[1] <= tol_l and errs[3] <= tol_l, (s, errs)
