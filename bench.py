#!/usr/bin/env python
"""Benchmark of the Orthros attention hot path on GB300.

Prints ONE JSON line (rank 0). The headline `value` is prefill attention
throughput (TFLOP/s of useful work: in-band query-key pairs of the base
stream plus the output rows' causal pairs, 4*d FLOP per pair and head) on a
128K-token prefill at the Llama-3.1-8B attention shape (GQA 32/8, d = 128,
window 4096, one output row at the last prompt token), through
orthros_prefill with inputs resident in HBM. The same line carries the
decoding throughput (KV-cache GB/s, every cached K/V byte counted once per
step) of 32 paged sequences with 16K-32K cached tokens over 128 steps.

A step = one orthros_prefill call: K/V cache fill, the fp16 key pre-pass,
the banded base-stream kernel, the output row(s), and their combine.

--impl reference runs the CPU oracle instead (the reference arm of this
repository: a deliberately plain program, timed on a bounded sample).
Multi-GPU: every rank runs its own replica of the workload (the work shards by
sequence and head with no exchange); value sums all ranks' work over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & decode KV GB/s (Llama-8B shape, 128K) vs roofline"


# ----------------------------------------------------------------------------
# work accounting (useful FLOPs / algorithmic bytes)
# ----------------------------------------------------------------------------
def band_pairs(T: int, w: int) -> int:
    """Query-key pairs of the sliding-window stream for one (sequence, head)."""
    if w >= T:
        return T * (T + 1) // 2
    return w * (w + 1) // 2 + (T - w) * w


def prefill_flops(wl, positions_per_seq) -> dict:
    """Useful FLOPs: 2*d for q.k plus 2*d for p*v per pair and query head."""
    per_pair = 4 * wl.d * wl.Hq * wl.B
    swa = band_pairs(wl.T, wl.window) * per_pair
    cross = sum(t + 1 for t in positions_per_seq) * 4 * wl.d * wl.Hq
    return dict(swa=swa, cross=cross, total=swa + cross)


def decode_bytes(lens0, steps, Hkv, d, elem=2) -> int:
    """Each cached K and V element read once per step (cache after the append)."""
    tot = 0
    for s in range(steps):
        tot += sum(int(L) + s + 1 for L in lens0) * Hkv * d * elem * 2
    return tot


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------
# distributed plumbing (replicas; torch.distributed only for barrier + max)
# ----------------------------------------------------------------------------
class Dist:
    """Replica bookkeeping: rank/world from the torchrun environment, a barrier,
    and the max over ranks (NCCL on GPUs; gloo where there is no GPU)."""

    def __init__(self, enable: bool, backend: str = "nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.backend = backend
        self.pg = None
        if self.world > 1 and enable:
            import torch
            import torch.distributed as dist

            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self.backend == "nccl" else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def whole_job_rate(work_per_rank: float, ms_local: float, dist) -> tuple[float, float]:
    """Weak scaling: every rank does the same work; the job's rate is all ranks'
    work over the slowest rank's time. Returns (rate per second, max ms)."""
    ms = dist.max(ms_local)
    return work_per_rank * dist.world / (ms * 1e-3), ms


def captured_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source has changed since that capture."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        ent = json.load(f).get(key)
    if not ent:
        return None
    with open(os.path.join(ROOT, ent["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != ent["sha256_16"]:
            return None
    return ent["bytes_per_launch"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d.get("bf16_tflops_sustained"),
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------
def oracle_sample(wl_inputs, wl, target_s: float, seed: int = 0):
    """Time the oracle on base rows of the prefill workload (full windows),
    growing the sample until it takes about target_s seconds. Returns
    (TFLOP/s, threads, description)."""
    import numpy as np

    import oracle

    f32 = wl_inputs.get("_f32")
    if f32 is None:  # widen once per workload (exact for bf16)
        f32 = {n: wl_inputs[n].float().numpy() for n in ("q", "k", "v", "alpha_base", "beta_base", "alpha_out",
                                                         "beta_out")}
        wl_inputs["_f32"] = f32
    nthreads = len(os.sched_getaffinity(0))
    empty_indptr = np.zeros(wl.B + 1, np.int32)
    empty_pos = np.zeros(0, np.int32)
    rng = np.random.default_rng(seed)
    n = 1
    while True:
        rows = np.sort(rng.choice(np.arange(wl.window, wl.T), size=n, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill(f32["q"], f32["k"], f32["v"], f32["alpha_base"], f32["beta_base"], f32["alpha_out"],
                       f32["beta_out"], empty_indptr, empty_pos, wl.window, wl.scale, base_rows=rows,
                       nthreads=nthreads)
        dt = time.perf_counter() - t0
        flops = n * wl.B * wl.Hq * wl.window * 4 * wl.d
        if dt >= target_s or n >= wl.T - wl.window:
            break
        n = min(wl.T - wl.window, max(n * 2, int(n * target_s / max(dt, 1e-3) * 1.05)))
    desc = (f"{n} base rows x {wl.Hq} heads with full {wl.window}-key windows of the {wl.T}-token prefill "
            f"({flops / 1e9:.1f} GFLOP useful, {dt:.1f} s)")
    return flops / dt / 1e12, nthreads, desc


def oracle_prefill_sample(inputs, wl, target_s: float, seed: int = 0):
    """Time the oracle on a sample of the workload's own rows: random base
    positions of every sequence (their true windows) and random output rows
    (their whole causal prefix), growing the sample until it takes about
    target_s seconds. Returns (TFLOP/s of the sampled rows' useful work,
    threads, description)."""
    import numpy as np

    import oracle

    f32 = inputs.get("_f32")
    if f32 is None:
        f32 = {n: inputs[n].float().numpy() for n in ("q", "k", "v", "alpha_base", "beta_base", "alpha_out",
                                                      "beta_out")}
        inputs["_f32"] = f32
    nthreads = len(os.sched_getaffinity(0))
    indptr = inputs["out_indptr"].numpy().astype(np.int64)
    pos = inputs["out_positions"].numpy()
    n_out = int(indptr[-1])
    rng = np.random.default_rng(seed)
    n = 1
    while True:
        rows = np.sort(rng.choice(wl.T, size=min(n, wl.T), replace=False)).astype(np.int32)
        orow = np.sort(rng.choice(n_out, size=min(n, n_out), replace=False)) if n_out else np.zeros(0, np.int64)
        seq = np.searchsorted(indptr, orow, side="right") - 1
        s_indptr = np.concatenate([[0], np.cumsum(np.bincount(seq, minlength=wl.B))]).astype(np.int32)
        s_pos = pos[orow].astype(np.int32)
        t0 = time.perf_counter()
        oracle.prefill(f32["q"], f32["k"], f32["v"], f32["alpha_base"], f32["beta_base"], f32["alpha_out"],
                       f32["beta_out"], s_indptr, s_pos, wl.window, wl.scale, base_rows=rows, nthreads=nthreads)
        dt = time.perf_counter() - t0
        pairs = wl.B * int(np.minimum(rows.astype(np.int64) + 1, wl.window).sum()) + int((s_pos.astype(np.int64) + 1).sum())
        flops = pairs * 4 * wl.d * wl.Hq
        if dt >= target_s or (n >= wl.T and n >= n_out):
            break
        n = max(n * 2, int(n * target_s / max(dt, 1e-3) * 1.05))
    desc = (f"{len(rows)} base positions of each of {wl.B} sequences and {len(orow)} output rows of the "
            f"{wl.name} workload ({flops / 1e9:.1f} GFLOP useful, {dt:.1f} s)")
    return flops / dt / 1e12, nthreads, desc


def oracle_decode_sample(st, target_s: float, n_seq: int = 4):
    """Time the oracle on decoding steps of the first n_seq sequences of the
    decoding workload (their caches copied to a compact float pool), repeating
    steps until about target_s seconds. Returns (GB/s of algorithmic cache
    bytes, threads, description)."""
    import numpy as np

    import oracle

    nthreads = len(os.sched_getaffinity(0))
    seqs = np.arange(min(n_seq, st.meta["B"]))
    bt = st.block_table[seqs].numpy()
    used = np.unique(bt[bt >= 0])
    remap = np.full(st.k_cache.shape[0], -1, np.int64)
    remap[used] = np.arange(len(used))
    obt = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
    import torch

    okc = st.k_cache[torch.as_tensor(used)].float().numpy()
    ovc = st.v_cache[torch.as_tensor(used)].float().numpy()
    lens = st.cache_lens.numpy()[seqs].astype(np.int32).copy()
    aff = [a.float().numpy() for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    m = st.meta
    nbytes, steps, t_all = 0, 0, 0.0
    while t_all < target_s and steps < m["steps"]:
        t0 = time.perf_counter()
        oracle.decode(st.q[steps][seqs].float().numpy(), st.k_new[steps][seqs].float().numpy(),
                      st.v_new[steps][seqs].float().numpy(), okc, ovc, obt, lens, *aff, m["window"], m["scale"],
                      nthreads=nthreads)
        t_all += time.perf_counter() - t0
        nbytes += int((lens.astype(np.int64) + 1).sum()) * m["Hkv"] * m["d"] * 2 * 2
        lens += 1
        steps += 1
    desc = (f"{steps} decoding steps of {len(seqs)} of the {m['B']} sequences ({nbytes / 1e9:.2f} GB of cache "
            f"read, {t_all:.1f} s)")
    return nbytes / t_all / 1e9, nthreads, desc


def run_reference(args, dist):
    """The reference arm: the CPU oracle as it stands, same metric and config."""
    if dist.rank != 0:
        return
    from efficient_long_context_gb300 import workloads as W

    import oracle

    oracle.build()
    wl = W.PREFILL_128K
    inputs = W.make_prefill(wl)
    per_step_s = float(os.environ.get("ORTHROS_REF_STEP_S", "4"))
    vals = []
    for _ in range(args.warmup):
        oracle_sample(inputs, wl, per_step_s / 4)
    desc = cores = None
    t_all = time.perf_counter()
    for s in range(args.steps):
        v, cores, desc = oracle_sample(inputs, wl, per_step_s, seed=s)
        vals.append(v)
    elapsed = time.perf_counter() - t_all
    value = statistics.mean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs of the 128K prefill workload)",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                       "window": wl.window, "out_rows": "last position"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------
def _timed(ola, torch, dist, stream, fn, steps):
    """Run fn(i) for i < steps between two CUDA events on `stream`, with the
    library's per-kernel event profiling on. Returns (max-over-ranks ms, profile)."""
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ola.orthros_profile_begin()
    ev0.record(stream)
    for i in range(steps):
        fn(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    prof = ola.orthros_profile_end()
    dist.barrier()
    return dist.max(ev0.elapsed_time(ev1)), prof


def headline_workload(args, W):
    wl = {"128k": W.PREFILL_128K, "pt": W.PT_2K, "sft": W.SFT_8K}[args.prefill_workload]
    if args.prefill_T:
        import dataclasses

        wl = dataclasses.replace(wl, T=args.prefill_T, name=f"{wl.name}@T{args.prefill_T}")
    return wl


def bench_prefill(args, dist, dev, stream, peaks, ola, torch, W, wl, e2e=False):
    inputs = W.make_prefill(wl)
    q, k, v = (inputs[n].to(dev) for n in ("q", "k", "v"))
    aff = [inputs[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    indptr = inputs["out_indptr"]
    pos = inputs["out_positions"].to(dev)
    n_out = int(indptr[-1])
    P = 64
    max_pages = (wl.T + P - 1) // P
    num_pages = wl.B * max_pages
    k_cache = torch.empty((num_pages, P, wl.Hkv, wl.d), dtype=wl.dtype, device=dev)
    v_cache = torch.empty_like(k_cache)
    block_table = torch.arange(num_pages, dtype=torch.int32, device=dev).view(wl.B, max_pages)
    outs = (torch.empty_like(q), torch.empty((wl.B, wl.Hq, wl.T), dtype=torch.float32, device=dev),
            torch.empty((n_out, wl.Hq, wl.d), dtype=wl.dtype, device=dev),
            torch.empty((n_out, wl.Hq), dtype=torch.float32, device=dev))
    ws = torch.empty(ola.orthros_prefill_workspace_size(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, n_out, wl.window,
                                                        wl.dtype), dtype=torch.uint8, device=dev)

    # training-shape workloads fit in L2: a buffer twice its size is rewritten before each step
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if in_bytes < 2 * l2_bytes else None

    def step(_=0):
        if flush is not None:
            flush.fill_(1)
        ola.orthros_prefill(q, k, v, *aff, indptr, pos, wl.window, wl.scale, out=outs, k_cache=k_cache,
                            v_cache=v_cache, block_table=block_table, page_size=P, workspace=ws, stream=stream)

    positions = [int(t) for t in inputs["out_positions"]]
    flops = prefill_flops(wl, positions)
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, bits = ola.orthros_check(ws)
    if rc != 0:
        raise RuntimeError(f"prefill flagged device status {rc} bits 0x{bits:x}")
    ms, prof = _timed(ola, torch, dist, stream, step, args.steps)
    ms_step = ms / args.steps  # already the max over ranks
    # dominant kernel and the useful FLOPs it alone performs: the base stream,
    # plus output rows of sequences dense enough to go to the tile kernel
    dom, (dom_n, dom_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    g = wl.Hq // wl.Hkv
    per_seq = [positions[int(indptr[b]):int(indptr[b + 1])] for b in range(wl.B)]
    tile_cross = sum(sum(t + 1 for t in ps) for ps in per_seq if len(ps) * g > 256) * 4 * wl.d * wl.Hq
    dom_flops = flops["swa"] + tile_cross if dom == "prefill_tc" else flops["total"]
    achieved = dom_flops / (dom_ms / dom_n * 1e-3) / 1e12
    res = dict(wl=wl, inputs=inputs, flops=flops, ms_step=ms_step, prof=prof, P=P,
               l2=(f"L2 flushed before each step ({2 * l2_bytes >> 20} MiB written, inside the step time)"
                   if flush is not None else "inputs larger than L2; no flush"),
               value=flops["total"] * dist.world / (ms_step * 1e-3) / 1e12,
               roofline={"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["bf16"],
                         "traffic": captured_traffic({W.PREFILL_128K.name: "prefill_tc", W.PT_2K.name: "prefill_tc_pt",
                                                      W.SFT_8K.name: "prefill_tc_sft"}.get(wl.name, ""))
                         if dom == "prefill_tc" else None,
                         "peak_source": f"{peaks['src']} bf16 dense (burst)", "avg_launch_ms": dom_ms / dom_n,
                         "useful_tflop_per_launch": dom_flops / 1e12})
    if e2e:
        # end to end through orthros_prefill_from_host: pinned host buffers in
        # and out, the copies inside the timed region (chunked, overlapping the
        # compute on the library's copy streams), the same cache fill
        h_in = {n: inputs[n].pin_memory() for n in ("q", "k", "v")}
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        h_pos = inputs["out_positions"].to(torch.int32).contiguous()
        ws_fh = torch.empty(ola.orthros_prefill_from_host_workspace_size(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, n_out,
                                                                         wl.window, wl.dtype),
                            dtype=torch.uint8, device=dev)

        def e2e_step(_):
            ola.orthros_prefill_from_host(h_in["q"], h_in["k"], h_in["v"], *aff, indptr, h_pos, wl.window, wl.scale,
                                          out=h_out, k_cache=k_cache, v_cache=v_cache, block_table=block_table,
                                          page_size=P, workspace=ws_fh, stream=stream)

        e2e_steps = max(1, min(args.steps, 3))
        e2e_step(0)
        torch.cuda.synchronize()
        rc, bits = ola.orthros_check(ws_fh)
        if rc != 0:
            raise RuntimeError(f"prefill from host flagged device status {rc} bits 0x{bits:x}")
        ms_e2e, prof_e2e = _timed(ola, torch, dist, stream, e2e_step, e2e_steps)
        ms_e2e /= e2e_steps
        # bytes copied per step: q, k, v, the output rows' queries and positions in; every output out
        qrow = wl.Hq * wl.d * q.element_size()
        h2d = sum(t.numel() * t.element_size() for t in h_in.values()) + n_out * (qrow + 4)
        res["e2e"] = {"value": flops["total"] * dist.world / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in h_out),
                      "ms_per_step": ms_e2e, "steps": e2e_steps, "api": "orthros_prefill_from_host",
                      "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in prof_e2e.items()}}
    return res


def bench_decode(args, dist, dev, stream, peaks, ola, torch, W):
    import dataclasses

    dec = W.DECODE_32
    if args.decode_B:
        dec = dataclasses.replace(dec, B=args.decode_B, name=f"{dec.name}@B{args.decode_B}")
    st = W.make_decode(dec, steps=args.decode_steps)
    dm = st.meta
    kc, vc = st.k_cache.to(dev), st.v_cache.to(dev)
    bt = st.block_table.to(dev)
    lens_steps = (st.cache_lens[None, :].to(torch.int64) + torch.arange(dm["steps"])[:, None]).to(torch.int32).to(dev)
    dq, dk, dv = st.q.to(dev), st.k_new.to(dev), st.v_new.to(dev)
    daff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    outs = (torch.empty((dec.B, dec.Hq, dec.d), dtype=dec.dtype, device=dev),
            torch.empty((dec.B, dec.Hq), dtype=torch.float32, device=dev),
            torch.empty((dec.B, dec.Hq, dec.d), dtype=dec.dtype, device=dev),
            torch.empty((dec.B, dec.Hq), dtype=torch.float32, device=dev))
    ws = torch.empty(ola.orthros_decode_workspace_size(dec.B, dec.Hq, dec.Hkv, dec.d, dm["max_pages"], dec.page_size,
                                                       dec.dtype), dtype=torch.uint8, device=dev)

    def step(s, strm=stream):
        ola.orthros_decode(dq[s], dk[s], dv[s], kc, vc, bt, lens_steps[s], *daff, dec.window, dec.scale,
                           out=outs, workspace=ws, stream=strm)

    for s in range(min(max(args.warmup, 3), dm["steps"])):
        step(s)
    torch.cuda.synchronize()
    rc, bits = ola.orthros_check(ws)
    if rc != 0:
        raise RuntimeError(f"decode flagged device status {rc} bits 0x{bits:x}")
    ms, prof = _timed(ola, torch, dist, stream, step, dm["steps"])
    nbytes = decode_bytes(st.cache_lens.tolist(), dm["steps"], dec.Hkv, dec.d)
    # the same steps captured once in a CUDA graph and replayed (no host work or
    # launch gaps between steps, as in a captured serving loop)
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for s in range(dm["steps"]):
                step(s, None)  # the capture stream
        torch.cuda.synchronize()
        g.replay()  # warm
        dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms_g = dist.max(e0.elapsed_time(e1))
        graph = {"ms_per_step": ms_g / dm["steps"], "value": nbytes * dist.world / (ms_g * 1e-3) / 1e9,
                 "unit": "GB/s", "frac_of_hbm": nbytes / (ms_g * 1e-3) / 1e9 / peaks["hbm"]}
        del g
    except RuntimeError as exc:  # capture is optional for the measurement
        graph = {"error": str(exc)[:200]}
    gbs = nbytes * dist.world / (ms * 1e-3) / 1e9
    dom, (dom_n, dom_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    achieved = nbytes / (dom_ms * 1e-3) / 1e9  # bytes of all steps over that kernel's summed time
    # end to end through the public call: every step's inputs (queries, new
    # keys/values, lengths) copied from pinned host memory and its outputs read
    # back, inside the timed region; the cache stays resident as serving state
    e2e = None
    if args.only == "all":
        h_in = [t.pin_memory() for t in (st.q, st.k_new, st.v_new)]
        h_lens = lens_steps.cpu().pin_memory()
        d_in = [torch.empty_like(dq[0]), torch.empty_like(dk[0]), torch.empty_like(dv[0])]
        d_len = torch.empty_like(lens_steps[0])
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]

        def e2e_step(s):
            for hb, db in zip(h_in, d_in):
                db.copy_(hb[s], non_blocking=True)
            d_len.copy_(h_lens[s], non_blocking=True)
            ola.orthros_decode(d_in[0], d_in[1], d_in[2], kc, vc, bt, d_len, *daff, dec.window, dec.scale, out=outs,
                               workspace=ws, stream=stream)
            for hb, db in zip(h_out, outs):
                hb.copy_(db, non_blocking=True)

        ms_e2e, _ = _timed(ola, torch, dist, stream, e2e_step, dm["steps"])
        e2e = {"value": nbytes * dist.world / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": sum(t[0].numel() * t.element_size() for t in h_in) + h_lens[0].numel() * 4,
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in h_out),
               "ms_per_step": ms_e2e / dm["steps"], "steps": dm["steps"]}
    return {"value": gbs, "unit": "GB/s", "workload": dec.name, "steps": dm["steps"], "ms_per_step": ms / dm["steps"],
            "bytes": nbytes, "frac_of_hbm": gbs / peaks["hbm"],
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm"],
                         "traffic": captured_traffic("splitkv_decode") if dom == "splitkv_decode" and dec.B == 32 else None,
                         "peak_source": f"{peaks['src']} HBM copy",
                         "avg_launch_ms": dom_ms / dom_n, "bytes_per_launch": nbytes / dm["steps"]},
            "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in prof.items()},
            "gpu_launches": sum(n for n, _ in prof.values()),
            "graph_replay": graph, "e2e": e2e, "_state": st}


def bench_backward(args, dist, dev, stream, peaks, ola, torch, W):
    """Backward of the fine-tuning workload (Llama-8B attention shape, 8K,
    answer span of 1024 output rows): one forward for o and lse, then K timed
    calls of orthros_prefill_backward. Algorithmic FLOPs: 5 products of 2d per
    useful (query, key) pair, i.e. 2.5x the forward's 4d."""
    wl = W.SFT_8K
    inputs = W.make_prefill(wl)
    q, k, v = (inputs[n].to(dev) for n in ("q", "k", "v"))
    aff = [inputs[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    indptr = inputs["out_indptr"]
    pos = inputs["out_positions"].to(dev)
    n_out = int(indptr[-1])
    fwd = ola.orthros_prefill(q, k, v, *aff, indptr, pos, wl.window, wl.scale, stream=stream)
    do_b, do_o = (t.to(dev) for t in W.make_grad_outputs(inputs, seed=wl.seed + 7))
    ws = torch.empty(ola.orthros_prefill_backward_workspace_size(wl.B, wl.T, wl.Hq, wl.Hkv, wl.d, n_out, wl.window,
                                                                 wl.dtype), dtype=torch.uint8, device=dev)
    grads = None

    def step(_=0):
        nonlocal grads
        grads = ola.orthros_prefill_backward(q, k, v, *aff, indptr, pos, wl.window, wl.scale, *fwd, do_b, do_o,
                                             out=grads, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, bits = ola.orthros_check(ws)
    if rc != 0:
        raise RuntimeError(f"backward flagged device status {rc} bits 0x{bits:x}")
    steps = args.steps
    ms, prof = _timed(ola, torch, dist, stream, step, steps)
    positions = [int(t) for t in inputs["out_positions"]]
    fwd_flops = prefill_flops(wl, positions)
    flops = 2.5 * fwd_flops["total"]
    dom, (dom_n, dom_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    achieved = flops / (dom_ms / dom_n * 1e-3) / 1e12
    return {"value": flops * dist.world / (ms / steps * 1e-3) / 1e12, "unit": "TFLOP/s", "workload": wl.name,
            "steps": steps, "ms_per_step": ms / steps, "useful_tflop_per_step": flops / 1e12,
            "flop_model": "10 d per useful (query, key) pair: recomputed S, dP, dV, dK, dQ",
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peaks["bf16"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["bf16"],
                         "traffic": captured_traffic("bwd_tc") if dom == "bwd_tc" else None,
                         "peak_source": f"{peaks['src']} bf16 dense (burst)", "avg_launch_ms": dom_ms / dom_n,
                         "useful_tflop_per_launch": flops / 1e12},
            "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in prof.items()},
            "gpu_launches": sum(n for n, _ in prof.values())}


def bench_extend(args, dist, dev, stream, peaks, ola, torch, W):
    """A continuous-batching step (MIXED_32: 28 sequences decode one token, 4
    append a 16-token prefill chunk, 16K-32K cached tokens each), timed over K
    calls with the same inputs. Algorithmic bytes: every sequence's cached K
    and V (L_b + n_b tokens) read once per step."""
    wl = W.make_extend(W.MIXED_32)
    w = W.MIXED_32
    kc, vc = wl["k_cache"].to(dev), wl["v_cache"].to(dev)
    bt, lens = wl["block_table"].to(dev), wl["cache_lens"].to(dev)
    q, kn, vn = (wl[n].to(dev) for n in ("q", "k_new", "v_new"))
    pos = wl["out_positions"].to(dev)
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    n_new, n_out = int(wl["new_indptr"][-1]), int(wl["out_indptr"][-1])
    outs = (torch.empty_like(q), torch.empty((n_new, w.Hq), dtype=torch.float32, device=dev),
            torch.empty((n_out, w.Hq, w.d), dtype=w.dtype, device=dev),
            torch.empty((n_out, w.Hq), dtype=torch.float32, device=dev))
    ws = torch.empty(ola.orthros_extend_workspace_size(w.B, n_new, n_out, w.Hq, w.Hkv, w.d, wl["max_pages"],
                                                       w.page_size, w.dtype), dtype=torch.uint8, device=dev)

    def step(_=0):
        ola.orthros_extend(q, kn, vn, kc, vc, bt, lens, wl["new_indptr"], wl["out_indptr"], pos, *aff, w.window,
                           w.scale, out=outs, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    rc, bits = ola.orthros_check(ws)
    if rc != 0:
        raise RuntimeError(f"extend flagged device status {rc} bits 0x{bits:x}")
    steps = max(args.steps, 20)
    ms, prof = _timed(ola, torch, dist, stream, step, steps)
    news = list(w.news)
    nbytes = sum((int(L) + n) * w.Hkv * w.d * 2 * 2 for L, n in zip(wl["cache_lens"].tolist(), news))
    dom, (dom_n, dom_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    achieved = nbytes / (dom_ms / dom_n * 1e-3) / 1e9
    return {"value": nbytes * dist.world / (ms / steps * 1e-3) / 1e9, "unit": "GB/s", "workload": w.name,
            "steps": steps, "ms_per_step": ms / steps, "bytes_per_step": nbytes,
            "new_tokens_per_step": n_new, "output_rows_per_step": n_out,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm"], "traffic": None,
                         "peak_source": f"{peaks['src']} HBM copy", "avg_launch_ms": dom_ms / dom_n},
            "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in prof.items()},
            "gpu_launches": sum(n for n, _ in prof.values())}


def bench_project(args, dist, dev, stream, peaks, ola, torch, W):
    """The shared Q/K/V projection at the Llama-8B shape: a 32-sequence decoding
    pair (64 rows share one read of the 50 MB weight; HBM-bound, reported in
    GB/s of weight + rows + outputs) and an 8192-token prefill chunk
    (tensor-bound, 2 * rows * d_model * N FLOP), with the K/V written to pages.
    The decoding weight fits in L2, so consecutive steps cycle through copies
    of it whose total is well above L2: every step reads its weight from HBM."""
    res = {}
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    for wdef, key in ((W.PROJ_DECODE_32, "decode"), (W.PROJ_PREFILL_8K, "prefill")):
        wl = W.make_projection(wdef)
        nb, no, dm, Hq, Hkv, d = wdef.n_base, wdef.n_out, wdef.d_model, wdef.Hq, wdef.Hkv, wdef.d
        x, w_t = wl["x"].to(dev), wl["w_t"].to(dev)
        w_bytes = w_t.numel() * w_t.element_size()
        copies = [w_t] + [w_t.clone() for _ in range(-(-3 * l2_bytes // w_bytes) - 1)] if key == "decode" else [w_t]
        aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
        P = 64
        max_pages = (nb + P - 1) // P
        kc = torch.empty((max_pages, P, Hkv, d), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        bt = torch.arange(max_pages, dtype=torch.int32, device=dev).view(1, max_pages)
        seq = torch.zeros(nb, dtype=torch.int32, device=dev)
        pos = torch.arange(nb, dtype=torch.int32, device=dev)
        out = (torch.empty((nb, Hq, d), dtype=torch.bfloat16, device=dev),
               torch.empty((no, Hq, d), dtype=torch.bfloat16, device=dev), None, None)
        ws = torch.empty(256, dtype=torch.uint8, device=dev)

        def step(i=0):
            ola.orthros_qkv_project(x, nb, copies[i % len(copies)], Hq, Hkv, d, *aff, k_cache=kc, v_cache=vc,
                                    block_table=bt, token_seq=seq, token_pos=pos, out=out, workspace=ws,
                                    stream=stream)

        for _ in range(max(args.warmup, 3)):
            step()
        torch.cuda.synchronize()
        steps = max(args.steps, 20)
        ms, prof = _timed(ola, torch, dist, stream, step, steps)
        N = (Hq + 2 * Hkv) * d
        nbytes = (N * dm + (nb + no) * dm + (nb + no) * Hq * d + nb * 2 * Hkv * d) * 2
        flops = 2.0 * (nb * N + no * Hq * d) * dm
        n_, t_ = prof["project_tc"]
        avg = t_ / n_
        if key == "decode":
            ach = nbytes / (avg * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s", "frac": ach / peaks["hbm"],
                    "bytes_per_launch": nbytes}
        else:
            ach = flops / (avg * 1e-3) / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16"], "unit": "TFLOP/s",
                    "frac": ach / peaks["bf16"], "flop_per_launch": flops}
        roof.update({"kernel": "project_tc", "avg_launch_ms": avg, "traffic": None,
                     "peak_source": f"{peaks['src']} " + ("HBM copy" if key == "decode" else "bf16 dense (burst)")})
        res[key] = {"workload": wdef.name, "ms_per_step": ms / steps, "steps": steps, "roofline": roof,
                    "l2": (f"{len(copies)} weight copies ({len(copies) * w_bytes / 2**20:.0f} MiB) cycled, "
                           "each step's weight read from HBM") if len(copies) > 1 else "operands larger than L2",
                    "gpu_launches": sum(c for c, _ in prof.values())}
    return res


def bench_seqpar(args, dist, dev, stream, ola, torch, W, pre, world=8):
    """Sequence-parallel split of the 128K prefill over `world` ranks, each
    rank's arithmetic timed on this GPU: its orthros_prefill_shard call
    (band rows of its chunk over [halo ; chunk], the output row's partial over
    its chunk) and the owner's orthros_merge_partials. The halo and partial
    transfers between GPUs are not part of it (one GPU here)."""
    from efficient_long_context_gb300 import seqpar as SP

    wl = pre["wl"]
    inputs = pre["inputs"]
    q, k, v = (inputs[n].to(dev) for n in ("q", "k", "v"))
    aff = [inputs[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    indptr, pos_all = inputs["out_indptr"], inputs["out_positions"]
    B, T = wl.B, wl.T
    pos = pos_all.long()
    seq = torch.repeat_interleave(torch.arange(B), (indptr[1:] - indptr[:-1]).long())
    q_rows_all = q[seq.to(dev), pos.to(dev)]
    rank_ms, parts = [], []
    for r in range(world):
        start, end = SP.chunk_bounds(T, world, r)
        H = SP.halo_len(T, wl.window, world, r)
        k_ext, v_ext = k[:, start - H:end].contiguous(), v[:, start - H:end].contiguous()
        qc = q[:, start:end].contiguous()
        sel, r_indptr, r_pos = SP.shard_rows(pos, seq, B, start, H)
        q_rows = q_rows_all[sel.to(dev)].contiguous()
        r_pos = r_pos.to(dev)
        ws = torch.empty(ola.orthros_prefill_shard_workspace_size(B, end - start, H + end - start, wl.Hq, wl.Hkv,
                                                                  wl.d, len(sel), wl.window), dtype=torch.uint8,
                         device=dev)
        out = None

        def call(_=0):
            nonlocal out
            out = ola.orthros_prefill_shard(qc, k_ext, v_ext, *aff, r_indptr, r_pos, wl.window, wl.scale,
                                            q_rows=q_rows, out=out, workspace=ws, stream=stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        ms, _ = _timed(ola, torch, dist, stream, call, 5)
        rank_ms.append(ms / 5)
        parts.append((out[2].clone(), out[3].clone()))
    o_parts = torch.stack([p[0] for p in parts])
    l_parts = torch.stack([p[1] for p in parts])
    merged = None

    def merge(_=0):
        nonlocal merged
        merged = ola.orthros_merge_partials(o_parts, l_parts, wl.dtype, out=merged, stream=stream)

    for _ in range(3):
        merge()
    torch.cuda.synchronize()
    ms_m, _ = _timed(ola, torch, dist, stream, merge, 10)
    return {"workload": wl.name, "world": world, "rank_ms": rank_ms, "max_rank_ms": max(rank_ms),
            "merge_ms": ms_m / 10, "single_gpu_step_ms": pre["ms_step"],
            "projected_speedup": pre["ms_step"] / (max(rank_ms) + ms_m / 10),
            "note": "ranks emulated one after the other on one GPU; halo and partial transfers not timed"}


def run_ours(args, dist):
    import torch

    import efficient_long_context_gb300 as ola
    from efficient_long_context_gb300 import build as B
    from efficient_long_context_gb300 import workloads as W

    B.build()
    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    stream = torch.cuda.current_stream(dev)
    peaks = load_peaks()
    clocks = ClockSampler(dist.local)
    clocks.start()
    pre = dec = bwd = ext = prj = None
    shapes = {}  # the pre-training and fine-tuning forward workloads
    if args.only in ("all", "prefill"):
        pre = bench_prefill(args, dist, dev, stream, peaks, ola, torch, W, headline_workload(args, W),
                            e2e=args.only == "all")
    seqpar = None
    if args.only == "all" and pre is not None and pre["wl"].name == W.PREFILL_128K.name:
        seqpar = bench_seqpar(args, dist, dev, stream, ola, torch, W, pre)
    if args.only == "all":
        for key, wl in (("pt", W.PT_2K), ("sft", W.SFT_8K)):
            shapes[key] = bench_prefill(args, dist, dev, stream, peaks, ola, torch, W, wl)
    if args.only in ("all", "decode"):
        dec = bench_decode(args, dist, dev, stream, peaks, ola, torch, W)
    if args.only in ("all", "backward"):
        bwd = bench_backward(args, dist, dev, stream, peaks, ola, torch, W)
    if args.only in ("all", "extend"):
        ext = bench_extend(args, dist, dev, stream, peaks, ola, torch, W)
    if args.only in ("all", "project"):
        prj = bench_project(args, dist, dev, stream, peaks, ola, torch, W)
    clk = clocks.stop()
    cpu = None
    base_on = dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline
    if pre is not None and base_on:
        v_cpu, cores, desc = oracle_sample(pre["inputs"], pre["wl"], args.cpu_seconds)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc}
    shape_lines = {}
    for key, r in shapes.items():
        line_r = {"value": r["value"], "unit": "TFLOP/s", "workload": r["wl"].name, "ms_per_step": r["ms_step"],
                  "useful_tflop_per_step": r["flops"]["total"] / 1e12, "l2": r["l2"], "roofline": r["roofline"],
                  "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in r["prof"].items()},
                  "gpu_launches": sum(n for n, _ in r["prof"].values()), "cpu_baseline": None}
        if base_on:
            v_cpu, cores, desc = oracle_prefill_sample(r["inputs"], r["wl"], args.cpu_seconds / 3)
            line_r["cpu_baseline"] = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                      "sample": desc}
        shape_lines[key] = line_r
    if dec is not None:
        st = dec.pop("_state")
        dec["cpu_baseline"] = None
        if base_on:
            v_cpu, cores, desc = oracle_decode_sample(st, args.cpu_seconds / 3)
            dec["cpu_baseline"] = {"value": v_cpu, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}
    if dist.rank != 0:
        return
    if pre is None:  # decode- or backward-only profiling run
        print(json.dumps({"decode": dec, "backward": bwd, "extend": ext, "project": prj, "clocks": clk}), flush=True)
        return
    wl = pre["wl"]
    line = {
        "metric": METRIC, "value": pre["value"], "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": pre["ms_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, affines 1+0.1N / 0.1N; no dataset)",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "window": wl.window, "page_size": pre["P"],
                   "out_rows": ("last position (prefill regime)" if wl.out_mode == "last" else
                                "every position (pre-training)" if wl.out_mode == "all" else
                                f"last {wl.out_mode[1]} positions of each sequence (fine-tuning answer span)"),
                   "useful_tflop_per_step": pre["flops"]["total"] / 1e12,
                   "l2": pre["l2"],
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": pre["roofline"],
        "kernels": {n: {"launches": c, "total_ms": t} for n, (c, t) in pre["prof"].items()},
        "gpu_launches": sum(n for n, _ in pre["prof"].values()),
        "e2e": pre.get("e2e"),
        "seqpar": seqpar,
        "pt": shape_lines.get("pt"),
        "sft": shape_lines.get("sft"),
        "decode": dec,
        "backward": bwd,
        "extend": ext,
        "project": prj,
        "cpu_baseline": cpu,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decoding steps to time (default: the workload's 128)")
    ap.add_argument("--only", choices=("all", "prefill", "decode", "backward", "extend", "project"), default="all",
                    help="run one part (profiling captures); the headline line needs 'all'")
    ap.add_argument("--prefill-workload", choices=("128k", "pt", "sft"), default="128k",
                    help="prefill workload: the 128K headline, or the pre-training / fine-tuning shapes")
    ap.add_argument("--prefill-T", type=int, default=None,
                    help="shorter prefill (a smaller case of the same kernels, for profiler captures)")
    ap.add_argument("--decode-B", type=int, default=None, help="fewer decoding sequences (profiler captures)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target length of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    dist = Dist(enable=args.impl == "ours")
    try:
        if args.impl == "reference":
            run_reference(args, dist)
        else:
            run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
