"""GPU parity of orthros_prefill against the CPU oracle (same seeded inputs).

Small shapes are compared in full (several tiles and a ragged tail); the
named workloads run at full size in the launch configuration the benchmark
times and are compared on sampled rows that the oracle computes one by one.
"""
import numpy as np
import pytest
import torch

from efficient_long_context_gb300 import workloads as W
from tests.parity_util import compare_prefill, prefill_tolerances, record_margin, run_gpu_prefill, sample_positions

pytestmark = pytest.mark.gpu

SMALL = [
    # (B, T, Hq, Hkv, d, window, out_mode, dtype)
    (1, 1, 1, 1, 128, 1, "last", torch.bfloat16),
    (1, 100, 2, 1, 128, 64, "all", torch.bfloat16),
    (2, 333, 4, 4, 128, 63, ("span", 70), torch.bfloat16),
    (1, 333, 8, 2, 128, 65, "last", torch.bfloat16),
    (1, 700, 4, 1, 128, 128, ("list", [[0, 5, 127, 128, 129, 400, 699]]), torch.bfloat16),
    (2, 257, 4, 2, 64, 256, "all", torch.bfloat16),
    (1, 300, 2, 2, 64, 1, "last", torch.bfloat16),
    (1, 300, 4, 2, 128, 299, ("span", 3), torch.bfloat16),
    (1, 300, 4, 2, 128, 300, "all", torch.bfloat16),
    (1, 300, 4, 2, 128, 307, ("list", [[]]), torch.bfloat16),
    (3, 129, 32, 8, 128, 64, ("list", [[128], [], [0, 64, 128]]), torch.bfloat16),
    (1, 200, 4, 2, 64, 50, "all", torch.float32),
    (2, 150, 2, 1, 128, 17, ("span", 40), torch.float32),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"B{c[0]}T{c[1]}h{c[2]}x{c[3]}d{c[4]}w{c[5]}{str(c[7])[6:]}")
@pytest.mark.parametrize("with_q_out", [False, True])
def test_small_shapes(case, with_q_out):
    B, T, Hq, Hkv, d, w, mode, dt = case
    wl = W.small_prefill(B, T, Hq, Hkv, d, w, dtype=dt, out_mode=mode, seed=T + w, with_q_out=with_q_out)
    compare_prefill(wl, run_gpu_prefill(wl), what=str(case))


def test_key_offsets_small():
    wl = W.small_prefill(2, 600, 8, 2, 128, 100, out_mode=("span", 200), seed=5, k_offset_std=0.5)
    compare_prefill(wl, run_gpu_prefill(wl), what="offsets")


def test_tiny_fp32_full():
    wl = W.make_prefill(W.TINY_FP32)
    errs = compare_prefill(wl, run_gpu_prefill(wl), what=W.TINY_FP32.name)
    record_margin(W.TINY_FP32.name, errs, prefill_tolerances(torch.float32), "max abs error vs the oracle, every row")


@pytest.mark.parametrize("work", [W.PT_2K, W.SFT_8K, W.PREFILL_128K], ids=lambda x: x.name)
def test_named_workload_sampled(work):
    wl = W.make_prefill(work)
    gpu = run_gpu_prefill(wl)
    rows = sample_positions(work.T, work.window, 24, seed=work.seed)
    n_out = int(wl["out_indptr"][-1])
    r = np.random.default_rng(work.seed)
    out_rows = np.unique(np.concatenate([[0, n_out - 1], r.choice(n_out, size=min(24, n_out), replace=False)]))
    errs = compare_prefill(wl, gpu, base_rows=rows, out_rows=out_rows, what=work.name)
    record_margin(work.name, errs, prefill_tolerances(work.dtype),
                  f"max abs error vs the oracle on {len(rows)} sampled positions x {work.B} sequences and "
                  f"{len(out_rows)} sampled output rows")
