"""GPU parity of orthros_prefill against the CPU oracle (same seeded inputs).

Small shapes are compared in full (several tiles and a ragged tail); the
named workloads run at full size in the launch configuration the benchmark
times and are compared on sampled rows that the oracle computes one by one.
"""
import os

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
    # windows of 4096 keys and more take the one-thread-per-row softmax
    (1, 300, 4, 2, 128, 4096, "all", torch.bfloat16),
    (2, 257, 4, 2, 64, 5000, ("span", 40), torch.bfloat16),
    (1, 700, 8, 2, 128, 4096, ("list", [[0, 5, 127, 128, 129, 400, 699]]), torch.bfloat16),
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


@pytest.mark.parametrize("window", [200, 4096], ids=["w200", "w4096_row_softmax"])
@pytest.mark.parametrize("mode", ["all", ("span", 70)], ids=["all", "span"])
def test_key_beyond_fp16_range(mode, window):
    """Single keys of 7e4 and -9e4 (fp16 stops at 65504): the fp16 key copy is
    scaled by 2^-2 and the logit scale by 2^2. The query channel that meets
    them is small (subnormal in fp16), so every logit stays moderate and the
    usual tolerances hold."""
    wl = W.small_prefill(2, 300, 4, 2, 128, window, out_mode=mode, seed=11)
    c = 5
    wl["k"][0, 100, 1, c] = 70000.0
    wl["k"][1, 7, 0, c] = -90000.0
    for a, b in (("alpha_base", "beta_base"), ("alpha_out", "beta_out")):
        wl[a][:, c] = 2e-5
        wl[b][:, c] = 0.0
    compare_prefill(wl, run_gpu_prefill(wl), what="keys beyond fp16")


@pytest.mark.parametrize("window", [200, 4096], ids=["w200", "w4096_row_softmax"])
@pytest.mark.parametrize("mode", ["all", ("span", 70)], ids=["all", "span"])
def test_query_beyond_fp16_range(mode, window):
    """Affine weights of +-1e5 on one channel lift about half of the rows of a
    base head and of an output head past 65504; those rows are staged as
    q * 2^-r and their logit scale takes 2^r, the other rows of the same tiles
    keep r = 0. The keys' values in that channel are small multiples of 2^-16
    (exact in bf16 and fp16), so the logits stay moderate. One query sits just
    below 2^17 (130781.25), where rounding the row maximum up crosses the
    power of two: both column halves must still pick the same shift (window
    200; with the 4096-key window one thread holds the whole row)."""
    wl = W.small_prefill(2, 300, 4, 2, 128, window, out_mode=mode, seed=12)
    c = 9
    wl["alpha_base"][0, c] = 1e5
    wl["beta_base"][0, c] = 0.0
    wl["alpha_out"][3, c] = -1e5
    wl["beta_out"][3, c] = 3e4
    wl["q"][0, 299, 3, c] = -1.0078125  # affined: 130781.25
    g = torch.Generator().manual_seed(3)
    m = torch.randint(-2, 3, wl["k"].shape[:-1] + (1,), generator=g).float()
    wl["k"][..., c:c + 1] = (m * 2.0 ** -16).to(wl["k"].dtype)
    compare_prefill(wl, run_gpu_prefill(wl), what="queries beyond fp16")


def test_tiny_fp32_full():
    wl = W.make_prefill(W.TINY_FP32)
    errs = compare_prefill(wl, run_gpu_prefill(wl), what=W.TINY_FP32.name)
    record_margin(W.TINY_FP32.name, errs, prefill_tolerances(torch.float32), "max abs error vs the oracle, every row")


@pytest.mark.parametrize("work", [W.PT_2K, W.SFT_8K], ids=lambda x: x.name)
def test_named_workload_every_row(work):
    """The pre-training and fine-tuning workloads at full size, in the
    benchmark's launch, compared with the oracle on every base position and
    every output row (the oracle takes a few seconds for these)."""
    wl = W.make_prefill(work)
    errs = compare_prefill(wl, run_gpu_prefill(wl), what=work.name)
    record_margin(work.name + ", every row", errs, prefill_tolerances(work.dtype),
                  "max abs error vs the oracle over every base position and every output row")


@pytest.mark.skipif(os.environ.get("ORTHROS_FULL_PARITY") != "1",
                    reason="about three minutes of oracle time on 16 cores; set ORTHROS_FULL_PARITY=1")
def test_128k_every_row():
    """The 128K prefill compared with the oracle on all 131072 positions x 32
    heads and the output row (8.66 TFLOP of oracle work)."""
    work = W.PREFILL_128K
    wl = W.make_prefill(work)
    errs = compare_prefill(wl, run_gpu_prefill(wl), what=work.name)
    record_margin(work.name + ", every row", errs, prefill_tolerances(work.dtype),
                  "max abs error vs the oracle over every base position and the output row")


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
