"""GPU parity of orthros_extend (continuous-batching step) against the oracle.

Mixed batches: sequences that append a prefill chunk, one decoding token, or
nothing, in one call; output rows at the new tokens (q read from the new
token) or anywhere in the history (q_out given). The bf16 path with pages of
64 tokens takes the TMA split-KV kernel, other page sizes and fp32 the
CUDA-core rows; the appended cache slots must match bit for bit.
"""
import numpy as np
import pytest
import torch

from efficient_long_context_gb300 import workloads as W
from tests.parity_util import TOL, f32, max_err

pytestmark = pytest.mark.gpu

CASES = [
    # name, B, Hq, Hkv, d, window, len_lo, len_hi, news, page_size, dtype, history_rows
    ("mix_bf16", 6, 8, 2, 128, 64, 0, 700, (37, 1, 0, 1, 5, 130), 64, torch.bfloat16, 0),
    ("mix_bf16_hist", 5, 8, 2, 128, 100, 10, 900, (3, 1, 1, 64, 0), 64, torch.bfloat16, 3),
    ("mix_bf16_mha", 4, 4, 4, 128, 33, 0, 300, (1, 20, 1, 0), 64, torch.bfloat16, 2),
    ("mix_bf16_gqa16", 3, 32, 2, 128, 50, 5, 400, (9, 1, 2), 64, torch.bfloat16, 0),
    ("mix_bf16_d64", 4, 8, 2, 64, 70, 0, 500, (1, 17, 1, 3), 64, torch.bfloat16, 2),
    ("mix_bf16_page16", 4, 8, 2, 128, 40, 0, 260, (5, 1, 0, 12), 16, torch.bfloat16, 2),
    ("mix_fp32", 4, 4, 2, 64, 30, 0, 200, (7, 1, 1, 0), 16, torch.float32, 2),
]


def run(case, with_q_out):
    import efficient_long_context_gb300 as ola
    import oracle

    name, B, Hq, Hkv, d, w, lo, hi, news, P, dt, hist = case
    wl_def = W.ExtendWorkload(name, B, Hq, Hkv, d, w, lo, hi, news, page_size=P, dtype=dt, history_rows=hist,
                              seed=len(name) + B)
    wl = W.make_extend(wl_def, with_q_out=with_q_out)
    dev = "cuda"
    kc, vc = wl["k_cache"].to(dev), wl["v_cache"].to(dev)
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    q_out = wl["q_out"].to(dev) if wl["q_out"] is not None else None
    got = ola.orthros_extend(wl["q"].to(dev), wl["k_new"].to(dev), wl["v_new"].to(dev), kc, vc,
                             wl["block_table"].to(dev), wl["cache_lens"].to(dev), wl["new_indptr"], wl["out_indptr"],
                             wl["out_positions"].to(dev), *aff, w, wl["scale"], q_out=q_out)
    torch.cuda.synchronize()
    kc_ref, vc_ref = f32(wl["k_cache"]).copy(), f32(wl["v_cache"]).copy()
    ref = oracle.extend(f32(wl["q"]), f32(wl["k_new"]), f32(wl["v_new"]), kc_ref, vc_ref, wl["block_table"].numpy(),
                        wl["cache_lens"].numpy(), wl["new_indptr"].numpy(), wl["out_indptr"].numpy(),
                        wl["out_positions"].numpy(), *(f32(wl[n]) for n in ("alpha_base", "beta_base", "alpha_out",
                                                                              "beta_out")),
                        w, wl["scale"], q_out=f32(wl["q_out"]) if wl["q_out"] is not None else None)
    tol_o, tol_l = TOL[dt]
    errs = dict(o_base=max_err(got[0], ref[0]), lse_base=max_err(got[1], ref[1]),
                o_out=max_err(got[2], ref[2]), lse_out=max_err(got[3], ref[3]))
    assert errs["o_base"] <= tol_o and errs["o_out"] <= tol_o, f"{name} {errs}"
    assert errs["lse_base"] <= tol_l and errs["lse_out"] <= tol_l, f"{name} {errs}"
    # the appends: every slot equals the oracle's cache after its own appends
    assert np.array_equal(kc.float().cpu().numpy(), kc_ref) and np.array_equal(vc.float().cpu().numpy(), vc_ref)
    return errs


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
@pytest.mark.parametrize("with_q_out", [False, True])
def test_extend_mixed_batch(case, with_q_out):
    run(case, with_q_out)


def test_extend_named_workload():
    """The benchmark's mixed step (32 sequences, 16K-32K cached tokens each)."""
    import dataclasses

    wl = dataclasses.replace(W.MIXED_32)
    errs = run((wl.name, wl.B, wl.Hq, wl.Hkv, wl.d, wl.window, wl.len_lo, wl.len_hi, wl.news, wl.page_size,
                wl.dtype, 0), False)
    assert errs
