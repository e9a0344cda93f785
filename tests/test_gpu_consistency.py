"""Prefill, then decoding steps, equals one longer prefill (on the GPU).

The paper's regimes share one formulation (Sec. 3.2, "strict algorithmic
consistency"): a prefill over T0 tokens that fills the paged cache, followed
by N decoding steps appending tokens T0..T0+N-1, must give at every new
position the base output of a single prefill over T0+N tokens, and the output
stream of that prefill with output rows at those positions. Checked against
the GPU prefill and against the oracle.
"""
import numpy as np
import pytest
import torch

import efficient_long_context_gb300 as ola
from efficient_long_context_gb300 import workloads as W
from tests.parity_util import TOL, f32, max_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,Hq,Hkv,d,w", [(torch.bfloat16, 32, 8, 128, 100), (torch.bfloat16, 8, 8, 64, 300),
                                              (torch.float32, 4, 2, 128, 50)])
def test_prefill_then_decode_matches_long_prefill(dtype, Hq, Hkv, d, w):
    import oracle

    B, T0, N, P = 2, 700, 6, 64
    T = T0 + N
    full = W.small_prefill(B, T, Hq, Hkv, d, w, dtype=dtype, out_mode=("span", N + 1), seed=9)
    dev = "cuda"
    aff = [full[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    # one long prefill (output rows at T0-1 .. T-1)
    q, k, v = (full[n].to(dev) for n in ("q", "k", "v"))
    long_out = ola.orthros_prefill(q, k, v, *aff, full["out_indptr"], full["out_positions"].to(dev), w,
                                   full["scale"])
    # prefill over the first T0 tokens with the paged cache fill (shuffled pages)
    pages_per = (T + P - 1) // P
    rng = np.random.default_rng(0)
    perm = torch.as_tensor(rng.permutation(B * pages_per).astype(np.int32))
    bt = perm.view(B, pages_per).to(dev)
    kc = torch.zeros((B * pages_per, P, Hkv, d), dtype=dtype, device=dev)
    vc = torch.zeros_like(kc)
    ind0 = torch.tensor([0, 1, 2], dtype=torch.int32)
    pos0 = torch.tensor([T0 - 1, T0 - 1], dtype=torch.int32, device=dev)
    pre = ola.orthros_prefill(q[:, :T0].contiguous(), k[:, :T0].contiguous(), v[:, :T0].contiguous(), *aff, ind0,
                              pos0, w, full["scale"], k_cache=kc, v_cache=vc, block_table=bt, page_size=P)
    tol_o, tol_l = TOL[dtype]
    # prefill's last output row equals the long prefill's first output row
    assert max_err(pre[2], long_out[2][[0, N + 1]].float().cpu().numpy()) <= tol_o
    lens = torch.full((B,), T0, dtype=torch.int32, device=dev)
    for s in range(N):
        t = T0 + s
        ob, lb, oo, lo = ola.orthros_decode(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(), kc, vc,
                                            bt, lens, *aff, w, full["scale"])
        lens += 1
        rows = [1 + s, N + 2 + s]  # output rows of position t in both sequences
        assert max_err(ob, long_out[0][:, t].float().cpu().numpy()) <= tol_o
        assert max_err(lb, long_out[1][:, :, t].float().cpu().numpy()) <= tol_l
        assert max_err(oo, long_out[2][rows].float().cpu().numpy()) <= tol_o
        assert max_err(lo, long_out[3][rows].float().cpu().numpy()) <= tol_l
    # and the long prefill itself against the oracle at the new positions
    ref = oracle.prefill(f32(full["q"]), f32(full["k"]), f32(full["v"]), *(f32(full[n]) for n in
                         ("alpha_base", "beta_base", "alpha_out", "beta_out")), full["out_indptr"].numpy(),
                         full["out_positions"].numpy(), w, full["scale"], base_rows=np.arange(T0, T, dtype=np.int32))
    assert max_err(long_out[0][:, T0:], ref[0]) <= tol_o
    assert max_err(long_out[1][:, :, T0:], ref[1]) <= tol_l
    assert max_err(long_out[2], ref[2]) <= tol_o
    assert max_err(long_out[3], ref[3]) <= tol_l
