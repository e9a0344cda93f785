"""orthros_decode_static: the decoding step for callers that cannot allocate.

Some callers have no way to hand the library a device workspace where they
run a decoding step (an operator interface that passes only inputs and
outputs, or an allocator that must not grow while serving). For them
orthros_decode_static takes its scratch from a fixed array inside the library.
These tests call it through the C ABI and check it against orthros_decode on
the same inputs, over two calls in a row (the array is shared between calls
and keeps the previous call's contents), and check that sizes beyond the
array are refused before any launch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import efficient_long_context_gb300 as ola
from efficient_long_context_gb300 import workloads as W
from tests.parity_util import TOL, max_err
from tests.test_gpu_status import bad_page_decode_case, check_bad_page_rows


@pytest.mark.gpu
def test_static_decode_matches_workspace_decode():
    wl = W.DecodeWorkload("static", 6, 32, 8, 128, 256, 64, 0, 0, 2, seed=77)
    st = W.make_decode(wl, lens=[0, 1, 300, 1000, 5000, 20000], with_q_out=True)
    m = st.meta
    dev = "cuda"
    kc_a, vc_a = st.k_cache.to(dev), st.v_cache.to(dev)
    kc_b, vc_b = kc_a.clone(), vc_a.clone()
    bt = st.block_table.to(dev)
    aff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    ws = torch.empty(ola.orthros_decode_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.d, m["max_pages"], wl.page_size),
                     dtype=torch.uint8, device=dev)
    tol_o, tol_l = TOL[torch.bfloat16]
    for s in range(2):  # two calls in a row, consecutive decoding steps
        lens = (st.cache_lens + s).to(dev)
        args = (st.q[s].to(dev), st.k_new[s].to(dev), st.v_new[s].to(dev))
        ref = ola.orthros_decode(*args, kc_a, vc_a, bt, lens, *aff, wl.window, wl.scale, q_out=st.q_out[s].to(dev),
                                 workspace=ws)
        ref = [t.clone() for t in ref]
        got = ola.orthros_decode_static(*args, kc_b, vc_b, bt, lens, *aff, wl.window, wl.scale,
                                        q_out=st.q_out[s].to(dev))
        torch.cuda.synchronize()
        for name, g, r, tol in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref,
                                   (tol_o, tol_l, tol_o, tol_l)):
            err = max_err(g, r.float().cpu().numpy())
            assert err <= tol, f"step {s} {name}: {err}"
        assert torch.equal(kc_a, kc_b) and torch.equal(vc_a, vc_b), "the appends differ"


@pytest.mark.gpu
def test_static_decode_bad_page_gives_nan_rows():
    # the status word of this entry point is not exposed, so rows that read a
    # block-table entry outside the page pool must come back as NaN
    wl, st, bt = bad_page_decode_case()
    dev = "cuda"
    aff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    out = ola.orthros_decode_static(st.q[0].to(dev), st.k_new[0].to(dev), st.v_new[0].to(dev), st.k_cache.to(dev),
                                    st.v_cache.to(dev), bt.to(dev), st.cache_lens.to(dev), *aff, wl.window,
                                    wl.scale)
    torch.cuda.synchronize()
    check_bad_page_rows(out)


def test_static_decode_refuses_sizes_beyond_the_array():
    # host-side refusal: no launch happens, so this also runs without a GPU
    lib = ola.load_library()
    fake = ctypes.c_void_p(1 << 12)
    B, Hq, Hkv, d, max_pages, page_size = 128, 32, 8, 128, 600, 64
    # 128 sequences x 8 kv heads over 600 pages of 64 tokens need ~43 MB of
    # partials; the fake pointers below are only safe because the host refuses
    # the call before any launch, so make sure first that the size is refused
    need = ola.orthros_decode_workspace_size(B, Hq, Hkv, d, max_pages, page_size)
    assert need > 32 << 20, need
    rc = lib.orthros_decode_static(fake, None, fake, fake, fake, fake, fake, max_pages, page_size, 20000, fake,
                                   fake, fake, fake, fake, B, Hq, Hkv, d, 4096, 0.088, 0,
                                   fake, fake, fake, fake, None)
    assert rc == 4, rc
    assert "static array" in ola.orthros_last_error()
