"""Bad device-side data is reported through the status word, never by a fault.

Each case hands the library data that only the GPU can see is wrong; the
kernels' own checks skip the affected rows and set a bit that orthros_check
returns. All accesses stay in bounds (the kernels clamp before they read).
"""
import pytest
import torch

import efficient_long_context_gb300 as ola
from efficient_long_context_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV_BAD_POSITION, DEV_BAD_PAGE, DEV_BAD_LENGTH = 0x1, 0x2, 0x4


def _prefill(wl, ws=None, **kw):
    dev = "cuda"
    q, k, v = (wl[n].to(dev) for n in ("q", "k", "v"))
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    if ws is None:
        n_out = int(wl["out_indptr"][-1])
        ws = torch.empty(ola.orthros_prefill_workspace_size(wl["B"], wl["T"], wl["Hq"], wl["Hkv"], wl["d"], n_out,
                                                            wl["window"], wl["dtype"]), dtype=torch.uint8, device=dev)
    out = ola.orthros_prefill(q, k, v, *aff, wl["out_indptr"], wl["out_positions"].to(dev), wl["window"],
                              wl["scale"], workspace=ws, **kw)
    return out, ws


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", [("list", [[3, 200, 50]]), ("list", [list(range(40))])])
def test_bad_output_position(dtype, mode):
    wl = W.small_prefill(1, 200, 4, 2, 128, 32, dtype=dtype, out_mode=mode, seed=1)
    wl["out_positions"][1] = 200  # == T: out of range
    out, ws = _prefill(wl)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_POSITION, (rc, bits)
    # the other rows are still right: row 0 equals a clean run's row 0
    wl2 = dict(wl)
    wl2["out_positions"] = wl["out_positions"].clone()
    wl2["out_positions"][1] = 199
    out2, ws2 = _prefill(wl2)
    assert ola.orthros_check(ws2) == (0, 0)
    torch.testing.assert_close(out[2][0].float(), out2[2][0].float(), rtol=0, atol=0)
    torch.testing.assert_close(out[0].float(), out2[0].float(), rtol=0, atol=0)


def test_key_beyond_fp16_range_is_no_error():
    """Keys past the fp16 range are rescaled, not flagged (values: test_parity_prefill)."""
    wl = W.small_prefill(1, 256, 2, 2, 128, 64, seed=2)
    wl["k"][0, 100, 1, 5] = 70000.0
    out, ws = _prefill(wl)
    assert ola.orthros_check(ws) == (0, 0)
    assert torch.isfinite(out[0]).all() and torch.isfinite(out[1]).all()


def test_prefill_cache_fill_bad_page():
    wl = W.small_prefill(1, 128, 2, 2, 128, 64, seed=3)
    kc = torch.zeros((4, 64, 2, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = torch.tensor([[1, 9]], dtype=torch.int32, device="cuda")  # page 9 is outside the pool of 4
    _, ws = _prefill(wl, k_cache=kc, v_cache=vc, block_table=bt, page_size=64)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_PAGE, (rc, bits)
    assert torch.equal(kc[1].cpu(), wl["k"][0, :64])  # the good page was written


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_bad_length_and_page(dtype):
    wl = W.DecodeWorkload("bad", 3, 8, 2, 128, 16, 16, 0, 0, 1, dtype=dtype, seed=4)
    st = W.make_decode(wl, lens=[5, 40, 70])
    dev = "cuda"
    kc, vc = st.k_cache.to(dev), st.v_cache.to(dev)
    bt = st.block_table.clone()
    bt[1, 1] = st.k_cache.shape[0] + 3  # a page id outside the pool, inside sequence 1's history
    lens = st.cache_lens.clone()
    lens[2] = bt.shape[1] * wl.page_size + 5  # past the block table
    aff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    ws = torch.empty(ola.orthros_decode_workspace_size(3, 8, 2, 128, bt.shape[1], 16, dtype), dtype=torch.uint8,
                     device=dev)
    out = ola.orthros_decode(st.q[0].to(dev), st.k_new[0].to(dev), st.v_new[0].to(dev), kc, vc, bt.to(dev),
                             lens.to(dev), *aff, wl.window, wl.scale, workspace=ws)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_PAGE and bits & DEV_BAD_LENGTH, (rc, bits)
    assert torch.isnan(out[2][2].float()).all()  # the sequence with a bad length: NaN output rows
    assert torch.isfinite(out[0][0].float()).all()  # an untouched sequence is fine


def bad_page_decode_case():
    """Three sequences on 64-token pages (the TMA-fed split-KV path); sequence
    1 (300 cached tokens) has a block-table entry outside the pool for its
    tokens 64..127. Its output row reads them, its 64-key window does not."""
    wl = W.DecodeWorkload("bad_page64", 3, 8, 2, 128, 64, 64, 0, 0, 1, seed=12)
    st = W.make_decode(wl, lens=[100, 300, 500])
    bt = st.block_table.clone()
    bt[1, 1] = st.k_cache.shape[0] + 7
    return wl, st, bt


def check_bad_page_rows(out):
    o_base, _, o_out, lse_out = (t.float() for t in out)
    assert torch.isnan(o_out[1]).all() and torch.isnan(lse_out[1]).all()  # reads the bad page
    assert torch.isfinite(o_base[1]).all()  # its window lies past the bad page
    for b in (0, 2):  # untouched sequences
        assert torch.isfinite(o_out[b]).all() and torch.isfinite(o_base[b]).all()


def test_decode_bad_page_on_tma_path_gives_nan_rows():
    wl, st, bt = bad_page_decode_case()
    dev = "cuda"
    aff = [a.to(dev) for a in (st.alpha_base, st.beta_base, st.alpha_out, st.beta_out)]
    ws = torch.empty(ola.orthros_decode_workspace_size(3, 8, 2, 128, bt.shape[1], 64), dtype=torch.uint8, device=dev)
    out = ola.orthros_decode(st.q[0].to(dev), st.k_new[0].to(dev), st.v_new[0].to(dev), st.k_cache.to(dev),
                             st.v_cache.to(dev), bt.to(dev), st.cache_lens.to(dev), *aff, wl.window, wl.scale,
                             workspace=ws)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_PAGE, (rc, bits)
    check_bad_page_rows(out)


@pytest.mark.parametrize("page_size,dtype", [(64, torch.bfloat16), (16, torch.bfloat16), (16, torch.float32)])
def test_extend_bad_rows_are_flagged(page_size, dtype):
    """A history output row without q_out and a sequence whose length runs past
    its block table are flagged; their rows come back NaN, the others are
    those of a clean call."""
    wdef = W.ExtendWorkload("bad_ext", 3, 8, 2, 128, 32, 10, 200, (3, 1, 2), page_size=page_size, dtype=dtype,
                            seed=6)
    wl = W.make_extend(wdef)
    dev = "cuda"

    def call(lens, pos):
        kc, vc = wl["k_cache"].to(dev), wl["v_cache"].to(dev)
        aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
        ws = torch.empty(ola.orthros_extend_workspace_size(3, 6, 3, 8, 2, 128, wl["max_pages"], page_size, dtype),
                         dtype=torch.uint8, device=dev)
        out = ola.orthros_extend(wl["q"].to(dev), wl["k_new"].to(dev), wl["v_new"].to(dev), kc, vc,
                                 wl["block_table"].to(dev), lens.to(dev), wl["new_indptr"], wl["out_indptr"],
                                 pos.to(dev), *aff, wdef.window, wdef.scale, workspace=ws)
        return out, ola.orthros_check(ws)

    clean, st = call(wl["cache_lens"], wl["out_positions"])
    assert st == (0, 0)
    pos = wl["out_positions"].clone()
    pos[0] = 0  # a history position of sequence 0, but no q_out: no query for it
    lens = wl["cache_lens"].clone()
    lens[2] = wl["max_pages"] * page_size  # sequence 2's appends fall past its block table
    bad, (rc, bits) = call(lens, pos)
    assert rc == 5 and bits & DEV_BAD_POSITION and bits & (DEV_BAD_LENGTH | DEV_BAD_PAGE), (rc, bits)
    assert torch.isnan(bad[2][0].float()).all() and torch.isnan(bad[3][0]).all()  # the flagged output row
    assert torch.isnan(bad[1][4:6]).all()  # sequence 2's base rows
    torch.testing.assert_close(bad[0][:4].float(), clean[0][:4].float(), rtol=0, atol=0)
    torch.testing.assert_close(bad[2][1].float(), clean[2][1].float(), rtol=0, atol=0)


def test_backward_bad_output_position():
    wl = W.small_prefill(1, 200, 4, 2, 128, 32, out_mode=("list", [[3, 150, 50]]), seed=7)
    dev = "cuda"
    q, k, v = (wl[n].to(dev) for n in ("q", "k", "v"))
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    fwd = ola.orthros_prefill(q, k, v, *aff, wl["out_indptr"], wl["out_positions"].to(dev), wl["window"],
                              wl["scale"])
    do_b, do_o = (t.to(dev) for t in W.make_grad_outputs(wl, 3))
    pos = wl["out_positions"].clone()
    pos[1] = 200  # == T
    ws = torch.empty(ola.orthros_prefill_backward_workspace_size(1, 200, 4, 2, 128, 3, 32), dtype=torch.uint8,
                     device=dev)
    ola.orthros_prefill_backward(q, k, v, *aff, wl["out_indptr"], pos.to(dev), wl["window"], wl["scale"], *fwd, do_b,
                                 do_o, workspace=ws)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_POSITION, (rc, bits)


def test_projection_bad_page():
    wdef = W.ProjectionWorkload("bad_proj", 4, 0, 128, 4, 2, 64, seed=8)
    wl = W.make_projection(wdef)
    dev = "cuda"
    kc = torch.zeros((2, 16, 2, 64), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    bt = torch.tensor([[1, 5]], dtype=torch.int32, device=dev)  # page 5 is outside the pool of 2
    seq = torch.zeros(4, dtype=torch.int32, device=dev)
    pos = torch.tensor([0, 1, 16, 17], dtype=torch.int32, device=dev)  # the last two rows land on page 5
    aff = [wl[n].to(dev) for n in ("alpha_base", "beta_base", "alpha_out", "beta_out")]
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    out = ola.orthros_qkv_project(wl["x"].to(dev), 4, wl["w_t"].to(dev), 4, 2, 64, *aff, kv_out=True, k_cache=kc,
                                  v_cache=vc, block_table=bt, token_seq=seq, token_pos=pos, workspace=ws)
    rc, bits = ola.orthros_check(ws)
    assert rc == 5 and bits & DEV_BAD_PAGE, (rc, bits)
    assert torch.equal(kc[1, :2].cpu(), out[2][:2].cpu())  # the rows with a page were written


def test_bounded_wait_runs_out_and_reports_a_timeout():
    """The failure path of every TMA / tensor-core kernel: a wait on a barrier
    that nothing arms runs out (here after 1e5 SM cycles), the kernel raises
    the timeout bit and returns, and the context stays usable."""
    import time

    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ola.orthros_selftest_wait_timeout(100_000, ws)
    rc, bits = ola.orthros_check(ws)
    elapsed = time.perf_counter() - t0
    assert rc == 6 and bits == 0x10, (rc, bits)  # ORTHROS_ETIMEOUT, ORTHROS_DEV_TIMEOUT only
    assert elapsed < 1.0, elapsed  # the other threads left on the abort flag, not on their own 2 s limit
    # the context still works: a normal call afterwards succeeds
    wl = W.small_prefill(1, 64, 2, 2, 128, 16, seed=13)
    _, ws2 = _prefill(wl)
    assert ola.orthros_check(ws2) == (0, 0)
