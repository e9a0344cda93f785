"""The seeded input recipe (CPU): same seed, same bits; the distributions and
structures the workloads promise (affines 1 + 0.1 N / 0.1 N per head and
channel, a per-(kv head, channel) key offset, output-row sets of each regime,
a decoding cache whose physical pages are a permutation)."""
import torch

from efficient_long_context_gb300 import workloads as W


def test_prefill_is_deterministic_per_seed():
    a = W.small_prefill(2, 40, 4, 2, 16, 9, seed=5, out_mode=("span", 7), with_q_out=True)
    b = W.small_prefill(2, 40, 4, 2, 16, 9, seed=5, out_mode=("span", 7), with_q_out=True)
    c = W.small_prefill(2, 40, 4, 2, 16, 9, seed=6, out_mode=("span", 7), with_q_out=True)
    for n in ("q", "k", "v", "alpha_base", "beta_base", "alpha_out", "beta_out", "q_out", "out_positions"):
        assert torch.equal(a[n], b[n]), n
    assert not torch.equal(a["q"], c["q"])


def test_affine_and_input_distributions():
    wl = W.small_prefill(1, 64, 32, 8, 128, 16, dtype=torch.float32, seed=3)
    for n, mean, std in (("alpha_base", 1.0, 0.1), ("beta_base", 0.0, 0.1), ("alpha_out", 1.0, 0.1),
                         ("beta_out", 0.0, 0.1), ("q", 0.0, 1.0), ("k", 0.0, 1.0), ("v", 0.0, 1.0)):
        x = wl[n].double()
        assert abs(float(x.mean()) - mean) < 0.05 * max(std, 0.2), (n, float(x.mean()))
        assert abs(float(x.std()) / std - 1) < 0.1, (n, float(x.std()))
    # the two streams' affines are drawn separately
    assert not torch.equal(wl["alpha_base"], wl["alpha_out"])


def test_key_offsets_are_shared_across_positions():
    """A key offset per (kv head, channel), the same at every position: the
    mean over positions of (k with offset) - (k without) is that offset."""
    base = W.small_prefill(1, 2000, 4, 2, 8, 5, dtype=torch.float32, seed=11)
    off = W.small_prefill(1, 2000, 4, 2, 8, 5, dtype=torch.float32, seed=11, k_offset_std=0.5)
    diff = (off["k"] - base["k"]).double()  # [1, T, Hkv, d]
    per = diff[0, 0]
    assert torch.allclose(diff, per.expand_as(diff), atol=1e-6)  # constant over positions
    assert 0.2 < float(per.std()) < 1.0  # ~0.5 N(0,1) over 16 values


def test_output_row_sets_of_the_regimes():
    T, B = 10, 3
    ip, pos = W.out_positions_for("last", B, T)
    assert ip.tolist() == [0, 1, 2, 3] and pos.tolist() == [9, 9, 9]
    ip, pos = W.out_positions_for("all", B, T)
    assert ip.tolist() == [0, 10, 20, 30] and pos.tolist() == list(range(10)) * 3
    ip, pos = W.out_positions_for(("span", 4), B, T)
    assert ip.tolist() == [0, 4, 8, 12] and pos.tolist() == [6, 7, 8, 9] * 3
    ip, pos = W.out_positions_for(("list", [[1, 5], [], [0]]), B, T)
    assert ip.tolist() == [0, 2, 2, 3] and pos.tolist() == [1, 5, 0]


def test_decode_cache_structure():
    w = W.DecodeWorkload("t", 5, 8, 2, 16, 64, 16, 10, 90, 3, seed=21)
    st = W.make_decode(w)
    m = st.meta
    lens = st.cache_lens.tolist()
    assert all(10 <= L <= 90 for L in lens)
    # every sequence has the pages its history plus all steps need; physical ids are a permutation
    used = []
    for b, L in enumerate(lens):
        n = (L + m["steps"] + w.page_size - 1) // w.page_size
        row = st.block_table[b].tolist()
        assert all(p >= 0 for p in row[:n]) and all(p == -1 for p in row[n:])
        used += row[:n]
    assert sorted(used) == list(range(m["num_pages"]))
    assert used != sorted(used)  # scattered, not the identity
    assert st.k_cache.shape == (m["num_pages"], w.page_size, w.Hkv, w.d)
    assert st.q.shape == (m["steps"], w.B, w.Hq, w.d) and st.k_new.shape == (m["steps"], w.B, w.Hkv, w.d)
    again = W.make_decode(w)
    assert torch.equal(st.k_cache, again.k_cache) and torch.equal(st.block_table, again.block_table)
