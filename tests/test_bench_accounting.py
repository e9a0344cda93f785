"""The benchmark's work accounting (what the roofline figures divide by),
checked on CPU against explicit counting and against the closed forms of the
workload definitions.

Useful prefill work is 4*d FLOP per (query, key) pair and query head: 2*d for
q.k and 2*d for p*v (Orthros paper, Sec. 3.3 counts the base stream's cost
as O(T w d) and the output rows' as O(T_out T d)). Decoding moves every cached
key and value once per step, the appended token included.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from efficient_long_context_gb300 import workloads as W  # noqa: E402


def pairs_by_loop(T, w):
    """(query, key) pairs of Eq. 4 for one sequence and head, counted one by one."""
    n = 0
    for t in range(T):
        for j in range(T):
            if max(0, t - w + 1) <= j <= t:
                n += 1
    return n


@pytest.mark.parametrize("T,w", [(1, 1), (5, 1), (5, 2), (7, 7), (7, 9), (64, 13), (130, 128), (257, 64)])
def test_band_pairs_counts_every_in_window_pair(T, w):
    assert bench.band_pairs(T, w) == pairs_by_loop(T, w)


def out_positions(wl):
    """Output positions of each sequence, restated from the workload's out_mode."""
    if wl.out_mode == "last":
        return [[wl.T - 1]] * wl.B
    if wl.out_mode == "all":
        return [list(range(wl.T))] * wl.B
    kind, n = wl.out_mode
    assert kind == "span"
    return [list(range(wl.T - n, wl.T))] * wl.B


def test_prefill_flops_small_case_by_loop():
    wl = W.PrefillWorkload("acct", 2, 40, 4, 2, 64, 9, None, ("span", 6))
    pos = out_positions(wl)
    f = bench.prefill_flops(wl, [t for p in pos for t in p])
    per_pair = 4 * wl.d * wl.Hq
    assert f["swa"] == wl.B * pairs_by_loop(wl.T, wl.window) * per_pair
    # an output row at position t sees keys 0 .. t
    cross_pairs = sum(sum(1 for j in range(wl.T) if j <= t) for p in pos for t in p)
    assert f["cross"] == cross_pairs * per_pair
    assert f["total"] == f["swa"] + f["cross"]


@pytest.mark.parametrize("wl,swa,cross", [
    # closed forms: w(w+1)/2 + (T-w)w band pairs per (sequence, head); output
    # rows sum (t+1); times 4 d Hq (and B for the band)
    (W.PT_2K, 8 * 16 * 4 * 128 * (512 * 513 // 2 + (2048 - 512) * 512), 8 * 16 * 4 * 128 * (2048 * 2049 // 2)),
    (W.SFT_8K, 4 * 32 * 4 * 128 * (1024 * 1025 // 2 + (8192 - 1024) * 1024),
     4 * 32 * 4 * 128 * sum(t + 1 for t in range(8192 - 1024, 8192))),
    (W.PREFILL_128K, 32 * 4 * 128 * (4096 * 4097 // 2 + (131072 - 4096) * 4096), 32 * 4 * 128 * 131072),
], ids=lambda x: getattr(x, "name", ""))
def test_prefill_flops_named_workloads(wl, swa, cross):
    f = bench.prefill_flops(wl, [t for p in out_positions(wl) for t in p])
    assert f["swa"] == swa and f["cross"] == cross


def test_prefill_flops_match_the_stated_totals():
    """The useful work the benchmark reports, to the precision it is quoted at:
    1.977e11 (pre-training shape), 1.031e12 (fine-tuning), 8.661e12 (128K)."""
    for wl, total in ((W.PT_2K, 1.977e11), (W.SFT_8K, 1.031e12), (W.PREFILL_128K, 8.661e12)):
        f = bench.prefill_flops(wl, [t for p in out_positions(wl) for t in p])
        assert abs(f["total"] / total - 1) < 5e-4, (wl.name, f["total"])


def test_decode_bytes_count_each_cached_element_once_per_step():
    lens0, steps, Hkv, d = [0, 5, 17], 4, 2, 64
    by_loop = 0
    for s in range(steps):
        for L in lens0:
            keys = L + s + 1  # the cache after this step's append
            by_loop += keys * Hkv * d * 2 * 2  # K and V, bf16
    assert bench.decode_bytes(lens0, steps, Hkv, d) == by_loop


def test_decode_bytes_at_the_mean_length():
    """32 sequences at the mean history of U[16384, 32768] (24576 tokens), GQA 8
    kv heads, d = 128: about 3.22 GB per step."""
    gb = bench.decode_bytes([24576] * 32, 1, 8, 128) / 1e9
    assert abs(gb - 3.2215) < 1e-3, gb
