"""Host logic of the split-KV plan: how many keys one work item covers and
how much workspace the partials take (no GPU needed).

Rule: an item covers the longest of 8192, 4096, ..., 512 keys that still gives
every SM three items; one partial slot (16 rows x (d + 2) floats) per
(group, chunk). Prefill and continuous batching plan their groups at launch,
so their workspace holds a bound over every group count up to the maximum;
the first test checks that bound exhaustively, the others that the library
sizes its workspace by the same rule.
"""
import pytest
import torch

import efficient_long_context_gb300 as ola

CHUNKS = (8192, 4096, 2048, 1024, 512)
STATUS_BYTES = 256
SLOT_ROWS = 16


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def cdiv(a, b):
    return -(-a // b)


def align(x, a=256):
    return cdiv(x, a) * a


def chunk_for(n_groups, keys, n_sm):
    for c in CHUNKS[:-1]:
        if n_groups * cdiv(keys, c) >= 3 * n_sm:
            return c
    return CHUNKS[-1]


def slots_bound(max_groups, keys, n_sm):
    lo = max_groups * cdiv(keys, CHUNKS[0])
    hi = max_groups * cdiv(keys, CHUNKS[-1])
    return min(hi, max(lo, 6 * n_sm))


def slot_bytes(d):
    return SLOT_ROWS * (d + 2) * 4


@pytest.mark.parametrize("n_sm", [8, 152])
@pytest.mark.parametrize("keys", [1, 100, 511, 512, 513, 2047, 4097, 8192, 8193, 30000, 131072])
def test_slot_bound_covers_every_group_count(n_sm, keys):
    for max_groups in (1, 3, 8, 40, 257):
        bound = slots_bound(max_groups, keys, n_sm)
        for n in range(1, max_groups + 1):
            c = chunk_for(n, keys, n_sm)
            assert n * cdiv(keys, c) <= bound, (n, max_groups, keys, c)


@pytest.mark.parametrize("B,Hkv,max_pages,page", [(32, 8, 514, 64), (1, 8, 512, 64), (6, 8, 320, 64), (3, 2, 9, 16)])
def test_decode_workspace_follows_the_rule(B, Hkv, max_pages, page):
    d = 128
    keys = max_pages * page
    c = chunk_for(B * Hkv, keys, sms())
    want = STATUS_BYTES + align(B * Hkv * cdiv(keys, c) * slot_bytes(d))
    assert ola.orthros_decode_workspace_size(B, 32 if Hkv == 8 else 4, Hkv, d, max_pages, page) == want


def test_decode_chunk_choice_at_the_benchmark_shapes():
    """32 sequences x 8 kv heads over 32K-token page tables take 8192-key items;
    one sequence takes short ones so that it still spreads over the GPU."""
    assert chunk_for(32 * 8, 514 * 64, 152) == 8192
    assert chunk_for(8, 32768, 152) == 512


@pytest.mark.parametrize("B,T,Hkv,n_out", [(1, 131072, 8, 1), (4, 8192, 8, 1024), (2, 300, 2, 5)])
def test_prefill_workspace_follows_the_rule(B, T, Hkv, n_out):
    d, Hq = 128, 4 * Hkv
    max_groups = min(n_out, 16 * B) * Hkv
    blocks = Hq * (B * (cdiv(T, 128) + 1) + cdiv(n_out, 128) + 2 * B)  # bound on the tile kernel's row blocks
    want = (STATUS_BYTES + align(4 * (3 * (B + 1) + 3 * max_groups)) + align(B * T * Hkv * d * 2)
            + align(slots_bound(max_groups, T, sms()) * slot_bytes(d))
            + align(4 * cdiv(blocks, 32)) + align(4 * (B * Hq * T + n_out * Hq))  # second-pass bitmap and list
            + align(4 * 4 * Hq * d))  # the scaled affine copies
    assert ola.orthros_prefill_workspace_size(B, T, Hq, Hkv, d, n_out, 4096) == want
