"""Sequence-parallel prefill (token axis sharded over ranks) against the oracle
on the whole sequence.

CPU: 1 to 4 gloo ranks, each rank's single-device arithmetic (its shard's band
rows and output-row partials, and the merge of the partials) done by the
oracle and a plain torch merge (test infrastructure), so what is checked is
the decomposition: the halo exchange (including halos that span several
ranks), the positions of the halo and of each rank's rows, and which partials
reach which owner. GPU: ranks 0..N-1 of a sequence run in one process
through the CUDA library (orthros_prefill_shard and orthros_merge_partials),
with halos and partials handed over in memory, against the oracle.
"""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [
    # (B, T, Hq, Hkv, d, window, positions per sequence, with q_out)
    (2, 37, 4, 2, 8, 5, [[36, 3, 20], [0, 12, 12, 30]], False),
    (1, 37, 4, 2, 8, 20, [[36, 5, 13, 24, 25]], True),   # halo wider than one chunk
    (2, 29, 2, 1, 8, 40, [[28], [7, 28]], False),        # window >= T: full causal
    (1, 30, 4, 4, 8, 3, [[]], False),                    # no output rows
    (2, 25, 4, 2, 8, 6, [list(range(25))] * 2, False),   # pre-training: every position an output row
]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case, seed=0):
    B, T, Hq, Hkv, d, w, lists, with_q_out = case
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, Hq, d), generator=g)
    k = torch.randn((B, T, Hkv, d), generator=g)
    v = torch.randn((B, T, Hkv, d), generator=g)
    aff = [1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g),
           1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g)]
    indptr = torch.zeros(B + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor([len(x) for x in lists]), 0)
    pos = torch.tensor([p for x in lists for p in x], dtype=torch.int32)
    n_out = int(indptr[-1])
    q_out = torch.randn((n_out, Hq, d), generator=g) if with_q_out else None
    return q, k, v, aff, indptr, pos, q_out


def oracle_attend(q, k, v, ab, bb, ao, bo, out_indptr, out_positions, window, scale, q_out=None, **_):
    """Single-device attention by the CPU oracle, in the shape of orthros_prefill's return."""
    import oracle

    f = lambda t: None if t is None else t.detach().cpu().float().numpy()  # noqa: E731
    res = oracle.prefill(f(q), f(k), f(v), f(ab), f(bb), f(ao), f(bo),
                         np.asarray(out_indptr, np.int32), np.asarray(out_positions.cpu(), np.int32),
                         window, scale, q_out=f(q_out))
    return tuple(torch.from_numpy(x) for x in res)


def oracle_shard(q, k_ext, v_ext, ab, bb, ao, bo, row_indptr, row_positions, window, scale, q_rows=None, **_):
    """orthros_prefill_shard's contract computed by the oracle: the chunk's
    band rows over [halo ; chunk] (halo rows given zero queries and dropped),
    and each row's partial over the chunk's keys only (a row before them is
    empty: o = 0, lse = -inf)."""
    B, C, Hq, d = q.shape
    Tkv = k_ext.shape[1]
    H = Tkv - C
    q_ext = torch.cat([q.new_zeros((B, H, Hq, d)), q], 1)
    no_rows = torch.zeros(B + 1, dtype=torch.int32)
    ob, lb, _, _ = oracle_attend(q_ext, k_ext, v_ext, ab, bb, ao, bo, no_rows, torch.zeros(0, dtype=torch.int32),
                                 window, scale)
    pos = torch.as_tensor(row_positions).cpu().long()
    n = len(pos)
    o_part = torch.zeros((n, Hq, d))
    lse_part = torch.full((n, Hq), float("-inf"))
    keep = torch.nonzero(pos >= H).flatten()
    if len(keep):
        indptr = torch.as_tensor(row_indptr).long()
        seq = torch.repeat_interleave(torch.arange(B), indptr[1:] - indptr[:-1])
        counts = torch.bincount(seq[keep], minlength=B)
        k_indptr = torch.zeros(B + 1, dtype=torch.int32)
        k_indptr[1:] = torch.cumsum(counts, 0)
        local = (torch.clamp(pos[keep], max=Tkv - 1) - H).to(torch.int32)  # rows past the chunk read all of it
        _, _, oo, lo = oracle_attend(q, k_ext[:, H:], v_ext[:, H:], ab, bb, ao, bo, k_indptr, local, 1, scale,
                                     q_out=q_rows[keep])
        o_part[keep] = oo.to(o_part.dtype)
        lse_part[keep] = lo.to(lse_part.dtype)
    return ob[:, H:], lb[:, :, H:], o_part, lse_part


def torch_merge(o_parts, lse_parts, dtype):
    """The merge identity in plain torch (lse = logsumexp, o = weighted sum)."""
    lse = torch.logsumexp(lse_parts, dim=0)
    w = torch.exp(lse_parts - lse[None])
    return (w[..., None] * o_parts).sum(0).to(dtype), lse


def _worker(rank, world, port, case, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    from efficient_long_context_gb300.seqpar import chunk_bounds, sp_prefill

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, T, Hq, Hkv, d, w, lists, with_q_out = case
        q, k, v, aff, indptr, pos, q_out = _inputs(case)
        s0, s1 = chunk_bounds(T, world, rank)
        scale = d ** -0.5
        ob, lb, rows, oo, lo = sp_prefill(q[:, s0:s1].contiguous(), k[:, s0:s1].contiguous(),
                                          v[:, s0:s1].contiguous(), *aff, indptr, pos, w, scale, T,
                                          q_out=q_out, attend=oracle_shard, merge=torch_merge)
        ref = oracle_attend(q, k, v, *aff, indptr, pos, w, scale, q_out=q_out)
        errs = dict(o_base=float((ob - ref[0][:, s0:s1]).abs().max()),
                    lse_base=float((lb - ref[1][:, :, s0:s1]).abs().max()))
        if len(rows):
            errs["o_out"] = float((oo - ref[2][rows]).abs().max())
            errs["lse_out"] = float((lo - ref[3][rows]).abs().max())
        out_q.put((rank, errs, rows.tolist()))
    finally:
        dist.destroy_process_group()


def _run_ranks(world, case):
    """Run `world` gloo ranks on one case; returns their (rank, errors, rows).
    Ranks still running when the results are in (or after a failure) are
    ended here, so a broken exchange cannot leave processes behind."""
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, case, out_q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = [out_q.get(timeout=180) for _ in procs]
        for p in procs:
            p.join(timeout=60)
            assert p.exitcode == 0
        return got
    finally:
        for p in procs:
            if p.is_alive():
                p.terminate()
                p.join(timeout=10)


@pytest.mark.parametrize("world", [1, 2, 3])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}T{c[1]}w{c[5]}{'qo' if c[7] else ''}")
def test_sequence_parallel_matches_whole_sequence(world, case, oracle_mod):
    got = _run_ranks(world, case)
    owned = sorted(r for _, _, rows in got for r in rows)
    n_out = sum(len(x) for x in case[6])
    assert owned == list(range(n_out))  # every output row has exactly one owner
    for rank, errs, _ in got:
        for name, e in errs.items():
            assert e <= 2e-5, f"rank {rank} {name}: {e}"


def _random_case(seed):
    """A seeded shape with halos that span several of four ranks and output
    rows (repeats included) spread over every owner."""
    import random

    r = random.Random(seed)
    B, T = r.choice([1, 2]), r.randint(9, 41)
    Hkv = r.choice([1, 2])
    Hq = Hkv * r.choice([1, 2, 3])
    w = r.choice([1, 2, r.randint(3, T), T + 3])
    lists = [sorted(r.choice(range(T)) for _ in range(r.randint(0, 6))) for _ in range(B)]
    return (B, T, Hq, Hkv, 8, w, lists, r.random() < 0.5)


@pytest.mark.parametrize("seed", range(6))
def test_sequence_parallel_random_shapes_four_ranks(seed, oracle_mod):
    case = _random_case(seed)
    got = _run_ranks(4, case)
    owned = sorted(r for _, _, rows in got for r in rows)
    assert owned == list(range(sum(len(x) for x in case[6]))), case
    for rank, errs, _ in got:
        for name, e in errs.items():
            assert e <= 2e-5, f"{case} rank {rank} {name}: {e}"


def test_local_ranks_match_oracle_on_cpu(oracle_mod):
    """sp_prefill_local (every rank in one process) with the oracle shard and
    the torch merge: the in-memory hand-over of halos and partials."""
    sys.path.insert(0, ROOT)
    from efficient_long_context_gb300.seqpar import sp_prefill_local

    for case in CASES:
        q, k, v, aff, indptr, pos, q_out = _inputs(case, seed=9)
        scale = case[4] ** -0.5
        ref = oracle_attend(q, k, v, *aff, indptr, pos, case[5], scale, q_out=q_out)
        for world in (1, 2, 4):
            got = sp_prefill_local(q, k, v, *aff, indptr, pos, case[5], scale, world, q_out=q_out,
                                   attend=oracle_shard, merge=torch_merge)
            for name, g, r in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref):
                assert float((g - r).abs().max()) <= 2e-5 if r.numel() else True, (case, world, name)


# GPU cases: (B, T, Hq, Hkv, d, window, positions per sequence, with q_out, worlds)
GPU_CASES = [
    # halos spanning several ranks (w - 1 > chunk), repeated positions, output rows on every rank
    (2, 700, 8, 2, 128, 400, [[699, 10, 150, 150, 351, 520], [5, 698]], False, (2, 3, 4)),
    # window >= T: every band row is full causal attention, halos of everything before the chunk
    (1, 530, 8, 2, 128, 4096, [[529, 0, 264, 265]], True, (2, 4)),
    # pre-training regime: every position an output row (tile kernel partials)
    (2, 512, 4, 4, 128, 96, [list(range(512))] * 2, False, (2, 3)),
    # GQA 32/8 at the prefilling regime's single last row, chunks of several key tiles
    (1, 2048, 32, 8, 128, 256, [[2047]], False, (4,)),
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", GPU_CASES, ids=lambda c: f"B{c[0]}T{c[1]}w{c[5]}n{len(c[6][0])}")
def test_local_ranks_on_gpu_match_oracle(case, oracle_mod):
    """Ranks 0..N-1 of one sequence-parallel prefill, one after the other on
    one GPU through the library: each rank's band rows over [halo ; chunk]
    and its output-row partials (orthros_prefill_shard), merged on each row's
    owner (orthros_merge_partials); compared with the oracle over the whole
    sequence at the parity contract's tolerances."""
    sys.path.insert(0, ROOT)
    from efficient_long_context_gb300.seqpar import sp_prefill_local
    from tests.parity_util import TOL

    *shape, worlds = case
    q, k, v, aff, indptr, pos, q_out = _inputs(tuple(shape), seed=4)
    dev = "cuda"
    qb, kb, vb = (t.to(torch.bfloat16) for t in (q, k, v))
    qob = q_out.to(torch.bfloat16) if q_out is not None else None
    window, scale = shape[5], shape[4] ** -0.5
    ref = oracle_attend(qb.float(), kb.float(), vb.float(), *aff, indptr, pos, window, scale,
                        q_out=qob.float() if qob is not None else None)
    tol_o, tol_l = TOL[torch.bfloat16]
    for world in worlds:
        got = sp_prefill_local(qb.to(dev), kb.to(dev), vb.to(dev), *(a.to(dev) for a in aff), indptr, pos, window,
                               scale, world, q_out=qob.to(dev) if qob is not None else None)
        torch.cuda.synchronize()
        for name, g, r, tol in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref,
                                   (tol_o, tol_l, tol_o, tol_l)):
            g = g.float().cpu()
            assert torch.isfinite(g).all(), (world, name)
            err = float((g - r).abs().max())
            assert err <= tol, f"world {world} {name}: {err}"


@pytest.mark.gpu
def test_shard_partials_on_gpu_match_oracle_shard(oracle_mod):
    """One shard call against the oracle's reading of its contract, rows
    before the chunk (empty partials), inside it and past it included; and
    the merge entry point against the merge identity."""
    import efficient_long_context_gb300 as ola
    from tests.parity_util import TOL

    g = torch.Generator().manual_seed(21)
    B, C, H, Hq, Hkv, d, w = 2, 300, 200, 8, 2, 128, 256
    q = torch.randn((B, C, Hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H + C, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H + C, Hkv, d), generator=g).to(torch.bfloat16)
    aff = [1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g),
           1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g)]
    indptr = torch.tensor([0, 4, 7], dtype=torch.int32)
    pos = torch.tensor([5, 200, 499, 900, 250, 200, 199], dtype=torch.int32)  # before, at, in, past the chunk
    q_rows = torch.randn((7, Hq, d), generator=g).to(torch.bfloat16)
    dev = "cuda"
    got = ola.orthros_prefill_shard(q.to(dev), k.to(dev), v.to(dev), *(a.to(dev) for a in aff), indptr, pos.to(dev),
                                    w, d ** -0.5, q_rows=q_rows.to(dev))
    ref = oracle_shard(q.float(), k.float(), v.float(), *aff, indptr, pos, w, d ** -0.5, q_rows=q_rows.float())
    tol_o, tol_l = TOL[torch.bfloat16]
    for name, a, r, tol in zip(("o_base", "lse_base", "o_part", "lse_part"), got, ref, (tol_o, tol_l, tol_o, tol_l)):
        a = a.float().cpu()
        fin = torch.isfinite(r)
        assert torch.equal(torch.isfinite(a), fin), name  # the empty rows' lse is -inf on both sides
        assert float((a[fin] - r[fin]).abs().max()) <= tol, name
    # merge: three partials of random rows, one of them empty for some rows
    parts = torch.randn((3, 5, Hq, d), generator=g)
    lses = torch.randn((3, 5, Hq), generator=g) * 3
    lses[1, 2] = float("-inf")
    parts[1, 2] = 0
    o, lse = ola.orthros_merge_partials(parts.to(dev), lses.to(dev), torch.float32)
    ro, rl = torch_merge(parts.double(), lses.double(), torch.float64)
    assert float((o.cpu().double() - ro).abs().max()) <= 1e-5
    assert float((lse.cpu().double() - rl).abs().max()) <= 1e-5


@pytest.mark.gpu
@pytest.mark.parametrize("w", [128, 4096], ids=["w128", "w4096_row_softmax"])
def test_shard_tile_path_rows_without_keys(oracle_mod, w):
    """Enough output rows that the sequence takes the tensor-core tile kernel
    (not the split-KV kernel), a third of them placed before the chunk's first
    key: those rows share tiles with rows that have keys, see only masked
    logits, and must come back exactly o = 0, lse = -inf."""
    import efficient_long_context_gb300 as ola
    from tests.parity_util import TOL

    g = torch.Generator().manual_seed(22)
    B, C, H, Hq, Hkv, d = 1, 256, 128, 8, 2, 128
    n = 1200  # more than 256 16-row groups of 4 query heads: the tile kernel
    q = torch.randn((B, C, Hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, H + C, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, H + C, Hkv, d), generator=g).to(torch.bfloat16)
    aff = [1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g),
           1 + 0.1 * torch.randn((Hq, d), generator=g), 0.1 * torch.randn((Hq, d), generator=g)]
    indptr = torch.tensor([0, n], dtype=torch.int32)
    pos = torch.sort(torch.randint(0, H + C, (n,), generator=g, dtype=torch.int32)).values
    assert int((pos < H).sum()) > n // 5
    q_rows = torch.randn((n, Hq, d), generator=g).to(torch.bfloat16)
    dev = "cuda"
    got = ola.orthros_prefill_shard(q.to(dev), k.to(dev), v.to(dev), *(a.to(dev) for a in aff), indptr, pos.to(dev),
                                    w, d ** -0.5, q_rows=q_rows.to(dev))
    ref = oracle_shard(q.float(), k.float(), v.float(), *aff, indptr, pos, w, d ** -0.5, q_rows=q_rows.float())
    tol_o, tol_l = TOL[torch.bfloat16]
    for name, a, r, tol in zip(("o_base", "lse_base", "o_part", "lse_part"), got, ref, (tol_o, tol_l, tol_o, tol_l)):
        a = a.float().cpu()
        fin = torch.isfinite(r)
        assert torch.equal(torch.isfinite(a), fin), name
        assert float((a[fin] - r[fin]).abs().max()) <= tol, name
    empty = pos < H
    assert torch.equal(got[2].cpu()[empty], torch.zeros_like(got[2].cpu()[empty]))  # exactly zero
    assert bool(torch.isneginf(got[3].cpu()[empty]).all())
