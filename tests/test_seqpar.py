"""Sequence-parallel prefill (token axis sharded over ranks) against the oracle
on the whole sequence.

CPU: 1, 2 and 3 gloo ranks, each rank's single-device attention done by the
oracle (test infrastructure), so what is checked is the decomposition: the
halo exchange (including halos that span several ranks), the discarded halo
rows, and the exact LSE merge of the output rows' partials. GPU: one rank
through the CUDA library.
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
                                          q_out=q_out, attend=oracle_attend)
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


@pytest.mark.gpu
def test_single_rank_on_gpu_matches_oracle(oracle_mod):
    sys.path.insert(0, ROOT)
    from efficient_long_context_gb300.seqpar import sp_prefill
    from tests.parity_util import TOL

    case = (2, 300, 8, 2, 128, 64, [[299, 10, 150], [5]], False)
    q, k, v, aff, indptr, pos, _ = _inputs(case, seed=4)
    dev = "cuda"
    qb, kb, vb = (t.to(torch.bfloat16) for t in (q, k, v))
    ob, lb, rows, oo, lo = sp_prefill(qb.to(dev), kb.to(dev), vb.to(dev), *(a.to(dev) for a in aff), indptr,
                                      pos, 64, 128 ** -0.5, 300)
    ref = oracle_attend(qb.float(), kb.float(), vb.float(), *aff, indptr, pos, 64, 128 ** -0.5)
    tol_o, tol_l = TOL[torch.bfloat16]
    assert float((ob.float().cpu() - ref[0]).abs().max()) <= tol_o
    assert float((lb.cpu() - ref[1]).abs().max()) <= tol_l
    assert rows.tolist() == [0, 1, 2, 3]
    assert float((oo.float().cpu() - ref[2]).abs().max()) <= tol_o
    assert float((lo.cpu() - ref[3]).abs().max()) <= tol_l
