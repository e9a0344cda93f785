"""Sequence-parallel prefill: Eq. 4 and Eq. 5 with the token axis sharded
across ranks (one process per GPU).

The paper runs its longest prefills (64K to 1M tokens) on 8 GPUs (Orthros,
Sec. 4.5) without spelling out the split. Sharding the token axis into
contiguous chunks needs exactly two exchanges; every arithmetic step runs in
the library's kernels:

* band rows (Eq. 4): rank r holds tokens [start_r, end_r). A row at position
  t needs keys back to t - w + 1, so the rank receives the last
  H = min(w - 1, start_r) keys and values before its chunk (the halo, point to
  point from the ranks that hold them) in front of its own, and
  ``orthros_prefill_shard`` runs its chunk's queries over [halo ; chunk]
  (query i at key position H + i): no halo row is computed.
* output rows (Eq. 5): a row at position t attends keys 0 .. t, spread over
  every rank whose chunk starts at or before t. The same call gives each such
  rank the row's normalised partial over its own chunk's keys (o_r, lse_r);
  the partials travel point to point to the owner of position t, and
  ``orthros_merge_partials`` combines them exactly
  (lse = log sum_r exp(lse_r), o = sum_r exp(lse_r - lse) o_r).

The rank step is split into functions that take the halo and the partials as
tensors, so the same arithmetic runs either across processes
(``sp_prefill``: torch.distributed point-to-point, NCCL between GPUs or gloo
for CPU tensors) or for all ranks of one sequence in one process
(``sp_prefill_local``: halos and partials handed over in memory).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def chunk_bounds(T: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced chunk [start, end) of T tokens owned by `rank`."""
    return rank * T // world, (rank + 1) * T // world


def halo_len(T: int, window: int, world: int, rank: int) -> int:
    """Keys before the chunk that its band rows read: min(w - 1, start)."""
    return min(window - 1, chunk_bounds(T, world, rank)[0])


def _world(group):
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(group), dist.get_rank(group)
    return 1, 0


def _owners(pos, T, world):
    """Rank that owns each position (-1 for positions outside [0, T))."""
    owner = torch.full_like(pos, -1)
    for s in range(world):
        s0, s1 = chunk_bounds(T, world, s)
        owner[(pos >= s0) & (pos < s1)] = s
    return owner


def _row_plan(out_indptr, out_positions, B):
    indptr = torch.as_tensor(out_indptr, dtype=torch.int32).cpu()
    pos = torch.as_tensor(out_positions, dtype=torch.int64).cpu()
    n_out = int(indptr[-1]) if indptr.numel() else 0
    seq = torch.repeat_interleave(torch.arange(B), (indptr[1:] - indptr[:-1]).long()) if n_out else \
        torch.zeros(0, dtype=torch.long)
    return indptr, pos, seq, n_out


def shard_rows(pos, seq, B, start, H):
    """The output rows a chunk starting at `start` holds keys for (position >=
    start), grouped by sequence: (row indices, host row indptr [B+1], their
    positions in the [halo ; chunk] buffer's coordinates)."""
    mine = torch.nonzero(pos >= start).flatten()
    order = torch.argsort(seq[mine], stable=True)
    sel = mine[order]
    counts = torch.bincount(seq[sel], minlength=B)
    indptr = torch.zeros(B + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(counts, 0)
    return sel, indptr, (pos[sel] - start + H).to(torch.int32)


def rank_attend(q, k_ext, v_ext, affines, pos, seq, start, q_rows_all, window, scale, attend=None):
    """One rank's arithmetic: band rows of its chunk over [halo ; chunk] and
    the partials of every output row at or after its chunk start.

    q [B, C, Hq, d] the chunk's queries; k_ext, v_ext [B, H + C, Hkv, d];
    q_rows_all [n_out, Hq, d] raw output-row queries (rows this rank does not
    hold keys for may be anything). Returns (o_base [B, C, Hq, d], lse_base
    [B, Hq, C], sel, o_part [len(sel), Hq, d] float, lse_part [len(sel), Hq])."""
    if attend is None:
        from . import orthros_prefill_shard as attend  # noqa: N813
    B, C, Hq, d = q.shape
    H = k_ext.shape[1] - C
    sel, r_indptr, r_pos = shard_rows(pos, seq, B, start, H)
    if C == 0:  # an empty chunk (more ranks than tokens) holds no keys
        return (q.new_empty((B, 0, Hq, d)), torch.empty((B, Hq, 0), dtype=torch.float32, device=q.device), sel,
                torch.zeros((len(sel), Hq, d), dtype=torch.float32, device=q.device),
                torch.full((len(sel), Hq), float("-inf"), dtype=torch.float32, device=q.device))
    q_rows = q_rows_all[sel.to(q_rows_all.device)].contiguous() if len(sel) else None
    o_base, lse_base, o_part, lse_part = attend(q, k_ext, v_ext, *affines, r_indptr, r_pos.to(q.device), window,
                                                scale, q_rows=q_rows)
    return o_base, lse_base, sel, o_part, lse_part


def merge_rows(o_parts, lse_parts, dtype, merge=None):
    """Exact merge of stacked partials [P, n, Hq, d] / [P, n, Hq] of the same rows."""
    if merge is None:
        from . import orthros_merge_partials as merge  # noqa: N813
    return merge(o_parts.contiguous(), lse_parts.contiguous(), dtype)


def _pick(sel, rows, device):
    """Positions inside `sel` (row indices) of each row index in `rows`."""
    where = {int(x): j for j, x in enumerate(sel.tolist())}
    return torch.tensor([where[int(x)] for x in rows.tolist()], dtype=torch.long, device=device)


def _local_queries(q, pos, seq, rows, start):
    """Raw queries of the output rows whose positions lie in this chunk."""
    return q[seq[rows].to(q.device), (pos[rows] - start).to(q.device)]


# ----------------------------------------------------------------------------
# all ranks of one sequence in one process (halos and partials in memory)
# ----------------------------------------------------------------------------
def sp_prefill_local(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions, window, scale,
                     world, *, q_out=None, attend=None, merge=None):
    """Run ranks 0 .. world-1 of a sequence-parallel prefill one after the
    other on the current device, with each rank's inputs cut from the whole
    tensors (its chunk, and its halo copied in front of it) and the partials
    handed to each row's owner in memory. Returns the whole-sequence
    (o_base [B,T,Hq,d], lse_base [B,Hq,T], o_out [n_out,Hq,d], lse_out [n_out,Hq])
    assembled from the ranks' results."""
    B, T, Hq, d = q.shape
    affines = (alpha_base, beta_base, alpha_out, beta_out)
    indptr, pos, seq, n_out = _row_plan(out_indptr, out_positions, B)
    if q_out is None and n_out:
        q_rows_all = q[seq.to(q.device), pos.to(q.device)]
    else:
        q_rows_all = q_out if q_out is not None else q.new_zeros((0, Hq, d))
    o_base = torch.empty_like(q)
    lse_base = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    owner = _owners(pos, T, world)
    parts = {}  # owner rank -> [(sel, o_part, lse_part) of every rank up to it]
    for r in range(world):
        start, end = chunk_bounds(T, world, r)
        if end == start:
            continue
        H = halo_len(T, window, world, r)
        k_ext = k[:, start - H:end].contiguous()  # [halo ; chunk], as received from the owners
        v_ext = v[:, start - H:end].contiguous()
        ob, lb, sel, op, lp = rank_attend(q[:, start:end].contiguous(), k_ext, v_ext, affines, pos, seq, start,
                                          q_rows_all, window, scale, attend)
        o_base[:, start:end] = ob
        lse_base[:, :, start:end] = lb
        for s in set(owner[sel].tolist()) - {-1}:
            parts.setdefault(s, []).append((sel, op, lp))
    o_out = q.new_empty((n_out, Hq, d))
    lse_out = torch.empty((n_out, Hq), dtype=torch.float32, device=q.device)
    for s, plist in parts.items():
        rows = torch.nonzero(owner == s).flatten()
        o_st = torch.empty((len(plist), len(rows), Hq, d), dtype=torch.float32, device=q.device)
        l_st = torch.empty((len(plist), len(rows), Hq), dtype=torch.float32, device=q.device)
        for i, (sel, op, lp) in enumerate(plist):
            # every rank up to the owner holds a partial of each of the owner's rows
            idx = _pick(sel, rows, q.device)
            o_st[i] = op[idx]
            l_st[i] = lp[idx]
        o, l = merge_rows(o_st, l_st, q.dtype, merge)
        rd = rows.to(q.device)
        o_out[rd] = o
        lse_out[rd] = l
    return o_base, lse_base, o_out, lse_out


# ----------------------------------------------------------------------------
# one rank per process (torch.distributed point to point)
# ----------------------------------------------------------------------------
def _exchange_halo(k, v, T, window, world, rank, group, k_ext, v_ext):
    """Receive positions [start - H, start) from the ranks that own them into
    k_ext[:, :H] / v_ext[:, :H], and send this chunk's share of every later
    rank's halo."""
    B, _, Hkv, d = k.shape
    start, end = chunk_bounds(T, world, rank)
    H = halo_len(T, window, world, rank)
    ops = []
    for s in range(rank + 1, world):
        s0, _ = chunk_bounds(T, world, s)
        lo, hi = max(start, s0 - halo_len(T, window, world, s)), min(end, s0)
        if lo < hi:
            ops.append(dist.P2POp(dist.isend, k[:, lo - start:hi - start].contiguous(), s, group))
            ops.append(dist.P2POp(dist.isend, v[:, lo - start:hi - start].contiguous(), s, group))
    recv = []
    for r in range(rank):
        r0, r1 = chunk_bounds(T, world, r)
        lo, hi = max(r0, start - H), min(r1, start)
        if lo < hi:
            kb = k.new_empty((B, hi - lo, Hkv, d))
            vb = v.new_empty((B, hi - lo, Hkv, d))
            ops.append(dist.P2POp(dist.irecv, kb, r, group))
            ops.append(dist.P2POp(dist.irecv, vb, r, group))
            recv.append((lo, kb, vb))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    for lo, kb, vb in recv:
        a = lo - (start - H)
        k_ext[:, a:a + kb.shape[1]] = kb
        v_ext[:, a:a + vb.shape[1]] = vb


def _queries_from_owners(qo, pos, rows, T, world, rank, group):
    """Fill qo's rows owned by later ranks with their raw queries: the owner of
    a row sends it to every earlier rank (each of those holds keys the row
    attends); this rank's own rows are already in qo."""
    owner = _owners(pos, T, world)
    ops = []
    if len(rows):
        mine = qo[rows.to(qo.device)].contiguous()
        for r in range(rank):
            ops.append(dist.P2POp(dist.isend, mine, r, group))
    recv = []
    for s in range(rank + 1, world):
        sel = torch.nonzero(owner == s).flatten().to(qo.device)
        if len(sel):
            buf = qo.new_empty((len(sel),) + tuple(qo.shape[1:]))
            ops.append(dist.P2POp(dist.irecv, buf, s, group))
            recv.append((sel, buf))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    for sel, buf in recv:
        qo[sel] = buf


def _partials_to_owners(sel, o_part, lse_part, pos, rows, T, world, rank, group):
    """Send this rank's partials of rows owned by later ranks to their owners
    and receive, from every earlier rank, its partials of the rows this rank
    owns (a rank holds a partial of every row at or after its chunk start).
    Returns the partials of this rank's rows, [rank + 1, len(rows), ...]: its
    own first, then those of ranks 0 .. rank-1."""
    owner = _owners(pos, T, world)
    dev = o_part.device
    ops = []
    for s in range(rank + 1, world):
        theirs = torch.nonzero(owner == s).flatten()
        if len(theirs):
            idx = _pick(sel, theirs, dev)
            ops.append(dist.P2POp(dist.isend, o_part[idx].contiguous(), s, group))
            ops.append(dist.P2POp(dist.isend, lse_part[idx].contiguous(), s, group))
    idx = _pick(sel, rows, dev)
    o_in, l_in = [o_part[idx]], [lse_part[idx]]
    if len(rows):
        for r in range(rank):
            ob = o_part.new_empty((len(rows),) + tuple(o_part.shape[1:]))
            lb = lse_part.new_empty((len(rows),) + tuple(lse_part.shape[1:]))
            ops.append(dist.P2POp(dist.irecv, ob, r, group))
            ops.append(dist.P2POp(dist.irecv, lb, r, group))
            o_in.append(ob)
            l_in.append(lb)
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return torch.stack(o_in), torch.stack(l_in)


def sp_prefill(q, k, v, alpha_base, beta_base, alpha_out, beta_out, out_indptr, out_positions, window, scale,
               T, *, q_out=None, group=None, attend=None, merge=None, kv_ext=None):
    """One rank's share of a sequence-parallel prefill, one rank per process.

    q [B, C, Hq, d], k, v [B, C, Hkv, d]: this rank's chunk of every sequence
    (tokens chunk_bounds(T, world, rank)). out_indptr [B+1] / out_positions
    [n_out] (host, global positions) and q_out [n_out, Hq, d] (or None) are the
    same on every rank. kv_ext: optional (k_ext, v_ext) [B, H + C, Hkv, d]
    buffers whose last C tokens already hold the chunk (H = halo_len(...));
    the halo is received into their front, so the chunk is never copied.
    Returns (o_base [B, C, Hq, d], lse_base [B, Hq, C], rows, o_out
    [len(rows), Hq, d], lse_out [len(rows), Hq]) where rows are the
    output-row indices whose position lies in this rank's chunk.
    """
    world, rank = _world(group)
    B, C, Hq, d = q.shape
    start, end = chunk_bounds(T, world, rank)
    assert C == end - start, (C, start, end)
    indptr, pos, seq, n_out = _row_plan(out_indptr, out_positions, B)
    H = halo_len(T, window, world, rank)
    if kv_ext is None:
        k_ext = k.new_empty((B, H + C) + tuple(k.shape[2:]))
        v_ext = v.new_empty((B, H + C) + tuple(v.shape[2:]))
        k_ext[:, H:] = k
        v_ext[:, H:] = v
    else:
        k_ext, v_ext = kv_ext
        assert k_ext.shape[1] == H + C and v_ext.shape[1] == H + C, (k_ext.shape, H, C)
    if world > 1:
        _exchange_halo(k, v, T, window, world, rank, group, k_ext, v_ext)

    rows = torch.nonzero((pos >= start) & (pos < end)).flatten()
    if q_out is None:
        # raw queries of the output rows this rank attends: its own, and those
        # of later ranks' rows, sent by their owners
        qo = q.new_zeros((n_out, Hq, d))
        if len(rows):
            qo[rows.to(q.device)] = _local_queries(q, pos, seq, rows, start)
        if world > 1:
            _queries_from_owners(qo, pos, rows, T, world, rank, group)
    else:
        qo = q_out
    o_base, lse_base, sel, o_part, lse_part = rank_attend(q, k_ext, v_ext, (alpha_base, beta_base, alpha_out,
                                                                              beta_out), pos, seq, start, qo,
                                                           window, scale, attend)
    if n_out == 0 or not len(rows):
        if world > 1 and n_out:
            _partials_to_owners(sel, o_part, lse_part, pos, rows, T, world, rank, group)
        return o_base, lse_base, rows, q.new_zeros((0, Hq, d)), lse_base.new_zeros((0, Hq))
    if world > 1:
        o_rows, l_rows = _partials_to_owners(sel, o_part, lse_part, pos, rows, T, world, rank, group)
    else:
        idx = _pick(sel, rows, o_part.device)
        o_rows, l_rows = o_part[idx][None], lse_part[idx][None]
    o_out, lse_out = merge_rows(o_rows, l_rows, q.dtype, merge)
    return o_base, lse_base, rows, o_out, lse_out
