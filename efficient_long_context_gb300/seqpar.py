"""Sequence-parallel prefill: Eq. 4 and Eq. 5 with the token axis sharded
across ranks (one process per GPU).

The paper runs its longest prefills (64K to 1M tokens) on 8 GPUs (Orthros,
Sec. 4.5) without spelling out the split. Sharding the token axis into
contiguous chunks needs exactly two exchanges, and every arithmetic step
stays in the library's kernels:

* band rows (Eq. 4): rank r holds tokens [start_r, end_r). A row at position
  t needs keys back to t - w + 1, so each rank receives the last
  min(w - 1, start_r) keys and values before its chunk (a halo, point to point
  from the ranks that hold them) and runs ``orthros_prefill`` on
  [halo ; chunk]; the halo rows' own outputs are discarded (their windows
  are incomplete there, complete on their owner).
* output rows (Eq. 5): a row at position t attends keys 0 .. t, spread over
  every rank whose chunk starts at or before t. Each such rank computes the
  row over its own keys only (an output row of a separate call on its chunk),
  giving a partial (o_r, lse_r), and sends it point to point to the owner of
  position t, which merges them exactly:
  lse = log sum_r exp(lse_r), o = sum_r exp(lse_r - lse) o_r.

``attend`` is the single-device attention call (``orthros_prefill`` on a GPU);
it receives torch tensors of one rank and returns (o_base, lse_base, o_out,
lse_out). The exchange uses torch.distributed (NCCL between GPUs, gloo for
CPU tensors). A rank receives only the partials of the rows it owns, from the
ranks before it, and (without q_out) the raw queries of later ranks' rows,
from their owners, so the output-row exchange moves each partial and each
query only to where it is used, however many rows there are (one per
sequence when prefilling, an answer span when fine-tuning, every position
when pre-training).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def chunk_bounds(T: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, balanced chunk [start, end) of T tokens owned by `rank`."""
    return rank * T // world, (rank + 1) * T // world


def _world(group):
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(group), dist.get_rank(group)
    return 1, 0


def _exchange_halo(k, v, T, window, world, rank, group):
    """Keys/values of positions [start - H, start), H = min(window - 1, start),
    received from the ranks that own them; returns (k_halo, v_halo)."""
    B, _, Hkv, d = k.shape
    start, end = chunk_bounds(T, world, rank)
    H = min(window - 1, start)
    k_halo = k.new_empty((B, H, Hkv, d))
    v_halo = v.new_empty((B, H, Hkv, d))
    ops = []
    # what this rank sends: to every later rank s, the part of this chunk inside s's halo
    for s in range(rank + 1, world):
        s0, _ = chunk_bounds(T, world, s)
        lo, hi = max(start, s0 - min(window - 1, s0)), min(end, s0)
        if lo < hi:
            ops.append(dist.P2POp(dist.isend, k[:, lo - start:hi - start].contiguous(), s, group))
            ops.append(dist.P2POp(dist.isend, v[:, lo - start:hi - start].contiguous(), s, group))
    # what it receives: from every earlier rank r, the part of r's chunk inside this halo
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
        k_halo[:, a:a + kb.shape[1]] = kb
        v_halo[:, a:a + vb.shape[1]] = vb
    return k_halo, v_halo


def _owners(pos, T, world):
    """Rank that owns each position (-1 for positions outside [0, T))."""
    owner = torch.full_like(pos, -1)
    for s in range(world):
        s0, s1 = chunk_bounds(T, world, s)
        owner[(pos >= s0) & (pos < s1)] = s
    return owner


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


def _partials_to_owners(o_part, lse_part, pos, rows, T, world, rank, group):
    """Send this rank's partials of rows owned by later ranks to their owners
    and receive, from every earlier rank, its partials of the rows this rank
    owns (a rank holds a partial of every row at or after its chunk start).
    Returns the partials of this rank's rows, [rank + 1, len(rows), ...]:
    its own first, then those of ranks 0 .. rank-1."""
    owner = _owners(pos, T, world)
    ops = []
    for s in range(rank + 1, world):
        sel = torch.nonzero(owner == s).flatten().to(o_part.device)
        if len(sel):
            ops.append(dist.P2POp(dist.isend, o_part[sel].contiguous(), s, group))
            ops.append(dist.P2POp(dist.isend, lse_part[sel].contiguous(), s, group))
    rd = rows.to(o_part.device)
    o_in, l_in = [o_part[rd]], [lse_part[rd]]
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
               T, *, q_out=None, group=None, attend=None):
    """One rank's share of a sequence-parallel ``orthros_prefill``.

    q [B, C, Hq, d], k, v [B, C, Hkv, d]: this rank's chunk of every sequence
    (tokens chunk_bounds(T, world, rank)). out_indptr [B+1] / out_positions
    [n_out] (host, global positions) and q_out [n_out, Hq, d] (or None) are the
    same on every rank. Returns (o_base [B, C, Hq, d], lse_base [B, Hq, C],
    rows, o_out [len(rows), Hq, d], lse_out [len(rows), Hq]) where rows are the
    output-row indices whose position lies in this rank's chunk.
    """
    if attend is None:
        from . import orthros_prefill as attend  # noqa: N813
    world, rank = _world(group)
    B, C, Hq, d = q.shape
    start, end = chunk_bounds(T, world, rank)
    assert C == end - start, (C, start, end)
    indptr = torch.as_tensor(out_indptr, dtype=torch.int32).cpu()
    pos = torch.as_tensor(out_positions, dtype=torch.int64).cpu()
    n_out = int(indptr[-1])
    seq = torch.repeat_interleave(torch.arange(B), (indptr[1:] - indptr[:-1]).long()) if n_out else \
        torch.zeros(0, dtype=torch.long)

    # ---- band rows over [halo ; chunk] -------------------------------------------------
    if world > 1:
        k_halo, v_halo = _exchange_halo(k, v, T, window, world, rank, group)
    else:
        k_halo, v_halo = k[:, :0], v[:, :0]
    H = k_halo.shape[1]
    q_ext = torch.cat([q.new_zeros((B, H, Hq, d)), q], 1) if H else q
    k_ext = torch.cat([k_halo, k], 1) if H else k
    v_ext = torch.cat([v_halo, v], 1) if H else v
    no_rows = torch.zeros(B + 1, dtype=torch.int32)
    o_ext, lse_ext, _, _ = attend(q_ext.contiguous(), k_ext.contiguous(), v_ext.contiguous(), alpha_base, beta_base,
                                  alpha_out, beta_out, no_rows, pos.new_zeros(0).to(torch.int32).to(q.device),
                                  window, scale)
    o_base = o_ext[:, H:].contiguous()
    lse_base = lse_ext[:, :, H:].contiguous()

    # ---- output rows: partial over this chunk's keys, merged on the owner ---------------
    rows = torch.nonzero((pos >= start) & (pos < end)).flatten()
    if n_out == 0:
        return o_base, lse_base, rows, q.new_zeros((0, Hq, d)), lse_base.new_zeros((0, Hq))
    if q_out is None:
        # raw queries of the output rows this rank attends: its own, and those
        # of later ranks' rows, sent by their owners
        qo = q.new_zeros((n_out, Hq, d))
        if len(rows):
            qo[rows.to(q.device)] = q[seq[rows], pos[rows] - start]
        if world > 1:
            _queries_from_owners(qo, pos, rows, T, world, rank, group)
    else:
        qo = q_out
    mine = torch.nonzero(pos >= start).flatten()  # rows that see at least one key of this chunk
    o_part = torch.zeros((n_out, Hq, d), dtype=torch.float32, device=q.device)
    lse_part = torch.full((n_out, Hq), float("-inf"), dtype=torch.float32, device=q.device)
    if len(mine):
        m_seq = seq[mine]
        counts = torch.bincount(m_seq, minlength=B)
        m_indptr = torch.zeros(B + 1, dtype=torch.int32)
        m_indptr[1:] = torch.cumsum(counts, 0)
        order = torch.argsort(m_seq, stable=True)
        sel = mine[order]
        local_pos = (torch.clamp(pos[sel], max=end - 1) - start).to(torch.int32)
        # window 1 keeps the (discarded) base rows of this call to one key each
        _, _, o_r, lse_r = attend(q, k, v, alpha_base, beta_base, alpha_out, beta_out, m_indptr,
                                  local_pos.to(q.device), 1, scale, q_out=qo[sel.to(qo.device)].contiguous())
        o_part[sel.to(q.device)] = o_r.float()
        lse_part[sel.to(q.device)] = lse_r.float()
    if world > 1:
        o_rows, l_rows = _partials_to_owners(o_part, lse_part, pos, rows, T, world, rank, group)
    else:
        rd = rows.to(q.device)
        o_rows, l_rows = o_part[rd][None], lse_part[rd][None]
    lse = torch.logsumexp(l_rows, dim=0)       # [rows, Hq]; a partial without keys carries -inf
    wgt = torch.exp(l_rows - lse[None])        # [ranks, rows, Hq]
    o_out = (wgt[..., None] * o_rows).sum(0)
    return o_base, lse_base, rows, o_out.to(q.dtype), lse
