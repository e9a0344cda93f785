"""Pins for the CPU oracle: checks against facts fixed by the paper and by mathematics.

Each ``pin_*`` function takes an oracle object (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with the fact it pins. The same
functions run against the real oracle (tests/test_oracle.py) and against
builds of the oracle source with a planted mistake (tests/test_oracle_mutants.py),
which must each fail at least one pin.

Sources of truth used here (none of them re-types the oracle's loops):
  * brute force: the dense T x T score matrix with a boolean band mask and the
    library softmax / logsumexp of scipy, on tiny inputs;
  * closed forms: window 1, zero query (uniform weights), a hand-worked example;
  * library routines the method reduces to: with identity affines the base
    stream is banded causal attention, i.e. torch's scaled_dot_product_attention
    with a band mask (Sec. 2.1 Eq. 1 and Eq. 3 of the Orthros paper);
  * invariances stated or implied by the paper: window >= T recovers full
    attention (third-party reproduction page, conversion check), grouped heads
    equal replicated heads, physical page order does not matter, prefill then
    decode equals one longer prefill (Sec. 3.2 "strict algorithmic consistency").
"""
from __future__ import annotations

import math

import numpy as np
import torch
from scipy.special import logsumexp, softmax

from efficient_long_context_gb300.workloads import make_affines

RTOL_EXACT = 1e-9  # double vs double


def rng_inputs(seed, B, T, Hq, Hkv, d, k_offset=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, T, Hq, d), generator=g).numpy()
    k = torch.randn((B, T, Hkv, d), generator=g).numpy()
    v = torch.randn((B, T, Hkv, d), generator=g).numpy()
    ab, bb, ao, bo = (x.numpy() for x in make_affines(g, Hq, d))
    if k_offset is not None:
        k = (k + k_offset[None, None]).astype(np.float32)
    return q, k, v, ab, bb, ao, bo


def csr(lists):
    indptr = np.zeros(len(lists) + 1, np.int32)
    indptr[1:] = np.cumsum([len(x) for x in lists])
    pos = np.concatenate([np.asarray(x, np.int32) for x in lists]) if lists else np.zeros(0, np.int32)
    return indptr, pos.astype(np.int32)


def brute_rows(qraw, alpha, beta, K, V, positions, lo_fn, scale):
    """Dense masked softmax attention of a set of query rows of one head.

    qraw [R, d] raw queries, K/V [T, d]; row r sits at positions[r] and sees
    keys j with lo_fn(t) <= j <= t. Builds the full R x T score matrix,
    puts -inf outside the band and calls the library softmax.
    """
    qa = qraw.astype(np.float64) * alpha.astype(np.float64) + beta.astype(np.float64)
    S = scale * (qa @ K.astype(np.float64).T)
    T = K.shape[0]
    j = np.arange(T)[None, :]
    t = np.asarray(positions)[:, None]
    lo = np.array([lo_fn(int(x)) for x in positions])[:, None]
    mask = (j >= lo) & (j <= t)
    S = np.where(mask, S, -np.inf)
    P = softmax(S, axis=1)
    return P @ V.astype(np.float64), logsumexp(S, axis=1)


def brute_prefill(q, k, v, ab, bb, ao, bo, indptr, pos, window, scale, q_out=None):
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    o_b = np.zeros((B, T, Hq, d))
    l_b = np.zeros((B, Hq, T))
    n_out = int(indptr[-1])
    o_o = np.zeros((n_out, Hq, d))
    l_o = np.zeros((n_out, Hq))
    for b in range(B):
        for h in range(Hq):
            kv = h // g
            o, l = brute_rows(q[b, :, h], ab[h], bb[h], k[b, :, kv], v[b, :, kv], np.arange(T),
                              lambda t: max(0, t - window + 1), scale)
            o_b[b, :, h] = o
            l_b[b, h] = l
            r0, r1 = int(indptr[b]), int(indptr[b + 1])
            if r1 > r0:
                p = pos[r0:r1]
                qr = q_out[r0:r1, h] if q_out is not None else q[b, p, h]
                o, l = brute_rows(qr, ao[h], bo[h], k[b, :, kv], v[b, :, kv], p, lambda t: 0, scale)
                o_o[r0:r1, h] = o
                l_o[r0:r1, h] = l
    return o_b, l_b, o_o, l_o


def _close(a, b, tol=RTOL_EXACT, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    if a.size:
        err = float(np.max(np.abs(a - b)))
        assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


BRUTE_CASES = [
    # (B, T, Hq, Hkv, d, window)
    (1, 1, 1, 1, 8, 1),
    (1, 17, 1, 1, 8, 1),
    (1, 17, 4, 2, 8, 2),
    (2, 17, 8, 2, 16, 7),
    (1, 40, 4, 2, 16, 39),
    (1, 40, 4, 4, 8, 40),
    (2, 33, 8, 2, 8, 38),
    (1, 64, 2, 1, 16, 5),
]


def pin_brute_force_prefill(orc, cases=BRUTE_CASES, seed=11):
    for i, (B, T, Hq, Hkv, d, w) in enumerate(cases):
        q, k, v, ab, bb, ao, bo = rng_inputs(seed + i, B, T, Hq, Hkv, d)
        r = np.random.default_rng(seed + i)
        lists = [sorted(r.choice(T, size=r.integers(0, T + 1), replace=False).tolist()) for _ in range(B)]
        lists[0] = sorted(set(lists[0]) | {T - 1})  # the prefill regime's last prompt token
        indptr, pos = csr(lists)
        scale = 1.0 / math.sqrt(d)
        for q_out in (None, torch.randn((int(indptr[-1]), Hq, d), generator=torch.Generator().manual_seed(i)).numpy()):
            got = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, scale, q_out=q_out)
            ref = brute_prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, scale, q_out=q_out)
            for name, a, b in zip(("o_base", "lse_base", "o_out", "lse_out"), got, ref):
                _close(a, b, what=f"case {i} {name}")


def pin_row_subset(orc):
    B, T, Hq, Hkv, d, w = 2, 30, 4, 2, 8, 9
    q, k, v, ab, bb, ao, bo = rng_inputs(3, B, T, Hq, Hkv, d)
    indptr, pos = csr([[], [29]])
    full = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3)
    rows = np.array([0, 8, 9, 29], np.int32)
    sub = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3, base_rows=rows)
    _close(sub[0], full[0][:, rows], what="o_base subset")
    _close(sub[1], full[1][:, :, rows], what="lse_base subset")


def pin_window_covers_all(orc):
    """w >= T: every base row equals the output row at the same position
    when both streams share their affine (full causal attention, Eq. 1)."""
    B, T, Hq, Hkv, d = 2, 23, 4, 2, 8
    q, k, v, ab, bb, _, _ = rng_inputs(5, B, T, Hq, Hkv, d)
    indptr, pos = csr([list(range(T))] * B)
    for w in (T, T + 3):
        ob, lb, oo, lo = orc.prefill(q, k, v, ab, bb, ab, bb, indptr, pos, w, 0.25)
        _close(oo.reshape(B, T, Hq, d), ob, what="o full window")
        _close(lo.reshape(B, T, Hq).transpose(0, 2, 1), lb, what="lse full window")


def pin_identity_affine_is_sdpa(orc):
    """alpha = 1, beta = 0 (the paper's 'w/o SO' ablation): the base stream is
    banded causal attention and the output stream causal attention; checked
    against torch's scaled_dot_product_attention with an explicit mask."""
    B, T, Hq, Hkv, d, w = 1, 37, 4, 4, 16, 6
    q, k, v, *_ = rng_inputs(9, B, T, Hq, Hkv, d)
    one = np.ones((Hq, d), np.float32)
    zero = np.zeros((Hq, d), np.float32)
    indptr, pos = csr([list(range(T))])
    ob, lb, oo, lo = orc.prefill(q, k, v, one, zero, one, zero, indptr, pos, w, d ** -0.5)
    qt = torch.from_numpy(q).double().permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).double().permute(0, 2, 1, 3)
    vt = torch.from_numpy(v).double().permute(0, 2, 1, 3)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    band = (j <= i) & (j > i - w)
    causal = j <= i
    ref_b = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=band)
    ref_o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=causal)
    _close(ob, ref_b.permute(0, 2, 1, 3).numpy(), 1e-10, "sdpa band")
    _close(oo.reshape(B, T, Hq, d), ref_o.permute(0, 2, 1, 3).numpy(), 1e-10, "sdpa causal")


def pin_window_one(orc):
    """w = 1: every base row attends only itself: o = v_t, lse = scale q_t.k_t."""
    B, T, Hq, Hkv, d = 1, 12, 2, 1, 8
    q, k, v, ab, bb, ao, bo = rng_inputs(13, B, T, Hq, Hkv, d)
    indptr, pos = csr([[]])
    ob, lb, _, _ = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, 1, 0.7)
    for h in range(Hq):
        _close(ob[0, :, h], v[0, :, 0], what="w=1 o")
        qa = q[0, :, h].astype(np.float64) * ab[h] + bb[h]
        _close(lb[0, h], 0.7 * np.sum(qa * k[0, :, 0], axis=1), 1e-9, "w=1 lse")


def pin_zero_query_uniform(orc):
    """alpha = beta = 0: all logits are 0, weights are uniform over the window:
    o_t = mean of v over [max(0,t-w+1), t] and lse = ln(min(t+1, w)).
    Pins both window edges exactly."""
    B, T, Hq, Hkv, d, w = 1, 20, 2, 1, 4, 6
    q, k, v, *_ = rng_inputs(17, B, T, Hq, Hkv, d)
    z = np.zeros((Hq, d), np.float32)
    indptr, pos = csr([[0, 7, 19]])
    ob, lb, oo, lo = orc.prefill(q, k, v, z, z, z, z, indptr, pos, w, 1.0)
    for t in range(T):
        lo_t = max(0, t - w + 1)
        mean = v[0, lo_t:t + 1, 0].astype(np.float64).mean(axis=0)
        for h in range(Hq):
            _close(ob[0, t, h], mean, 1e-12, f"uniform o t={t}")
            _close(lb[0, h, t], math.log(t - lo_t + 1), 1e-12, f"uniform lse t={t}")
    for r, t in enumerate([0, 7, 19]):
        _close(oo[r, 0], v[0, :t + 1, 0].astype(np.float64).mean(axis=0), 1e-12, "uniform out o")
        _close(lo[r, 0], math.log(t + 1), 1e-12, "uniform out lse")


def pin_key_offset_shift(orc):
    """A per-channel offset c added to every key shifts every logit of a row by
    scale * qa.c: softmax weights (so o) are unchanged and lse moves by exactly that.
    Keys and offsets are put on coarse binary grids so that k + c is exact in float32."""
    B, T, Hq, Hkv, d, w = 1, 25, 4, 2, 8, 5
    q, k, v, ab, bb, ao, bo = rng_inputs(19, B, T, Hq, Hkv, d)
    k = (np.round(k * 1024.0) / 1024.0).astype(np.float32)
    c = (np.round(0.5 * np.random.default_rng(1).standard_normal((Hkv, d)) * 16.0) / 16.0).astype(np.float32)
    k2 = (k + c[None, None]).astype(np.float32)
    assert np.array_equal(k2.astype(np.float64) - k.astype(np.float64),
                          np.broadcast_to(c[None, None].astype(np.float64), k.shape))
    indptr, pos = csr([[3, 24]])
    a = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.35)
    b_ = orc.prefill(q, k2, v, ab, bb, ao, bo, indptr, pos, w, 0.35)
    _close(b_[0], a[0], 1e-11, "offset o_base")
    _close(b_[2], a[2], 1e-11, "offset o_out")
    for h in range(Hq):
        kv = h // (Hq // Hkv)
        qa = q[0, :, h].astype(np.float64) * ab[h] + bb[h]
        _close(b_[1][0, h] - a[1][0, h], 0.35 * (qa @ c[kv].astype(np.float64)), 1e-11, "offset lse_base")
        qa_o = q[0, [3, 24], h].astype(np.float64) * ao[h] + bo[h]
        _close(b_[3][:, h] - a[3][:, h], 0.35 * (qa_o @ c[kv].astype(np.float64)), 1e-11, "offset lse_out")


def pin_gqa_equals_replicated(orc):
    """Grouped K/V heads (kv = h // (Hq/Hkv)) equal MHA with each K/V head copied
    to its group of query heads."""
    B, T, Hq, Hkv, d, w = 2, 19, 8, 2, 8, 4
    q, k, v, ab, bb, ao, bo = rng_inputs(23, B, T, Hq, Hkv, d)
    g = Hq // Hkv
    k_rep = np.repeat(k, g, axis=2)
    v_rep = np.repeat(v, g, axis=2)
    indptr, pos = csr([[18], [0, 5, 18]])
    a = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3)
    b_ = orc.prefill(q, k_rep, v_rep, ab, bb, ao, bo, indptr, pos, w, 0.3)
    for x, y, n in zip(a, b_, ("o_base", "lse_base", "o_out", "lse_out")):
        _close(x, y, 1e-12, "gqa " + n)


def _paged_from_seq(k_seq, v_seq, lens, page_size, extra, rng):
    """Scatter per-sequence K/V [B][L_b, Hkv, d] into a shuffled page pool."""
    B = len(k_seq)
    Hkv, d = k_seq[0].shape[1], k_seq[0].shape[2]
    pages_per = [(int(lens[b]) + extra + page_size - 1) // page_size for b in range(B)]
    num_pages = sum(pages_per)
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, max(pages_per)), -1, np.int32)
    at = 0
    for b in range(B):
        bt[b, :pages_per[b]] = perm[at:at + pages_per[b]]
        at += pages_per[b]
    kc = rng.standard_normal((num_pages, page_size, Hkv, d)).astype(np.float32)
    vc = rng.standard_normal((num_pages, page_size, Hkv, d)).astype(np.float32)
    for b in range(B):
        for j in range(int(lens[b])):
            kc[bt[b, j // page_size], j % page_size] = k_seq[b][j]
            vc[bt[b, j // page_size], j % page_size] = v_seq[b][j]
    return kc, vc, bt


def pin_decode_brute_force(orc):
    """One decoding step against dense brute force over the logical sequence
    (history plus the appended token): base row keys max(0,L-w+1)..L, output
    row keys 0..L, both after the append (Sec. 3.2 'Decoding')."""
    rng = np.random.default_rng(29)
    B, Hq, Hkv, d, P = 3, 4, 2, 8, 4
    lens = np.array([0, 5, 13], np.int32)
    for w in (1, 3, 6, 50):
        g = torch.Generator().manual_seed(w)
        ab, bb, ao, bo = (x.numpy() for x in make_affines(g, Hq, d))
        k_seq = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
        v_seq = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
        kc, vc, bt = _paged_from_seq(k_seq, v_seq, lens, P, 1, rng)
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        qo = rng.standard_normal((B, Hq, d)).astype(np.float32)
        kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
        for q_out in (None, qo):
            kc2, vc2 = kc.copy(), vc.copy()
            ob, lb, oo, lo = orc.decode(q, kn, vn, kc2, vc2, bt, lens, ab, bb, ao, bo, w, 0.4, q_out=q_out)
            for b in range(B):
                L = int(lens[b])
                K = np.concatenate([k_seq[b], kn[b][None]], 0)
                V = np.concatenate([v_seq[b], vn[b][None]], 0)
                for h in range(Hq):
                    kv = h // (Hq // Hkv)
                    o, l = brute_rows(q[b, h][None], ab[h], bb[h], K[:, kv], V[:, kv], [L],
                                      lambda t: max(0, t - w + 1), 0.4)
                    _close(ob[b, h], o[0], what="decode base o")
                    _close(lb[b, h], l[0], what="decode base lse")
                    qr = (q_out if q_out is not None else q)[b, h][None]
                    o, l = brute_rows(qr, ao[h], bo[h], K[:, kv], V[:, kv], [L], lambda t: 0, 0.4)
                    _close(oo[b, h], o[0], what="decode out o")
                    _close(lo[b, h], l[0], what="decode out lse")
                # the append landed where the block table says
                pg = bt[b, L // P]
                assert np.array_equal(kc2[pg, L % P], kn[b]) and np.array_equal(vc2[pg, L % P], vn[b])


def pin_decode_page_permutation(orc):
    """Relabelling physical pages (and moving their contents) changes nothing."""
    rng = np.random.default_rng(31)
    B, Hq, Hkv, d, P, w = 2, 4, 2, 8, 4, 5
    lens = np.array([9, 14], np.int32)
    k_seq = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    v_seq = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    kc, vc, bt = _paged_from_seq(k_seq, v_seq, lens, P, 1, rng)
    ab, bb, ao, bo = (x.numpy() for x in make_affines(torch.Generator().manual_seed(2), Hq, d))
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    kn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((B, Hkv, d)).astype(np.float32)
    a = orc.decode(q, kn, vn, kc.copy(), vc.copy(), bt, lens, ab, bb, ao, bo, w, 0.3)
    perm = rng.permutation(kc.shape[0])
    inv = np.argsort(perm)
    kc_p = kc[perm].copy()
    vc_p = vc[perm].copy()
    bt_p = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    b_ = orc.decode(q, kn, vn, kc_p, vc_p, bt_p, lens, ab, bb, ao, bo, w, 0.3)
    for x, y in zip(a, b_):
        _close(x, y, 0.0, "page permutation")


def pin_prefill_decode_consistency(orc):
    """Sec. 3.2: one formulation for every regime. A prefill over T0 tokens,
    then N decoding steps that append tokens T0..T0+N-1, gives at every new
    position the same base output as one prefill over T0+N tokens, and the same
    output-stream result as that prefill with output rows at those positions."""
    B, T0, N, Hq, Hkv, d, w, P = 2, 11, 6, 4, 2, 8, 5, 4
    T = T0 + N
    q, k, v, ab, bb, ao, bo = rng_inputs(37, B, T, Hq, Hkv, d)
    indptr, pos = csr([list(range(T0 - 1, T))] * B)
    full = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.33)
    rng = np.random.default_rng(3)
    lens = np.full(B, T0, np.int32)
    kc, vc, bt = _paged_from_seq([k[b, :T0] for b in range(B)], [v[b, :T0] for b in range(B)], lens, P, N, rng)
    for s in range(N):
        t = T0 + s
        ob, lb, oo, lo = orc.decode(q[:, t], k[:, t], v[:, t], kc, vc, bt, lens, ab, bb, ao, bo, w, 0.33)
        _close(ob, full[0][:, t], 1e-12, f"consistency base o step {s}")
        _close(lb, full[1][:, :, t], 1e-12, f"consistency base lse step {s}")
        rows = indptr[:-1] + (t - (T0 - 1))
        _close(oo, full[2][rows], 1e-12, f"consistency out o step {s}")
        _close(lo, full[3][rows], 1e-12, f"consistency out lse step {s}")
        lens = lens + 1


def pin_hand_worked(orc):
    """The closed-form example in tests/golden/hand_worked.txt (derivation there)."""
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")
    with open(path) as f:
        g = json.load(f)
    q = np.array(g["q"], np.float32)[None, :, None, :]
    k = np.array(g["k"], np.float32)[None, :, None, :]
    v = np.array(g["v"], np.float32)[None, :, None, :]
    one = np.ones((1, q.shape[-1]), np.float32)
    zero = np.zeros((1, q.shape[-1]), np.float32)
    indptr, pos = csr([g["out_positions"]])
    ob, lb, oo, lo = orc.prefill(q, k, v, one, zero, one, zero, indptr, pos, g["window"], g["scale"])
    _close(ob[0, :, 0], np.array(g["o_base"]), 1e-12, "hand o_base")
    _close(lb[0, 0], np.log(np.array(g["exp_lse_base"])), 1e-12, "hand lse_base")
    _close(oo[:, 0], np.array(g["o_out"]), 1e-12, "hand o_out")
    _close(lo[:, 0], np.log(np.array(g["exp_lse_out"])), 1e-12, "hand lse_out")


# ---------------------------------------------------------------------------
# Shared Q/K/V projection (the step upstream of the hot path)
# ---------------------------------------------------------------------------

def pin_project_selection_weight(orc):
    """A weight whose every output column selects one input column times a
    power of two: each projection output is that input times the factor, so q
    is alpha * (s x_c) + beta and k, v are s x_c, exactly."""
    rng = np.random.default_rng(51)
    n_base, n_out, d_model, Hq, Hkv, d = 3, 2, 24, 4, 2, 4
    N = (Hq + 2 * Hkv) * d
    x = rng.standard_normal((n_base + n_out, d_model)).astype(np.float32)
    sel = rng.integers(0, d_model, N)
    fac = (2.0 ** rng.integers(-2, 3, N)).astype(np.float32)
    w_t = np.zeros((N, d_model), np.float32)
    w_t[np.arange(N), sel] = fac
    ab, bb, ao, bo = (a.numpy() for a in make_affines(torch.Generator().manual_seed(3), Hq, d))
    qb, qo, k, v = orc.qkv_project(x, n_base, w_t, Hq, Hkv, d, ab, bb, ao, bo)
    y = x.astype(np.float64)[:, sel] * fac.astype(np.float64)
    Nq, Nkv = Hq * d, Hkv * d
    _close(qb.reshape(n_base, Nq), ab.reshape(-1) * y[:n_base, :Nq] + bb.reshape(-1), 1e-15, "select q_base")
    _close(qo.reshape(n_out, Nq), ao.reshape(-1) * y[n_base:, :Nq] + bo.reshape(-1), 1e-15, "select q_out")
    _close(k.reshape(n_base, Nkv), y[:n_base, Nq:Nq + Nkv], 0.0, "select k")
    _close(v.reshape(n_base, Nkv), y[:n_base, Nq + Nkv:], 0.0, "select v")


def pin_project_rank_one(orc):
    """w_t[j, c] = a_j b_c: every output is a_j (x . b), with the dot product
    taken by numpy; values on a binary grid so all products are exact."""
    rng = np.random.default_rng(53)
    n_base, n_out, d_model, Hq, Hkv, d = 2, 1, 40, 2, 1, 8
    N = (Hq + 2 * Hkv) * d
    x = (np.round(rng.standard_normal((n_base + n_out, d_model)) * 8) / 8).astype(np.float32)
    a = (np.round(rng.standard_normal(N) * 4) / 4).astype(np.float32)
    b = (np.round(rng.standard_normal(d_model) * 4) / 4).astype(np.float32)
    w_t = np.outer(a, b).astype(np.float32)
    one = np.ones((Hq, d), np.float32)
    zero = np.zeros((Hq, d), np.float32)
    qb, qo, k, v = orc.qkv_project(x, n_base, w_t, Hq, Hkv, d, one, zero, one, zero)
    y = np.outer(x.astype(np.float64) @ b.astype(np.float64), a.astype(np.float64))
    Nq, Nkv = Hq * d, Hkv * d
    _close(qb.reshape(n_base, Nq), y[:n_base, :Nq], 1e-12, "rank-1 q_base")
    _close(qo.reshape(n_out, Nq), y[n_base:, :Nq], 1e-12, "rank-1 q_out")
    _close(k.reshape(n_base, Nkv), y[:n_base, Nq:Nq + Nkv], 1e-12, "rank-1 k")
    _close(v.reshape(n_base, Nkv), y[:n_base, Nq + Nkv:], 1e-12, "rank-1 v")


def pin_project_feeds_decode(orc):
    """Alg. 1 line 5 applies each stream's affine once: projecting a decoding
    pair with the affines in the projection and then decoding with identity
    affines equals decoding the raw projections with the stream affines; the
    projection's cache writes are the decoding step's appends."""
    rng = np.random.default_rng(57)
    B, Hq, Hkv, d, P, w, d_model = 3, 4, 2, 8, 4, 5, 16
    lens = np.array([2, 7, 0], np.int32)
    k_hist = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    v_hist = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    kc, vc, bt = _paged_from_seq(k_hist, v_hist, lens, P, 1, rng)
    x = rng.standard_normal((2 * B, d_model)).astype(np.float32)
    w_t = (0.25 * rng.standard_normal(((Hq + 2 * Hkv) * d, d_model))).astype(np.float32)
    ab, bb, ao, bo = (a.numpy() for a in make_affines(torch.Generator().manual_seed(6), Hq, d))
    one = np.ones((Hq, d), np.float32)
    zero = np.zeros((Hq, d), np.float32)
    kc1, vc1 = kc.copy(), vc.copy()
    qb, qo, k, v = orc.qkv_project(x, B, w_t, Hq, Hkv, d, ab, bb, ao, bo, k_cache=kc1, v_cache=vc1,
                                   block_table=bt, token_seq=np.arange(B, dtype=np.int32), token_pos=lens)
    raw = orc.qkv_project(x, B, w_t, Hq, Hkv, d, one, zero, one, zero)
    kc2, vc2 = kc.copy(), vc.copy()
    a = orc.decode(qb.astype(np.float32), k.astype(np.float32), v.astype(np.float32), kc2, vc2, bt, lens,
                   one, zero, one, zero, w, 0.4, q_out=qo.astype(np.float32))
    kc3, vc3 = kc.copy(), vc.copy()
    b_ = orc.decode(raw[0].astype(np.float32), raw[2].astype(np.float32), raw[3].astype(np.float32), kc3, vc3, bt,
                    lens, ab, bb, ao, bo, w, 0.4, q_out=raw[1].astype(np.float32))
    for x1, x2, n in zip(a, b_, ("o_base", "lse_base", "o_out", "lse_out")):
        _close(x1, x2, 2e-6, "projection affine " + n)  # the affine runs in float32 on one side
    assert np.array_equal(kc1, kc2) and np.array_equal(vc1, vc2), "projection cache writes != decode appends"


# ---------------------------------------------------------------------------
# Continuous-batching step (appends of several tokens per sequence)
# ---------------------------------------------------------------------------

def _extend_setup(seed, B, Hq, Hkv, d, P, lens, news, extra=0):
    """Random history of lens[b] tokens per sequence in a shuffled page pool
    with room for news[b] more; returns the logical per-sequence K/V too."""
    rng = np.random.default_rng(seed)
    k_hist = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    v_hist = [rng.standard_normal((int(L), Hkv, d)).astype(np.float32) for L in lens]
    kc, vc, bt = _paged_from_seq(k_hist, v_hist, np.asarray(lens), P, max(news) + extra, rng)
    new_indptr = np.zeros(B + 1, np.int32)
    new_indptr[1:] = np.cumsum(news)
    n_new = int(new_indptr[-1])
    q = rng.standard_normal((n_new, Hq, d)).astype(np.float32)
    kn = rng.standard_normal((n_new, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((n_new, Hkv, d)).astype(np.float32)
    return rng, k_hist, v_hist, kc, vc, bt, new_indptr, q, kn, vn


def pin_extend_brute_force(orc):
    """Base rows of the new tokens and output rows anywhere in the sequence,
    against dense brute force over the logical sequence (history + new)."""
    B, Hq, Hkv, d, P, w = 3, 4, 2, 8, 4, 5
    lens, news = [0, 6, 13], [4, 1, 0]
    rng, k_hist, v_hist, kc, vc, bt, new_indptr, q, kn, vn = _extend_setup(41, B, Hq, Hkv, d, P, lens, news, extra=1)
    ab, bb, ao, bo = (x.numpy() for x in make_affines(torch.Generator().manual_seed(8), Hq, d))
    scale = 0.37
    for with_q_out in (False, True):
        if with_q_out:  # output rows may sit in the history when their query is given
            lists = [[3, 0], [2, 6], [12, 5]]
        else:  # otherwise only at new positions
            lists = [[0, 3, 2], [6], []]
        out_indptr, pos = csr(lists)
        q_out = rng.standard_normal((int(out_indptr[-1]), Hq, d)).astype(np.float32) if with_q_out else None
        kc2, vc2 = kc.copy(), vc.copy()
        ob, lb, oo, lo = orc.extend(q, kn, vn, kc2, vc2, bt, np.asarray(lens, np.int32), new_indptr, out_indptr, pos,
                                    ab, bb, ao, bo, w, scale, q_out=q_out)
        for b in range(B):
            i0, i1 = int(new_indptr[b]), int(new_indptr[b + 1])
            K = np.concatenate([k_hist[b], kn[i0:i1]], 0)
            V = np.concatenate([v_hist[b], vn[i0:i1]], 0)
            L = lens[b]
            for h in range(Hq):
                kv = h // (Hq // Hkv)
                if i1 > i0:
                    o, l = brute_rows(q[i0:i1, h], ab[h], bb[h], K[:, kv], V[:, kv], np.arange(L, L + i1 - i0),
                                      lambda t: max(0, t - w + 1), scale)
                    _close(ob[i0:i1, h], o, what="extend base o")
                    _close(lb[i0:i1, h], l, what="extend base lse")
                r0, r1 = int(out_indptr[b]), int(out_indptr[b + 1])
                if r1 > r0:
                    p = pos[r0:r1]
                    qr = q_out[r0:r1, h] if q_out is not None else q[i0 + p - L, h]
                    o, l = brute_rows(qr, ao[h], bo[h], K[:, kv], V[:, kv], p, lambda t: 0, scale)
                    _close(oo[r0:r1, h], o, what="extend out o")
                    _close(lo[r0:r1, h], l, what="extend out lse")
            for i in range(i0, i1):  # the appends landed where the block table says
                t = L + i - i0
                assert np.array_equal(kc2[bt[b, t // P], t % P], kn[i])
                assert np.array_equal(vc2[bt[b, t // P], t % P], vn[i])


def pin_extend_chunked_consistency(orc):
    """Sec. 3.2: a prefill of T0 tokens followed by steps that append chunks of
    3, 0, 5, 1 and 7 tokens gives every new token the base row of one prefill
    over all tokens, and the output rows (last token of each chunk) its output rows."""
    B, T0, Hq, Hkv, d, w, P = 2, 6, 4, 2, 8, 4, 4
    chunks = [3, 0, 5, 1, 7]
    T = T0 + sum(chunks)
    q, k, v, ab, bb, ao, bo = rng_inputs(43, B, T, Hq, Hkv, d)
    ends = np.cumsum([T0] + chunks) - 1
    out_pos = sorted(set(int(e) for e in ends[1:]))
    indptr, pos = csr([out_pos] * B)
    full = orc.prefill(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3)
    rng = np.random.default_rng(4)
    lens = np.full(B, T0, np.int32)
    kc, vc, bt = _paged_from_seq([k[b, :T0] for b in range(B)], [v[b, :T0] for b in range(B)], lens, P, T - T0, rng)
    at = T0
    for c in chunks:
        new_indptr = np.arange(B + 1, dtype=np.int32) * c
        qn = np.concatenate([q[b, at:at + c] for b in range(B)], 0)
        kn = np.concatenate([k[b, at:at + c] for b in range(B)], 0)
        vn = np.concatenate([v[b, at:at + c] for b in range(B)], 0)
        lists = [[at + c - 1] if c else [] for _ in range(B)]
        oi, op = csr(lists)
        ob, lb, oo, lo = orc.extend(qn.reshape(B * c, Hq, d), kn.reshape(B * c, Hkv, d), vn.reshape(B * c, Hkv, d),
                                    kc, vc, bt, lens, new_indptr, oi, op, ab, bb, ao, bo, w, 0.3)
        for b in range(B):
            _close(ob[b * c:(b + 1) * c], full[0][b, at:at + c], 1e-12, f"chunk base o at {at}")
            _close(lb[b * c:(b + 1) * c].T, full[1][b, :, at:at + c], 1e-12, f"chunk base lse at {at}")
            if c:
                r = int(indptr[b]) + out_pos.index(at + c - 1)
                _close(oo[b], full[2][r], 1e-12, f"chunk out o at {at}")
                _close(lo[b], full[3][r], 1e-12, f"chunk out lse at {at}")
        lens = lens + c
        at += c


def pin_extend_single_token_is_decode(orc):
    """One new token per sequence with an output row at it is a decoding step."""
    rng = np.random.default_rng(47)
    B, Hq, Hkv, d, P, w = 3, 4, 2, 8, 4, 6
    lens = [0, 5, 11]
    _, k_hist, v_hist, kc, vc, bt, new_indptr, q, kn, vn = _extend_setup(47, B, Hq, Hkv, d, P, lens, [1, 1, 1])
    ab, bb, ao, bo = (x.numpy() for x in make_affines(torch.Generator().manual_seed(9), Hq, d))
    qo = rng.standard_normal((B, Hq, d)).astype(np.float32)
    out_indptr, pos = csr([[L] for L in lens])
    a = orc.extend(q, kn, vn, kc.copy(), vc.copy(), bt, np.asarray(lens, np.int32), new_indptr, out_indptr, pos,
                   ab, bb, ao, bo, w, 0.5, q_out=qo)
    b_ = orc.decode(q, kn, vn, kc.copy(), vc.copy(), bt, np.asarray(lens, np.int32), ab, bb, ao, bo, w, 0.5, q_out=qo)
    for x, y, n in zip(a, b_, ("o_base", "lse_base", "o_out", "lse_out")):
        _close(x, y, 1e-12, "extend as decode " + n)


# ---------------------------------------------------------------------------
# Backward (gradients of Eq. 4 and Eq. 5 and of the query affines)
# ---------------------------------------------------------------------------

def torch_forward(q, k, v, ab, bb, ao, bo, indptr, pos, window, scale, q_out=None):
    """Dense masked forward in torch float64 (library softmax), differentiable.

    Arguments are float64 torch tensors; returns (o_base [B,T,Hq,d], o_out [n_out,Hq,d]).
    The gradients that torch.autograd derives from it are what the oracle's
    hand-derived backward is checked against.
    """
    B, T, Hq, d = q.shape
    Hkv = k.shape[2]
    g = Hq // Hkv
    kr = k.repeat_interleave(g, dim=2)  # [B,T,Hq,d], kv = h // g
    vr = v.repeat_interleave(g, dim=2)
    i = torch.arange(T)[:, None]
    j = torch.arange(T)[None, :]
    band = (j <= i) & (j > i - window)
    qa = q * ab + bb
    S = scale * torch.einsum("bthc,bjhc->bhtj", qa, kr)
    S = S.masked_fill(~band, float("-inf"))
    o_base = torch.einsum("bhtj,bjhc->bthc", torch.softmax(S, dim=-1), vr)
    outs = []
    for b in range(B):
        r0, r1 = int(indptr[b]), int(indptr[b + 1])
        if r1 == r0:
            continue
        p = torch.as_tensor(pos[r0:r1], dtype=torch.long)
        qr = q_out[r0:r1] if q_out is not None else q[b, p]
        qo = qr * ao + bo  # [R,Hq,d]
        So = scale * torch.einsum("rhc,jhc->rhj", qo, kr[b])
        causal = torch.arange(T)[None, None, :] <= p[:, None, None]
        So = So.masked_fill(~causal, float("-inf"))
        outs.append(torch.einsum("rhj,jhc->rhc", torch.softmax(So, dim=-1), vr[b]))
    o_out = torch.cat(outs, 0) if outs else torch.zeros((0, Hq, d), dtype=q.dtype)
    return o_base, o_out


BACKWARD_CASES = [
    # (B, T, Hq, Hkv, d, window)
    (1, 1, 1, 1, 4, 1),
    (1, 13, 2, 1, 8, 1),
    (1, 17, 4, 2, 8, 5),
    (2, 21, 4, 1, 8, 21),
    (2, 19, 6, 2, 4, 30),
]


def _backward_inputs(i, B, T, Hq, Hkv, d, with_q_out):
    q, k, v, ab, bb, ao, bo = rng_inputs(101 + i, B, T, Hq, Hkv, d)
    r = np.random.default_rng(101 + i)
    lists = [sorted(r.choice(T, size=r.integers(0, T + 1), replace=False).tolist()) for _ in range(B)]
    lists[-1] = sorted(set(lists[-1]) | {T - 1})
    indptr, pos = csr(lists)
    n_out = int(indptr[-1])
    q_out = r.standard_normal((n_out, Hq, d)).astype(np.float32) if with_q_out else None
    do_b = r.standard_normal((B, T, Hq, d)).astype(np.float32)
    do_o = r.standard_normal((n_out, Hq, d)).astype(np.float32)
    return q, k, v, ab, bb, ao, bo, indptr, pos, q_out, do_b, do_o


def pin_backward_autograd(orc, cases=BACKWARD_CASES):
    """Every gradient equals torch.autograd (float64) through the dense masked forward."""
    for i, (B, T, Hq, Hkv, d, w) in enumerate(cases):
        for with_q_out in (False, True):
            q, k, v, ab, bb, ao, bo, indptr, pos, q_out, do_b, do_o = _backward_inputs(i, B, T, Hq, Hkv, d, with_q_out)
            scale = 0.9 / math.sqrt(d)
            got = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, scale, do_b, do_o, q_out=q_out)
            leaves = {n: torch.tensor(x, dtype=torch.float64, requires_grad=True)
                      for n, x in (("q", q), ("k", k), ("v", v), ("ab", ab), ("bb", bb), ("ao", ao), ("bo", bo))}
            qo_t = torch.tensor(q_out, dtype=torch.float64, requires_grad=True) if q_out is not None else None
            ob, oo = torch_forward(leaves["q"], leaves["k"], leaves["v"], leaves["ab"], leaves["bb"],
                                   leaves["ao"], leaves["bo"], indptr, pos, w, scale, qo_t)
            loss = (ob * torch.from_numpy(do_b).double()).sum() + (oo * torch.from_numpy(do_o).double()).sum()
            loss.backward()
            tag = f"case {i} q_out={with_q_out}"
            for name, leaf in (("dq", "q"), ("dk", "k"), ("dv", "v"), ("d_alpha_base", "ab"),
                               ("d_beta_base", "bb"), ("d_alpha_out", "ao"), ("d_beta_out", "bo")):
                _close(got[name], leaves[leaf].grad.numpy(), 1e-9, f"{tag} {name}")
            if q_out is not None:
                _close(got["dq_out"], qo_t.grad.numpy(), 1e-9, f"{tag} dq_out")
            else:
                assert got["dq_out"] is None


def pin_backward_finite_difference(orc):
    """Directional derivatives of L = <do_base, o_base> + <do_out, o_out>, taken
    by central differences of the oracle's own (pinned) forward, equal the
    gradients contracted with the same direction, one input at a time."""
    B, T, Hq, Hkv, d, w = 2, 11, 4, 2, 8, 4
    q, k, v, ab, bb, ao, bo, indptr, pos, q_out, do_b, do_o = _backward_inputs(7, B, T, Hq, Hkv, d, True)
    scale = 0.4
    got = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, scale, do_b, do_o, q_out=q_out)
    base = dict(q=q, k=k, v=v, ab=ab, bb=bb, ao=ao, bo=bo, q_out=q_out)
    grad_of = dict(q="dq", k="dk", v="dv", ab="d_alpha_base", bb="d_beta_base",
                   ao="d_alpha_out", bo="d_beta_out", q_out="dq_out")

    def loss(x):
        ob, _, oo, _ = orc.prefill(x["q"], x["k"], x["v"], x["ab"], x["bb"], x["ao"], x["bo"],
                                   indptr, pos, w, scale, q_out=x["q_out"])
        return float(np.sum(ob * do_b) + np.sum(oo * do_o))

    r = np.random.default_rng(5)
    h = 2.0 ** -9
    for name, gname in grad_of.items():
        u = r.standard_normal(base[name].shape)
        xp, xm = dict(base), dict(base)
        xp[name] = (base[name] + h * u).astype(np.float32)
        xm[name] = (base[name] - h * u).astype(np.float32)
        step = xp[name].astype(np.float64) - xm[name].astype(np.float64)  # the float32 step actually taken
        fd = loss(xp) - loss(xm)
        pred = float(np.sum(got[gname] * step))
        assert abs(fd - pred) <= 1e-6 * max(1.0, abs(pred)), f"finite difference {name}: {fd} vs {pred}"


def pin_backward_translation_sums(orc):
    """Adding one vector c to every key of a (b, kv) sequence leaves every
    output unchanged, so the keys' gradients sum to zero; adding c to every
    value adds c to every output of that group, so the values' gradients sum
    to the sum of all dO rows (both streams) of the group's query heads."""
    B, T, Hq, Hkv, d, w = 2, 16, 6, 2, 8, 5
    q, k, v, ab, bb, ao, bo, indptr, pos, q_out, do_b, do_o = _backward_inputs(11, B, T, Hq, Hkv, d, False)
    got = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3, do_b, do_o)
    g = Hq // Hkv
    for b in range(B):
        r0, r1 = int(indptr[b]), int(indptr[b + 1])
        for kv in range(Hkv):
            hs = slice(kv * g, (kv + 1) * g)
            _close(got["dk"][b, :, kv].sum(axis=0), np.zeros(d), 1e-11, "sum dk")
            want = do_b[b, :, hs].astype(np.float64).sum(axis=(0, 1)) + do_o[r0:r1, hs].astype(np.float64).sum(axis=(0, 1))
            _close(got["dv"][b, :, kv].sum(axis=0), want, 1e-11, "sum dv")


def pin_backward_row_range(orc):
    """Restricting the rows to positions [t0, T) leaves the gradients of every
    key j >= t0 and of every row in the range unchanged (no earlier row sees
    those keys); restricting to [0, t1) leaves dq of rows < t1 unchanged."""
    B, T, Hq, Hkv, d, w = 1, 30, 4, 2, 8, 6
    for with_q_out in (False, True):
        q, k, v, ab, bb, ao, bo, indptr, pos, q_out, do_b, do_o = _backward_inputs(13, B, T, Hq, Hkv, d, with_q_out)
        full = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3, do_b, do_o, q_out=q_out)
        t0, t1 = 17, 12
        tail = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3, do_b, do_o, q_out=q_out,
                                    row_range=(t0, T))
        head = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, w, 0.3, do_b, do_o, q_out=q_out,
                                    row_range=(0, t1))
        _close(tail["dk"][:, t0:], full["dk"][:, t0:], 1e-12, "tail dk")
        _close(tail["dv"][:, t0:], full["dv"][:, t0:], 1e-12, "tail dv")
        if q_out is None:
            _close(tail["dq"][:, t0:], full["dq"][:, t0:], 1e-12, "tail dq")
            _close(head["dq"][:, :t1], full["dq"][:, :t1], 1e-12, "head dq")
            _close(tail["dq"][:, :t0], np.zeros_like(full["dq"][:, :t0]), 0.0, "tail dq outside")
        else:
            sel = pos >= t0
            _close(tail["dq_out"][sel], full["dq_out"][sel], 1e-12, "tail dq_out")
            _close(tail["dq"][:, t0:], full["dq"][:, t0:], 1e-12, "tail dq")


def pin_backward_window_one(orc):
    """w = 1 and no output rows: o_base[t] = v_t, so dv_t is the sum of dO over
    the group's heads and every other gradient is zero."""
    B, T, Hq, Hkv, d = 1, 9, 4, 2, 8
    q, k, v, ab, bb, ao, bo = rng_inputs(41, B, T, Hq, Hkv, d)
    indptr, pos = csr([[]])
    do_b = np.random.default_rng(2).standard_normal((B, T, Hq, d)).astype(np.float32)
    got = orc.prefill_backward(q, k, v, ab, bb, ao, bo, indptr, pos, 1, 0.5, do_b, None)
    want = do_b.astype(np.float64).reshape(B, T, Hkv, Hq // Hkv, d).sum(axis=3)
    _close(got["dv"], want, 1e-12, "w=1 dv")
    for n in ("dq", "dk", "d_alpha_base", "d_beta_base", "d_alpha_out", "d_beta_out"):
        _close(got[n], np.zeros_like(got[n]), 1e-12, f"w=1 {n}")


ALL_PINS = [
    pin_brute_force_prefill,
    pin_row_subset,
    pin_window_covers_all,
    pin_identity_affine_is_sdpa,
    pin_window_one,
    pin_zero_query_uniform,
    pin_key_offset_shift,
    pin_gqa_equals_replicated,
    pin_decode_brute_force,
    pin_decode_page_permutation,
    pin_prefill_decode_consistency,
    pin_hand_worked,
    pin_project_selection_weight,
    pin_project_rank_one,
    pin_project_feeds_decode,
    pin_extend_brute_force,
    pin_extend_chunked_consistency,
    pin_extend_single_token_is_decode,
    pin_backward_autograd,
    pin_backward_finite_difference,
    pin_backward_translation_sums,
    pin_backward_row_range,
    pin_backward_window_one,
]
