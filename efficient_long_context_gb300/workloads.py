"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke check.

This module only draws random inputs and describes their shapes; it holds none
of the attention arithmetic. Every tensor is drawn on the CPU from a
``torch.Generator`` seeded per workload, in a fixed order, so the CUDA path and
the CPU oracle always see identical bits.

The workloads stand in for the Orthros paper's regimes (Sec. 3.2: pre-training
with every position an output row, supervised fine-tuning with an answer span,
prefilling with one output row at the last prompt token, decoding with one
decoupled token pair per step) at the shapes of the attention layers they run
in. The paper measures only model-level latency; these synthetic inputs take
the place of its datasets.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    window: int
    dtype: torch.dtype
    # "last": out = {T-1}; "all": out = every position; ("span", n): last n positions
    out_mode: object
    k_offset_std: float = 0.0  # per-(kv head, channel) offset added to every key
    seed: int = 0

    @property
    def scale(self) -> float:
        return self.d ** -0.5


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    window: int
    page_size: int
    len_lo: int  # cached lengths drawn uniformly from [len_lo, len_hi]
    len_hi: int
    steps: int
    dtype: torch.dtype = torch.bfloat16
    seed: int = 0

    @property
    def scale(self) -> float:
        return self.d ** -0.5


# The five workloads: tiny fp32 prefill; pre-training shape (every position an
# output row); SFT shape with a 1024-token answer span and offset keys; a 128K
# prefill at the Llama-3.1-8B attention shape; batched paged decoding.
TINY_FP32 = PrefillWorkload("tiny_fp32_T512_w64", 1, 512, 4, 4, 64, 64, torch.float32, "last", seed=1000)
PT_2K = PrefillWorkload("pt_b8_T2048_h16_w512", 8, 2048, 16, 16, 128, 512, torch.bfloat16, "all", seed=1001)
SFT_8K = PrefillWorkload("sft_b4_T8192_gqa32x8_w1024", 4, 8192, 32, 8, 128, 1024, torch.bfloat16,
                         ("span", 1024), k_offset_std=0.5, seed=1002)
PREFILL_128K = PrefillWorkload("prefill_T131072_gqa32x8_d128_w4096", 1, 131072, 32, 8, 128, 4096,
                               torch.bfloat16, "last", seed=1003)
DECODE_32 = DecodeWorkload("decode_b32_L16k-32k_gqa32x8_w4096_p64", 32, 32, 8, 128, 4096, 64,
                           16384, 32768, 128, seed=1004)

PREFILL_WORKLOADS = {w.name: w for w in (TINY_FP32, PT_2K, SFT_8K, PREFILL_128K)}


def out_positions_for(mode, B: int, T: int):
    """CSR (indptr [B+1] int32, positions [n_out] int32) of output rows."""
    if mode == "last":
        per = [torch.tensor([T - 1], dtype=torch.int32)] if T > 0 else [torch.zeros(0, dtype=torch.int32)]
        per = per * B
    elif mode == "all":
        per = [torch.arange(T, dtype=torch.int32)] * B
    elif isinstance(mode, tuple) and mode[0] == "span":
        n = min(int(mode[1]), T)
        per = [torch.arange(T - n, T, dtype=torch.int32)] * B
    elif isinstance(mode, tuple) and mode[0] == "list":
        per = [torch.as_tensor(p, dtype=torch.int32) for p in mode[1]]
        assert len(per) == B
    else:
        raise ValueError(f"unknown output-row mode {mode!r}")
    counts = torch.tensor([len(p) for p in per], dtype=torch.int64)
    indptr = torch.zeros(B + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(counts, 0).to(torch.int32)
    pos = torch.cat(per) if per else torch.zeros(0, dtype=torch.int32)
    return indptr, pos.to(torch.int32)


def _normal(gen, shape, dtype):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def make_affines(gen, Hq: int, d: int):
    """alpha ~ 1 + 0.1 N(0,1), beta ~ 0.1 N(0,1), per (query head, channel), fp32."""
    ab = 1.0 + 0.1 * torch.randn((Hq, d), generator=gen, dtype=torch.float32)
    bb = 0.1 * torch.randn((Hq, d), generator=gen, dtype=torch.float32)
    ao = 1.0 + 0.1 * torch.randn((Hq, d), generator=gen, dtype=torch.float32)
    bo = 0.1 * torch.randn((Hq, d), generator=gen, dtype=torch.float32)
    return ab, bb, ao, bo


def make_prefill(w: PrefillWorkload, seed: int | None = None, out_mode=None, with_q_out: bool = False):
    """Draw one prefill workload on the CPU. Returns a dict of CPU tensors.

    Draw order: q, k, v, alpha_base, beta_base, alpha_out, beta_out, the key
    offsets (if any), then q_out (if asked for).
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    B, T, Hq, Hkv, d = w.B, w.T, w.Hq, w.Hkv, w.d
    q = _normal(gen, (B, T, Hq, d), w.dtype)
    k32 = torch.randn((B, T, Hkv, d), generator=gen, dtype=torch.float32)
    v = _normal(gen, (B, T, Hkv, d), w.dtype)
    ab, bb, ao, bo = make_affines(gen, Hq, d)
    if w.k_offset_std > 0:
        off = w.k_offset_std * torch.randn((Hkv, d), generator=gen, dtype=torch.float32)
        k32 += off
    k = k32.to(w.dtype)
    del k32
    indptr, pos = out_positions_for(w.out_mode if out_mode is None else out_mode, B, T)
    q_out = _normal(gen, (int(indptr[-1]), Hq, d), w.dtype) if with_q_out else None
    return dict(q=q, k=k, v=v, alpha_base=ab, beta_base=bb, alpha_out=ao, beta_out=bo,
                out_indptr=indptr, out_positions=pos, q_out=q_out,
                B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, window=w.window, scale=w.scale, dtype=w.dtype)


def make_grad_outputs(wl: dict, seed: int):
    """Seeded gradients dL/do for a prefill workload (the backward's inputs):
    do_base [B,T,Hq,d] and do_out [n_out,Hq,d], N(0,1) in the workload's dtype."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    B, T, Hq, d = wl["B"], wl["T"], wl["Hq"], wl["d"]
    n_out = int(wl["out_indptr"][-1])
    do_base = _normal(gen, (B, T, Hq, d), wl["dtype"])
    do_out = _normal(gen, (n_out, Hq, d), wl["dtype"])
    return do_base, do_out


def small_prefill(B, T, Hq, Hkv, d, window, dtype=torch.bfloat16, out_mode="last", seed=7,
                  with_q_out=False, k_offset_std=0.0):
    """A small prefill case for parity sweeps (same recipe as the named workloads)."""
    w = PrefillWorkload(f"small_{B}x{T}x{Hq}x{Hkv}x{d}_w{window}", B, T, Hq, Hkv, d, window, dtype,
                        out_mode, k_offset_std=k_offset_std, seed=seed)
    return make_prefill(w, with_q_out=with_q_out)


@dataclass
class DecodeState:
    """Paged cache plus the per-step inputs of a decoding run (CPU tensors)."""
    k_cache: torch.Tensor  # [num_pages, page_size, Hkv, d]
    v_cache: torch.Tensor
    block_table: torch.Tensor  # [B, max_pages] int32, physical page ids
    cache_lens: torch.Tensor  # [B] int32, lengths before the first step
    q: torch.Tensor  # [steps, B, Hq, d]
    k_new: torch.Tensor  # [steps, B, Hkv, d]
    v_new: torch.Tensor
    alpha_base: torch.Tensor
    beta_base: torch.Tensor
    alpha_out: torch.Tensor
    beta_out: torch.Tensor
    q_out: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)


def make_decode(w: DecodeWorkload, steps: int | None = None, seed: int | None = None,
                with_q_out: bool = False, lens=None) -> DecodeState:
    """Draw a decoding workload: lengths, a shuffled page pool, cache contents, step inputs.

    Every slot of every page is filled with N(0,1) (slots past a sequence's
    length hold values that the attention must never read). Physical page ids
    are a seeded random permutation, so logically adjacent pages are scattered.
    Draw order: lengths, permutation, k_cache, v_cache, affines, q, k_new, v_new, q_out.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    steps = w.steps if steps is None else steps
    B, P = w.B, w.page_size
    if lens is None:
        lens = torch.randint(w.len_lo, w.len_hi + 1, (B,), generator=gen, dtype=torch.int64)
    else:
        lens = torch.as_tensor(lens, dtype=torch.int64)
    pages_per = [(int(L) + steps + P - 1) // P for L in lens]
    max_pages = max(pages_per)
    num_pages = sum(pages_per)
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = perm[at:at + n]
        at += n
    k_cache = _normal(gen, (num_pages, P, w.Hkv, w.d), w.dtype)
    v_cache = _normal(gen, (num_pages, P, w.Hkv, w.d), w.dtype)
    ab, bb, ao, bo = make_affines(gen, w.Hq, w.d)
    q = _normal(gen, (steps, B, w.Hq, w.d), w.dtype)
    k_new = _normal(gen, (steps, B, w.Hkv, w.d), w.dtype)
    v_new = _normal(gen, (steps, B, w.Hkv, w.d), w.dtype)
    q_out = _normal(gen, (steps, B, w.Hq, w.d), w.dtype) if with_q_out else None
    return DecodeState(k_cache, v_cache, block_table, lens.to(torch.int32), q, k_new, v_new,
                       ab, bb, ao, bo, q_out,
                       meta=dict(B=B, Hq=w.Hq, Hkv=w.Hkv, d=w.d, window=w.window, page_size=P,
                                 max_pages=max_pages, num_pages=num_pages, steps=steps,
                                 scale=w.scale, dtype=w.dtype))


@dataclass(frozen=True)
class ExtendWorkload:
    """A continuous-batching step: histories in a paged cache, then per
    sequence a number of new tokens (a prefill chunk, one decoding token or
    none). Output rows: the last new token of every sequence that has one,
    plus `history_rows` rows at earlier positions (these need q_out)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    window: int
    len_lo: int
    len_hi: int
    news: tuple
    page_size: int = 64
    dtype: torch.dtype = torch.bfloat16
    history_rows: int = 0
    seed: int = 0

    @property
    def scale(self) -> float:
        return self.d ** -0.5


# 32 sequences with 16K-32K cached tokens: 28 decode one token, 4 append a 16-token prefill chunk
MIXED_32 = ExtendWorkload("mixed_b32_L16k-32k_gqa32x8_w4096_4x16+28x1", 32, 32, 8, 128, 4096, 16384, 32768,
                          tuple([16] * 4 + [1] * 28), seed=1005)


def make_extend(w: ExtendWorkload, with_q_out: bool = False, seed: int | None = None) -> dict:
    """Draw one continuous-batching step (CPU tensors). Draw order: lengths,
    page permutation, k_cache, v_cache, affines, q, k_new, v_new, history-row
    positions, q_out."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed if seed is None else seed)
    B, P = w.B, w.page_size
    news = list(w.news)
    assert len(news) == B
    lens = torch.randint(w.len_lo, w.len_hi + 1, (B,), generator=gen, dtype=torch.int64)
    pages_per = [max(1, (int(L) + n + P - 1) // P) for L, n in zip(lens, news)]
    max_pages = max(pages_per)
    num_pages = sum(pages_per)
    perm = torch.randperm(num_pages, generator=gen).to(torch.int32)
    block_table = torch.full((B, max_pages), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(pages_per):
        block_table[b, :n] = perm[at:at + n]
        at += n
    k_cache = _normal(gen, (num_pages, P, w.Hkv, w.d), w.dtype)
    v_cache = _normal(gen, (num_pages, P, w.Hkv, w.d), w.dtype)
    ab, bb, ao, bo = make_affines(gen, w.Hq, w.d)
    new_indptr = torch.zeros(B + 1, dtype=torch.int32)
    new_indptr[1:] = torch.cumsum(torch.tensor(news), 0)
    n_new = int(new_indptr[-1])
    q = _normal(gen, (n_new, w.Hq, w.d), w.dtype)
    k_new = _normal(gen, (n_new, w.Hkv, w.d), w.dtype)
    v_new = _normal(gen, (n_new, w.Hkv, w.d), w.dtype)
    lists = []
    for b in range(B):
        L, n = int(lens[b]), news[b]
        rows = [L + n - 1] if n else []
        if w.history_rows and with_q_out:
            hist = torch.randint(0, max(L + n, 1), (w.history_rows,), generator=gen).tolist()
            rows = sorted(rows + hist)
        lists.append(rows)
    out_indptr = torch.zeros(B + 1, dtype=torch.int32)
    out_indptr[1:] = torch.cumsum(torch.tensor([len(r) for r in lists]), 0)
    out_positions = torch.tensor([t for r in lists for t in r], dtype=torch.int32)
    n_out = int(out_indptr[-1])
    q_out = _normal(gen, (n_out, w.Hq, w.d), w.dtype) if with_q_out else None
    return dict(k_cache=k_cache, v_cache=v_cache, block_table=block_table, cache_lens=lens.to(torch.int32),
                new_indptr=new_indptr, out_indptr=out_indptr, out_positions=out_positions, q=q, k_new=k_new,
                v_new=v_new, q_out=q_out, alpha_base=ab, beta_base=bb, alpha_out=ao, beta_out=bo,
                B=B, Hq=w.Hq, Hkv=w.Hkv, d=w.d, window=w.window, scale=w.scale, dtype=w.dtype,
                page_size=P, max_pages=max_pages, num_pages=num_pages)


@dataclass(frozen=True)
class ProjectionWorkload:
    """The shared Q/K/V projection: n_base base-token rows and n_out output
    rows of width d_model through one weight of (Hq + 2 Hkv) d columns."""
    name: str
    n_base: int
    n_out: int
    d_model: int
    Hq: int
    Hkv: int
    d: int
    seed: int = 0


# Llama-3.1-8B attention projection: a 32-sequence decoding step (32 base +
# 32 output tokens share the weight read) and an 8192-token prefill chunk.
PROJ_DECODE_32 = ProjectionWorkload("proj_decode_b32x2_d4096_gqa32x8", 32, 32, 4096, 32, 8, 128, seed=1006)
PROJ_PREFILL_8K = ProjectionWorkload("proj_prefill_8192_d4096_gqa32x8", 8192, 0, 4096, 32, 8, 128, seed=1007)


def make_projection(w: ProjectionWorkload, seed: int | None = None) -> dict:
    """Hidden rows ~ N(0,1), weights ~ N(0,1)/sqrt(d_model) (unit-variance
    outputs), affines as elsewhere; bf16. Draw order: x, w_t, affines."""
    gen = torch.Generator()
    gen.manual_seed(w.seed if seed is None else seed)
    N = (w.Hq + 2 * w.Hkv) * w.d
    x = _normal(gen, (w.n_base + w.n_out, w.d_model), torch.bfloat16)
    w_t = (torch.randn((N, w.d_model), generator=gen) * w.d_model ** -0.5).to(torch.bfloat16)
    ab, bb, ao, bo = make_affines(gen, w.Hq, w.d)
    return dict(x=x, w_t=w_t, alpha_base=ab, beta_base=bb, alpha_out=ao, beta_out=bo, n_base=w.n_base,
                n_out=w.n_out, d_model=w.d_model, Hq=w.Hq, Hkv=w.Hkv, d=w.d)
