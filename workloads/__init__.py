"""Seeded synthetic inputs for paged extend attention.

This module is shared by the FP64 oracle tests, the GPU parity tests and the
benchmark.  It holds none of the attention arithmetic: it only draws random
numbers, rounds the draws to bf16, and lays out page tables (which physical page
of the shuffled pool each sequence owns).  Slot mapping, KV append and attention
live on each side separately (``oracle/`` and the CUDA library).

Every array is numpy.  bf16 tensors are carried as ``uint16`` bit patterns so
both sides read exactly the same values.

Workload shapes follow the chunked-prefill workloads of the source pages
(AReno PR #642 "How was it tested?": one-token chunks, GQA, page boundaries,
sliding windows; the 1025/4097-token incoming prompts of its "Performance"
section) and the sizes fixed for this implementation (Qwen3-8B-like GQA
attention, a mixed scheduler batch, a page-boundary stress, a long context).
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "Batch", "bf16_bits", "bf16_to_f32", "make_batch", "tiny_case",
    "zero_score_steps", "gqa_prefill", "mixed_batch", "stress_case",
    "long_context", "random_mask", "CONFIGS", "config_by_name",
]


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and
    return the 16-bit patterns.  Inputs are finite draws."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Batch:
    """One call's worth of inputs.

    qo_indptr   int32 [B+1]  prefix sums of chunk lengths (rows of q)
    prefix_lens int32 [B]    cached tokens before each chunk
    kv_indptr   int32 [B+1]  CSR offsets into kv_indices, in pages
    kv_indices  int32 [...]  physical page ids; -1 marks padding after the
                             pages a sequence needs
    q           uint16 [total_q, Hq, D]     bf16 bits
    k_new/v_new uint16 [total_q, Hkv, D]    the chunk's K/V (to be appended)
    k_pool/v_pool uint16 [num_pages*page_size, Hkv, D]  pool before append
    """
    name: str
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    window: int
    sm_scale: float
    qo_indptr: np.ndarray
    prefix_lens: np.ndarray
    kv_indptr: np.ndarray
    kv_indices: np.ndarray
    num_pages: int
    q: np.ndarray
    k_new: np.ndarray
    v_new: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray

    @property
    def batch(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def chunk_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int64)

    @property
    def kv_lens(self) -> np.ndarray:
        return self.prefix_lens.astype(np.int64) + self.chunk_lens

    @property
    def pool_slots(self) -> int:
        return int(self.num_pages * self.page_size)


def _normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return bf16_bits(x)


def make_batch(
    prefix_lens: Sequence[int],
    chunk_lens: Sequence[int],
    n_q_heads: int,
    n_kv_heads: int,
    head_dim: int,
    page_size: int,
    *,
    seed: int,
    window: int = 0,
    sm_scale: float = 0.0,
    name: str = "custom",
    pad_to_pages: Optional[int] = None,
    share_groups: Optional[Sequence[Sequence[int]]] = None,
    slack_pages: int = 3,
    pool_pages: Optional[int] = None,
) -> Batch:
    """Build a ragged batch with a scattered page table.

    Pages come from a seeded shuffle of the pool; each sequence (or each
    group in ``share_groups``, whose members list the same physical pages as
    successive chunks of one prompt) takes the next ceil(L/page_size) pages.
    ``pad_to_pages`` lays the table out densely, ``pad_to_pages`` entries per
    row, padded with -1.  The whole pool (including the slots the chunk will
    be appended to) is filled with bf16 ~N(0,1) draws.
    """
    rng = np.random.default_rng(seed)
    P = np.asarray(prefix_lens, dtype=np.int64).reshape(-1)
    C = np.asarray(chunk_lens, dtype=np.int64).reshape(-1)
    assert P.shape == C.shape
    B = int(P.shape[0])
    L = P + C
    need = [(-(-int(l) // page_size)) for l in L]

    groups = share_groups if share_groups is not None else [[b] for b in range(B)]
    owner = {}
    for gi, grp in enumerate(groups):
        for b in grp:
            owner[b] = gi
    assert len(owner) == B
    group_pages_needed = [max(need[b] for b in grp) if grp else 0 for grp in groups]
    total_needed = int(sum(group_pages_needed))
    num_pages = int(pool_pages) if pool_pages is not None else total_needed + slack_pages
    assert num_pages >= total_needed
    perm = rng.permutation(num_pages).astype(np.int32)
    group_pages = []
    off = 0
    for n in group_pages_needed:
        group_pages.append(perm[off:off + n])
        off += n

    rows = []
    for b in range(B):
        pages = group_pages[owner[b]][: need[b]]
        if pad_to_pages is not None:
            assert pad_to_pages >= need[b]
            row = np.full(pad_to_pages, -1, dtype=np.int32)
            row[: need[b]] = pages
        else:
            row = np.asarray(pages, dtype=np.int32)
        rows.append(row)
    kv_indptr = np.zeros(B + 1, dtype=np.int32)
    kv_indptr[1:] = np.cumsum([r.shape[0] for r in rows]) if B else []
    kv_indices = np.concatenate(rows).astype(np.int32) if rows else np.zeros(0, np.int32)

    qo_indptr = np.zeros(B + 1, dtype=np.int32)
    qo_indptr[1:] = np.cumsum(C) if B else []
    total_q = int(qo_indptr[-1])
    slots = num_pages * page_size
    q = _normal_bf16(rng, (total_q, n_q_heads, head_dim))
    k_new = _normal_bf16(rng, (total_q, n_kv_heads, head_dim))
    v_new = _normal_bf16(rng, (total_q, n_kv_heads, head_dim))
    k_pool = _normal_bf16(rng, (slots, n_kv_heads, head_dim))
    v_pool = _normal_bf16(rng, (slots, n_kv_heads, head_dim))
    return Batch(
        name=name, n_q_heads=n_q_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
        page_size=page_size, window=int(window), sm_scale=float(sm_scale),
        qo_indptr=qo_indptr, prefix_lens=P.astype(np.int32), kv_indptr=kv_indptr,
        kv_indices=kv_indices, num_pages=num_pages, q=q, k_new=k_new, v_new=v_new,
        k_pool=k_pool, v_pool=v_pool,
    )


# ---------------------------------------------------------------------------
# The workloads.  Seeds are 1000 + the workload number.
# ---------------------------------------------------------------------------

def tiny_case(seed: int = 1001) -> Batch:
    """2 sequences, prefix {0, 37}, chunk {5, 40}, 2 query heads / 1 KV head,
    head_dim 64, page_size 16, a seeded permutation of a 16-page pool laid out
    as a dense 2 x 8 table padded with -1, sm_scale 1/8, no window."""
    return make_batch([0, 37], [5, 40], 2, 1, 64, 16, seed=seed, sm_scale=0.125,
                      name="tiny: 2 seqs, prefix {0,37}, chunk {5,40}, 2q/1kv, D64, ps16",
                      pad_to_pages=8, pool_pages=16)


def zero_score_steps(page_size: int = 2, head_dim: int = 64,
                     chunks: Sequence[int] = (2, 2), n_q_heads: int = 1,
                     n_kv_heads: int = 1):
    """The zero-score regression of AReno PR #642 ("What does this PR do?"):
    a prompt split into chunks, Q = 0 and V_j = 2j + 1 in every lane.

    Returns a list of per-step Batches over one shared pool; step s holds the
    s-th chunk with the earlier chunks as its cached prefix.  The pool arrays
    of every step are the same objects: the caller appends each step's chunk
    before attending, exactly as a serving loop does."""
    total = int(sum(chunks))
    need = -(-total // page_size)
    rng = np.random.default_rng(7)
    num_pages = need + 2
    perm = rng.permutation(num_pages).astype(np.int32)
    pages = perm[:need]
    slots = num_pages * page_size
    k_pool = _normal_bf16(rng, (slots, n_kv_heads, head_dim))
    v_pool = _normal_bf16(rng, (slots, n_kv_heads, head_dim))
    steps = []
    start = 0
    for c in chunks:
        L = start + c
        npg = -(-L // page_size)
        pos = np.arange(start, L, dtype=np.float32)
        v_new = np.broadcast_to((2.0 * pos + 1.0)[:, None, None],
                                (c, n_kv_heads, head_dim)).astype(np.float32)
        steps.append(Batch(
            name=f"zero-score chunk at {start}", n_q_heads=n_q_heads,
            n_kv_heads=n_kv_heads, head_dim=head_dim, page_size=page_size, window=0,
            sm_scale=0.125, qo_indptr=np.array([0, c], np.int32),
            prefix_lens=np.array([start], np.int32),
            kv_indptr=np.array([0, npg], np.int32), kv_indices=pages[:npg].copy(),
            num_pages=num_pages, q=np.zeros((c, n_q_heads, head_dim), np.uint16),
            k_new=_normal_bf16(rng, (c, n_kv_heads, head_dim)),
            v_new=bf16_bits(v_new), k_pool=k_pool, v_pool=v_pool))
        start = L
    return steps


def gqa_prefill(seed: int = 1002, batch: int = 8, n_q_heads: int = 32, n_kv_heads: int = 8,
                head_dim: int = 128, page_size: int = 16, chunk: int = 512,
                max_prefix: int = 8192) -> Batch:
    """GQA chunked prefill (Qwen3-8B-like attention): prefix_lens uniform in
    [0, max_prefix], one chunk of ``chunk`` tokens per sequence, scattered
    pages from a shuffled pool, bottom-right causal, no window."""
    rng = np.random.default_rng(seed + 10_000)
    P = rng.integers(0, max_prefix + 1, size=batch)
    return make_batch(P, [chunk] * batch, n_q_heads, n_kv_heads, head_dim, page_size,
                      seed=seed,
                      name=f"GQA chunked prefill: B={batch}, {n_q_heads}q/{n_kv_heads}kv, "
                           f"D={head_dim}, ps={page_size}, chunk={chunk}, "
                           f"prefix~U[0,{max_prefix}]")


def mixed_batch(seed: int = 1003, prompt: int = 4097, chunk: int = 2048, n_decode: int = 31,
                n_q_heads: int = 16, n_kv_heads: int = 4, head_dim: int = 128,
                page_size: int = 64, decode_min: int = 32, decode_max: int = 8192) -> Batch:
    """A mixed scheduler batch in one ragged call: one ``prompt``-token prompt
    split into chunks of ``chunk`` tokens (the last one holds the remainder),
    all chunks sharing the prompt's page list, plus ``n_decode`` decode rows
    (one query each) with KV lengths uniform in [decode_min, decode_max]."""
    rng = np.random.default_rng(seed + 10_000)
    P, C = [], []
    start = 0
    while start < prompt:
        c = min(chunk, prompt - start)
        P.append(start)
        C.append(c)
        start += c
    n_prompt_rows = len(P)
    Ld = rng.integers(decode_min, decode_max + 1, size=n_decode)
    P += [int(l) - 1 for l in Ld]
    C += [1] * n_decode
    groups = [list(range(n_prompt_rows))] + [[n_prompt_rows + i] for i in range(n_decode)]
    return make_batch(P, C, n_q_heads, n_kv_heads, head_dim, page_size, seed=seed,
                      share_groups=groups,
                      name=f"mixed: {prompt}-token prompt as chunks of {chunk} + {n_decode} "
                           f"decode rows, {n_q_heads}q/{n_kv_heads}kv, D={head_dim}, "
                           f"ps={page_size}")


def decode_rows(seed: int = 1003, n_decode: int = 31, n_q_heads: int = 16, n_kv_heads: int = 4,
                head_dim: int = 128, page_size: int = 64, decode_min: int = 32,
                decode_max: int = 8192) -> Batch:
    """The decode rows of the mixed batch on their own (same lengths)."""
    rng = np.random.default_rng(seed + 10_000)
    Ld = rng.integers(decode_min, decode_max + 1, size=n_decode)
    return make_batch([int(l) - 1 for l in Ld], [1] * n_decode, n_q_heads, n_kv_heads,
                      head_dim, page_size, seed=seed,
                      name=f"decode rows: {n_decode} rows, KV~U[{decode_min},{decode_max}], "
                           f"{n_q_heads}q/{n_kv_heads}kv, D={head_dim}, ps={page_size}")


def stress_case(page_size: int, window: int, seed: int = 1004, batch: int = 64,
                n_q_heads: int = 8, n_kv_heads: int = 2, head_dim: int = 64,
                chunk_choices: Sequence[int] = (1, 7, 65, 128), max_prefix: int = 12288,
                pad_extra: int = 2) -> Batch:
    """Page-boundary and window stress: every chunk starts inside a page
    (prefix mod page_size uniform in [1, page_size-1]; for page_size 1 the
    prefix is uniform in [1, max_prefix]), chunk lengths drawn from
    ``chunk_choices``, a dense table padded with -1."""
    rng = np.random.default_rng(seed + 10_000 + 17 * page_size + (window > 0))
    if page_size > 1:
        base = rng.integers(0, max_prefix // page_size, size=batch) * page_size
        r = rng.integers(1, page_size, size=batch)
        P = base + r
    else:
        P = rng.integers(1, max_prefix + 1, size=batch)
    C = rng.choice(np.asarray(chunk_choices), size=batch)
    L = P + C
    width = int(max(-(-int(l) // page_size) for l in L)) + pad_extra
    return make_batch(P, C, n_q_heads, n_kv_heads, head_dim, page_size, seed=seed,
                      window=window, pad_to_pages=width,
                      name=f"stress: B={batch}, chunks {tuple(chunk_choices)}, ps={page_size}, "
                           f"window={window}, {n_q_heads}q/{n_kv_heads}kv, D={head_dim}")


def long_context(seed: int = 1005, batch: int = 4, prefix: int = 32768, chunk: int = 8192,
                 n_q_heads: int = 64, n_kv_heads: int = 8, head_dim: int = 128,
                 page_size: int = 64) -> Batch:
    """Long context: every sequence has ``prefix`` cached tokens and a
    ``chunk``-token chunk."""
    return make_batch([prefix] * batch, [chunk] * batch, n_q_heads, n_kv_heads, head_dim,
                      page_size, seed=seed,
                      name=f"long context: B={batch}, prefix={prefix}, chunk={chunk}, "
                           f"{n_q_heads}q/{n_kv_heads}kv, D={head_dim}, ps={page_size}")


def random_mask(batch: Batch, kind: str, seed: int, keep: float = 0.6) -> np.ndarray:
    """A seeded boolean attention mask (True = keep) for ``batch``, laid out
    as the attention call takes it:

    * ``"2d"``       [B, kv]          one key mask per sequence
    * ``"4d_bcast"`` [B, 1, q, kv]    per query row, shared by all heads
    * ``"4d_heads"`` [B, Hq, q, kv]   per query row and head
    * ``"4d_q1"``    [B, 1, 1, kv]    broadcast over rows and heads

    q is the longest chunk, kv the longest KV length rounded up to a multiple
    of 16 (entries past a sequence's end are never read).  Each entry is True
    with probability ``keep``."""
    rng = np.random.default_rng(seed)
    B = batch.batch
    qmax = int(batch.chunk_lens.max()) if B else 1
    kv = int(-(-int(batch.kv_lens.max()) // 16) * 16) if B else 16
    shape = {"2d": (B, kv), "4d_bcast": (B, 1, max(qmax, 1), kv),
             "4d_heads": (B, batch.n_q_heads, max(qmax, 1), kv),
             "4d_q1": (B, 1, 1, kv)}[kind]
    return rng.random(shape) < keep


CONFIGS = {
    "tiny": tiny_case,
    "gqa_prefill": gqa_prefill,
    "mixed": mixed_batch,
    "decode_rows": decode_rows,
    "stress_ps1_w4096": lambda: stress_case(1, 4096),
    "stress_ps1_w0": lambda: stress_case(1, 0),
    "stress_ps16_w4096": lambda: stress_case(16, 4096),
    "stress_ps16_w0": lambda: stress_case(16, 0),
    "long_context": long_context,
}


def config_by_name(name: str) -> Batch:
    return CONFIGS[name]()
