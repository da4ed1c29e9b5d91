"""Shared test helpers: move a workload to the GPU, run the CUDA path through
the C ABI, sample rows, and compare with the FP64 oracle.

Tolerances: bf16 out max-abs 2e-2 and mean-abs 2e-3, lse 1e-3 absolute;
out_cache_loc and the appended pools bit-exact.
"""
from __future__ import annotations

import numpy as np

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3


def torch_mod():
    import torch
    return torch


def to_device(batch, device="cuda"):
    torch = torch_mod()
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).to(device)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)
    return dict(
        q=t16(batch.q), k_new=t16(batch.k_new), v_new=t16(batch.v_new),
        k_pool=t16(batch.k_pool), v_pool=t16(batch.v_pool),
        qo_indptr=i32(batch.qo_indptr), kv_indptr=i32(batch.kv_indptr),
        kv_indices=i32(batch.kv_indices if len(batch.kv_indices) else np.zeros(1, np.int32)),
        prefix_lens=i32(batch.prefix_lens if len(batch.prefix_lens) else np.zeros(1, np.int32)),
    )


def bf16_tensor_to_f64(t) -> np.ndarray:
    torch = torch_mod()
    u = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_tensor_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(batch, d=None, check=True, host_hint=True, causal=True, mask=None):
    """out_cache_loc -> kv_append -> paged_extend_attn on the GPU (with the
    host copy of qo_indptr unless host_hint is False; ``mask`` a numpy bool
    array, moved to the device)."""
    import paged_chunked_prefill_gb300 as pcp
    if d is None:
        d = to_device(batch)
    loc = pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                    d["prefix_lens"], batch.page_size, batch.num_pages,
                                    total_q=batch.total_q, check=check)
    pcp.kv_append(d["k_new"], d["v_new"], loc, d["k_pool"], d["v_pool"], check=check)
    out, lse = pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["prefix_lens"], d["k_pool"], d["v_pool"],
                                     batch.page_size, batch.n_q_heads, batch.n_kv_heads,
                                     batch.head_dim, batch.window, batch.sm_scale, check=check,
                                     qo_indptr_host=batch.qo_indptr if host_hint else None,
                                     causal=causal,
                                     mask=None if mask is None else
                                     torch_mod().from_numpy(np.ascontiguousarray(mask)).to(
                                         d["q"].device))
    return loc, d, out, lse


def sample_rows(batch, n_random=256, seed=0):
    """(tokens, heads): random rows plus the first/last row of every chunk and
    rows at page and 128-key tile boundaries, every head for the edge rows of
    the first sequences."""
    rng = np.random.default_rng(seed)
    toks, heads = [], []
    Hq = batch.n_q_heads
    for b in range(batch.batch):
        q0, q1 = int(batch.qo_indptr[b]), int(batch.qo_indptr[b + 1])
        if q1 == q0:
            continue
        P = int(batch.prefix_lens[b])
        edge = {q0, q1 - 1}
        for i in range(q1 - q0):
            p = P + i
            if p % batch.page_size == 0 or p % 128 in (0, 127) or (
                    batch.window > 0 and i < 2):
                edge.add(q0 + i)
            if len(edge) > 8:
                break
        for t in sorted(edge):
            hs = range(Hq) if b < 2 else [int(rng.integers(0, Hq))]
            for h in hs:
                toks.append(t)
                heads.append(h)
    toks += list(rng.integers(0, max(batch.total_q, 1), size=n_random))
    heads += list(rng.integers(0, Hq, size=n_random))
    return np.asarray(toks, np.int64), np.asarray(heads, np.int32)


def assert_close(out_gpu: np.ndarray, lse_gpu: np.ndarray, out_ref: np.ndarray,
                 lse_ref: np.ndarray, what: str = "") -> dict:
    err = np.abs(out_gpu - out_ref)
    lerr = np.abs(lse_gpu - lse_ref)
    stats = dict(max_abs=float(err.max(initial=0.0)), mean_abs=float(err.mean()) if err.size else 0.0,
                 lse_max=float(lerr.max(initial=0.0)))
    assert np.isfinite(out_gpu).all(), f"{what}: non-finite output"
    assert stats["max_abs"] <= OUT_MAX_ABS, f"{what}: out max-abs {stats}"
    assert stats["mean_abs"] <= OUT_MEAN_ABS, f"{what}: out mean-abs {stats}"
    assert stats["lse_max"] <= LSE_ABS, f"{what}: lse {stats}"
    return stats
