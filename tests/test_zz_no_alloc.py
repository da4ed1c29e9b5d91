"""pcp_paged_extend_attn_noalloc: extend attention for callers that cannot
allocate device memory.

Callers such as code inside a host framework that owns every device
allocation, or a plugin interface with no allocation hook, cannot hand the
library a workspace.  This entry point takes its scratch from a fixed
device array inside the library instead.  The test calls it through the C ABI
twice in a row, on two different batches (both with split-KV decode rows, so
the shared scratch's counters and partials from the first call are still
there when the second one runs), and compares each result with the regular
entry point, which gets a workspace from PyTorch.  Both run the same
deterministic kernels on the same inputs, so the results must be identical
bit for bit.  It also checks that a call needing more than the fixed scratch
is refused before anything runs, after the same argument checks as the
regular entry point.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it.
"""
import ctypes

import pytest

import workloads as W
from helpers import to_device

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import paged_chunked_prefill_gb300 as pcp
    f = pcp.lib().pcp_paged_extend_attn_noalloc
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, i32, i64, P, P, i64, i32, i32, i32, i32, i32, f32, P, P, P,
                  P]
    f.restype = i32
    return f


def _run_both(batch):
    import torch
    import paged_chunked_prefill_gb300 as pcp
    d = to_device(batch)
    loc = pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                    d["prefix_lens"], batch.page_size, batch.num_pages,
                                    total_q=batch.total_q)
    pcp.kv_append(d["k_new"], d["v_new"], loc, d["k_pool"], d["v_pool"])
    ref_out, ref_lse = pcp.paged_extend_attn(
        d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"], d["k_pool"],
        d["v_pool"], batch.page_size, batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
        batch.window, batch.sm_scale)
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full((batch.total_q, batch.n_q_heads), float("nan"), dtype=torch.float32,
                     device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = _noalloc_fn()(ptr(d["q"]), ptr(d["qo_indptr"]), ptr(d["kv_indptr"]),
                       ptr(d["kv_indices"]), ptr(d["prefix_lens"]), ctypes.c_void_p(0),
                       batch.batch, batch.total_q,
                       ptr(d["k_pool"]), ptr(d["v_pool"]), batch.num_pages, batch.page_size,
                       batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.window,
                       float(batch.sm_scale), ptr(out), ptr(lse), ptr(err), stream)
    assert st == 0, pcp.lib().pcp_status_string(st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # same kernels, same inputs: bit-identical results
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    first = W.mixed_batch(prompt=700, chunk=300, n_decode=9, decode_max=3000)
    second = W.make_batch([0, 1200, 4000, 31], [260, 1, 1, 97], 32, 8, 128, 16, seed=91,
                          window=0)
    _run_both(first)
    _run_both(second)


def test_noalloc_refuses_oversized_calls():
    import paged_chunked_prefill_gb300 as pcp
    need = pcp.workspace_size(4096, 65536, 32, 8, 128)
    assert need > 16 * 1024 * 1024
    P = ctypes.c_void_p
    one = P(0x1000)  # never dereferenced: both calls return before any launch
    err = P(0x2000)
    st = _noalloc_fn()(one, one, one, one, one, P(0), 4096, 65536, one, one, 1, 16, 32, 8,
                       128, 0, 0.0, one, one, err, P(0))
    assert st == pcp.Status.WORKSPACE
    # a bad argument is reported as such, also on an oversized call
    st = _noalloc_fn()(one, one, one, one, one, P(0), 4096, 65536, one, one, 1, 16, 30, 8,
                       128, 0, 0.0, one, one, err, P(0))
    assert st == pcp.Status.INVALID_ARG
