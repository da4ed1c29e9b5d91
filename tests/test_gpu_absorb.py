"""Decode-shaped chunks in a call with tensor-core work.

The planner takes a call's decode-shaped chunks (chunk_len * G <= 16 rows)
onto the tensor cores, as one-Q-tile items in the longest-first queue, when
the longest of them stays within 1.1 times the schedule's expected length
(its longest prompt item, or the average work per SM); otherwise they stay
on the split-KV row kernel.  Both outcomes are checked here against the FP64
oracle over every row, and the workspace header (n_tc_items, n_row_groups,
tc_next, row_tiles, row_ctas: the first five int32 of the workspace) shows
which one the planner took.  The call runs without host copies (the planner
decides on the device), with the host copy of qo_indptr only (the same), and
with host copies of qo_indptr and prefix_lens (the host decides with the
same rule and skips the kernels without work); the outcome is the same in
all three.  Either way out_cache_loc and the pools are bit-exact.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_bits, bf16_tensor_to_f64, to_device

pytestmark = pytest.mark.gpu


HINTS = ["none", "qo_indptr", "qo_indptr+prefix_lens"]


def _run(batch, hint):
    import torch
    import paged_chunked_prefill_gb300 as pcp
    d = to_device(batch)
    loc = pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                    d["prefix_lens"], batch.page_size, batch.num_pages,
                                    total_q=batch.total_q)
    pcp.kv_append(d["k_new"], d["v_new"], loc, d["k_pool"], d["v_pool"])
    ws = torch.zeros(pcp.workspace_size(batch.batch, batch.total_q, batch.n_q_heads,
                                        batch.n_kv_heads, batch.head_dim),
                     dtype=torch.uint8, device="cuda")
    out, lse = pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["prefix_lens"], d["k_pool"], d["v_pool"],
                                     batch.page_size, batch.n_q_heads, batch.n_kv_heads,
                                     batch.head_dim, batch.window, batch.sm_scale, workspace=ws,
                                     qo_indptr_host=None if hint == "none" else batch.qo_indptr,
                                     prefix_lens_host=batch.prefix_lens
                                     if hint == "qo_indptr+prefix_lens" else None)
    header = ws[:20].view(torch.int32).cpu().numpy()
    loc_ref, kp_ref, vp_ref, out_ref, lse_ref = oracle.run_batch(batch)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["k_pool"]), kp_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["v_pool"]), vp_ref)
    assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref,
                 lse_ref, batch.name)
    return header


def _items(batch, rmax):
    """Tensor-core items of a call whose decode-shaped chunks are taken on."""
    G = batch.n_q_heads // batch.n_kv_heads
    item_pos = 2 * (128 // G)
    n = 0
    for c in batch.chunk_lens:
        if c > 0:
            n += -(-int(c) // item_pos) if c > rmax else 1
    return n * batch.n_kv_heads


@pytest.mark.parametrize("hint", HINTS)
@pytest.mark.parametrize("window", [0, 300])
def test_short_decode_rows_join_the_tensor_core_queue(hint, window):
    """A 1000-token prompt as chunks 512 / 488 beside 12 decode rows (and a
    4-token chunk) whose KV lengths stay under 1000: every decode-shaped item
    is shorter than the longest prompt item, so all of them go to the tensor
    cores and the row path gets nothing."""
    rng = np.random.default_rng(11)
    Ld = rng.integers(32, 1000, size=12)
    P = [0, 512] + [int(l) - 1 for l in Ld] + [600]
    C = [512, 488] + [1] * 12 + [4]
    groups = [[0, 1]] + [[i] for i in range(2, len(C))]
    b = W.make_batch(P, C, 16, 4, 128, 16, seed=12, window=window, share_groups=groups,
                     name=f"prompt 512+488 beside 12 short decode rows, window {window}")
    h = _run(b, hint)
    assert h[1] == 0 and h[3] == 0          # no row groups, no row tiles
    assert h[0] == _items(b, rmax=4)


@pytest.mark.parametrize("hint", HINTS)
def test_long_decode_rows_stay_on_the_row_kernel(hint):
    """A 64-token prompt beside 8 decode rows of 3000 to 6000 keys: one
    decode-shaped item would outlast the whole tensor-core schedule, so the
    decode rows stay on the split-KV row kernel."""
    rng = np.random.default_rng(13)
    Ld = rng.integers(3000, 6000, size=8)
    P = [0] + [int(l) - 1 for l in Ld]
    C = [64] + [1] * 8
    b = W.make_batch(P, C, 16, 4, 128, 16, seed=14,
                     name="prompt 64 beside 8 decode rows of 3000-6000 keys")
    h = _run(b, hint)
    assert h[1] == 8 * 4 and h[3] > 0       # one row group per (sequence, KV head)
    assert h[0] == 4                         # the prompt's one item per KV head


@pytest.mark.parametrize("hint", ["none", "qo_indptr+prefix_lens"])
def test_stress_page_size_one_absorbs_its_one_token_chunks(hint):
    """The page-boundary stress batch over a one-slot-per-token pool (chunks of
    1, 7, 65 and 128 tokens, prefixes up to 12288): its longest items are the
    prompt chunks' own, so the 1-token chunks join the tensor-core queue."""
    b = W.stress_case(1, 0, batch=24, max_prefix=3000)
    h = _run(b, hint)
    assert (b.chunk_lens == 1).any()
    assert h[1] == 0 and h[3] == 0
