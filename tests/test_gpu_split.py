"""Tensor-core items split along their KV tiles.

With host copies of qo_indptr and prefix_lens, a call whose longest
tensor-core item is more than 1.3 times the average work per SM has its
longest items split in two (the items above half that average and above 16
KV tiles, at most 64): each part is an item of its own in the longest-first
queue, and the part that ends second merges the other's partial result (per
warp, through a ticket and a ready flag, part 0's terms first).  The
workspace header's item count shows the split; every row is compared with
the FP64 oracle.  Without the host copy of prefix_lens the same call runs
unsplit, within the same tolerance.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_bits, bf16_tensor_to_f64, to_device

pytestmark = pytest.mark.gpu


def _run(batch, prefix_host):
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
                                     qo_indptr_host=batch.qo_indptr,
                                     prefix_lens_host=batch.prefix_lens if prefix_host else None)
    n_items = int(ws[:4].view(torch.int32).item())
    loc_ref, kp_ref, vp_ref, out_ref, lse_ref = oracle.run_batch(batch)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    np.testing.assert_array_equal(bf16_tensor_bits(d["k_pool"]), kp_ref)
    assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref,
                 lse_ref, f"{batch.name}, prefix_lens host copy {prefix_host}")
    return n_items


def _unsplit_items(batch):
    """Tensor-core items with the decode-shaped chunks taken on (they are, in
    every batch here)."""
    G = batch.n_q_heads // batch.n_kv_heads
    rmax = 16 // G if G <= 16 else 0
    item_pos = 2 * (128 // G)
    n = sum((-(-int(c) // item_pos) if c > rmax else 1) for c in batch.chunk_lens if c > 0)
    return n * batch.n_kv_heads


CASES = {
    # page-boundary stress batches at head_dim 64: page boxes and cp.async gathers
    "stress_ps16": lambda: W.stress_case(16, 0, batch=24, max_prefix=6000),
    "stress_ps1": lambda: W.stress_case(1, 0, batch=24, max_prefix=6000),
    # head_dim 128: one long prefix beside short ones, a decode row among them
    "long_beside_short": lambda: W.make_batch([9000, 100, 2500, 40], [64, 64, 100, 1], 16, 4,
                                              128, 16, seed=5, name="long beside short"),
    "long_beside_short_window": lambda: W.make_batch([9000, 100, 2500, 40], [64, 64, 100, 1],
                                                     16, 4, 128, 16, seed=5, window=5000,
                                                     name="long beside short, window 5000"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_split_items_match_the_oracle(case):
    b = CASES[case]()
    n_split = _run(b, True)
    n_plain = _run(b, False)
    assert n_plain == _unsplit_items(b)
    assert n_split > n_plain   # every split item adds a part
