"""The append of a step's new K/V rows inside the attention call.

With k_new / v_new in the call options the call does what pcp_kv_append_paged
does (slot mapping from the page table, scatter into the pools), in the
planner's launch beside the planning CTA (when it fits in one wave there),
or as a kernel of its own ahead of the planner or of a self-planned row
kernel, and then attends.  Pools, slots, out, lse and the error code equal
those of pcp_kv_append_paged followed by the same call, bit for bit; one case
is also compared with the FP64 oracle.
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_to_f64, to_device

pytestmark = pytest.mark.gpu


def _run(batch, fused, hints, mask=None):
    import torch
    import paged_chunked_prefill_gb300 as pcp
    d = to_device(batch)
    loc = torch.full((batch.total_q,), -7, dtype=torch.int64, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(qo_indptr_host=batch.qo_indptr, prefix_lens_host=batch.prefix_lens) if hints else {}
    if mask is not None:
        kw["mask"] = torch.from_numpy(mask).cuda()
    args = (d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"],
            d["k_pool"], d["v_pool"], batch.page_size, batch.n_q_heads, batch.n_kv_heads,
            batch.head_dim, batch.window, batch.sm_scale)
    if fused:
        out, lse = pcp.paged_extend_attn(*args, k_new=d["k_new"], v_new=d["v_new"],
                                         out_cache_loc=loc, dev_err=err, check=False, **kw)
    else:
        pcp.kv_append_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["prefix_lens"],
                            batch.page_size, d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                            out_cache_loc=loc, dev_err=err, check=False)
        out, lse = pcp.paged_extend_attn(*args, dev_err=err, check=False, **kw)
    code = pcp.read_error(err)
    return loc, d["k_pool"], d["v_pool"], out, lse, code


def _assert_same(batch, hints, mask=None):
    import torch
    a = _run(batch, False, hints, mask)
    b = _run(batch, True, hints, mask)
    assert a[5] == b[5]
    assert torch.equal(a[0], b[0])
    for x, y in zip(a[1:5], b[1:5]):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32))
    return b


CASES = {
    "tiny": lambda: W.tiny_case(),
    "mixed": lambda: W.mixed_batch(prompt=700, chunk=300, n_decode=9, decode_max=3000),
    "stress_ps1": lambda: W.stress_case(1, 0, batch=24, max_prefix=3000),
    "stress_ps16_w4096": lambda: W.stress_case(16, 4096, batch=24, max_prefix=6000),
    "gqa_d64": lambda: W.gqa_prefill(batch=3, head_dim=64, chunk=200, max_prefix=2000),
    # 5120 new tokens of 8 KV heads at D=128: 160 spans of 4096 chunks, more
    # than one wave beside the planner, so the append runs as its own kernel
    "gqa_long_append": lambda: W.gqa_prefill(batch=10, chunk=512, max_prefix=1000),
    # empty chunks among the others, a chunk starting mid-page, one at prefix 0
    "empty_chunks": lambda: W.make_batch([0, 37, 500, 9, 1200], [0, 70, 0, 1, 300], 16, 4, 128,
                                         16, seed=12, window=600),
    # decode-shaped rows only: self-planned by the row kernel with the hints,
    # planned by the planner kernel without them
    "decode_only": lambda: W.decode_rows(n_decode=12, decode_max=3000),
}


@pytest.mark.parametrize("hints", [False, True])
@pytest.mark.parametrize("case", sorted(CASES))
def test_append_in_call_is_bit_identical(case, hints):
    b = _assert_same(CASES[case](), hints)
    assert b[5] == 0


def test_append_in_call_without_new_rows():
    """A call with no query rows at all: nothing to append, nothing launched,
    the pools untouched."""
    import torch
    import paged_chunked_prefill_gb300 as pcp
    b = W.make_batch([40, 7], [0, 0], 8, 2, 64, 16, seed=13)
    d = to_device(b)
    before = d["k_pool"].clone()
    empty = torch.empty(0, b.n_kv_heads, b.head_dim, dtype=torch.bfloat16, device="cuda")
    out, lse = pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["prefix_lens"], d["k_pool"], d["v_pool"], b.page_size,
                                     b.n_q_heads, b.n_kv_heads, b.head_dim,
                                     qo_indptr_host=b.qo_indptr, prefix_lens_host=b.prefix_lens,
                                     k_new=empty, v_new=empty)
    torch.cuda.synchronize()
    assert out.numel() == 0 and lse.numel() == 0
    assert torch.equal(d["k_pool"].view(torch.int16), before.view(torch.int16))


def test_append_in_call_with_mask():
    batch = CASES["mixed"]()
    mask = W.random_mask(batch, "2d", seed=7)
    _assert_same(batch, True, mask)


def test_append_in_call_matches_the_oracle():
    batch = CASES["mixed"]()
    loc, kp, vp, out, lse, code = _run(batch, True, True)
    assert code == 0
    loc_ref, kp_ref, vp_ref, out_ref, lse_ref = oracle.run_batch(batch)
    np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
    assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref, lse_ref,
                 "append in the call")


def test_append_in_call_reports_bad_page():
    """A bad page id among a chunk's pages: the same error code, slots and
    pools as the separate append followed by the call."""
    b = W.make_batch([10, 300], [50, 130], 8, 2, 64, 16, seed=41)
    bad = b.kv_indices.copy()
    bad[3] = -1
    b2 = W.Batch(**{**b.__dict__, "kv_indices": bad})
    import paged_chunked_prefill_gb300 as pcp
    res = _assert_same(b2, True)
    assert res[5] == pcp.Status.BAD_INDEX
