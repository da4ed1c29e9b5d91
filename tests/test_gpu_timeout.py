"""The bounded waits of the tensor-core and row kernels, made to run out.

Every producer/consumer wait of the two kernels gives up after 2 s.  A wait
that gives up records PCP_ERR_TIMEOUT in the error word, the CTA's other
warps give up their waits, and the CTA lets the copies and MMAs it has in
flight complete, frees its tensor memory and exits.  Here a call runs with the
test stall of the per-call options: every CTA's first pipeline wait is made
on an mbarrier that nothing arrives on, with a limit of 0.2 ms, while its
load warps have copies in flight.  The call must report PCP_ERR_TIMEOUT, and
an ordinary call on the same stream right after it must match the FP64
oracle.  Nothing here faults or hangs a GPU: every wait has a limit, and the
waits that drain a giving-up CTA keep theirs at 2 s.

The cases cover the tensor-core kernel with TMA page boxes (page size 64)
and with cp.async page gathers (page size 1), and the split-KV row kernel
(decode rows only, so the tensor-core kernel has no work).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import assert_close, bf16_tensor_to_f64, to_device

pytestmark = pytest.mark.gpu


def _append(batch, d):
    import paged_chunked_prefill_gb300 as pcp
    loc = pcp.compute_out_cache_loc(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                    d["prefix_lens"], batch.page_size, batch.num_pages,
                                    total_q=batch.total_q)
    pcp.kv_append(d["k_new"], d["v_new"], loc, d["k_pool"], d["v_pool"])


def _attend(batch, d, err, test_stall_ns=0):
    import paged_chunked_prefill_gb300 as pcp
    return pcp.paged_extend_attn(d["q"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                 d["prefix_lens"], d["k_pool"], d["v_pool"], batch.page_size,
                                 batch.n_q_heads, batch.n_kv_heads, batch.head_dim,
                                 batch.window, batch.sm_scale, dev_err=err,
                                 qo_indptr_host=batch.qo_indptr, test_stall_ns=test_stall_ns)


CASES = {
    # prefill chunks only: the tensor-core kernel, TMA page boxes
    "tc_boxes": lambda: W.make_batch([0, 300, 1000], [384, 256, 200], 16, 4, 128, 64, seed=71),
    # the same over a one-slot-per-token pool: cp.async page gathers
    "tc_gathers": lambda: W.make_batch([0, 300, 1000], [384, 256, 200], 16, 4, 128, 1,
                                       seed=72),
    # decode rows only: the split-KV row kernel and the combine
    "rows": lambda: W.decode_rows(n_decode=24, decode_max=6000),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_wait_timeout_is_reported_and_the_next_call_is_correct(case):
    import torch
    import paged_chunked_prefill_gb300 as pcp
    batch = CASES[case]()
    d = to_device(batch)
    _append(batch, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _attend(batch, d, err, test_stall_ns=200_000)
    assert pcp.read_error(err) == pcp.Status.TIMEOUT
    # the same stream goes on: an ordinary call matches the oracle
    err.zero_()
    out, lse = _attend(batch, d, err)
    assert pcp.read_error(err) == 0
    kp = d["k_pool"].view(torch.int16).cpu().numpy().view(np.uint16)
    vp = d["v_pool"].view(torch.int16).cpu().numpy().view(np.uint16)
    out_ref, lse_ref = oracle.paged_extend_attn(
        batch.q, batch.qo_indptr, batch.kv_indptr, batch.kv_indices, batch.prefix_lens, kp, vp,
        batch.page_size, batch.n_q_heads, batch.n_kv_heads, batch.head_dim, batch.window,
        batch.sm_scale)
    assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref,
                 lse_ref, f"after a timed-out call ({case})")
