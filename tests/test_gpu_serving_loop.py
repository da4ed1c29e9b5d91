"""A serving loop planned by the library's chunk planner, run on the GPU.

Every step: ``Pager.schedule_step`` chooses the chunks (token budget 2048,
decode-shaped rows first) and hands out pages; the GPU maps the new tokens to
slots, appends their K/V and runs extend attention; the FP64 oracle runs the
same step on its own copy of the pools.  The workload is the mixed scheduler
batch of the pages: a 4097-token prompt (chunks 2048 / 2048 / 1 under the
budget) arriving while shorter requests prefill and then decode.

Checked: slots and pools bit-exact every step, out / lse within tolerance.
"""
import numpy as np
import pytest

import oracle
import paged_chunked_prefill_gb300 as pcp
import workloads as W
from helpers import assert_close, bf16_tensor_bits, bf16_tensor_to_f64

pytestmark = pytest.mark.gpu


def test_planned_serving_loop():
    import torch
    rng = np.random.default_rng(2024)
    Hq, Hkv, D, ps = 16, 4, 128, 64
    num_pages = 200
    # token streams of each request (prompt + the tokens it will decode)
    prompts = [4097, 300, 45, 1000, 130]
    decodes = [2, 6, 6, 3, 6]
    streams = []
    for P, n in zip(prompts, decodes):
        T = P + n
        streams.append({
            "q": W.bf16_bits(rng.standard_normal((T, Hq, D), dtype=np.float32)),
            "k": W.bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32)),
            "v": W.bf16_bits(rng.standard_normal((T, Hkv, D), dtype=np.float32)),
        })
    pool_k = W.bf16_bits(rng.standard_normal((num_pages * ps, Hkv, D), dtype=np.float32))
    pool_v = W.bf16_bits(rng.standard_normal((num_pages * ps, Hkv, D), dtype=np.float32))
    t16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()
    gk, gv = t16(pool_k), t16(pool_v)
    ok, ov = pool_k.copy(), pool_v.copy()

    pager = pcp.Pager(num_pages, ps)
    total = [p for p in prompts]
    computed = [0] * len(prompts)
    left = list(decodes)
    active = [0, 1, 2]          # the 4097-token prompt arrives with two others
    arrivals = {2: [3], 4: [4]}
    n_rows_seen = 0
    for step in range(40):
        active += arrivals.get(step, [])
        if not active:
            break
        st = pager.schedule_step(active, [total[r] for r in active],
                                 [computed[r] for r in active], 2048)
        rows = [active[i] for i in st["row_req"]]
        qo = st["qo_indptr"]
        if len(rows) == 0:
            continue
        n_rows_seen += len(rows)
        q = np.concatenate([streams[r]["q"][st["prefix_lens"][n]:st["prefix_lens"][n] +
                                            qo[n + 1] - qo[n]] for n, r in enumerate(rows)])
        k = np.concatenate([streams[r]["k"][st["prefix_lens"][n]:st["prefix_lens"][n] +
                                            qo[n + 1] - qo[n]] for n, r in enumerate(rows)])
        v = np.concatenate([streams[r]["v"][st["prefix_lens"][n]:st["prefix_lens"][n] +
                                            qo[n + 1] - qo[n]] for n, r in enumerate(rows)])
        # GPU
        dq, dqo, dkvp = t16(q), i32(qo), i32(st["kv_indptr"])
        dkvi, dpre = i32(st["kv_indices"]), i32(st["prefix_lens"])
        loc = pcp.compute_out_cache_loc(dqo, dkvp, dkvi, dpre, ps, num_pages,
                                        total_q=int(qo[-1]))
        pcp.kv_append(t16(k), t16(v), loc, gk, gv)
        out, lse = pcp.paged_extend_attn(dq, dqo, dkvp, dkvi, dpre, gk, gv, ps, Hq, Hkv, D,
                                         qo_indptr_host=qo)
        # oracle
        loc_ref = oracle.out_cache_loc(qo, st["kv_indptr"], st["kv_indices"], st["prefix_lens"],
                                       ps, num_pages)
        np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
        oracle.kv_append(k, v, loc_ref, ok, ov)
        out_ref, lse_ref = oracle.paged_extend_attn(q, qo, st["kv_indptr"], st["kv_indices"],
                                                    st["prefix_lens"], ok, ov, ps, Hq, Hkv, D)
        assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), out_ref,
                     lse_ref, f"step {step}")
        # advance: chunks ran; a sampled request decodes its next token or ends
        for n, r in enumerate(rows):
            computed[r] += int(qo[n + 1] - qo[n])
            if st["sample"][n]:
                if left[r] > 0:
                    total[r] += 1
                    left[r] -= 1
                else:
                    pager.release(r)
                    active.remove(r)
    assert not active and n_rows_seen > 20
    np.testing.assert_array_equal(bf16_tensor_bits(gk), ok)
    np.testing.assert_array_equal(bf16_tensor_bits(gv), ov)
    assert pager.num_free() == num_pages
