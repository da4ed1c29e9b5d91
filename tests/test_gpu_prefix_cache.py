"""Shared pages on the GPU: the copy-on-write kernel, and attention over a
re-asked prompt's reused pages and over forked continuations.

* ``pcp_copy_page_slots`` is bit-exact against a numpy copy of the same
  slots;
* a request whose prompt repeats a cached prompt's first 250 tokens reuses
  floor(249 / 16) * 16 = 240 of them (the pages' hit law), computes only the
  rest, and its outputs match the oracle run over the same page lists;
* a prompt forked into a second continuation: the first write into the
  shared, partly filled page copies it on the device; both continuations
  then match the oracle, and the pools match a numpy model of the copies and
  appends bit for bit.
"""
import numpy as np
import pytest

import oracle
import paged_chunked_prefill_gb300 as pcp
import workloads as W
from helpers import assert_close, bf16_tensor_bits, bf16_tensor_to_f64

pytestmark = pytest.mark.gpu

HQ, HKV, D, PS = 8, 2, 128, 16


def t16(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def test_copy_page_slots_bit_exact():
    rng = np.random.default_rng(5)
    num_pages = 12
    k = W.bf16_bits(rng.standard_normal((num_pages * PS, HKV, D), dtype=np.float32))
    v = W.bf16_bits(rng.standard_normal((num_pages * PS, HKV, D), dtype=np.float32))
    src, dst, n = [3, 7, 0], [10, 2, 11], [5, 16, 0]
    gk, gv = t16(k), t16(v)
    pcp.copy_page_slots(gk, gv, PS, i32(src), i32(dst), i32(n))
    for s, d, c in zip(src, dst, n):
        k[d * PS:d * PS + c] = k[s * PS:s * PS + c]
        v[d * PS:d * PS + c] = v[s * PS:s * PS + c]
    np.testing.assert_array_equal(bf16_tensor_bits(gk), k)
    np.testing.assert_array_equal(bf16_tensor_bits(gv), v)


class Runner:
    """Runs planned steps on the GPU and on the oracle side by side."""

    def __init__(self, num_pages, seed):
        rng = np.random.default_rng(seed)
        self.num_pages = num_pages
        kp = W.bf16_bits(rng.standard_normal((num_pages * PS, HKV, D), dtype=np.float32))
        vp = W.bf16_bits(rng.standard_normal((num_pages * PS, HKV, D), dtype=np.float32))
        self.gk, self.gv = t16(kp), t16(vp)
        self.ok, self.ov = kp.copy(), vp.copy()
        self.pager = pcp.Pager(num_pages, PS)

    def step(self, ids, streams, total, computed, budget=4096):
        st = self.pager.schedule_step(ids, [total[i] for i in ids], [computed[i] for i in ids],
                                      budget)
        if st["copy_src"].size:
            pcp.copy_page_slots(self.gk, self.gv, PS, i32(st["copy_src"]), i32(st["copy_dst"]),
                                i32(st["copy_slots"]))
            for s, d, c in zip(st["copy_src"], st["copy_dst"], st["copy_slots"]):
                self.ok[d * PS:d * PS + c] = self.ok[s * PS:s * PS + c]
                self.ov[d * PS:d * PS + c] = self.ov[s * PS:s * PS + c]
        qo = st["qo_indptr"]
        rows = [ids[i] for i in st["row_req"]]
        part = lambda key: np.concatenate(
            [streams[r][key][st["prefix_lens"][n]:st["prefix_lens"][n] + qo[n + 1] - qo[n]]
             for n, r in enumerate(rows)])
        q, k, v = part("q"), part("k"), part("v")
        dqo, dkvp, dkvi, dpre = i32(qo), i32(st["kv_indptr"]), i32(st["kv_indices"]), \
            i32(st["prefix_lens"])
        loc = pcp.compute_out_cache_loc(dqo, dkvp, dkvi, dpre, PS, self.num_pages,
                                        total_q=int(qo[-1]))
        pcp.kv_append(t16(k), t16(v), loc, self.gk, self.gv)
        out, lse = pcp.paged_extend_attn(t16(q), dqo, dkvp, dkvi, dpre, self.gk, self.gv, PS,
                                         HQ, HKV, D, qo_indptr_host=qo)
        loc_ref = oracle.out_cache_loc(qo, st["kv_indptr"], st["kv_indices"], st["prefix_lens"],
                                       PS, self.num_pages)
        np.testing.assert_array_equal(loc.cpu().numpy(), loc_ref)
        oracle.kv_append(k, v, loc_ref, self.ok, self.ov)
        o_ref, l_ref = oracle.paged_extend_attn(q, qo, st["kv_indptr"], st["kv_indices"],
                                                st["prefix_lens"], self.ok, self.ov, PS, HQ, HKV,
                                                D)
        assert_close(bf16_tensor_to_f64(out), lse.cpu().numpy().astype(np.float64), o_ref, l_ref,
                     "shared-page step")
        for n, r in enumerate(rows):
            computed[r] += int(qo[n + 1] - qo[n])
        return st

    def check_pools(self):
        np.testing.assert_array_equal(bf16_tensor_bits(self.gk), self.ok)
        np.testing.assert_array_equal(bf16_tensor_bits(self.gv), self.ov)


def stream(rng, T):
    return {"q": W.bf16_bits(rng.standard_normal((T, HQ, D), dtype=np.float32)),
            "k": W.bf16_bits(rng.standard_normal((T, HKV, D), dtype=np.float32)),
            "v": W.bf16_bits(rng.standard_normal((T, HKV, D), dtype=np.float32))}


def test_reask_reuses_cached_pages():
    rng = np.random.default_rng(6)
    run = Runner(64, 7)
    tok_a = rng.integers(0, 1000, size=300).astype(np.int32)
    tok_b = np.concatenate([tok_a[:250], rng.integers(0, 1000, size=60).astype(np.int32)])
    sa = stream(rng, 300)
    sb = stream(rng, 310)
    for key in ("k", "v"):                 # the shared prefix has the same K/V
        sb[key][:250] = sa[key][:250]
    streams = {0: sa, 1: sb}
    total, computed = {0: 300, 1: 310}, {0: 0, 1: 0}
    run.step([0], streams, total, computed)
    run.pager.cache_prompt(0, tok_a)
    hit = run.pager.match_prefix(1, tok_b)
    assert hit == 240
    computed[1] = hit
    free_before = run.pager.num_free()
    st = run.step([1], streams, total, computed)
    assert st["prefix_lens"].tolist() == [240]
    assert (run.pager.request_pages(1)[:15] == run.pager.request_pages(0)[:15]).all()
    assert free_before - run.pager.num_free() == -(-310 // PS) - 15
    run.check_pools()


def test_fork_copy_on_write_continuations():
    rng = np.random.default_rng(8)
    run = Runner(40, 9)
    base = stream(rng, 300)
    s1, s2 = stream(rng, 305), stream(rng, 305)
    for s in (s1, s2):
        for key in ("q", "k", "v"):
            s[key][:300] = base[key][:300]
    streams = {0: s1, 1: s2}
    total, computed = {0: 300, 1: 300}, {0: 0, 1: 0}
    run.step([0], streams, total, computed)
    run.pager.share(0, 1, 300)
    computed[1] = 300
    n_copies = 0
    for _ in range(5):
        total[0] += 1
        total[1] += 1
        st = run.step([0, 1], streams, total, computed)
        n_copies += st["copy_src"].size
    assert n_copies == 1
    p0, p1 = run.pager.request_pages(0), run.pager.request_pages(1)
    assert (p0[:18] == p1[:18]).all() and p0[18] != p1[18]
    run.check_pools()
