"""Shared pages: the prefix index, forks and copy-on-write of the host page
pool (``pcp_pager_*``, ``pcp_schedule_step``; no GPU) against the
brute-force model ``oracle.chunk_plan.PagePool``, and the model against the
pages' numbers.

Pins of the model:
* vLLM PR #54076 (golden fixture prefix_hit.json): re-asking a P-token prompt
  reuses floor((P - 1) / B) * B tokens -- 16,480 of a 16,764-token prompt
  with 1648-token blocks, and the law at exact multiples of 1568;
* a fork worked out by hand: the first continuation to write into the
  shared, partly filled page copies it, the second then owns the original.
"""
import json
import os

import numpy as np
import pytest

import paged_chunked_prefill_gb300 as pcp
from oracle import chunk_plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def serve_whole(pool_plan, rid, P):
    """Compute a P-token prompt in one step (budget P)."""
    st = pool_plan([rid], [P], [0], P, 0)
    assert st["qo_indptr"][-1] == P


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "prefix_hit.json")))["cases"])
def test_hit_law_golden(case):
    B, P = case["block"], case["prompt_len"]
    tokens = np.random.default_rng(P).integers(0, 50000, size=P).astype(np.int32)
    pages = -(-P // B) + 2
    model = chunk_plan.PagePool(pages, B)
    serve_whole(model.plan_step, 1, P)
    model.cache_prompt(1, tokens.tolist())
    assert model.match_prefix(2, tokens.tolist()) == case["reused"]
    lib = pcp.Pager(pages, B)
    serve_whole(lambda *a: {k: v.tolist() for k, v in lib.schedule_step(*a).items()}, 1, P)
    lib.cache_prompt(1, tokens)
    assert lib.match_prefix(2, tokens) == case["reused"]
    # the reused pages are the first request's
    assert (lib.request_pages(2) == lib.request_pages(1)[:case["reused"] // B]).all()


def test_fork_copy_on_write_by_hand():
    """Page size 16: request 1 computes 37 tokens (pages 0, 1, 2; page 2
    holds 5 slots).  Request 2 shares them.  A step where both decode one
    token: request 1 starts inside the shared page 2, copies its 5 slots to
    the lowest free page (3) and writes there; request 2 is then the only
    holder of page 2 and writes into it without a copy."""
    for pool, plan in ((chunk_plan.PagePool(8, 16), None), (pcp.Pager(8, 16), None)):
        lib = isinstance(pool, pcp.Pager)
        step = (lambda *a: {k: v.tolist() for k, v in pool.schedule_step(*a).items()}) \
            if lib else pool.plan_step
        step([1], [37], [0], 64, 0)
        pool.share(1, 2, 37)
        st = step([1, 2], [38, 38], [37, 37], 64, 0)
        assert st["copy_src"] == [2] and st["copy_dst"] == [3] and st["copy_slots"] == [5]
        assert st["kv_indices"] == [0, 1, 3, 0, 1, 2]
        assert st["kv_indptr"] == [0, 3, 6] and st["qo_indptr"] == [0, 1, 2]
        pages1 = pool.request_pages(1) if lib else pool.pages[1]
        assert list(pages1) == [0, 1, 3]


def test_copy_needs_a_free_page():
    """A chunk starting inside a shared page waits when no page is free for
    the copy; the budget goes to the next request."""
    for lib in (False, True):
        pool = pcp.Pager(3, 16) if lib else chunk_plan.PagePool(3, 16)
        step = (lambda *a: {k: v.tolist() for k, v in pool.schedule_step(*a).items()}) \
            if lib else pool.plan_step
        step([1], [40], [0], 64, 0)          # pages 0, 1, 2 (page 2 half full)
        pool.share(1, 2, 40)
        st = step([1, 2], [41, 41], [40, 40], 64, 0)
        assert st["row_req"] == [] and st["copy_src"] == []


def random_tokens(rng, parents, n):
    """A prompt that continues a random earlier prompt's prefix (or starts
    fresh), so prompts share prefixes of random lengths."""
    if parents and rng.random() < 0.7:
        base = parents[int(rng.integers(0, len(parents)))]
        cut = int(rng.integers(0, len(base) + 1))
        return base[:cut] + rng.integers(0, 5, size=max(n - cut, 1)).tolist()
    return rng.integers(0, 5, size=n).tolist()


def run_loop(make_pool, wrap, seed, steps=50):
    """A serving loop with prefix reuse, forks and a cache clear; returns a
    trace of every observable (plans, hits, free counts)."""
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([2, 4, 16]))
    pool = make_pool(int(rng.integers(20, 120)), ps)
    plan = wrap(pool)
    prompts, reqs, trace = [], {}, []
    nid = 0
    for step in range(steps):
        if rng.random() < 0.5:
            toks = random_tokens(rng, prompts, int(rng.integers(1, 70)))
            hit = pool.match_prefix(nid, toks)
            trace.append(("hit", nid, hit))
            reqs[nid] = {"tokens": toks, "computed": hit, "total": len(toks),
                         "decodes": int(rng.integers(0, 3))}
            nid += 1
        if reqs and rng.random() < 0.2:
            src = list(reqs)[int(rng.integers(0, len(reqs)))]
            r = reqs[src]
            if r["computed"] > 0:
                pool.share(src, nid, r["computed"])
                reqs[nid] = {"tokens": list(r["tokens"][:r["computed"]]),
                             "computed": r["computed"], "total": r["computed"] + 1,
                             "decodes": 1}
                trace.append(("fork", src, nid))
                nid += 1
        if step == steps // 2:
            pool.clear_cache()
        if not reqs:
            continue
        ids = list(reqs)
        st = plan(ids, [reqs[i]["total"] for i in ids], [reqs[i]["computed"] for i in ids],
                  int(rng.choice([3, 40, 300])), int(rng.choice([0, 0, 8])))
        trace.append(("plan", st))
        qo = st["qo_indptr"]
        for n, ri in enumerate(st["row_req"]):
            r = reqs[ids[ri]]
            r["computed"] += qo[n + 1] - qo[n]
            if st["sample"][n]:
                if r["computed"] == len(r["tokens"]):
                    pool.cache_prompt(ids[ri], r["tokens"])
                if r["decodes"] > 0:
                    r["decodes"] -= 1
                    r["total"] += 1
                    r["tokens"].append(int(rng.integers(0, 5)))
                else:
                    pool.release(ids[ri])
                    del reqs[ids[ri]]
        trace.append(("free", pool.num_free() if hasattr(pool, "num_free") else len(pool.free)))
    return trace


def lib_wrap(pool):
    return lambda *a: {k: v.tolist() for k, v in pool.schedule_step(*a).items()}


@pytest.mark.parametrize("seed", range(16))
def test_library_matches_model_with_sharing(seed):
    a = run_loop(pcp.Pager, lib_wrap, seed)
    b = run_loop(chunk_plan.PagePool, lambda p: p.plan_step, seed)
    assert a == b
    kinds = {t[0] for t in a}
    assert "plan" in kinds


def test_model_reference_counts_stay_consistent():
    """Every page's count equals its holders (requests plus the index); free
    pages are exactly those with no holder."""
    for seed in range(5):
        rng = np.random.default_rng(seed)
        pool = chunk_plan.PagePool(60, 4)
        run_loop(lambda n, ps: pool, lambda p: p.plan_step, seed, steps=30)
        holders = [0] * len(pool.refs)
        for pages in pool.pages.values():
            for p in pages:
                holders[p] += 1
        for p in pool.index.values():
            holders[p] += 1
        assert holders == pool.refs
        assert sorted(pool.free) == [p for p, h in enumerate(holders) if h == 0]
