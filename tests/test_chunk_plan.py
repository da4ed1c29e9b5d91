"""The host chunk planner and page pool (``pcp_schedule_step``, through the
C ABI; no GPU) against the brute-force model in ``oracle.chunk_plan``, and that
model against the pages' worked examples.

Pins of the model:
* vLLM PR #54076 (follow-up comment): a 5-block prompt walked with the full
  remaining budget ends its chunks at every state-block boundary,
  [1648, 3296, 4944, 6592, 8240] (golden fixture boundary_stop.json);
* AReno PR #642: the 4097-token prompt under a 2048 / 512 / 128 token budget
  is prefilled in 3 / 9 / 33 chunks, the last one token long, and samples
  only after the last chunk;
* a small step worked out by hand (decode row first, a prefill chunk cut by
  the budget, page ids handed out lowest first in request order).
"""
import json
import os

import numpy as np
import pytest

import paged_chunked_prefill_gb300 as pcp
from oracle import chunk_plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def serve_prompt(plan, prompt_len, budget, state_block, page_size=16, num_pages=1024):
    """Chunk ends of one prompt served alone, step after step."""
    free, pages = list(range(num_pages)), {}
    computed, ends = 0, []
    while computed < prompt_len:
        st = plan(free, pages, [0], [prompt_len], [computed], budget(prompt_len - computed),
                  state_block, page_size)
        c = st["qo_indptr"][1] - st["qo_indptr"][0]
        computed += c
        ends.append(computed)
        assert st["sample"][0] == (computed == prompt_len)
    return ends


def test_boundary_stop_golden():
    g = json.load(open(os.path.join(GOLDEN, "boundary_stop.json")))
    ends = serve_prompt(chunk_plan.plan_step, g["prompt_len"], lambda rem: rem,
                        g["state_block"], page_size=16, num_pages=1024)
    assert ends == g["chunk_ends"]


@pytest.mark.parametrize("budget,n_chunks", [(2048, 3), (512, 9), (128, 33)])
def test_budget_chunking_of_a_4097_token_prompt(budget, n_chunks):
    ends = serve_prompt(chunk_plan.plan_step, 4097, lambda rem: budget, 0)
    assert len(ends) == n_chunks
    assert ends[-1] == 4097 and ends[-1] - ends[-2] == 1
    assert all(b - a == budget for a, b in zip([0] + ends[:-2], ends[:-1]))


def hand_step_state():
    # page size 4; request 5 (decode: 9 tokens known, 8 computed) holds pages
    # [5, 6]; request 8 is a fresh 13-token prompt; request 9 has 2 of 6
    # prompt tokens computed and holds page [4]
    free = [0, 1, 2, 3, 7, 8, 9]
    pages = {5: [5, 6], 9: [4]}
    return free, pages


def test_hand_worked_step():
    """Budget 8: the decode row takes 1 token (position 8 needs a new page:
    the lowest free one, 0); the fresh prompt takes the remaining 7
    (positions 0..6, two new pages 1 and 2); request 9 gets nothing."""
    free, pages = hand_step_state()
    st = chunk_plan.plan_step(free, pages, [5, 8, 9], [9, 13, 6], [8, 0, 2], 8, 0, 4)
    assert st == {"row_req": [0, 1], "qo_indptr": [0, 1, 8], "prefix_lens": [8, 0],
                  "kv_indptr": [0, 3, 5], "kv_indices": [5, 6, 0, 1, 2],
                  "sample": [True, False]}
    assert free == [3, 7, 8, 9]


def library_plan(pager):
    def plan(free, pages, ids, tot, comp, budget, sb, ps):
        st = pager.schedule_step(ids, tot, comp, budget, sb)
        return {k: v.tolist() for k, v in st.items()}
    return plan


def test_library_hand_worked_step():
    """The library on the hand-worked step: the same pool state, the same
    plan as the model (and the model's plan is the one worked out above)."""
    pg = pcp.Pager(10, 4)
    # requests 5 and 9 take pages in id order: 5 gets [0, 1], 9 gets [2]
    pg.schedule_step([5, 9], [8, 2], [0, 0], 16)
    free_before = pg.num_free()
    st = pg.schedule_step([5, 8, 9], [9, 13, 6], [8, 0, 2], 8)
    for k in ("copy_src", "copy_dst", "copy_slots"):
        assert st.pop(k).size == 0
    model_free = list(range(3, 10))
    model_pages = {5: [0, 1], 9: [2]}
    want = chunk_plan.plan_step(model_free, model_pages, [5, 8, 9], [9, 13, 6], [8, 0, 2], 8, 0,
                                4)
    assert {k: v.tolist() for k, v in st.items()} == want
    assert want["kv_indices"] == [0, 1, 3, 4, 5] and want["qo_indptr"] == [0, 1, 8]
    assert pg.num_free() == free_before - 3 == len(model_free)
    # a zero budget plans nothing and takes no page
    assert pg.schedule_step([8], [13], [7], 0)["row_req"].size == 0
    assert pg.num_free() == len(model_free)


def simulate(plan_fn, pager_factory, seed, steps=60):
    """Random serving loop: new prompts arrive, chunks run, finished requests
    generate a few tokens and then release their pages.  Returns the list of
    step plans and the pool's free counts."""
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([1, 4, 16]))
    num_pages = int(rng.integers(8, 200))
    budget_choices = [1, 7, 64, 512]
    sb = int(rng.choice([0, 0, 5, 64]))
    state = pager_factory(num_pages, ps)
    reqs = []      # [id, total, computed, decode_left]
    next_id = 0
    log = []
    for _ in range(steps):
        for _ in range(int(rng.integers(0, 3))):
            reqs.append([next_id, int(rng.integers(1, 300)), 0, int(rng.integers(0, 4))])
            next_id += 1
        if not reqs:
            continue
        budget = int(rng.choice(budget_choices))
        ids = [r[0] for r in reqs]
        tot = [r[1] for r in reqs]
        comp = [r[2] for r in reqs]
        st = plan_fn(state, ids, tot, comp, budget, sb)
        log.append(st)
        qo = st["qo_indptr"]
        for n, ri in enumerate(st["row_req"]):
            reqs[ri][2] += qo[n + 1] - qo[n]
            if st["sample"][n]:
                if reqs[ri][3] > 0:      # generate one more token
                    reqs[ri][1] += 1
                    reqs[ri][3] -= 1
        done = [r for r in reqs if r[2] == r[1] and r[3] == 0]
        for r in done:
            state["release"](r[0])
        reqs = [r for r in reqs if not (r[2] == r[1] and r[3] == 0)]
    return log


def lib_factory(num_pages, ps):
    pg = pcp.Pager(num_pages, ps)
    return {"pg": pg, "release": pg.release}


def model_factory(num_pages, ps):
    pool = chunk_plan.PagePool(num_pages, ps)
    return {"pool": pool, "release": pool.release}


def lib_plan(state, ids, tot, comp, budget, sb):
    st = state["pg"].schedule_step(ids, tot, comp, budget, sb)
    return {k: v.tolist() for k, v in st.items()}


def model_plan(state, ids, tot, comp, budget, sb):
    return state["pool"].plan_step(ids, tot, comp, budget, sb)


@pytest.mark.parametrize("seed", range(12))
def test_library_matches_model_over_a_serving_loop(seed):
    a = simulate(lib_plan, lib_factory, seed)
    b = simulate(model_plan, model_factory, seed)
    assert a == b
    assert sum(len(s["row_req"]) for s in a) > 0


@pytest.mark.parametrize("seed", range(4))
def test_step_invariants(seed):
    """Every step stays within its budget; no page is held twice; pages held
    plus free pages make up the pool; a chunk's tokens land in consecutive
    slots of its request's pages."""
    rng = np.random.default_rng(100 + seed)
    pg = pcp.Pager(64, 8)
    ids, tot, comp = [0, 1, 2, 3], [300, 41, 9, 120], [0, 0, 0, 0]
    for _ in range(30):
        budget = int(rng.integers(1, 100))
        st = pg.schedule_step(ids, tot, comp, budget, 0)
        assert st["qo_indptr"][-1] <= budget
        held = [pg.request_pages(i) for i in ids]
        allp = np.concatenate(held)
        assert len(set(allp.tolist())) == allp.size
        assert allp.size + pg.num_free() == 64
        for n, r in enumerate(st["row_req"]):
            pages = st["kv_indices"][st["kv_indptr"][n]:st["kv_indptr"][n + 1]]
            assert (pages == held[r]).all()
            c = st["qo_indptr"][n + 1] - st["qo_indptr"][n]
            comp[r] += int(c)
        if all(c == t for c, t in zip(comp, tot)):
            break


def test_errors():
    pg = pcp.Pager(4, 16)
    with pytest.raises(pcp.PCPError) as e:
        pg.schedule_step([1, 1], [10, 10], [0, 0], 8)           # repeated id
    assert e.value.status == pcp.Status.INVALID_ARG
    with pytest.raises(pcp.PCPError):
        pg.schedule_step([1], [10], [11], 8)                     # computed > total
    with pytest.raises(pcp.PCPError):
        pg.schedule_step([1], [40], [20], 8)                     # holds no pages for 20 tokens
    with pytest.raises(ValueError):
        pcp.Pager(-1, 16)
    L = pcp.lib()
    import ctypes
    P = ctypes.c_void_p
    n = ctypes.c_int32(0)
    ids = np.array([3], np.int64)
    tot = np.array([64], np.int32)
    comp = np.array([0], np.int32)
    z = np.zeros(4, np.int32)
    smp = np.zeros(4, np.uint8)
    ptr = lambda a: a.ctypes.data_as(P)
    nc = ctypes.c_int32(0)
    st = L.pcp_schedule_step(pg._h, 1, ptr(ids), ptr(tot), ptr(comp), 64, 0, ctypes.byref(n),
                             ptr(z), ptr(z), ptr(z), ptr(z), ptr(z), 1, ptr(smp),
                             ctypes.byref(nc), ptr(z), ptr(z), ptr(z))
    assert st == pcp.Status.WORKSPACE and pg.num_free() == 4   # nothing taken
