"""Brute-force model of the page pool and of one serving step's chunk plan.

TEST INFRASTRUCTURE.  Only ``tests/`` may import this module; the library
never does, and it shares no code with the library's planner.

It follows the step the pages describe, one token at a time:

* a step runs at most ``budget`` tokens; prompts longer than that are
  prefilled over several steps, decode rows run alongside, and a request
  samples only when its final chunk has run (AReno PR #642, "What does this PR
  do?" and "How was it tested?");
* with a recurrent-state grid of S tokens, a chunk ends at the first grid
  point past its start, also when it starts on the grid (vLLM PR #54076,
  "Fix", and the follow-up comment that makes the boundary stop
  unconditional);
* a request's tokens fill its pages in order, so a chunk continues inside the
  last, partly filled page (AReno PR #642, third bullet);
* a re-asked prompt reuses the cached pages of its prefix, whole pages only
  and never its last token, so a P-token prompt reuses at most
  floor((P - 1) / page_size) * page_size tokens (vLLM PR #54076, "E2E" and
  the hit law in the follow-up comments); a page several requests hold is
  read-only, so a write into a shared, partly filled page first copies it.

The order of service is the one the library documents: requests with one
pending token first, then prefill chunks, both in request order; the chunk
lengths are fixed first (each token needs room in a held or free page, and a
chunk starting inside a shared page needs one more free page for its copy),
then each scheduled request, in request order, copies its shared page if
it still shares it and takes the lowest-numbered free pages it needs.

The prefix index here is a trie of page-sized token blocks (exact keys), not a
hash.
"""
from __future__ import annotations

import bisect
from typing import Dict, List, Sequence, Tuple


class PagePool:
    def __init__(self, num_pages: int, page_size: int):
        self.ps = page_size
        self.free: List[int] = list(range(num_pages))
        self.refs: List[int] = [0] * num_pages
        self.pages: Dict[int, List[int]] = {}
        # a trie of page-sized token blocks: (parent node, block tokens) -> node
        self.nodes: Dict[Tuple[int, Tuple[int, ...]], int] = {}
        self.index: Dict[int, int] = {}          # trie node -> cached page
        self.node_of_page: Dict[int, int] = {}

    # ------------------------------------------------------------ pages
    def take(self) -> int:
        pg = self.free.pop(0)
        self.refs[pg] = 1
        return pg

    def drop(self, pg: int) -> None:
        self.refs[pg] -= 1
        if self.refs[pg] == 0:
            bisect.insort(self.free, pg)

    def release(self, req: int) -> None:
        for pg in self.pages.pop(req, []):
            self.drop(pg)

    def share(self, src: int, dst: int, n_tokens: int) -> None:
        need = -(-n_tokens // self.ps)
        assert dst != src and not self.pages.get(dst) and need <= len(self.pages.get(src, []))
        if need:
            self.pages[dst] = list(self.pages[src][:need])
            for pg in self.pages[dst]:
                self.refs[pg] += 1

    # ----------------------------------------------------- prefix index
    def node(self, parent: int, tokens: Sequence[int], i: int) -> int:
        key = (parent, tuple(tokens[i * self.ps:(i + 1) * self.ps]))
        return self.nodes.setdefault(key, len(self.nodes) + 1)

    def cache_prompt(self, req: int, tokens: Sequence[int]) -> int:
        held = self.pages.get(req, [])
        added = 0
        parent = 0
        for i in range(min(len(tokens) // self.ps, len(held))):
            nd = self.node(parent, tokens, i)
            parent = nd
            if nd in self.index:
                continue
            pg = held[i]
            if pg in self.node_of_page:
                break
            self.index[nd] = pg
            self.node_of_page[pg] = nd
            self.refs[pg] += 1
            added += 1
        return added

    def match_prefix(self, req: int, tokens: Sequence[int]) -> int:
        assert not self.pages.get(req)
        hit = []
        parent = 0
        for i in range((len(tokens) - 1) // self.ps if len(tokens) else 0):
            nd = self.node(parent, tokens, i)
            if nd not in self.index:
                break
            hit.append(self.index[nd])
            parent = nd
        if hit:
            self.pages[req] = hit
            for pg in hit:
                self.refs[pg] += 1
        return len(hit) * self.ps

    def clear_cache(self) -> None:
        for pg in self.index.values():
            self.drop(pg)
        self.index = {}
        self.node_of_page = {}

    # -------------------------------------------------------------- step
    def plan_step(self, req_ids: Sequence[int], total_lens: Sequence[int],
                  num_computed: Sequence[int], budget: int, state_block: int) -> dict:
        ps = self.ps
        n = len(req_ids)
        chunk = [0] * n
        left = budget
        free_count = len(self.free)
        held = [len(self.pages.get(r, [])) for r in req_ids]
        extra = [0] * n

        def shared_start(r: int) -> bool:
            start = num_computed[r]
            pages = self.pages.get(req_ids[r], [])
            return start % ps != 0 and start // ps < len(pages) and \
                self.refs[pages[start // ps]] > 1

        def place_tokens(r: int, limit: int) -> None:
            nonlocal left, free_count
            reserve = 1 if shared_start(r) else 0
            if free_count < reserve:
                return
            placed = 0
            while placed < limit and left > 0:
                pos = num_computed[r] + placed
                if pos // ps >= held[r] + extra[r]:
                    if free_count - reserve == 0:
                        break
                    free_count -= 1
                    extra[r] += 1
                placed += 1
                left -= 1
                if state_block > 0 and (pos + 1) % state_block == 0:
                    break
            if placed:
                free_count -= reserve
            chunk[r] = placed

        for r in range(n):
            if total_lens[r] - num_computed[r] == 1 and left > 0:
                place_tokens(r, 1)
        for r in range(n):
            if total_lens[r] - num_computed[r] > 1 and left > 0:
                place_tokens(r, total_lens[r] - num_computed[r])

        out = {"row_req": [], "qo_indptr": [0], "prefix_lens": [], "kv_indptr": [0],
               "kv_indices": [], "sample": [], "copy_src": [], "copy_dst": [],
               "copy_slots": []}
        for r in range(n):
            if chunk[r] == 0:
                continue
            if shared_start(r):
                pages = self.pages[req_ids[r]]
                i = num_computed[r] // ps
                new = self.take()
                out["copy_src"].append(pages[i])
                out["copy_dst"].append(new)
                out["copy_slots"].append(num_computed[r] % ps)
                self.drop(pages[i])
                pages[i] = new
            pages = self.pages.setdefault(req_ids[r], [])
            end = num_computed[r] + chunk[r]
            while len(pages) * ps < end:
                pages.append(self.take())
            out["row_req"].append(r)
            out["prefix_lens"].append(num_computed[r])
            out["qo_indptr"].append(out["qo_indptr"][-1] + chunk[r])
            out["kv_indices"].extend(pages)
            out["kv_indptr"].append(len(out["kv_indices"]))
            out["sample"].append(end == total_lens[r])
        return out


def plan_step(free_pages: List[int], req_pages: Dict[int, List[int]], req_ids: Sequence[int],
              total_lens: Sequence[int], num_computed: Sequence[int], budget: int,
              state_block: int, page_size: int) -> dict:
    """One step on an explicit pool state where every page has one holder
    (no sharing): ``free_pages`` and ``req_pages`` are updated in place."""
    pool = PagePool(0, page_size)
    n_pages = max([0] + free_pages + [p for v in req_pages.values() for p in v]) + 1
    pool.refs = [0] * n_pages
    pool.free = sorted(free_pages)
    pool.pages = {k: list(v) for k, v in req_pages.items()}
    for v in pool.pages.values():
        for p in v:
            pool.refs[p] = 1
    out = pool.plan_step(req_ids, total_lens, num_computed, budget, state_block)
    free_pages[:] = pool.free
    req_pages.clear()
    req_pages.update(pool.pages)
    for k in ("copy_src", "copy_dst", "copy_slots"):
        assert not out.pop(k)
    return out
