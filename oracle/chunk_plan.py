"""Brute-force model of one serving step's chunk plan and page allocation.

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
  last, partly filled page (AReno PR #642, third bullet).

The step's order of service is the one the library documents: requests with
one pending token first, then prefill chunks, both in request order; the
chunk lengths are fixed first (each token needs room in a held or free
page), then each scheduled request, in request order, takes the
lowest-numbered free pages it needs.
"""
from __future__ import annotations

from typing import Dict, List, Sequence


def plan_step(free_pages: List[int], req_pages: Dict[int, List[int]], req_ids: Sequence[int],
              total_lens: Sequence[int], num_computed: Sequence[int], budget: int,
              state_block: int, page_size: int) -> dict:
    """One step.  Mutates ``free_pages`` (kept sorted) and ``req_pages``.

    Returns row_req, qo_indptr, prefix_lens, kv_indptr, kv_indices, sample
    as Python lists."""
    n = len(req_ids)
    chunk = [0] * n
    left = budget
    free_count = len(free_pages)
    held = [len(req_pages.get(r, [])) for r in req_ids]
    extra = [0] * n                      # pages a chunk takes from the free list

    def place_tokens(r: int, limit: int) -> None:
        nonlocal left, free_count
        placed = 0
        while placed < limit and left > 0:
            pos = num_computed[r] + placed
            page_index = pos // page_size
            if page_index >= held[r] + extra[r]:
                if free_count == 0:
                    break
                free_count -= 1
                extra[r] += 1
            placed += 1
            left -= 1
            if state_block > 0 and (pos + 1) % state_block == 0:
                break                    # the chunk ends on a grid point
        chunk[r] = placed

    for r in range(n):
        if total_lens[r] - num_computed[r] == 1 and left > 0:
            place_tokens(r, 1)
    for r in range(n):
        pending = total_lens[r] - num_computed[r]
        if pending > 1 and left > 0:
            place_tokens(r, pending)

    out = {"row_req": [], "qo_indptr": [0], "prefix_lens": [], "kv_indptr": [0],
           "kv_indices": [], "sample": []}
    for r in range(n):
        if chunk[r] == 0:
            continue
        pages = req_pages.setdefault(req_ids[r], [])
        end = num_computed[r] + chunk[r]
        while len(pages) * page_size < end:
            pages.append(free_pages.pop(0))
        out["row_req"].append(r)
        out["prefix_lens"].append(num_computed[r])
        out["qo_indptr"].append(out["qo_indptr"][-1] + chunk[r])
        out["kv_indices"].extend(pages)
        out["kv_indptr"].append(len(out["kv_indices"]))
        out["sample"].append(end == total_lens[r])
    return out
