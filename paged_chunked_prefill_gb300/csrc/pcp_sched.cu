// Host-side chunk planner and page pool (no device code).
//
// The step upstream of the attention path: which tokens of which requests a
// serving step runs, and where their K/V goes.
//
//  * Token budget.  A step runs at most `budget` tokens (AReno PR #642: the
//    scheduler token budget is kept; a prompt longer than it is prefilled in
//    chunks, decode rows run alongside, and a request samples only when its
//    final chunk has run).  Requests whose pending work is one token
//    (decode-shaped) are served first, in the given order; prefill chunks
//    then fill what is left of the budget, in order.
//  * State-block boundary stop (vLLM PR #54076, "Fix" and the follow-up
//    comment): with a state grid of S tokens, a chunk that starts at `start`
//    ends no later than the next multiple of S strictly above `start` -- also
//    from an aligned start -- so a recurrent state can be written at every
//    grid point a prompt crosses.
//  * Pages.  A request owns a list of pages; its tokens fill them in order,
//    so a chunk continues inside the last, partly filled page (AReno PR #642,
//    third bullet) and new pages come from the pool's free list, lowest id
//    first.  A chunk is shortened to the tokens the free pages can hold.
#include <algorithm>
#include <cstdint>
#include <map>
#include <new>
#include <set>
#include <vector>

#include "pcp.h"

struct pcp_pager {
    int64_t num_pages;
    int page_size;
    std::set<int32_t> free_pages;                          // lowest id first
    std::map<int64_t, std::vector<int32_t>> req_pages;     // request id -> its pages
    int64_t held_entries = 0;                              // sum of the page lists' lengths
};

namespace {

int64_t pages_for(int64_t tokens, int page_size) { return (tokens + page_size - 1) / page_size; }

}  // namespace

extern "C" {

pcp_pager* pcp_pager_create(int64_t num_pages, int page_size) {
    if (num_pages < 0 || num_pages > INT32_MAX || page_size < 1) return nullptr;
    pcp_pager* p = new (std::nothrow) pcp_pager();
    if (p == nullptr) return nullptr;
    p->num_pages = num_pages;
    p->page_size = page_size;
    for (int64_t i = 0; i < num_pages; ++i) p->free_pages.insert((int32_t)i);
    return p;
}

void pcp_pager_destroy(pcp_pager* p) { delete p; }

int64_t pcp_pager_num_free(const pcp_pager* p) {
    return p == nullptr ? -1 : (int64_t)p->free_pages.size();
}

int64_t pcp_pager_num_held(const pcp_pager* p) { return p == nullptr ? -1 : p->held_entries; }

int64_t pcp_pager_request_pages(const pcp_pager* p, int64_t req_id, int32_t* pages,
                                int64_t capacity) {
    if (p == nullptr) return -1;
    auto it = p->req_pages.find(req_id);
    if (it == p->req_pages.end()) return 0;
    const int64_t n = (int64_t)it->second.size();
    if (pages != nullptr)
        for (int64_t i = 0; i < std::min(n, capacity); ++i) pages[i] = it->second[i];
    return n;
}

pcp_status pcp_pager_release(pcp_pager* p, int64_t req_id) {
    if (p == nullptr) return PCP_ERR_INVALID_ARG;
    auto it = p->req_pages.find(req_id);
    if (it == p->req_pages.end()) return PCP_OK;
    for (int32_t pg : it->second) p->free_pages.insert(pg);
    p->held_entries -= (int64_t)it->second.size();
    p->req_pages.erase(it);
    return PCP_OK;
}

pcp_status pcp_schedule_step(pcp_pager* p, int n_reqs, const int64_t* req_ids,
                             const int32_t* total_lens, const int32_t* num_computed, int budget,
                             int state_block, int32_t* n_rows, int32_t* row_req,
                             int32_t* qo_indptr, int32_t* prefix_lens, int32_t* kv_indptr,
                             int32_t* kv_indices, int64_t kv_indices_cap, uint8_t* sample) {
    if (p == nullptr || n_reqs < 0 || budget < 0 || state_block < 0 || n_rows == nullptr ||
        kv_indices_cap < 0)
        return PCP_ERR_INVALID_ARG;
    if (n_reqs > 0 && (req_ids == nullptr || total_lens == nullptr || num_computed == nullptr ||
                       row_req == nullptr || qo_indptr == nullptr || prefix_lens == nullptr ||
                       kv_indptr == nullptr || sample == nullptr))
        return PCP_ERR_INVALID_ARG;
    {
        std::set<int64_t> seen;
        for (int r = 0; r < n_reqs; ++r) {
            if (total_lens[r] < 0 || num_computed[r] < 0 || num_computed[r] > total_lens[r] ||
                !seen.insert(req_ids[r]).second)
                return PCP_ERR_INVALID_ARG;
            // the pages a request holds must cover its computed tokens
            auto it = p->req_pages.find(req_ids[r]);
            const int64_t held = it == p->req_pages.end() ? 0 : (int64_t)it->second.size();
            if (held < pages_for(num_computed[r], p->page_size)) return PCP_ERR_INVALID_ARG;
        }
    }
    // ---- choose the chunk of every request
    std::vector<int32_t> chunk(n_reqs, 0);
    int64_t left = budget;
    int64_t free_pages = (int64_t)p->free_pages.size();
    auto grant = [&](int r, int64_t want) {
        const int64_t start = num_computed[r];
        auto it = p->req_pages.find(req_ids[r]);
        const int64_t held = it == p->req_pages.end() ? 0 : (int64_t)it->second.size();
        // tokens that fit in the held pages plus the free ones
        const int64_t room = (held + free_pages) * p->page_size - start;
        const int64_t n = std::max<int64_t>(0, std::min(want, room));
        free_pages -= std::max<int64_t>(0, pages_for(start + n, p->page_size) - held);
        left -= n;
        chunk[r] = (int32_t)n;
    };
    // decode-shaped work first: one pending token
    for (int r = 0; r < n_reqs && left > 0; ++r)
        if (total_lens[r] - num_computed[r] == 1) grant(r, 1);
    // then prefill chunks, stopping at the next state-grid point
    for (int r = 0; r < n_reqs && left > 0; ++r) {
        const int64_t pending = (int64_t)total_lens[r] - num_computed[r];
        if (pending <= 1) continue;
        int64_t want = std::min<int64_t>(pending, left);
        if (state_block > 0) {
            const int64_t start = num_computed[r];
            const int64_t next = (start / state_block + 1) * state_block;
            want = std::min<int64_t>(want, next - start);
        }
        grant(r, want);
    }
    // ---- rows, pages and the step's metadata (rows in request order)
    int rows = 0;
    int64_t entries = 0;
    for (int r = 0; r < n_reqs; ++r) {
        if (chunk[r] == 0) continue;
        const int64_t end = (int64_t)num_computed[r] + chunk[r];
        auto it = p->req_pages.find(req_ids[r]);
        const int64_t held = it == p->req_pages.end() ? 0 : (int64_t)it->second.size();
        entries += std::max<int64_t>(held, pages_for(end, p->page_size));  // the row's page list
        ++rows;
    }
    if (kv_indices_cap < entries || (entries > 0 && kv_indices == nullptr))
        return PCP_ERR_WORKSPACE;
    rows = 0;
    entries = 0;
    qo_indptr[0] = 0;
    kv_indptr[0] = 0;
    for (int r = 0; r < n_reqs; ++r) {
        if (chunk[r] == 0) continue;
        std::vector<int32_t>& pages = p->req_pages[req_ids[r]];
        const int64_t end = (int64_t)num_computed[r] + chunk[r];
        while ((int64_t)pages.size() < pages_for(end, p->page_size)) {
            auto f = p->free_pages.begin();
            pages.push_back(*f);
            p->free_pages.erase(f);
            ++p->held_entries;
        }
        row_req[rows] = r;
        prefix_lens[rows] = num_computed[r];
        qo_indptr[rows + 1] = qo_indptr[rows] + chunk[r];
        for (int32_t pg : pages) kv_indices[entries++] = pg;
        kv_indptr[rows + 1] = (int32_t)entries;
        sample[rows] = end == total_lens[r] ? 1 : 0;
        ++rows;
    }
    *n_rows = rows;
    return PCP_OK;
}

}  // extern "C"
