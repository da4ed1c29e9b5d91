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
//  * Shared pages (vLLM PR #54076, "E2E": an immediate re-ask of a prompt
//    reuses its cached blocks; the hit is quantised to whole blocks,
//    floor((P - 1) / B) * B tokens of a P-token prompt).  Pages carry
//    reference counts.  The prefix index maps each full page of a cached
//    prompt, keyed by the prompt's tokens up to that page's end, to the page;
//    a new request takes the longest matching run of full pages read-only.
//    A request can also share another's pages (a fork); the first write into
//    a shared, partly filled page copies it to a fresh page first
//    (copy-on-write), and the step reports that copy for the device.
#include <algorithm>
#include <cstdint>
#include <map>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pcp.h"

namespace {

// Prefix-index entry: one full page of a cached prompt.  The key chains the
// previous page's key with this page's tokens; the tokens and the parent key
// are kept to check a match exactly (no trust in the hash alone).
struct CacheEntry {
    int32_t page;
    uint64_t parent;
    std::vector<int32_t> tokens;
};

uint64_t mix64(uint64_t x) {  // the SplitMix64 finaliser
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

uint64_t block_key(uint64_t parent, const int32_t* tokens, int n) {
    uint64_t h = mix64(parent ^ 0x5851f42d4c957f2dull);
    for (int i = 0; i < n; ++i) h = mix64(h ^ (uint32_t)tokens[i]);
    return h == 0 ? 1 : h;  // 0 is the empty prefix
}

int64_t pages_for(int64_t tokens, int page_size) { return (tokens + page_size - 1) / page_size; }

}  // namespace

struct pcp_pager {
    int64_t num_pages;
    int page_size;
    std::set<int32_t> free_pages;                          // lowest id first
    std::vector<int32_t> refs;                             // holders of each page
    std::map<int64_t, std::vector<int32_t>> req_pages;     // request id -> its pages
    int64_t held_entries = 0;                              // sum of the page lists' lengths
    std::unordered_map<uint64_t, CacheEntry> index;        // prefix index
    std::vector<uint64_t> cached_key;                      // page -> its index key (0: none)

    int32_t take_page() {
        auto f = free_pages.begin();
        const int32_t pg = *f;
        free_pages.erase(f);
        refs[pg] = 1;
        return pg;
    }
    void drop_page(int32_t pg) {
        if (--refs[pg] == 0) free_pages.insert(pg);
    }
};

extern "C" {

pcp_pager* pcp_pager_create(int64_t num_pages, int page_size) {
    if (num_pages < 0 || num_pages > INT32_MAX || page_size < 1) return nullptr;
    pcp_pager* p = new (std::nothrow) pcp_pager();
    if (p == nullptr) return nullptr;
    p->num_pages = num_pages;
    p->page_size = page_size;
    p->refs.assign((size_t)num_pages, 0);
    p->cached_key.assign((size_t)num_pages, 0);
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
    for (int32_t pg : it->second) p->drop_page(pg);
    p->held_entries -= (int64_t)it->second.size();
    p->req_pages.erase(it);
    return PCP_OK;
}

pcp_status pcp_pager_share(pcp_pager* p, int64_t src_req, int64_t dst_req, int64_t n_tokens) {
    if (p == nullptr || n_tokens < 0 || src_req == dst_req) return PCP_ERR_INVALID_ARG;
    auto src = p->req_pages.find(src_req);
    const int64_t need = pages_for(n_tokens, p->page_size);
    const int64_t have = src == p->req_pages.end() ? 0 : (int64_t)src->second.size();
    if (need > have) return PCP_ERR_INVALID_ARG;
    auto dst = p->req_pages.find(dst_req);
    if (dst != p->req_pages.end() && !dst->second.empty()) return PCP_ERR_INVALID_ARG;
    if (need == 0) return PCP_OK;
    std::vector<int32_t>& out = p->req_pages[dst_req];
    for (int64_t i = 0; i < need; ++i) {
        const int32_t pg = p->req_pages[src_req][i];
        ++p->refs[pg];
        out.push_back(pg);
    }
    p->held_entries += need;
    return PCP_OK;
}

int64_t pcp_pager_cache_prompt(pcp_pager* p, int64_t req_id, const int32_t* tokens,
                               int64_t n_tokens) {
    if (p == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr)) return -1;
    auto it = p->req_pages.find(req_id);
    const int64_t held = it == p->req_pages.end() ? 0 : (int64_t)it->second.size();
    const int64_t full = std::min<int64_t>(n_tokens / p->page_size, held);
    uint64_t parent = 0;
    int64_t added = 0;
    for (int64_t i = 0; i < full; ++i) {
        const int32_t* blk = tokens + i * p->page_size;
        const uint64_t key = block_key(parent, blk, p->page_size);
        auto e = p->index.find(key);
        if (e == p->index.end()) {
            const int32_t pg = it->second[i];
            if (p->cached_key[pg] != 0) break;  // the page is cached under another prefix
            p->index.emplace(key, CacheEntry{pg, parent,
                                             std::vector<int32_t>(blk, blk + p->page_size)});
            p->cached_key[pg] = key;
            ++p->refs[pg];
            ++added;
        } else if (e->second.parent != parent ||
                   !std::equal(blk, blk + p->page_size, e->second.tokens.begin())) {
            break;  // a different prefix under the same key: stop here
        }
        parent = key;
    }
    return added;
}

pcp_status pcp_pager_match_prefix(pcp_pager* p, int64_t req_id, const int32_t* tokens,
                                  int64_t n_tokens, int64_t* n_hit) {
    if (p == nullptr || n_hit == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
        return PCP_ERR_INVALID_ARG;
    auto it = p->req_pages.find(req_id);
    if (it != p->req_pages.end() && !it->second.empty()) return PCP_ERR_INVALID_ARG;
    *n_hit = 0;
    // whole pages only, and at least the prompt's last token is left to compute
    const int64_t max_blocks = n_tokens > 0 ? (n_tokens - 1) / p->page_size : 0;
    std::vector<int32_t> hit;
    uint64_t parent = 0;
    for (int64_t i = 0; i < max_blocks; ++i) {
        const int32_t* blk = tokens + i * p->page_size;
        const uint64_t key = block_key(parent, blk, p->page_size);
        auto e = p->index.find(key);
        if (e == p->index.end() || e->second.parent != parent ||
            !std::equal(blk, blk + p->page_size, e->second.tokens.begin()))
            break;
        hit.push_back(e->second.page);
        parent = key;
    }
    if (hit.empty()) return PCP_OK;
    std::vector<int32_t>& pages = p->req_pages[req_id];
    for (int32_t pg : hit) {
        ++p->refs[pg];
        pages.push_back(pg);
    }
    p->held_entries += (int64_t)hit.size();
    *n_hit = (int64_t)hit.size() * p->page_size;
    return PCP_OK;
}

pcp_status pcp_pager_clear_cache(pcp_pager* p) {
    if (p == nullptr) return PCP_ERR_INVALID_ARG;
    for (auto& kv : p->index) {
        p->cached_key[kv.second.page] = 0;
        p->drop_page(kv.second.page);
    }
    p->index.clear();
    return PCP_OK;
}

pcp_status pcp_schedule_step(pcp_pager* p, int n_reqs, const int64_t* req_ids,
                             const int32_t* total_lens, const int32_t* num_computed, int budget,
                             int state_block, int32_t* n_rows, int32_t* row_req,
                             int32_t* qo_indptr, int32_t* prefix_lens, int32_t* kv_indptr,
                             int32_t* kv_indices, int64_t kv_indices_cap, uint8_t* sample,
                             int32_t* n_copies, int32_t* copy_src, int32_t* copy_dst,
                             int32_t* copy_slots) {
    if (p == nullptr || n_reqs < 0 || budget < 0 || state_block < 0 || n_rows == nullptr ||
        kv_indices_cap < 0 || n_copies == nullptr)
        return PCP_ERR_INVALID_ARG;
    if (n_reqs > 0 && (copy_src == nullptr || copy_dst == nullptr || copy_slots == nullptr))
        return PCP_ERR_INVALID_ARG;
    if (n_reqs > 0 && (req_ids == nullptr || total_lens == nullptr || num_computed == nullptr ||
                       row_req == nullptr || qo_indptr == nullptr || prefix_lens == nullptr ||
                       kv_indptr == nullptr || sample == nullptr))
        return PCP_ERR_INVALID_ARG;
    // each request's page list, looked up once (null: it holds no pages yet;
    // the map keeps element addresses stable while others are inserted)
    std::vector<std::vector<int32_t>*> held_pages(n_reqs, nullptr);
    {
        std::vector<int64_t> ids(req_ids, req_ids + n_reqs);
        std::sort(ids.begin(), ids.end());
        if (std::adjacent_find(ids.begin(), ids.end()) != ids.end()) return PCP_ERR_INVALID_ARG;
        for (int r = 0; r < n_reqs; ++r) {
            if (total_lens[r] < 0 || num_computed[r] < 0 || num_computed[r] > total_lens[r])
                return PCP_ERR_INVALID_ARG;
            auto it = p->req_pages.find(req_ids[r]);
            if (it != p->req_pages.end()) held_pages[r] = &it->second;
            // the pages a request holds must cover its computed tokens
            const int64_t held = held_pages[r] ? (int64_t)held_pages[r]->size() : 0;
            if (held < pages_for(num_computed[r], p->page_size)) return PCP_ERR_INVALID_ARG;
        }
    }
    auto n_held = [&](int r) -> int64_t {
        return held_pages[r] ? (int64_t)held_pages[r]->size() : 0;
    };
    // ---- choose the chunk of every request
    std::vector<int32_t> chunk(n_reqs, 0);
    int64_t left = budget;
    int64_t free_pages = (int64_t)p->free_pages.size();
    // does the first token of a chunk of request r land in a shared page
    // (which it must copy to a fresh page first)?
    auto needs_copy = [&](int r) {
        const int64_t start = num_computed[r];
        if (start % p->page_size == 0) return false;
        const int64_t idx = start / p->page_size;
        return idx < n_held(r) && p->refs[(*held_pages[r])[idx]] > 1;
    };
    auto grant = [&](int r, int64_t want) {
        const int64_t start = num_computed[r];
        const int64_t held = n_held(r);
        int64_t avail = free_pages;
        if (needs_copy(r)) {
            if (avail == 0) return;  // no page to copy the shared one into
            --avail;
        }
        // tokens that fit in the held pages plus the free ones
        const int64_t room = (held + avail) * p->page_size - start;
        const int64_t n = std::max<int64_t>(0, std::min(want, room));
        if (n == 0) return;
        free_pages = avail - std::max<int64_t>(0, pages_for(start + n, p->page_size) - held);
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
        entries += std::max<int64_t>(n_held(r), pages_for(end, p->page_size));  // the row's page list
        ++rows;
    }
    if (kv_indices_cap < entries || (entries > 0 && kv_indices == nullptr))
        return PCP_ERR_WORKSPACE;
    rows = 0;
    entries = 0;
    int copies = 0;
    qo_indptr[0] = 0;
    kv_indptr[0] = 0;
    for (int r = 0; r < n_reqs; ++r) {
        if (chunk[r] == 0) continue;
        const bool copy = needs_copy(r);
        if (held_pages[r] == nullptr) held_pages[r] = &p->req_pages[req_ids[r]];
        std::vector<int32_t>& pages = *held_pages[r];
        const int64_t end = (int64_t)num_computed[r] + chunk[r];
        if (copy) {  // copy-on-write of the shared page the chunk continues in
            const int64_t idx = num_computed[r] / p->page_size;
            const int32_t old_pg = pages[idx];
            const int32_t new_pg = p->take_page();
            copy_src[copies] = old_pg;
            copy_dst[copies] = new_pg;
            copy_slots[copies] = num_computed[r] % p->page_size;
            ++copies;
            pages[idx] = new_pg;
            p->drop_page(old_pg);
        }
        while ((int64_t)pages.size() < pages_for(end, p->page_size)) {
            pages.push_back(p->take_page());
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
    *n_copies = copies;
    return PCP_OK;
}

}  // extern "C"
