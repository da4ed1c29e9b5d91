// Work planning on the device (one CTA).
//
// From the device copies of qo_indptr / prefix_lens / kv_indptr it builds the
// two work lists of one pcp_paged_extend_attn call, so the host needs no copy
// of the metadata and no synchronisation:
//
//  * tensor-core items {b, kv head, first position, cost}: each covers
//    kQTiles * (128 / G) positions of one chunk for one KV head (all G query
//    heads of that KV head packed into the MMA rows).  Items are ordered by
//    cost (number of KV tiles) descending -- longest-processing-time first
//    for the persistent kernel's dynamic scheduler -- with a counting sort
//    over cost buckets (exact below 64 tiles, 16 tiles wide above).  Inside
//    a bucket every warp places the items of one (sequence, KV head) next to
//    each other, so the CTAs running at the same time stream few sequences'
//    K/V and each tile is read from DRAM about once (with one item per
//    bucket slot in any order, a long prefix is re-read by every item from
//    DRAM once the groups' K/V together exceed the L2).
//  * row groups for decode-shaped chunks (chunk_len * G <= 16 rows), one per
//    (sequence, KV head): their 128-key tiles are laid end to end and the
//    row kernel's CTA i of n takes tiles [i*T/n, (i+1)*T/n), so every SM
//    streams the same number of K/V bytes.  A group held by several CTAs is
//    split at their boundaries; each piece owns a partial slot for the
//    log-sum-exp combine.  This is the split-KV idea of the AstrAI paged
//    decode kernel (splits from the SM count, partials merged by a combine
//    step) with the split points chosen for equal work per SM.
//  * a call that has tensor-core work takes its decode-shaped chunks onto the
//    tensor cores as one-Q-tile items when the longest of them ends within
//    the tensor-core schedule's expected length: the longest-first queue
//    then fills the SMs that the prompt items leave idle, and the row kernel
//    and the combine find no work.  A decode-shaped item costs about 0.8 of
//    a two-Q-tile step per KV tile (its one Q tile alone: measured 1.66 us
//    against 2.07 us on the GQA workload), so it is charged that in the
//    longest-first order and in the test.
//  * a call whose longest item far exceeds the average work per SM (the
//    host's decision, split_longest_items) splits its longest items in two
//    along their KV tiles: the items above half the average work per SM and
//    above 16 tiles, longest first, at most kTcMaxSplitItems.  The two parts
//    are items of their own in the longest-first order; the part that ends
//    second merges the first one's partial result.
#include "pcp_append_body.cuh"
#include "pcp_device.cuh"
#include "pcp_internal.h"
#include "pcp_launch.h"

namespace pcp {

namespace {

struct SeqInfo {
    int c, P, L, q0, kvb;
    bool ok;
};

__device__ __forceinline__ SeqInfo seq_info(const PlanParams& p, int b) {
    SeqInfo s;
    const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    s.q0 = q0;
    s.kvb = p.kv_indptr[b];
    s.c = q1 - q0;
    s.P = p.prefix_lens[b];
    s.L = s.P + s.c;
    const int pages = p.kv_indptr[b + 1] - s.kvb;
    s.ok = q0 >= 0 && s.c >= 0 && q1 <= p.total_q && s.P >= 0 && pages >= 0 &&
           (int64_t)pages * p.page_size >= (int64_t)s.L;
    return s;
}

// First visible key of absolute position `pos`.
__device__ __forceinline__ int first_key(int pos, int window) {
    return window > 0 ? max(0, pos - window + 1) : 0;
}

// Bucket of a tensor-core item's cost in the longest-first counting sort:
// the cost itself below 64 KV tiles, 16-tile buckets above.
__device__ __forceinline__ int cost_bucket(int cost) {
    return cost < 64 ? cost : min(1023, 64 + ((cost - 64) >> 4));
}

// Lowest cost in a bucket of cost_bucket.
__device__ __forceinline__ int bucket_min_cost(int bucket) {
    return bucket < 64 ? bucket : 64 + ((bucket - 64) << 4);
}


// KV tiles of tensor-core item k of a chunk (tc_item_tiles).
__device__ __forceinline__ int tc_cost(int P, int c, int k, int item_pos, int window,
                                       int causal) {
    return tc_item_tiles(P, c, k, item_pos, window, causal);
}

// Turn a 1024-bucket histogram into descending exclusive offsets (bucket
// 1023 first) in place and return the total.  1024 threads; warp-shuffle
// scans, three block barriers.
__device__ __forceinline__ int desc_offsets(int* hist, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int own = hist[1023 - tid];
    int v = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int x = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        warp_sums[32 + lane] = x;  // inclusive prefix over warps
    }
    __syncthreads();
    const int before = w > 0 ? warp_sums[32 + w - 1] : 0;
    hist[1023 - tid] = before + v - own;
    const int total = warp_sums[32 + 31];
    __syncthreads();
    return total;
}

// Exclusive prefix sum of a[0..1023] into a[0..1024] (a[1024] = total);
// returns the total.  1024 threads.
__device__ __forceinline__ int excl_scan(int* a, int* warp_sums) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int own = a[tid];
    int v = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int x = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += n;
        }
        warp_sums[32 + lane] = x;
    }
    __syncthreads();
    a[tid] = (w > 0 ? warp_sums[32 + w - 1] : 0) + v - own;
    const int total = warp_sums[32 + 31];
    if (tid == 0) a[1024] = total;
    __syncthreads();
    return total;
}

// Position of flattened index f among segments with exclusive starts a[0..n]:
// the last s with a[s] <= f.
__device__ __forceinline__ int segment_of(const int* a, int n, int f) {
    int lo = 0, hi = n;  // answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a[mid] <= f) lo = mid;
        else hi = mid;
    }
    return lo;
}

// atomicAdd(&base[key], inc) for every active lane, one atomic per distinct
// key in the warp; returns this lane's old value (lanes with the same key
// get consecutive ranges).
__device__ __forceinline__ int warp_agg_add(int* base, int key, int inc) {
    const unsigned act = __activemask();
    const unsigned same = __match_any_sync(act, key);
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(same) - 1;
    const int rank = __popc(same & ((1u << lane) - 1));
    int old = 0;
    if (lane == leader) old = atomicAdd(&base[key], inc * __popc(same));
    old = __shfl_sync(same, old, leader);
    return old + rank * inc;
}

}  // namespace

// Sequences are processed in chunks of 1024 (one per thread); within a chunk
// the per-sequence items and row groups are flattened across all threads
// through prefix sums, so a long chunk does not serialise on one thread.
// kSplit: the call splits its longest tensor-core items (the host's decision);
// the other instantiation carries none of that code.
// The planner's shared memory (the planning CTA's, in both kernels below).
struct PlanSmem {
    int hist[1025];      // cost buckets; entry 1024 takes no-op additions
    int hist_dec[1024];  // decode-shaped chunks as tensor-core items
    int s_cut;           // lowest bucket whose items are split in two (1024: none)
    int s_nsplit;        // split items placed so far
    int warp_sums[64];
    unsigned long long s_w_tc, s_w_dec;  // summed costs (two-Q-tile steps)
    int s_max_tc, s_max_dec;             // longest item of each kind
    int s_a[1025];       // per-sequence counts, then their exclusive prefix
    int s_b[1025];
    int s_c[1025];
    int4 s_seq[1024];    // {c, P, ok, row tiles}
    int2 s_off[1024];    // {qo_indptr[b], kv_indptr[b]}
    unsigned long long s_row_tiles;
};

template <bool kSplit>
__device__ __forceinline__ void plan_body(const PlanParams& p, PlanSmem& S) {
    auto& hist = S.hist;
    auto& hist_dec = S.hist_dec;
    auto& s_cut = S.s_cut;
    auto& s_nsplit = S.s_nsplit;
    auto& warp_sums = S.warp_sums;
    auto& s_w_tc = S.s_w_tc;
    auto& s_w_dec = S.s_w_dec;
    auto& s_max_tc = S.s_max_tc;
    auto& s_max_dec = S.s_max_dec;
    auto& s_a = S.s_a;
    auto& s_b = S.s_b;
    auto& s_c = S.s_c;
    auto& s_seq = S.s_seq;
    auto& s_off = S.s_off;
    auto& s_row_tiles = S.s_row_tiles;

    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
    int4* tc = reinterpret_cast<int4*>(p.ws + p.lay.tc_items);
    int4* rg = reinterpret_cast<int4*>(p.ws + p.lay.row_groups);
    int* row_first = reinterpret_cast<int*>(p.ws + p.lay.row_first);
    int4* gdesc = reinterpret_cast<int4*>(p.ws + p.lay.group_desc);
    const int tid = threadIdx.x, lane = tid & 31;
    const int item_pos = q_positions_per_tile(p.group) * kQTiles;
    const int rmax = row_path_max_chunk(p.group);
    const int H = p.n_kv_heads;
    const int n_ctas = row_grid(p.sm_count);

    // The call's metadata are not the previous kernel's output, so they are
    // read and the tensor-core histogram built while that kernel finishes;
    // the wait for it comes before the first write to global memory (the
    // workspace may still be read by the previous call's kernels).
    pdl_launch_dependents();
    hist[tid] = 0;
    hist_dec[tid] = 0;
    if (tid == 0) {
        hist[1024] = 0;
        s_cut = 1024;
        s_nsplit = 0;
        s_row_tiles = 0;
        s_w_tc = s_w_dec = 0;
        s_max_tc = s_max_dec = 0;
    }
    bool bad_meta = false;  // this thread saw contradictory metadata

    // metadata of sequence chunk0 + tid (kept in s_seq); notes bad sequences
    auto load_chunk = [&](int chunk0, bool report) {
        const int b = chunk0 + tid;
        int4 v = make_int4(0, 0, 0, 0);
        int2 off = make_int2(0, 0);
        if (b < p.batch) {
            const SeqInfo q = seq_info(p, b);
            off = make_int2(q.q0, q.kvb);
            // qo_indptr[batch] must be total_q (the last sequence's end)
            if (report && (!q.ok || (b == p.batch - 1 && q.q0 + q.c != p.total_q)))
                bad_meta = true;
            const int tiles = (q.ok && q.c > 0 && q.c <= rmax)
                                  ? (q.L - 1) / kRowTile - first_key(q.P, p.window) / kRowTile + 1
                                  : 0;
            v = make_int4(q.c, q.P, q.ok ? 1 : 0, tiles);
        }
        s_seq[tid] = v;
        s_off[tid] = off;
    };
    // tensor-core items of one KV head (decode-shaped chunks: one, when
    // the call takes them onto the tensor cores)
    auto n_tc_of = [&](int4 v, bool absorb) {
        return (v.z && (v.x > rmax || (absorb && v.w > 0))) ? (v.x + item_pos - 1) / item_pos
                                                            : 0;
    };
    const bool one_chunk = p.batch <= 1024;

    // ---- sweep 1: tensor-core cost histogram, row tile total, and both
    // kinds' total and longest cost
    unsigned long long w_tc = 0, w_dec = 0;
    int max_tc = 0, max_dec = 0;
    for (int chunk0 = 0; chunk0 < p.batch; chunk0 += 1024) {
        __syncthreads();
        load_chunk(chunk0, true);
        s_a[tid] = n_tc_of(s_seq[tid], false);
        if (p.tc_work && s_seq[tid].w > 0) {
            // a decode-shaped chunk: one item of its row tiles per KV head
            const int wc = dec_weight(s_seq[tid].w);
            w_dec += (unsigned long long)wc * H;
            max_dec = max(max_dec, wc);
            warp_agg_add(hist_dec, cost_bucket(wc), H);
        }
        // each row group adds its virtual start tiles to the split
        unsigned long long rt =
            s_seq[tid].w > 0 ? (unsigned long long)(s_seq[tid].w + kRowGroupStartTiles) * H : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) rt += __shfl_xor_sync(0xffffffffu, rt, o);
        if (lane == 0 && rt) atomicAdd(&s_row_tiles, rt);
        __syncthreads();
        if (p.tc_work) {
            const int total = excl_scan(s_a, warp_sums);
            for (int f = tid; f < total; f += 1024) {
                const int sl = segment_of(s_a, 1024, f);
                const int4 v = s_seq[sl];
                const int cost = tc_cost(v.y, v.x, f - s_a[sl], item_pos, p.window, p.causal);
                w_tc += (unsigned long long)cost * H;
                max_tc = max(max_tc, cost);
                warp_agg_add(hist, cost_bucket(cost), H);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        w_tc += __shfl_xor_sync(0xffffffffu, w_tc, o);
        w_dec += __shfl_xor_sync(0xffffffffu, w_dec, o);
        max_tc = max(max_tc, __shfl_xor_sync(0xffffffffu, max_tc, o));
        max_dec = max(max_dec, __shfl_xor_sync(0xffffffffu, max_dec, o));
    }
    if (lane == 0) {
        if (w_tc) atomicAdd(&s_w_tc, w_tc);
        if (w_dec) atomicAdd(&s_w_dec, w_dec);
        atomicMax(&s_max_tc, max_tc);
        atomicMax(&s_max_dec, max_dec);
    }
    __syncthreads();
    // Decode-shaped chunks go to the tensor cores when the call has prompt
    // items and the longest decode-shaped item stays within 1.1 times the
    // schedule's expected length (its longest item or its average per SM);
    // the host's decision, when it made one, stands.
    const bool absorb =
        p.tc_work && (p.absorb >= 0 ? p.absorb == 1
                                    : absorb_decode_rows(s_w_tc, s_max_tc, s_w_dec, s_max_dec,
                                                         p.sm_count));
    if (absorb) hist[tid] += hist_dec[tid];
    __syncthreads();
    int n_tc = p.tc_work ? desc_offsets(hist, warp_sums) : 0;
    const unsigned long long row_tiles_all = absorb ? 0ull : s_row_tiles;

    // The item of KV-tile cost `tiles` and bucket `bk` is split when bk >= cut:
    // part 0 takes its first (tiles + 1) / 2 tiles.  A part's weight: its
    // tiles, or for a decode-shaped item dec_weight of them.
    auto part_weight = [&](int tiles, bool dec) { return dec ? dec_weight(tiles) : tiles; };
    if (kSplit && p.tc_work && p.lay.cap_split > 0) {
        // hist[b] now counts the items in the buckets above b, so the items in
        // buckets >= b number hist[b - 1]; the buckets to split are the top ones
        const unsigned long long w_all = s_w_tc + (absorb ? s_w_dec : 0ull);
        const unsigned long long theta =
            max(w_all / (2ull * (unsigned long long)max(p.sm_count, 1)), 16ull);
        const int above = tid > 0 ? hist[tid - 1] : n_tc;
        if (above <= p.lay.cap_split && (unsigned long long)bucket_min_cost(tid) > theta)
            atomicMin(&s_cut, tid);
        __syncthreads();
        if (s_cut < 1024) {
            // ---- sweep 1b: the histogram again, with the parts' own costs
            hist[tid] = 0;
            if (tid == 0) hist[1024] = 0;
            for (int chunk0 = 0; chunk0 < p.batch; chunk0 += 1024) {
                __syncthreads();
                if (!one_chunk) load_chunk(chunk0, false);
                s_a[tid] = n_tc_of(s_seq[tid], absorb);
                __syncthreads();
                const int total = excl_scan(s_a, warp_sums);
                for (int f = tid; f < total; f += 1024) {
                    const int sl = segment_of(s_a, 1024, f);
                    const int4 v = s_seq[sl];
                    const int k = f - s_a[sl];
                    const bool dec = v.x <= rmax;
                    const int tiles = tc_cost(v.y, v.x, k, item_pos, p.window, p.causal);
                    const int bk = cost_bucket(part_weight(tiles, dec));
                    const int first =
                        first_key(v.y + k * item_pos, p.window) / kTileN;
                    const bool split = bk >= s_cut && first + tiles <= kSplitMaxTile;
                    const int c0 = (tiles + 1) / 2;
                    warp_agg_add(hist, split ? cost_bucket(part_weight(c0, dec)) : bk, H);
                    warp_agg_add(hist, split ? cost_bucket(part_weight(tiles - c0, dec)) : 1024,
                                 H);
                }
            }
            __syncthreads();
            n_tc = desc_offsets(hist, warp_sums);
        }
    }
    const int cut = kSplit ? s_cut : 1024;

    // ---- from here on global memory is written: the previous kernel is done
    pdl_wait();
    if (bad_meta) report_error(p.dev_err, PCP_ERR_INVALID_ARG);
    if (tid == 0 && row_tiles_all >= (1ull << 31)) report_error(p.dev_err, PCP_ERR_UNSUPPORTED);
    for (int64_t i = tid; i < (int64_t)p.batch * H; i += 1024) gdesc[i] = make_int4(0, 0, 0, 0);
    if (kSplit && cut < 1024) {  // split items' tickets and ready flags start at zero
        int* tc_sync = reinterpret_cast<int*>(p.ws + p.lay.tc_sync);
        for (int64_t i = tid; i < p.lay.cap_split * kQTiles * 4 * 2; i += 1024) tc_sync[i] = 0;
    }
    const int64_t cap_items = p.lay.cap_tc + p.lay.cap_split;
    // a CTA whose tiles are all virtual has no row group
    if (tid < kRowMaxCtas) row_first[tid] = -1;
    const int T = (int)min(row_tiles_all, (unsigned long long)INT32_MAX);
    // the split uses min(n, T) CTAs, so every one of them holds at least one
    // tile and every partial slot of a group is written
    const int n_use = row_ctas_used(n_ctas, T);
    // the row-kernel CTA holding tile x: the last i with i*T/n_use <= x
    auto cta_of = [&](int x) {
        return (int)((((int64_t)x + 1) * n_use + T - 1) / T) - 1;
    };

    // ---- sweep 2: scatter tensor-core items and row groups
    int grp_base = 0;   // row groups of earlier chunks
    int tile_base = 0;  // row tiles of earlier chunks
    for (int chunk0 = 0; chunk0 < p.batch; chunk0 += 1024) {
        __syncthreads();
        if (!one_chunk) load_chunk(chunk0, false);
        // items flattened as (sequence, KV head, item)
        s_a[tid] = n_tc_of(s_seq[tid], absorb) * H;
        s_b[tid] = !absorb && s_seq[tid].w > 0 ? H : 0;
        s_c[tid] = !absorb && s_seq[tid].w > 0 ? s_seq[tid].w + kRowGroupStartTiles : 0;
        __syncthreads();
        const int total_a = p.tc_work ? excl_scan(s_a, warp_sums) : 0;
        const int total_b = excl_scan(s_b, warp_sums);
        const int total_c = excl_scan(s_c, warp_sums);
        for (int f = tid; f < total_a; f += 1024) {
            const int sl = segment_of(s_a, 1024, f);
            const int4 v = s_seq[sl];
            const int n = n_tc_of(v, absorb);
            const int g = (f - s_a[sl]) / n;
            const int k = (f - s_a[sl]) - g * n;
            const int cost = tc_cost(v.y, v.x, k, item_pos, p.window, p.causal);
            if constexpr (!kSplit) {
                // a decode-shaped chunk's item is in the bucket of its weight
                const int wc = v.x > rmax ? cost : dec_weight(v.w);
                // lanes with one bucket get consecutive slots in lane order
                const int slot = warp_agg_add(hist, cost_bucket(wc), 1);
                if (slot >= p.lay.cap_tc) {
                    report_error(p.dev_err, PCP_ERR_WORKSPACE);
                    continue;
                }
                tc[slot] = make_int4(chunk0 + sl, g, k * item_pos, cost);
            } else {
                // a decode-shaped chunk's item is in the bucket of its weight
                const bool dec = v.x <= rmax;
                const int bk = cost_bucket(part_weight(cost, dec));
                const int first = first_key(v.y + k * item_pos, p.window) / kTileN;
                const bool split = bk >= cut && first + cost <= kSplitMaxTile;
                const int c0 = (cost + 1) / 2;
                // lanes with one bucket get consecutive slots in lane order; a split
                // item places its second part too (the others add nothing to the
                // spare entry)
                const int slot =
                    warp_agg_add(hist, split ? cost_bucket(part_weight(c0, dec)) : bk, 1);
                // (cut is the same for the whole block, so every lane of a warp
                // takes this branch or none)
                const int slot1 =
                    cut < 1024 ? warp_agg_add(
                                     hist, split ? cost_bucket(part_weight(cost - c0, dec)) : 1024, 1)
                               : 0;
                int w0 = cost, w1 = 0;
                if (split) {
                    const int sp = atomicAdd(&s_nsplit, 1);  // < cap_split by the cut
                    w0 = kSplitTag | ((first + c0) << 12) | (sp << 1);
                    w1 = w0 | 1;
                }
                if (slot >= cap_items || (split && slot1 >= cap_items)) {
                    report_error(p.dev_err, PCP_ERR_WORKSPACE);
                    continue;
                }
                tc[slot] = make_int4(chunk0 + sl, g, k * item_pos, w0);
                if (split) tc[slot1] = make_int4(chunk0 + sl, g, k * item_pos, w1);
            }
        }
        for (int f = tid; f < total_b; f += 1024) {
            const int sl = segment_of(s_b, 1024, f);
            const int b = chunk0 + sl;
            const int g = f - s_b[sl];
            const int k = grp_base + f;
            const int4 v = s_seq[sl];
            const int tiles = v.w;
            // the group's span on the tile line starts with its virtual tiles;
            // its pieces are the CTAs' shares of its real tiles [S, S + tiles)
            const int S0 = tile_base + s_c[sl] * H + g * (tiles + kRowGroupStartTiles);
            const int S = S0 + kRowGroupStartTiles;
            const int i_first = cta_of(S), i_last = cta_of(S + tiles - 1);
            const int ns = i_last - i_first + 1;
            const int base = k + i_first;
            if (k >= p.lay.cap_groups || base + ns > p.lay.cap_row) {
                report_error(p.dev_err, PCP_ERR_WORKSPACE);
                continue;
            }
            const int P = v.y, L = v.x + v.y;
            const int q0 = s_off[sl].x;
            rg[3 * k] = make_int4(b, g, S, tiles);
            rg[3 * k + 1] = make_int4(first_key(P, p.window), q0, base, ns);
            rg[3 * k + 2] = make_int4(v.x, P, s_off[sl].y, L);
            gdesc[(int64_t)b * H + g] = make_int4(base, ns, q0, v.x);
            // CTAs whose range starts in this group's span start with it
            for (int i = i_first; i <= i_last; ++i)
                if (row_tile_begin(i, n_use, T) >= S0) row_first[i] = k;
        }
        grp_base += total_b;
        tile_base += total_c * H;
    }
    __syncthreads();
    if (tid == 0) {
        hdr->n_tc_items = (int)min((int64_t)n_tc, cap_items);
        hdr->n_row_groups = (int)min((int64_t)grp_base, p.lay.cap_groups);
        // with cp.async page gathers, the tensor-core kernel's CTA i (one per
        // SM) starts with item i and the counter hands out the rest
        hdr->tc_next = p.tc_gather ? p.sm_count : 0;
        hdr->row_tiles = T;
        hdr->row_ctas = n_ctas;
    }
}

template <bool kSplit>
__global__ void __launch_bounds__(1024, 1) plan_kernel(const __grid_constant__ PlanParams p) {
    __shared__ PlanSmem S;
    plan_body<kSplit>(p, S);
}

// The planner in CTA 0 and the append of the call's new K/V rows in the other
// CTAs (a span of 4096 chunks each), in one launch: both run at once, one
// CTA per SM, instead of the planner waiting for an SM that the append has
// left.
constexpr int kPlanAppendThreads = 1024;
constexpr size_t kPlanAppendSmem = sizeof(PlanSmem) > sizeof(AppendSmem<kPlanAppendThreads>)
                                       ? sizeof(PlanSmem)
                                       : sizeof(AppendSmem<kPlanAppendThreads>);

template <bool kSplit>
__global__ void __launch_bounds__(kPlanAppendThreads, 1)
    plan_append_kernel(const __grid_constant__ PlanParams p, const __grid_constant__ AppendParams a) {
    extern __shared__ __align__(16) unsigned char smem[];
    if (blockIdx.x == 0) {
        plan_body<kSplit>(p, *reinterpret_cast<PlanSmem*>(smem));
    } else {
        // the new K/V rows may be the previous kernel's output, and the pools
        // may still be read by it
        pdl_wait();
        pdl_launch_dependents();
        append_paged_span<kPlanAppendThreads>(
            a, *reinterpret_cast<AppendSmem<kPlanAppendThreads>*>(smem), blockIdx.x - 1);
    }
}

cudaError_t launch_plan(cudaStream_t stream, const PlanParams& p) {
    if (p.split) return launch_pdl(plan_kernel<true>, dim3(1), dim3(1024), 0, stream, p);
    return launch_pdl(plan_kernel<false>, dim3(1), dim3(1024), 0, stream, p);
}

// Append CTAs of plan_append_kernel for the call (one span each).
int64_t plan_append_spans(const AppendParams& a) {
    constexpr int64_t span = (int64_t)kPlanAppendThreads * kAppendUnroll;
    return (a.total_q * a.chunks_per_token + span - 1) / span;
}

cudaError_t launch_plan_append(cudaStream_t stream, const PlanParams& p, const AppendParams& a) {
    const dim3 grid((unsigned)(1 + plan_append_spans(a)));
    if (p.split)
        return launch_pdl(plan_append_kernel<true>, grid, dim3(kPlanAppendThreads),
                          kPlanAppendSmem, stream, p, a);
    return launch_pdl(plan_append_kernel<false>, grid, dim3(kPlanAppendThreads),
                      kPlanAppendSmem, stream, p, a);
}

}  // namespace pcp
