// Decode-shaped rows: split-KV attention, HBM-bound.
//
// A chunk with chunk_len * G <= 16 query rows (a decode row is chunk_len 1)
// uses each key for at most 16 rows, so this path is bound by reading the
// K/V pages, not by arithmetic.  The KV range of each (sequence, KV head) is
// split across CTAs (AstrAI paged decode "split-KV" kernel, prior art); each
// split writes an fp32 partial (unnormalised O, running max, normaliser) to
// the workspace and combine_kernel merges the partials with the log-sum-exp
// identity afterwards (the AstrAI combine kernel's job).  Merging inside the
// last split to finish was tried: its dependent L2 reads stalled that SM's
// load pipeline for ~10 us per group.  Masking is the same bottom-right
// causal / window rule as the tensor-core path, per row.
//
// Layout: one CTA per SM, 4 consumer warps and 1 load warp, a ring of
// 128-key K+V stages with full/empty mbarriers.  The load warp fills a stage
// by TMA (one box per page run of >= 8 keys and 64-column block; the V page
// run holding the sequence end by zero-filling cp.async) or, for smaller
// pages, by 16-byte cp.async gathers; both land in the 128-byte-swizzled
// layout.  The up to 16 query rows (position x head) form the M = 16 side of
// warp-level m16n8k16 bf16 MMAs: consumer warp w takes keys 32w..32w+31 of a
// tile, computes S = Q K^T with K fragments from ldmatrix, keeps an online
// softmax in fp32, reuses the S accumulators as the P operand, and adds P V
// with V fragments from ldmatrix.trans.  The four warp states are merged at
// the end of each item.
#include "pcp_device.cuh"
#include "pcp_internal.h"
#include "pcp_launch.h"

namespace pcp {

namespace {

template <int D>
struct RowCfg {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = kRowTile * 128;            // one 64-column block
    static constexpr int kTileBytes = kRowTile * D * 2;          // a K or a V tile
    static constexpr int kStages = D == 128 ? 3 : 5;
    static constexpr int kItemSlots = 2;
    static constexpr int kQStride = D * 2 + 16;                  // padded Q row (bytes)
    static constexpr int kOffStage = 0;                          // [stage][K | V]
    static constexpr int kOffQ = kOffStage + kStages * 2 * kTileBytes;  // [slot][16][kQStride]
    static constexpr int kOffDesc = kOffQ + kItemSlots * kRowMaxRows * kQStride;  // int4 [slot][3]
    static constexpr int kOffBar = kOffDesc + kItemSlots * 48;
    static constexpr int kOffM = kOffBar + (2 * kStages + 2 * kItemSlots) * 8;  // float [4][16] m, l
    // merge buffer of an item's four warp states, four rows at a time:
    // [4 warps][4 rows][D + 8] fp32 (the padding puts the rows of one float2
    // store on different banks)
    static constexpr int kMergeRows = 4;
    static constexpr int kMergeStride = D + 8;
    static constexpr int kOffMerge = kOffM + 2 * 4 * kRowMaxRows * 4;
    static constexpr int kSmemBytes =
        kOffMerge + 4 * kMergeRows * kMergeStride * 4 + 64 + 1024;
    static_assert(kOffDesc % 16 == 0 && kOffBar % 8 == 0 && kOffStage % 1024 == 0 &&
                      kOffMerge % 16 == 0,
                  "smem alignment");
};

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// Byte offset of (row, dim) in a 128-byte-swizzled tile (16-byte granules).
template <int D>
__device__ __forceinline__ uint32_t swz(int row, int dim) {
    return (uint32_t)((dim >> 6) * RowCfg<D>::kHalfBytes + row * 128 +
                      ((((dim & 63) >> 3) ^ (row & 7)) << 4));
}

}  // namespace

// kMask: the call passes a boolean mask (a separate instantiation).
template <int D, bool kMask>
__global__ void __launch_bounds__(kRowThreads, 1)
    row_attn_kernel(const __grid_constant__ RowParams p, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
    using C = RowCfg<D>;
    constexpr int S = C::kStages;
    constexpr int NI = C::kItemSlots;
    constexpr int kConsumerThreads = 128;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* sm = smem_raw + (base - raw);
    float* m_s = reinterpret_cast<float*>(sm + C::kOffM);
    float* l_s = m_s + 4 * kRowMaxRows;
    int4* s_desc = reinterpret_cast<int4*>(sm + C::kOffDesc);  // published by mbarrier
    __shared__ int s_abort, s_zero;
    // consumer warps' posts at their joint decision points
    __shared__ int s_post[4], s_fail[4];
    __shared__ __align__(8) uint64_t s_stall;  // nothing arrives on it (timeout test)
    // self-planned calls: per sequence {chunk_len, prefix_len, kv_indptr[b],
    // qo_indptr[b]}, and exclusive prefix sums over the sequences of their
    // row tiles and of their row-group counts (1 for a decode-shaped chunk)
    __shared__ int4 s_sp_seq[kRowSelfPlanMaxSeqs];
    __shared__ int s_sp_ts[kRowSelfPlanMaxSeqs + 1], s_sp_gs[kRowSelfPlanMaxSeqs + 1];
    __shared__ long long s_sp_wsum[2][kRowThreads / 32];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int H = p.n_kv_heads;
    const int rmax = row_path_max_chunk(p.group);
    // ---- self-planned call: the split of the row tiles, from the metadata
    // alone (read before the wait below; they are inputs of the call)
    long long sp_total = 0;   // row tiles of one KV head, all sequences
    long long sp_groups = 0;  // row sequences (row groups of one KV head)
    bool sp_bad = false;     // this thread saw contradictory metadata
    if (p.self_plan) {
        // thread i takes sequences 4i .. 4i + 3
        long long t_run = 0, g_run = 0;
        int tl[4], rw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = 4 * tid + j;
            tl[j] = rw[j] = 0;
            if (b < p.batch) {
                const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
                const int kvb = p.kv_indptr[b], pages = p.kv_indptr[b + 1] - kvb;
                const int P = p.prefix_lens[b], c = q1 - q0;
                const bool ok = q0 >= 0 && c >= 0 && q1 <= p.total_q && P >= 0 && pages >= 0 &&
                                (int64_t)pages * p.page_size >= (int64_t)P + c;
                sp_bad = sp_bad || !ok || (b == p.batch - 1 && q1 != p.total_q);
                if (ok && c > 0 && c <= rmax) {
                    const int lo = p.window > 0 ? max(0, P - p.window + 1) : 0;
                    tl[j] = (P + c - 1) / kRowTile - lo / kRowTile + 1;
                    rw[j] = 1;
                }
                s_sp_seq[b] = make_int4(c, P, kvb, q0);
            }
            t_run += tl[j];
            g_run += rw[j];
        }
        // exclusive scans over the threads: warp shuffles, then the warps
        long long ti = t_run, gi = g_run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long a = __shfl_up_sync(0xffffffffu, ti, o);
            const long long c = __shfl_up_sync(0xffffffffu, gi, o);
            if (lane >= o) {
                ti += a;
                gi += c;
            }
        }
        if (lane == 31) {
            s_sp_wsum[0][warp] = ti;
            s_sp_wsum[1][warp] = gi;
        }
        __syncthreads();
        long long tb = 0, gb = 0;
        for (int w = 0; w < kRowThreads / 32; ++w) {
            if (w < warp) {
                tb += s_sp_wsum[0][w];
                gb += s_sp_wsum[1][w];
            }
            sp_total += s_sp_wsum[0][w];
            sp_groups += s_sp_wsum[1][w];
        }
        tb += ti - t_run;
        gb += gi - g_run;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = 4 * tid + j;
            if (b <= p.batch) {  // entry `batch` holds the totals
                s_sp_ts[b] = (int)min(tb, (long long)INT32_MAX);
                s_sp_gs[b] = (int)gb;
            }
            tb += tl[j];
            gb += rw[j];
        }
        __syncthreads();
    }
    pdl_wait();  // the work list is the planner's output (or, self-planned,
                 // the workspace may still be read by the kernel before)
    pdl_launch_dependents();
    const WsHeader* hdr = reinterpret_cast<const WsHeader*>(p.ws + p.lay.header);
    const int4* rg = reinterpret_cast<const int4*>(p.ws + p.lay.row_groups);
    float* part_o = reinterpret_cast<float*>(p.ws + p.lay.partial_o);
    float2* part_ml = reinterpret_cast<float2*>(p.ws + p.lay.partial_ml);
    const int G = p.group;
    const float sl2 = p.scale_log2;
    const uint32_t sStage = base + C::kOffStage;
    const uint32_t sQ = base + C::kOffQ;
    const uint32_t sBar = base + C::kOffBar;
    auto full_bar = [&](int s) { return sBar + 8u * (uint32_t)s; };
    auto empty_bar = [&](int s) { return sBar + 8u * (uint32_t)(S + s); };
    auto item_full = [&](int s) { return sBar + 8u * (uint32_t)(2 * S + s); };
    auto item_empty = [&](int s) { return sBar + 8u * (uint32_t)(2 * S + NI + s); };
    volatile int* abort_flag = &s_abort;
    // the four consumer warps only (named barrier 1)
    auto consumer_sync = [] { asm volatile("bar.sync 1, 128;" ::: "memory"); };

    // This CTA streams row tiles [x0, x1) of the T tiles of all row groups
    // laid end to end: the same amount of K/V for every CTA.  Each row group
    // it meets (from row_first[blockIdx.x] on) is one item; the load warp
    // resolves the next item and reads its first page ids during this one.
    int T;
    if (p.self_plan) {
        if (sp_bad) report_error(p.dev_err, PCP_ERR_INVALID_ARG);
        // the tile line holds every group's virtual start tiles too
        const long long t_all = (sp_total + (long long)kRowGroupStartTiles * sp_groups) * H;
        if (t_all >= (1ll << 31)) {
            if (tid == 0 && blockIdx.x == 0) report_error(p.dev_err, PCP_ERR_UNSUPPORTED);
            return;
        }
        T = (int)t_all;
    } else {
        T = hdr->row_tiles;
        if (hdr->row_ctas != (int)gridDim.x) {  // the plan was made for another grid
            if (tid == 0 && T > 0) report_error(p.dev_err, PCP_ERR_INVALID_ARG);
            return;
        }
    }
    const int n_use = row_ctas_used(gridDim.x, T);
    // the row-kernel CTA holding tile x: the last i with i*T/n_use <= x
    auto cta_of = [&](int x) { return (int)((((int64_t)x + 1) * n_use + T - 1) / T) - 1; };
    // self-planned calls: where sequence b's groups start on the tile line
    // (each group: kRowGroupStartTiles virtual tiles, then its real ones)
    auto sp_line = [&](int b) { return H * (s_sp_ts[b] + kRowGroupStartTiles * s_sp_gs[b]); };
    if (p.self_plan) {
        // the combine kernel's descriptor of every (sequence, KV head) group,
        // {first partial slot, splits, qo_indptr[b], chunk_len}, zeros for a
        // sequence without decode-shaped rows: the entries are spread over
        // all CTAs of the grid
        int4* gdesc = reinterpret_cast<int4*>(p.ws + p.lay.group_desc);
        for (int64_t e = (int64_t)blockIdx.x * kRowThreads + tid; e < (int64_t)p.batch * H;
             e += (int64_t)gridDim.x * kRowThreads) {
            const int b = (int)(e / H), g = (int)(e - (int64_t)b * H);
            const int tiles = s_sp_ts[b + 1] - s_sp_ts[b];
            int4 gd = make_int4(0, 0, 0, 0);
            if (tiles > 0) {
                const int4 sq = s_sp_seq[b];
                const int k = H * s_sp_gs[b] + g;
                const int R0 = sp_line(b) + g * (tiles + kRowGroupStartTiles) + kRowGroupStartTiles;
                const int i0 = cta_of(R0), i1 = cta_of(R0 + tiles - 1);
                gd = make_int4(k + i0, i1 - i0 + 1, sq.w, sq.x);
            }
            gdesc[e] = gd;
        }
    }
    if ((int)blockIdx.x >= n_use) return;
    const int x0 = row_tile_begin(blockIdx.x, n_use, T);
    const int x1 = row_tile_begin(blockIdx.x + 1, n_use, T);
    if (tid == 0) {
        const uint32_t full_count = p.box_rows > 0 ? 1u : 32u;
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), full_count);
            mbar_init(empty_bar(s), 4);
        }
        for (int s = 0; s < NI; ++s) {
            mbar_init(item_full(s), 33);  // 32 lanes' Q copies + the descriptor
            mbar_init(item_empty(s), 4);
        }
        mbar_init(smem_addr(&s_stall), 1);
        fence_mbarrier_init();
        s_abort = 0;
        s_zero = 0;
    }
    __syncthreads();

    if (warp == 4) {
        // ==================================================== load warp
        const int ps = p.page_size;
        // box geometry: nsub page runs of br = 2^box_shift rows per tile
        const int nsub_shift = 7 - p.box_shift;  // kRowTile = 128 = 2^7
        const int nsub = 1 << nsub_shift;
        // page-table entry of key (a shift for power-of-two page sizes)
        auto entry_of = [&](int key) { return p.page_shift >= 0 ? key >> p.page_shift : key / ps; };
        // slot (TMA: first slot of this lane's page run; gather: slots of
        // rows lane + 32k) of tile t of a sequence with page list `pages`
        auto fetch = [&](const int32_t* pages, int L, int t, int (&sl)[4]) {
#pragma unroll
            for (int k = 0; k < 4; ++k) sl[k] = -1;
            if (p.box_rows > 0) {
                const int key = t * kRowTile + ((lane & (nsub - 1)) << p.box_shift);
                sl[0] = p.num_slots;
                if (lane < nsub * C::kHalves && key < L) {
                    const int e = entry_of(key);
                    const int page = pages[e];
                    if (page >= 0 && page < p.num_pages)
                        sl[0] = page * ps + (key - e * ps);
                    else
                        report_error(p.dev_err, PCP_ERR_BAD_INDEX);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int key = t * kRowTile + lane + 32 * k;
                    if (key < L) {
                        const int e = entry_of(key);
                        const int page = pages[e];
                        if (page >= 0 && page < p.num_pages)
                            sl[k] = page * ps + (key - e * ps);
                        else
                            report_error(p.dev_err, PCP_ERR_BAD_INDEX);
                    }
                }
            }
        };
        // the piece of row group kg = {A, B, C} that lies in [x0, x1) as a
        // row item {b, g, split, n_splits}, {kv_begin, kv_end, first partial
        // slot, q0}, {chunk_len, prefix_len, kv_indptr[b], kv_len}; its split
        // index is blockIdx.x - (first CTA of the group) = blockIdx.x + kg - slot
        // row group kg's descriptor (planner layout): {b, g, S_k, tiles_k},
        // {first key, qo_indptr[b], first partial slot, n_splits},
        // {chunk_len, prefix_len, kv_indptr[b], kv_len}; self-planned calls
        // build it from the shared-memory sums
        auto group = [&](int kg, int4& A, int4& B, int4& Cg) {
            if (!p.self_plan) {
                A = rg[3 * kg];
                B = rg[3 * kg + 1];
                Cg = rg[3 * kg + 2];
                return;
            }
            const int j = kg / H, g = kg - j * H;
            int lo = 0, hi = p.batch;  // the sequence of row group j: last b with gs[b] <= j
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_sp_gs[mid] <= j) lo = mid;
                else hi = mid;
            }
            const int b = lo;
            const int4 sq = s_sp_seq[b];
            const int tiles = s_sp_ts[b + 1] - s_sp_ts[b];
            const int R0 = sp_line(b) + g * (tiles + kRowGroupStartTiles) + kRowGroupStartTiles;
            const int i0 = cta_of(R0), i1 = cta_of(R0 + tiles - 1);
            A = make_int4(b, g, R0, tiles);
            B = make_int4(p.window > 0 ? max(0, sq.y - p.window + 1) : 0, sq.w, kg + i0,
                          i1 - i0 + 1);
            Cg = make_int4(sq.x, sq.y, sq.z, sq.x + sq.y);
        };
        // the first row group with real tiles in [x, x1) (self-planned
        // calls): the group whose span holds tile x, unless x lies among its
        // virtual tiles and its real ones start at or past x1 (-1: none)
        auto group_at = [&](int x) {
            int lo = 0, hi = p.batch;  // last b with sp_line(b) <= x
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (sp_line(mid) <= x) lo = mid;
                else hi = mid;
            }
            const int span = s_sp_ts[lo + 1] - s_sp_ts[lo] + kRowGroupStartTiles;
            const int g = (x - sp_line(lo)) / span;
            const int real0 = sp_line(lo) + g * span + kRowGroupStartTiles;
            if (x < real0 && real0 >= x1) return -1;
            return H * s_sp_gs[lo] + g;
        };
        auto resolve = [&](int kg, int4 A, int4 B, int4 Cg, int4& e0, int4& e1, int4& e2) {
            const int a = max(x0, A.z) - A.z, e = min(x1, A.z + A.w) - A.z;
            const int t0 = B.x / kRowTile;
            e0 = make_int4(A.x, A.y, (int)blockIdx.x + kg - B.z, B.w);
            e1 = make_int4(max(B.x, (t0 + a) * kRowTile), min(Cg.w, (t0 + e) * kRowTile), B.z,
                           B.y);
            e2 = Cg;
        };
        uint32_t it = 0;  // ring position
        int last_issued = -1;
        int last_item = -1;  // last item (or end marker) handed to the consumers
        int kg = p.self_plan ? group_at(x0)
                             : reinterpret_cast<const int*>(p.ws + p.lay.row_first)[blockIdx.x];
        bool have = kg >= 0;  // n0..n2 hold an item (a CTA of virtual tiles only has none)
        int4 gA = make_int4(0, 0, 0, 0), gB = gA, gC = gA;
        int4 n0 = gA, n1 = gA, n2 = gA;
        int next_sl[4] = {-1, -1, -1, -1};
        if (have) {
            group(kg, gA, gB, gC);
            resolve(kg, gA, gB, gC, n0, n1, n2);
            fetch(p.kv_indices + n2.z, n2.w, n1.x / kRowTile, next_sl);
        }
        for (int k = 0;; ++k) {
            const int qs = k % NI;
            // every decision of this warp is taken for all its lanes (the
            // abort flag is read once per warp)
            const bool valid = have && !__any_sync(0xffffffffu, *abort_flag != 0);
            const int4 d0 = n0, d1 = n1, d2 = n2;
            int cur_sl[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) cur_sl[j] = next_sl[j];
            // the range goes on past this group: the next group follows
            // the next group's real tiles start after its virtual ones
            const bool next_valid = valid && gA.z + gA.w + kRowGroupStartTiles < x1;
            if (next_valid) {  // loads in flight during this item
                ++kg;
                group(kg, gA, gB, gC);
            }
            // hand the item (or the end marker) and its Q rows to the consumers
            if (!__all_sync(0xffffffffu, mbar_wait(item_empty(qs), ((uint32_t)(k / NI) & 1u) ^ 1u,
                                                   abort_flag, p.dev_err, kSpinLimitNs)))
                break;
            const int g = d0.y;
            if (valid) {
                const int R = d2.x * G;
                const uint32_t qd = sQ + qs * kRowMaxRows * C::kQStride;
                for (int idx = lane; idx < kRowMaxRows * (D / 8); idx += 32) {
                    const int r = idx / (D / 8), cc = idx % (D / 8);
                    const bool ok = r < R;
                    const uint16_t* src =
                        ok ? p.q + ((int64_t)(d1.w + r / G) * p.n_q_heads + g * G + r % G) * D + cc * 8
                           : p.q;
                    cp_async_16(qd + r * C::kQStride + cc * 16, src, ok ? 16u : 0u);
                }
            }
            cp_async_mbar_arrive_noinc(item_full(qs));
            if (lane == 0) {
                s_desc[qs * 3 + 0] = valid ? d0 : make_int4(-1, 0, 0, 0);
                s_desc[qs * 3 + 1] = d1;
                s_desc[qs * 3 + 2] = d2;
                mbar_arrive(item_full(qs));
            }
            last_item = k;
            if (!valid) break;
            const int kb = d1.x, ke = d1.y, L = d2.w;
            const int32_t* pages = p.kv_indices + d2.z;
            const int t_first = kb / kRowTile, t_last = (ke - 1) / kRowTile;
            const int ntiles = t_last - t_first + 1;
            for (int i = 0; i < ntiles; ++i) {
                const int t = t_first + i;
                const uint32_t itp = it + i;
                const int st = itp % S;
                int nsl[4];
                if (i + 1 < ntiles) fetch(pages, L, t + 1, nsl);
                if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(st), ((itp / S) & 1u) ^ 1u,
                                                       abort_flag, p.dev_err, kSpinLimitNs)))
                    break;
                const uint32_t kd = sStage + st * 2 * C::kTileBytes;
                const uint32_t vd = kd + C::kTileBytes;
                if (p.box_rows > 0) {
                    const int br = p.box_rows, nloads = nsub * C::kHalves;
                    const int key0 = t * kRowTile;
                    // the V page run holding the sequence end is zero-filled past it
                    int strad = -1;
                    if (L > key0 && L < key0 + kRowTile && ((L - key0) & (br - 1)) != 0)
                        strad = (L - key0) >> p.box_shift;
                    if (strad >= 0) {
                        const int slot0 = __shfl_sync(0xffffffffu, cur_sl[0], strad);
                        const bool bad = slot0 >= p.num_slots;
                        const int ks = key0 + strad * br;
                        for (int idx = lane; idx < br * C::kHalves * 8; idx += 32) {
                            const int row = idx / (C::kHalves * 8), cc = idx % (C::kHalves * 8);
                            const int rt = strad * br + row;
                            const bool ok = !bad && ks + row < L;
                            const uint16_t* src =
                                ok ? p.v_pool + ((int64_t)(slot0 + row) * p.n_kv_heads + g) * D + cc * 8
                                   : p.v_pool;
                            cp_async_16(vd + swz<D>(rt, cc * 8), src, ok ? 16u : 0u);
                        }
                        cp_async_mbar_arrive(full_bar(st));
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_expect_tx(
                            full_bar(st),
                            (uint32_t)(2 * nloads - (strad >= 0 ? C::kHalves : 0)) * br * 128);
                    __syncwarp();
                    if (lane < nloads) {
                        const int sb = lane & (nsub - 1), h = lane >> nsub_shift;
                        tma_load_3d(kd + h * C::kHalfBytes + sb * br * 128, &tm_k, full_bar(st),
                                    h * 64, g, cur_sl[0]);
                        if (sb != strad)
                            tma_load_3d(vd + h * C::kHalfBytes + sb * br * 128, &tm_v,
                                        full_bar(st), h * 64, g, cur_sl[0]);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int row = lane + 32 * j;
                        const bool ok = cur_sl[j] >= 0;
                        const int64_t off = ((int64_t)(ok ? cur_sl[j] : 0) * p.n_kv_heads + g) * D;
#pragma unroll
                        for (int cc = 0; cc < C::kHalves * 8; ++cc) {
                            cp_async_16(kd + swz<D>(row, cc * 8), p.k_pool + off + cc * 8, ok ? 16u : 0u);
                            cp_async_16(vd + swz<D>(row, cc * 8), p.v_pool + off + cc * 8, ok ? 16u : 0u);
                        }
                    }
                    cp_async_mbar_arrive_noinc(full_bar(st));
                }
                last_issued = (int)itp;
                if (i == 0 && next_valid) {  // the next item and its first page ids
                    resolve(kg, gA, gB, gC, n0, n1, n2);
                    fetch(p.kv_indices + n2.z, n2.w, n1.x / kRowTile, next_sl);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i + 1 < ntiles) cur_sl[j] = nsl[j];
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            it += (uint32_t)ntiles;
            have = next_valid;
        }
        // nothing may still be landing in shared memory when the CTA exits
        cp_async_wait_all();
        if (*abort_flag && lane == 0) {
            // the copies of the last tiles and of the last item's Q rows (and
            // the mbarrier arrivals they trigger) land before the CTA exits;
            // these waits watch s_zero, never raised, and run to their limit
            volatile int* no_abort = &s_zero;
            for (int j = last_issued - S + 1; j <= last_issued; ++j)
                if (j >= 0)
                    mbar_wait(full_bar(j % S), ((uint32_t)j / S) & 1u, no_abort, p.dev_err,
                              kSpinLimitNs);
            if (last_item >= 0)
                mbar_wait(item_full(last_item % NI), ((uint32_t)(last_item / NI)) & 1u, no_abort,
                          p.dev_err, kSpinLimitNs);
        }
        return;
    }

    // ======================================================== consumer warps
    // The four consumer warps meet at named barriers, so they leave the item
    // loop together: each warp posts its state at a decision point and all of
    // them read every post after the barrier.  (A wait gives up for the whole
    // warp at once.)
    uint32_t it = 0;
    bool failed = false;  // this warp gave up a wait
    for (int k = 0;; ++k) {
        const int qs = k % NI;
        // 0: an item, 1: the end marker, 2: the wait gave up
        int post = 2;
        // the timeout test: the consumers' first wait is one nothing ends
        if (k == 0 && p.stall_ns != 0 &&
            !__all_sync(0xffffffffu,
                        mbar_wait(smem_addr(&s_stall), 0u, abort_flag, p.dev_err, p.stall_ns)))
            failed = true;
        if (!failed &&
            __all_sync(0xffffffffu, mbar_wait(item_full(qs), (uint32_t)(k / NI) & 1u, abort_flag,
                                              p.dev_err, kSpinLimitNs)))
            post = s_desc[qs * 3 + 0].x < 0 ? 1 : 0;
        if (lane == 0) s_post[warp] = post;
        consumer_sync();
        if (s_post[0] | s_post[1] | s_post[2] | s_post[3]) break;
        const int4 d0 = s_desc[qs * 3 + 0];
        const int4 d1 = s_desc[qs * 3 + 1];
        const int4 d2 = s_desc[qs * 3 + 2];
        const int g = d0.y, split = d0.z, nsplit = d0.w;
        const int kb = d1.x, ke = d1.y, first_item = d1.z, q0 = d1.w;
        const int P = d2.y;
        const int R = d2.x * G;
        const int t_first = kb / kRowTile, t_last = (ke - 1) / kRowTile;
        const int ntiles = t_last - t_first + 1;

        // Q as the A operand (rows gid and gid + 8, 16 dims per k-step), from
        // the item slot; rows >= R were zero-filled
        const int row_lo = gid, row_hi = gid + 8;
        uint32_t qa[D / 16][4];
        {
            const uint32_t qb = sQ + qs * kRowMaxRows * C::kQStride;
            const int qrow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ldsm_x4(qb + qrow * C::kQStride + (kk * 16 + (lane >> 4) * 8) * 2, qa[kk][0],
                        qa[kk][1], qa[kk][2], qa[kk][3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(item_empty(qs));
        const int pos_lo = P + row_lo / G, pos_hi = P + row_hi / G;
        const int L = d2.w;
        // rows of the boolean mask for this lane's two query rows (null: the
        // row is past the mask and sees nothing, or there is no such row)
        const uint8_t* mrow_lo = nullptr;
        const uint8_t* mrow_hi = nullptr;
        if constexpr (kMask) {
            const int b = d0.x;
            auto mrow = [&](int row) -> const uint8_t* {
                const int qi = row / G;
                if (row >= R || (p.mask.q_stride != 0 && qi >= p.mask.q_len)) return nullptr;
                return p.mask.data + (int64_t)b * p.mask.b_stride +
                       (int64_t)(g * G + row % G) * p.mask.h_stride +
                       (int64_t)qi * p.mask.q_stride;
            };
            mrow_lo = mrow(row_lo);
            mrow_hi = mrow(row_hi);
        }
        float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
        float o[D / 8][4];
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
            for (int j = 0; j < 4; ++j) o[dn][j] = 0.f;

        for (int i = 0; i < ntiles; ++i) {
            const int t = t_first + i;
            const uint32_t itp = it + i;
            const int st = itp % S;
            if (!__all_sync(0xffffffffu, mbar_wait(full_bar(st), (itp / S) & 1u, abort_flag,
                                                   p.dev_err, kSpinLimitNs))) {
                failed = true;
                break;
            }
                const uint32_t kbase = sStage + st * 2 * C::kTileBytes;
                const uint32_t vbase = kbase + C::kTileBytes;
                const int key_w = t * kRowTile + warp * 32;

                // S = Q K^T for this warp's 32 keys: [block of 16 keys][n8 half][4]
                float sc[2][2][4];
#pragma unroll
                for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                        for (int j = 0; j < 4; ++j) sc[bl][nb][j] = 0.f;
#pragma unroll
                for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int krow = warp * 32 + bl * 16 + (lane >> 4) * 8 + (lane & 7);
                        const int dcol = kk * 16 + ((lane >> 3) & 1) * 8;
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(kbase + swz<D>(krow, dcol), b0, b1, b2, b3);
                        mma_16816(sc[bl][0], qa[kk], b0, b1);
                        mma_16816(sc[bl][1], qa[kk], b2, b3);
                    }
                // mask and scale; element j: row lo (j < 2) or hi, key = ... + 2 * tig + (j & 1)
                float mx_lo = -INFINITY, mx_hi = -INFINITY;
                // every row of the item sees all 32 keys of this warp (the
                // interior of a long KV range): scale only.  Rows past R hold
                // zero queries; their results are never read.
                bool all_vis = !kMask && key_w >= kb && key_w + 32 <= ke;
                if (p.causal)
                    all_vis = all_vis && key_w + 31 <= P &&
                              (p.window <= 0 || key_w > P + d2.x - 1 - p.window);
                else
                    all_vis = all_vis && key_w + 32 <= L;
                if (all_vis) {
#pragma unroll
                    for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float v = sc[bl][nb][j] * sl2;
                                sc[bl][nb][j] = v;
                                if (j < 2) mx_lo = fmaxf(mx_lo, v);
                                else mx_hi = fmaxf(mx_hi, v);
                            }
                } else {
#pragma unroll
                for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int key = key_w + bl * 16 + nb * 8 + tig * 2 + (j & 1);
                            const int pos = j < 2 ? pos_lo : pos_hi;
                            const int row = j < 2 ? row_lo : row_hi;
                            bool vis = row < R && key >= kb && key < ke &&
                                       (p.causal ? key <= pos &&
                                                       (p.window <= 0 || key > pos - p.window)
                                                 : key < L);
                            if constexpr (kMask) {
                                const uint8_t* mr = j < 2 ? mrow_lo : mrow_hi;
                                vis = vis && mr != nullptr && key < p.mask.kv_len && mr[key] != 0;
                            }
                            const float v = vis ? sc[bl][nb][j] * sl2 : -INFINITY;
                            sc[bl][nb][j] = v;
                            if (j < 2) mx_lo = fmaxf(mx_lo, v);
                            else mx_hi = fmaxf(mx_hi, v);
                        }
                }
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
                mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
                mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
                const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
                const float a_lo = mn_lo == -INFINITY ? 1.f : fast_exp2(m_lo - mn_lo);
                const float a_hi = mn_hi == -INFINITY ? 1.f : fast_exp2(m_hi - mn_hi);
                const float r_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
                const float r_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
                m_lo = mn_lo;
                m_hi = mn_hi;
                float s_lo = 0.f, s_hi = 0.f;
                uint32_t pa[2][4];
#pragma unroll
                for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                    for (int nb = 0; nb < 2; ++nb) {
                        const float e0 = fast_exp2(sc[bl][nb][0] - r_lo);
                        const float e1 = fast_exp2(sc[bl][nb][1] - r_lo);
                        const float e2 = fast_exp2(sc[bl][nb][2] - r_hi);
                        const float e3 = fast_exp2(sc[bl][nb][3] - r_hi);
                        s_lo += e0 + e1;
                        s_hi += e2 + e3;
                        pa[bl][nb * 2 + 0] = pack_bf16x2(e0, e1);
                        pa[bl][nb * 2 + 1] = pack_bf16x2(e2, e3);
                    }
                l_lo = l_lo * a_lo + s_lo;
                l_hi = l_hi * a_hi + s_hi;
                // O is rescaled only when some row's running max moved
                if (__any_sync(0xffffffffu, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
                    for (int dn = 0; dn < D / 8; ++dn) {
                        o[dn][0] *= a_lo;
                        o[dn][1] *= a_lo;
                        o[dn][2] *= a_hi;
                        o[dn][3] *= a_hi;
                    }
                }
                // O += P V; V fragments for two 8-wide column chunks per ldmatrix.trans
#pragma unroll
                for (int bl = 0; bl < 2; ++bl)
#pragma unroll
                    for (int dn2 = 0; dn2 < D / 16; ++dn2) {
                        const int vrow = warp * 32 + bl * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
                        const int dcol = (dn2 * 2 + (lane >> 4)) * 8;
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_trans(vbase + swz<D>(vrow, dcol), v0, v1, v2, v3);
                        mma_16816(o[2 * dn2], pa[bl], v0, v1);
                        mma_16816(o[2 * dn2 + 1], pa[bl], v2, v3);
                    }
            // every tile's stage goes back to the load warp as soon as its
            // PV is done (the merge below does not use the stages)
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(st));
        }
        it += (uint32_t)ntiles;
        if (lane == 0) s_fail[warp] = failed ? 1 : 0;

        // Merge the four warps' states (each holds its 32 keys of every tile):
        // (m, l) per row through m_s / l_s, then, four rows at a time, every
        // warp leaves its O rows in its slice of the merge buffer and the
        // threads sum the four slices element by element (warps in a fixed
        // order, so the rounding does not depend on timing).  All stages are
        // back with the load warp, which keeps streaming the next item.
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        if (tig == 0) {
            m_s[warp * kRowMaxRows + row_lo] = m_lo;
            m_s[warp * kRowMaxRows + row_hi] = m_hi;
            l_s[warp * kRowMaxRows + row_lo] = l_lo;
            l_s[warp * kRowMaxRows + row_hi] = l_hi;
        }
        consumer_sync();
        if (s_fail[0] | s_fail[1] | s_fail[2] | s_fail[3]) break;
        float* mbuf = reinterpret_cast<float*>(sm + C::kOffMerge);
        constexpr int MR = C::kMergeRows;
        for (int r0 = 0; r0 < R; r0 += MR) {
            if (row_lo >= r0 && row_lo < r0 + MR) {
                float* dst = mbuf + (warp * MR + row_lo - r0) * C::kMergeStride + tig * 2;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn)
                    *reinterpret_cast<float2*>(dst + dn * 8) = make_float2(o[dn][0], o[dn][1]);
            }
            if (row_hi >= r0 && row_hi < r0 + MR) {
                float* dst = mbuf + (warp * MR + row_hi - r0) * C::kMergeStride + tig * 2;
#pragma unroll
                for (int dn = 0; dn < D / 8; ++dn)
                    *reinterpret_cast<float2*>(dst + dn * 8) = make_float2(o[dn][2], o[dn][3]);
            }
            consumer_sync();
            for (int idx = tid; idx < MR * D; idx += kConsumerThreads) {
                const int r = r0 + idx / D, d = idx % D;
                if (r >= R) continue;
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * kRowMaxRows + r]);
                float acc = 0.f, lsum = 0.f;
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float mw = m_s[w * kRowMaxRows + r];
                        const float e = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
                        acc += e * mbuf[(w * MR + r - r0) * C::kMergeStride + d];
                        lsum += e * l_s[w * kRowMaxRows + r];
                    }
                }
                const int64_t orow = (int64_t)(q0 + r / G) * p.n_q_heads + g * G + r % G;
                if (nsplit == 1) {
                    const float v = lsum > 0.f ? acc / lsum : 0.f;
                    p.out[orow * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                    if (d == 0 && p.lse != nullptr)
                        p.lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * 0.69314718055994531f
                                                 : -INFINITY;
                } else {
                    part_o[((int64_t)(first_item + split) * kRowMaxRows + r) * D + d] = acc;
                    if (d == 0)
                        part_ml[(int64_t)(first_item + split) * kRowMaxRows + r] =
                            make_float2(M, lsum);
                }
            }
            consumer_sync();  // the buffer is free for the next rows (or item)
        }
    }
}

// Merge the split-KV partials of one (sequence, KV head) group: one CTA per
// group, out[row, h, :] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s and
// lse = (M + log2 L) ln 2, with M the largest split maximum (log2 units).
// Each thread computes whole output elements: after the group descriptor it
// issues the loads of all its elements' partials ((m, l) and o of every
// split, eight splits at a time with a running maximum) at once, so the
// kernel costs two dependent memory round trips and no block barrier.
template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ CombineParams p) {
    constexpr int kBatch = 8;  // splits whose loads are in flight together
    pdl_wait();
    pdl_launch_dependents();
    const int4 gd = reinterpret_cast<const int4*>(p.ws + p.lay.group_desc)[blockIdx.x];
    const int base = gd.x, ns = gd.y, q0 = gd.z;
    if (ns <= 1) return;
    const int g = blockIdx.x % p.n_kv_heads;
    const int G = p.group;
    const int R = gd.w * G;
    const float* part_o = reinterpret_cast<const float*>(p.ws + p.lay.partial_o);
    const float2* part_ml = reinterpret_cast<const float2*>(p.ws + p.lay.partial_ml);
    for (int idx = threadIdx.x; idx < R * D; idx += blockDim.x) {
        const int r = idx / D, d = idx % D;
        float M = -INFINITY, L = 0.f, acc = 0.f;
        for (int s0 = 0; s0 < ns; s0 += kBatch) {
            float2 ml[kBatch];
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int sp = s0 + j;
                const int64_t slot = (int64_t)(base + sp) * kRowMaxRows + r;
                ml[j] = sp < ns ? part_ml[slot] : make_float2(-INFINITY, 0.f);
                v[j] = sp < ns ? part_o[slot * D + d] : 0.f;
            }
            float Mb = M;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) Mb = fmaxf(Mb, ml[j].x);
            if (Mb == -INFINITY) continue;
            const float a = M == -INFINITY ? 0.f : fast_exp2(M - Mb);
            L *= a;
            acc *= a;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const float e = ml[j].x == -INFINITY ? 0.f : fast_exp2(ml[j].x - Mb);
                L += e * ml[j].y;
                acc += e * v[j];
            }
            M = Mb;
        }
        const int64_t orow = (int64_t)(q0 + r / G) * p.n_q_heads + g * G + r % G;
        p.out[orow * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(L > 0.f ? acc / L : 0.f));
        if (d == 0 && p.lse != nullptr)
            p.lse[orow] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
}

cudaError_t launch_combine(int head_dim, cudaStream_t stream, const CombineParams& p) {
    if (p.n_groups <= 0) return cudaSuccess;
    if (head_dim == 128)
        return launch_pdl(combine_kernel<128>, dim3(p.n_groups), dim3(256), 0, stream, p);
    return launch_pdl(combine_kernel<64>, dim3(p.n_groups), dim3(256), 0, stream, p);
}

size_t row_smem_bytes(int head_dim) {
    return head_dim == 128 ? RowCfg<128>::kSmemBytes : RowCfg<64>::kSmemBytes;
}

template <int D, bool kMask>
cudaError_t launch_rows_t(int grid, cudaStream_t stream, const RowParams& p,
                          const CUtensorMap& tk, const CUtensorMap& tv) {
    const size_t smem = RowCfg<D>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(row_attn_kernel<D, kMask>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(row_attn_kernel<D, kMask>, dim3(grid), dim3(kRowThreads), smem, stream, p,
                      tk, tv);
}

cudaError_t launch_rows(int head_dim, int grid, cudaStream_t stream, const RowParams& p,
                        const CUtensorMap& tk, const CUtensorMap& tv) {
    const bool mask = p.mask.data != nullptr;
    if (head_dim == 128)
        return mask ? launch_rows_t<128, true>(grid, stream, p, tk, tv)
                    : launch_rows_t<128, false>(grid, stream, p, tk, tv);
    return mask ? launch_rows_t<64, true>(grid, stream, p, tk, tv)
                : launch_rows_t<64, false>(grid, stream, p, tk, tv);
}

}  // namespace pcp
