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
//    for the persistent kernel's dynamic scheduler -- with a counting sort.
//  * row items for decode-shaped chunks (chunk_len * G <= 16 rows): the KV
//    range of each (sequence, KV head) is split into pieces of
//    `tiles_per_split` 128-key tiles, chosen so the whole call has about
//    three items per SM, and ordered longest first like the tensor-core
//    items.  Each split owns a partial slot (the group's first slot + split
//    index) for the log-sum-exp combine.  This is the split-KV idea of the
//    AstrAI paged decode kernel (split count from the SM count, partials
//    merged by a combine step).
#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

struct SeqInfo {
    int c, P, L;
    bool ok;
};

__device__ __forceinline__ SeqInfo seq_info(const PlanParams& p, int b) {
    SeqInfo s;
    const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
    s.c = q1 - q0;
    s.P = p.prefix_lens[b];
    s.L = s.P + s.c;
    const int pages = p.kv_indptr[b + 1] - p.kv_indptr[b];
    s.ok = q0 >= 0 && s.c >= 0 && q1 <= p.total_q && s.P >= 0 && pages >= 0 &&
           (int64_t)pages * p.page_size >= (int64_t)s.L;
    return s;
}

// First visible key of absolute position `pos`.
__device__ __forceinline__ int first_key(int pos, int window) {
    return window > 0 ? max(0, pos - window + 1) : 0;
}

__device__ __forceinline__ int tc_cost(int P, int c, int k, int item_pos, int window) {
    const int first = P + k * item_pos;
    const int last = P + min((k + 1) * item_pos, c) - 1;
    return last / kTileN - first_key(first, window) / kTileN + 1;
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

}  // namespace

__global__ void __launch_bounds__(1024, 1) plan_kernel(const __grid_constant__ PlanParams p) {
    __shared__ int hist[1024];
    __shared__ int hist_r[1024];
    __shared__ int warp_sums[64];
    __shared__ unsigned long long s_row_tiles;
    __shared__ int s_rows;
    __shared__ int s_tps;
    __shared__ int4 s_seq[1024];  // {c, P, ok} of the first 1024 sequences

    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
    int4* tc = reinterpret_cast<int4*>(p.ws + p.lay.tc_items);
    int4* rows = reinterpret_cast<int4*>(p.ws + p.lay.row_items);
    int* gcnt = reinterpret_cast<int*>(p.ws + p.lay.group_cnt);
    const int tid = threadIdx.x, nt = blockDim.x;
    const int item_pos = q_positions_per_tile(p.group) * kQTiles;
    const int rmax = row_path_max_chunk(p.group);
    const int H = p.n_kv_heads;

    for (int i = tid; i < 1024; i += nt) hist[i] = hist_r[i] = 0;
    // the metadata is read from global memory once; later passes use shared memory
    for (int b = tid; b < min(p.batch, 1024); b += nt) {
        const SeqInfo q = seq_info(p, b);
        s_seq[b] = make_int4(q.c, q.P, q.ok ? 1 : 0, 0);
    }
    auto get_seq = [&](int b) {
        if (b >= 1024) return seq_info(p, b);
        const int4 v = s_seq[b];
        SeqInfo q;
        q.c = v.x;
        q.P = v.y;
        q.L = v.x + v.y;
        q.ok = v.z != 0;
        return q;
    };
    for (int64_t i = tid; i < (int64_t)p.batch * H; i += nt) gcnt[i] = 0;
    if (tid == 0) {
        s_row_tiles = 0;
        s_rows = 0;
        if (p.batch > 0 && p.qo_indptr[p.batch] != p.total_q)
            report_error(p.dev_err, PCP_ERR_INVALID_ARG);
    }
    __syncthreads();

    // pass 1: validate, histogram of tensor-core costs, total row-path tiles
    for (int b = tid; b < p.batch; b += nt) {
        const SeqInfo s = get_seq(b);
        if (!s.ok) {
            report_error(p.dev_err, PCP_ERR_INVALID_ARG);
            continue;
        }
        if (s.c == 0) continue;
        if (s.c <= rmax) {
            const int tiles = (s.L - 1) / kRowTile - first_key(s.P, p.window) / kRowTile + 1;
            atomicAdd(&s_row_tiles, (unsigned long long)tiles * H);
        } else {
            const int n = (s.c + item_pos - 1) / item_pos;
            for (int k = 0; k < n; ++k)
                atomicAdd(&hist[min(tc_cost(s.P, s.c, k, item_pos, p.window), 1023)], H);
        }
    }
    __syncthreads();

    // descending exclusive offsets of the cost histogram
    const int n_tc = desc_offsets(hist, warp_sums);
    if (tid == 0) {
        const unsigned long long tot = s_row_tiles;
        const int target = min(3 * max(p.sm_count, 1), kRowTargetItems);
        unsigned long long tps = (tot + target - 1) / target;
        s_tps = (int)(tps < 1 ? 1 : tps);
    }
    __syncthreads();
    const int tps = s_tps;

    // histogram of row-item lengths (tiles), for longest-first order
    for (int b = tid; b < p.batch; b += nt) {
        const SeqInfo s = get_seq(b);
        if (!s.ok || s.c == 0 || s.c > rmax) continue;
        const int tiles = (s.L - 1) / kRowTile - first_key(s.P, p.window) / kRowTile + 1;
        const int ns = (tiles + tps - 1) / tps;
        if (ns > 1) atomicAdd(&hist_r[min(tps, 1023)], (ns - 1) * H);
        atomicAdd(&hist_r[min(tiles - (ns - 1) * tps, 1023)], H);
    }
    __syncthreads();
    desc_offsets(hist_r, warp_sums);

    // pass 2: scatter tensor-core items, emit row items
    for (int b = tid; b < p.batch; b += nt) {
        const SeqInfo s = get_seq(b);
        if (!s.ok || s.c == 0) continue;
        if (s.c <= rmax) {
            const int lo = first_key(s.P, p.window);
            const int t0 = lo / kRowTile, t1 = (s.L - 1) / kRowTile;
            const int tiles = t1 - t0 + 1;
            const int ns = (tiles + tps - 1) / tps;
            for (int g = 0; g < H; ++g) {
                const int base = atomicAdd(&s_rows, ns);  // the group's partial slots
                for (int sp = 0; sp < ns; ++sp) {
                    const int len = min(tps, tiles - sp * tps);
                    const int it = atomicAdd(&hist_r[min(len, 1023)], 1);
                    if (it >= p.lay.cap_row || base + sp >= p.lay.cap_row) {
                        report_error(p.dev_err, PCP_ERR_WORKSPACE);
                        break;
                    }
                    const int kb = max(lo, (t0 + sp * tps) * kRowTile);
                    const int ke = min(s.L, (t0 + (sp + 1) * tps) * kRowTile);
                    rows[2 * it] = make_int4(b, g, sp, ns);
                    rows[2 * it + 1] = make_int4(kb, ke, base, 0);
                }
            }
        } else {
            const int n = (s.c + item_pos - 1) / item_pos;
            for (int k = 0; k < n; ++k) {
                const int cost = tc_cost(s.P, s.c, k, item_pos, p.window);
                const int slot = atomicAdd(&hist[min(cost, 1023)], H);
                for (int g = 0; g < H; ++g) {
                    if (slot + g >= p.lay.cap_tc) {
                        report_error(p.dev_err, PCP_ERR_WORKSPACE);
                        break;
                    }
                    tc[slot + g] = make_int4(b, g, k * item_pos, cost);
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        hdr->n_tc_items = (int)min((int64_t)n_tc, p.lay.cap_tc);
        hdr->n_row_items = (int)min((int64_t)s_rows, p.lay.cap_row);
        hdr->tc_next = 0;
        hdr->row_next = 0;
        hdr->tiles_per_split = tps;
    }
}

cudaError_t launch_plan(cudaStream_t stream, const PlanParams& p) {
    plan_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pcp
