// The fused slot mapping and KV append of one span of new K/V chunks, shared
// by the stand-alone append kernel and the kernel that runs the append beside
// the planner.
//
// AReno PR #642 ("What does this PR do?", third bullet): prefill continues
// inside the last allocated KV page, so the first new token of a chunk whose
// prefix is not a multiple of the page size lands mid-page.  AstrAI's
// PagePool.bind_tasks builds out_cache_loc once per step and the backend writes
// k_buffer[layer, out_cache_loc] = k before attending.
#pragma once

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

// A thread moves kAppendUnroll 16-byte chunks of K and as many of V, kThreads
// apart; a span is kThreads * kAppendUnroll consecutive chunks of the
// flattened (token, chunk) space.
constexpr int kAppendUnroll = 4;
// qo_indptr is staged in shared memory up to this many sequences.
constexpr int kAppendStagedSeqs = 2048;

template <int kThreads>
struct AppendSmem {
    int qo[kAppendStagedSeqs + 1];
    int64_t slot[kThreads * kAppendUnroll + 1];  // slots of the span's tokens
};

// Slot of new token t from the page table; qo is qo_indptr (staged or
// global).  -1 when the page id is bad or the metadata do not place t.
__device__ __forceinline__ int64_t slot_of_token(const int32_t* qo, int batch, int64_t t,
                                                 const int32_t* __restrict__ kv_indptr,
                                                 const int32_t* __restrict__ kv_indices,
                                                 const int32_t* __restrict__ prefix_lens,
                                                 int page_size, int64_t num_pages) {
    int lo = 0, hi = batch;  // sequence of row t: the last b with qo[b] <= t
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (qo[mid] <= t) lo = mid;
        else hi = mid;
    }
    const int b = lo;
    if (!(t >= qo[b] && t < qo[b + 1])) return -1;
    const int64_t pos = (int64_t)__ldg(prefix_lens + b) + (t - qo[b]);
    const int kb = __ldg(kv_indptr + b);
    const int64_t entry = pos / page_size;
    if (pos < 0 || entry >= (int64_t)__ldg(kv_indptr + b + 1) - kb) return -1;
    const int64_t page = __ldg(kv_indices + kb + entry);
    return (page >= 0 && page < num_pages) ? page * page_size + pos % page_size : -1;
}

// Span `span` of the append, by a block of kThreads threads: every load is
// issued first, the slots of the span's tokens are found meanwhile (one
// thread per token: qo_indptr from shared memory, then prefix_lens, kv_indptr
// and the page id), then the stores go out.  The block holding a token's
// first chunk writes loc[t] when asked and reports a bad slot.
template <int kThreads>
__device__ __forceinline__ void append_paged_span(const AppendParams& a, AppendSmem<kThreads>& S,
                                                  int64_t span) {
    constexpr int kSpan = kThreads * kAppendUnroll;
    const uint4* __restrict__ k = static_cast<const uint4*>(a.k);
    const uint4* __restrict__ v = static_cast<const uint4*>(a.v);
    uint4* __restrict__ k_pool = static_cast<uint4*>(a.k_pool);
    uint4* __restrict__ v_pool = static_cast<uint4*>(a.v_pool);
    const int cpt = a.chunks_per_token;
    const int64_t total = a.total_q * cpt;
    const int64_t c0 = span * kSpan;
    uint4 kr[kAppendUnroll], vr[kAppendUnroll];
#pragma unroll
    for (int j = 0; j < kAppendUnroll; ++j) {
        const int64_t idx = c0 + j * kThreads + threadIdx.x;
        if (idx < total) {
            kr[j] = __ldcs(k + idx);
            vr[j] = __ldcs(v + idx);
        }
    }
    const bool staged = a.batch <= kAppendStagedSeqs;
    if (staged) {
        for (int i = threadIdx.x; i <= a.batch; i += kThreads) S.qo[i] = a.qo_indptr[i];
        __syncthreads();
    }
    const int32_t* qo = staged ? S.qo : a.qo_indptr;
    const int64_t t0 = c0 / cpt;
    const int64_t t1 = (min(total, c0 + kSpan) - 1) / cpt;
    for (int64_t t = t0 + threadIdx.x; t <= t1; t += kThreads) {
        const int64_t s = slot_of_token(qo, a.batch, t, a.kv_indptr, a.kv_indices, a.prefix_lens,
                                        a.page_size, a.num_pages);
        if (t * cpt >= c0) {
            if (s < 0) report_error(a.dev_err, PCP_ERR_BAD_INDEX);
            if (a.loc != nullptr) a.loc[t] = s;
        }
        S.slot[t - t0] = s;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kAppendUnroll; ++j) {
        const int64_t idx = c0 + j * kThreads + threadIdx.x;
        if (idx >= total) continue;
        const int64_t t = idx / cpt;
        const int64_t s = S.slot[t - t0];
        if (s < 0) continue;
        const int64_t ch = idx - t * cpt;
        __stcs(k_pool + s * cpt + ch, kr[j]);
        __stcs(v_pool + s * cpt + ch, vr[j]);
    }
}

}  // namespace pcp
