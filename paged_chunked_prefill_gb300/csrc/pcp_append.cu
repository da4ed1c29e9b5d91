// Slot mapping of a step's new tokens and the KV append (scatter into pages).
//
// AReno PR #642 ("What does this PR do?", third bullet): prefill continues
// inside the last allocated KV page, so the first new token of a chunk whose
// prefix is not a multiple of the page size lands mid-page.  AstrAI's
// PagePool.bind_tasks builds out_cache_loc once per step and the backend writes
// k_buffer[layer, out_cache_loc] = k before attending; here both are kernels.
#include <algorithm>

#include "pcp_append_body.cuh"
#include "pcp_device.cuh"
#include "pcp_internal.h"
#include "pcp_launch.h"

namespace pcp {

__global__ void out_cache_loc_kernel(const int32_t* __restrict__ qo_indptr,
                                     const int32_t* __restrict__ kv_indptr,
                                     const int32_t* __restrict__ kv_indices,
                                     const int32_t* __restrict__ prefix_lens, int batch,
                                     int64_t total_q, int page_size, int64_t num_pages,
                                     int64_t* __restrict__ loc, int32_t* dev_err) {
    // qo_indptr in shared memory (one coalesced read per CTA) when it fits,
    // so the search below costs no global round trips
    constexpr int kStagedSeqs = 2048;
    __shared__ int s_qo[kStagedSeqs + 1];
    pdl_wait();
    pdl_launch_dependents();
    const bool staged = batch <= kStagedSeqs;
    if (staged) {
        for (int i = threadIdx.x; i <= batch; i += blockDim.x) s_qo[i] = qo_indptr[i];
        __syncthreads();
    }
    const int32_t* qo = staged ? s_qo : qo_indptr;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total_q;
         t += (int64_t)gridDim.x * blockDim.x) {
        // sequence owning row t: the last b with qo_indptr[b] <= t
        int lo = 0, hi = batch;  // answer in [lo, hi)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (qo[mid] <= t) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        int64_t out = -1;
        if (t >= qo[b] && t < qo[b + 1]) {
            const int64_t pos = (int64_t)prefix_lens[b] + (t - qo[b]);
            const int64_t entry = pos / page_size;
            if (pos >= 0 && entry < (int64_t)kv_indptr[b + 1] - kv_indptr[b]) {
                const int64_t page = kv_indices[kv_indptr[b] + entry];
                if (page >= 0 && page < num_pages) out = page * page_size + pos % page_size;
            }
        }
        if (out < 0) report_error(dev_err, PCP_ERR_BAD_INDEX);
        loc[t] = out;
    }
}

// Both append kernels move a token row (n_kv_heads * head_dim bf16 values,
// `chunks_per_token` 16-byte chunks) of K and of V.  A block owns a span of
// kAppendSpan consecutive chunks of the flattened (token, chunk) space, each
// thread kAppendUnroll of them, 256 apart: every thread issues all its K/V
// loads first, the slots of the span's tokens are found meanwhile (one
// thread per token, into shared memory), then the stores go out.  One wave
// of such blocks keeps 32 KB in flight per block.
constexpr int kAppendThreads = 256;
constexpr int kAppendSpan = kAppendThreads * kAppendUnroll;

// KV append from precomputed slots: k_pool[loc[t]] = k[t], v_pool[loc[t]] = v[t].
__global__ void __launch_bounds__(kAppendThreads, 4)
    kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     const int64_t* __restrict__ loc, int64_t n_tokens, int chunks_per_token,
                     uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int64_t pool_slots,
                     int32_t* dev_err) {
    __shared__ int64_t s_slot[kAppendSpan + 1];
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = n_tokens * chunks_per_token;
    const int64_t c0 = (int64_t)blockIdx.x * kAppendSpan;
    uint4 kr[kAppendUnroll], vr[kAppendUnroll];
#pragma unroll
    for (int j = 0; j < kAppendUnroll; ++j) {
        const int64_t idx = c0 + j * kAppendThreads + threadIdx.x;
        if (idx < total) {
            kr[j] = __ldcs(k + idx);
            vr[j] = __ldcs(v + idx);
        }
    }
    const int64_t t0 = c0 / chunks_per_token;
    const int64_t t1 = (min(total, c0 + kAppendSpan) - 1) / chunks_per_token;
    for (int64_t t = t0 + threadIdx.x; t <= t1; t += kAppendThreads) {
        const int64_t s = __ldg(loc + t);
        const bool ok = s >= 0 && s < pool_slots;
        // the block holding the token's first chunk reports a bad slot
        if (!ok && t * chunks_per_token >= c0) report_error(dev_err, PCP_ERR_BAD_INDEX);
        s_slot[t - t0] = ok ? s : -1;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kAppendUnroll; ++j) {
        const int64_t idx = c0 + j * kAppendThreads + threadIdx.x;
        if (idx >= total) continue;
        const int64_t t = idx / chunks_per_token;
        const int64_t s = s_slot[t - t0];
        if (s < 0) continue;
        const int64_t ch = idx - t * chunks_per_token;
        __stcs(k_pool + s * chunks_per_token + ch, kr[j]);
        __stcs(v_pool + s * chunks_per_token + ch, vr[j]);
    }
}

// Slot mapping and KV append in one pass (append_paged_span): the slots of
// the span's tokens come from the page table while the span's K/V loads are
// in flight, so no out_cache_loc array is read back.
__global__ void __launch_bounds__(kAppendThreads, 4)
    kv_append_paged_kernel(const __grid_constant__ AppendParams a) {
    __shared__ AppendSmem<kAppendThreads> S;
    pdl_wait();
    pdl_launch_dependents();
    append_paged_span<kAppendThreads>(a, S, blockIdx.x);
}

cudaError_t launch_kv_append_paged(const AppendParams& a, cudaStream_t stream) {
    const int64_t blocks = (a.total_q * a.chunks_per_token + kAppendSpan - 1) / kAppendSpan;
    return launch_pdl(kv_append_paged_kernel, dim3((unsigned)blocks), dim3(kAppendThreads), 0,
                      stream, a);
}

// Copy-on-write of shared pages: for copy c, slots [0, n_slots[c]) of page
// src[c] go to the same slots of page dst[c], K and V.  One CTA row per copy;
// a thread moves one 16-byte chunk.
__global__ void copy_page_slots_kernel(const int32_t* __restrict__ src,
                                       const int32_t* __restrict__ dst,
                                       const int32_t* __restrict__ n_slots, int64_t num_pages,
                                       int page_size, int chunks_per_slot,
                                       uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                       int32_t* dev_err) {
    pdl_wait();
    pdl_launch_dependents();
    const int c = blockIdx.y;
    const int64_t s = src[c], d = dst[c];
    const int n = n_slots[c];
    if (s < 0 || s >= num_pages || d < 0 || d >= num_pages || n < 0 || n > page_size) {
        if (blockIdx.x == 0 && threadIdx.x == 0) report_error(dev_err, PCP_ERR_BAD_INDEX);
        return;
    }
    const int64_t total = (int64_t)n * chunks_per_slot;
    const int64_t s0 = s * page_size * chunks_per_slot, d0 = d * page_size * chunks_per_slot;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 kv = k_pool[s0 + i];
        const uint4 vv = v_pool[s0 + i];
        k_pool[d0 + i] = kv;
        v_pool[d0 + i] = vv;
    }
}

cudaError_t launch_copy_page_slots(const int32_t* src, const int32_t* dst,
                                   const int32_t* n_slots, int n_copies, int64_t num_pages,
                                   int page_size, int chunks_per_slot, void* k_pool,
                                   void* v_pool, int32_t* dev_err, cudaStream_t stream) {
    const int threads = 256;
    const int64_t per_copy = (int64_t)page_size * chunks_per_slot;
    const int64_t bx = std::min<int64_t>((per_copy + threads - 1) / threads, 64);
    return launch_pdl(copy_page_slots_kernel, dim3((unsigned)bx, (unsigned)n_copies),
                      dim3(threads), 0, stream, src, dst, n_slots, num_pages, page_size,
                      chunks_per_slot, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                      dev_err);
}

cudaError_t launch_out_cache_loc(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* prefix_lens,
                                 int batch, int64_t total_q, int page_size, int64_t num_pages,
                                 int64_t* loc, int32_t* dev_err, int sm_count,
                                 cudaStream_t stream) {
    const int threads = 256;
    int64_t blocks = (total_q + threads - 1) / threads;
    if (blocks > (int64_t)sm_count * 8) blocks = (int64_t)sm_count * 8;
    return launch_pdl(out_cache_loc_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      qo_indptr, kv_indptr, kv_indices, prefix_lens, batch, total_q, page_size,
                      num_pages, loc, dev_err);
}

cudaError_t launch_kv_append(const void* k, const void* v, const int64_t* loc, int64_t n_tokens,
                             int chunks_per_token, void* k_pool, void* v_pool, int64_t pool_slots,
                             int32_t* dev_err, int sm_count, cudaStream_t stream) {
    (void)sm_count;
    const int64_t blocks = (n_tokens * chunks_per_token + kAppendSpan - 1) / kAppendSpan;
    return launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(kAppendThreads), 0, stream,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), loc, n_tokens,
                      chunks_per_token, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                      pool_slots, dev_err);
}

}  // namespace pcp
