// Slot mapping of a step's new tokens and the KV append (scatter into pages).
//
// AReno PR #642 ("What does this PR do?", third bullet): prefill continues
// inside the last allocated KV page, so the first new token of a chunk whose
// prefix is not a multiple of the page size lands mid-page.  AstrAI's
// PagePool.bind_tasks builds out_cache_loc once per step and the backend writes
// k_buffer[layer, out_cache_loc] = k before attending; here both are kernels.
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
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total_q;
         t += (int64_t)gridDim.x * blockDim.x) {
        // sequence owning row t: the last b with qo_indptr[b] <= t
        int lo = 0, hi = batch;  // answer in [lo, hi)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (qo_indptr[mid] <= t) lo = mid;
            else hi = mid;
        }
        const int b = lo;
        int64_t out = -1;
        if (t >= qo_indptr[b] && t < qo_indptr[b + 1]) {
            const int64_t pos = (int64_t)prefix_lens[b] + (t - qo_indptr[b]);
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

// One thread moves one 16-byte chunk of a token's K row and the same chunk of
// its V row; a token row is n_kv_heads * head_dim bf16 values.
__global__ void kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 const int64_t* __restrict__ loc, int64_t n_tokens,
                                 int chunks_per_token, uint4* __restrict__ k_pool,
                                 uint4* __restrict__ v_pool, int64_t pool_slots,
                                 int32_t* dev_err) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t total = n_tokens * chunks_per_token;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / chunks_per_token;
        const int ch = (int)(idx - t * chunks_per_token);
        const int64_t s = __ldg(loc + t);
        if (s < 0 || s >= pool_slots) {
            if (ch == 0) report_error(dev_err, PCP_ERR_BAD_INDEX);
            continue;
        }
        const uint4 kv = __ldcs(k + idx);
        const uint4 vv = __ldcs(v + idx);
        __stcs(k_pool + s * chunks_per_token + ch, kv);
        __stcs(v_pool + s * chunks_per_token + ch, vv);
    }
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
    const int threads = 256;
    const int64_t total = n_tokens * chunks_per_token;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
    return launch_pdl(kv_append_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), loc, n_tokens,
                      chunks_per_token, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool),
                      pool_slots, dev_err);
}

}  // namespace pcp
