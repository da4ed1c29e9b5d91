// Extend attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running
// inside a host framework that owns every allocation (a custom allocator
// that must not be re-entered, a plugin ABI with no allocation hook, a
// process that pre-reserves all device memory at start-up) or a caller that
// must not call cudaMalloc at all on its hot path.  For them,
// pcp_paged_extend_attn_noalloc runs the same kernels as
// pcp_paged_extend_attn with the scratch taken from a fixed array that lives
// in this library's device image.
#include <cuda_runtime.h>

#include <mutex>

#include "pcp.h"
#include "pcp_internal.h"

namespace {

// The scratch every call of the entry point shares.  Each GPU that loads the
// library keeps this much memory reserved until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device.  The array's
// name in host code is only a stand-in for the symbol, so the address is
// looked up once per device with that device current.
pcp_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PCP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PCP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return PCP_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PCP_OK;
}

}  // namespace

extern "C" pcp_status pcp_paged_extend_attn_noalloc(
    const void* q, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* kv_indices, const int32_t* prefix_lens, const int32_t* qo_indptr_host,
    int batch, int64_t total_q,
    const void* k_pool, const void* v_pool, int64_t num_pages, int page_size, int n_q_heads,
    int n_kv_heads, int head_dim, int window, float sm_scale, void* out, float* lse,
    int32_t* dev_err, void* stream) {
    pcp::ExtendArgs a = {};
    a.q = q;
    a.qo_indptr = qo_indptr;
    a.kv_indptr = kv_indptr;
    a.kv_indices = kv_indices;
    a.prefix_lens = prefix_lens;
    a.qo_indptr_host = qo_indptr_host;
    a.batch = batch;
    a.total_q = total_q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.num_pages = num_pages;
    a.page_size = page_size;
    a.n_q_heads = n_q_heads;
    a.n_kv_heads = n_kv_heads;
    a.head_dim = head_dim;
    a.window = window;
    a.sm_scale = sm_scale;
    a.causal = 1;
    a.out = out;
    a.lse = lse;
    a.dev_err = dev_err;
    a.stream = stream;
    // the same argument checks as the workspace entry point, first
    pcp::WsLayout lay;
    const pcp_status chk = pcp::check_extend_args(a, &lay);
    if (chk != PCP_OK || total_q == 0) return chk;
    // (this entry point never splits items: it needs the layout up to the
    // split buffers)
    if (lay.split_begin > (size_t)PCP_NOALLOC_SCRATCH_BYTES) return PCP_ERR_WORKSPACE;
    void* scratch = nullptr;
    const pcp_status st = scratch_for_current_device(&scratch);
    if (st != PCP_OK) return st;
    a.workspace = scratch;
    a.workspace_bytes = (size_t)PCP_NOALLOC_SCRATCH_BYTES;
    return pcp::run_extend(a, nullptr);
}
