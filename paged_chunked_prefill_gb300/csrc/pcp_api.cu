// The C ABI: argument validation, workspace layout, tensor-map encoding and
// the launches of the planner, tensor-core and row kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "pcp.h"
#include "pcp_internal.h"


namespace pcp {

bool pdl_enabled() {
    static const bool on = std::getenv("PCP_DISABLE_PDL") == nullptr;
    return on;
}

cudaError_t launch_plan(cudaStream_t stream, const PlanParams& p);
cudaError_t launch_plan_append(cudaStream_t stream, const PlanParams& p, const AppendParams& a);
int64_t plan_append_spans(const AppendParams& a);
cudaError_t launch_extend_tc(int head_dim, int grid, cudaStream_t stream, const TcParams& p,
                             const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv);
cudaError_t launch_rows(int head_dim, int grid, cudaStream_t stream, const RowParams& p,
                        const CUtensorMap& tk, const CUtensorMap& tv);
cudaError_t launch_combine(int head_dim, cudaStream_t stream, const CombineParams& p);
cudaError_t launch_out_cache_loc(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                 const int32_t* kv_indices, const int32_t* prefix_lens,
                                 int batch, int64_t total_q, int page_size, int64_t num_pages,
                                 int64_t* loc, int32_t* dev_err, int sm_count,
                                 cudaStream_t stream);
cudaError_t launch_copy_page_slots(const int32_t* src, const int32_t* dst,
                                   const int32_t* n_slots, int n_copies, int64_t num_pages,
                                   int page_size, int chunks_per_slot, void* k_pool,
                                   void* v_pool, int32_t* dev_err, cudaStream_t stream);
cudaError_t launch_kv_append_paged(const AppendParams& a, cudaStream_t stream);
cudaError_t launch_kv_append(const void* k, const void* v, const int64_t* loc, int64_t n_tokens,
                             int chunks_per_token, void* k_pool, void* v_pool, int64_t pool_slots,
                             int32_t* dev_err, int sm_count, cudaStream_t stream);

namespace {

// The CUDA error behind the last PCP_ERR_CUDA returned on this thread.
thread_local cudaError_t t_last_cuda = cudaSuccess;

bool failed(cudaError_t e) {
    if (e == cudaSuccess) return false;
    t_last_cuda = e;
    return true;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices] = {0};
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;

// SM count of the current device, cached per device.
pcp_status sm_count(int* out) {
    int dev = 0;
    if (failed(cudaGetDevice(&dev))) return PCP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev < 0 || dev >= kMaxDevices) return PCP_ERR_UNSUPPORTED;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        if (failed(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)))
            return PCP_ERR_CUDA;
        g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return PCP_OK;
}

pcp_status get_encoder(EncodeFn* fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (failed(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                    cudaEnableDefault, &q)) ||
            q != cudaDriverEntryPointSuccess || p == nullptr)
            return PCP_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeFn>(p);
    }
    *fn = g_encode;
    return PCP_OK;
}

// 3-D bf16 tensor map over [d2][d1][d0] with a 128-byte-swizzled box.
pcp_status encode_3d(EncodeFn enc, CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                     uint64_t d2, uint32_t b0, uint32_t b1, uint32_t b2) {
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PCP_OK : PCP_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

}  // namespace

pcp_status check_extend_args(const ExtendArgs& a, WsLayout* lay) {
    if (a.batch < 0 || a.total_q < 0 || a.total_q >= (int64_t(1) << 31) || a.n_q_heads < 1 ||
        a.n_kv_heads < 1 || a.page_size < 1 || a.window < 0 || a.num_pages < 0 ||
        a.dev_err == nullptr)
        return PCP_ERR_INVALID_ARG;
    if ((a.causal != 0 && a.causal != 1) || (!a.causal && a.window > 0))
        return PCP_ERR_INVALID_ARG;
    const MaskParams& m = a.mask;
    if (m.data != nullptr &&
        (m.b_stride < 0 || m.h_stride < 0 || m.q_stride < 0 || m.q_len < 0 || m.kv_len < 0 ||
         !aligned(m.data, 16) || m.b_stride % 16 != 0 || m.h_stride % 16 != 0 ||
         m.q_stride % 16 != 0))
        return PCP_ERR_INVALID_ARG;
    if (a.batch == 0 && a.total_q != 0) return PCP_ERR_INVALID_ARG;
    if (a.n_q_heads % a.n_kv_heads != 0) return PCP_ERR_INVALID_ARG;
    if (a.head_dim != 64 && a.head_dim != 128) return PCP_ERR_UNSUPPORTED;
    if (a.n_q_heads / a.n_kv_heads > kTileM) return PCP_ERR_UNSUPPORTED;
    if (!std::isfinite(a.sm_scale)) return PCP_ERR_INVALID_ARG;
    if (a.num_pages * (int64_t)a.page_size >= (int64_t(1) << 31)) return PCP_ERR_UNSUPPORTED;
    if (!ws_layout(a.batch, a.total_q, a.n_q_heads, a.n_kv_heads, a.head_dim, lay))
        return PCP_ERR_INVALID_ARG;
    if (a.total_q == 0) return PCP_OK;
    if (!a.q || !a.qo_indptr || !a.kv_indptr || !a.kv_indices || !a.prefix_lens || !a.k_pool ||
        !a.v_pool || !a.out)
        return PCP_ERR_INVALID_ARG;
    if (a.num_pages < 1) return PCP_ERR_INVALID_ARG;
    if (!aligned(a.q, 16) || !aligned(a.out, 16) || !aligned(a.k_pool, 16) ||
        !aligned(a.v_pool, 16))
        return PCP_ERR_INVALID_ARG;
    if (a.qo_indptr_host != nullptr) {
        const int32_t* h = a.qo_indptr_host;
        if (h[0] != 0 || h[a.batch] != a.total_q) return PCP_ERR_INVALID_ARG;
        for (int b = 0; b < a.batch; ++b)
            if (h[b + 1] < h[b]) return PCP_ERR_INVALID_ARG;
    }
    return PCP_OK;
}

pcp_status run_extend(const ExtendArgs& a, const pcp_call_options* opts) {
    // ---- host-visible checks, before anything is launched
    WsLayout lay;
    pcp_status st = check_extend_args(a, &lay);
    if (st != PCP_OK) return st;
    pcp_call_options o = {};
    if (opts != nullptr) o = *opts;
    if ((o.tc_event_before == nullptr) != (o.tc_event_after == nullptr) ||
        (o.rows_event_before == nullptr) != (o.rows_event_after == nullptr))
        return PCP_ERR_INVALID_ARG;
    // the step's new K/V rows, appended before attending: both or neither
    const bool append = o.k_new != nullptr || o.v_new != nullptr;
    if (append && (o.k_new == nullptr || o.v_new == nullptr ||
                   (a.total_q > 0 && (!aligned(o.k_new, 16) || !aligned(o.v_new, 16)))))
        return PCP_ERR_INVALID_ARG;
    if (o.out_cache_loc != nullptr && !append) return PCP_ERR_INVALID_ARG;
    if (a.total_q == 0) return PCP_OK;
    // a call needs the workspace up to the split buffers; it splits items only
    // when the whole layout fits
    if (a.workspace == nullptr || a.workspace_bytes < lay.split_begin ||
        !aligned(a.workspace, 256))
        return PCP_ERR_WORKSPACE;
    const int group = a.n_q_heads / a.n_kv_heads;
    const int head_dim = a.head_dim;
    const int page_size = a.page_size;
    // With the host copy of qo_indptr the call launches only the kernels that
    // have work: the tensor-core kernel for chunks of more than
    // row_path_max_chunk(G) rows, the row kernel and combine for the others.
    const int rmax = row_path_max_chunk(group);
    bool run_tc = true, run_rows = rmax > 0;
    if (a.qo_indptr_host != nullptr) {
        bool any_tc = false, any_row = false;
        for (int b = 0; b < a.batch; ++b) {
            const int64_t c = (int64_t)a.qo_indptr_host[b + 1] - a.qo_indptr_host[b];
            if (c > rmax) any_tc = true;
            else if (c > 0) any_row = true;
        }
        run_tc = any_tc;
        run_rows = run_rows && any_row;
    }

    int sms = 0;
    st = sm_count(&sms);
    if (st != PCP_OK) return st;

    // With host copies of qo_indptr and prefix_lens the host decides whether
    // a call with both kinds of chunks takes its decode-shaped ones onto the
    // tensor cores (the planner's rule, absorb_decode_rows, on the same
    // figures) and then launches only the kernels that have work.
    // With both host copies the host also decides whether the call splits its
    // longest tensor-core items along their KV tiles (split_longest_items):
    // not for masked calls, and only when the workspace holds the split
    // buffers.
    int absorb = -1;
    int split = 0;
    if (run_tc && a.qo_indptr_host != nullptr && o.prefix_lens_host != nullptr) {
        const int item_pos = q_positions_per_tile(group) * kQTiles;
        unsigned long long w_tc = 0, w_dec = 0;
        int max_tc = 0, max_dec = 0;
        for (int b = 0; b < a.batch; ++b) {
            const int c = a.qo_indptr_host[b + 1] - a.qo_indptr_host[b];
            const int P = o.prefix_lens_host[b];
            if (c <= 0 || P < 0 || (int64_t)P + c >= INT32_MAX) continue;
            if (c > rmax) {
                for (int k = 0; k * item_pos < c; ++k) {
                    const int t = tc_item_tiles(P, c, k, item_pos, a.window, a.causal);
                    w_tc += (unsigned long long)t * a.n_kv_heads;
                    max_tc = t > max_tc ? t : max_tc;
                }
            } else {
                const int t = dec_weight(tc_item_tiles(P, c, 0, item_pos, a.window, a.causal));
                w_dec += (unsigned long long)t * a.n_kv_heads;
                max_dec = t > max_dec ? t : max_dec;
            }
        }
        if (run_rows) {
            absorb = absorb_decode_rows(w_tc, max_tc, w_dec, max_dec, sms) ? 1 : 0;
            if (absorb == 1) run_rows = false;
        }
        const bool dec_tc = absorb == 1;
        const unsigned long long w_all = w_tc + (dec_tc ? w_dec : 0ull);
        const int longest = dec_tc && max_dec > max_tc ? max_dec : max_tc;
        split = a.mask.data == nullptr && a.workspace_bytes >= lay.total &&
                        split_longest_items(w_all, longest, sms)
                    ? 1
                    : 0;
    }
    EncodeFn enc = nullptr;
    st = get_encoder(&enc);
    if (st != PCP_OK) return st;

    const float scale = a.sm_scale > 0.f ? a.sm_scale : 1.0f / std::sqrt((float)head_dim);
    const float scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);
    unsigned char* ws = static_cast<unsigned char*>(a.workspace);
    const int qpos = q_positions_per_tile(group);
    const int num_slots = (int)(a.num_pages * page_size);
    // TMA boxes for page runs of >= kTmaMinRows keys; smaller pages go to
    // the cp.async gather warps
    const int g128 = gcd_int(page_size, kTileN);
    const int box_rows = g128 >= kTmaMinRows ? g128 : 0;
    const int page_shift =
        (page_size & (page_size - 1)) == 0 ? __builtin_ctz((unsigned)page_size) : -1;

    // ---- tensor maps: Q boxes of (64 dims, G heads, qpos positions); K/V
    // boxes of (64 dims, one KV head, one page run)
    CUtensorMap tq, tk, tv;
    if ((st = encode_3d(enc, &tq, a.q, head_dim, a.n_q_heads, a.total_q, 64, group, qpos)) !=
        PCP_OK)
        return st;
    const uint32_t kv_box = box_rows > 0 ? box_rows : 8;
    if ((st = encode_3d(enc, &tk, a.k_pool, head_dim, a.n_kv_heads, num_slots, 64, 1, kv_box)) !=
        PCP_OK)
        return st;
    if ((st = encode_3d(enc, &tv, a.v_pool, head_dim, a.n_kv_heads, num_slots, 64, 1, kv_box)) !=
        PCP_OK)
        return st;

    // A decode-only call of at most kRowSelfPlanMaxSeqs sequences is planned
    // by the row kernel itself; everything else by the planner kernel.
    const bool self_plan = !run_tc && run_rows && a.batch <= kRowSelfPlanMaxSeqs;

    // ---- 1. plan
    PlanParams pp;
    pp.qo_indptr = a.qo_indptr;
    pp.kv_indptr = a.kv_indptr;
    pp.prefix_lens = a.prefix_lens;
    pp.batch = a.batch;
    pp.total_q = a.total_q;
    pp.n_kv_heads = a.n_kv_heads;
    pp.group = group;
    pp.page_size = page_size;
    pp.window = a.window;
    pp.causal = a.causal;
    pp.tc_work = run_tc ? 1 : 0;
    pp.absorb = absorb;
    pp.split = split;
    pp.sm_count = sms;
    pp.tc_gather = box_rows == 0 ? 1 : 0;
    pp.ws = ws;
    pp.lay = lay;
    pp.dev_err = a.dev_err;
    // The append (slot mapping and scatter of the step's new K/V rows) runs in
    // the planner's launch, in CTAs of its own beside the planning CTA: as a
    // kernel of its own ahead of the planner it filled every SM's register
    // file, so the planner could start only once the append drained.  A
    // self-planned call launches the append kernel ahead of the row kernel.
    AppendParams ap;
    if (append) {
        ap.qo_indptr = a.qo_indptr;
        ap.kv_indptr = a.kv_indptr;
        ap.kv_indices = a.kv_indices;
        ap.prefix_lens = a.prefix_lens;
        ap.batch = a.batch;
        ap.total_q = a.total_q;
        ap.page_size = page_size;
        ap.num_pages = a.num_pages;
        ap.k = o.k_new;
        ap.v = o.v_new;
        ap.chunks_per_token = a.n_kv_heads * head_dim * 2 / 16;
        ap.k_pool = const_cast<void*>(a.k_pool);
        ap.v_pool = const_cast<void*>(a.v_pool);
        ap.loc = o.out_cache_loc;
        ap.dev_err = a.dev_err;
    }
    // Beside the planner only while the append fits in one wave of its
    // 1024-thread CTAs (one per SM): a longer append runs faster as a kernel
    // of its own, whose four 256-thread blocks per SM overlap one another's
    // load and store phases (32,768 tokens: 43.5 us against 56-60 us), and
    // the planner after it is then a small part of the step.
    const bool beside = append && !self_plan && plan_append_spans(ap) <= sms - 1;
    if (append && !beside && failed(launch_kv_append_paged(ap, s))) return PCP_ERR_CUDA;
    if (!self_plan &&
        failed(beside ? launch_plan_append(s, pp, ap) : launch_plan(s, pp)))
        return PCP_ERR_CUDA;

    // ---- 2. tensor-core extend kernel (persistent, one CTA per SM)
    TcParams tp;
    tp.qo_indptr = a.qo_indptr;
    tp.kv_indptr = a.kv_indptr;
    tp.kv_indices = a.kv_indices;
    tp.prefix_lens = a.prefix_lens;
    tp.ws = ws;
    tp.lay = lay;
    tp.k_pool = static_cast<const uint16_t*>(a.k_pool);
    tp.v_pool = static_cast<const uint16_t*>(a.v_pool);
    tp.out = static_cast<uint16_t*>(a.out);
    tp.lse = a.lse;
    tp.n_q_heads = a.n_q_heads;
    tp.n_kv_heads = a.n_kv_heads;
    tp.group = group;
    tp.qpos = qpos;
    tp.page_size = page_size;
    tp.box_rows = box_rows;
    tp.page_shift = page_shift;
    tp.num_pages = a.num_pages;
    tp.num_slots = num_slots;
    tp.window = a.window;
    tp.causal = a.causal;
    tp.mask = a.mask;
    tp.scale_log2 = scale_log2;
    tp.stall_ns = o.test_stall_ns;
    tp.dev_err = a.dev_err;
    tp.split = split;
    // One-Q-tile items (decode-shaped chunks that join the tensor cores, and
    // a chunk's last item when it holds at most one Q tile of positions) take
    // the instantiation that alternates their S/P buffers (with split items
    // too, on the page-box path); with the host copy of qo_indptr the host
    // knows whether the call has any.  Calls without
    // them keep the instantiation that carries none of that code.
    int ping = 0;
    if (run_tc && a.causal && a.mask.data == nullptr && a.qo_indptr_host != nullptr) {
        const int item_pos = qpos * kQTiles;
        for (int b = 0; b < a.batch && !ping; ++b) {
            const int c = a.qo_indptr_host[b + 1] - a.qo_indptr_host[b];
            if (c <= 0) continue;
            if (c <= rmax) ping = 1;  // decode-shaped: a one-Q-tile item if it joins
            else if (((c - 1) / item_pos) * item_pos + qpos >= c) ping = 1;
        }
    }
    tp.ping = ping;
    cudaEvent_t evb = static_cast<cudaEvent_t>(o.tc_event_before);
    cudaEvent_t eva = static_cast<cudaEvent_t>(o.tc_event_after);
    if (evb && failed(cudaEventRecord(evb, s))) return PCP_ERR_CUDA;
    if (run_tc && failed(launch_extend_tc(head_dim, sms, s, tp, tq, tk, tv))) return PCP_ERR_CUDA;
    if (eva && failed(cudaEventRecord(eva, s))) return PCP_ERR_CUDA;

    // ---- 3. decode-shaped rows (split-KV on CUDA cores, equal tiles per CTA)
    if (run_rows) {
        RowParams rp;
        rp.self_plan = self_plan ? 1 : 0;
        rp.batch = a.batch;
        rp.total_q = a.total_q;
        rp.q = static_cast<const uint16_t*>(a.q);
        rp.qo_indptr = a.qo_indptr;
        rp.kv_indptr = a.kv_indptr;
        rp.kv_indices = a.kv_indices;
        rp.prefix_lens = a.prefix_lens;
        rp.ws = ws;
        rp.lay = lay;
        rp.k_pool = static_cast<const uint16_t*>(a.k_pool);
        rp.v_pool = static_cast<const uint16_t*>(a.v_pool);
        rp.out = static_cast<uint16_t*>(a.out);
        rp.lse = a.lse;
        rp.n_q_heads = a.n_q_heads;
        rp.n_kv_heads = a.n_kv_heads;
        rp.group = group;
        rp.page_size = page_size;
        rp.box_rows = box_rows;
        rp.box_shift = box_rows > 0 ? __builtin_ctz((unsigned)box_rows) : 0;
        rp.page_shift = page_shift;
        rp.num_pages = a.num_pages;
        rp.num_slots = num_slots;
        rp.window = a.window;
        rp.causal = a.causal;
        rp.mask = a.mask;
        rp.scale_log2 = scale_log2;
        rp.stall_ns = o.test_stall_ns;
        rp.dev_err = a.dev_err;
        cudaEvent_t erb = static_cast<cudaEvent_t>(o.rows_event_before);
        cudaEvent_t era = static_cast<cudaEvent_t>(o.rows_event_after);
        if (erb && failed(cudaEventRecord(erb, s))) return PCP_ERR_CUDA;
        if (failed(launch_rows(head_dim, row_grid(sms), s, rp, tk, tv))) return PCP_ERR_CUDA;
        if (era && failed(cudaEventRecord(era, s))) return PCP_ERR_CUDA;
        // ---- 4. merge split-KV partials (one CTA per split group)
        CombineParams cp;
        cp.ws = ws;
        cp.lay = lay;
        cp.out = static_cast<uint16_t*>(a.out);
        cp.lse = a.lse;
        cp.n_q_heads = a.n_q_heads;
        cp.n_kv_heads = a.n_kv_heads;
        cp.group = group;
        cp.n_groups = a.batch * a.n_kv_heads;
        if (failed(launch_combine(head_dim, s, cp))) return PCP_ERR_CUDA;
    }
    return PCP_OK;
}

}  // namespace pcp

using namespace pcp;

extern "C" {

const char* pcp_status_string(int status) {
    switch (status) {
        case PCP_OK: return "PCP_OK";
        case PCP_ERR_INVALID_ARG: return "PCP_ERR_INVALID_ARG: invalid argument";
        case PCP_ERR_UNSUPPORTED: return "PCP_ERR_UNSUPPORTED: unsupported shape";
        case PCP_ERR_BAD_INDEX: return "PCP_ERR_BAD_INDEX: page id or slot outside the pool";
        case PCP_ERR_WORKSPACE: return "PCP_ERR_WORKSPACE: workspace too small or misaligned";
        case PCP_ERR_CUDA: return "PCP_ERR_CUDA: CUDA call failed";
        case PCP_ERR_TIMEOUT: return "PCP_ERR_TIMEOUT: a bounded device wait ran out";
        default: return "PCP_ERR_UNKNOWN";
    }
}

int pcp_abi_version(void) { return 5; }

const char* pcp_last_cuda_error(void) {
    return t_last_cuda == cudaSuccess ? "no error" : cudaGetErrorString(t_last_cuda);
}

pcp_status pcp_compute_out_cache_loc(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                     const int32_t* kv_indices, const int32_t* prefix_lens,
                                     int batch, int64_t total_q, int page_size,
                                     int64_t num_pages, int64_t* out_cache_loc,
                                     int32_t* dev_err, void* stream) {
    if (batch < 0 || total_q < 0 || page_size < 1 || num_pages < 0 || dev_err == nullptr)
        return PCP_ERR_INVALID_ARG;
    if (batch == 0 && total_q != 0) return PCP_ERR_INVALID_ARG;
    if (total_q == 0) return PCP_OK;
    if (!qo_indptr || !kv_indptr || !kv_indices || !prefix_lens || !out_cache_loc)
        return PCP_ERR_INVALID_ARG;
    int sms = 0;
    pcp_status st = sm_count(&sms);
    if (st != PCP_OK) return st;
    cudaError_t e = launch_out_cache_loc(qo_indptr, kv_indptr, kv_indices, prefix_lens, batch,
                                         total_q, page_size, num_pages, out_cache_loc, dev_err,
                                         sms, static_cast<cudaStream_t>(stream));
    return failed(e) ? PCP_ERR_CUDA : PCP_OK;
}

pcp_status pcp_kv_append(const void* k, const void* v, const int64_t* out_cache_loc,
                         int64_t n_tokens, int n_kv_heads, int head_dim, void* k_pool,
                         void* v_pool, int64_t pool_slots, int32_t* dev_err, void* stream) {
    if (n_tokens < 0 || n_kv_heads < 1 || head_dim < 1 || pool_slots < 0 || dev_err == nullptr)
        return PCP_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PCP_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PCP_OK;
    if (!k || !v || !out_cache_loc || !k_pool || !v_pool) return PCP_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16))
        return PCP_ERR_INVALID_ARG;
    int sms = 0;
    pcp_status st = sm_count(&sms);
    if (st != PCP_OK) return st;
    const int chunks = n_kv_heads * head_dim * 2 / 16;
    cudaError_t e = launch_kv_append(k, v, out_cache_loc, n_tokens, chunks, k_pool, v_pool,
                                     pool_slots, dev_err, sms, static_cast<cudaStream_t>(stream));
    return failed(e) ? PCP_ERR_CUDA : PCP_OK;
}

pcp_status pcp_kv_append_paged(const int32_t* qo_indptr, const int32_t* kv_indptr,
                               const int32_t* kv_indices, const int32_t* prefix_lens, int batch,
                               int64_t total_q, int page_size, int64_t num_pages, const void* k,
                               const void* v, int n_kv_heads, int head_dim, void* k_pool,
                               void* v_pool, int64_t* out_cache_loc, int32_t* dev_err,
                               void* stream) {
    if (batch < 0 || total_q < 0 || page_size < 1 || num_pages < 0 || n_kv_heads < 1 ||
        head_dim < 1 || dev_err == nullptr)
        return PCP_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PCP_ERR_UNSUPPORTED;
    if (batch == 0 && total_q != 0) return PCP_ERR_INVALID_ARG;
    if (total_q == 0) return PCP_OK;
    if (!qo_indptr || !kv_indptr || !kv_indices || !prefix_lens || !k || !v || !k_pool ||
        !v_pool)
        return PCP_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16))
        return PCP_ERR_INVALID_ARG;
    AppendParams ap;
    ap.qo_indptr = qo_indptr;
    ap.kv_indptr = kv_indptr;
    ap.kv_indices = kv_indices;
    ap.prefix_lens = prefix_lens;
    ap.batch = batch;
    ap.total_q = total_q;
    ap.page_size = page_size;
    ap.num_pages = num_pages;
    ap.k = k;
    ap.v = v;
    ap.chunks_per_token = n_kv_heads * head_dim * 2 / 16;
    ap.k_pool = k_pool;
    ap.v_pool = v_pool;
    ap.loc = out_cache_loc;
    ap.dev_err = dev_err;
    cudaError_t e = launch_kv_append_paged(ap, static_cast<cudaStream_t>(stream));
    return failed(e) ? PCP_ERR_CUDA : PCP_OK;
}

pcp_status pcp_copy_page_slots(void* k_pool, void* v_pool, int64_t num_pages, int page_size,
                               int n_kv_heads, int head_dim, const int32_t* src_pages,
                               const int32_t* dst_pages, const int32_t* n_slots, int n_copies,
                               int32_t* dev_err, void* stream) {
    if (num_pages < 0 || page_size < 1 || n_kv_heads < 1 || head_dim < 1 || n_copies < 0 ||
        n_copies > 65535 || dev_err == nullptr)
        return PCP_ERR_INVALID_ARG;
    if ((head_dim * 2) % 16 != 0) return PCP_ERR_UNSUPPORTED;
    if (n_copies == 0) return PCP_OK;
    if (!k_pool || !v_pool || !src_pages || !dst_pages || !n_slots) return PCP_ERR_INVALID_ARG;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16)) return PCP_ERR_INVALID_ARG;
    const int chunks = n_kv_heads * head_dim * 2 / 16;
    return failed(launch_copy_page_slots(src_pages, dst_pages, n_slots, n_copies, num_pages,
                                         page_size, chunks, k_pool, v_pool, dev_err,
                                         static_cast<cudaStream_t>(stream)))
               ? PCP_ERR_CUDA
               : PCP_OK;
}

size_t pcp_extend_workspace_size(int batch, int64_t total_q, int n_q_heads, int n_kv_heads,
                                 int head_dim) {
    if (head_dim != 64 && head_dim != 128) return 0;
    WsLayout L;
    if (!ws_layout(batch, total_q, n_q_heads, n_kv_heads, head_dim, &L)) return 0;
    return L.total;
}

pcp_status pcp_paged_extend_attn_ex(
    const void* q, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
    const int32_t* prefix_lens, const int32_t* qo_indptr_host, int batch, int64_t total_q,
    const void* k_pool, const void* v_pool, int64_t num_pages, int page_size, int n_q_heads,
    int n_kv_heads, int head_dim, int window, float sm_scale, int causal, const uint8_t* mask,
    int64_t mask_b_stride, int64_t mask_h_stride, int64_t mask_q_stride, int32_t mask_q_len,
    int32_t mask_kv_len, void* out, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* dev_err, void* stream, const pcp_call_options* options) {
    ExtendArgs a;
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
    a.causal = causal;
    a.mask.data = mask;
    a.mask.b_stride = mask_b_stride;
    a.mask.h_stride = mask_h_stride;
    a.mask.q_stride = mask_q_stride;
    a.mask.q_len = mask_q_len;
    a.mask.kv_len = mask_kv_len;
    a.out = out;
    a.lse = lse;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
    a.dev_err = dev_err;
    a.stream = stream;
    return run_extend(a, options);
}

pcp_status pcp_paged_extend_attn_masked(
    const void* q, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
    const int32_t* prefix_lens, const int32_t* qo_indptr_host, int batch, int64_t total_q,
    const void* k_pool, const void* v_pool, int64_t num_pages, int page_size, int n_q_heads,
    int n_kv_heads, int head_dim, int window, float sm_scale, int causal, const uint8_t* mask,
    int64_t mask_b_stride, int64_t mask_h_stride, int64_t mask_q_stride, int32_t mask_q_len,
    int32_t mask_kv_len, void* out, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* dev_err, void* stream) {
    return pcp_paged_extend_attn_ex(q, qo_indptr, kv_indptr, kv_indices, prefix_lens,
                                    qo_indptr_host, batch, total_q, k_pool, v_pool, num_pages,
                                    page_size, n_q_heads, n_kv_heads, head_dim, window, sm_scale,
                                    causal, mask, mask_b_stride, mask_h_stride, mask_q_stride,
                                    mask_q_len, mask_kv_len, out, lse, workspace,
                                    workspace_bytes, dev_err, stream, nullptr);
}

pcp_status pcp_paged_extend_attn(const void* q, const int32_t* qo_indptr,
                                 const int32_t* kv_indptr, const int32_t* kv_indices,
                                 const int32_t* prefix_lens, const int32_t* qo_indptr_host,
                                 int batch, int64_t total_q, const void* k_pool,
                                 const void* v_pool, int64_t num_pages, int page_size,
                                 int n_q_heads, int n_kv_heads, int head_dim, int window,
                                 float sm_scale, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream) {
    return pcp_paged_extend_attn_ex(q, qo_indptr, kv_indptr, kv_indices, prefix_lens,
                                    qo_indptr_host, batch, total_q, k_pool, v_pool, num_pages,
                                    page_size, n_q_heads, n_kv_heads, head_dim, window, sm_scale,
                                    1, nullptr, 0, 0, 0, 0, 0, out, lse, workspace,
                                    workspace_bytes, dev_err, stream, nullptr);
}

pcp_status pcp_read_error(const int32_t* dev_err, void* stream, int32_t* host_err) {
    if (dev_err == nullptr || host_err == nullptr) return PCP_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (failed(cudaMemcpyAsync(host_err, dev_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s)))
        return PCP_ERR_CUDA;
    if (failed(cudaStreamSynchronize(s))) return PCP_ERR_CUDA;
    return PCP_OK;
}

}  // extern "C"
