// Decode-shaped rows: split-KV attention on CUDA cores.
//
// A chunk with chunk_len * G <= 16 query rows (a decode row is chunk_len 1)
// is HBM-bound: each key is used by at most 16 rows, so this path streams the
// K/V pages at full bandwidth instead of padding 128-row tensor-core tiles.
// The KV range of each (sequence, KV head) is split across CTAs (AstrAI paged
// decode "split-KV" kernel, prior art); each split writes an fp32 partial
// (unnormalised O, running max, normaliser) to the workspace and the last
// split to finish merges the partials with the log-sum-exp identity (the
// AstrAI combine kernel's job, fused here so a mixed batch needs no extra
// launch).  Masking is the same bottom-right causal / window rule as the
// tensor-core path, per row.
//
// Layout: 4 warps; a 128-key tile is gathered through the page table with
// 16-byte cp.async (any page size, zero-filled past the split end), double
// buffered.  Warp w scores keys 32w..32w+31 of the tile (one key per lane),
// keeps its own online-softmax state, and accumulates P V with lanes split
// over head_dim.  The four warp states are merged at the end of the item.
#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

template <int D>
struct RowCfg {
    static constexpr int kRowStride = D * 2 + 16;           // padded smem row (bytes)
    static constexpr int kTileBytes = kRowTile * kRowStride;
    static constexpr int kOffQ = 0;                          // float [16][D]
    static constexpr int kOffK = kOffQ + kRowMaxRows * D * 4;
    static constexpr int kOffV = kOffK + 2 * kTileBytes;
    static constexpr int kOffP = kOffV + 2 * kTileBytes;     // float [4][32][16]
    static constexpr int kOffM = kOffP + 4 * 32 * kRowMaxRows * 4;  // float [4][16] m, l
    static constexpr int kSmemBytes = kOffM + 2 * 4 * kRowMaxRows * 4 + 64;
    static constexpr int kDPerLane = D / 32;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace

template <int D>
__global__ void __launch_bounds__(kRowThreads) row_attn_kernel(const __grid_constant__ RowParams p) {
    using C = RowCfg<D>;
    extern __shared__ __align__(128) uint8_t sm[];
    float* q_s = reinterpret_cast<float*>(sm + C::kOffQ);
    float* p_s = reinterpret_cast<float*>(sm + C::kOffP);
    float* m_s = reinterpret_cast<float*>(sm + C::kOffM);
    float* l_s = m_s + 4 * kRowMaxRows;
    __shared__ int s_item;
    __shared__ int s_last;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    WsHeader* hdr = reinterpret_cast<WsHeader*>(p.ws + p.lay.header);
    const int n_items = hdr->n_row_items;
    const int4* items = reinterpret_cast<const int4*>(p.ws + p.lay.row_items);
    float* part_o = reinterpret_cast<float*>(p.ws + p.lay.partial_o);
    float2* part_ml = reinterpret_cast<float2*>(p.ws + p.lay.partial_ml);
    int* gcnt = reinterpret_cast<int*>(p.ws + p.lay.group_cnt);
    const int G = p.group;
    const float sl2 = p.scale_log2;

    for (;;) {
        if (tid == 0) s_item = atomicAdd(&hdr->row_next, 1);
        __syncthreads();
        const int item = s_item;
        if (item >= n_items) break;
        const int4 i0 = items[2 * item], i1 = items[2 * item + 1];
        const int b = i0.x, g = i0.y, nsplit = i0.w;
        const int kb = i1.x, ke = i1.y, first_item = i1.z;
        const int q0 = p.qo_indptr[b];
        const int c = p.qo_indptr[b + 1] - q0;
        const int P = p.prefix_lens[b];
        const int R = c * G;
        const int32_t* pages = p.kv_indices + p.kv_indptr[b];

        // query rows, pre-scaled into log2 units
        for (int idx = tid; idx < R * D; idx += kRowThreads) {
            const int r = idx / D, d = idx % D;
            const uint16_t qb = p.q[((int64_t)(q0 + r / G) * p.n_q_heads + g * G + r % G) * D + d];
            q_s[idx] = __uint_as_float((uint32_t)qb << 16) * sl2;
        }

        const int t_first = kb / kRowTile, t_last = (ke - 1) / kRowTile;
        auto issue_tile = [&](int t, int stage) {
            uint8_t* kd = sm + C::kOffK + stage * C::kTileBytes;
            uint8_t* vd = sm + C::kOffV + stage * C::kTileBytes;
            constexpr int chunks = D * 2 / 16;
            for (int idx = tid; idx < kRowTile * chunks; idx += kRowThreads) {
                const int row = idx / chunks, ch = idx % chunks;
                const int key = t * kRowTile + row;
                bool ok = key >= kb && key < ke;
                int64_t slot = 0;
                if (ok) {
                    const int page = pages[key / p.page_size];
                    if (page >= 0 && page < p.num_pages) {
                        slot = (int64_t)page * p.page_size + key % p.page_size;
                    } else {
                        ok = false;
                        report_error(p.dev_err, PCP_ERR_BAD_INDEX);
                    }
                }
                const int64_t off = (slot * p.n_kv_heads + g) * D + ch * 8;
                cp_async_16(smem_addr(kd + row * C::kRowStride + ch * 16),
                            ok ? (const void*)(p.k_pool + off) : (const void*)p.k_pool,
                            ok ? 16u : 0u);
                cp_async_16(smem_addr(vd + row * C::kRowStride + ch * 16),
                            ok ? (const void*)(p.v_pool + off) : (const void*)p.v_pool,
                            ok ? 16u : 0u);
            }
            cp_async_commit();
        };

        // per-warp online softmax state (log2 units), replicated across lanes
        float m_r[kRowMaxRows], l_r[kRowMaxRows];
        float o_r[kRowMaxRows][C::kDPerLane];
#pragma unroll
        for (int r = 0; r < kRowMaxRows; ++r) {
            m_r[r] = -INFINITY;
            l_r[r] = 0.f;
#pragma unroll
            for (int i = 0; i < C::kDPerLane; ++i) o_r[r][i] = 0.f;
        }

        issue_tile(t_first, 0);
        for (int t = t_first; t <= t_last; ++t) {
            const int stage = (t - t_first) & 1;
            if (t < t_last) {
                issue_tile(t + 1, stage ^ 1);
                cp_async_wait_group<1>();
            } else {
                cp_async_wait_group<0>();
            }
            __syncthreads();
            const uint8_t* kt = sm + C::kOffK + stage * C::kTileBytes;
            const uint8_t* vt = sm + C::kOffV + stage * C::kTileBytes;
            const int key = t * kRowTile + warp * 32 + lane;

            // scores: one key per lane
            float s[kRowMaxRows];
#pragma unroll
            for (int r = 0; r < kRowMaxRows; ++r) s[r] = 0.f;
            const uint8_t* krow = kt + (warp * 32 + lane) * C::kRowStride;
#pragma unroll 2
            for (int ch = 0; ch < D / 8; ++ch) {
                const uint4 kv = *reinterpret_cast<const uint4*>(krow + ch * 16);
                const float k8[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                                     bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
                for (int r = 0; r < kRowMaxRows; ++r) {
                    if (r < R) {
                        const float4 qa = *reinterpret_cast<const float4*>(q_s + r * D + ch * 8);
                        const float4 qb = *reinterpret_cast<const float4*>(q_s + r * D + ch * 8 + 4);
                        float acc = s[r];
                        acc = fmaf(qa.x, k8[0], acc);
                        acc = fmaf(qa.y, k8[1], acc);
                        acc = fmaf(qa.z, k8[2], acc);
                        acc = fmaf(qa.w, k8[3], acc);
                        acc = fmaf(qb.x, k8[4], acc);
                        acc = fmaf(qb.y, k8[5], acc);
                        acc = fmaf(qb.z, k8[6], acc);
                        acc = fmaf(qb.w, k8[7], acc);
                        s[r] = acc;
                    }
                }
            }
            // mask, online softmax, publish p to shared memory
            const bool in_split = key >= kb && key < ke;
#pragma unroll
            for (int r = 0; r < kRowMaxRows; ++r) {
                if (r < R) {
                    const int pos = P + r / G;
                    const bool vis = in_split && key <= pos && (p.window <= 0 || key > pos - p.window);
                    const float sv = vis ? s[r] : -INFINITY;
                    const float mx = warp_max(sv);
                    const float m_new = fmaxf(m_r[r], mx);
                    float pr = 0.f, alpha = 1.f;
                    if (m_new != -INFINITY) {
                        alpha = fast_exp2(m_r[r] - m_new);
                        pr = fast_exp2(sv - m_new);
                        m_r[r] = m_new;
                    }
                    l_r[r] = l_r[r] * alpha + pr;
#pragma unroll
                    for (int i = 0; i < C::kDPerLane; ++i) o_r[r][i] *= alpha;
                    p_s[(warp * 32 + lane) * kRowMaxRows + r] = pr;
                }
            }
            __syncwarp();
            // O += P V over this warp's 32 keys; lanes split head_dim
#pragma unroll 4
            for (int tk = 0; tk < 32; ++tk) {
                const uint8_t* vrow = vt + (warp * 32 + tk) * C::kRowStride + lane * C::kDPerLane * 2;
                float vv[C::kDPerLane];
                if constexpr (C::kDPerLane == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(vrow);
                    vv[0] = bf16_lo(w.x); vv[1] = bf16_hi(w.x); vv[2] = bf16_lo(w.y); vv[3] = bf16_hi(w.y);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(vrow);
                    vv[0] = bf16_lo(w); vv[1] = bf16_hi(w);
                }
                const float* pp = p_s + (warp * 32 + tk) * kRowMaxRows;
#pragma unroll
                for (int r = 0; r < kRowMaxRows; ++r) {
                    if (r < R) {
                        const float pr = pp[r];
#pragma unroll
                        for (int i = 0; i < C::kDPerLane; ++i) o_r[r][i] = fmaf(pr, vv[i], o_r[r][i]);
                    }
                }
            }
            __syncthreads();
        }

        // merge the four warps' states through shared memory (reusing the K stages)
        float* wo = reinterpret_cast<float*>(sm + C::kOffK);  // [4][16][D]
#pragma unroll
        for (int r = 0; r < kRowMaxRows; ++r) {
            if (r < R) {
                const float lsum = warp_sum(l_r[r]);
                if (lane == 0) {
                    m_s[warp * kRowMaxRows + r] = m_r[r];
                    l_s[warp * kRowMaxRows + r] = lsum;
                }
#pragma unroll
                for (int i = 0; i < C::kDPerLane; ++i)
                    wo[(warp * kRowMaxRows + r) * D + lane * C::kDPerLane + i] = o_r[r][i];
            }
        }
        __syncthreads();
        for (int idx = tid; idx < R * D; idx += kRowThreads) {
            const int r = idx / D, d = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w) M = fmaxf(M, m_s[w * kRowMaxRows + r]);
            float acc = 0.f, lsum = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const float e = fast_exp2(m_s[w * kRowMaxRows + r] - M);
                    acc += e * wo[(w * kRowMaxRows + r) * D + d];
                    lsum += e * l_s[w * kRowMaxRows + r];
                }
            }
            const int64_t orow = (int64_t)(q0 + r / G) * p.n_q_heads + g * G + r % G;
            if (nsplit == 1) {
                const float v = lsum > 0.f ? acc / lsum : 0.f;
                p.out[orow * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                if (d == 0 && p.lse != nullptr)
                    p.lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
            } else {
                part_o[((int64_t)item * kRowMaxRows + r) * D + d] = acc;
                if (d == 0) part_ml[(int64_t)item * kRowMaxRows + r] = make_float2(M, lsum);
            }
        }
        if (nsplit > 1) {
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int prev = atomicAdd(&gcnt[b * p.n_kv_heads + g], 1);
                s_last = prev == nsplit - 1;
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                for (int idx = tid; idx < R * D; idx += kRowThreads) {
                    const int r = idx / D, d = idx % D;
                    float M = -INFINITY;
                    for (int sp = 0; sp < nsplit; ++sp)
                        M = fmaxf(M, __ldcg(&part_ml[(int64_t)(first_item + sp) * kRowMaxRows + r]).x);
                    float acc = 0.f, lsum = 0.f;
                    if (M != -INFINITY) {
                        for (int sp = 0; sp < nsplit; ++sp) {
                            const int64_t it = first_item + sp;
                            const float2 ml = __ldcg(&part_ml[it * kRowMaxRows + r]);
                            const float e = fast_exp2(ml.x - M);
                            acc += e * __ldcg(&part_o[(it * kRowMaxRows + r) * D + d]);
                            lsum += e * ml.y;
                        }
                    }
                    const int64_t orow = (int64_t)(q0 + r / G) * p.n_q_heads + g * G + r % G;
                    const float v = lsum > 0.f ? acc / lsum : 0.f;
                    p.out[orow * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                    if (d == 0 && p.lse != nullptr)
                        p.lse[orow] = lsum > 0.f ? (M + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
                }
                if (tid == 0) gcnt[b * p.n_kv_heads + g] = 0;
            }
        }
        __syncthreads();
    }
}

size_t row_smem_bytes(int head_dim) {
    return head_dim == 128 ? RowCfg<128>::kSmemBytes : RowCfg<64>::kSmemBytes;
}

cudaError_t launch_rows(int head_dim, int grid, cudaStream_t stream, const RowParams& p) {
    const size_t smem = row_smem_bytes(head_dim);
    cudaError_t e;
    if (head_dim == 128) {
        e = cudaFuncSetAttribute(row_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        row_attn_kernel<128><<<grid, kRowThreads, smem, stream>>>(p);
    } else {
        e = cudaFuncSetAttribute(row_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        row_attn_kernel<64><<<grid, kRowThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pcp
