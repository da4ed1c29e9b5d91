// Tensor-core paged extend attention for sm_103a (tcgen05 + TMEM + TMA).
//
// Computes, for the tensor-core work items built by the planner, the extend
// attention of AReno PR #642 ("What does this PR do?": later chunks attend to
// the cached prefix plus their own chunk, bottom-right causal alignment) over
// a paged KV pool, with GQA and an optional sliding window.  The AstrAI paged
// prefill kernel (split-Q, mma.sync, one query head per CTA) is prior art for
// the semantics only; this kernel is laid out for Blackwell:
//
//  * A work item is (sequence b, KV head g, 2 x 128 query rows).  The rows of
//    one 128-row Q tile are (position, head) pairs of the G = Hq/Hkv query
//    heads of KV head g, so every K/V tile fetched from HBM feeds 2 x G query
//    heads (GQA head-group sharing) and 4 tcgen05 MMAs.
//  * Warp roles (384 threads, persistent CTA per SM, dynamic item counter):
//      warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1: one thread
//                  per row, tcgen05.ld of S, mask only on diagonal / window
//                  edge tiles, online softmax in fp32 with exp2 and a lazy O
//                  rescale (only when the running max grows by > 2^8), P
//                  written back to TMEM as bf16, epilogue O / l -> bf16, lse;
//      warp 8      TMA: Q, and K/V when pages hold runs of >= 8 keys (one box
//                  per page run and 64-column block);
//      warp 9      one thread issues tcgen05.mma: S_u = Q_u K^T into TMEM,
//                  then O_u += P_u V with P_u read from TMEM;
//      warps 10-11 page gathers of K/V for pages below 8 keys, with the TMA
//                  warp as a third gatherer: 16 lanes cover one 256-byte row
//                  with 16-byte cp.async (fully coalesced), rows past the
//                  sequence end zero-filled.  (The TMA unit takes about one box
//                  per ~100 cycles, so one-key boxes are hopeless.)
//    K and V land in 128-byte-swizzled shared-memory stages either way.
//  * Ping-pong: while one softmax group works on its S tile, the tensor core
//    runs the other group's QK^T or PV.
//  * Every wait is bounded; a wait that runs out records PCP_ERR_TIMEOUT,
//    the CTA drains its copies and MMAs, frees TMEM and exits.
#include "pcp_device.cuh"
#include "pcp_internal.h"
#include "pcp_launch.h"

namespace pcp {

namespace {

template <int D>
struct TcCfg {
    static constexpr int kHalves = D / 64;                   // 128-byte column blocks
    // K gets one more stage than V when shared memory allows: K(t+1) is
    // needed half a tile before V(t+1)
    static constexpr int kStagesK = D == 128 ? 3 : 4;
    static constexpr int kStagesV = D == 128 ? 2 : 4;
    static constexpr uint32_t kHalfBytes = kTileN * 128;     // one column block of a tile
    static constexpr uint32_t kTileBytes = kTileN * D * 2;   // a K or V tile
    static constexpr uint32_t kQBytes = kTileM * D * 2;      // a Q tile
    static constexpr uint32_t kOffQ = 0;
    // V stages sit before the K stages: the MN-major V operand is read with
    // the largest descriptor strides, and this keeps every read of it inside
    // the CTA's shared memory.
    static constexpr uint32_t kOffV = kOffQ + kQTiles * kQBytes;
    static constexpr uint32_t kOffK = kOffV + kStagesV * kTileBytes;
    static constexpr uint32_t kOffBar = kOffK + kStagesK * kTileBytes;
    static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 6 + 3;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    static constexpr uint32_t kSmemBytes = kOffMisc + 128 + 1024;
    static_assert(kOffBar % 8 == 0 && kOffMisc % 4 == 0, "smem alignment");
    static_assert(kOffQ % 1024 == 0 && kOffK % 1024 == 0 && kOffV % 1024 == 0,
                  "128-byte-swizzled operands need 1024-byte alignment");
    // barrier indices
    static constexpr int bQFull = 0;
    static constexpr int bKFull = 1;
    static constexpr int bKEmpty = 1 + kStagesK;
    static constexpr int bVFull = 1 + 2 * kStagesK;
    static constexpr int bVEmpty = 1 + 2 * kStagesK + kStagesV;
    static constexpr int bSFull = 1 + 2 * kStagesK + 2 * kStagesV;
    static constexpr int bPFull = bSFull + 2;
    static constexpr int bODone = bSFull + 4;
    static constexpr int bDrain = bSFull + 6;
    static constexpr int bGatherDrain = bSFull + 7;
    static constexpr int bStall = bSFull + 8;  // nothing arrives on it (timeout test)
};

struct Geo {
    int b, g, pos0, c, P, L, q_row0, nq;
    int first[2], last[2];  // KV tile range of each Q tile (first > last: inactive)
    int pl[2], ph[2];       // first / last valid absolute position of each Q tile
    int t_begin, t_end;
};

// Geometry of item `it` of sequence b = it.x, whose qo_indptr[b], [b + 1]
// and prefix length are q0, q1 and P.
template <bool kCausal, bool kSplit>
__device__ __forceinline__ Geo make_geo(const TcParams& p, int4 it, int q0, int q1, int P) {
    Geo g;
    g.b = it.x;
    g.g = it.y;
    g.pos0 = it.z;
    g.c = q1 - q0;
    g.P = P;
    g.L = g.P + g.c;
    g.q_row0 = q0 + g.pos0;
    g.nq = (g.pos0 + p.qpos < g.c) ? 2 : 1;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int start = g.pos0 + u * p.qpos;
        if (start < g.c) {
            g.pl[u] = g.P + start;
            g.ph[u] = g.P + min(start + p.qpos, g.c) - 1;
            const int lo = p.window > 0 ? max(0, g.pl[u] - p.window + 1) : 0;
            g.first[u] = lo / kTileN;
            // causal: up to the tile's last row; otherwise every key of the sequence
            g.last[u] = (kCausal ? g.ph[u] : g.L - 1) / kTileN;
        } else {
            g.pl[u] = g.ph[u] = 0;
            g.first[u] = 1;
            g.last[u] = 0;
        }
    }
    // a part of a split item: its Q tiles' KV ranges end below the item's
    // middle tile tm (part 0) or start at it (part 1).  Items are split only
    // above 16 KV tiles, so tm lies at least 8 tiles inside the item and both
    // Q tiles keep KV tiles in both parts (their ranges differ by at most one
    // tile at either end).
    if constexpr (kSplit) {
        if (it.w & kSplitTag) {
            const int tm = (it.w >> 12) & (kSplitMaxTile - 1);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (it.w & 1) g.first[u] = max(g.first[u], tm);
                else g.last[u] = min(g.last[u], tm - 1);
            }
        }
    }
    g.t_begin = g.first[0];
    g.t_end = g.nq == 2 ? g.last[1] : g.last[0];
    return g;
}

__device__ __forceinline__ bool tile_active(const Geo& g, int u, int t) {
    return g.first[u] <= t && t <= g.last[u];
}

// First slot of the page run one TMA lane loads for a KV tile (num_slots
// when the run is past the sequence end or its page id is bad: the TMA then
// writes zeros).  Read one tile ahead of the load that uses it.
template <int D>
__device__ __forceinline__ int fetch_box_slot(const TcParams& p, const Geo& geo,
                                              const int32_t* pages, int t, int lane) {
    using C = TcCfg<D>;
    const int nsub = kTileN / p.box_rows;
    const int key = t * kTileN + (lane % nsub) * p.box_rows;
    int z = p.num_slots;
    if (lane < nsub * C::kHalves && key < geo.L) {
        const int page = pages[key / p.page_size];
        if (page >= 0 && page < p.num_pages)
            z = page * p.page_size + key % p.page_size;
        else
            report_error(p.dev_err, PCP_ERR_BAD_INDEX);
    }
    return z;
}

// Load one K or V tile (keys [t*128, t*128+128) of sequence b, KV head g)
// by TMA into a 128-byte-swizzled stage: column block h at h * 16 KB, row r at
// r * 128 bytes, 16-byte chunk c of a row at position c ^ (r % 8).  For V, the
// page run holding the sequence end is copied with cp.async and zero-filled
// past the end, so stale pool contents (possibly NaN) never meet P = 0.
template <int D>
__device__ __forceinline__ void tma_kv_tile(const TcParams& p, const Geo& geo, int t, int z,
                                            const CUtensorMap* map, const uint16_t* pool,
                                            uint32_t dst, uint32_t bar, bool zero_tail,
                                            int lane) {
    using C = TcCfg<D>;
    const int key0 = t * kTileN;
    const int br = p.box_rows;
    const int nsub = kTileN / br;
    const int nloads = nsub * C::kHalves;
    int strad = -1;
    if (zero_tail && geo.L > key0 && geo.L < key0 + kTileN && (geo.L - key0) % br != 0)
        strad = (geo.L - key0) / br;
    if (strad >= 0) {
        const int ks = key0 + strad * br;
        const int slot0 = __shfl_sync(0xffffffffu, z, strad);
        const bool bad = slot0 >= p.num_slots;
        for (int idx = lane; idx < br * C::kHalves * 8; idx += 32) {
            const int row = idx / (C::kHalves * 8);
            const int c = idx % (C::kHalves * 8);
            const int rt = strad * br + row;
            const bool ok = !bad && ks + row < geo.L;
            const uint16_t* src =
                ok ? pool + ((int64_t)(slot0 + row) * p.n_kv_heads + geo.g) * D + c * 8 : pool;
            cp_async_16(dst + (c >> 3) * C::kHalfBytes + rt * 128 + (((c & 7) ^ (rt & 7)) << 4),
                        src, ok ? 16u : 0u);
        }
        cp_async_mbar_arrive(bar);
    }
    __syncwarp();
    if (lane == 0)
        mbar_arrive_expect_tx(bar, (uint32_t)(nloads - (strad >= 0 ? C::kHalves : 0)) * br * 128);
    __syncwarp();
    if (lane < nloads) {
        const int sb = lane % nsub;
        const int h = lane / nsub;
        if (sb != strad)
            tma_load_3d(dst + h * C::kHalfBytes + sb * br * 128, map, bar, h * 64, geo.g, z);
    }
}

// Nonzero bytes of a 32-bit word as 4 bits (bit e: byte e is nonzero).
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t w) {
    uint32_t t = w | (w >> 4);
    t |= t >> 2;
    t |= t >> 1;
    t &= 0x01010101u;
    return (t | (t >> 7) | (t >> 14) | (t >> 21)) & 0xFu;
}

// Keep-bits of keys [key0, key0 + 128) of one mask row: bit j of mb[j / 32]
// is set when the mask keeps key key0 + j.  The row starts 16-byte aligned
// (the host checks the base and the strides) and key0 is a multiple of 128;
// keys at or past kv_len read as masked.  A null row is all masked.
__device__ __forceinline__ void mask_bits_128(const uint8_t* mrow, int key0, int kv_len,
                                              uint32_t (&mb)[4]) {
#pragma unroll
    for (int w = 0; w < 4; ++w) mb[w] = 0u;
    if (mrow == nullptr) return;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int k = key0 + c * 16;
        uint32_t bits = 0u;
        if (k + 16 <= kv_len) {
            const uint4 x = __ldg(reinterpret_cast<const uint4*>(mrow + k));
            bits = nonzero_bytes(x.x) | (nonzero_bytes(x.y) << 4) | (nonzero_bytes(x.z) << 8) |
                   (nonzero_bytes(x.w) << 12);
        } else {
            for (int e = 0; e < 16 && k + e < kv_len; ++e)
                if (mrow[k + e]) bits |= 1u << e;
        }
        mb[c >> 1] |= bits << ((c & 1) * 16);
    }
}

// The same 128 keep-bits when every lane of the warp reads one mask row: lane
// l reads keys key0 + 4l .. key0 + 4l + 3 and the warp assembles the words
// with shuffles.
__device__ __forceinline__ void mask_bits_128_warp(const uint8_t* mrow, int key0, int kv_len,
                                                   int lane, uint32_t (&mb)[4]) {
    const int k = key0 + 4 * lane;
    uint32_t nib = 0u;
    if (k + 4 <= kv_len) {
        nib = nonzero_bytes(__ldg(reinterpret_cast<const uint32_t*>(mrow + k)));
    } else {
        for (int e = 0; e < 4 && k + e < kv_len; ++e)
            if (mrow[k + e]) nib |= 1u << e;
    }
    uint32_t part = nib << (4 * (lane & 7));
    part |= __shfl_xor_sync(0xffffffffu, part, 1);
    part |= __shfl_xor_sync(0xffffffffu, part, 2);
    part |= __shfl_xor_sync(0xffffffffu, part, 4);
#pragma unroll
    for (int w = 0; w < 4; ++w) mb[w] = __shfl_sync(0xffffffffu, part, 8 * w);
}

// Bits j of [0, 32) with lo <= j < hi.
__device__ __forceinline__ uint32_t range_bits(int lo, int hi) {
    lo = max(0, min(lo, 32));
    hi = max(0, min(hi, 32));
    const uint32_t below_hi = hi >= 32 ? ~0u : (1u << hi) - 1u;
    const uint32_t below_lo = lo >= 32 ? ~0u : (1u << lo) - 1u;
    return below_hi & ~below_lo;
}

// One gather warp's share (rows [gw * 43, min(128, gw * 43 + 43)) of the
// three warps) of a K or V tile: lanes split into groups covering one 256-byte
// (128-byte for D = 64) row each.
template <int D>
struct GatherShape {
    static constexpr int kChunks = D / 8;                     // 16-byte chunks per row
    static constexpr int kRowsPerInst = 32 / kChunks;         // rows per warp instruction
    static constexpr int kRows = (kTileN + kGatherWarps - 1) / kGatherWarps;  // 43 rows at most
    static constexpr int kInsts = (kRows + kRowsPerInst - 1) / kRowsPerInst;  // instructions
    static_assert(kRows > 32 && kRows <= 64, "two 32-row lookups per gather warp");
};

// sa / sb: the slots of the warp's rows `lane` and `lane + 32` of its share
// (-1: none); the copy lanes of a row take its slot by shuffle.  Rows past
// the share (`nrows`) belong to the next warp and are skipped.
template <int D>
__device__ __forceinline__ void gather_kv_rows(const TcParams& p, const Geo& geo, int sa, int sb,
                                               const uint16_t* pool, uint32_t dst, int gw,
                                               int nrows, int lane) {
    using C = TcCfg<D>;
    using GS = GatherShape<D>;
    const int c = lane % GS::kChunks;
    const int rsub = lane / GS::kChunks;
#pragma unroll
    for (int j = 0; j < GS::kInsts; ++j) {
        const int rw = j * GS::kRowsPerInst + rsub;  // row among the warp's share
        const int slot = __shfl_sync(0xffffffffu, j * GS::kRowsPerInst < 32 ? sa : sb, rw & 31);
        if (rw >= nrows) continue;
        const int row = gw * GS::kRows + rw;
        const bool ok = slot >= 0;
        const uint16_t* src =
            ok ? pool + ((int64_t)slot * p.n_kv_heads + geo.g) * D + c * 8 : pool;
        cp_async_16(dst + (c >> 3) * C::kHalfBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4),
                    src, ok ? 16u : 0u);
    }
}

}  // namespace

// Epilogue of Q tile u of a split item's part, one row per thread (row r of
// the tile).  Each warp (32 rows) settles its rows with the warp holding the
// same rows in the other part, through a ticket and a ready flag of its own,
// so nothing waits on a warp of this CTA that might have given up (only
// warp-level synchronisation).  The warp that takes ticket 0 writes its O
// rows (fp32, unnormalised) and (m, l) in the log2 domain to the item's
// partial buffer and then raises the flag; the other one waits for the flag
// (its partner is past its ticket, so it is running and the wait ends;
// bounded all the same) and writes
//   out = (2^(m_0 - M) O_0 + 2^(m_1 - M) O_1) / (2^(m_0 - M) l_0 + 2^(m_1 - M) l_1),
//   lse = (M + log2 L) ln 2,  M = max(m_0, m_1),
// always with part 0's terms first (explicit fma/mul, no contraction left to
// the compiler), so the result does not depend on which part finished first.
template <int D>
__device__ __forceinline__ void split_epilogue(const TcParams& p, int sp, int part, int u, int r,
                                               uint32_t tO, float m_ref, float l_run,
                                               bool row_valid, int64_t orow) {
    const int lane = r & 31;
    const int64_t pidx = ((int64_t)sp * kQTiles + u) * kTileM + r;
    unsigned char* ws = const_cast<unsigned char*>(p.ws);
    float* po = reinterpret_cast<float*>(ws + p.lay.tc_part_o) + pidx * D;
    float2* pml = reinterpret_cast<float2*>(ws + p.lay.tc_part_ml) + pidx;
    // {ticket, ready} of this warp's rows
    int* sync = reinterpret_cast<int*>(ws + p.lay.tc_sync) +
                (((int64_t)sp * kQTiles + u) * 4 + (r >> 5)) * 2;
    int ticket = 0;
    if (lane == 0) ticket = atomicAdd(sync, 1);
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    if (ticket == 0) {
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            uint32_t o[32];
            tmem_ld32(tO + 32u * i, o);
            tmem_ld_wait();
            float4* dst = reinterpret_cast<float4*>(po + i * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                __stcg(dst + j, make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                            __uint_as_float(o[4 * j + 2]),
                                            __uint_as_float(o[4 * j + 3])));
        }
        __stcg(pml, make_float2(m_ref, l_run));
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(sync + 1, 1);
        return;
    }
    if (lane == 0) {
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu(sync + 1) == 0) {
            if (global_timer_ns() - t0 > kSpinLimitNs) {
                report_error(p.dev_err, PCP_ERR_TIMEOUT);
                break;
            }
        }
    }
    __syncwarp();
    const float2 ot = __ldcg(pml);
    const float M = fmaxf(m_ref, ot.x);
    const float e_s = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - M);
    const float e_o = ot.x == -INFINITY ? 0.f : fast_exp2(ot.x - M);
    // part 0's (weight, normaliser) first
    const float e0 = part == 0 ? e_s : e_o, e1 = part == 0 ? e_o : e_s;
    const float l0 = part == 0 ? l_run : ot.y, l1 = part == 0 ? ot.y : l_run;
    const float L = __fmaf_rn(l0, e0, __fmul_rn(l1, e1));
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float a0 = __fmul_rn(e0, inv), a1 = __fmul_rn(e1, inv);
    // O of part 0 and of part 1 from this part's TMEM row (s) and the partial (x)
    auto mix = [&](float sv, float x) {
        return part == 0 ? __fmaf_rn(sv, a0, __fmul_rn(x, a1)) : __fmaf_rn(x, a0, __fmul_rn(sv, a1));
    };
    uint16_t* op = p.out + orow * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        uint32_t o[32];
        tmem_ld32(tO + 32u * i, o);
        tmem_ld_wait();
        const float4* src = reinterpret_cast<const float4*>(po + i * 32);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 x = __ldcg(src + j);
            w[2 * j] = pack_bf16x2(mix(__uint_as_float(o[4 * j]), x.x),
                                   mix(__uint_as_float(o[4 * j + 1]), x.y));
            w[2 * j + 1] = pack_bf16x2(mix(__uint_as_float(o[4 * j + 2]), x.z),
                                       mix(__uint_as_float(o[4 * j + 3]), x.w));
        }
        if (row_valid) {
            uint4* dst = reinterpret_cast<uint4*>(op + i * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
    }
    if (row_valid && p.lse != nullptr)
        p.lse[orow] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
}

// kMask: the call passes a boolean mask; kCausal: bottom-right causal (else
// every row sees all keys); kGather: the instantiation that holds the
// cp.async gathers for pages below kTmaMinRows keys (it takes TMA page
// boxes too when box_rows > 0; the host launches it only for box_rows 0).
// Separate instantiations, so the plain causal path carries none of the
// other paths' instructions or registers: the gather code alone, never run
// with page boxes, cost the page-box kernel 1-3%, and a gathering
// instantiation without the page-box code spilled and lost 8%.
template <int D, bool kMask, bool kCausal, bool kGather, bool kSplit, bool kPing>
__global__ void __launch_bounds__(kTcThreads, 1)
    extend_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v) {
    using C = TcCfg<D>;
    constexpr int SK = C::kStagesK;
    constexpr int SV = C::kStagesV;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t sQ = base + C::kOffQ;
    const uint32_t sK = base + C::kOffK;
    const uint32_t sV = base + C::kOffV;
    const uint32_t sBar = base + C::kOffBar;
    volatile int* misc = reinterpret_cast<volatile int*>(gbase + C::kOffMisc);
    // misc[0] TMEM base, misc[1] current item, misc[2] abort flag, misc[3] 0;
    // page boxes: misc[4 + 8 s ..]: the next item, its record, its sequence's
    // qo_indptr[b], qo_indptr[b + 1] and prefix length, in slot s = the
    // item's parity (written during the item before, read at its start: the
    // slot is not rewritten before every thread has passed the next start)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::bQFull), 1);
        // TMA path: one arrive.expect_tx; gather path: one arrival per gather lane
        const uint32_t full_count = kGather && p.box_rows == 0 ? 32u * kGatherWarps : 1u;
        // the warps that issue cp.async (or stand by for it) and drain it on
        // the abort path: 10 and 11 with page boxes, 8, 10 and 11 gathering
        const uint32_t drain_count = kGather && p.box_rows == 0 ? 32u * kGatherWarps : 64u;
        for (int s = 0; s < SK; ++s) {
            mbar_init(bar(C::bKFull + s), full_count);
            mbar_init(bar(C::bKEmpty + s), 1);
        }
        for (int s = 0; s < SV; ++s) {
            mbar_init(bar(C::bVFull + s), full_count);
            mbar_init(bar(C::bVEmpty + s), 1);
        }
        for (int u = 0; u < 2; ++u) {
            mbar_init(bar(C::bSFull + u), 1);
            mbar_init(bar(C::bPFull + u), 4);  // one arrival per softmax warp
            mbar_init(bar(C::bODone + u), 1);
        }
        mbar_init(bar(C::bDrain), 1);
        mbar_init(bar(C::bGatherDrain), drain_count);
        mbar_init(bar(C::bStall), 1);
        fence_mbarrier_init();
        misc[2] = 0;
        misc[3] = 0;
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    // the work list is the planner's output
    pdl_wait();
    // a call without tensor-core work (decode rows only) leaves at once
    if (reinterpret_cast<const WsHeader*>(p.ws + p.lay.header)->n_tc_items == 0) return;
    if (warp == kWarpMma) {
        tmem_alloc(smem_addr((const void*)&misc[0]), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];

    WsHeader* hdr = reinterpret_cast<WsHeader*>(const_cast<unsigned char*>(p.ws) + p.lay.header);
    const int n_items = hdr->n_tc_items;
    const int4* items = reinterpret_cast<const int4*>(p.ws + p.lay.tc_items);
    volatile int* abort_flag = &misc[2];
    const int G = p.group;
    const float sl2 = p.scale_log2;

    uint32_t kv_iter = 0;          // KV tiles handled so far by this CTA
    uint32_t act0 = 0u, act1 = 0u;  // active (Q tile, KV tile) pairs so far, per Q tile
    // kPing: S/P rounds per buffer (act0/act1) and O rounds per accumulator
    // (oct0/oct1) differ once a one-Q-tile item alternated its S buffers
    uint32_t oct0 = 0u, oct1 = 0u;
    uint32_t n_done = 0;            // items finished (q_full phase)
    int last_issued = -1;           // TMA-issuing warps: last KV iteration they loaded

    for (;;) {
        // The TMA warp claims the next item and reads its record and metadata
        // during this one (after the item's last K tile, or its last gathered
        // tile), so an item starts without the atomic and the dependent
        // loads; the first item loads them here.
        int item, q0, q1, Pl;
        int4 rec;
        if (n_done == 0) {
            // gathering: the first item of CTA i is item i (the planner starts
            // the counter at the grid size); page boxes: the first item from
            // the counter too (item i there moved the page-box kernel's
            // registers and cost it 1.4%)
            if (threadIdx.x == 0) misc[1] = kGather ? (int)blockIdx.x : atomicAdd(&hdr->tc_next, 1);
            __syncthreads();
            item = misc[1];
            if (item >= n_items || *abort_flag) break;
            rec = items[item];
            q0 = p.qo_indptr[rec.x];
            q1 = p.qo_indptr[rec.x + 1];
            Pl = p.prefix_lens[rec.x];
        } else {
            __syncthreads();
            volatile int* nx = misc + 4 + 8 * (n_done & 1u);
            item = nx[0];
            if (item >= n_items || *abort_flag) break;
            rec = make_int4(nx[1], nx[2], nx[3], nx[4]);
            q0 = nx[5];
            q1 = nx[6];
            Pl = nx[7];
        }
        const Geo geo = make_geo<kCausal, kSplit>(p, rec, q0, q1, Pl);
        const int ntiles = geo.t_end - geo.t_begin + 1;

        // Page boxes: the TMA warp issues the K tiles and the first gather warp
        // the V tiles.  The TMA unit accepts a warp's boxes one lane after the
        // other (about 140 cycles per 2 KB box), so two issuing warps double
        // the rate at which small pages arrive.
        if (warp == kWarpTma || warp >= kWarpGather0) {
            if (warp == kWarpTma && lane == 0) {  // Q, by TMA on both paths
                mbar_arrive_expect_tx(bar(C::bQFull),
                                      (uint32_t)(geo.nq * C::kHalves * G * p.qpos * 128));
                for (int u = 0; u < geo.nq; ++u)
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(sQ + u * C::kQBytes + h * (kTileM * 128), &tm_q,
                                    bar(C::bQFull), h * 64, geo.g * G, geo.q_row0 + u * p.qpos);
            }
            if (!kGather || p.box_rows > 0) {
                // ------------------------------------------------ TMA: K / V page boxes
                const bool is_k = warp == kWarpTma;
                if (warp == kWarpTma || warp == kWarpGather0) {
                    const int32_t* pages = p.kv_indices + p.kv_indptr[geo.b];
                    int z_cur = fetch_box_slot<D>(p, geo, pages, geo.t_begin, lane);
                    for (int i = 0; i < ntiles; ++i) {
                        const int t = geo.t_begin + i;
                        const uint32_t cur = kv_iter + i;
                        // the next tile's page ids are in flight while this one waits
                        const int z_next =
                            i + 1 < ntiles ? fetch_box_slot<D>(p, geo, pages, t + 1, lane) : z_cur;
                        // every wait is decided for the whole warp: the box issue
                        // below has warp-collective steps
                        if (is_k) {
                            const int sk = cur % SK;
                            if (!__all_sync(0xffffffffu,
                                            mbar_wait(bar(C::bKEmpty + sk), ((cur / SK) & 1u) ^ 1u,
                                                      abort_flag, p.dev_err, kSpinLimitNs)))
                                break;
                            tma_kv_tile<D>(p, geo, t, z_cur, &tm_k, p.k_pool,
                                           sK + sk * C::kTileBytes, bar(C::bKFull + sk), false,
                                           lane);
                        } else {
                            const int sv = cur % SV;
                            if (!__all_sync(0xffffffffu,
                                            mbar_wait(bar(C::bVEmpty + sv), ((cur / SV) & 1u) ^ 1u,
                                                      abort_flag, p.dev_err, kSpinLimitNs)))
                                break;
                            tma_kv_tile<D>(p, geo, t, z_cur, &tm_v, p.v_pool,
                                           sV + sv * C::kTileBytes, bar(C::bVFull + sv), true,
                                           lane);
                        }
                        last_issued = (int)cur;
                        z_cur = z_next;
                    }
                    // The next item, claimed once this item's last K tile is
                    // issued: a few tile steps before this item ends, late
                    // enough that the longest-first queue stays greedy (a claim
                    // at the item's start cost items-poor launches 20%), early
                    // enough that the claim and its loads are done by then.
                    if constexpr (!kGather) {
                        if (is_k && lane == 0) {
                            volatile int* nx = misc + 4 + 8 * ((n_done + 1u) & 1u);
                            const int ni = atomicAdd(&hdr->tc_next, 1);
                            nx[0] = ni;
                            if (ni < n_items) {
                                const int4 r = items[ni];
                                nx[1] = r.x;
                                nx[2] = r.y;
                                nx[3] = r.z;
                                nx[4] = r.w;
                                nx[5] = p.qo_indptr[r.x];
                                nx[6] = p.qo_indptr[r.x + 1];
                                nx[7] = p.prefix_lens[r.x];
                            }
                        }
                    }
                }
            } else {
                // ------------------------------------------------ cp.async page gathers
                // warps 10, 11 and 8 each copy a third of the rows of every K and
                // V tile (three warps issuing cp.async in parallel)
                {
                    using GS = GatherShape<D>;
                    const int gw = warp == kWarpTma ? 2 : warp - kWarpGather0;
                    const int nrows = min(GS::kRows, kTileN - gw * GS::kRows);
                    const int32_t* pages = p.kv_indices + p.kv_indptr[geo.b];
                    // Slot of key `key` (-1 past the sequence end or for a bad page).
                    auto slot_of = [&](int key) {
                        int slot = -1;
                        if (key < geo.L) {
                            const int entry = p.page_shift >= 0 ? key >> p.page_shift
                                                                : key / p.page_size;
                            const int page = pages[entry];
                            if (page >= 0 && page < p.num_pages)
                                slot = page * p.page_size + (key - entry * p.page_size);
                            else
                                report_error(p.dev_err, PCP_ERR_BAD_INDEX);
                        }
                        return slot;
                    };
                    // The warp's rows of tile t: lane l looks up rows l and l + 32
                    // of its share (consecutive page-table entries, one coalesced
                    // load each), one tile ahead of their use; a row's copy lanes
                    // take its slot by shuffle.
                    const int row0 = gw * GS::kRows;
                    const bool hi_ok = 32 + lane < nrows;
                    int sa = slot_of(geo.t_begin * kTileN + row0 + lane);
                    int sb = hi_ok ? slot_of(geo.t_begin * kTileN + row0 + 32 + lane) : -1;
                    for (int i = 0; i < ntiles; ++i) {
                        const int t = geo.t_begin + i;
                        const uint32_t cur = kv_iter + i;
                        const int sk = cur % SK, sv = cur % SV;
                        const int ca = sa, cb = sb;
                        if (i + 1 < ntiles) {  // the next tile's lookups are in flight meanwhile
                            sa = slot_of((t + 1) * kTileN + row0 + lane);
                            sb = hi_ok ? slot_of((t + 1) * kTileN + row0 + 32 + lane) : -1;
                        }
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(bar(C::bKEmpty + sk), ((cur / SK) & 1u) ^ 1u,
                                                  abort_flag, p.dev_err, kSpinLimitNs)))
                            break;
                        gather_kv_rows<D>(p, geo, ca, cb, p.k_pool, sK + sk * C::kTileBytes, gw,
                                          nrows, lane);
                        cp_async_mbar_arrive_noinc(bar(C::bKFull + sk));
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(bar(C::bVEmpty + sv), ((cur / SV) & 1u) ^ 1u,
                                                  abort_flag, p.dev_err, kSpinLimitNs)))
                            break;
                        gather_kv_rows<D>(p, geo, ca, cb, p.v_pool, sV + sv * C::kTileBytes, gw,
                                          nrows, lane);
                        cp_async_mbar_arrive_noinc(bar(C::bVFull + sv));
                    }
                    // the next item claimed once this one's last tile is issued,
                    // as on the page-box path
                    if (warp == kWarpTma && lane == 0) {
                        volatile int* nx = misc + 4 + 8 * ((n_done + 1u) & 1u);
                        const int ni = atomicAdd(&hdr->tc_next, 1);
                        nx[0] = ni;
                        if (ni < n_items) {
                            const int4 r = items[ni];
                            nx[1] = r.x;
                            nx[2] = r.y;
                            nx[3] = r.z;
                            nx[4] = r.w;
                            nx[5] = p.qo_indptr[r.x];
                            nx[6] = p.qo_indptr[r.x + 1];
                            nx[7] = p.prefix_lens[r.x];
                        }
                    }
                }
            }
        } else if (warp == kWarpMma) {
            // ------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t idesc_qk = idesc_bf16_f32(kTileM, kTileN, false);
                constexpr uint32_t idesc_pv = idesc_bf16_f32(kTileM, D, true);
                // Descriptors are built once; a k-step, Q tile or stage only moves the
                // start address, which sits in the low 14 bits in 16-byte units.
                const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
                const uint64_t dk = sdesc_sw128(sK, 16, 1024);
                const uint64_t dv = sdesc_sw128(sV, C::kHalfBytes, 1024);
                auto issue_qk = [&](int u, int st) {
                    const uint64_t a0 = dq + ((uint32_t)u * C::kQBytes >> 4);
                    const uint64_t b0 = dk + ((uint32_t)st * C::kTileBytes >> 4);
                    const uint32_t d = tmem + (uint32_t)u * 128u;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        constexpr uint32_t kHalf16 = (kTileM * 128) >> 4;
                        const uint32_t off = (uint32_t)(kk >> 2) * kHalf16 + (uint32_t)(kk & 3) * 2u;
                        umma_ss(d, a0 + off, b0 + off, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                };
                auto issue_pv = [&](int u, int st, bool acc) {
                    const uint64_t b0 = dv + ((uint32_t)st * C::kTileBytes >> 4);
                    const uint32_t d = tmem + 256u + (uint32_t)u * 128u;
                    const uint32_t a = tmem + (uint32_t)u * 128u;
#pragma unroll
                    for (int kk = 0; kk < kTileN / 16; ++kk)
                        umma_ts(d, a + kk * 8, b0 + (uint32_t)kk * (2048u >> 4), idesc_pv,
                                (acc || kk > 0) ? 1u : 0u);
                };
                // the timeout test: the CTA's first wait is one nothing ends
                bool ok = p.stall_ns == 0 || n_done > 0 ||
                          mbar_wait(bar(C::bStall), 0u, abort_flag, p.dev_err, p.stall_ns);
                ok = ok && mbar_wait(bar(C::bQFull), n_done & 1u, abort_flag, p.dev_err,
                                     kSpinLimitNs);
                uint32_t aidx0 = act0, aidx1 = act1;
                bool pp = false;  // a one-Q-tile item alternating its S/P buffers
                if constexpr (kPing) pp = geo.nq == 1;
                if constexpr (kPing) {
                    if (pp) {
                        // Q tile 0 only: the QK^T of KV tile i goes to S buffer i % 2,
                        // two tiles ahead of its PV, so the softmax of tile i + 1 finds
                        // its S ready while PV(i) runs
                        auto qk_to = [&](int sbuf, int st) {
                            const uint64_t b0 = dk + ((uint32_t)st * C::kTileBytes >> 4);
                            const uint32_t d = tmem + (uint32_t)sbuf * 128u;
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                constexpr uint32_t kHalf16 = (kTileM * 128) >> 4;
                                const uint32_t off =
                                    (uint32_t)(kk >> 2) * kHalf16 + (uint32_t)(kk & 3) * 2u;
                                umma_ss(d, dq + off, b0 + off, idesc_qk, kk > 0 ? 1u : 0u);
                            }
                        };
                        auto pv_from = [&](int sbuf, int st, bool acc) {
                            const uint64_t b0 = dv + ((uint32_t)st * C::kTileBytes >> 4);
                            const uint32_t d = tmem + 256u;
                            const uint32_t a = tmem + (uint32_t)sbuf * 128u;
#pragma unroll
                            for (int kk = 0; kk < kTileN / 16; ++kk)
                                umma_ts(d, a + kk * 8, b0 + (uint32_t)kk * (2048u >> 4), idesc_pv,
                                        (acc || kk > 0) ? 1u : 0u);
                        };
                        if (ok) {
                            tc_fence_after();
                            const int npro = ntiles < 2 ? ntiles : 2;
                            for (int i = 0; ok && i < npro; ++i) {
                                const uint32_t c = kv_iter + (uint32_t)i;
                                ok = mbar_wait(bar(C::bKFull + c % SK), (c / SK) & 1u, abort_flag,
                                               p.dev_err, kSpinLimitNs);
                                if (ok) {
                                    if (kGather && p.box_rows == 0) fence_proxy_async_smem();
                                    qk_to(i, c % SK);
                                    umma_commit(bar(C::bSFull + i));
                                    umma_commit(bar(C::bKEmpty + c % SK));
                                }
                            }
                        }
                        for (int i = 0; ok && i < ntiles; ++i) {
                            const int t = geo.t_begin + i;
                            const uint32_t cur = kv_iter + (uint32_t)i;
                            const int st = cur % SV;
                            if (!mbar_wait(bar(C::bVFull + st), (cur / SV) & 1u, abort_flag,
                                           p.dev_err, kSpinLimitNs)) {
                                ok = false;
                                break;
                            }
                            if ((kGather && p.box_rows == 0) ||
                                (geo.L > t * kTileN && geo.L < t * kTileN + kTileN &&
                                 (geo.L - t * kTileN) % p.box_rows != 0))
                                fence_proxy_async_smem();
                            const int sbuf = i & 1;
                            const uint32_t pr = sbuf ? aidx1 : aidx0;
                            if (!mbar_wait(bar(C::bPFull + sbuf), pr & 1u, abort_flag, p.dev_err,
                                           kSpinLimitNs)) {
                                ok = false;
                                break;
                            }
                            if (sbuf) ++aidx1;
                            else ++aidx0;
                            tc_fence_after();
                            pv_from(sbuf, st, i > 0);
                            umma_commit(bar(C::bODone + 0));
                            umma_commit(bar(C::bVEmpty + st));
                            if (i + 2 < ntiles) {
                                const uint32_t c = cur + 2u;
                                if (!mbar_wait(bar(C::bKFull + c % SK), (c / SK) & 1u, abort_flag,
                                               p.dev_err, kSpinLimitNs)) {
                                    ok = false;
                                    break;
                                }
                                if (kGather && p.box_rows == 0) fence_proxy_async_smem();
                                qk_to(sbuf, c % SK);
                                umma_commit(bar(C::bSFull + sbuf));
                                umma_commit(bar(C::bKEmpty + c % SK));
                            }
                        }
                    }
                }
                if (ok && !pp) {
                    tc_fence_after();
                    const uint32_t c0 = kv_iter;
                    ok = mbar_wait(bar(C::bKFull + c0 % SK), (c0 / SK) & 1u, abort_flag,
                                   p.dev_err, kSpinLimitNs);
                    if (ok) {
                        if (kGather && p.box_rows == 0) fence_proxy_async_smem();
                        if (tile_active(geo, 0, geo.t_begin)) {
                            issue_qk(0, c0 % SK);
                            umma_commit(bar(C::bSFull + 0));
                        }
                        if (tile_active(geo, 1, geo.t_begin)) {
                            issue_qk(1, c0 % SK);
                            umma_commit(bar(C::bSFull + 1));
                        }
                        umma_commit(bar(C::bKEmpty + c0 % SK));
                    }
                }
                for (int i = 0; ok && !pp && i < ntiles; ++i) {
                    const int t = geo.t_begin + i;
                    const uint32_t cur = kv_iter + i;
                    const int st = cur % SV;
                    if (!mbar_wait(bar(C::bVFull + st), (cur / SV) & 1u, abort_flag, p.dev_err,
                                   kSpinLimitNs)) {
                        ok = false;
                        break;
                    }
                    // cp.async wrote part of this V tile: small pages, or the page
                    // run that holds the sequence end (zero-filled past it)
                    if ((kGather && p.box_rows == 0) ||
                        (geo.L > t * kTileN && geo.L < t * kTileN + kTileN &&
                         (geo.L - t * kTileN) % p.box_rows != 0))
                        fence_proxy_async_smem();
                    const bool has_next = i + 1 < ntiles;
                    const int nst = (cur + 1) % SK;
                    bool k_next = false;
                    // PV of Q tile u for this KV tile, then its QK^T for the next one
                    auto step_u = [&](const int u, uint32_t& ai, const int first_u) -> bool {
                        if (tile_active(geo, u, t)) {
                            if (!mbar_wait(bar(C::bPFull + u), ai & 1u, abort_flag, p.dev_err,
                                           kSpinLimitNs))
                                return false;
                            tc_fence_after();
                            issue_pv(u, st, t != first_u);
                            umma_commit(bar(C::bODone + u));
                            ++ai;
                        }
                        if (has_next && tile_active(geo, u, t + 1)) {
                            if (!k_next) {
                                if (!mbar_wait(bar(C::bKFull + nst), ((cur + 1) / SK) & 1u,
                                               abort_flag, p.dev_err, kSpinLimitNs))
                                    return false;
                                if (kGather && p.box_rows == 0) fence_proxy_async_smem();
                                k_next = true;
                            }
                            issue_qk(u, nst);
                            umma_commit(bar(C::bSFull + u));
                        }
                        return true;
                    };
                    if (!step_u(0, aidx0, geo.first[0]) || !step_u(1, aidx1, geo.first[1])) {
                        ok = false;
                        break;
                    }
                    umma_commit(bar(C::bVEmpty + st));
                    if (k_next) umma_commit(bar(C::bKEmpty + nst));
                }
            }
            __syncwarp();
        } else {
            // ------------------------------------------------ softmax + epilogue
            const int u = warp >> 2;
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
            const uint32_t tS = tmem + lane_off + (uint32_t)u * 128u;
            const uint32_t tO = tmem + lane_off + 256u + (uint32_t)u * 128u;
            if (u < geo.nq) {
                const int first_u = u == 0 ? geo.first[0] : geo.first[1];
                const int last_u = u == 0 ? geo.last[0] : geo.last[1];
                const int pl_u = u == 0 ? geo.pl[0] : geo.pl[1];
                const int ph_u = u == 0 ? geo.ph[0] : geo.ph[1];
                const uint32_t act_u = u == 0 ? act0 : act1;
                // kPing: O rounds of this Q tile's accumulator, and whether the
                // item alternates S/P buffers 0 and 1 over its KV tiles
                const uint32_t oct_u = kPing ? (u == 0 ? oct0 : oct1) : act_u;
                bool pp = false;
                if constexpr (kPing) pp = geo.nq == 1;
                const int pos_local = u * p.qpos + r / G;
                const bool row_valid = r < p.qpos * G && geo.pos0 + pos_local < geo.c;
                const int pabs = geo.P + geo.pos0 + pos_local;
                const int head = geo.g * G + r % G;
                float m_run = -INFINITY, l_run = 0.f;
                bool ok = true;
                for (int t = first_u; t <= last_u; ++t) {
                    const uint32_t a = act_u + (uint32_t)(t - first_u);
                    // S/P buffer, its round, this tile's O round, its S columns
                    uint32_t sb = (uint32_t)u, sa = a, oa = a, tSi = tS;
                    if constexpr (kPing) {
                        const uint32_t i = (uint32_t)(t - first_u);
                        oa = oct_u + i;
                        if (pp) {
                            sb = i & 1u;
                            sa = (sb ? act1 : act0) + (i >> 1);
                            tSi = tmem + lane_off + sb * 128u;
                        }
                    }
                    const int key0 = t * kTileN;
                    constexpr bool has_mask = kMask;
                    // causal: the diagonal and window-edge tiles; otherwise the
                    // tile holding the sequence end; with a mask, every tile
                    const bool need_mask =
                        has_mask ||
                        (kCausal ? (key0 + kTileN - 1 > pl_u) ||
                                        (p.window > 0 && key0 < ph_u - p.window + 1)
                                  : key0 + kTileN > geo.L);
                    // keep-bits of this row's keys in the tile (bit j of mb[j / 32]):
                    // the boolean mask's entries, and'ed with the causal / length
                    // range, so each key costs one bit test.  They do not depend
                    // on S: their loads are issued before the wait for S, so the
                    // load latency overlaps the QK^T MMA.
                    uint32_t mb[4] = {~0u, ~0u, ~0u, ~0u};
                    if constexpr (has_mask) {
                        if (p.mask.h_stride == 0 && p.mask.q_stride == 0) {
                            // one mask row for the whole tile: the warp builds it
                            const uint8_t* mrow =
                                p.mask.data + (int64_t)geo.b * p.mask.b_stride;
                            mask_bits_128_warp(mrow, key0, p.mask.kv_len, lane, mb);
                        } else {
                            const int qi = geo.pos0 + pos_local;
                            const bool in_mask =
                                row_valid && (p.mask.q_stride == 0 || qi < p.mask.q_len);
                            const uint8_t* mrow =
                                in_mask ? p.mask.data + (int64_t)geo.b * p.mask.b_stride +
                                              (int64_t)head * p.mask.h_stride +
                                              (int64_t)qi * p.mask.q_stride
                                        : nullptr;
                            mask_bits_128(mrow, key0, p.mask.kv_len, mb);
                        }
                        // visible key range of the row in tile coordinates
                        const int hi = kCausal ? pabs - key0 + 1 : geo.L - key0;
                        const int lo = kCausal && p.window > 0 ? pabs - p.window + 1 - key0 : 0;
#pragma unroll
                        for (int w = 0; w < 4; ++w) mb[w] &= range_bits(lo - 32 * w, hi - 32 * w);
                    }
                    // waits decide per warp (tcgen05.ld/st and the P arrival are
                    // warp-collective)
                    if (!__all_sync(0xffffffffu, mbar_wait(bar(C::bSFull + sb), sa & 1u, abort_flag,
                                                           p.dev_err, kSpinLimitNs))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the whole S row of this thread: one TMEM load
                    uint32_t v[128];
                    tmem_ld128(tSi, v);
                    tmem_ld_wait();
                    if (need_mask) {
                        // keys this row does not see become -inf: tile columns
                        // [lo, hi) are visible
                        const int hi = kCausal ? pabs - key0 + 1 : geo.L - key0;
                        const int lo = kCausal && p.window > 0 ? pabs - p.window + 1 - key0 : 0;
#pragma unroll
                        for (int j = 0; j < 128; ++j) {
                            bool vis;
                            if constexpr (has_mask) {
                                vis = (mb[j >> 5] >> (j & 31)) & 1u;
                            } else {
                                vis = j < hi && j >= lo;
                            }
                            if (!vis) v[j] = __float_as_uint(-INFINITY);
                        }
                    }
                    // row maximum: eight independent chains of 3-input max
                    float mx8[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 128; j += 2)
                        mx8[(j >> 1) & 7] = max3f(mx8[(j >> 1) & 7], __uint_as_float(v[j]),
                                                  __uint_as_float(v[j + 1]));
                    const float mx = max3f(max3f(mx8[0], mx8[1], mx8[2]),
                                           max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
                    const float m_new = fmaxf(m_run, mx);
                    float alpha = 1.f;
                    bool resc = false;
                    if (m_run == -INFINITY) {
                        m_run = m_new;
                    } else if ((m_new - m_run) * sl2 > 8.f) {
                        alpha = fast_exp2((m_run - m_new) * sl2);
                        m_run = m_new;
                        resc = true;
                    }
                    const float nref = m_run == -INFINITY ? 0.f : -m_run * sl2;
                    // P = exp2(s * scale * log2e - m): packed scale-and-subtract, MUFU
                    // ex2 (MUFU), packed row sums, bf16 pairs (P column c holds keys
                    // 2c, 2c+1)
                    const uint64_t sl2x2 = f2(sl2, sl2), nref2 = f2(nref, nref);
                    uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
                    uint32_t pk[64];
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const uint64_t x = fma_f2(f2(__uint_as_float(v[2 * c]),
                                                     __uint_as_float(v[2 * c + 1])),
                                                  sl2x2, nref2);
                        const uint64_t e = f2(fast_exp2(f2_lo(x)), fast_exp2(f2_hi(x)));
                        acc2[c & 3] = add_f2(acc2[c & 3], e);
                        pk[c] = pack_bf16x2(f2_lo(e), f2_hi(e));
                        // P goes to TMEM in 16-column pieces while the rest is computed
                        if ((c & 15) == 15) tmem_st16(tSi + (uint32_t)(c - 15), &pk[c - 15]);
                    }
                    if (t > first_u) {
                        if (!__all_sync(0xffffffffu,
                                        mbar_wait(bar(C::bODone + u), (oa - 1u) & 1u, abort_flag,
                                                  p.dev_err, kSpinLimitNs))) {
                            tmem_st_wait();
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                            for (int i = 0; i < D / 32; ++i) {
                                uint32_t o[32];
                                tmem_ld32(tO + 32u * i, o);
                                tmem_ld_wait();
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                                tmem_st32(tO + 32u * i, o);
                            }
                        }
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    // one arrival per warp once all its lanes' P is in TMEM
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::bPFull + sb));
                    // the row sum is off the MMA's critical path
                    const uint64_t acc = add_f2(add_f2(acc2[0], acc2[1]), add_f2(acc2[2], acc2[3]));
                    l_run = l_run * alpha + (f2_lo(acc) + f2_hi(acc));
                }
                if (ok) {
                    const uint32_t a_last = oct_u + (uint32_t)(last_u - first_u);
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(C::bODone + u), a_last & 1u,
                                                           abort_flag, p.dev_err, kSpinLimitNs));
                }
                // a part of a split item merges with the other part (its split
                // state is read from the item again, not kept live through the
                // tile loop)
                int wsplit = 0;
                if constexpr (kSplit) {
                    wsplit = n_done > 0 ? misc[4 + 8 * (n_done & 1u) + 4] : items[misc[1]].w;
                    if (!(wsplit & kSplitTag)) wsplit = 0;
                }
                if (ok && wsplit != 0) {
                    tc_fence_after();
                    split_epilogue<D>(p, (wsplit >> 1) & 0x7FF, wsplit & 1, u, r, tO,
                                      m_run == -INFINITY ? -INFINITY : m_run * sl2, l_run,
                                      row_valid,
                                      (int64_t)(geo.q_row0 + pos_local) * p.n_q_heads + head);
                } else if (ok) {
                    tc_fence_after();
                    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                    const int64_t orow = (int64_t)(geo.q_row0 + pos_local) * p.n_q_heads + head;
                    uint16_t* op = p.out + orow * D;
#pragma unroll
                    for (int i = 0; i < D / 32; ++i) {
                        uint32_t o[32];
                        tmem_ld32(tO + 32u * i, o);
                        tmem_ld_wait();
                        uint32_t w[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv,
                                               __uint_as_float(o[2 * j + 1]) * inv);
                        if (row_valid) {
                            uint4* dst = reinterpret_cast<uint4*>(op + i * 32);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2],
                                                    w[4 * j + 3]);
                        }
                    }
                    if (row_valid && p.lse != nullptr)
                        p.lse[orow] = l_run > 0.f ? (m_run * sl2 + __log2f(l_run)) * 0.69314718055994531f
                                                  : -INFINITY;
                }
            }
        }
        kv_iter += (uint32_t)ntiles;
        if constexpr (kPing) {
            const uint32_t n0 = (uint32_t)(geo.last[0] - geo.first[0] + 1);
            if (geo.nq == 1) {  // S/P buffers alternated; every PV went to O0
                act0 += (n0 + 1u) / 2u;
                act1 += n0 / 2u;
                oct0 += n0;
            } else {
                const uint32_t n1 = (uint32_t)(geo.last[1] - geo.first[1] + 1);
                act0 += n0;
                oct0 += n0;
                act1 += n1;
                oct1 += n1;
            }
        } else {
            act0 += (uint32_t)(geo.last[0] - geo.first[0] + 1);
            if (geo.nq == 2) act1 += (uint32_t)(geo.last[1] - geo.first[1] + 1);
        }
        ++n_done;
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }

    // ---------------------------------------------------------- teardown
    // no work left here: the next kernel on the stream may start launching
    pdl_launch_dependents();
    const bool aborted = *abort_flag != 0;
    // drain waits are never cut short by the abort flag: they watch misc[3],
    // which stays 0, and run to their own limit
    volatile int* no_abort = &misc[3];
    if (warp == kWarpTma || warp >= kWarpGather0) {
        cp_async_wait_all();
        if (aborted && (warp >= kWarpGather0 || (kGather && p.box_rows == 0))) {
            // the mbarrier arrivals the gathers' cp.async copies trigger have
            // been made once this one, triggered after all of them, lands
            cp_async_mbar_arrive_noinc(bar(C::bGatherDrain));
            if (warp == kWarpGather0 && lane == 0)
                mbar_wait(bar(C::bGatherDrain), 0u, no_abort, p.dev_err, kSpinLimitNs);
            __syncwarp();
        }
        if (aborted && lane == 0) {
            // let every TMA load this warp issued land before the CTA exits
            if (warp == kWarpTma && n_done > 0)
                mbar_wait(bar(C::bQFull), (n_done - 1) & 1u, no_abort, p.dev_err, kSpinLimitNs);
            if (warp == kWarpTma)
                for (int it = last_issued - SK + 1; it <= last_issued; ++it)
                    if (it >= 0)
                        mbar_wait(bar(C::bKFull + it % SK), ((uint32_t)it / SK) & 1u, no_abort,
                                  p.dev_err, kSpinLimitNs);
            if (warp == kWarpGather0)
                for (int it = last_issued - SV + 1; it <= last_issued; ++it)
                    if (it >= 0)
                        mbar_wait(bar(C::bVFull + it % SV), ((uint32_t)it / SV) & 1u, no_abort,
                                  p.dev_err, kSpinLimitNs);
        }
    } else if (warp == kWarpMma && lane == 0) {
        // every MMA (and its mbarrier arrivals) completes before TMEM is freed
        umma_commit(bar(C::bDrain));
        mbar_wait(bar(C::bDrain), 0u, no_abort, p.dev_err, kSpinLimitNs);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

size_t tc_smem_bytes(int head_dim) {
    return head_dim == 128 ? TcCfg<128>::kSmemBytes : TcCfg<64>::kSmemBytes;
}

template <int D, bool kMask, bool kCausal, bool kGather, bool kSplit, bool kPing>
cudaError_t launch_extend_tc_s(int grid, cudaStream_t stream, const TcParams& p,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv) {
    const size_t smem = TcCfg<D>::kSmemBytes;
    auto* kern = extend_tc_kernel<D, kMask, kCausal, kGather, kSplit, kPing>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kTcThreads), smem, stream, p, tq, tk, tv);
}

// a plan with split items (never with a mask) takes the instantiation that
// merges them; a causal unmasked call with one-Q-tile items (the host's
// decision, p.ping) the one that alternates their S/P buffers, split items
// or not
template <int D, bool kMask, bool kCausal, bool kGather>
cudaError_t launch_extend_tc_g(int grid, cudaStream_t stream, const TcParams& p,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv) {
    if constexpr (!kMask) {
        if (p.split) {
            // (with page boxes only: the gathering one spilled 36 / 92 bytes and
            // lost 5% on the page-size-1 stress batch)
            if constexpr (kCausal && !kGather) {
                if (p.ping)
                    return launch_extend_tc_s<D, kMask, kCausal, kGather, true, true>(
                        grid, stream, p, tq, tk, tv);
            }
            return launch_extend_tc_s<D, kMask, kCausal, kGather, true, false>(grid, stream, p,
                                                                              tq, tk, tv);
        }
        if constexpr (kCausal) {
            if (p.ping)
                return launch_extend_tc_s<D, kMask, kCausal, kGather, false, true>(grid, stream, p,
                                                                                  tq, tk, tv);
        }
    }
    return launch_extend_tc_s<D, kMask, kCausal, kGather, false, false>(grid, stream, p, tq, tk,
                                                                        tv);
}

// pages below kTmaMinRows keys (box_rows 0) take the gathering instantiation
template <int D, bool kMask, bool kCausal>
cudaError_t launch_extend_tc_t(int grid, cudaStream_t stream, const TcParams& p,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv) {
    return p.box_rows > 0
               ? launch_extend_tc_g<D, kMask, kCausal, false>(grid, stream, p, tq, tk, tv)
               : launch_extend_tc_g<D, kMask, kCausal, true>(grid, stream, p, tq, tk, tv);
}

template <int D>
cudaError_t launch_extend_tc_d(int grid, cudaStream_t stream, const TcParams& p,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv) {
    const bool mask = p.mask.data != nullptr;
    if (p.causal)
        return mask ? launch_extend_tc_t<D, true, true>(grid, stream, p, tq, tk, tv)
                    : launch_extend_tc_t<D, false, true>(grid, stream, p, tq, tk, tv);
    return mask ? launch_extend_tc_t<D, true, false>(grid, stream, p, tq, tk, tv)
                : launch_extend_tc_t<D, false, false>(grid, stream, p, tq, tk, tv);
}

cudaError_t launch_extend_tc(int head_dim, int grid, cudaStream_t stream, const TcParams& p,
                             const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv) {
    return head_dim == 128 ? launch_extend_tc_d<128>(grid, stream, p, tq, tk, tv)
                           : launch_extend_tc_d<64>(grid, stream, p, tq, tk, tv);
}

}  // namespace pcp
