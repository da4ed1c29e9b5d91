// Shared host/device definitions: tile sizes, the workspace layout, work-item
// formats and kernel parameter blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "pcp.h"

namespace pcp {

// ---- tensor-core extend kernel geometry
constexpr int kTileM = 128;       // query rows per Q tile (tcgen05 M)
constexpr int kTileN = 128;       // keys per KV tile
constexpr int kQTiles = 2;        // Q tiles per work item (share each K/V tile)
constexpr int kTcThreads = 384;   // 2 x 4 softmax warps, TMA warp, MMA warp, 2 gather warps
constexpr int kWarpTma = 8;       // Q (and the K page boxes) by TMA
constexpr int kWarpMma = 9;       // one thread issues tcgen05.mma
constexpr int kWarpGather0 = 10;  // warps 10, 11 (and the TMA warp): cp.async page gathers of K/V
constexpr int kGatherWarps = 3;   // gathering warps on the cp.async path: 10, 11 and 8
// Pages whose runs inside a 128-key tile hold at least this many keys are
// loaded by TMA boxes; smaller ones by the cp.async gather warps (below 8
// rows the TMA unit's per-box cost dominates; above, TMA out-runs them).
constexpr int kTmaMinRows = 8;

// ---- CUDA-core row kernel (decode-shaped rows, split-KV)
constexpr int kRowMaxRows = 16;   // query rows (positions x heads) per row item
constexpr int kRowTile = 128;     // keys per row-kernel tile
constexpr int kRowThreads = 160;      // 4 consumer warps + 1 load warp
constexpr int kRowMaxCtas = 512;       // row-kernel CTAs at most (one per SM below that)
// A call whose chunks are all decode-shaped (known from the host copy of
// qo_indptr) and that has at most this many sequences is planned inside the
// row kernel: every CTA builds the split in shared memory, no planner launch.
constexpr int kRowSelfPlanMaxSeqs = 512;

// Default limit of the kernels' bounded pipeline waits, and the fixed limit of
// the waits that drain a CTA's in-flight copies and MMAs before it exits
// (nanoseconds).
constexpr uint64_t kSpinLimitNs = 2000000000ull;

// A sequence's chunk goes to the row kernel when its rows (chunk_len * G)
// fit one row item and G <= kRowMaxRows; everything else to the tensor cores.
__host__ __device__ inline int row_path_max_chunk(int group) {
    return group <= kRowMaxRows ? (kRowMaxRows / group) : 0;
}

__host__ __device__ inline int q_positions_per_tile(int group) { return kTileM / group; }

// Whether a call with tensor-core work takes its decode-shaped chunks onto
// the tensor cores as one-Q-tile items: the longest of them (w: 4/5 of its
// KV tiles, rounded up, in two-Q-tile steps) within 1.1 times the larger of
// the longest prompt item and the average work per SM.  w_tc / max_tc: the
// prompt items' summed and largest cost in KV tiles; w_dec / max_dec: the
// decode-shaped items' weighted ones (per KV head included in the sums).
__host__ __device__ inline int dec_weight(int tiles) { return (4 * tiles + 4) / 5; }
__host__ __device__ inline bool absorb_decode_rows(unsigned long long w_tc, int max_tc,
                                                   unsigned long long w_dec, int max_dec,
                                                   int sm_count) {
    if (w_tc == 0 || w_dec == 0) return false;
    // 10 * max_dec <= 11 * max(max_tc, (w_tc + w_dec) / sms), in integers
    const unsigned long long sms = sm_count > 0 ? (unsigned long long)sm_count : 1ull;
    const unsigned long long lhs = 10ull * (unsigned long long)max_dec * sms;
    const unsigned long long a = 11ull * (unsigned long long)max_tc * sms;
    const unsigned long long b = 11ull * (w_tc + w_dec);
    return lhs <= (a > b ? a : b);
}

// Whether a call splits its longest tensor-core items in two: its longest
// item (in two-Q-tile steps, as absorb_decode_rows weighs them) above 1.3
// times the average work per SM (w_all: the summed cost, per KV head
// included).  The planner then splits the items above half that average
// (and above 16 tiles), longest first, at most kTcMaxSplitItems.
__host__ __device__ inline bool split_longest_items(unsigned long long w_all, int longest,
                                                    int sm_count) {
    const unsigned long long sms = sm_count > 0 ? (unsigned long long)sm_count : 1ull;
    return w_all > 0 && 10ull * (unsigned long long)longest * sms > 13ull * w_all;
}

// KV tiles of tensor-core item k (positions [k * item_pos, ...)) of a chunk
// of c rows after a prefix of P keys: from the first key its first row sees
// to its last row (causal) or the sequence end.
__host__ __device__ inline int tc_item_tiles(int P, int c, int k, int item_pos, int window,
                                             int causal) {
    const int first = P + k * item_pos;
    const int end = (k + 1) * item_pos < c ? (k + 1) * item_pos : c;
    const int last = causal ? P + end - 1 : P + c - 1;
    const int lo = window > 0 ? (first - window + 1 > 0 ? first - window + 1 : 0) : 0;
    return last / kTileN - lo / kTileN + 1;
}

// The row-tile split charges every row group's start as this many extra
// tiles: a CTA's time grows with the group pieces it takes (their Q loads,
// boundary tiles and four-warp merges cost about two tiles' streaming time
// each), so a CTA that starts more groups takes fewer real tiles.  The
// groups' tiles are laid end to end as [kRowGroupStartTiles virtual tiles,
// then the real ones].
constexpr int kRowGroupStartTiles = 2;

// CTAs of the row kernel: one per SM.  The planner splits the row work for
// exactly this many.
__host__ __device__ inline int row_grid(int sm_count) {
    return sm_count < 1 ? 1 : (sm_count > kRowMaxCtas ? kRowMaxCtas : sm_count);
}

// CTAs of a row grid of n that get row tiles: min(n, T), so each of them
// gets at least one of the T tiles (the others exit at once).
__host__ __device__ inline int row_ctas_used(int n, int T) { return T < n ? T : n; }

// Row-kernel CTA `i` of the `n` used owns tiles [row_tile_begin(i),
// row_tile_begin(i + 1)) of the T row tiles (all row groups' 128-key tiles
// laid end to end).
__host__ __device__ inline int row_tile_begin(int i, int n, int T) {
    return (int)(((int64_t)i * T) / n);
}

// ---- workspace
struct WsHeader {
    int n_tc_items;
    int n_row_groups;  // (sequence, KV head) groups on the row path
    int tc_next;       // dynamic scheduler counter of the tensor-core kernel
    int row_tiles;     // T: 128-key tiles of all row groups, with each group's virtual start tiles
    int row_ctas;      // n: row-kernel CTAs the split was made for
    int pad[59];       // 256 bytes
};

// Tensor-core work item: {b, kv head g, first chunk position, w}: w is the
// cost in KV tiles, or, for a part of an item split along its KV tiles,
// kSplitTag | (first KV tile of part 1) << 12 | (split index) << 1 | part.
//
// A call whose longest item far exceeds the average work per SM splits its
// longest items in two (at most kTcMaxSplitItems of them); each split item
// keeps the partial result of its first-finishing part in the workspace.
constexpr int kTcMaxSplitItems = 64;
constexpr int kSplitTag = 1 << 30;
constexpr int kSplitMaxTile = 1 << 18;  // a split tile index must fit its 18 bits

//
// Row path.  The row groups' tiles are laid end to end (group k covers tiles
// [S_k, S_k + tiles_k)) and CTA i of n takes tiles [i*T/n, (i+1)*T/n), so
// every CTA streams the same number of tiles (within one).  The piece of
// group k that CTA i holds writes partial slot k + i: for two non-empty
// pieces (k, i) != (k', i') with k + i = k' + i' the group and CTA orders
// would have to cross, so the slots are distinct, and the pieces of one group
// use consecutive slots.  A group held by one CTA writes out and lse directly.
// Row group descriptor (three int4): {b, g, S_k, tiles_k},
// {first key, qo_indptr[b], first partial slot, n_splits},
// {chunk_len, prefix_len, kv_indptr[b], kv_len}.

struct WsLayout {
    size_t header;        // offset of WsHeader
    size_t tc_items;      // int4 [cap_tc + cap_split]
    size_t row_groups;    // int4 [3 * cap_groups]: row group descriptors
    size_t row_first;     // int [kRowMaxCtas]: first row group of each row-kernel CTA (-1: none)
    size_t group_desc;    // int4 [cap_groups]: {first partial slot, n_splits, q0, chunk_len}
    size_t partial_o;     // float [cap_row * kRowMaxRows * head_dim]
    size_t partial_ml;    // float2 [cap_row * kRowMaxRows]
    size_t split_begin;   // bytes a call without split items uses (the split buffers follow)
    size_t tc_part_o;     // float [cap_split][2 Q tiles][128 rows][head_dim]: split partials
    size_t tc_part_ml;    // float2 [cap_split][2][128]: their (max, normaliser), log2 domain
    size_t tc_sync;       // int [cap_split][2 Q tiles][4 warps][2]: {ticket, partial ready}
    size_t total;
    int64_t cap_tc;
    int64_t cap_split;
    int64_t cap_row;
    int64_t cap_groups;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool ws_layout(int batch, int64_t total_q, int n_q_heads, int n_kv_heads, int head_dim,
                      WsLayout* L) {
    if (batch < 0 || total_q < 0 || n_q_heads < 1 || n_kv_heads < 1 ||
        n_q_heads % n_kv_heads != 0)
        return false;
    const int group = n_q_heads / n_kv_heads;
    if (group > kTileM) return false;
    const int64_t qpos = (int64_t)q_positions_per_tile(group) * kQTiles;
    L->cap_tc = (int64_t)n_kv_heads * ((total_q + qpos - 1) / qpos + batch);
    L->cap_split = L->cap_tc < kTcMaxSplitItems ? L->cap_tc : kTcMaxSplitItems;
    L->cap_groups = (int64_t)n_kv_heads * batch;
    L->cap_row = L->cap_groups + kRowMaxCtas;  // partial slots: k + i < groups + CTAs
    size_t off = 0;
    L->header = off;
    off += sizeof(WsHeader);
    L->tc_items = off = align_up(off, 256);
    off += (size_t)(L->cap_tc + L->cap_split > 0 ? L->cap_tc + L->cap_split : 1) * 16;
    L->row_groups = off = align_up(off, 256);
    off += (size_t)(L->cap_groups > 0 ? L->cap_groups : 1) * 48;
    L->row_first = off = align_up(off, 256);
    off += (size_t)kRowMaxCtas * 4;
    L->group_desc = off = align_up(off, 256);
    off += (size_t)(L->cap_groups > 0 ? L->cap_groups : 1) * 16;
    L->partial_o = off = align_up(off, 256);
    off += (size_t)L->cap_row * kRowMaxRows * head_dim * 4;
    L->partial_ml = off = align_up(off, 256);
    off += (size_t)L->cap_row * kRowMaxRows * 8;
    L->split_begin = off = align_up(off, 256);
    L->tc_part_o = off;
    off += (size_t)L->cap_split * kQTiles * kTileM * head_dim * 4;
    L->tc_part_ml = off = align_up(off, 256);
    off += (size_t)L->cap_split * kQTiles * kTileM * 8;
    L->tc_sync = off = align_up(off, 256);
    off += (size_t)(L->cap_split > 0 ? L->cap_split : 1) * kQTiles * 4 * 2 * 4;
    L->total = align_up(off, 256);
    return true;
}

// ---- visibility beyond the causal rule: causal flag and boolean mask
// (True = keep) indexed [b * b_stride + h * h_stride + i * q_stride + j] with
// i the row inside the chunk and j the key position; rows i >= q_len (when
// q_stride != 0) and keys j >= kv_len read as masked.
struct MaskParams {
    const uint8_t* data;  // nullptr: no mask
    int64_t b_stride;
    int64_t h_stride;
    int64_t q_stride;
    int q_len;
    int kv_len;
};

// ---- parameters of the planner kernel
struct PlanParams {
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* prefix_lens;
    int batch;
    int64_t total_q;
    int n_kv_heads;
    int group;
    int page_size;
    int window;
    int causal;
    int tc_work;       // 0: the host knows no chunk goes to the tensor cores
    int split;         // 1: split the longest tensor-core items (the host's decision)
    int absorb;        // decode-shaped chunks on the tensor cores: 1 / 0 as the host
                       // decided, -1: the planner decides (absorb_decode_rows)
    int sm_count;
    int tc_gather;     // 1: the tensor-core kernel gathers pages below kTmaMinRows keys
    unsigned char* ws;
    WsLayout lay;
    int32_t* dev_err;
};

// ---- the fused slot mapping and KV append (pcp_kv_append_paged, and the
// append a call runs beside its planner)
struct AppendParams {
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* prefix_lens;
    int batch;
    int64_t total_q;
    int page_size;
    int64_t num_pages;
    const void* k;           // [total_q, n_kv_heads, head_dim] bf16
    const void* v;
    int chunks_per_token;    // n_kv_heads * head_dim * 2 / 16
    void* k_pool;
    void* v_pool;
    int64_t* loc;            // nullptr, or out_cache_loc [total_q]
    int32_t* dev_err;
};

// ---- parameters of the tensor-core extend kernel
struct TcParams {
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* prefix_lens;
    const unsigned char* ws;
    WsLayout lay;
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    uint16_t* out;
    float* lse;
    int n_q_heads;
    int n_kv_heads;
    int group;
    int qpos;          // positions per Q tile
    int page_size;
    int box_rows;      // rows per TMA page box; 0 selects the cp.async gather warps
    int page_shift;    // log2(page_size) for a power of two, else -1
    int64_t num_pages;
    int num_slots;
    int window;
    int causal;
    MaskParams mask;
    float scale_log2;  // sm_scale * log2(e)
    uint64_t stall_ns; // test hook (0: off): see pcp_call_options.test_stall_ns
    int32_t* dev_err;
    int split;         // host: the plan may hold split items (the instantiation that merges them)
    int ping;          // host: one-Q-tile items alternate their S/P buffers (causal, unmasked
                       // calls that have such items)
};

// ---- parameters of the split-KV combine kernel
struct CombineParams {
    const unsigned char* ws;
    WsLayout lay;
    uint16_t* out;
    float* lse;
    int n_q_heads;
    int n_kv_heads;
    int group;
    int n_groups;      // batch * n_kv_heads
};

// ---- parameters of the row (split-KV) kernel
struct RowParams {
    int self_plan;     // 1: plan in the kernel (batch <= kRowSelfPlanMaxSeqs, no planner run)
    int batch;
    int64_t total_q;
    const uint16_t* q;
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* prefix_lens;
    unsigned char* ws;
    WsLayout lay;
    const uint16_t* k_pool;
    const uint16_t* v_pool;
    uint16_t* out;
    float* lse;
    int n_q_heads;
    int n_kv_heads;
    int group;
    int page_size;
    int box_rows;      // rows per TMA page box; 0 selects cp.async gathers
    int box_shift;     // log2(box_rows) (a power of two), when box_rows > 0
    int page_shift;    // log2(page_size) when it is a power of two, else -1
    int64_t num_pages;
    int num_slots;
    int window;
    int causal;
    MaskParams mask;
    float scale_log2;
    uint64_t stall_ns; // test hook (0: off): see pcp_call_options.test_stall_ns
    int32_t* dev_err;
};

// ---- one extend-attention call as the entry points receive it
struct ExtendArgs {
    const void* q;
    const int32_t* qo_indptr;
    const int32_t* kv_indptr;
    const int32_t* kv_indices;
    const int32_t* prefix_lens;
    const int32_t* qo_indptr_host;
    int batch;
    int64_t total_q;
    const void* k_pool;
    const void* v_pool;
    int64_t num_pages;
    int page_size;
    int n_q_heads;
    int n_kv_heads;
    int head_dim;
    int window;
    float sm_scale;
    int causal;
    MaskParams mask;
    void* out;
    float* lse;
    void* workspace;
    size_t workspace_bytes;
    int32_t* dev_err;
    void* stream;
};

// Host-side checks of an extend-attention call, everything but the
// workspace: PCP_OK or the status the call returns before launching anything.
// On PCP_OK *lay is the call's workspace layout.
pcp_status check_extend_args(const ExtendArgs& a, WsLayout* lay);

// The whole call (checks, workspace, launches); opts may be null.
pcp_status run_extend(const ExtendArgs& a, const pcp_call_options* opts);

}  // namespace pcp
