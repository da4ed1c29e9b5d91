/*
 * pcp.h -- C ABI of the GB300 (sm_103a) paged chunked-prefill attention library.
 *
 * The library implements the hot path of chunked prefill over a paged KV
 * cache:
 *
 *   1. pcp_compute_out_cache_loc -- where each new token of a chunk goes in
 *      the page pool, continuing inside the last partly filled page
 *      (AReno PR #642, "What does this PR do?", third bullet; AstrAI
 *      compare "scalar paged prefill fallback and decode causal fix",
 *      PagePool.bind_tasks, out_cache_loc).
 *   2. pcp_kv_append -- the scatter of the chunk's K/V into the pool
 *      (AstrAI CudaBackend.fwd_prefill, the k_buffer[layer, out_cache_loc]
 *      write).
 *   3. pcp_paged_extend_attn -- extend attention: every query row of a ragged
 *      batch attends to its sequence's cached prefix plus its own chunk,
 *      read through a page table, with bottom-right causal alignment
 *      (AReno PR #642, "What does this PR do?"; AstrAI paged prefill kernels,
 *      causal offset = KV length - query length), GQA, an optional sliding
 *      window, and split-KV with a log-sum-exp combine for decode-shaped rows
 *      (AstrAI paged decode split-KV kernel and its combine kernel).
 *   1-3 in one call: pcp_paged_extend_attn_ex with the step's new K/V rows in
 *      its pcp_call_options (k_new / v_new) maps their slots and appends them
 *      beside the planner, then attends.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers named q, k, v, *_pool, out, lse, indptr/indices/lens,
 *    out_cache_loc, workspace and dev_err are DEVICE pointers; only the
 *    optional *_host arguments are host pointers.  The caller
 *    owns every buffer and the stream; the library allocates no device
 *    memory and keeps no state except a per-device cache of the SM count and
 *    of the driver's tensor-map encoder.
 *  - bf16 tensors are passed as void* (IEEE bfloat16, 2 bytes, row major).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call is asynchronous on that stream.
 *  - Errors the host can see return a status before anything is launched.
 *    Errors only the device can see are recorded in *dev_err, a
 *    caller-owned device int32 that the caller zeroes; the first error wins.
 *    A page id or slot outside the pool (PCP_ERR_BAD_INDEX) skips the
 *    offending access (its data read as zeros, its write dropped); device
 *    metadata that contradicts itself (a chunk ending past total_q,
 *    qo_indptr[batch] != total_q, fewer page entries than ceil(L_b /
 *    page_size); PCP_ERR_INVALID_ARG) skips that sequence; a spin-wait that
 *    ran out (PCP_ERR_TIMEOUT) ends the CTA after its copies have landed.
 *    No kernel traps.  Read the word with pcp_read_error.
 *
 * Layouts
 * -------
 *  q         [total_q, n_q_heads, head_dim]        bf16
 *  k, v      [n_tokens, n_kv_heads, head_dim]      bf16 (the chunk's new K/V)
 *  k_pool,
 *  v_pool    [num_pages * page_size, n_kv_heads, head_dim] bf16; slot
 *            s = page * page_size + offset
 *  qo_indptr [batch + 1] int32, prefix sums of chunk lengths (rows of q)
 *  prefix_lens [batch] int32, cached tokens before each chunk; the KV length
 *            of sequence b is L_b = prefix_lens[b] + chunk_len_b
 *  kv_indptr [batch + 1] int32, CSR offsets into kv_indices, in PAGES
 *  kv_indices int32 page ids; sequence b owns entries
 *            [kv_indptr[b], kv_indptr[b+1]); at least ceil(L_b / page_size)
 *            entries, all in [0, num_pages).  Entries after those may hold
 *            anything (e.g. -1 padding of a dense page table) and are never
 *            read.  Several sequences may list the same pages (successive
 *            chunks of one prompt in one call).
 *  out       [total_q, n_q_heads, head_dim] bf16 (round to nearest even)
 *  lse       [total_q, n_q_heads] float32, natural log of the sum of
 *            exp(sm_scale * q.k) over the visible keys; -inf for a row that
 *            sees no key (impossible with a causal mask and window >= 1)
 */
#ifndef PCP_H_
#define PCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pcp_status {
    PCP_OK = 0,
    PCP_ERR_INVALID_ARG = 1,  /* a null pointer, a negative or inconsistent size */
    PCP_ERR_UNSUPPORTED = 2,  /* a shape this build has no kernel for */
    PCP_ERR_BAD_INDEX = 3,    /* device: a page id or slot outside the pool */
    PCP_ERR_WORKSPACE = 4,    /* workspace smaller than pcp_extend_workspace_size */
    PCP_ERR_CUDA = 5,         /* a CUDA runtime or driver call failed */
    PCP_ERR_TIMEOUT = 6       /* device: a bounded spin-wait gave up */
} pcp_status;

/* Static string naming a status code; never NULL. */
const char* pcp_status_string(int status);

/* ABI version of this header (incremented on incompatible changes). */
int pcp_abi_version(void);

/*
 * Text of the CUDA error behind the last PCP_ERR_CUDA an entry point returned
 * on the calling thread ("no error" if there was none).  Static string;
 * never NULL.
 */
const char* pcp_last_cuda_error(void);

/*
 * Slot mapping for the new tokens of every sequence (integer, bit-exact):
 *   out_cache_loc[t] = kv_indices[kv_indptr[b] + p / page_size] * page_size
 *                      + p % page_size,   p = prefix_lens[b] + (t - qo_indptr[b])
 * for qo_indptr[b] <= t < qo_indptr[b+1].  Writes begin inside the last
 * partly filled page when prefix_lens[b] % page_size != 0 (AReno PR #642,
 * "What does this PR do?": continue prefill inside the last allocated KV
 * page).  A page id outside [0, num_pages) sets *dev_err = PCP_ERR_BAD_INDEX
 * and writes -1 for that token.
 * out_cache_loc: device int64 [total_q], written.
 */
pcp_status pcp_compute_out_cache_loc(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                     const int32_t* kv_indices, const int32_t* prefix_lens,
                                     int batch, int64_t total_q, int page_size,
                                     int64_t num_pages, int64_t* out_cache_loc,
                                     int32_t* dev_err, void* stream);

/*
 * KV append (a pure copy, bit-exact):
 *   k_pool[out_cache_loc[t], :, :] = k[t, :, :],  v_pool[...] = v[t, :, :]
 * for 0 <= t < n_tokens (AstrAI CudaBackend.fwd_prefill / fwd_decode, the
 * write of the step's K/V at out_cache_loc before attention).  A location
 * outside [0, pool_slots) sets *dev_err = PCP_ERR_BAD_INDEX and that token is
 * skipped.  Slots not named in out_cache_loc are left untouched.
 * head_dim * 2 bytes must be a multiple of 16; k, v and the pools must be
 * 16-byte aligned.
 */
pcp_status pcp_kv_append(const void* k, const void* v, const int64_t* out_cache_loc,
                         int64_t n_tokens, int n_kv_heads, int head_dim, void* k_pool,
                         void* v_pool, int64_t pool_slots, int32_t* dev_err, void* stream);

/*
 * Slot mapping and KV append in one kernel (integer and copy, bit-exact):
 * for every new token t of sequence b (qo_indptr[b] <= t < qo_indptr[b+1]),
 * its slot s = kv_indices[kv_indptr[b] + p / page_size] * page_size
 * + p % page_size with p = prefix_lens[b] + (t - qo_indptr[b]) (as
 * pcp_compute_out_cache_loc), then k_pool[s] = k[t] and v_pool[s] = v[t] (as
 * pcp_kv_append).  The same two steps of a serving step (AReno PR #642,
 * "What does this PR do?", third bullet: prefill continues inside the last
 * allocated page; AstrAI CudaBackend.fwd_prefill, the k_buffer write at
 * out_cache_loc) without the round trip through an out_cache_loc array.
 * k, v: [total_q, n_kv_heads, head_dim] bf16; the pools hold num_pages *
 * page_size slots.  out_cache_loc: NULL, or device int64 [total_q] that
 * receives the slots (-1 for a token whose page id is bad).  A page id
 * outside [0, num_pages) sets *dev_err = PCP_ERR_BAD_INDEX and that token is
 * not written.  head_dim * 2 bytes must be a multiple of 16; k, v and the
 * pools must be 16-byte aligned.
 */
pcp_status pcp_kv_append_paged(const int32_t* qo_indptr, const int32_t* kv_indptr,
                               const int32_t* kv_indices, const int32_t* prefix_lens, int batch,
                               int64_t total_q, int page_size, int64_t num_pages, const void* k,
                               const void* v, int n_kv_heads, int head_dim, void* k_pool,
                               void* v_pool, int64_t* out_cache_loc, int32_t* dev_err,
                               void* stream);

/*
 * Bytes of device workspace pcp_paged_extend_attn needs for a call with at
 * most `batch` sequences and `total_q` query rows (work lists, split-KV
 * partials and counters, and at the end the partials of split tensor-core
 * items).  Pure host arithmetic; 0 for an unsupported shape.  A call whose
 * workspace holds everything but the split items' buffers runs, unsplit.
 */
size_t pcp_extend_workspace_size(int batch, int64_t total_q, int n_q_heads, int n_kv_heads,
                                 int head_dim);

/*
 * Paged extend attention (AReno PR #642, "What does this PR do?": one
 * paged varlen attention call for mixed prefix/chunk lengths with
 * bottom-right causal alignment; AstrAI attn_paged_prefill / attn_paged_decode).
 * For sequence b, query row i (position p = prefix_lens[b] + i) and query
 * head h (KV head g = h / (n_q_heads / n_kv_heads)), the visible keys are
 * j in [lo, p] with lo = max(0, p - window + 1) when window > 0, else 0:
 *   s_j = sm_scale * q[row, h, :] . K[slot(b, j), g, :]
 *   out[row, h, :] = sum_j softmax(s)_j * V[slot(b, j), g, :]
 *   lse[row, h]    = log(sum_j exp(s_j))
 * sm_scale <= 0 selects 1 / sqrt(head_dim) (AstrAI parameter packing).
 * A chunk of length 0 is allowed (no rows); prefix_lens[b] == 0 is a plain
 * prefill; a chunk of length 1 is a decode row.
 *
 * qo_indptr_host: NULL, or a HOST copy of qo_indptr ([batch + 1] int32, the
 * same values as the device array; read during the call only, not kept).
 * With it the call launches only the kernels that have work: chunks of at
 * most 16 / (n_q_heads / n_kv_heads) rows go to the split-KV row kernel, the
 * others to the tensor-core kernel, and a call whose chunks are all of one
 * kind skips the other kernel's launch.  A host copy that does not start at
 * 0, does not end at total_q or decreases returns PCP_ERR_INVALID_ARG before
 * anything is launched.  Results are bit-identical with and without it.
 *
 * The K/V of the chunk itself must already be in the pool (pcp_kv_append
 * first, as a serving step does).  The call starts reading qo_indptr,
 * kv_indptr and prefix_lens while the kernel before it on the stream is
 * still running (a programmatic dependent launch): a kernel of the caller's
 * that writes them right before this call must not trigger programmatic
 * dependents before those writes (a kernel that does not use that feature
 * is always fine).  Supported: head_dim in {64, 128},
 * n_q_heads % n_kv_heads == 0, n_q_heads / n_kv_heads <= 128, page_size >= 1,
 * window >= 0, num_pages * page_size < 2^31.  q, out, the pools and the
 * workspace must be 16-byte aligned (256-byte aligned workspace).
 * workspace: device memory of at least pcp_extend_workspace_size(...) bytes;
 * its contents need no initialisation and are scratch between calls.  Calls
 * that share one workspace must be ordered on the GPU (same stream).
 * lse may be NULL.
 */
pcp_status pcp_paged_extend_attn(const void* q, const int32_t* qo_indptr,
                                 const int32_t* kv_indptr, const int32_t* kv_indices,
                                 const int32_t* prefix_lens, const int32_t* qo_indptr_host,
                                 int batch, int64_t total_q,
                                 const void* k_pool, const void* v_pool, int64_t num_pages,
                                 int page_size, int n_q_heads, int n_kv_heads, int head_dim,
                                 int window, float sm_scale, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                 void* stream);

/*
 * Extend attention with a causal switch and an optional boolean mask (AstrAI
 * attn_paged_prefill: `is_causal` and `mask`, True = keep, indexed by the
 * request-local query row and key; its prefill-with-mask regression test runs
 * a 4-D causal-pattern mask with causality off).  Arguments, layouts, results
 * and errors are those of pcp_paged_extend_attn (which is this call with
 * causal = 1 and no mask), plus:
 *   causal    1: bottom-right causal (query row i sees keys j <= P_b + i, and
 *                the window applies); 0: every row sees all keys j < L_b
 *                (window must be 0).  Anything else is PCP_ERR_INVALID_ARG.
 *   mask      NULL, or a DEVICE array of bytes (0 = masked, nonzero = keep).
 *             Key j of query row i of sequence b, query head h is kept when
 *             mask[b * mask_b_stride + h * mask_h_stride + i * mask_q_stride
 *             + j] is nonzero, on top of the causal rule.  i is the row inside
 *             the chunk (0 .. chunk_len_b - 1), j the key position
 *             (0 .. L_b - 1).  A stride of 0 broadcasts that dimension (a 2-D
 *             key mask [batch, kv] has h and q strides 0; a 4-D mask
 *             [batch, 1, q, kv] has h stride 0).  Rows i >= mask_q_len (when
 *             mask_q_stride != 0) and keys j >= mask_kv_len read as masked.
 *             The mask must be 16-byte aligned and the three strides
 *             non-negative multiples of 16 (bytes); otherwise
 *             PCP_ERR_INVALID_ARG before anything is launched.
 * A row whose visible set is empty gets out = 0 and lse = -inf.
 */
pcp_status pcp_paged_extend_attn_masked(
    const void* q, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
    const int32_t* prefix_lens, const int32_t* qo_indptr_host, int batch, int64_t total_q,
    const void* k_pool, const void* v_pool, int64_t num_pages, int page_size, int n_q_heads,
    int n_kv_heads, int head_dim, int window, float sm_scale, int causal, const uint8_t* mask,
    int64_t mask_b_stride, int64_t mask_h_stride, int64_t mask_q_stride, int32_t mask_q_len,
    int32_t mask_kv_len, void* out, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* dev_err, void* stream);

/*
 * Size of the fixed device scratch array behind
 * pcp_paged_extend_attn_noalloc (16 MiB).  Every GPU that loads the library
 * keeps this much memory reserved until the process exits.
 */
#define PCP_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * pcp_paged_extend_attn without a caller-supplied workspace.  The pages this
 * library follows have no counterpart: it exists for callers that cannot
 * allocate device memory -- code inside a host framework that owns every
 * allocation, a plugin ABI with no allocation hook, or a hot path that must
 * not call cudaMalloc -- and so cannot pass a workspace.  Arguments, layouts,
 * results and errors are those of pcp_paged_extend_attn; the work lists,
 * split-KV partials and counters go to a file-scope device array of
 * PCP_NOALLOC_SCRATCH_BYTES instead.  The arguments are checked first, as
 * pcp_paged_extend_attn checks them (a bad argument returns the same
 * status); then a call whose pcp_extend_workspace_size(...) exceeds the
 * array returns PCP_ERR_WORKSPACE before launching anything.  Nothing is
 * allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  The cached address belongs to the device's primary context: after
 * cudaDeviceReset (or any other teardown of that context) it is stale, and
 * this entry point must not be called again in the process.  All calls on a
 * device share the one array and it keeps the last call's contents; each call
 * re-initialises what must start at zero, but calls whose GPU work overlaps
 * (different streams, or several host threads) race on the array and must be
 * ordered by the caller.
 */
pcp_status pcp_paged_extend_attn_noalloc(const void* q, const int32_t* qo_indptr,
                                         const int32_t* kv_indptr, const int32_t* kv_indices,
                                         const int32_t* prefix_lens,
                                         const int32_t* qo_indptr_host, int batch,
                                         int64_t total_q,
                                         const void* k_pool, const void* v_pool,
                                         int64_t num_pages, int page_size, int n_q_heads,
                                         int n_kv_heads, int head_dim, int window,
                                         float sm_scale, void* out, float* lse,
                                         int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Host-side chunk planner and page pool.  Pure host code: every pointer
 * below is a HOST pointer and nothing touches a GPU.  Not thread-safe: one
 * pool is used from one thread at a time.
 *
 * The step upstream of the attention path (AReno PR #642: prompts longer
 * than the scheduler's token budget are prefilled in chunks, decode rows run
 * alongside, a request samples only once its final chunk has run, and prefill
 * continues inside the last allocated KV page; vLLM PR #54076: with a
 * recurrent-state grid of S tokens every chunk stops at the next grid point,
 * also from an aligned start).
 * ---------------------------------------------------------------------- */
typedef struct pcp_pager pcp_pager;

/* A pool of num_pages pages of page_size slots, all free.  NULL on a bad
 * argument (num_pages < 0 or > INT32_MAX, page_size < 1) or out of memory.
 * The caller owns it and frees it with pcp_pager_destroy. */
pcp_pager* pcp_pager_create(int64_t num_pages, int page_size);
void pcp_pager_destroy(pcp_pager* pager);

/* Free pages in the pool (-1 for a NULL pool). */
int64_t pcp_pager_num_free(const pcp_pager* pager);

/* Entries of all requests' page lists together (-1 for a NULL pool): with the
 * free pages, a bound on the kv_indices entries of any step. */
int64_t pcp_pager_num_held(const pcp_pager* pager);

/* The pages request req_id holds, in token order: writes up to `capacity`
 * of them to `pages` (may be NULL) and returns how many it holds (0 for an
 * unknown request, -1 for a NULL pool). */
int64_t pcp_pager_request_pages(const pcp_pager* pager, int64_t req_id, int32_t* pages,
                                int64_t capacity);

/* Drop request req_id's hold on its pages (a finished request); a page
 * nobody holds any more (no request, not the prefix index) is free again. */
pcp_status pcp_pager_release(pcp_pager* pager, int64_t req_id);

/*
 * Shared pages (vLLM PR #54076, "E2E": an immediate re-ask of a prompt
 * reuses its cached blocks, and the hit is quantised to whole blocks: at
 * most floor((P - 1) / page_size) * page_size tokens of a P-token prompt,
 * so the prompt's last token is always computed).  Pages carry reference
 * counts; a shared page is read-only.
 *
 * pcp_pager_share: request dst_req (holding no pages) takes read-only
 * references to the first ceil(n_tokens / page_size) pages of src_req, e.g.
 * for several continuations of one prompt; the caller then treats dst_req as
 * having n_tokens computed.  PCP_ERR_INVALID_ARG if src_req holds fewer
 * pages, dst_req already holds pages, or the ids are equal.
 *
 * pcp_pager_cache_prompt: enter request req_id's full pages into the prefix
 * index, keyed by tokens[0 .. (i + 1) * page_size) for page i (a chained
 * 64-bit hash, with the page's tokens kept and compared on lookup).  Call it
 * once those tokens' K/V are computed.  Only whole pages are entered; a key
 * that is already present keeps its page.  The index holds a reference to
 * each page it names.  Returns the pages newly entered (-1 on a bad
 * argument).
 *
 * pcp_pager_match_prefix: request req_id (holding no pages) takes read-only
 * references to the longest run of indexed pages that matches tokens[0 ..
 * n_tokens), at most floor((n_tokens - 1) / page_size) of them, and
 * *n_hit = their tokens; the caller starts it with that many computed.
 *
 * pcp_pager_clear_cache: empty the prefix index (pages only it held are
 * freed).  There is no other eviction.
 *
 * A step whose chunk starts inside a shared, partly filled page copies that
 * page first (copy-on-write, see pcp_schedule_step).
 */
pcp_status pcp_pager_share(pcp_pager* pager, int64_t src_req, int64_t dst_req, int64_t n_tokens);
int64_t pcp_pager_cache_prompt(pcp_pager* pager, int64_t req_id, const int32_t* tokens,
                               int64_t n_tokens);
pcp_status pcp_pager_match_prefix(pcp_pager* pager, int64_t req_id, const int32_t* tokens,
                                  int64_t n_tokens, int64_t* n_hit);
pcp_status pcp_pager_clear_cache(pcp_pager* pager);

/*
 * Plan one serving step.  Request r (0 <= r < n_reqs, distinct req_ids[r])
 * knows total_lens[r] tokens (prompt plus generated) of which num_computed[r]
 * already have their K/V in the pool; its pending work is the difference.
 *   1. Requests with exactly one pending token (decode-shaped) get it, in
 *      order, while the budget lasts.
 *   2. The others get chunks in order: as many pending tokens as the budget
 *      left allows, stopping at the next multiple of state_block strictly
 *      above num_computed[r] when state_block > 0.
 *   Each chunk is cut to the tokens its request's pages plus the free pages
 *   can hold (the pages are counted in the order the chunks are chosen); a
 *   chunk that starts inside a page other holders share also counts one
 *   page for its copy, and gets no tokens when no page is free for it.
 *   3. Every request with a non-empty chunk, in request order, becomes one
 *      row of the step: if its chunk starts inside a page whose reference
 *      count (as the rows before left it) is above one, it takes the lowest
 *      free page, which replaces the shared one in its list, and the step
 *      reports the copy (copy_src[c] -> copy_dst[c], the first copy_slots[c]
 *      slots, to run with pcp_copy_page_slots before the step's KV append);
 *      then it takes the lowest free pages its new tokens need.
 * Outputs (host arrays the caller sizes; n_reqs + 1 entries bound the rows):
 *   *n_rows; row_req[n] (index r of row n); qo_indptr[n + 1] (chunk
 *   offsets); prefix_lens[n] (= num_computed of the row's request);
 *   kv_indptr[n + 1] / kv_indices (each row's full page list, the CSR the
 *   attention call takes, in pages); sample[n] (1 when the row's chunk ends
 *   at total_lens, i.e. the step samples a token for it); *n_copies and
 *   copy_src / copy_dst / copy_slots (n_reqs entries bound them).
 * The caller advances num_computed by the chunk lengths afterwards.
 * Errors: PCP_ERR_INVALID_ARG for a NULL pool or array, a negative size,
 * num_computed > total_lens, repeated req_ids, or a request holding fewer
 * pages than its computed tokens need; PCP_ERR_WORKSPACE when kv_indices_cap
 * is smaller than the page entries of the step (nothing is allocated then).
 */
pcp_status pcp_schedule_step(pcp_pager* pager, int n_reqs, const int64_t* req_ids,
                             const int32_t* total_lens, const int32_t* num_computed, int budget,
                             int state_block, int32_t* n_rows, int32_t* row_req,
                             int32_t* qo_indptr, int32_t* prefix_lens, int32_t* kv_indptr,
                             int32_t* kv_indices, int64_t kv_indices_cap, uint8_t* sample,
                             int32_t* n_copies, int32_t* copy_src, int32_t* copy_dst,
                             int32_t* copy_slots);

/*
 * Copy-on-write of shared pages on the device (integer copy, bit-exact): for
 * each c < n_copies, slots [0, n_slots[c]) of page src_pages[c] of k_pool
 * and v_pool ([num_pages * page_size, n_kv_heads, head_dim] bf16) are
 * copied to the same slots of page dst_pages[c].  src_pages, dst_pages and
 * n_slots are DEVICE int32 arrays.  A page id outside [0, num_pages) or a
 * slot count outside [0, page_size] sets *dev_err = PCP_ERR_BAD_INDEX and
 * that copy is skipped.  The destinations must not overlap the sources.
 * n_copies <= 65535.
 */
pcp_status pcp_copy_page_slots(void* k_pool, void* v_pool, int64_t num_pages, int page_size,
                               int n_kv_heads, int head_dim, const int32_t* src_pages,
                               const int32_t* dst_pages, const int32_t* n_slots, int n_copies,
                               int32_t* dev_err, void* stream);

/*
 * Synchronise `stream` and copy *dev_err to *host_err (host pointer).
 * Returns PCP_ERR_CUDA if the synchronisation or copy fails.
 */
pcp_status pcp_read_error(const int32_t* dev_err, void* stream, int32_t* host_err);

/*
 * Per-call options: instrumentation for profiling and for tests of the
 * device-side error paths (the pages have no counterpart), a host copy of
 * prefix_lens for the launch decision, and the step's new K/V rows to append
 * before attending.  A zeroed struct (or a NULL pointer) means: no events,
 * the default wait limit, no host copy, no append.
 *   tc_event_before / tc_event_after: NULL, or cudaEvent_t values (as void*)
 *     recorded on the call's stream right before and right after the launch
 *     of the tensor-core kernel, so the caller can time that kernel alone
 *     (recorded even when the call has no tensor-core work).  Both or
 *     neither.  Recording them orders the kernel after its predecessor and
 *     its successor after it: the call loses the launch overlap it has
 *     without events.
 *   rows_event_before / rows_event_after: the same around the split-KV row
 *     kernel (recorded only when the call launches it).
 *   test_stall_ns: 0, or a test of the kernels' timeout path: in every CTA
 *     of the tensor-core and row kernels the call launches, one pipeline
 *     wait (the tensor-core MMA issuer's first one; the row kernel's
 *     consumers' first one) is made on an mbarrier that nothing arrives on,
 *     with this limit instead of the default 2 s.  It runs out, as any wait
 *     of the kernels does after 2 s when the GPU stops making progress:
 *     PCP_ERR_TIMEOUT goes to *dev_err, the CTA's other warps give up their
 *     waits, its in-flight copies and MMAs complete (those drain waits keep
 *     the 2 s limit), its tensor memory is freed and it exits.  The call's
 *     results are then undefined; the device, the stream and the library
 *     stay usable.
 *   prefix_lens_host: NULL, or a HOST copy of prefix_lens ([batch] int32,
 *     read during the call only), used together with qo_indptr_host.  A call
 *     with tensor-core work takes its decode-shaped chunks onto the tensor
 *     cores (one-Q-tile items in the longest-first queue) when the longest
 *     of them, charged 4/5 of a two-Q-tile step per 128-key tile, stays
 *     within 1.1 times the larger of the longest prompt item and the
 *     average work per SM.  Without both host copies the planner kernel
 *     decides this on the device, and the row kernel and the combine are
 *     launched and find no work when it takes them on; with both, the host
 *     makes the same decision and launches only the kernels that have work.
 *     The decision moves work between kernels only: results are correct
 *     either way (bit-identical whenever the decision is the same).
 *     With both host copies, an unmasked call whose longest tensor-core item
 *     is more than 1.3 times the average work per SM also splits its longest
 *     items in two along their 128-key tiles (the items above half that
 *     average and above 16 tiles, longest first, at most 64).  The two
 *     parts are separate items of the queue; the part that finishes second
 *     merges the first one's partial output and (max, normaliser) into the
 *     result.  A split changes only the rounding order of those rows.  It
 *     needs the full pcp_extend_workspace_size: with a smaller workspace
 *     the call runs unsplit.
 *   k_new / v_new: NULL, or the step's new K and V rows, [total_q,
 *     n_kv_heads, head_dim] bf16 on the device, 16-byte aligned; both or
 *     neither.  The call first does what pcp_kv_append_paged does with them
 *     (slot mapping from the page table, scatter into k_pool / v_pool; a bad
 *     page id sets *dev_err = PCP_ERR_BAD_INDEX and that token is not
 *     written), then attends over the pools it wrote (AReno PR #642, "What
 *     does this PR do?": the chunk's own keys are in the cache when it
 *     attends).  The pools and the results are bit-identical to
 *     pcp_kv_append_paged followed by the same call without k_new / v_new.
 *     The append runs in the planner's launch, beside the planning, when it
 *     fits in one wave of that launch's CTAs (one per SM, 4096 16-byte
 *     chunks of K and as many of V each); a longer one, and the append of a
 *     decode-only call planned inside the row kernel, runs as the kernel of
 *     pcp_kv_append_paged ahead of the rest.  The pools are written while the
 *     call runs: the caller orders other readers of the same slots.
 *   out_cache_loc: NULL, or (with k_new / v_new) device int64 [total_q] that
 *     receives each new token's slot (-1 for a token whose page id is bad).
 * The library keeps nothing of it after the call returns.
 */
typedef struct pcp_call_options {
    void* tc_event_before;
    void* tc_event_after;
    void* rows_event_before;
    void* rows_event_after;
    uint64_t test_stall_ns;
    const int32_t* prefix_lens_host;
    const void* k_new;
    const void* v_new;
    int64_t* out_cache_loc;
} pcp_call_options;

/*
 * pcp_paged_extend_attn_masked with per-call options (NULL: none).  Events
 * given one without the other return PCP_ERR_INVALID_ARG before anything is
 * launched.
 */
pcp_status pcp_paged_extend_attn_ex(
    const void* q, const int32_t* qo_indptr, const int32_t* kv_indptr, const int32_t* kv_indices,
    const int32_t* prefix_lens, const int32_t* qo_indptr_host, int batch, int64_t total_q,
    const void* k_pool, const void* v_pool, int64_t num_pages, int page_size, int n_q_heads,
    int n_kv_heads, int head_dim, int window, float sm_scale, int causal, const uint8_t* mask,
    int64_t mask_b_stride, int64_t mask_h_stride, int64_t mask_q_stride, int32_t mask_q_len,
    int32_t mask_kv_len, void* out, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* dev_err, void* stream, const pcp_call_options* options);

#ifdef __cplusplus
}
#endif

#endif /* PCP_H_ */
