/*
 * qasa.h -- C ABI of the query-aware sparse paged decode library (GB300, sm_103a).
 *
 * Method: "TinyServe: Query-Aware Cache Selection for Efficient LLM Serving"
 * (arXiv 2509.12211).  Section 方法详解 / 关键设计 of that summary: every KV-cache
 * block (page) carries a bounding box of what it holds; at decode time the
 * query is compared with every page's box and only the most similar pages are
 * loaded; the abstract: page scoring, sparse memory access and masked
 * attention form one decode step.  The edgentiq post ("How TinyServe Works")
 * names the retriever (page selection over page-level metadata) and the sparse
 * attention executor (attention over the selected pages only).
 *
 * Readings fixed by this library (the pages give no formula or layout):
 *   box      lo[c] / hi[c] = per-channel min / max of the keys in the page's
 *            valid slots, stored in the KV dtype (min/max are exact).
 *   score    s(p) = max over the G query heads of the group of
 *            sum_c max(q_c * lo_c, q_c * hi_c), accumulated in fp32.
 *   select   logical page 0 (sink) and page N-1 (newest) always kept; the rest
 *            of a budget of k pages goes to the highest scores, equal scores
 *            to the lower page index; k >= N keeps every page.  Kept ids are
 *            written in ascending order.
 *   attend   softmax(scale * q.k) over the tokens of the kept pages whose
 *            position is < seq_len, times V; scale <= 0 selects 1/sqrt(d);
 *            fp32 accumulation; the output has the KV dtype.
 *
 * Layout (all row-major, caller-owned DEVICE memory unless stated):
 *   k_pool, v_pool  [num_phys_pages][num_kv_heads][page_size][head_dim]
 *   page_bounds     [num_phys_pages][num_kv_heads][2][head_dim]  (lo row, hi row)
 *   block_table     [batch][max_pages_per_seq] int32: physical page of each
 *                   logical page of each sequence
 *   q, out          [batch][num_q_heads][head_dim]; query head j uses KV head
 *                   j / (num_q_heads / num_kv_heads)
 *   selected        [batch][num_kv_heads][max_budget] int32, -1 padded
 *
 * Supported: dtype f32 / f16 / bf16; head_dim 64 or 128; page_size 16 or 32;
 * group size G = num_q_heads / num_kv_heads in 1..8; max_pages_per_seq up to
 * 16384; every device pointer 16-byte aligned.
 *
 * Ownership and threading: the library allocates nothing, keeps no state
 * between calls and only enqueues work on the given stream (asynchronous).
 * Calls on different streams that share a workspace race.
 *
 * Errors: argument problems found on the host return a nonzero status before
 * any launch.  Problems in device data (a block-table entry outside
 * [0, num_phys_pages), a seq_len beyond the block table, a budget above
 * max_budget, a bounded wait that gave up) never trap: the kernel skips the
 * offending page (or clamps the length/budget), ORs a QASA_DEVERR_* bit into
 * *device_status when that pointer is non-NULL, and finishes.
 */
#ifndef QASA_H
#define QASA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QASA_DTYPE_F32 = 0,
    QASA_DTYPE_F16 = 1,
    QASA_DTYPE_BF16 = 2,
    QASA_DTYPE_E4M3 = 3        /* FP8 KV codes with per-(page, KV head) scales; q, out, k_new, v_new are f16 */
} qasa_dtype;

typedef enum {
    QASA_OK = 0,
    QASA_ERR_NULL = 1,         /* a required pointer is NULL */
    QASA_ERR_DTYPE = 2,        /* unknown dtype, or one the call does not support */
    QASA_ERR_SHAPE = 3,        /* unsupported head_dim / page_size / group / sizes */
    QASA_ERR_ALIGN = 4,        /* a device pointer is not 16-byte aligned */
    QASA_ERR_BUDGET = 5,       /* max_budget < 2 */
    QASA_ERR_WORKSPACE = 6,    /* workspace NULL or smaller than qasa_decode_workspace_size */
    QASA_ERR_CUDA = 7,         /* a CUDA runtime call or launch failed */
    QASA_ERR_DRIVER = 8        /* the tensor-map encoder could not be obtained or failed */
} qasa_status;

/* Bits ORed into *device_status by the kernels. */
#define QASA_DEVERR_PAGE_ID   0x1  /* block-table entry outside [0, num_phys_pages): page skipped */
#define QASA_DEVERR_SEQ_LEN   0x2  /* seq_len < 0 or beyond max_pages_per_seq*page_size: clamped */
#define QASA_DEVERR_BUDGET    0x4  /* kept pages would exceed max_budget: clamped */
#define QASA_DEVERR_TIMEOUT   0x8  /* a bounded wait in a pipelined kernel gave up */
#define QASA_DEVERR_APPEND    0x10 /* append_lens[b] outside [0, max_new_tokens]: clamped */
#define QASA_DEVERR_SELECTED  0x20 /* a selected id outside [0, N_b): page skipped */

typedef struct {
    void *k_pool;            /* [num_phys_pages][num_kv_heads][page_size][head_dim] */
    void *v_pool;            /* same shape as k_pool */
    void *page_bounds;       /* [num_phys_pages][num_kv_heads][2][head_dim] */
    int32_t num_phys_pages;
    int32_t num_kv_heads;
    int32_t page_size;
    int32_t head_dim;
    qasa_dtype dtype;
    float *page_scales;      /* QASA_DTYPE_E4M3 only: [num_phys_pages][num_kv_heads][4] =
                                (amax of K, amax of V, unused, unused); NULL otherwise */
} qasa_kv_cache;

/*
 * FP8 KV (QASA_DTYPE_E4M3; the TinyServe summary lists support for several KV
 * formats).  k_pool, v_pool and page_bounds hold FP8 E4M3 codes (OCP 8-bit
 * floating point: bias 7, 3 mantissa bits, largest finite 448).  Every
 * (page, KV head) keeps amax, the largest |x| of the K (resp. V) values written
 * into it, and the scale s = amax / 448 (fp32 division): a value x is stored as
 * code(x / s) (round to nearest even, saturating, zero stored as +0; s = 0
 * stores 0), and its value is code * s.  When an append raises a page's amax,
 * the codes already in the page are re-quantized to the new scale,
 * code(value(c) * s_old / s_new) in fp32, so the page keeps one scale.  The box
 * holds the per-channel minimum and maximum K codes of the page: exact bounds of
 * the dequantized keys, since they share the page's scale.  Scores and
 * attention use code * s.  page_scales entries start at any value: a page's
 * first append (the one writing slot 0) sets them.
 */

/*
 * Append new tokens to every sequence and keep the page boxes current
 * (the bounding-box metadata of 方法详解 / 关键设计; maintained at write time).
 *
 * Sequence b has seq_lens[b] tokens before the call; its new tokens are
 * k_new[b][t] / v_new[b][t] for t < n_b, where n_b = append_lens[b] if
 * append_lens is non-NULL, else max_new_tokens.  Token at position
 * pos = seq_lens[b] + t goes to slot pos % page_size of physical page
 * block_table[b][pos / page_size], in both pools.  The page's box becomes the
 * min / max of its previous box and the new keys, except that a page whose
 * slot 0 is written by this call starts a fresh box.
 *   k_new, v_new   [batch][max_new_tokens][num_kv_heads][head_dim], cache dtype
 *   seq_lens       [batch] int32, lengths BEFORE the call (not modified: the
 *                  caller advances them)
 *   append_lens    [batch] int32 or NULL
 *   device_status  int32 or NULL (see QASA_DEVERR_*)
 * A page written by one call must belong to one sequence only.
 */
qasa_status qasa_kv_append(const qasa_kv_cache *cache, const int32_t *block_table,
                           int32_t max_pages_per_seq, const int32_t *seq_lens,
                           const int32_t *append_lens, const void *k_new, const void *v_new,
                           int32_t batch, int32_t max_new_tokens, int32_t *device_status,
                           cudaStream_t stream);

/*
 * Rebuild the page boxes of whole sequences from the keys already in k_pool:
 * for every sequence b and logical page p < ceil(seq_lens[b] / page_size), the
 * box of physical page block_table[b][p] becomes the per-channel min / max of
 * the keys in its valid slots (slot < seq_lens[b] - p * page_size).  For
 * caches whose keys were written by something other than qasa_kv_append (a
 * prefill kernel storing K/V directly, a pool restored or migrated), or to
 * re-derive the boxes after the fact.  Bit-identical to the boxes
 * qasa_kv_append maintains for the same keys (min / max are exact).
 *   seq_lens       [batch] int32, current lengths
 *   device_status  int32 or NULL (QASA_DEVERR_PAGE_ID: page skipped,
 *                  QASA_DEVERR_SEQ_LEN: length clamped)
 * A physical page listed by several sequences (shared prefix) must have the
 * same number of valid slots in each, else the last writer wins.  Reads every
 * valid key once; only page_bounds is written.
 */
qasa_status qasa_rebuild_page_bounds(const qasa_kv_cache *cache, const int32_t *block_table,
                                     int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch,
                                     int32_t *device_status, cudaStream_t stream);

/*
 * Bytes of device workspace the decode calls need for this shape on the
 * CURRENT device (split-K partials and per-(sequence, KV head) counters).
 * The workspace is scratch: its contents need no initialisation and are
 * meaningless between calls.
 */
size_t qasa_decode_workspace_size(int32_t batch, int32_t num_q_heads,
                                  const qasa_kv_cache *cache, int32_t max_pages_per_seq);

/*
 * Query-aware page selection alone: score every page of every
 * (sequence, KV head) against the box metadata and keep the budget
 * (方法详解 / 关键设计: similarity of the query to each block's box, the most
 * similar blocks are loaded).
 *   q              [batch][num_q_heads][head_dim], cache dtype
 *   budget_pages   [batch] int32: requested pages per sequence.  The kept count
 *                  is k_b = min(N_b, max(budget_pages[b], forced)) with
 *                  forced = min(N_b, 2); k_b > max_budget is clamped and flagged.
 *   selected       [batch][num_kv_heads][max_budget] int32 out: ascending
 *                  logical page ids, -1 padded
 *   scores_out     [batch][num_kv_heads][max_pages_per_seq] float out, or NULL;
 *                  entries >= N_b are left untouched
 */
qasa_status qasa_select_pages(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                              const int32_t *block_table, int32_t max_pages_per_seq,
                              const int32_t *seq_lens, const int32_t *budget_pages,
                              int32_t max_budget, int32_t *selected, float *scores_out,
                              void *workspace, size_t workspace_bytes, int32_t batch,
                              int32_t *device_status, cudaStream_t stream);

/*
 * Masked attention over a given selection (the sparse attention executor of
 * the edgentiq post): for every (sequence, KV head) the first k_b entries of
 * its `selected` row (k_b as in qasa_select_pages) are logical page ids.
 *   out            [batch][num_q_heads][head_dim], cache dtype
 * A sequence with seq_len 0 gets zeros.
 */
qasa_status qasa_sparse_attention(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                                  const int32_t *block_table, int32_t max_pages_per_seq,
                                  const int32_t *seq_lens, const int32_t *budget_pages,
                                  int32_t max_budget, const int32_t *selected, float scale,
                                  void *out, void *workspace, size_t workspace_bytes,
                                  int32_t batch, int32_t *device_status, cudaStream_t stream);

/*
 * One decode step: the scoring and selection of qasa_select_pages and the
 * attention of qasa_sparse_attention, with the same results.  Arguments as in
 * those two calls.
 *
 * By default it runs as two kernels on the stream: selection, then attention
 * (the attention kernel's prologue overlaps the selection's tail through
 * programmatic dependent launch).  With QASA_SINGLE_LAUNCH=1 in the
 * environment it runs as ONE cooperative launch of a persistent kernel (one
 * CTA per SM) that scores, selects and attends (the single pass of the
 * TinyServe abstract): each CTA selects the (sequence, KV head) units whose
 * first kept page falls in its share of the kept pages and publishes each
 * unit's ids with a flag, which the CTA's copy engine acquires (bounded wait)
 * before reading them; the kept count of every unit follows from seq_lens and
 * budget_pages alone, so the split of the attention work is known before any
 * score; an 8-byte-per-unit region of the workspace is zeroed on the stream
 * first.  If the cooperative launch is refused, the two kernels run instead.
 * Selected ids and scores are identical in both forms; outputs agree to fp32
 * summation order.
 */
qasa_status qasa_sparse_decode_attention(const qasa_kv_cache *cache, const void *q,
                                         int32_t num_q_heads, const int32_t *block_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens,
                                         const int32_t *budget_pages, int32_t max_budget,
                                         float scale, void *out, int32_t *selected,
                                         float *scores_out, void *workspace,
                                         size_t workspace_bytes, int32_t batch,
                                         int32_t *device_status, cudaStream_t stream);

/*
 * Dense paged decode attention over every page (the comparison path: what the
 * decode step costs without selection).  Arguments as in qasa_sparse_attention.
 */
qasa_status qasa_dense_decode_attention(const qasa_kv_cache *cache, const void *q,
                                        int32_t num_q_heads, const int32_t *block_table,
                                        int32_t max_pages_per_seq, const int32_t *seq_lens,
                                        float scale, void *out, void *workspace,
                                        size_t workspace_bytes, int32_t batch,
                                        int32_t *device_status, cudaStream_t stream);

/* Bytes of the fixed device buffer that qasa_sparse_decode_attention_noalloc
 * uses in place of a workspace (held by every device that loads the library). */
#define QASA_NOALLOC_SCRATCH_BYTES (4u << 20)

/*
 * The decode step of qasa_sparse_decode_attention for callers that cannot
 * allocate device memory: callers whose device memory belongs to a host
 * framework that forbids allocating behind its back, and callers on paths
 * where a device-synchronising call such as cudaMalloc is not allowed.  The
 * paper has no counterpart; this is a deployment convenience.
 *
 * Arguments and results as in qasa_sparse_decode_attention, without the
 * workspace: the library's own fixed buffer of QASA_NOALLOC_SCRATCH_BYTES
 * serves instead, and nothing is allocated (no cudaMalloc, cudaFree or other
 * allocating routine).  A shape whose qasa_decode_workspace_size exceeds that
 * size is rejected with QASA_ERR_WORKSPACE before any launch.
 *   - Every call made outside stream capture looks up the buffer's device
 *     address on the current device (so a context re-created after
 *     cudaDeviceReset is followed); a call made while the stream is being
 *     captured reuses the last address seen on that device, so make the
 *     first call on a device before any stream capture, and make one more
 *     call outside capture after a cudaDeviceReset before capturing again.
 *   - All calls on a device share the buffer, which keeps the last call's
 *     contents; what must start at zero is cleared inside each call.  Calls
 *     that overlap on the GPU (other streams) race: serialise them.
 */
qasa_status qasa_sparse_decode_attention_noalloc(const qasa_kv_cache *cache, const void *q,
                                                 int32_t num_q_heads, const int32_t *block_table,
                                                 int32_t max_pages_per_seq, const int32_t *seq_lens,
                                                 const int32_t *budget_pages, int32_t max_budget,
                                                 float scale, void *out, int32_t *selected,
                                                 float *scores_out, int32_t batch,
                                                 int32_t *device_status, cudaStream_t stream);

/*
 * Page hit-rate instrumentation (the TinyServe abstract lists the page hit
 * rate among its analyses and gives no definition; this library measures it
 * against dense attention).  Neither call is on the decode path.
 *
 * qasa_page_attention_mass: for every (sequence, KV head), the share of the
 * dense softmax(scale * q.k) weight of its G query heads (over ALL tokens
 * below seq_len) that falls on each logical page, averaged over the G heads.
 *   mass     [batch][num_kv_heads][max_pages_per_seq] float out; entries of a
 *            sequence sum to 1 (to fp32 rounding); entries >= N_b are left
 *            untouched; a page with an invalid block-table entry gets 0 and
 *            sets QASA_DEVERR_PAGE_ID.  4-byte alignment suffices.
 * Other arguments as in qasa_dense_decode_attention.  Reads every key twice.
 * 16- and 32-bit caches only (an FP8 cache returns QASA_ERR_DTYPE).
 */
qasa_status qasa_page_attention_mass(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                                     const int32_t *block_table, int32_t max_pages_per_seq,
                                     const int32_t *seq_lens, float scale, float *mass,
                                     int32_t batch, int32_t *device_status, cudaStream_t stream);

/*
 * qasa_page_hit_rate: compare a selection with the page mass.  For every
 * (sequence, KV head) with k_b kept pages (k_b as in qasa_select_pages) and
 * T = the k_b pages of largest mass (equal masses: the lower page id first):
 *   hits          [batch][num_kv_heads] int32 out: |first k_b selected ids ∩ T|
 *                 (the hit rate is hits / k_b)
 *   covered_mass  [batch][num_kv_heads] float out: mass summed over the
 *                 selected pages
 *   best_mass     [batch][num_kv_heads] float out: mass summed over T (the
 *                 most any selection of k_b pages can cover)
 * mass comes from qasa_page_attention_mass; selected ids are assumed distinct
 * (as qasa_select_pages writes them); an id outside [0, N_b) is skipped and
 * sets QASA_DEVERR_SELECTED.  Only the cache's shape fields are read.
 * Device arrays need 4-byte alignment.
 */
qasa_status qasa_page_hit_rate(const qasa_kv_cache *cache, const float *mass, int32_t max_pages_per_seq,
                               const int32_t *seq_lens, const int32_t *budget_pages,
                               int32_t max_budget, const int32_t *selected, int32_t batch,
                               int32_t *hits, float *covered_mass, float *best_mass,
                               int32_t *device_status, cudaStream_t stream);

/*
 * The decode step with its per-call inputs and outputs in HOST memory (the
 * KV cache stays on the device).  The paper has no counterpart; this is the
 * call a host-driven server makes.  Two transfer forms, same kernels, same bits:
 *   direct  every host buffer is page-locked memory the device can address
 *           at the same pointer (cudaHostAlloc / cudaHostRegister on a device
 *           with cudaDevAttrCanUseHostPointerForRegisteredMem, e.g. a
 *           Grace-Blackwell node over NVLink-C2C): the kernels of
 *           qasa_sparse_decode_attention read q, the block table, lengths and
 *           budgets and write out and selected in host memory themselves, with
 *           no copy launched;
 *   staged  otherwise, or when the environment sets QASA_HOST_DIRECT=0: one
 *           cudaMemcpyAsync per input into `workspace`, the step, and one copy
 *           per output back, all on `stream`.
 *   q_host, out_host            [batch][num_q_heads][head_dim] (f16 for FP8 KV)
 *   block_table_host            [batch][max_pages_per_seq] int32
 *   seq_lens_host, budget_pages_host  [batch] int32
 *   selected_host               [batch][num_kv_heads][max_budget] int32
 *   workspace                   device memory of qasa_host_decode_workspace_size
 *                               bytes, 256-byte aligned (scratch, no initialisation)
 * The outputs are valid once the stream has been synchronised; the host must
 * not touch the buffers before that.  Pageable host buffers take the staged
 * form (their copies are synchronous to the host).  Errors as in
 * qasa_sparse_decode_attention.
 *
 * qasa_host_call_is_direct returns 1 when a call with these six buffers takes
 * the direct form, 0 when it takes the staged form.
 */
size_t qasa_host_decode_workspace_size(int32_t batch, int32_t num_q_heads, const qasa_kv_cache *cache,
                                       int32_t max_pages_per_seq, int32_t max_budget);
qasa_status qasa_sparse_decode_attention_host(const qasa_kv_cache *cache, const void *q_host,
                                              int32_t num_q_heads, const int32_t *block_table_host,
                                              int32_t max_pages_per_seq, const int32_t *seq_lens_host,
                                              const int32_t *budget_pages_host, int32_t max_budget,
                                              float scale, void *out_host, int32_t *selected_host,
                                              void *workspace, size_t workspace_bytes, int32_t batch,
                                              int32_t *device_status, cudaStream_t stream);
int32_t qasa_host_call_is_direct(const void *q_host, const int32_t *block_table_host,
                                 const int32_t *seq_lens_host, const int32_t *budget_pages_host,
                                 const void *out_host, const int32_t *selected_host);

/*
 * Diagnostics (the paper has no counterpart): per-CTA timestamps of the
 * decode-step kernels, for reading a step's timeline (when each CTA started,
 * finished scoring, waited for the selection, issued its first copy, ...).
 *
 * qasa_debug_trace(buffer, bytes): every later launch of the selection and
 * attention kernels in this process records %globaltimer values (ns) into
 * `buffer` (device memory, 8-byte aligned, at least qasa_debug_trace_bytes()
 * bytes, zeroed by the caller: a slot that stays 0 was not reached).  NULL
 * turns recording off.  Process-wide and not thread-safe; a launch captured
 * in a CUDA graph keeps the pointer it was captured with.  Returns
 * QASA_ERR_WORKSPACE when `bytes` is too small, QASA_ERR_ALIGN when the
 * buffer is misaligned.
 *
 * Layout (uint64): QASA_TRACE_MAX_CTAS rows of QASA_TRACE_SELECT_EVENTS for
 * the selection kernel's CTAs, then QASA_TRACE_MAX_CTAS rows of
 * QASA_TRACE_ATTN_EVENTS for the attention kernel's CTAs (CTAs beyond
 * QASA_TRACE_MAX_CTAS record nothing).  Selection events: 0 CTA start,
 * 1 the CTA's last tile scored, 2 the CTA's last warp done (selections
 * included), 3 the SM the CTA ran on (an index, not a time).  Attention
 * events: 0 CTA start, 1 prologue done, 2 wait for the preceding kernel done,
 * 3 first page copy issued, 4 first page consumed, 5 last page copy issued,
 * 6 last consumer warp done, 7 combiner done, 8 the SM the CTA ran on,
 * 9 the states of the range's last segment (when it is a whole unit) are all
 * in shared memory, 10 that segment merged and written, 11 unused.
 */
#define QASA_TRACE_MAX_CTAS 4096
#define QASA_TRACE_SELECT_EVENTS 4
#define QASA_TRACE_ATTN_EVENTS 12
size_t qasa_debug_trace_bytes(void);
qasa_status qasa_debug_trace(unsigned long long *buffer, size_t bytes);

/* Static description of a status code. */
const char *qasa_status_string(qasa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t qasa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QASA_H */
