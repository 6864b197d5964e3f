// api.cu -- C entry points of libqasa: argument checks, workspace carve-up,
// TMA descriptor encoding and kernel launches.  Every declaration lives in
// include/qasa.h together with its contract.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "qasa_launch.h"

using namespace qasa;

namespace {

constexpr int kMaxPagesPerSeq = 16384;
constexpr int kMaxBatch = 8192;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr int kAttnUnitWeight = 4;

// Limit of the waits on other warps, CTAs and flags.  QASA_WAIT_LIMIT_NS
// (diagnostic, for tests of the time-out path) shortens it, down to 1 us; the
// waits for a CTA's own copies in flight always keep kWaitLimitNs.
unsigned long long wait_limit_ns() {
    const char *v = std::getenv("QASA_WAIT_LIMIT_NS");
    if (!v) return kWaitLimitNs;
    const unsigned long long n = std::strtoull(v, nullptr, 10);
    if (n < 1000ull) return 1000ull;
    return n < kWaitLimitNs ? n : kWaitLimitNs;
}

// Page-equivalents of work a unit adds to an attention CTA's range (its query
// load, the hand-over of the working warps' states and their merge): ranges
// balance pages plus this per unit, so that a range of many short units gets
// fewer pages.  The cost is about fixed in time, so it is worth more of the
// smaller pages: 4 pages of 8 KiB (K + V), 8 of 4 KiB, 2 of 16 KiB (measured
// best or level on the workloads of each size).  QASA_ATTN_UNIT_WEIGHT
// (diagnostic) overrides it, 0 .. 256.
int attn_unit_weight(size_t page_kv_bytes) {
    if (const char *v = std::getenv("QASA_ATTN_UNIT_WEIGHT")) {
        const long n = std::strtol(v, nullptr, 10);
        return n < 0 ? 0 : n > 256 ? 256 : (int)n;
    }
    const size_t w = (size_t)kAttnUnitWeight * 8192 / (page_kv_bytes ? page_kv_bytes : 1);
    return w < 1 ? 1 : w > 16 ? 16 : (int)w;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(qasa_dtype dt) { return dt == QASA_DTYPE_F32 ? 4 : dt == QASA_DTYPE_E4M3 ? 1 : 2; }

qasa_status check_cache(const qasa_kv_cache *c) {
    if (!c || !c->k_pool || !c->v_pool || !c->page_bounds) return QASA_ERR_NULL;
    if (c->dtype != QASA_DTYPE_F32 && c->dtype != QASA_DTYPE_F16 && c->dtype != QASA_DTYPE_BF16 &&
        c->dtype != QASA_DTYPE_E4M3)
        return QASA_ERR_DTYPE;
    if (c->dtype == QASA_DTYPE_E4M3 && !c->page_scales) return QASA_ERR_NULL;
    if (c->dtype == QASA_DTYPE_E4M3 && !aligned16(c->page_scales)) return QASA_ERR_ALIGN;
    if (c->head_dim != 64 && c->head_dim != 128) return QASA_ERR_SHAPE;
    if (c->page_size != 16 && c->page_size != 32) return QASA_ERR_SHAPE;
    if (c->num_kv_heads < 1 || c->num_phys_pages < 1) return QASA_ERR_SHAPE;
    if ((long long)c->num_phys_pages * c->num_kv_heads * c->page_size > 0x7fffffffLL)
        return QASA_ERR_SHAPE;
    if (!aligned16(c->k_pool) || !aligned16(c->v_pool) || !aligned16(c->page_bounds))
        return QASA_ERR_ALIGN;
    return QASA_OK;
}

qasa_status check_decode(const qasa_kv_cache *c, const void *q, int num_q_heads,
                         const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                         const void *out, int batch) {
    qasa_status st = check_cache(c);
    if (st != QASA_OK) return st;
    if (!q || !block_table || !seq_lens || !out) return QASA_ERR_NULL;
    if (batch < 0 || batch > kMaxBatch) return QASA_ERR_SHAPE;
    if (num_q_heads < 1 || num_q_heads % c->num_kv_heads != 0) return QASA_ERR_SHAPE;
    const int G = num_q_heads / c->num_kv_heads;
    if (G > 8) return QASA_ERR_SHAPE;
    if (max_pages < 1 || max_pages > kMaxPagesPerSeq) return QASA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(out)) return QASA_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return QASA_ERR_ALIGN;
    return QASA_OK;
}

// Per-device attributes, queried once per device (they cannot change).
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];

int device_attr(std::atomic<int> *cache, cudaDeviceAttr attr) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) {
        const int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int sm_count() { return device_attr(g_sm_count, cudaDevAttrMultiProcessorCount); }

size_t smem_optin() { return (size_t)device_attr(g_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin); }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Diagnostics: the trace buffer set by qasa_debug_trace (NULL: off).
unsigned long long *g_trace = nullptr;

unsigned long long *select_trace() { return g_trace; }
unsigned long long *attn_trace() {
    return g_trace ? g_trace + (size_t)QASA_TRACE_MAX_CTAS * QASA_TRACE_SELECT_EVENTS : nullptr;
}

// Internal status: the cooperative launch of the single-launch kernel was
// refused (not every CTA can be resident); the caller falls back to two.
constexpr qasa_status QASA_ERR_COOPERATIVE = static_cast<qasa_status>(100);

// Fewest kept pages per attention CTA before the grid shrinks below one CTA per SM.
constexpr int kMinPagesPerCta = 8;

// The decode step runs as two kernels (selection, then attention) unless
// QASA_SINGLE_LAUNCH=1 asks for the single cooperative launch.  On GB300 the
// two-kernel form is faster for every measured workload: inside one launch
// only four warps per SM select, and a unit's selection (block-table row, box
// scoring, top-k; ~20 us per unit, latency-bound) then paces the
// attention streaming.
bool single_launch_enabled() {
    const char *v = std::getenv("QASA_SINGLE_LAUNCH");
    return v && v[0] == '1';
}

// Workspace carve-up: counters [units], ready flags [units] | partial (m, l)
// [(units + C) * G * 2] | partial o [(units + C) * G * D], each region
// 256-byte aligned.
struct WsLayout {
    size_t counters, ready, part_ml, part_o, total;
};

WsLayout ws_layout(int batch, int num_q_heads, const qasa_kv_cache *c, int grid) {
    const size_t units = (size_t)batch * c->num_kv_heads;
    const size_t G = (size_t)(num_q_heads / c->num_kv_heads);
    const size_t slots = units + (size_t)grid;
    WsLayout w;
    w.counters = 0;
    w.ready = units * 4;
    w.part_ml = align_up(units * 8, 256);
    w.part_o = w.part_ml + align_up(slots * G * 2 * 4, 256);
    w.total = w.part_o + align_up(slots * G * (size_t)c->head_dim * 4, 256);
    return w;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// Views of a KV pool for TMA, 128-byte swizzle in both.
//  3-D (one box per (page, head) tile): dim0 = 128 bytes of head dim, dim1 =
//      rows (page, head, slot) with stride head_dim*es, dim2 = the 128-byte
//      column blocks with stride 128 B; box = (128 B, page_size, all blocks), so
//      the tile lands as [block][slot][128 B].
//  2-D fallback: rows x head_dim, box = 128 bytes x page_size, one box per
//      column block.
// One map over both pools when V sits at a fixed positive offset from K
// (e.g. both pools carved from one allocation): an extra outer dimension of
// extent 2 and stride (v_pool - k_pool) selects K or V, so a single box brings
// a page's K tile and V tile, laid out back to back in shared memory.
qasa_status kv_tensor_map(CUtensorMap *map, const qasa_kv_cache *c) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return QASA_ERR_DRIVER;
    const intptr_t kv = reinterpret_cast<intptr_t>(c->v_pool) - reinterpret_cast<intptr_t>(c->k_pool);
    if (kv <= 0 || (kv & 15) || (unsigned long long)kv >= (1ull << 40)) return QASA_ERR_SHAPE;
    const size_t es = elem_size(c->dtype);
    const cuuint64_t rows = (cuuint64_t)c->num_phys_pages * c->num_kv_heads * c->page_size;
    CUresult r;
    if (c->dtype == QASA_DTYPE_E4M3) {
        cuuint64_t dims[3] = {(cuuint64_t)c->head_dim, rows, 2};
        cuuint64_t strides[2] = {(cuuint64_t)c->head_dim, (cuuint64_t)kv};
        cuuint32_t box[3] = {(cuuint32_t)c->head_dim, (cuuint32_t)c->page_size, 2};
        cuuint32_t estr[3] = {1, 1, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c->k_pool, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                c->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const CUtensorMapDataType t = c->dtype == QASA_DTYPE_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                      : c->dtype == QASA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const cuuint32_t boxw = (cuuint32_t)(128 / es);
        const cuuint32_t nsub = (cuuint32_t)(c->head_dim * es / 128);
        cuuint64_t dims[4] = {boxw, rows, nsub, 2};
        cuuint64_t strides[3] = {(cuuint64_t)c->head_dim * es, 128, (cuuint64_t)kv};
        cuuint32_t box[4] = {boxw, (cuuint32_t)c->page_size, nsub, 2};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        r = enc(map, t, 4, c->k_pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? QASA_OK : QASA_ERR_DRIVER;
}

qasa_status pool_tensor_map(CUtensorMap *map, void *base, const qasa_kv_cache *c, bool three_d) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return QASA_ERR_DRIVER;
    const size_t es = elem_size(c->dtype);
    const CUtensorMapDataType t = c->dtype == QASA_DTYPE_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : c->dtype == QASA_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t rows = (cuuint64_t)c->num_phys_pages * c->num_kv_heads * c->page_size;
    if (c->dtype == QASA_DTYPE_E4M3) {
        // FP8 codes: one box of head_dim bytes x page_size rows per tile; 128-byte
        // swizzle at head_dim 128 (the tensor-core path reads it with ldmatrix),
        // none at 64 (converted with plain row reads)
        cuuint64_t dims[2] = {(cuuint64_t)c->head_dim, rows};
        cuuint64_t strides[1] = {(cuuint64_t)c->head_dim};
        cuuint32_t box[2] = {(cuuint32_t)c->head_dim, (cuuint32_t)c->page_size};
        cuuint32_t estr[2] = {1, 1};
        CUresult r8 = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          c->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        return r8 == CUDA_SUCCESS ? QASA_OK : QASA_ERR_DRIVER;
    }
    const cuuint32_t boxw = (cuuint32_t)(128 / es);
    const cuuint32_t nsub = (cuuint32_t)(c->head_dim * es / 128);
    CUresult r;
    if (three_d) {
        cuuint64_t dims[3] = {boxw, rows, nsub};
        cuuint64_t strides[2] = {(cuuint64_t)c->head_dim * es, 128};
        cuuint32_t box[3] = {boxw, (cuuint32_t)c->page_size, nsub};
        cuuint32_t estr[3] = {1, 1, 1};
        r = enc(map, t, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[2] = {(cuuint64_t)c->head_dim, rows};
        cuuint64_t strides[1] = {(cuuint64_t)c->head_dim * es};
        cuuint32_t box[2] = {boxw, (cuuint32_t)c->page_size};
        cuuint32_t estr[2] = {1, 1};
        r = enc(map, t, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS ? QASA_OK : QASA_ERR_DRIVER;
}

qasa_status run_select(const qasa_kv_cache *cache, const void *q, int num_q_heads,
                       const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                       const int32_t *budget_pages, int max_budget, int32_t *selected,
                       float *scores_out, void *workspace, int batch, int32_t *status,
                       cudaStream_t stream) {
    SelectParams p;
    p.bounds = cache->page_bounds;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.budget = budget_pages;
    p.q = q;
    p.selected = selected;
    p.scores_out = scores_out;
    p.counters = static_cast<int32_t *>(workspace);   // cleared by the selection kernel
    p.status = status;
    p.B = batch;
    p.num_phys = cache->num_phys_pages;
    p.Hkv = cache->num_kv_heads;
    p.P = cache->page_size;
    p.G = num_q_heads / cache->num_kv_heads;
    p.Hq = num_q_heads;
    p.max_pages = max_pages;
    p.max_budget = max_budget;
    p.scales = cache->page_scales;
    p.trace = select_trace();
    cudaError_t e = launch_select(cache->dtype, cache->head_dim, p, batch * cache->num_kv_heads, stream);
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

// Attention over kept pages (or every page when `dense`).  With `fused` the
// same persistent kernel also scores and selects (one launch for the step);
// it then writes `selected` and `scores_out`.
qasa_status run_attention(const qasa_kv_cache *cache, const void *q, int num_q_heads,
                          const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                          const int32_t *budget_pages, int max_budget, const int32_t *selected,
                          float scale, void *out, void *workspace, size_t ws_bytes, int batch,
                          int32_t *status, bool dense, bool pdl, cudaStream_t stream,
                          bool fused = false, float *scores_out = nullptr) {
    const int grid = sm_count();
    if (grid <= 0) return QASA_ERR_CUDA;
    const WsLayout w = ws_layout(batch, num_q_heads, cache, grid);
    if (!workspace) return QASA_ERR_WORKSPACE;
    if (ws_bytes < w.total || !aligned16(workspace)) return QASA_ERR_WORKSPACE;
    CUtensorMap km, vm;
    int one_box = 1;
    const char *no_kv = std::getenv("QASA_KV_SEPARATE");   // diagnostic: two boxes per page
    if (!(no_kv && no_kv[0] == '1') && kv_tensor_map(&km, cache) == QASA_OK) {
        one_box = 2;
        vm = km;
    } else if (pool_tensor_map(&km, cache->k_pool, cache, true) != QASA_OK ||
               pool_tensor_map(&vm, cache->v_pool, cache, true) != QASA_OK) {
        one_box = 0;
        qasa_status st = pool_tensor_map(&km, cache->k_pool, cache, false);
        if (st != QASA_OK) return st;
        st = pool_tensor_map(&vm, cache->v_pool, cache, false);
        if (st != QASA_OK) return st;
    }
    if (const char *force = std::getenv("QASA_TMA_2D")) {   // diagnostic: force the 2-D path
        if (force[0] == '1') {
            one_box = 0;
            qasa_status st = pool_tensor_map(&km, cache->k_pool, cache, false);
            if (st != QASA_OK) return st;
            st = pool_tensor_map(&vm, cache->v_pool, cache, false);
            if (st != QASA_OK) return st;
        }
    }
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    const size_t units = (size_t)batch * cache->num_kv_heads;
    // tickets (and, for one launch, the ready flags) must start at zero
    if ((dense || fused) && cudaMemsetAsync(ws + w.counters, 0, units * (fused ? 8 : 4), stream) != cudaSuccess)
        return QASA_ERR_CUDA;
    AttnParams p;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.budget = budget_pages;
    p.selected = const_cast<int32_t *>(selected);   // written only by the single-launch kernel
    p.q = q;
    p.out = out;
    p.part_o = reinterpret_cast<float *>(ws + w.part_o);
    p.part_ml = reinterpret_cast<float *>(ws + w.part_ml);
    p.counters = reinterpret_cast<int32_t *>(ws + w.counters);
    p.status = status;
    p.B = batch;
    p.Hkv = cache->num_kv_heads;
    p.G = num_q_heads / cache->num_kv_heads;
    p.Hq = num_q_heads;
    p.max_pages = max_pages;
    p.max_budget = max_budget;
    p.num_phys = cache->num_phys_pages;
    const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)cache->head_dim);
    p.scale_log2 = (float)(sc * 1.4426950408889634);
    p.dense = dense ? 1 : 0;
    p.unit_weight = attn_unit_weight(2 * (size_t)cache->page_size * cache->head_dim * elem_size(cache->dtype));
    p.one_box = one_box;
    p.stages = 0;
    p.consumers = 0;
    p.wait_limit_ns = wait_limit_ns();
    p.drain_limit_ns = kWaitLimitNs;
    p.bounds = cache->page_bounds;
    p.scores_out = scores_out;
    p.ready = reinterpret_cast<int32_t *>(ws + w.ready);
    p.scales = cache->page_scales;
    p.trace = attn_trace();
    size_t budget = smem_optin();
    if (budget == 0) return QASA_ERR_CUDA;
    budget = budget > 1024 ? budget - 1024 : budget;   // leave room for static shared memory
    // Small batches: at least kMinPagesPerCta pages per CTA for the most pages
    // the batch can attend to, so a unit is not spread over dozens of CTAs
    // whose partials its last arriver then merges one after another.  (The
    // workspace is sized for the full grid; fewer CTAs use fewer slots.)
    int attn_grid = grid;
    if (!fused) {
        const long long most = (long long)units * (dense ? max_pages : max_budget);
        const long long want = (most + kMinPagesPerCta - 1) / kMinPagesPerCta;
        if (want < attn_grid) attn_grid = want < 1 ? 1 : (int)want;
    }
    cudaError_t e = fused ? launch_fused_decode(cache->dtype, cache->head_dim, cache->page_size, km, vm, p,
                                                grid, budget, stream)
                          : launch_attention(cache->dtype, cache->head_dim, cache->page_size, km, vm, p,
                                             attn_grid, budget, pdl, stream);
    if (e == cudaErrorInvalidConfiguration) return QASA_ERR_SHAPE;
    if (e == cudaErrorCooperativeLaunchTooLarge) {   // not every CTA could be resident: two launches
        (void)cudaGetLastError();
        return QASA_ERR_COOPERATIVE;
    }
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

}  // namespace

extern "C" {

qasa_status qasa_kv_append(const qasa_kv_cache *cache, const int32_t *block_table,
                           int32_t max_pages_per_seq, const int32_t *seq_lens,
                           const int32_t *append_lens, const void *k_new, const void *v_new,
                           int32_t batch, int32_t max_new_tokens, int32_t *device_status,
                           cudaStream_t stream) {
    qasa_status st = check_cache(cache);
    if (st != QASA_OK) return st;
    if (batch == 0 || max_new_tokens == 0) return QASA_OK;
    if (!block_table || !seq_lens || !k_new || !v_new) return QASA_ERR_NULL;
    if (batch < 0 || max_new_tokens < 0 || max_pages_per_seq < 1 || max_pages_per_seq > kMaxPagesPerSeq)
        return QASA_ERR_SHAPE;
    if (batch > 65535) return QASA_ERR_SHAPE;
    if (!aligned16(k_new) || !aligned16(v_new)) return QASA_ERR_ALIGN;
    if (batch == 0 || max_new_tokens == 0) return QASA_OK;
    AppendParams p;
    p.k_pool = cache->k_pool;
    p.v_pool = cache->v_pool;
    p.bounds = cache->page_bounds;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.append_lens = append_lens;
    p.k_new = k_new;
    p.v_new = v_new;
    p.status = device_status;
    p.num_phys = cache->num_phys_pages;
    p.Hkv = cache->num_kv_heads;
    p.P = cache->page_size;
    p.max_pages = max_pages_per_seq;
    p.T = max_new_tokens;
    p.scales = cache->page_scales;
    cudaError_t e = launch_append(cache->dtype, cache->head_dim, p, batch, stream);
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

qasa_status qasa_rebuild_page_bounds(const qasa_kv_cache *cache, const int32_t *block_table,
                                     int32_t max_pages_per_seq, const int32_t *seq_lens, int32_t batch,
                                     int32_t *device_status, cudaStream_t stream) {
    qasa_status st = check_cache(cache);
    if (st != QASA_OK || batch == 0) return st;
    if (!block_table || !seq_lens) return QASA_ERR_NULL;
    if (batch < 0 || batch > kMaxBatch || max_pages_per_seq < 1 || max_pages_per_seq > kMaxPagesPerSeq)
        return QASA_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return QASA_ERR_ALIGN;
    RebuildParams p;
    p.k_pool = cache->k_pool;
    p.bounds = cache->page_bounds;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.status = device_status;
    p.num_phys = cache->num_phys_pages;
    p.Hkv = cache->num_kv_heads;
    p.P = cache->page_size;
    p.max_pages = max_pages_per_seq;
    cudaError_t e = launch_rebuild_bounds(cache->dtype, cache->head_dim, p, batch, stream);
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

size_t qasa_decode_workspace_size(int32_t batch, int32_t num_q_heads, const qasa_kv_cache *cache,
                                  int32_t max_pages_per_seq) {
    if (!cache || cache->num_kv_heads < 1 || batch < 0 || num_q_heads < cache->num_kv_heads) return 0;
    if (max_pages_per_seq < 1 || max_pages_per_seq > kMaxPagesPerSeq) return 0;
    const int grid = sm_count();
    if (grid <= 0) return 0;
    return ws_layout(batch, num_q_heads, cache, grid).total;
}

qasa_status qasa_select_pages(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                              const int32_t *block_table, int32_t max_pages_per_seq,
                              const int32_t *seq_lens, const int32_t *budget_pages,
                              int32_t max_budget, int32_t *selected, float *scores_out,
                              void *workspace, size_t workspace_bytes, int32_t batch,
                              int32_t *device_status, cudaStream_t stream) {
    if (batch == 0) return check_cache(cache);
    qasa_status st = check_decode(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                  selected, batch);
    if (st != QASA_OK) return st;
    if (!budget_pages) return QASA_ERR_NULL;
    if (max_budget < 2) return QASA_ERR_BUDGET;
    if (!workspace) return QASA_ERR_WORKSPACE;
    const int grid = sm_count();
    if (grid <= 0) return QASA_ERR_CUDA;
    if (workspace_bytes < ws_layout(batch, num_q_heads, cache, grid).total ||
        !aligned16(workspace))
        return QASA_ERR_WORKSPACE;
    if (batch == 0) return QASA_OK;
    return run_select(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, budget_pages,
                      max_budget, selected, scores_out, workspace, batch, device_status, stream);
}

qasa_status qasa_sparse_attention(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                                  const int32_t *block_table, int32_t max_pages_per_seq,
                                  const int32_t *seq_lens, const int32_t *budget_pages,
                                  int32_t max_budget, const int32_t *selected, float scale,
                                  void *out, void *workspace, size_t workspace_bytes,
                                  int32_t batch, int32_t *device_status, cudaStream_t stream) {
    if (batch == 0) return check_cache(cache);
    qasa_status st = check_decode(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                  out, batch);
    if (st != QASA_OK) return st;
    if (!budget_pages || !selected) return QASA_ERR_NULL;
    if (max_budget < 2) return QASA_ERR_BUDGET;
    if (batch == 0) return QASA_OK;
    // counters must start at zero: the selection kernel normally clears them
    const int grid = sm_count();
    if (grid <= 0) return QASA_ERR_CUDA;
    if (!workspace || workspace_bytes < ws_layout(batch, num_q_heads, cache, grid).total)
        return QASA_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, (size_t)batch * cache->num_kv_heads * 4, stream) != cudaSuccess)
        return QASA_ERR_CUDA;
    return run_attention(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, budget_pages,
                         max_budget, selected, scale, out, workspace, workspace_bytes, batch,
                         device_status, false, false, stream);
}

qasa_status qasa_sparse_decode_attention(const qasa_kv_cache *cache, const void *q,
                                         int32_t num_q_heads, const int32_t *block_table,
                                         int32_t max_pages_per_seq, const int32_t *seq_lens,
                                         const int32_t *budget_pages, int32_t max_budget,
                                         float scale, void *out, int32_t *selected,
                                         float *scores_out, void *workspace,
                                         size_t workspace_bytes, int32_t batch,
                                         int32_t *device_status, cudaStream_t stream) {
    if (batch == 0) return check_cache(cache);
    qasa_status st = check_decode(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                  out, batch);
    if (st != QASA_OK) return st;
    if (!budget_pages || !selected) return QASA_ERR_NULL;
    if (max_budget < 2) return QASA_ERR_BUDGET;
    const int grid = sm_count();
    if (grid <= 0) return QASA_ERR_CUDA;
    if (!workspace || workspace_bytes < ws_layout(batch, num_q_heads, cache, grid).total ||
        !aligned16(workspace))
        return QASA_ERR_WORKSPACE;
    if (batch == 0) return QASA_OK;
    if (single_launch_enabled() && cache->dtype != QASA_DTYPE_E4M3) {
        st = run_attention(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, budget_pages,
                           max_budget, selected, scale, out, workspace, workspace_bytes, batch,
                           device_status, false, false, stream, true, scores_out);
        if (st != QASA_ERR_COOPERATIVE) return st;
    }
    st = run_select(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, budget_pages,
                    max_budget, selected, scores_out, workspace, batch, device_status, stream);
    if (st != QASA_OK) return st;
    return run_attention(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, budget_pages,
                         max_budget, selected, scale, out, workspace, workspace_bytes, batch,
                         device_status, false, true, stream);
}

qasa_status qasa_dense_decode_attention(const qasa_kv_cache *cache, const void *q,
                                        int32_t num_q_heads, const int32_t *block_table,
                                        int32_t max_pages_per_seq, const int32_t *seq_lens,
                                        float scale, void *out, void *workspace,
                                        size_t workspace_bytes, int32_t batch,
                                        int32_t *device_status, cudaStream_t stream) {
    if (batch == 0) return check_cache(cache);
    qasa_status st = check_decode(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                  out, batch);
    if (st != QASA_OK) return st;
    if (batch == 0) return QASA_OK;
    return run_attention(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens, seq_lens,
                         2, nullptr, scale, out, workspace, workspace_bytes, batch, device_status,
                         true, false, stream);
}

qasa_status qasa_page_attention_mass(const qasa_kv_cache *cache, const void *q, int32_t num_q_heads,
                                     const int32_t *block_table, int32_t max_pages_per_seq,
                                     const int32_t *seq_lens, float scale, float *mass,
                                     int32_t batch, int32_t *device_status, cudaStream_t stream) {
    if (batch == 0) return check_cache(cache);
    qasa_status st = check_decode(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                  q, batch);
    if (st != QASA_OK) return st;
    if (!mass) return QASA_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(mass) & 3u) return QASA_ERR_ALIGN;
    if (cache->dtype == QASA_DTYPE_E4M3) return QASA_ERR_DTYPE;   // measured on 16/32-bit caches
    MassParams p;
    p.k_pool = cache->k_pool;
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.q = q;
    p.mass = mass;
    p.status = device_status;
    p.num_phys = cache->num_phys_pages;
    p.Hkv = cache->num_kv_heads;
    p.P = cache->page_size;
    p.G = num_q_heads / cache->num_kv_heads;
    p.Hq = num_q_heads;
    p.max_pages = max_pages_per_seq;
    const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)cache->head_dim);
    p.scale_log2 = (float)(sc * 1.4426950408889634);
    cudaError_t e = launch_page_mass(cache->dtype, cache->head_dim, p, batch * cache->num_kv_heads, stream);
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

qasa_status qasa_page_hit_rate(const qasa_kv_cache *cache, const float *mass, int32_t max_pages_per_seq,
                               const int32_t *seq_lens, const int32_t *budget_pages,
                               int32_t max_budget, const int32_t *selected, int32_t batch,
                               int32_t *hits, float *covered_mass, float *best_mass,
                               int32_t *device_status, cudaStream_t stream) {
    qasa_status st = check_cache(cache);
    if (st != QASA_OK || batch == 0) return st;
    if (!mass || !seq_lens || !budget_pages || !selected || !hits || !covered_mass || !best_mass)
        return QASA_ERR_NULL;
    if (batch < 0 || batch > kMaxBatch) return QASA_ERR_SHAPE;
    if (max_pages_per_seq < 1 || max_pages_per_seq > kMaxPagesPerSeq) return QASA_ERR_SHAPE;
    if (max_budget < 2) return QASA_ERR_BUDGET;
    const void *ptrs[] = {mass, seq_lens, budget_pages, selected, hits, covered_mass, best_mass};
    for (const void *ptr : ptrs)
        if (reinterpret_cast<uintptr_t>(ptr) & 3u) return QASA_ERR_ALIGN;
    HitParams p;
    p.mass = mass;
    p.seq_lens = seq_lens;
    p.budget = budget_pages;
    p.selected = selected;
    p.hits = hits;
    p.covered = covered_mass;
    p.best = best_mass;
    p.status = device_status;
    p.Hkv = cache->num_kv_heads;
    p.P = cache->page_size;
    p.max_pages = max_pages_per_seq;
    p.max_budget = max_budget;
    cudaError_t e = launch_page_hit(p, batch * cache->num_kv_heads, stream);
    return e == cudaSuccess ? QASA_OK : QASA_ERR_CUDA;
}

const char *qasa_status_string(qasa_status s) {
    switch (s) {
    case QASA_OK: return "ok";
    case QASA_ERR_NULL: return "a required pointer is NULL";
    case QASA_ERR_DTYPE: return "unknown dtype, or a dtype this call does not support";
    case QASA_ERR_SHAPE: return "unsupported shape (head_dim, page_size, group size or sizes)";
    case QASA_ERR_ALIGN: return "a device pointer is not 16-byte aligned";
    case QASA_ERR_BUDGET: return "max_budget must be at least 2";
    case QASA_ERR_WORKSPACE: return "workspace missing or too small";
    case QASA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case QASA_ERR_DRIVER: return "the TMA descriptor encoder is unavailable or rejected the pool";
    }
    return "unknown status";
}

int32_t qasa_version(void) { return 100; }

size_t qasa_debug_trace_bytes(void) {
    return (size_t)QASA_TRACE_MAX_CTAS * (QASA_TRACE_SELECT_EVENTS + QASA_TRACE_ATTN_EVENTS) *
           sizeof(unsigned long long);
}

qasa_status qasa_debug_trace(unsigned long long *buffer, size_t bytes) {
    if (!buffer) {
        g_trace = nullptr;
        return QASA_OK;
    }
    if (reinterpret_cast<uintptr_t>(buffer) & 7u) return QASA_ERR_ALIGN;
    if (bytes < qasa_debug_trace_bytes()) return QASA_ERR_WORKSPACE;
    g_trace = buffer;
    return QASA_OK;
}

}  // extern "C"
