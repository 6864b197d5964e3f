// hostio.cu -- the decode step with its inputs and outputs in host memory.
//
// qasa_sparse_decode_attention_host runs the decode step of
// qasa_sparse_decode_attention for a host that keeps its per-step tensors
// (queries, block table, lengths, budgets; output and kept page ids) on the
// CPU side; the KV cache stays in device memory.  Where the device can address
// every one of those page-locked buffers at its host pointer (Grace-Blackwell:
// coherent NVLink-C2C), the kernels read and write them in place and no copy
// is launched: the transfers ride on the kernels' own loads and stores.
// Otherwise the inputs are staged into the device workspace with one
// cudaMemcpyAsync per buffer and the outputs copied back the same way, all on
// one stream.
#include <cstdlib>

#include "qasa_launch.h"

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

size_t elem_bytes_q(const qasa_kv_cache *c) { return c->dtype == QASA_DTYPE_F32 ? 4 : 2; }

struct HostLayout {
    size_t decode, q, bt, lens, budget, out, sel, total;
};

bool host_layout(int batch, int num_q_heads, const qasa_kv_cache *cache, int max_pages, int max_budget,
                 HostLayout *l) {
    const size_t ws = qasa_decode_workspace_size(batch, num_q_heads, cache, max_pages);
    if (batch > 0 && ws == 0) return false;
    const size_t qbytes = (size_t)batch * num_q_heads * cache->head_dim * elem_bytes_q(cache);
    l->decode = 0;
    l->q = align256(ws);
    l->bt = l->q + align256(qbytes);
    l->lens = l->bt + align256((size_t)batch * max_pages * 4);
    l->budget = l->lens + align256((size_t)batch * 4);
    l->out = l->budget + align256((size_t)batch * 4);
    l->sel = l->out + align256(qbytes);
    l->total = l->sel + align256((size_t)batch * cache->num_kv_heads * max_budget * 4);
    return true;
}

// Direct form: the device can dereference every host buffer at its host
// address (page-locked memory known to the driver, on a device that accepts
// host pointers for it), unless QASA_HOST_DIRECT is "0".
bool host_memory_direct(const void *a, const void *b, const void *c, const void *d, const void *e, const void *f) {
    const char *v = std::getenv("QASA_HOST_DIRECT");
    if (v && v[0] == '0') return false;
    int dev = 0, ok = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&ok, cudaDevAttrCanUseHostPointerForRegisteredMem, dev) != cudaSuccess || !ok)
        return false;
    const void *ptrs[] = {a, b, c, d, e, f};
    for (const void *p : ptrs) {
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        if (attr.type != cudaMemoryTypeHost || attr.devicePointer != p) return false;
    }
    return true;
}

}  // namespace

extern "C" size_t qasa_host_decode_workspace_size(int32_t batch, int32_t num_q_heads, const qasa_kv_cache *cache,
                                                  int32_t max_pages_per_seq, int32_t max_budget) {
    if (!cache || batch < 0 || num_q_heads < 1 || max_pages_per_seq < 1 || max_budget < 2) return 0;
    HostLayout l;
    if (!host_layout(batch, num_q_heads, cache, max_pages_per_seq, max_budget, &l)) return 0;
    return l.total;
}

extern "C" qasa_status qasa_sparse_decode_attention_host(
    const qasa_kv_cache *cache, const void *q_host, int32_t num_q_heads, const int32_t *block_table_host,
    int32_t max_pages_per_seq, const int32_t *seq_lens_host, const int32_t *budget_pages_host, int32_t max_budget,
    float scale, void *out_host, int32_t *selected_host, void *workspace, size_t workspace_bytes, int32_t batch,
    int32_t *device_status, cudaStream_t stream) {
    if (!cache) return QASA_ERR_NULL;
    if (batch == 0) return QASA_OK;
    if (!q_host || !block_table_host || !seq_lens_host || !budget_pages_host || !out_host || !selected_host)
        return QASA_ERR_NULL;
    if (batch < 0 || num_q_heads < 1 || max_pages_per_seq < 1) return QASA_ERR_SHAPE;
    if (max_budget < 2) return QASA_ERR_BUDGET;
    HostLayout l;
    if (!host_layout(batch, num_q_heads, cache, max_pages_per_seq, max_budget, &l)) return QASA_ERR_SHAPE;
    if (!workspace || workspace_bytes < l.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return QASA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    if (host_memory_direct(q_host, block_table_host, seq_lens_host, budget_pages_host, out_host, selected_host)) {
        // the kernels read the inputs and write the outputs in host memory
        // themselves (coherent device access to host memory, e.g. NVLink-C2C)
        return qasa_sparse_decode_attention(cache, q_host, num_q_heads, block_table_host, max_pages_per_seq,
                                            seq_lens_host, budget_pages_host, max_budget, scale, out_host,
                                            selected_host, nullptr, ws + l.decode, l.q, batch, device_status,
                                            stream);
    }
    const size_t qbytes = (size_t)batch * num_q_heads * cache->head_dim * elem_bytes_q(cache);
    const size_t btbytes = (size_t)batch * max_pages_per_seq * 4;
    const size_t selbytes = (size_t)batch * cache->num_kv_heads * max_budget * 4;
    struct Copy { void *dst; const void *src; size_t n; };
    const Copy in[] = {{ws + l.q, q_host, qbytes}, {ws + l.bt, block_table_host, btbytes},
                       {ws + l.lens, seq_lens_host, (size_t)batch * 4},
                       {ws + l.budget, budget_pages_host, (size_t)batch * 4}};
    for (const Copy &c : in)
        if (cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, stream) != cudaSuccess) return QASA_ERR_CUDA;
    const qasa_status st = qasa_sparse_decode_attention(
        cache, ws + l.q, num_q_heads, reinterpret_cast<const int32_t *>(ws + l.bt), max_pages_per_seq,
        reinterpret_cast<const int32_t *>(ws + l.lens), reinterpret_cast<const int32_t *>(ws + l.budget), max_budget,
        scale, ws + l.out, reinterpret_cast<int32_t *>(ws + l.sel), nullptr, ws + l.decode, l.q, batch,
        device_status, stream);
    if (st != QASA_OK) return st;
    if (cudaMemcpyAsync(out_host, ws + l.out, qbytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(selected_host, ws + l.sel, selbytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return QASA_ERR_CUDA;
    return QASA_OK;
}

extern "C" int32_t qasa_host_call_is_direct(const void *q_host, const int32_t *block_table_host,
                                            const int32_t *seq_lens_host, const int32_t *budget_pages_host,
                                            const void *out_host, const int32_t *selected_host) {
    if (!q_host || !block_table_host || !seq_lens_host || !budget_pages_host || !out_host || !selected_host)
        return 0;
    return host_memory_direct(q_host, block_table_host, seq_lens_host, budget_pages_host, out_host, selected_host)
               ? 1 : 0;
}
