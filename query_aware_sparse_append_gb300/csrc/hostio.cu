// hostio.cu -- the decode step with its inputs and outputs in host memory.
//
// qasa_sparse_decode_attention_host stages the step's per-call inputs (queries,
// block table, lengths, budgets) from host buffers into a device workspace,
// runs the decode step of qasa_sparse_decode_attention, and copies the outputs
// (attention output and kept page ids) back, all enqueued on one stream: one
// call for a host that keeps its per-step tensors on the CPU side.  The KV
// cache itself stays in device memory.  Copies are plain cudaMemcpyAsync, one
// per buffer; with page-locked host buffers they overlap nothing but are
// asynchronous to the host.
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
