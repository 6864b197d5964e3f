// noalloc.cu -- the decode step for callers that cannot allocate device memory.
//
// qasa_sparse_decode_attention needs a caller-provided workspace (per
// (sequence, KV head) tickets and split-K partials).  Some callers cannot
// obtain one: their device memory is owned by a host framework that forbids
// allocating behind its back, or they run where a device-synchronising call
// such as cudaMalloc is not allowed.  qasa_sparse_decode_attention_noalloc
// runs the same two kernels with this file's fixed device buffer as the
// workspace, so it performs no allocation of any kind.
//
// Properties of the buffer (all stated in include/qasa.h):
//   - QASA_NOALLOC_SCRATCH_BYTES bytes, a file-scope __device__ array: every
//     device that loads the library holds it until the process exits;
//   - its device address is looked up with cudaGetSymbolAddress on every call
//     made outside stream capture (so a context torn down and re-created, e.g.
//     after cudaDeviceReset, is followed), and the last address seen per
//     device is reused while the stream is being captured; the first call on
//     a device should therefore come before any stream capture;
//   - every call on a device shares it and it keeps the last call's contents;
//     the parts that must start at zero (the tickets) are cleared by the
//     selection kernel of each call; calls that overlap on the GPU race.
#include <mutex>

#include "qasa_launch.h"

static __device__ __align__(256) unsigned char qasa_noalloc_scratch[QASA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_scratch[kMaxDevices] = {};

// Device address of the scratch buffer for the current device: looked up
// again on every call made outside stream capture; during a capture the last
// address seen on this device is used (none yet: an error).
qasa_status scratch_for_current_device(cudaStream_t stream, void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QASA_ERR_CUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return QASA_ERR_CUDA;
    std::lock_guard<std::mutex> guard(g_lock);
    if (cap == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, qasa_noalloc_scratch) != cudaSuccess || !p) return QASA_ERR_CUDA;
        g_scratch[dev] = p;
    }
    if (!g_scratch[dev]) return QASA_ERR_CUDA;
    *ptr = g_scratch[dev];
    return QASA_OK;
}

}  // namespace

extern "C" qasa_status qasa_sparse_decode_attention_noalloc(
    const qasa_kv_cache *cache, const void *q, int32_t num_q_heads, const int32_t *block_table,
    int32_t max_pages_per_seq, const int32_t *seq_lens, const int32_t *budget_pages, int32_t max_budget,
    float scale, void *out, int32_t *selected, float *scores_out, int32_t batch, int32_t *device_status,
    cudaStream_t stream) {
    const size_t need = qasa_decode_workspace_size(batch, num_q_heads, cache, max_pages_per_seq);
    if (batch > 0 && need == 0) return cache ? QASA_ERR_SHAPE : QASA_ERR_NULL;
    if (need > (size_t)QASA_NOALLOC_SCRATCH_BYTES) return QASA_ERR_WORKSPACE;   // beyond the fixed buffer
    void *scratch = nullptr;
    const qasa_status st = scratch_for_current_device(stream, &scratch);
    if (st != QASA_OK) return st;
    return qasa_sparse_decode_attention(cache, q, num_q_heads, block_table, max_pages_per_seq, seq_lens,
                                        budget_pages, max_budget, scale, out, selected, scores_out, scratch,
                                        (size_t)QASA_NOALLOC_SCRATCH_BYTES, batch, device_status, stream);
}
