// qasa_launch.h -- kernel parameter blocks and launchers shared by the
// kernel translation units and the C entry points (host + device visible).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qasa.h"

namespace qasa {

struct AppendParams {
    void *k_pool;
    void *v_pool;
    void *bounds;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *append_lens;
    const void *k_new;
    const void *v_new;
    int32_t *status;
    int num_phys, Hkv, P, max_pages, T;
    float *scales;       // FP8 KV: [num_phys][Hkv][4] (amax K, amax V, -, -)
};

struct SelectParams {
    const void *bounds;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *budget;
    const void *q;
    int32_t *selected;
    float *scores_out;
    int32_t *counters;       // [units] the attention kernel's page tickets, cleared here
    int32_t *status;
    int B, num_phys, Hkv, P, G, Hq, max_pages, max_budget;
    const float *scales;   // FP8 KV: [num_phys][Hkv][4] (amax K, amax V, -, -)
    unsigned long long *trace;   // diagnostics: [QASA_TRACE_MAX_CTAS][QASA_TRACE_SELECT_EVENTS] or NULL
};

struct AttnParams {
    const int32_t *block_table;
    const int32_t *seq_lens;
    const int32_t *budget;
    int32_t *selected;       // read; written too by the single-launch kernel
    const void *q;
    void *out;
    float *part_o;     // [(units + C) * G * D]
    float *part_ml;    // [(units + C) * G * 2]  (running max in log2 units, sum of weights)
    int32_t *counters; // [units]
    int32_t *status;
    int B, Hkv, G, Hq, max_pages, max_budget, num_phys;
    float scale_log2;
    int dense;
    int unit_weight;   // page-equivalents a unit adds to a CTA range's work (ranges balance pages + this per unit)
    int one_box;       // 2: one box per page holding its K and V tiles (kmap only);
                       // 1: one 3-D TMA box per K/V tile; 0: one 2-D box per 128 bytes of head dim
    int stages;        // ring depth, a multiple of `consumers`
    int consumers;     // consumer warps that take pages (<= the compiled count)
    unsigned long long wait_limit_ns;    // waits on other warps, CTAs or flags
    unsigned long long drain_limit_ns;   // waits for this CTA's own copies in flight (never shortened)
    // single-launch decode only: the selection inputs and outputs
    const void *bounds;
    float *scores_out;
    int32_t *ready;    // [units] 1 once a unit's kept ids are published (zero at launch)
    const float *scales;   // FP8 KV: [num_phys][Hkv][4] (amax K, amax V, -, -)
    unsigned long long *trace;   // diagnostics: [QASA_TRACE_MAX_CTAS][QASA_TRACE_ATTN_EVENTS] or NULL
};

struct MassParams {
    const void *k_pool;
    const int32_t *block_table;
    const int32_t *seq_lens;
    const void *q;
    float *mass;       // [B][Hkv][max_pages]
    int32_t *status;
    int num_phys, Hkv, P, G, Hq, max_pages;
    float scale_log2;
};

struct HitParams {
    const float *mass;        // [B][Hkv][max_pages]
    const int32_t *seq_lens;
    const int32_t *budget;
    const int32_t *selected;  // [B][Hkv][max_budget]
    int32_t *hits;            // [B][Hkv]
    float *covered;           // [B][Hkv]
    float *best;              // [B][Hkv]
    int32_t *status;
    int Hkv, P, max_pages, max_budget;
};

struct RebuildParams {
    const void *k_pool;
    void *bounds;
    const int32_t *block_table;
    const int32_t *seq_lens;
    int32_t *status;
    int num_phys, Hkv, P, max_pages;
};

cudaError_t launch_append(qasa_dtype dt, int D, const AppendParams &p, int batch, cudaStream_t stream);
cudaError_t launch_select(qasa_dtype dt, int D, const SelectParams &p, int units, cudaStream_t stream);
cudaError_t launch_attention(qasa_dtype dt, int D, int P, const CUtensorMap &km, const CUtensorMap &vm,
                             const AttnParams &p, int grid, size_t smem_budget, bool pdl,
                             cudaStream_t stream);
// One launch for the whole decode step (scoring, selection, attention);
// cooperative, grid = one CTA per SM.
cudaError_t launch_fused_decode(qasa_dtype dt, int D, int P, const CUtensorMap &km, const CUtensorMap &vm,
                                const AttnParams &p, int grid, size_t smem_budget, cudaStream_t stream);

cudaError_t launch_rebuild_bounds(qasa_dtype dt, int D, const RebuildParams &p, int batch,
                                  cudaStream_t stream);
cudaError_t launch_page_mass(qasa_dtype dt, int D, const MassParams &p, int units, cudaStream_t stream);
cudaError_t launch_page_hit(const HitParams &p, int units, cudaStream_t stream);

}  // namespace qasa
