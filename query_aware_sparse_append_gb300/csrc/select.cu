// select.cu -- query-aware page scoring and top-k page selection.
//
// "TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
// 方法详解 / 关键设计: at decode time the query is compared with the bounding
// box of every KV block and the most similar blocks are kept.  Per
// (sequence, KV head) this kernel computes, for every page p of the sequence,
//
//     s(p) = max_g  sum_c max(q[g][c] * lo[p][c], q[g][c] * hi[p][c])      (fp32)
//
// over the G query heads of the group, then keeps the sink page 0, the newest
// page N-1, and the best (k - 2) remaining pages (ties to the lower index),
// written as ascending logical ids.
//
// One CTA per (sequence, KV head), or a cluster of C CTAs per (sequence, KV
// head) that split its 16-page tiles evenly and store their scores straight
// into the first CTA's shared memory (distributed shared memory), which then
// selects; the scoring paths (tensor-core contraction through the sign split,
// or FFMA) and the top-k selection live in select_device.cuh, shared with the
// single-launch decode kernel.
#include <cstdlib>

#include "select_device.cuh"

namespace qasa {


// NT threads per (sequence, KV head): 128, 256 or 512 (see launch_select_t).
template <typename T, int D, bool MMA, int GMAX, int NT>
__global__ void __launch_bounds__(NT, NT >= 512 ? 1 : 512 / NT) select_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *sc = reinterpret_cast<float *>(smem_raw);   // [max_pages] scores, then keys in place
    __shared__ SelScratch scratch;

    pdl_launch_dependents();

    const int u = blockIdx.x;
    unsigned long long *tr =
        p.trace && blockIdx.x < QASA_TRACE_MAX_CTAS ? p.trace + (size_t)blockIdx.x * QASA_TRACE_SELECT_EVENTS : nullptr;
    if (threadIdx.x == 0) {
        trace_stamp(tr);
        trace_smid(tr ? tr + 3 : nullptr);
        p.counters[u] = 0;
    }
    const SelGroup<NT, -1> grp{(int)threadIdx.x};
    select_unit<T, D, MMA, GMAX>(grp, p, u, sc, scratch, nullptr, nullptr, tr ? tr + 1 : nullptr);
    if (tr) {
        __syncthreads();
        if (threadIdx.x == 0) trace_stamp(tr + 2);
    }
}

// CTAs per unit of the cluster form
constexpr int kSplit = 4;

// ---- thread-block cluster primitives (PTX ISA: barrier.cluster, mapa)

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Generic address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ float *cluster_map(float *local, uint32_t rank) {
    uint64_t out;
    asm volatile("mapa.u64 %0, %1, %2;" : "=l"(out) : "l"(reinterpret_cast<uint64_t>(local)), "r"(rank));
    return reinterpret_cast<float *>(out);
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// C CTAs of NT threads per (sequence, KV head), launched as clusters of C:
// CTA r scores tiles [r*T/C, (r+1)*T/C) of the unit's T tiles into CTA 0's
// score array; after the cluster barrier CTA 0 selects.  Every thread of every
// CTA passes both cluster barriers (the arrive at entry / wait before the first
// remote store makes sure each CTA of the cluster is running; the second makes
// the scores visible to CTA 0), so no CTA exits while another still writes
// into its shared memory.
template <typename T, int D, bool MMA, int GMAX, int NT, int C>
__global__ void __launch_bounds__(NT, NT >= 512 ? 1 : 512 / NT) select_cluster_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *sc = reinterpret_cast<float *>(smem_raw);   // [max_pages], used by CTA 0
    __shared__ SelScratch scratch;

    cluster_arrive_relaxed();
    pdl_launch_dependents();

    const int u = blockIdx.x / C;
    const uint32_t rank = cluster_ctarank();
    unsigned long long *tr =
        p.trace && blockIdx.x < QASA_TRACE_MAX_CTAS ? p.trace + (size_t)blockIdx.x * QASA_TRACE_SELECT_EVENTS : nullptr;
    if (threadIdx.x == 0) {
        trace_stamp(tr);
        trace_smid(tr ? tr + 3 : nullptr);
    }
    if (rank == 0 && threadIdx.x == 0) p.counters[u] = 0;
    const SelGroup<NT, -1> grp{(int)threadIdx.x};
    const UnitPlan s = plan_unit(p, u, rank == 0 && threadIdx.x == 0);
    float *lead = cluster_map(sc, 0);
    cluster_wait_acquire();
    if (s.need_scores) {
        const int tiles = (s.N + 15) >> 4;
        score_window<T, D, MMA, GMAX>(grp, p, s, lead, (int)rank * tiles / C, ((int)rank + 1) * tiles / C);
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    if (threadIdx.x == 0) trace_stamp(tr ? tr + 1 : nullptr);
    if (rank != 0) return;
    select_from_scores(grp, p, u, s, sc, scratch);
    if (tr) {
        __syncthreads();
        if (threadIdx.x == 0) trace_stamp(tr + 2);
    }
}

template <typename T, int D, bool MMA, int GMAX, int NT>
static cudaError_t launch_select_nt(const SelectParams &p, int units, int split, cudaStream_t stream) {
    const size_t smem = (size_t)p.max_pages * sizeof(float);
    if (split == 1) {
        auto kern = select_kernel<T, D, MMA, GMAX, NT>;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        kern<<<units, NT, smem, stream>>>(p);
        return cudaGetLastError();
    }
    void (*kern)(SelectParams) = select_cluster_kernel<T, D, MMA, GMAX, NT, kSplit>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * split));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename T, int D, bool MMA, int GMAX>
static cudaError_t launch_select_t(const SelectParams &p, int units, cudaStream_t stream) {
    // Few units for the SMs: give each more warps (its scoring is a per-warp
    // chain of dependent tile loads); many units: 4 warps each keeps several
    // units resident per SM, which hides that latency better.
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    // Few units (a small batch): kSplit CTAs per unit, as a cluster, so the
    // scoring of one unit runs on several SMs.  With units for every SM the
    // split only adds launch and cluster-scheduling cost.
    int split = units * kSplit <= sms ? kSplit : 1;
    if (const char *f = std::getenv("QASA_SELECT_SPLIT")) {     // diagnostic: force CTAs per unit
        const int want = std::atoi(f);
        if (want == 1 || want == kSplit) split = want;
    }
    const int ctas = units * split;
    int nt = ctas * 2 <= sms ? 512 : ctas <= 2 * sms ? 256 : 128;
    if (const char *f = std::getenv("QASA_SELECT_THREADS")) {   // diagnostic: force the CTA size
        const int want = std::atoi(f);
        if (want == 128 || want == 256 || want == 512) nt = want;
    }
    if (nt == 512) return launch_select_nt<T, D, MMA, GMAX, 512>(p, units, split, stream);
    if (nt == 256) return launch_select_nt<T, D, MMA, GMAX, 256>(p, units, split, stream);
    return launch_select_nt<T, D, MMA, GMAX, 128>(p, units, split, stream);
}

cudaError_t launch_select(qasa_dtype dt, int D, const SelectParams &p, int units,
                          cudaStream_t stream) {
    // tensor-core scoring for 16-bit and FP8 boxes at every group size (unused
    // query heads of the 8-wide MMA are zero); FFMA for fp32
    switch (dt) {
    case QASA_DTYPE_F32:
        return D == 64 ? launch_select_t<float, 64, false, 8>(p, units, stream)
                       : launch_select_t<float, 128, false, 8>(p, units, stream);
    case QASA_DTYPE_E4M3:
        return D == 64 ? launch_select_t<fp8e4m3, 64, true, 1>(p, units, stream)
                       : launch_select_t<fp8e4m3, 128, true, 1>(p, units, stream);
    case QASA_DTYPE_F16:
        return D == 64 ? launch_select_t<__half, 64, true, 1>(p, units, stream)
                       : launch_select_t<__half, 128, true, 1>(p, units, stream);
    default:
        return D == 64 ? launch_select_t<__nv_bfloat16, 64, true, 1>(p, units, stream)
                       : launch_select_t<__nv_bfloat16, 128, true, 1>(p, units, stream);
    }
}

}  // namespace qasa
