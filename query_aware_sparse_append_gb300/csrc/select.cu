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
// One CTA (4 warps) per (sequence, KV head); the scoring paths (tensor-core
// contraction through the sign split, or FFMA) and the radix selection live in
// select_device.cuh, shared with the single-launch decode kernel.
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
    if (threadIdx.x == 0) p.counters[u] = 0;
    const SelGroup<NT, -1> grp{(int)threadIdx.x};
    select_unit<T, D, MMA, GMAX>(grp, p, u, sc, scratch);
}

template <typename T, int D, bool MMA, int GMAX, int NT>
static cudaError_t launch_select_nt(const SelectParams &p, int units, cudaStream_t stream) {
    const size_t smem = (size_t)p.max_pages * sizeof(float);
    auto kern = select_kernel<T, D, MMA, GMAX, NT>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<units, NT, smem, stream>>>(p);
    return cudaGetLastError();
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
    int nt = units * 2 <= sms ? 512 : units <= 2 * sms ? 256 : 128;
    if (const char *f = std::getenv("QASA_SELECT_THREADS")) {   // diagnostic: force the CTA size
        const int want = std::atoi(f);
        if (want == 128 || want == 256 || want == 512) nt = want;
    }
    if (nt == 512) return launch_select_nt<T, D, MMA, GMAX, 512>(p, units, stream);
    if (nt == 256) return launch_select_nt<T, D, MMA, GMAX, 256>(p, units, stream);
    return launch_select_nt<T, D, MMA, GMAX, 128>(p, units, stream);
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
