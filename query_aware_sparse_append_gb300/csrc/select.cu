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
// Work split (persistent, balanced over pages).  The 16-page tiles of every
// (sequence, KV head) unit that needs scores are laid out in one flattened
// order (unit-major); warp w of the grid's W warps scores the contiguous tile
// range [w*T/W, (w+1)*T/W) into the unit's score row in global memory (L2),
// then adds the number of tiles it scored to the unit's ticket
// (acquire-release).  The warp that completes a unit's ticket selects that
// unit on its own (warp_select_unit) while the other warps keep streaming
// page boxes, so the selection does not leave HBM idle and ragged batches
// spread evenly over the SMs.  Units that need no scores (no pages, or every
// page kept) are written directly.  The scoring paths (tensor-core
// contraction through the sign split, or FFMA) live in select_device.cuh,
// shared with the single-launch decode kernel.
#include <cstdlib>

#include "select_device.cuh"

namespace qasa {

constexpr int kSelWarps = 8;          // warps per CTA
constexpr int kSelCtasPerSm = 2;      // resident CTAs per SM (16 warps: one box tile in flight each)
constexpr int kSelKeySlots = 32;      // keys per lane the selecting warp keeps in registers (N <= 1024)

// One warp scoring on its own (the scoring paths stride tiles by the group's
// warp count; here that count is one).
struct OneWarp {
    int tid;   // lane
    __device__ __forceinline__ void sync() const { __syncwarp(); }
    __device__ __forceinline__ int lane() const { return tid; }
    __device__ __forceinline__ int warp() const { return 0; }
    static constexpr int warps = 1;
};

template <typename T, int D, bool MMA, int GMAX>
__global__ void __launch_bounds__(32 * kSelWarps, kSelCtasPerSm) select_tiles_kernel(SelectParams p) {
    extern __shared__ __align__(16) int sm_i[];
    int *prefix = sm_i;                 // [B + 1] scored tiles of the sequences before b (one KV head)
    int *npages = prefix + p.B + 1;     // [B] pages of sequence b
    __shared__ int s_wsum[kSelWarps];

    pdl_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = gridDim.x, c = blockIdx.x;
    const int Hkv = p.Hkv, B = p.B;
    unsigned long long *const tr =
        p.trace && c < QASA_TRACE_MAX_CTAS ? p.trace + (size_t)c * QASA_TRACE_SELECT_EVENTS : nullptr;
    if (tid == 0) {
        trace_stamp(tr);
        trace_smid(tr ? tr + 3 : nullptr);
    }

    // page counts and the scored-tile prefix over the sequences (every CTA;
    // CTA 0 reports length and budget errors, once per sequence)
    {
        int carry = 0;
        for (int base = 0; base < B; base += blockDim.x) {
            const int b = base + tid;
            int cnt = 0;
            if (b < B) {
                const int L = valid_len(p.seq_lens[b], p.max_pages, p.P, c == 0 ? p.status : nullptr);
                const int N = (L + p.P - 1) / p.P;
                const int k = kept_pages(N, p.budget[b], p.max_budget, p.status, c == 0);
                npages[b] = N;
                cnt = (N > 0 && (k < N || p.scores_out != nullptr)) ? (N + 15) >> 4 : 0;
            }
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += x;
            }
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            int wbase = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kSelWarps; ++w) {
                const int v = s_wsum[w];
                wbase += w < warp ? v : 0;
                total += v;
            }
            if (b < B) prefix[b] = carry + wbase + incl - cnt;
            carry += total;
            __syncthreads();
        }
        if (tid == 0) prefix[B] = carry;
        __syncthreads();
    }

    // units whose kept set needs no scores: no pages (all -1) or every page kept
    const int units = B * Hkv;
    for (int u = c; u < units; u += C) {
        const int b = u / Hkv;
        if (prefix[b + 1] != prefix[b]) continue;
        const int N = npages[b];
        int32_t *row = p.selected + (size_t)u * p.max_budget;
        for (int j = tid; j < p.max_budget; j += blockDim.x) row[j] = j < N ? j : -1;
    }

    // this warp's range of the flattened tiles
    const long long Tt = (long long)Hkv * prefix[B];
    const int GW = C * kSelWarps, gw = c * kSelWarps + warp;
    long long t = (long long)gw * Tt / GW;
    const long long t1 = (long long)(gw + 1) * Tt / GW;
    const OneWarp one{lane};
    float *const score_base = p.scores_out ? p.scores_out : p.scratch_scores;
    while (t < t1) {
        int lo = 0, hi = B - 1;   // largest b with Hkv * prefix[b] <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)Hkv * prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int cnt = prefix[b + 1] - prefix[b];          // tiles per unit of sequence b (> 0 here)
        const long long off = t - (long long)Hkv * prefix[b];
        const int h = (int)(off / cnt);
        const int j0 = (int)(off - (long long)h * cnt);
        const long long ue = (long long)Hkv * prefix[b] + (long long)(h + 1) * cnt;
        const long long s1 = ue < t1 ? ue : t1;
        const int j1 = j0 + (int)(s1 - t);
        const int u = b * Hkv + h;
        UnitPlan s;
        s.b = b;
        s.h = h;
        s.N = npages[b];
        s.k = 0;
        s.need_scores = true;
        float *sc = score_base + (size_t)u * p.max_pages;
        score_window<T, D, MMA, GMAX>(one, p, s, sc, j0, j1);
        if (s1 == t1 && lane == 0) trace_latest(tr ? tr + 1 : nullptr);
        // publish this warp's scores and count its tiles; the warp that
        // completes the unit selects it
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            const int n = j1 - j0;
            last = atomic_add_acq_rel_gpu(&p.tickets[u], n) + n == cnt;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __syncwarp();
            const int k = kept_pages(s.N, p.budget[b], p.max_budget, nullptr, false);
            warp_select_unit<kSelKeySlots>(sc, s.N, k, p.selected + (size_t)u * p.max_budget, p.max_budget);
        }
        t = s1;
    }
    if (lane == 0) trace_latest(tr ? tr + 2 : nullptr);
}

template <typename T, int D, bool MMA, int GMAX>
static cudaError_t launch_select_t(const SelectParams &p, int units, cudaStream_t stream) {
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        sms = 1;
    // one warp per tile at most: small batches launch fewer CTAs
    const long long max_tiles = (long long)units * ((p.max_pages + 15) / 16);
    long long grid = (max_tiles + kSelWarps - 1) / kSelWarps;
    if (grid > (long long)kSelCtasPerSm * sms) grid = (long long)kSelCtasPerSm * sms;
    if (const char *f = std::getenv("QASA_SELECT_CTAS")) {   // diagnostic: force the grid size
        const long long want = std::atoll(f);
        if (want >= 1 && want <= 65535) grid = want;
    }
    if (grid < 1) grid = 1;
    const size_t smem = (size_t)(2 * p.B + 1) * sizeof(int);
    auto kern = select_tiles_kernel<T, D, MMA, GMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<(unsigned)grid, 32 * kSelWarps, smem, stream>>>(p);
    return cudaGetLastError();
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
