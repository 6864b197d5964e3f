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
// One CTA (4 warps) per (sequence, KV head).  Two scoring paths:
//
//  * tensor cores (16-bit KV, G >= 2).  Because lo <= hi, the per-channel
//    maximum equals q+ * hi + q- * lo with q+ = max(q,0), q- = min(q,0): the
//    scores of 16 pages are one [16 x 2d] x [2d x 8] contraction, run as
//    m16n8k16 MMAs with the box rows (lo | hi, contiguous) as the A operand and
//    [q- ; q+] as the B operand.  Products of 16-bit values are exact in fp32.
//    Each lane loads 16-byte chunks of the box rows straight into A-fragment
//    registers: the channel order inside the contraction is permuted
//    consistently for A and B, which the sum does not see.
//  * FFMA (G == 1, or fp32 KV): a warp scores a few pages at a time with
//    16-byte loads and shuffle reductions.
//
// Selection: radix select (4 passes of 8 bits, warp-aggregated shared-memory
// histograms) finds the key of the (k-2)-th best candidate; an ordered block
// scan then keeps every candidate above it and the lowest-index ones equal to
// it, and compacts the kept ids in ascending order.
#include "qasa_device.cuh"
#include "qasa_launch.h"

namespace qasa {


constexpr int SEL_THREADS = 128;

// Key whose unsigned order is the ranking order: larger score first; -0 and +0
// are the same score; NaN ranks below every number.
__device__ __forceinline__ uint32_t rank_key(float f) {
    if (f != f) return 0u;
    if (f == 0.0f) f = 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the 128 threads of the CTA.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    __syncthreads();
    return base + incl - v;
}

// ----------------------------------------------------------- scoring paths

// Tensor-core scores of all N pages into sc[] (16-bit KV, 2 <= G <= 8).
template <typename T, int D>
__device__ void score_pages_mma(const SelectParams &p, int b, int h, int N, float *sc) {
    constexpr int J = D / 16;          // 16-byte chunks per lane per box row (2D elements / 8 / 4 lanes)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane & 3, n = lane >> 2;

    // B fragments: chunk x = c + 4*jj of the [q- (lo half) | q+ (hi half)] row of head n.
    uint32_t qf[J][4];
    const T *qrow = static_cast<const T *>(p.q) + ((size_t)b * p.Hq + (size_t)h * p.G + n) * D;
#pragma unroll
    for (int jj = 0; jj < J; ++jj) {
        const int x = c + 4 * jj;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (n < p.G) raw = *reinterpret_cast<const uint4 *>(qrow + (x % (D / 8)) * 8);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t neg = ((w[i] & 0x80008000u) >> 15) * 0xffffu;   // 0xffff per negative half
            qf[jj][i] = (x < D / 8) ? (w[i] & neg) : (w[i] & ~neg);
        }
    }

    const T *bounds = static_cast<const T *>(p.bounds);
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages;
    const int ntiles = (N + 15) >> 4;
    for (int t = warp; t < ntiles; t += SEL_THREADS / 32) {
        const int r0 = t * 16 + n, r1 = r0 + 8;
        int ph0 = r0 < N ? bt[r0] : -1;
        int ph1 = r1 < N ? bt[r1] : -1;
        const bool ok0 = ph0 >= 0 && ph0 < p.num_phys, ok1 = ph1 >= 0 && ph1 < p.num_phys;
        if (((r0 < N && !ok0) || (r1 < N && !ok1)) && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        const T *row0 = bounds + ((size_t)(ok0 ? ph0 : 0) * p.Hkv + h) * 2 * D;
        const T *row1 = bounds + ((size_t)(ok1 ? ph1 : 0) * p.Hkv + h) * 2 * D;
        uint4 a0[J], a1[J];
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            a0[jj] = ok0 ? ld_global_nc_v4(row0 + (c + 4 * jj) * 8) : make_uint4(0, 0, 0, 0);
            a1[jj] = ok1 ? ld_global_nc_v4(row1 + (c + 4 * jj) * 8) : make_uint4(0, 0, 0, 0);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            const uint32_t fa[4] = {a0[jj].x, a1[jj].x, a0[jj].y, a1[jj].y};
            mma16816<T>::run(acc, fa, qf[jj][0], qf[jj][1]);
            const uint32_t fb[4] = {a0[jj].z, a1[jj].z, a0[jj].w, a1[jj].w};
            mma16816<T>::run(acc, fb, qf[jj][2], qf[jj][3]);
        }
        // acc = S[r0][2c], S[r0][2c+1], S[r1][2c], S[r1][2c+1]; maximum over valid heads
        const bool g0 = 2 * c < p.G, g1 = 2 * c + 1 < p.G;
        float m0 = fmaxf(g0 ? acc[0] : -INFINITY, g1 ? acc[1] : -INFINITY);
        float m1 = fmaxf(g0 ? acc[2] : -INFINITY, g1 ? acc[3] : -INFINITY);
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
        if (c == 0) {
            if (r0 < N) sc[r0] = ok0 ? m0 : -INFINITY;
            if (r1 < N) sc[r1] = ok1 ? m1 : -INFINITY;
        }
    }
}

// FFMA scores (any dtype, G <= GMAX).
template <typename T, int D, int GMAX>
__device__ void score_pages_ffma(const SelectParams &p, int b, int h, int N, float *sc) {
    constexpr int EPC = chunk16<T>::n;
    constexpr int CPR = 2 * D / EPC;             // chunks per box row (lo | hi)
    constexpr int LPR = CPR < 32 ? CPR : 32;     // lanes per row
    constexpr int CPL = CPR / LPR;               // chunks per lane
    constexpr int RPW = 32 / LPR;                // rows per warp pass
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rsub = lane / LPR, csub = lane % LPR;
    const int G = p.G;

    float qq[GMAX][CPL][EPC];
    const T *qb = static_cast<const T *>(p.q) + ((size_t)b * p.Hq + (size_t)h * G) * D;
#pragma unroll
    for (int g = 0; g < GMAX; ++g)
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                const int idx = (csub + LPR * i) * EPC + e;   // element of the lo|hi row
                float v = 0.f;
                if (g < G) {
                    const float qv = elem<T>::to_f(qb[(size_t)g * D + (idx % D)]);
                    v = idx < D ? fminf(qv, 0.f) : fmaxf(qv, 0.f);
                }
                qq[g][i][e] = v;
            }

    const T *bounds = static_cast<const T *>(p.bounds);
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages;
    const int npass = (N + RPW - 1) / RPW;
    for (int pass = warp; pass < npass; pass += SEL_THREADS / 32) {
        const int page = pass * RPW + rsub;
        int ph = page < N ? bt[page] : -1;
        const bool ok = ph >= 0 && ph < p.num_phys;
        if (page < N && !ok && csub == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        const T *row = bounds + ((size_t)(ok ? ph : 0) * p.Hkv + h) * 2 * D;
        float acc[GMAX];
#pragma unroll
        for (int g = 0; g < GMAX; ++g) acc[g] = 0.f;
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
            float f[EPC];
            uint4 raw = ok ? ld_global_nc_v4(row + (csub + LPR * i) * EPC) : make_uint4(0, 0, 0, 0);
            chunk16<T>::unpack(raw, f);
#pragma unroll
            for (int g = 0; g < GMAX; ++g)
#pragma unroll
                for (int e = 0; e < EPC; ++e) acc[g] = fmaf(qq[g][i][e], f[e], acc[g]);
        }
        float best = -INFINITY;
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            float a = acc[g];
#pragma unroll
            for (int off = 1; off < LPR; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (g < G) best = fmaxf(best, a);
        }
        if (csub == 0 && page < N) sc[page] = ok ? best : -INFINITY;
    }
}

// ------------------------------------------------------------------ kernel

template <typename T, int D, bool MMA, int GMAX>
__global__ void __launch_bounds__(SEL_THREADS, 4) select_kernel(SelectParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float *sc = reinterpret_cast<float *>(smem_raw);   // [max_pages] scores, then keys in place
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw);
    __shared__ int hist[256];
    __shared__ int warp_tot[SEL_THREADS / 32];
    __shared__ int s_digit, s_above;

    pdl_launch_dependents();

    const int u = blockIdx.x;
    const int b = u / p.Hkv, h = u % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = valid_len(p.seq_lens[b], p.max_pages, p.P, (h == 0 && tid == 0) ? p.status : nullptr);
    const int N = (L + p.P - 1) / p.P;
    const int k = kept_pages(N, p.budget[b], p.max_budget, p.status, h == 0 && tid == 0);
    int32_t *selrow = p.selected + (size_t)u * p.max_budget;
    if (tid == 0) p.counters[u] = 0;

    if (N == 0) {
        for (int j = tid; j < p.max_budget; j += SEL_THREADS) selrow[j] = -1;
        return;
    }
    const bool need_scores = (k < N) || (p.scores_out != nullptr);
    if (need_scores) {
        if constexpr (MMA) score_pages_mma<T, D>(p, b, h, N, sc);
        else score_pages_ffma<T, D, GMAX>(p, b, h, N, sc);
        __syncthreads();
        if (p.scores_out)
            for (int i = tid; i < N; i += SEL_THREADS)
                p.scores_out[(size_t)u * p.max_pages + i] = sc[i];
    }
    if (k >= N) {
        for (int j = tid; j < p.max_budget; j += SEL_THREADS) selrow[j] = j < N ? j : -1;
        return;
    }
    // here N >= 2: forced pages {0, N-1}; candidates 1..N-2; choose kc of them
    const int kc = k - 2;
    const int last = N - 1;
    if (kc == 0) {
        for (int j = tid; j < p.max_budget; j += SEL_THREADS) selrow[j] = j == 0 ? 0 : (j == 1 ? last : -1);
        return;
    }
    for (int i = tid; i < N; i += SEL_THREADS) keys[i] = rank_key(sc[i]);
    __syncthreads();

    // radix select: tau = key of the kc-th largest candidate
    uint32_t prefix = 0, pmask = 0;
    int need = kc;
    const int iters = (N - 2 + SEL_THREADS - 1) / SEL_THREADS;
#pragma unroll 1
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += SEL_THREADS) hist[i] = 0;
        __syncthreads();
        for (int it = 0; it < iters; ++it) {
            const int i = 1 + it * SEL_THREADS + tid;
            const bool in = i <= N - 2;
            const uint32_t key = in ? keys[i] : 0u;
            const bool match = in && ((key & pmask) == prefix);
            const unsigned active = __ballot_sync(0xffffffffu, match);
            if (match) {
                const int digit = (key >> shift) & 255;
                const unsigned peers = __match_any_sync(active, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
            }
        }
        __syncthreads();
        if (warp == 0) {
            int cnt[8], tot = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) { cnt[j] = hist[255 - 8 * lane - j]; tot += cnt[j]; }
            int incl = tot;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            const int excl = incl - tot;
            if (excl < need && need <= incl) {
                int run = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (run + cnt[j] >= need) { s_digit = 255 - 8 * lane - j; s_above = run; break; }
                    run += cnt[j];
                }
            }
        }
        __syncthreads();
        need -= s_above;
        prefix |= (uint32_t)s_digit << shift;
        pmask |= 0xffu << shift;
    }
    const uint32_t tau = prefix;   // `need` candidates equal to tau are kept (lowest indices)

    // ordered passes over contiguous index segments: rank among equals, then compaction
    const int E = (N + SEL_THREADS - 1) / SEL_THREADS;
    const int i0 = min(N, tid * E), i1 = min(N, i0 + E);
    int eq = 0;
    for (int i = i0; i < i1; ++i)
        if (i >= 1 && i <= N - 2 && keys[i] == tau) ++eq;
    int eq_rank = block_excl_scan(eq, warp_tot);
    int kept = 0;
    {
        int r = eq_rank;
        for (int i = i0; i < i1; ++i) {
            bool take;
            if (i == 0 || i == last) take = true;
            else {
                const uint32_t key = keys[i];
                take = key > tau || (key == tau && r < need);
                if (key == tau) ++r;
            }
            kept += take;
        }
    }
    int pos = block_excl_scan(kept, warp_tot);
    {
        int r = eq_rank;
        for (int i = i0; i < i1; ++i) {
            bool take;
            if (i == 0 || i == last) take = true;
            else {
                const uint32_t key = keys[i];
                take = key > tau || (key == tau && r < need);
                if (key == tau) ++r;
            }
            if (take && pos < p.max_budget) selrow[pos++] = i;
        }
    }
    for (int j = k + tid; j < p.max_budget; j += SEL_THREADS) selrow[j] = -1;
}

template <typename T, int D, bool MMA, int GMAX>
static cudaError_t launch_select_t(const SelectParams &p, int units, cudaStream_t stream) {
    const size_t smem = (size_t)p.max_pages * sizeof(float);
    auto kern = select_kernel<T, D, MMA, GMAX>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<units, SEL_THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_select(qasa_dtype dt, int D, const SelectParams &p, int units,
                          cudaStream_t stream) {
    const bool mma = dt != QASA_DTYPE_F32 && p.G >= 2;
    if (dt == QASA_DTYPE_F32)
        return D == 64 ? launch_select_t<float, 64, false, 8>(p, units, stream)
                       : launch_select_t<float, 128, false, 8>(p, units, stream);
    if (dt == QASA_DTYPE_F16) {
        if (mma) return D == 64 ? launch_select_t<__half, 64, true, 1>(p, units, stream)
                                : launch_select_t<__half, 128, true, 1>(p, units, stream);
        return D == 64 ? launch_select_t<__half, 64, false, 1>(p, units, stream)
                       : launch_select_t<__half, 128, false, 1>(p, units, stream);
    }
    if (mma) return D == 64 ? launch_select_t<__nv_bfloat16, 64, true, 1>(p, units, stream)
                            : launch_select_t<__nv_bfloat16, 128, true, 1>(p, units, stream);
    return D == 64 ? launch_select_t<__nv_bfloat16, 64, false, 1>(p, units, stream)
                   : launch_select_t<__nv_bfloat16, 128, false, 1>(p, units, stream);
}

}  // namespace qasa
