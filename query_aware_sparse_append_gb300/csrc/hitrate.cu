// hitrate.cu -- page hit-rate instrumentation: how much of the true attention
// a page selection covers.
//
// The TinyServe abstract ("TinyServe: Query-Aware Cache Selection for Efficient
// LLM Serving") lists the page hit rate among its analyses without defining
// it.  Here it is measured against the dense attention the selection
// approximates:
//   mass(p)   share of the dense softmax weight of the unit's G query heads
//             that falls on the tokens of page p, averaged over the heads
//             (sums to 1 over the N pages of a sequence);
//   T_k       the k pages of largest mass (equal masses: lower page first),
//             k the number of pages the selection keeps;
//   hits      |selected ∩ T_k|, so the hit rate is hits / k;
//   covered   sum of mass over the selected pages;
//   best      sum of mass over T_k (the most any k-page selection can cover).
//
// page_mass_kernel: one CTA of 8 warps per (sequence, KV head).  Pass 1 reads
// every key once and keeps the online softmax maximum and sum of each query
// head; pass 2 reads the keys again and sums the normalised weights page by
// page.  A page belongs to warp (page % 8) in both passes; inside a page a
// group of lanes holds one key row (16 bytes per lane), the rows of a page are
// split over the groups, and each lane issues the loads of up to 4 rows before
// it uses the first (the kernel would otherwise wait on one load at a time).
// The per-head partial dot products are reduced by a transposing butterfly
// that leaves each lane with one head's logit, so a row costs 8 shuffles and
// one exp2 per lane instead of 8 x log2(lanes) shuffles and 8 exp2.  The logits
// are formed the same way in both passes, so every weight is exp2(z - max) <= 1.
//
// page_hit_kernel: one CTA per (sequence, KV head).  The k-th largest mass is
// found by a bitwise search over the order-preserving 32-bit key of the float;
// the pages equal to it enter T_k in page order up to the quota, decided by an
// ordered block scan.  Sums run in a fixed order (strided per-thread partials,
// butterfly inside the warp, warps in index order): the results are
// deterministic.
#include "qasa_device.cuh"
#include "qasa_launch.h"

namespace qasa {

namespace {

constexpr int kMassWarps = 8;
constexpr int kGMax = 8;
constexpr int kHitThreads = 256;
constexpr int kBatch = 4;          // key rows per lane loaded ahead of use

template <typename T, int D>
struct RowSplit {
    static constexpr int EPC = chunk16<T>::n;           // elements per 16-byte chunk
    static constexpr int CPR = D / EPC;                 // chunks per key row
    static_assert(CPR <= 32, "a key row must fit one warp at 16 bytes per lane");
    static constexpr int LPR = CPR;                     // lanes per row
    static constexpr int RPP = 32 / LPR;                // rows per warp pass
    static_assert(LPR >= 8, "the transposing reduction needs a lane per head");
    static constexpr int DUP = LPR / 8;                 // lanes holding the same head of a row
};

// Transposing reduction of the kGMax per-head partial dot products across the
// LPR lanes of a row group: at each butterfly step a lane keeps half of its
// heads and sends the other half to its partner, so after log2(kGMax) steps a
// lane holds ONE head's sum, head = (lane % LPR) / (LPR / kGMax); the remaining
// steps are plain xor adds.  kGMax + ... + 1 shuffles instead of kGMax per step.
// Partner lanes add the same two operands, so duplicates hold identical bits.
template <int OFF, int NH>
struct TransposeReduce {
    __device__ static __forceinline__ float run(float *v, int lane) {
        if constexpr (OFF == 0) {
            return v[0];
        } else if constexpr (NH > 1) {
            const bool up = (lane & OFF) != 0;
#pragma unroll
            for (int i = 0; i < NH / 2; ++i) {
                const float send = up ? v[i] : v[i + NH / 2];
                const float keep = up ? v[i + NH / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
            }
            return TransposeReduce<OFF / 2, NH / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], OFF);
            return TransposeReduce<OFF / 2, 1>::run(v, lane);
        }
    }
};

// This lane's logit scale_log2 * q_g . k for its head g (see TransposeReduce);
// heads g >= G have q = 0 and give 0.
template <typename T, int D>
__device__ __forceinline__ float row_logit(const float (&qf)[kGMax][chunk16<T>::n], const uint4 &kv,
                                           int lane) {
    using S = RowSplit<T, D>;
    float kf[S::EPC];
    chunk16<T>::unpack(kv, kf);
    float v[kGMax];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < S::EPC; ++e) acc = __fmaf_rn(qf[g][e], kf[e], acc);
        v[g] = acc;
    }
    return TransposeReduce<S::LPR / 2, kGMax>::run(v, lane);
}

// The key rows r, r + RPP, ..., r + (kBatch-1)*RPP of a page tile (16 bytes per
// lane), all loads issued before any is used; rows >= `rows` read as zero.
template <typename T, int D>
__device__ __forceinline__ void load_rows(const T *kp, int r, int rows, int csub, uint4 (&kv)[kBatch]) {
    using S = RowSplit<T, D>;
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        const int rr = r + j * S::RPP;
        kv[j] = rr < rows ? ld_global_nc_v4(kp + (size_t)rr * D + csub * S::EPC) : make_uint4(0, 0, 0, 0);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kMassWarps * 32, 2) page_mass_kernel(MassParams p) {
    using S = RowSplit<T, D>;
    constexpr int GROUPS = kMassWarps * S::RPP;
    __shared__ float st_m[GROUPS][kGMax], st_s[GROUPS][kGMax];
    __shared__ float fin_m[kGMax], fin_inv[kGMax];

    const int u = blockIdx.x, b = u / p.Hkv, h = u % p.Hkv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int rsub = lane / S::LPR, csub = lane % S::LPR;
    const int P = p.P, G = p.G;
    const int L = valid_len(p.seq_lens[b], p.max_pages, P, threadIdx.x == 0 ? p.status : nullptr);
    const int N = (L + P - 1) / P;

    float qf[kGMax][S::EPC];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
            const T *qg = static_cast<const T *>(p.q) + ((size_t)b * p.Hq + (size_t)h * G + g) * D;
            chunk16<T>::unpack(ld_global_nc_v4(qg + csub * S::EPC), qf[g]);
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) qf[g][e] *= p.scale_log2;
        } else {
#pragma unroll
            for (int e = 0; e < S::EPC; ++e) qf[g][e] = 0.f;
        }
    }
    const T *kbase = static_cast<const T *>(p.k_pool);
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages;

    // pass 1: per lane (one head of one row group), online maximum and sum of
    // exp2(z - max) over the rows of its group
    const int head = (lane % S::LPR) / S::DUP;
    float m = -INFINITY, s = 0.f;
    for (int pg = warp; pg < N; pg += kMassWarps) {
        const int phys = bt[pg];
        if (phys < 0 || phys >= p.num_phys) {
            if (lane == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
            continue;
        }
        const int rows = min(P, L - pg * P);
        const T *kp = kbase + ((size_t)phys * p.Hkv + h) * P * D;
        for (int r0 = 0; r0 < rows; r0 += kBatch * S::RPP) {
            uint4 kv[kBatch];
            load_rows<T, D>(kp, r0 + rsub, rows, csub, kv);
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (r0 + j * S::RPP >= rows) break;      // warp-uniform: no live row left
                const float z = row_logit<T, D>(qf, kv[j], lane);
                if (r0 + rsub + j * S::RPP < rows) {
                    if (z > m) {
                        s = s * exp2f(m - z) + 1.f;
                        m = z;
                    } else {
                        s += exp2f(z - m);
                    }
                }
            }
        }
    }
    if (csub % S::DUP == 0) {
        st_m[warp * S::RPP + rsub][head] = m;
        st_s[warp * S::RPP + rsub][head] = s;
    }
    __syncthreads();
    if (threadIdx.x < G) {
        const int g = threadIdx.x;
        float M = -INFINITY;
        for (int i = 0; i < GROUPS; ++i) M = fmaxf(M, st_m[i][g]);
        float Ssum = 0.f;
        if (M != -INFINITY)
            for (int i = 0; i < GROUPS; ++i)
                if (st_m[i][g] != -INFINITY) Ssum += st_s[i][g] * exp2f(st_m[i][g] - M);
        fin_m[g] = M;
        fin_inv[g] = Ssum > 0.f ? 1.f / Ssum : 0.f;
    }
    __syncthreads();
    // this lane's head: its final maximum and 1/sum, or a zero weight for a
    // duplicate lane or a head beyond the group
    const bool counts = head < G && (csub % S::DUP) == 0;
    const float Mh = counts ? fin_m[head] : 0.f;
    const float Ih = counts ? fin_inv[head] : 0.f;
    const float invG = 1.f / (float)G;

    // pass 2: normalised weights summed page by page
    float *mass = p.mass + (size_t)u * p.max_pages;
    for (int pg = warp; pg < N; pg += kMassWarps) {
        const int phys = bt[pg];
        float acc = 0.f;
        if (phys >= 0 && phys < p.num_phys) {
            const int rows = min(P, L - pg * P);
            const T *kp = kbase + ((size_t)phys * p.Hkv + h) * P * D;
            for (int r0 = 0; r0 < rows; r0 += kBatch * S::RPP) {
                uint4 kv[kBatch];
                load_rows<T, D>(kp, r0 + rsub, rows, csub, kv);
#pragma unroll
                for (int j = 0; j < kBatch; ++j) {
                    if (r0 + j * S::RPP >= rows) break;  // warp-uniform: no live row left
                    const float z = row_logit<T, D>(qf, kv[j], lane);
                    if (counts && r0 + rsub + j * S::RPP < rows) acc += exp2f(z - Mh) * Ih;
                }
            }
        }
        // add the lanes: every (row group, head) pair once
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) mass[pg] = acc * invG;
    }
}

// Order-preserving key of a float (larger float -> larger unsigned key).
__device__ __forceinline__ uint32_t float_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ int block_sum_int(int v, int *red) {
    v = __reduce_add_sync(0xffffffffu, v);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kHitThreads / 32; ++w) t += red[w];
    return t;
}

__device__ __forceinline__ float block_sum_float(float v, float *red) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kHitThreads / 32; ++w) t += red[w];
    return t;
}

__global__ void __launch_bounds__(kHitThreads) page_hit_kernel(HitParams p) {
    __shared__ uint32_t in_top[16384 / 32];
    __shared__ int ired[kHitThreads / 32];
    __shared__ float fred[kHitThreads / 32];
    const int u = blockIdx.x, b = u / p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = valid_len(p.seq_lens[b], p.max_pages, p.P, tid == 0 ? p.status : nullptr);
    const int N = (L + p.P - 1) / p.P;
    const int k = kept_pages(N, p.budget[b], p.max_budget, p.status, false);
    const float *mass = p.mass + (size_t)u * p.max_pages;

    if (k == 0) {
        if (tid == 0) { p.hits[u] = 0; p.covered[u] = 0.f; p.best[u] = 0.f; }
        return;
    }
    // the k-th largest key: largest tau with #{key >= tau} >= k
    uint32_t tau = 0;
    for (int bit = 31; bit >= 0; --bit) {
        const uint32_t cand = tau | (1u << bit);
        int c = 0;
        for (int i = tid; i < N; i += kHitThreads) c += float_key(mass[i]) >= cand;
        if (block_sum_int(c, ired) >= k) tau = cand;
    }
    int c_gt = 0;
    for (int i = tid; i < N; i += kHitThreads) c_gt += float_key(mass[i]) > tau;
    const int quota = k - block_sum_int(c_gt, ired);     // pages equal to tau that enter T_k

    for (int i = tid; i < (N + 31) / 32; i += kHitThreads) in_top[i] = 0u;
    __syncthreads();
    // ordered scan of the pages equal to tau: the first `quota` of them count
    int base = 0;
    for (int i0 = 0; i0 < N; i0 += kHitThreads) {
        const int i = i0 + tid;
        const uint32_t key = i < N ? float_key(mass[i]) : 0u;
        const bool eq = i < N && key == tau;
        const unsigned bal = __ballot_sync(0xffffffffu, eq);
        __syncthreads();
        if (lane == 0) ired[warp] = __popc(bal);
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; ++w) before += ired[w];
        before += __popc(bal & ((1u << lane) - 1u));
        const bool top = i < N && (key > tau || (eq && before < quota));
        if (top) atomicOr(&in_top[i >> 5], 1u << (i & 31));
        for (int w = 0; w < kHitThreads / 32; ++w) base += ired[w];
    }
    __syncthreads();

    float bsum = 0.f;
    for (int i = tid; i < N; i += kHitThreads)
        if (in_top[i >> 5] & (1u << (i & 31))) bsum += mass[i];
    const float best = block_sum_float(bsum, fred);

    const int32_t *sel = p.selected + (size_t)u * p.max_budget;
    float csum = 0.f;
    int h = 0;
    for (int j = tid; j < k; j += kHitThreads) {
        const int sp = sel[j];
        if (sp < 0 || sp >= N) {
            if (p.status) atomicOr(p.status, QASA_DEVERR_SELECTED);
            continue;
        }
        csum += mass[sp];
        h += (in_top[sp >> 5] >> (sp & 31)) & 1u;
    }
    const float covered = block_sum_float(csum, fred);
    const int hits = block_sum_int(h, ired);
    if (tid == 0) {
        p.hits[u] = hits;
        p.covered[u] = covered;
        p.best[u] = best;
    }
}

template <typename T, int D>
cudaError_t launch_mass_t(const MassParams &p, int units, cudaStream_t stream) {
    page_mass_kernel<T, D><<<units, kMassWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_page_mass(qasa_dtype dt, int D, const MassParams &p, int units, cudaStream_t stream) {
    if (units == 0) return cudaSuccess;
    if (dt == QASA_DTYPE_F32) return D == 64 ? launch_mass_t<float, 64>(p, units, stream)
                                             : launch_mass_t<float, 128>(p, units, stream);
    if (dt == QASA_DTYPE_F16) return D == 64 ? launch_mass_t<__half, 64>(p, units, stream)
                                             : launch_mass_t<__half, 128>(p, units, stream);
    return D == 64 ? launch_mass_t<__nv_bfloat16, 64>(p, units, stream)
                   : launch_mass_t<__nv_bfloat16, 128>(p, units, stream);
}

cudaError_t launch_page_hit(const HitParams &p, int units, cudaStream_t stream) {
    if (units == 0) return cudaSuccess;
    page_hit_kernel<<<units, kHitThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace qasa
