// select_device.cuh -- query-aware page scoring and top-k selection of ONE
// (sequence, KV head), run by a group of NT threads.  Used by the standalone
// selection kernel (the whole CTA is the group), by its cluster form (each CTA
// of a cluster scores a window of the unit's tiles with score_window, the first
// runs select_from_scores) and by the single-launch decode kernel (four
// selector warps of a larger CTA, synchronised by a named barrier).
//
// "TinyServe: Query-Aware Cache Selection for Efficient LLM Serving",
// 方法详解 / 关键设计: at decode time the query is compared with the bounding
// box of every KV block and the most similar blocks are kept.  For every page
// p of the sequence
//
//     s(p) = max_g  sum_c max(q[g][c] * lo[p][c], q[g][c] * hi[p][c])      (fp32)
//
// over the G query heads of the group; the sink page 0, the newest page N-1
// and the best (k - 2) remaining pages (ties to the lower index) are kept and
// written as ascending logical ids.
//
// Two scoring paths:
//  * tensor cores (16-bit and FP8 KV, any group size: the unused query heads
//    of the 8-wide MMA are zero).  Because lo <= hi, the per-channel
//    maximum equals q+ * hi + q- * lo with q+ = max(q,0), q- = min(q,0): the
//    scores of 16 pages are one [16 x 2d] x [2d x 8] contraction, run as
//    m16n8k16 MMAs with the box rows (lo | hi, contiguous) as the A operand and
//    [q- ; q+] as the B operand.  Products of 16-bit values are exact in fp32.
//    Each lane loads 16-byte chunks of the box rows straight into A-fragment
//    registers: the channel order inside the contraction is permuted
//    consistently for A and B, which the sum does not see.
//  * FFMA (fp32 KV): a warp scores a few pages at a time with 16-byte loads
//    and shuffle reductions.
//
// Selection: the key of the (k-2)-th best candidate is narrowed down by
// shared-memory histograms of 10-bit digits (usually one pass); an ordered
// group scan then keeps every candidate above it and the lowest-index ones
// equal to it, and compacts the kept ids in ascending order.
#pragma once

#include "qasa_device.cuh"
#include "qasa_launch.h"

namespace qasa {

// A group of NT threads (a multiple of 32) that selects together.  BAR < 0:
// the group is the whole CTA (__syncthreads); otherwise named barrier BAR.
template <int NT, int BAR>
struct SelGroup {
    static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
    int tid;   // 0 .. NT-1
    __device__ __forceinline__ void sync() const {
        if constexpr (BAR < 0) __syncthreads();
        else named_barrier_sync(BAR, NT);
    }
    __device__ __forceinline__ int lane() const { return tid & 31; }
    __device__ __forceinline__ int warp() const { return tid >> 5; }
    static constexpr int warps = NT / 32;
};

// Shared scratch of one group: histogram, per-warp totals, search results.
constexpr int kSelBins = 1024;   // histogram bins of the selection (10-bit digits)

struct __align__(16) SelScratch {
    union {
        int hist[kSelBins];
        uint32_t list[kSelBins];   // keys sharing the final prefix (once the histogram is done)
    };
    int warp_tot[32];
    uint32_t kmin[32], kmax[32];
    int digit, above, cnt, gathered;
    uint32_t tau;
};

// Key whose unsigned order is the ranking order: larger score first; -0 and +0
// are the same score; NaN ranks below every number.
__device__ __forceinline__ uint32_t rank_key(float f) {
    if (f != f) return 0u;
    if (f == 0.0f) f = 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive scan over the threads of the group.
template <class Grp>
__device__ __forceinline__ int group_excl_scan(const Grp &g, int v, int *warp_tot) {
    const int lane = g.lane(), warp = g.warp();
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    g.sync();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    g.sync();
    return base + incl - v;
}

// Exclusive scan over the threads of the group, and the group's total.
template <class Grp>
__device__ __forceinline__ int group_excl_scan_total(const Grp &g, int v, int *warp_tot, int &total) {
    const int lane = g.lane(), warp = g.warp();
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    if (lane == 31) warp_tot[warp] = incl;
    g.sync();
    int base = 0, tot = 0;
    for (int w = 0; w < Grp::warps; ++w) {
        const int x = warp_tot[w];
        base += w < warp ? x : 0;
        tot += x;
    }
    g.sync();
    total = tot;
    return base + incl - v;
}

// ----------------------------------------------------------- scoring paths

// Tensor-core scores of the pages of 16-page tiles [t_begin, t_end) (pages
// below N) into sc[] (16-bit KV, 1 <= G <= 8).
template <typename T, int D, class Grp>
__device__ void score_pages_mma(const Grp &grp, const SelectParams &p, int b, int h, int N, float *sc,
                                int t_begin, int t_end) {
    constexpr int J = D / 16;          // 16-byte chunks per lane per box row (2D elements / 8 / 4 lanes)
    const int lane = grp.lane(), warp = grp.warp();
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
    // the block-table entries of a warp's next tile are loaded while its
    // current tile's boxes are in flight (one dependent round trip per tile),
    // and the next tile's box rows are prefetched into L2 (one bulk prefetch
    // per page row from lanes 0-15) together with the current tile's loads,
    // so that every warp keeps two tiles on their way from HBM
    constexpr int ROWB = 2 * D * (int)sizeof(T);
    const int tw = t_begin + warp;
    int nph0 = tw < t_end && tw * 16 + n < N ? bt[tw * 16 + n] : -1;
    int nph1 = tw < t_end && tw * 16 + n + 8 < N ? bt[tw * 16 + n + 8] : -1;
    int pf = tw + Grp::warps < t_end && lane < 16 && (tw + Grp::warps) * 16 + lane < N
                 ? bt[(tw + Grp::warps) * 16 + lane] : -1;
    for (int t = tw; t < t_end; t += Grp::warps) {
        const int r0 = t * 16 + n, r1 = r0 + 8;
        const int ph0 = nph0, ph1 = nph1;
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
        if (pf >= 0 && pf < p.num_phys) bulk_prefetch_l2(bounds + ((size_t)pf * p.Hkv + h) * 2 * D, ROWB);
        {
            const bool more = t + Grp::warps < t_end;
            const int q0 = (t + Grp::warps) * 16 + n;
            nph0 = more && q0 < N ? bt[q0] : -1;
            nph1 = more && q0 + 8 < N ? bt[q0 + 8] : -1;
            const int f = (t + 2 * Grp::warps) * 16 + lane;
            pf = t + 2 * Grp::warps < t_end && lane < 16 && f < N ? bt[f] : -1;
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

// Shared-memory staging of box rows for the tensor-core scoring of the
// single-launch kernel, where only four warps per SM select and loading box
// rows straight into registers would leave them waiting on one round trip
// per 16-page tile.  Each (page, KV head) box is 2*d*es contiguous bytes; one
// bulk async copy per page lands it in a slot row padded to 2*d*es + 64 bytes,
// so that the fragment reads (8 rows x 4 chunks per quarter warp) hit 8
// different 16-byte bank groups.  Every selector warp owns `slots_per_warp`
// slots (one mbarrier each) and keeps that many tiles in flight.
struct BoxStage {
    unsigned char *buf;           // [4 warps * slots_per_warp][16 rows][pitch]
    uint64_t *bar;                // [4 warps * slots_per_warp], arrival count 1
    int32_t *phys;                // [max_pages] the unit's physical pages (-1: invalid)
    int slots_per_warp;
    unsigned long long wait_limit_ns;
};

template <typename T, int D>
struct BoxStageShape {
    static constexpr int ROWB = 2 * D * (int)sizeof(T);   // one box: lo row, hi row
    static constexpr int PITCH = ROWB + 64;
    static constexpr int TILEB = 16 * PITCH;
};

// Tensor-core scores of all N pages into sc[] from staged box rows (16-bit KV,
// 1 <= G <= 8).  phase_bits holds the parity of this warp's slot barriers and
// persists across units.  Every copy issued here is waited for before return.
template <typename T, int D, class Grp>
__device__ void score_pages_mma_staged(const Grp &grp, const SelectParams &p, int b, int h, int N,
                                       float *sc, const BoxStage &st, uint32_t &phase_bits) {
    using SH = BoxStageShape<T, D>;
    constexpr int J = D / 16;
    constexpr int NT = Grp::warps * 32;
    const int lane = grp.lane(), warp = grp.warp();
    const int c = lane & 3, n = lane >> 2;

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
            const uint32_t neg = ((w[i] & 0x80008000u) >> 15) * 0xffffu;
            qf[jj][i] = (x < D / 8) ? (w[i] & neg) : (w[i] & ~neg);
        }
    }

    // the unit's block-table row, checked once
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages;
    for (int i = grp.tid; i < N; i += NT) {
        const int ph = bt[i];
        const bool ok = ph >= 0 && ph < p.num_phys;
        if (!ok && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        st.phys[i] = ok ? ph : -1;
    }
    grp.sync();

    const T *bounds = static_cast<const T *>(p.bounds);
    const int ntiles = (N + 15) >> 4;
    const int SPW = st.slots_per_warp;
    auto issue = [&](int t, int k) {                 // tile t into this warp's slot k
        const int slot = warp * SPW + k;
        const int r = t * 16 + lane;
        const int ph = (lane < 16 && r < N) ? st.phys[r] : -1;
        const unsigned m = __ballot_sync(0xffffffffu, ph >= 0);
        if (lane == 0) mbar_arrive_expect_tx(&st.bar[slot], (uint32_t)__popc(m) * SH::ROWB);
        __syncwarp();
        if (ph >= 0)
            bulk_load(st.buf + (size_t)slot * SH::TILEB + lane * SH::PITCH,
                      bounds + ((size_t)ph * p.Hkv + h) * 2 * D, SH::ROWB, &st.bar[slot]);
    };
    for (int k = 0; k < SPW; ++k) {
        const int t = warp + k * Grp::warps;
        if (t < ntiles) issue(t, k);
    }
    int k = 0;
    for (int t = warp; t < ntiles; t += Grp::warps) {
        const int slot = warp * SPW + k;
        if (!mbar_wait_bounded(&st.bar[slot], (phase_bits >> k) & 1u, st.wait_limit_ns)) {
            if (lane == 0 && p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
        }
        phase_bits ^= 1u << k;
        const unsigned char *src = st.buf + (size_t)slot * SH::TILEB;
        const int r0 = t * 16 + n, r1 = r0 + 8;
        const bool ok0 = r0 < N && st.phys[r0] >= 0, ok1 = r1 < N && st.phys[r1] >= 0;
        uint4 a0[J], a1[J];
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            a0[jj] = ok0 ? *reinterpret_cast<const uint4 *>(src + n * SH::PITCH + (c + 4 * jj) * 16)
                         : make_uint4(0, 0, 0, 0);
            a1[jj] = ok1 ? *reinterpret_cast<const uint4 *>(src + (n + 8) * SH::PITCH + (c + 4 * jj) * 16)
                         : make_uint4(0, 0, 0, 0);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
            const uint32_t fa[4] = {a0[jj].x, a1[jj].x, a0[jj].y, a1[jj].y};
            mma16816<T>::run(acc, fa, qf[jj][0], qf[jj][1]);
            const uint32_t fb[4] = {a0[jj].z, a1[jj].z, a0[jj].w, a1[jj].w};
            mma16816<T>::run(acc, fb, qf[jj][2], qf[jj][3]);
        }
        // the MMAs have consumed every fragment of the slot: refill it
        __syncwarp();
        {
            const int tn = t + SPW * Grp::warps;
            if (tn < ntiles) issue(tn, k);
        }
        if (++k == SPW) k = 0;
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

// FP8 boxes (E4M3 codes, scale amax_K / 448 per page): tensor-core scores of the
// codes, converted to halves exactly, times the page's scale (the common
// factor of every box value of the page).  Lane c holds 16-byte code chunks
// k = c + 4m of the [lo | hi] row, i.e. half chunks 2k and 2k+1, which feed MMA
// slots 2m and 2m+1; the q fragments use the same channel order.
template <int D, class Grp>
__device__ void score_pages_fp8_mma(const Grp &grp, const SelectParams &p, int b, int h, int N, float *sc,
                                    int t_begin, int t_end) {
    constexpr int J = D / 16;          // MMA slots per lane per box row, as in the 16-bit path
    constexpr int JC = J / 2;          // 16-byte code chunks per lane per box row
    const int lane = grp.lane(), warp = grp.warp();
    const int c = lane & 3, n = lane >> 2;

    uint32_t qf[J][4];
    const __half *qrow = static_cast<const __half *>(p.q) + ((size_t)b * p.Hq + (size_t)h * p.G + n) * D;
#pragma unroll
    for (int jj = 0; jj < J; ++jj) {
        const int x = 2 * c + 8 * (jj >> 1) + (jj & 1);   // half chunk of the [lo | hi] row
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (n < p.G) raw = *reinterpret_cast<const uint4 *>(qrow + (x % (D / 8)) * 8);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t neg = ((w[i] & 0x80008000u) >> 15) * 0xffffu;
            qf[jj][i] = (x < D / 8) ? (w[i] & neg) : (w[i] & ~neg);
        }
    }

    const uint8_t *bounds = static_cast<const uint8_t *>(p.bounds);
    const int32_t *bt = p.block_table + (size_t)b * p.max_pages;
    const int tw = t_begin + warp;
    int nph0 = tw < t_end && tw * 16 + n < N ? bt[tw * 16 + n] : -1;
    int nph1 = tw < t_end && tw * 16 + n + 8 < N ? bt[tw * 16 + n + 8] : -1;
    for (int t = tw; t < t_end; t += Grp::warps) {
        const int r0 = t * 16 + n, r1 = r0 + 8;
        const int ph0 = nph0, ph1 = nph1;
        {
            const bool more = t + Grp::warps < t_end;
            const int q0 = (t + Grp::warps) * 16 + n;
            nph0 = more && q0 < N ? bt[q0] : -1;
            nph1 = more && q0 + 8 < N ? bt[q0 + 8] : -1;
        }
        const bool ok0 = ph0 >= 0 && ph0 < p.num_phys, ok1 = ph1 >= 0 && ph1 < p.num_phys;
        if (((r0 < N && !ok0) || (r1 < N && !ok1)) && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        const size_t e0 = (size_t)(ok0 ? ph0 : 0) * p.Hkv + h, e1 = (size_t)(ok1 ? ph1 : 0) * p.Hkv + h;
        const uint8_t *row0 = bounds + e0 * 2 * D;
        const uint8_t *row1 = bounds + e1 * 2 * D;
        const float am0 = ok0 ? p.scales[e0 * 4] : 0.f, am1 = ok1 ? p.scales[e1 * 4] : 0.f;
        uint4 c0[JC], c1[JC];
#pragma unroll
        for (int m = 0; m < JC; ++m) {
            c0[m] = ok0 ? ld_global_nc_v4(row0 + (c + 4 * m) * 16) : make_uint4(0, 0, 0, 0);
            c1[m] = ok1 ? ld_global_nc_v4(row1 + (c + 4 * m) * 16) : make_uint4(0, 0, 0, 0);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < JC; ++m) {
            uint4 l0, h0, l1, h1;
            e4m3x16_to_h(c0[m], l0, h0);
            e4m3x16_to_h(c1[m], l1, h1);
            {
                const uint32_t fa[4] = {l0.x, l1.x, l0.y, l1.y};
                mma16816<__half>::run(acc, fa, qf[2 * m][0], qf[2 * m][1]);
                const uint32_t fb[4] = {l0.z, l1.z, l0.w, l1.w};
                mma16816<__half>::run(acc, fb, qf[2 * m][2], qf[2 * m][3]);
            }
            {
                const uint32_t fa[4] = {h0.x, h1.x, h0.y, h1.y};
                mma16816<__half>::run(acc, fa, qf[2 * m + 1][0], qf[2 * m + 1][1]);
                const uint32_t fb[4] = {h0.z, h1.z, h0.w, h1.w};
                mma16816<__half>::run(acc, fb, qf[2 * m + 1][2], qf[2 * m + 1][3]);
            }
        }
        const bool g0 = 2 * c < p.G, g1 = 2 * c + 1 < p.G;
        float m0 = fmaxf(g0 ? acc[0] : -INFINITY, g1 ? acc[1] : -INFINITY);
        float m1 = fmaxf(g0 ? acc[2] : -INFINITY, g1 ? acc[3] : -INFINITY);
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 1));
        m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, 2));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 1));
        m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, 2));
        if (c == 0) {
            if (r0 < N) sc[r0] = ok0 ? __fmul_rn(m0, fp8_scale(am0)) : -INFINITY;
            if (r1 < N) sc[r1] = ok1 ? __fmul_rn(m1, fp8_scale(am1)) : -INFINITY;
        }
    }
}

// FFMA scores (fp32 boxes, G <= GMAX) of the pages of 16-page tiles
// [t_begin, t_end) below N.
template <typename T, int D, int GMAX, class Grp>
__device__ void score_pages_ffma(const Grp &grp, const SelectParams &p, int b, int h, int N, float *sc,
                                 int t_begin, int t_end) {
    constexpr int EPC = chunk16<T>::n;
    constexpr int CPR = 2 * D / EPC;             // chunks per box row (lo | hi)
    constexpr int LPR = CPR < 32 ? CPR : 32;     // lanes per row
    constexpr int CPL = CPR / LPR;               // chunks per lane
    constexpr int RPW = 32 / LPR;                // rows per warp pass
    static_assert(16 % RPW == 0, "a tile holds whole passes");
    const int lane = grp.lane(), warp = grp.warp();
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
    const int pass_begin = t_begin * 16 / RPW;
    const int npass = (min(N, t_end * 16) + RPW - 1) / RPW;
    // NB passes per round: their block-table loads, then their box loads, are
    // all in flight together (two round trips per NB passes, not per pass)
    constexpr int NB = 4;
    for (int pass0 = pass_begin + warp; pass0 < npass; pass0 += Grp::warps * NB) {
        int page[NB];
        bool ok[NB];
        uint4 raw[NB][CPL];
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            page[q] = (pass0 + q * Grp::warps) * RPW + rsub;
            const bool in = pass0 + q * Grp::warps < npass && page[q] < N;
            const int ph = in ? bt[page[q]] : -1;
            ok[q] = ph >= 0 && ph < p.num_phys;
            if (in && !ok[q] && csub == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
            const T *row = bounds + ((size_t)(ok[q] ? ph : 0) * p.Hkv + h) * 2 * D;
#pragma unroll
            for (int i = 0; i < CPL; ++i)
                raw[q][i] = ok[q] ? ld_global_nc_v4(row + (csub + LPR * i) * EPC) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < NB; ++q) {
            if (pass0 + q * Grp::warps >= npass) break;      // warp-uniform
            float acc[GMAX];
#pragma unroll
            for (int g = 0; g < GMAX; ++g) acc[g] = 0.f;
#pragma unroll
            for (int i = 0; i < CPL; ++i) {
                float f[EPC];
                chunk16<T>::unpack(raw[q][i], f);
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
            if (csub == 0 && page[q] < N) sc[page[q]] = ok[q] ? best : -INFINITY;
        }
    }
}

// ------------------------------------------------------------ one unit

// What every thread (and, in a cluster split, every CTA) of unit u = (b, h)
// knows before scoring: its page count, its kept count, whether scores are
// needed.  `report`: this thread reports the sequence's length and budget
// errors (one thread per sequence does).
struct UnitPlan {
    int b, h, N, k;
    bool need_scores;
};

__device__ __forceinline__ UnitPlan plan_unit(const SelectParams &p, int u, bool report) {
    UnitPlan s;
    s.b = u / p.Hkv;
    s.h = u % p.Hkv;
    const bool rep = report && s.h == 0;
    const int L = valid_len(p.seq_lens[s.b], p.max_pages, p.P, rep ? p.status : nullptr);
    s.N = (L + p.P - 1) / p.P;
    s.k = kept_pages(s.N, p.budget[s.b], p.max_budget, p.status, rep);
    // The scores decide the kept set only when some candidate is left out and
    // at least one is kept beside the two forced pages (k > 2).
    s.need_scores = s.N > 0 && ((s.k < s.N && s.k > 2) || (p.scores_out != nullptr));
    return s;
}

// Scores of the unit's pages in 16-page tiles [t_begin, t_end) into sc[page]
// (sc may point into another CTA's shared memory of the cluster).
template <typename T, int D, bool MMA, int GMAX, class Grp>
__device__ __forceinline__ void score_window(const Grp &grp, const SelectParams &p, const UnitPlan &s, float *sc,
                                             int t_begin, int t_end) {
    if constexpr (is_fp8<T>::value) {
        score_pages_fp8_mma<D>(grp, p, s.b, s.h, s.N, sc, t_begin, t_end);
    } else if constexpr (MMA) {
        score_pages_mma<T, D>(grp, p, s.b, s.h, s.N, sc, t_begin, t_end);
    } else {
        score_pages_ffma<T, D, GMAX>(grp, p, s.b, s.h, s.N, sc, t_begin, t_end);
    }
}

template <class Grp>
__device__ void select_from_scores(const Grp &grp, const SelectParams &p, int u, const UnitPlan &s, float *sc,
                                   SelScratch &x);

// Score and select unit u = (b, h) of the batch: writes its row of
// p.selected (ascending ids, -1 padded) and, if requested, its scores.  sc
// holds max_pages floats of shared memory (scores, then keys in place).
// Every thread of the group must call it with the same u.
template <typename T, int D, bool MMA, int GMAX, class Grp>
__device__ void select_unit(const Grp &grp, const SelectParams &p, int u, float *sc, SelScratch &x,
                            const BoxStage *stage = nullptr, uint32_t *phase_bits = nullptr,
                            unsigned long long *trace_scored = nullptr) {
    const UnitPlan s = plan_unit(p, u, grp.tid == 0);
    if (s.need_scores) {
        if constexpr (MMA && !is_fp8<T>::value) {
            if (stage) score_pages_mma_staged<T, D>(grp, p, s.b, s.h, s.N, sc, *stage, *phase_bits);
            else score_window<T, D, MMA, GMAX>(grp, p, s, sc, 0, (s.N + 15) >> 4);
        } else {
            score_window<T, D, MMA, GMAX>(grp, p, s, sc, 0, (s.N + 15) >> 4);
        }
        grp.sync();
    }
    if (grp.tid == 0) trace_stamp(trace_scored);
    select_from_scores(grp, p, u, s, sc, x);
}

// The unit's selection once sc[0, N) holds its scores (when s.need_scores).
//
// tau, the key of the (k-2)-th best candidate, is narrowed down digit by
// digit over the bits where the candidate keys differ: a 1024-bin shared
// histogram of the next 10 bits of the keys sharing the prefix found so far
// gives the digit that holds the wanted rank (one warp scans the bins).  Once
// no more keys share the prefix than the group has threads, they are
// gathered, one per thread, and the key of the wanted rank is read off by
// comparing every pair.  One scan over contiguous index segments of the
// candidates above tau and equal to tau then gives every thread its output
// position: kept are the candidates above tau, the lowest-index ones equal to
// it up to the quota, and the two forced pages, in ascending order.  The
// sequence of group barriers is the latency of the selection, so it is kept
// short (seven for one histogram pass).
template <class Grp>
__device__ void select_from_scores(const Grp &grp, const SelectParams &p, int u, const UnitPlan &s, float *sc,
                                   SelScratch &x) {
    uint32_t *keys = reinterpret_cast<uint32_t *>(sc);
    constexpr int NT = Grp::warps * 32;
    constexpr int BPL = kSelBins / 32;   // histogram bins per lane of the scanning warp
    const int tid = grp.tid, lane = grp.lane(), warp = grp.warp();
    const int N = s.N, k = s.k;
    int32_t *selrow = p.selected + (size_t)u * p.max_budget;

    if (N == 0) {
        for (int j = tid; j < p.max_budget; j += NT) selrow[j] = -1;
        return;
    }
    if (s.need_scores && p.scores_out) {
        for (int i = tid; i < N; i += NT) p.scores_out[(size_t)u * p.max_pages + i] = sc[i];
        grp.sync();   // the scores are read before the keys overwrite them in place
    }
    if (k >= N) {
        for (int j = tid; j < p.max_budget; j += NT) selrow[j] = j < N ? j : -1;
        return;
    }
    // here N >= 3: forced pages {0, N-1}; candidates 1..N-2; choose kc of them
    const int kc = k - 2;
    const int last = N - 1;
    if (kc == 0) {
        for (int j = tid; j < p.max_budget; j += NT) selrow[j] = j == 0 ? 0 : (j == 1 ? last : -1);
        return;
    }
    // contiguous index segment of this thread; candidates [c0, c1) in it
    const int E = (N + NT - 1) / NT;
    const int i0 = min(N, tid * E), i1 = min(N, i0 + E);
    const int c0 = max(i0, 1), c1 = min(i1, N - 1);
    for (int i = tid; i < kSelBins; i += NT) x.hist[i] = 0;
    if (tid == 0) x.gathered = 0;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = rank_key(sc[i]);
        keys[i] = key;
        if (i >= c0 && i < c1) { lo = min(lo, key); hi = max(hi, key); }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) { x.kmin[warp] = lo; x.kmax[warp] = hi; }
    grp.sync();
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int w = 0; w < Grp::warps; ++w) { kmin = min(kmin, x.kmin[w]); kmax = max(kmax, x.kmax[w]); }

    uint32_t tau = kmax;
    if (kmin != kmax) {
        const int hb = 31 - __clz(kmin ^ kmax);
        uint32_t pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);   // bits shared by every candidate
        uint32_t prefix = kmax & pmask;
        int need = kc;     // rank (1 = largest) of tau among the keys matching (prefix, pmask)
        int low = hb + 1;  // bits [low, 32) of tau are known
        int m = 0;         // keys matching the prefix
        for (int pass = 0;; ++pass) {
            const int shift = low > 10 ? low - 10 : 0;
            const uint32_t dmask = (1u << (low - shift)) - 1u;
            if (pass > 0) {
                for (int i = tid; i < kSelBins; i += NT) x.hist[i] = 0;
                grp.sync();
            }
            for (int i = c0; i < c1; ++i) {
                const uint32_t key = keys[i];
                if ((key & pmask) == prefix) atomicAdd(&x.hist[(key >> shift) & dmask], 1);
            }
            grp.sync();
            if (warp == 0) {
                // lane l holds the digits kSelBins-1-BPL*l down to kSelBins-BPL*(l+1)
                const int top = kSelBins - BPL * lane;
                int tot = 0;
#pragma unroll
                for (int j = 0; j < BPL; j += 4) {
                    const int4 v = *reinterpret_cast<const int4 *>(&x.hist[top - 4 - j]);
                    tot += v.x + v.y + v.z + v.w;
                }
                int incl = tot;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += t;
                }
                const int excl = incl - tot;
                if (excl < need && need <= incl) {
                    int run = excl;
                    for (int j = 1; j <= BPL; ++j) {
                        const int c = x.hist[top - j];
                        if (run + c >= need) {
                            x.digit = top - j;
                            x.above = run;
                            x.cnt = c;
                            break;
                        }
                        run += c;
                    }
                }
            }
            grp.sync();
            need -= x.above;
            m = x.cnt;
            prefix |= (uint32_t)x.digit << shift;
            pmask |= dmask << shift;
            low = shift;
            if (low == 0 || m <= NT) break;
            grp.sync();   // every thread has read the digit before the histogram is cleared
        }
        if (low == 0) {
            tau = prefix;
        } else {
            // gather the m <= NT keys sharing the prefix (any order) and read
            // off the key of rank `need` among them
            for (int i = c0; i < c1; ++i) {
                const uint32_t key = keys[i];
                if ((key & pmask) == prefix) x.list[atomicAdd(&x.gathered, 1)] = key;
            }
            grp.sync();
            if (tid < m) {
                const uint32_t v = x.list[tid];
                int gt = 0, eq = 0;
                for (int j = 0; j < m; ++j) {
                    const uint32_t w = x.list[j];
                    gt += w > v;
                    eq += w == v;
                }
                if (gt < need && need <= gt + eq) x.tau = v;   // every writer writes the same value
            }
            grp.sync();
            tau = x.tau;
        }
    }

    // candidates above tau are kept; of those equal to tau, the lowest indices
    // up to the quota need_eq = kc - (candidates above tau).  One scan of the
    // packed counts (above << 16 | equal) gives both prefixes and totals.
    int gt = 0, eq = 0;
    for (int i = c0; i < c1; ++i) {
        gt += (int)(keys[i] > tau);
        eq += (int)(keys[i] == tau);
    }
    int total;
    const int before = group_excl_scan_total(grp, (gt << 16) | eq, x.warp_tot, total);
    const int need_eq = kc - (total >> 16);
    int r = before & 0xffff;                            // candidates equal to tau before this segment
    int pos = (i0 > 0 ? 1 : 0) + (before >> 16) + min(r, need_eq);
    for (int i = i0; i < i1; ++i) {
        bool take;
        if (i == 0 || i == last) take = true;
        else {
            const uint32_t key = keys[i];
            take = key > tau || (key == tau && r < need_eq);
            if (key == tau) ++r;
        }
        if (take && pos < p.max_budget) selrow[pos++] = i;
    }
    for (int j = k + tid; j < p.max_budget; j += NT) selrow[j] = -1;
}

}  // namespace qasa
