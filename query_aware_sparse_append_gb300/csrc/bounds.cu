// bounds.cu -- rebuild the page boxes of whole sequences from the keys already
// in the pool.
//
// The box of a KV block ("TinyServe: Query-Aware Cache Selection for Efficient
// LLM Serving", 方法详解 / 关键设计) is normally kept current by the append
// kernel as tokens arrive.  A cache whose keys were written some other way (a
// prefill kernel that stores K/V directly, a pool restored or migrated from
// elsewhere) needs its boxes built in bulk: for every logical page p < N_b of
// every sequence b, lo / hi = per-channel min / max of the keys in the page's
// valid slots (slot < seq_len - p * P).  The result is bit-identical to the
// boxes the append path maintains for the same keys (min / max are exact).
//
// Work unit: one warp per (sequence, logical page, KV head); grid x = logical
// page, y = sequence, the 4 warps of a CTA stride over the KV heads.  A group
// of lanes holds one key row at 16 bytes per lane; every lane issues the loads
// of up to 8 rows before folding them, then the row groups are folded by
// shuffles and one lane per chunk writes the lo and hi rows.  HBM-bound: the
// valid keys are read once, the boxes written once.
#include "qasa_device.cuh"
#include "qasa_launch.h"

namespace qasa {

namespace {

constexpr int kRebuildBatch = 8;

template <typename T, int D>
__global__ void __launch_bounds__(128) rebuild_bounds_kernel(RebuildParams p) {
    constexpr int EPC = chunk16<T>::n;           // elements per 16-byte chunk
    constexpr int CPR = D / EPC;                 // chunks per row
    static_assert(CPR <= 32, "a key row must fit one warp at 16 bytes per lane");
    constexpr int LPR = CPR;                     // lanes per row
    constexpr int RPP = 32 / LPR;                // rows per warp pass

    const int b = blockIdx.y, pg = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = p.P;
    const int L = valid_len(p.seq_lens[b], p.max_pages, P,
                            (threadIdx.x == 0 && pg == 0) ? p.status : nullptr);
    const int rows = min(P, L - pg * P);
    if (rows <= 0) return;
    const int phys = p.block_table[(size_t)b * p.max_pages + pg];
    if (phys < 0 || phys >= p.num_phys) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        return;
    }
    const int rsub = lane / LPR, csub = lane % LPR;
    for (int h = warp; h < p.Hkv; h += blockDim.x >> 5) {
        const T *kp = static_cast<const T *>(p.k_pool) + ((size_t)phys * p.Hkv + h) * P * D + csub * EPC;
        float lo[EPC], hi[EPC];
#pragma unroll
        for (int e = 0; e < EPC; ++e) { lo[e] = INFINITY; hi[e] = -INFINITY; }
        for (int r0 = rsub; r0 < rows; r0 += kRebuildBatch * RPP) {
            uint4 kv[kRebuildBatch];
#pragma unroll
            for (int j = 0; j < kRebuildBatch; ++j) {
                const int r = r0 + j * RPP;
                kv[j] = r < rows ? ld_global_nc_v4(kp + (size_t)r * D) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < kRebuildBatch; ++j) {
                if (r0 + j * RPP < rows) {
                    float f[EPC];
                    chunk16<T>::unpack(kv[j], f);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        lo[e] = fminf(lo[e], f[e]);
                        hi[e] = fmaxf(hi[e], f[e]);
                    }
                }
            }
        }
        // fold the row groups of the warp (a group with no row holds +-inf)
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                lo[e] = fminf(lo[e], __shfl_xor_sync(0xffffffffu, lo[e], off));
                hi[e] = fmaxf(hi[e], __shfl_xor_sync(0xffffffffu, hi[e], off));
            }
        }
        if (rsub == 0) {
            T *bl = static_cast<T *>(p.bounds) + ((size_t)phys * p.Hkv + h) * 2 * D + csub * EPC;
            *reinterpret_cast<uint4 *>(bl) = chunk16<T>::pack(lo);
            *reinterpret_cast<uint4 *>(bl + D) = chunk16<T>::pack(hi);
        }
    }
}

// FP8 (E4M3) codes: the box is the per-channel minimum and maximum code by
// value (the page's keys share one scale, so these bound the dequantized keys
// exactly); 16 codes per lane.
template <int D>
__global__ void __launch_bounds__(128) rebuild_bounds_fp8_kernel(RebuildParams p) {
    constexpr int LPR = D / 16;                  // lanes per row
    constexpr int RPP = 32 / LPR;                // rows per warp pass
    const int b = blockIdx.y, pg = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int P = p.P;
    const int L = valid_len(p.seq_lens[b], p.max_pages, P,
                            (threadIdx.x == 0 && pg == 0) ? p.status : nullptr);
    const int rows = min(P, L - pg * P);
    if (rows <= 0) return;
    const int phys = p.block_table[(size_t)b * p.max_pages + pg];
    if (phys < 0 || phys >= p.num_phys) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        return;
    }
    const int rsub = lane / LPR, csub = lane % LPR;
    for (int h = warp; h < p.Hkv; h += blockDim.x >> 5) {
        const uint8_t *kp = static_cast<const uint8_t *>(p.k_pool) + ((size_t)phys * p.Hkv + h) * P * D + csub * 16;
        float lo[16], hi[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) { lo[e] = INFINITY; hi[e] = -INFINITY; }
        for (int r = rsub; r < rows; r += RPP) {
            const uint4 c = ld_global_nc_v4(kp + (size_t)r * D);
            const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float v = e4m3_to_f((w[e >> 2] >> (8 * (e & 3))) & 0xffu);
                lo[e] = fminf(lo[e], v);
                hi[e] = fmaxf(hi[e], v);
            }
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                lo[e] = fminf(lo[e], __shfl_xor_sync(0xffffffffu, lo[e], off));
                hi[e] = fmaxf(hi[e], __shfl_xor_sync(0xffffffffu, hi[e], off));
            }
        if (rsub == 0) {
            uint32_t wl[4] = {0, 0, 0, 0}, wh[4] = {0, 0, 0, 0};
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                wl[e >> 2] |= e4m3_from_f(lo[e]) << (8 * (e & 3));    // exact: lo, hi are code values
                wh[e >> 2] |= e4m3_from_f(hi[e]) << (8 * (e & 3));
            }
            uint8_t *bl = static_cast<uint8_t *>(p.bounds) + ((size_t)phys * p.Hkv + h) * 2 * D + csub * 16;
            *reinterpret_cast<uint4 *>(bl) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            *reinterpret_cast<uint4 *>(bl + D) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        }
    }
}

template <int D>
cudaError_t launch_rebuild_fp8_t(const RebuildParams &p, int batch, cudaStream_t stream) {
    dim3 grid(p.max_pages, batch);
    rebuild_bounds_fp8_kernel<D><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_rebuild_t(const RebuildParams &p, int batch, cudaStream_t stream) {
    dim3 grid(p.max_pages, batch);
    rebuild_bounds_kernel<T, D><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rebuild_bounds(qasa_dtype dt, int D, const RebuildParams &p, int batch,
                                  cudaStream_t stream) {
    if (batch == 0) return cudaSuccess;
    switch (dt) {
    case QASA_DTYPE_E4M3:
        return D == 64 ? launch_rebuild_fp8_t<64>(p, batch, stream) : launch_rebuild_fp8_t<128>(p, batch, stream);
    case QASA_DTYPE_F32:
        return D == 64 ? launch_rebuild_t<float, 64>(p, batch, stream)
                       : launch_rebuild_t<float, 128>(p, batch, stream);
    case QASA_DTYPE_F16:
        return D == 64 ? launch_rebuild_t<__half, 64>(p, batch, stream)
                       : launch_rebuild_t<__half, 128>(p, batch, stream);
    default:
        return D == 64 ? launch_rebuild_t<__nv_bfloat16, 64>(p, batch, stream)
                       : launch_rebuild_t<__nv_bfloat16, 128>(p, batch, stream);
    }
}

}  // namespace qasa
