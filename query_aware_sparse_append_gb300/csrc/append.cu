// append.cu -- kv append with page-box maintenance.
//
// TinyServe ("TinyServe: Query-Aware Cache Selection for Efficient LLM
// Serving", 方法详解 / 关键设计) attaches to every KV block a bounding box of
// what it holds.  This kernel keeps that box current while tokens are
// written: for each page touched by the call it stores the new K/V rows in
// their slots and folds the new keys into the page's per-channel min / max.
// A page whose slot 0 is written by the call starts a fresh box, so recycled
// pages never inherit a previous owner's box.
//
// Work unit: one warp per (sequence, touched page, KV head).  Grid:
// x = page index among the pages the call can touch, y = sequence; the warps of
// a CTA stride over KV heads.  Every row is moved with 16-byte vector accesses;
// the min / max fold runs in fp32 registers (exact for all three dtypes).
#include "qasa_device.cuh"
#include "qasa_launch.h"

namespace qasa {


template <typename T, int D>
__global__ void __launch_bounds__(128) append_kernel(AppendParams p) {
    constexpr int EPC = chunk16<T>::n;           // elements per 16-byte chunk
    constexpr int CPR = D / EPC;                 // chunks per row
    constexpr int LPR = CPR < 32 ? CPR : 32;     // lanes per row
    constexpr int CPL = CPR / LPR;               // chunks per lane
    constexpr int RPP = 32 / LPR;                // rows per warp pass

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int L0 = p.seq_lens[b];
    int n = p.append_lens ? p.append_lens[b] : p.T;
    if (n < 0 || n > p.T) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_APPEND);
        n = n < 0 ? 0 : p.T;
    }
    if (L0 < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_SEQ_LEN);
        return;
    }
    if (n == 0) return;
    const int P = p.P;
    const int pi = L0 / P + (int)blockIdx.x;                       // logical page
    const int t_lo = max(L0, pi * P), t_hi = min(L0 + n, (pi + 1) * P);
    if (t_lo >= t_hi) return;
    if (pi >= p.max_pages) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_SEQ_LEN);
        return;
    }
    const int phys = p.block_table[(size_t)b * p.max_pages + pi];
    if (phys < 0 || phys >= p.num_phys) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        return;
    }
    const bool fresh = (t_lo == pi * P);

    const int rsub = lane / LPR, csub = lane % LPR;
    for (int h = warp; h < p.Hkv; h += blockDim.x >> 5) {
        const size_t tile = ((size_t)phys * p.Hkv + h) * P;   // first row of this (page, head)
        float lo[CPL][EPC], hi[CPL][EPC];
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int e = 0; e < EPC; ++e) { lo[c][e] = INFINITY; hi[c][e] = -INFINITY; }

        for (int t = t_lo + rsub; t < t_hi; t += RPP) {
            const size_t src = (((size_t)b * p.T + (t - L0)) * p.Hkv + h) * D;
            const size_t dst = (tile + (t - pi * P)) * D;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int e0 = (csub + c * LPR) * EPC;
                uint4 kv = ld_global_nc_v4(static_cast<const T *>(p.k_new) + src + e0);
                uint4 vv = ld_global_nc_v4(static_cast<const T *>(p.v_new) + src + e0);
                *reinterpret_cast<uint4 *>(static_cast<T *>(p.k_pool) + dst + e0) = kv;
                *reinterpret_cast<uint4 *>(static_cast<T *>(p.v_pool) + dst + e0) = vv;
                float f[EPC];
                chunk16<T>::unpack(kv, f);
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    lo[c][e] = fminf(lo[c][e], f[e]);
                    hi[c][e] = fmaxf(hi[c][e], f[e]);
                }
            }
        }
        // fold the RPP row groups of the warp together
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int c = 0; c < CPL; ++c)
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    lo[c][e] = fminf(lo[c][e], __shfl_xor_sync(0xffffffffu, lo[c][e], off));
                    hi[c][e] = fmaxf(hi[c][e], __shfl_xor_sync(0xffffffffu, hi[c][e], off));
                }
        }
        if (rsub == 0) {
            T *bl = static_cast<T *>(p.bounds) + ((size_t)phys * p.Hkv + h) * 2 * D;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int e0 = (csub + c * LPR) * EPC;
                if (!fresh) {
                    float ol[EPC], oh[EPC];
                    chunk16<T>::unpack(*reinterpret_cast<const uint4 *>(bl + e0), ol);
                    chunk16<T>::unpack(*reinterpret_cast<const uint4 *>(bl + D + e0), oh);
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        lo[c][e] = fminf(lo[c][e], ol[e]);
                        hi[c][e] = fmaxf(hi[c][e], oh[e]);
                    }
                }
                *reinterpret_cast<uint4 *>(bl + e0) = chunk16<T>::pack(lo[c]);
                *reinterpret_cast<uint4 *>(bl + D + e0) = chunk16<T>::pack(hi[c]);
            }
        }
    }
}

// FP8 (E4M3) KV: the same work unit, plus the page's scales.  For K and for V:
// amax' = max(amax, max |new value|) (amax = 0 for a page whose slot 0 this
// call writes); if amax grew, the codes already in the page (and the K box)
// are re-quantized from scale amax/448 to amax'/448; the new values are
// quantized with amax'/448; the box folds the new K codes.  Re-quantization is
// monotone, so re-quantizing the old box equals the box of the re-quantized
// codes.  All steps are single fp32 operations rounded to nearest.
template <int D>
__global__ void __launch_bounds__(128) append_fp8_kernel(AppendParams p) {
    constexpr int EPC = 8;                       // f16 values per 16-byte input chunk
    constexpr int LPR = D / EPC;                 // lanes per row (8 or 16)
    constexpr int RPP = 32 / LPR;                // rows per warp pass

    const int b = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int L0 = p.seq_lens[b];
    int n = p.append_lens ? p.append_lens[b] : p.T;
    if (n < 0 || n > p.T) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_APPEND);
        n = n < 0 ? 0 : p.T;
    }
    if (L0 < 0) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_SEQ_LEN);
        return;
    }
    if (n == 0) return;
    const int P = p.P;
    const int pi = L0 / P + (int)blockIdx.x;
    const int t_lo = max(L0, pi * P), t_hi = min(L0 + n, (pi + 1) * P);
    if (t_lo >= t_hi) return;
    if (pi >= p.max_pages) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_SEQ_LEN);
        return;
    }
    const int phys = p.block_table[(size_t)b * p.max_pages + pi];
    if (phys < 0 || phys >= p.num_phys) {
        if (threadIdx.x == 0 && p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
        return;
    }
    const bool fresh = (t_lo == pi * P);
    const int rsub = lane / LPR, csub = lane % LPR;
    const int c0 = csub * EPC;                   // first channel of this lane's chunk

    for (int h = warp; h < p.Hkv; h += blockDim.x >> 5) {
        const size_t tile = ((size_t)phys * p.Hkv + h) * P;     // first row of this (page, head)
        float *sc = p.scales + ((size_t)phys * p.Hkv + h) * 4;
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {         // 0: K (with its box), 1: V
            const __half *src = static_cast<const __half *>(kv ? p.v_new : p.k_new);
            uint8_t *pool = static_cast<uint8_t *>(kv ? p.v_pool : p.k_pool);
            // amax of the new values
            float mx = 0.f;
            for (int t = t_lo + rsub; t < t_hi; t += RPP) {
                float f[EPC];
                chunk16<__half>::unpack(ld_global_nc_v4(src + (((size_t)b * p.T + (t - L0)) * p.Hkv + h) * D + c0), f);
#pragma unroll
                for (int e = 0; e < EPC; ++e) mx = fmaxf(mx, fabsf(f[e]));
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float old = fresh ? 0.f : sc[kv];
            const float amax = fmaxf(old, mx);
            const float s_old = fp8_scale(old), s_new = fp8_scale(amax);
            const bool requant = !fresh && amax > old;
            auto quant = [&](float x) -> uint32_t { return s_new == 0.f ? 0u : e4m3_from_f(__fdiv_rn(x, s_new)); };
            auto requant_code = [&](uint32_t c) -> uint32_t { return quant(__fmul_rn(e4m3_to_f(c), s_old)); };
            // re-scale the codes already in the page
            if (requant) {
                for (int t = pi * P + rsub; t < t_lo; t += RPP) {
                    uint2 *row = reinterpret_cast<uint2 *>(pool + (tile + (t - pi * P)) * D + c0);
                    const uint2 w = *row;
                    uint32_t o0 = 0, o1 = 0;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o0 |= requant_code((w.x >> (8 * e)) & 0xffu) << (8 * e);
                        o1 |= requant_code((w.y >> (8 * e)) & 0xffu) << (8 * e);
                    }
                    *row = make_uint2(o0, o1);
                }
            }
            // the new values; K also folds its codes into the box
            float lo[EPC], hi[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e) { lo[e] = INFINITY; hi[e] = -INFINITY; }
            for (int t = t_lo + rsub; t < t_hi; t += RPP) {
                float f[EPC];
                chunk16<__half>::unpack(ld_global_nc_v4(src + (((size_t)b * p.T + (t - L0)) * p.Hkv + h) * D + c0), f);
                uint32_t o0 = 0, o1 = 0;
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    const uint32_t c = quant(f[e]);
                    if (e < 4) o0 |= c << (8 * e); else o1 |= c << (8 * (e - 4));
                    const float v = e4m3_to_f(c);
                    lo[e] = fminf(lo[e], v);
                    hi[e] = fmaxf(hi[e], v);
                }
                *reinterpret_cast<uint2 *>(pool + (tile + (t - pi * P)) * D + c0) = make_uint2(o0, o1);
            }
            if (kv == 0) {
#pragma unroll
                for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        lo[e] = fminf(lo[e], __shfl_xor_sync(0xffffffffu, lo[e], off));
                        hi[e] = fmaxf(hi[e], __shfl_xor_sync(0xffffffffu, hi[e], off));
                    }
                if (rsub == 0) {
                    uint8_t *bl = static_cast<uint8_t *>(p.bounds) + ((size_t)phys * p.Hkv + h) * 2 * D + c0;
                    if (!fresh) {
                        const uint2 wl = *reinterpret_cast<const uint2 *>(bl);
                        const uint2 wh = *reinterpret_cast<const uint2 *>(bl + D);
#pragma unroll
                        for (int e = 0; e < EPC; ++e) {
                            uint32_t cl = ((e < 4 ? wl.x : wl.y) >> (8 * (e & 3))) & 0xffu;
                            uint32_t ch = ((e < 4 ? wh.x : wh.y) >> (8 * (e & 3))) & 0xffu;
                            if (requant) { cl = requant_code(cl); ch = requant_code(ch); }
                            lo[e] = fminf(lo[e], e4m3_to_f(cl));
                            hi[e] = fmaxf(hi[e], e4m3_to_f(ch));
                        }
                    }
                    uint32_t l0 = 0, l1 = 0, h0 = 0, h1 = 0;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        const uint32_t cl = e4m3_from_f(lo[e]), ch = e4m3_from_f(hi[e]);   // exact
                        if (e < 4) { l0 |= cl << (8 * e); h0 |= ch << (8 * e); }
                        else { l1 |= cl << (8 * (e - 4)); h1 |= ch << (8 * (e - 4)); }
                    }
                    *reinterpret_cast<uint2 *>(bl) = make_uint2(l0, l1);
                    *reinterpret_cast<uint2 *>(bl + D) = make_uint2(h0, h1);
                }
            }
            __syncwarp();
            if (lane == 0) sc[kv] = amax;
        }
    }
}

template <int D>
static cudaError_t launch_append_fp8_t(const AppendParams &p, int batch, cudaStream_t stream) {
    const int pages = (p.T + p.P - 1) / p.P + 1;
    dim3 grid(pages, batch);
    append_fp8_kernel<D><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_append_t(const AppendParams &p, int batch, cudaStream_t stream) {
    const int pages = (p.T + p.P - 1) / p.P + 1;   // a span of T tokens touches at most this many
    dim3 grid(pages, batch);
    append_kernel<T, D><<<grid, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append(qasa_dtype dt, int D, const AppendParams &p, int batch,
                          cudaStream_t stream) {
    switch (dt) {
    case QASA_DTYPE_E4M3:
        return D == 64 ? launch_append_fp8_t<64>(p, batch, stream) : launch_append_fp8_t<128>(p, batch, stream);
    case QASA_DTYPE_F32:
        return D == 64 ? launch_append_t<float, 64>(p, batch, stream)
                       : launch_append_t<float, 128>(p, batch, stream);
    case QASA_DTYPE_F16:
        return D == 64 ? launch_append_t<__half, 64>(p, batch, stream)
                       : launch_append_t<__half, 128>(p, batch, stream);
    default:
        return D == 64 ? launch_append_t<__nv_bfloat16, 64>(p, batch, stream)
                       : launch_append_t<__nv_bfloat16, 128>(p, batch, stream);
    }
}

}  // namespace qasa
