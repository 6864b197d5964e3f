// qasa_device.cuh -- device helpers shared by the qasa kernels (sm_103a).
//
// Inline PTX wrappers for the Blackwell data-movement and tensor paths used by
// the kernels: mbarrier transaction barriers, tiled TMA loads
// (cp.async.bulk.tensor) with 128-byte swizzle, ldmatrix / movmatrix, the
// m16n8k16 tensor-core MMA with fp32 accumulation, and programmatic dependent
// launch.  Also the element-type traits and the rules that every kernel must
// apply identically (valid length, kept-page count).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qasa.h"

namespace qasa {

// ---------------------------------------------------------------- dtypes

template <typename T> struct elem;
template <> struct elem<float> {
    static constexpr qasa_dtype id = QASA_DTYPE_F32;
    __device__ static float to_f(float x) { return x; }
    __device__ static float from_f(float x) { return x; }
};
template <> struct elem<__half> {
    static constexpr qasa_dtype id = QASA_DTYPE_F16;
    __device__ static float to_f(__half x) { return __half2float(x); }
    __device__ static __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct elem<__nv_bfloat16> {
    static constexpr qasa_dtype id = QASA_DTYPE_BF16;
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Unpack a 16-byte chunk into floats (8 halves / 8 bf16 / 4 floats).
template <typename T> struct chunk16;
template <> struct chunk16<float> {
    static constexpr int n = 4;
    __device__ static void unpack(const uint4 &v, float *f) {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float *f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};
template <> struct chunk16<__half> {
    static constexpr int n = 8;
    __device__ static void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    __device__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct chunk16<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void unpack(const uint4 &v, float *f) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float *f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ------------------------------------------------------------- FP8 codes

// Tag type of FP8 (E4M3) KV: the pools hold one-byte codes with a scale per
// (page, KV head); queries, outputs and appended values are __half.
struct fp8e4m3 {};
template <typename T> struct is_fp8 { static constexpr bool value = false; };
template <> struct is_fp8<fp8e4m3> { static constexpr bool value = true; };

// Value of one E4M3 code (exact in fp32).
__device__ __forceinline__ float e4m3_to_f(uint32_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
    return __half2float(__half(h));
}
// Nearest E4M3 code (ties to even, finite overflow saturates to +-448), with a
// zero result stored as +0 so that equal values always have equal codes.
__device__ __forceinline__ uint32_t e4m3_from_f(float x) {
    const uint32_t c = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
    return (c & 0x7Fu) ? c : 0u;
}
// Two codes (low byte first) to a half2 word, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two & 0xffffu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}
// 16 codes (one 16-byte chunk) to 16 halves: channels 0..7 in lo, 8..15 in hi.
__device__ __forceinline__ void e4m3x16_to_h(const uint4 &c, uint4 &lo, uint4 &hi) {
    lo = make_uint4(e4m3x2_to_h2(c.x), e4m3x2_to_h2(c.x >> 16), e4m3x2_to_h2(c.y), e4m3x2_to_h2(c.y >> 16));
    hi = make_uint4(e4m3x2_to_h2(c.z), e4m3x2_to_h2(c.z >> 16), e4m3x2_to_h2(c.w), e4m3x2_to_h2(c.w >> 16));
}
// Scale of a page from its amax (the fp32 division of the format).
__device__ __forceinline__ float fp8_scale(float amax) { return __fdiv_rn(amax, 448.0f); }

// ------------------------------------------------------------ shared rules

// Sequence length after validation against the block table width.
__device__ __forceinline__ int valid_len(int L, int max_pages, int P, int32_t *status) {
    if (L < 0 || (long long)L > (long long)max_pages * P) {
        if (status) atomicOr(status, QASA_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : max_pages * P;
    }
    return L;
}

// Pages kept for one (sequence, KV head): every page when the budget reaches
// the page count, otherwise max(budget, forced pages), capped by max_budget.
__device__ __forceinline__ int kept_pages(int N, int budget, int max_budget, int32_t *status,
                                          bool report) {
    if (N <= 0) return 0;
    int forced = N >= 2 ? 2 : 1;
    int k = budget >= N ? N : (budget > forced ? budget : forced);
    if (k > max_budget) {
        if (report && status) atomicOr(status, QASA_DEVERR_BUDGET);
        k = max_budget;
    }
    return k;
}

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Diagnostics: record the current time in trace slot `t` (no-op when NULL),
// or raise it to the current time (several writers, the latest one wins).
__device__ __forceinline__ void trace_stamp(unsigned long long *t) {
    if (t) *t = global_timer_ns();
}
__device__ __forceinline__ void trace_latest(unsigned long long *t) {
    if (t) atomicMax(t, (unsigned long long)global_timer_ns());
}
__device__ __forceinline__ void trace_smid(unsigned long long *t) {
    if (t) {
        uint32_t id;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
        *t = id;
    }
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (for lane-parallel polling of many barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the given parity to complete, giving up after
// `limit_ns` nanoseconds.  Returns false on time-out (the caller records it).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Plain (untiled) bulk copy of `bytes` contiguous bytes from global to shared
// memory, completing on `bar`; both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bulk prefetch of `bytes` contiguous bytes (16-byte aligned, a multiple of
// 16) into L2: no register, shared memory or barrier is involved.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

// Tiled 2-D TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// Tiled 3-D TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Tiled 4-D TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t c0, int32_t c1, int32_t c2, int32_t c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                            uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                  uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// D += A(16x16, row) * B(16x8, col), fp32 accumulators.
template <typename T> struct mma16816;
template <> struct mma16816<__half> {
    __device__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};
template <> struct mma16816<__nv_bfloat16> {
    __device__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
            "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    __device__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
};

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Device-scope atomic add with acquire-release semantics (one instruction in
// place of fence + atomic + fence).
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// Device-scope acquire load / release store of a flag published by another CTA.
__device__ __forceinline__ int ld_acquire_gpu(const int *addr) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int *addr, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Offset of 16-byte chunk `chunk` of row `row` inside a tile staged by a TMA
// box with 128-byte swizzle: the tile is split in sub-tiles of 128-byte rows
// (one per 128 bytes of the head dimension); within each 1024-byte group of
// 8 rows the chunk index is XORed with the row index modulo 8.
template <int ROWS>
__device__ __forceinline__ uint32_t swz128_offset(int row, int chunk) {
    return (uint32_t)((chunk >> 3) * (ROWS * 128) + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

}  // namespace qasa
