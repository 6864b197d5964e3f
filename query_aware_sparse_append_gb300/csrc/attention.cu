// attention.cu -- masked paged decode attention over the selected pages.
//
// The sparse-attention half of TinyServe's decode step ("TinyServe:
// Query-Aware Cache Selection for Efficient LLM Serving", abstract: sparse
// memory access and masked attention; edgentiq post, "How TinyServe Works":
// the sparse attention executor computes attention over the selected KV pages
// only).  For every (sequence b, KV head h) and each of its G query heads:
//
//     out = sum_t softmax_t(scale * q.k_t) v_t   over the tokens t of the kept
//                                               pages whose position < seq_len
//
// Work split (persistent, balanced).  All kept (unit, page) pairs of the batch
// are laid out in one flattened order (unit-major, pages ascending); CTA c of C
// takes the contiguous range [c*T/C, (c+1)*T/C).  A range covers whole units
// (written straight to `out`) and at most two partial units at its ends,
// whose partial (m, l, o) go to workspace slot (unit + c); the CTA that
// finishes a unit last (acquire-release ticket counting the unit's pages, no
// waiting) merges its partials.  Each CTA walks its range rotated (the part of
// its last unit first), so both of its partial units finish early.
//
// Inside a CTA: warp 0 is the producer.  Its lanes turn up to 32 kept page ids
// into physical tiles through the block table at once and each lane issues its
// page's K and V copies: one 3-D tiled TMA box per tile (cp.async.bulk.tensor,
// 128-byte swizzle; a 2-D box per 128 bytes of head dimension where the 3-D
// map is refused) into a ring of shared-memory stages guarded by mbarriers.
// NWK working warps consume the pages (page i of the range goes to warp
// i % NWK and stage i % S, S a multiple of NWK, so a stage is only ever used by
// one warp); the remaining warps merge the working warps' softmax states at
// every unit boundary (a few heads each) and write the output or the partial,
// while the working warps go on.  Nothing follows the range's last segment, so
// when it is a whole unit the working warps merge it themselves.  For 16-bit and FP8 KV
// (any group size) a consumer computes S^T = K q^T and O^T += V^T P^T as m16n8k16
// tensor-core MMAs (16 tokens x 8
// query heads per MMA; ldmatrix reads the swizzled tiles conflict-free;
// movmatrix turns the S accumulators into the P operand) with an online
// softmax in fp32.  fp32 KV uses FFMA and warp shuffles.
//
// Every wait is bounded: a wait that gives up sets QASA_DEVERR_TIMEOUT, the CTA
// stops issuing, drains the copies it issued (again bounded) and returns.
// Waits on other warps, other CTAs or flags use p.wait_limit_ns; waits for the
// CTA's own copies in flight use p.drain_limit_ns, so that no CTA exits while
// a copy into its shared memory can still land.
#include <cstdlib>
#include <type_traits>

#include "select_device.cuh"

namespace qasa {


struct StageInfo {
    int page;    // logical page id
    int nvalid;  // valid tokens in the page (0: nothing to attend)
};

constexpr int kSelThreads = 128;   // selector warps of the single-launch kernel
constexpr int kSelBarrier = 1;     // their named barrier
constexpr int kSelSlotsPerWarp = 2;                    // box tiles in flight per selector warp
constexpr int kSelStageSlots = 4 * kSelSlotsPerWarp;

// Host-side size of the dynamic shared memory (mirrors the device carve-up).
size_t attn_smem_bytes(int stages, int stage_bytes, int nw, int gmax, int D, int P, bool mma, int B, int grid,
                       bool fused, int max_pages, bool fp8 = false, bool fp8_scratch = false) {
    size_t s = 1024;                                   // alignment slack for the ring
    s += (size_t)stages * stage_bytes;
    s += (size_t)stages * 2 * sizeof(uint64_t);        // full / empty barriers
    s += (size_t)stages * (sizeof(StageInfo) + sizeof(int));
    if (fp8) s += 16 + (size_t)stages * 16;            // per-stage page scales
    if (fp8_scratch) s += 1024 + (size_t)nw * 2 * P * D * 2;   // per-warp half copies of the K and V tiles
    s += (size_t)nw * gmax * (D + 2) * sizeof(float);  // combine scratch
    if (!mma) s += (size_t)nw * gmax * (D + P) * sizeof(float);
    s += (size_t)(2 * B + 2) * sizeof(int);            // prefix, lengths
    s += 8 + (size_t)(grid + 1) * sizeof(long long);   // every CTA's first page
    if (fused) {
        // selector scratch: scores, block-table row, box staging slots + barriers
        s += 16 + (size_t)max_pages * sizeof(float) + 16 + sizeof(SelScratch);
        s += 16 + (size_t)max_pages * sizeof(int32_t);
        if (mma) s += 16 + (size_t)kSelStageSlots * (16 * (2 * D * 2 + 64) + sizeof(uint64_t));
    }
    s += 64;
    return s;
}

// CTA ranges are balanced on weighted work: the flattened page g of unit u
// (unit-major order) sits at v(g) = g + W0 * (u + 1), so that every unit adds
// W0 page-equivalents (its query, its state hand-over and merge) before its
// pages; CTA c of C takes the pages with v in [c*V/C, (c+1)*V/C), V = T + W0*U.
// CTA whose range holds the page at weighted position v (0 <= v < V).
__device__ __forceinline__ int cta_of_v(long long v, int C, long long V) {
    return (int)(((v + 1) * C - 1) / V);
}

// Online merge of one softmax state (m, l, o[]) into a running one (log2 domain).
template <int J>
__device__ __forceinline__ void merge_state(float &M, float &L, float *o, float m, float l, const float *ox) {
    if (m == -INFINITY) return;
    const float nm = fmaxf(M, m);
    const float a = exp2f(M - nm), b = exp2f(m - nm);   // a = 0 while the running state is empty
    L = L * a + l * b;
#pragma unroll
    for (int j = 0; j < J; ++j) o[j] = o[j] * a + ox[j] * b;
    M = nm;
}

template <typename T, int D, int P, bool MMA, int GMAX, int NW, bool FUSED>
__global__ void __launch_bounds__(32 * (NW + 1) + (FUSED ? kSelThreads : 0), 1)
attn_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
            AttnParams p) {
    constexpr bool F8 = is_fp8<T>::value;
    using MT = typename std::conditional<F8, __half, T>::type;   // q, out and MMA operand type
    constexpr int ES = F8 ? 1 : (int)sizeof(T);  // bytes per stored KV element
    constexpr int MES = (int)sizeof(MT);         // bytes per element of the tiles the consumers read
    // FP8, d = 128: the 16-bit tensor-core path on K and V fragments
    // converted from the (128-byte swizzled) code tiles in registers;
    // otherwise FP8 tiles are converted to half copies in shared memory
    constexpr bool F8MMA = F8 && MMA && D == 128;
    constexpr bool F8CONV = F8 && !F8MMA;
    constexpr int TILE = P * D * ES;            // one (page, head) tile of K or V
    constexpr int STAGE = 2 * TILE;
    constexpr int NSUB = F8 ? 1 : D * ES / 128; // 128-byte column boxes per tile
    constexpr int BOXW = 128 / ES;              // elements per box row
    static_assert(TILE % 1024 == 0, "tile must keep 1024-byte swizzle alignment");

    extern __shared__ unsigned char smem_raw[];
    const int S = p.stages;
    const int NWK = p.consumers;   // working consumer warps (<= NW, divides S)
    unsigned char *ring = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(ring + (size_t)S * STAGE);
    uint64_t *empty_bar = full_bar + S;
    StageInfo *info = reinterpret_cast<StageInfo *>(empty_bar + S);
    int *last_ph = reinterpret_cast<int *>(info + S);             // [S] phase of the last copy
    float4 *st_scale = reinterpret_cast<float4 *>(                 // FP8: [S] the page's amax (K, V, -, -)
        (reinterpret_cast<uintptr_t>(last_ph + S) + 15) & ~uintptr_t(15));
    float *scr_o = reinterpret_cast<float *>(st_scale + (F8 ? S : 0));   // [NWK][GMAX][D]
    float *scr_m = scr_o + NWK * GMAX * D;                         // [NWK][GMAX]
    float *scr_l = scr_m + NWK * GMAX;                             // [NWK][GMAX]
    float *ff_q = scr_l + NWK * GMAX;                              // FFMA only: [NWK][GMAX][D]
    float *ff_p = ff_q + (MMA ? 0 : NWK * GMAX * D);               // FFMA only: [NWK][GMAX][P]
    int *prefix = reinterpret_cast<int *>(ff_p + (MMA ? 0 : NWK * GMAX * P));  // [B + 1]
    int *lens = prefix + (p.B + 1);                                // [B]
    long long *rstart = reinterpret_cast<long long *>(                 // [C + 1] every CTA's first page
        (reinterpret_cast<uintptr_t>(lens + p.B) + 7) & ~uintptr_t(7));
    // single launch: the selector warps' scores [max_pages], scratch, the
    // unit's block-table row [max_pages] and (tensor-core scoring) the box
    // staging slots with their barriers
    float *sel_sc = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(rstart + gridDim.x + 1) + 15) & ~uintptr_t(15));
    SelScratch *sel_x = reinterpret_cast<SelScratch *>(
        (reinterpret_cast<uintptr_t>(sel_sc + (FUSED ? p.max_pages : 0)) + 15) & ~uintptr_t(15));
    int32_t *sel_phys = reinterpret_cast<int32_t *>(
        (reinterpret_cast<uintptr_t>(sel_x + (FUSED ? 1 : 0)) + 15) & ~uintptr_t(15));
    unsigned char *sel_buf = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(sel_phys + (FUSED ? p.max_pages : 0)) + 15) & ~uintptr_t(15));
    constexpr int kSelTileB = 16 * (2 * D * ES + 64);
    uint64_t *sel_bar = reinterpret_cast<uint64_t *>(sel_buf + (FUSED && MMA ? kSelStageSlots * kSelTileB : 0));
    // FP8: per working warp, half-precision copies of its current K and V tiles
    // (laid out like a 128-byte-swizzled 16-bit tile, so the MMA path reads them
    // with the same ldmatrix addressing)
    unsigned char *f8_scr = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(sel_bar + (FUSED && MMA ? kSelStageSlots : 0)) + 1023) & ~uintptr_t(1023));
    __shared__ int s_abort;      // a bounded wait gave up
    // segment hand-off: [0] completes when the NWK working warps have written
    // their states for a segment; [1] completes when the combiners have read them;
    // [2] completes when they have written their states for the range's last
    // segment, if that is a whole unit (merged by the working warps themselves)
    __shared__ __align__(8) uint64_t seg_bar[3];
    volatile int *abort_flag = &s_abort;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = gridDim.x, c = blockIdx.x;
    const int Hkv = p.Hkv, G = p.G;
    unsigned long long *const tr =
        p.trace && c < QASA_TRACE_MAX_CTAS ? p.trace + (size_t)c * QASA_TRACE_ATTN_EVENTS : nullptr;
    if (tid == 0) {
        trace_stamp(tr);
        trace_smid(tr ? tr + 8 : nullptr);
    }

    // warp 0 sets up the stage barriers while the other warps start the scan
    if (warp == 0) {
        for (int s = lane; s < S; s += 32) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
            last_ph[s] = -1;
        }
        if (lane == 0) {
            s_abort = 0;
            mbar_init(&seg_bar[0], (uint32_t)NWK);
            mbar_init(&seg_bar[1], (uint32_t)(NW - NWK));
            mbar_init(&seg_bar[2], (uint32_t)NWK);
        }
        if constexpr (FUSED && MMA)
            for (int i = lane; i < kSelStageSlots; i += 32) mbar_init(&sel_bar[i], 1);
        fence_barrier_init();
        if (lane == 0) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
    }
    // per-sequence kept counts (the selection kernel's rule) and their prefix
    int any_empty = 0;
    {
        __shared__ int s_wsum[32];
        int carry = 0;
        for (int base = 0; base < p.B; base += blockDim.x) {
            const int b = base + tid;
            int cnt = 0;
            if (b < p.B) {
                const int L = valid_len(p.seq_lens[b], p.max_pages, P, c == 0 ? p.status : nullptr);
                const int N = (L + P - 1) / P;
                cnt = p.dense ? N : kept_pages(N, p.budget[b], p.max_budget, nullptr, false);
                lens[b] = L;
                any_empty |= (cnt == 0);
            }
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                int t = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += t;
            }
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            int wbase = 0, total = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
                const int v = s_wsum[w];
                wbase += w < warp ? v : 0;
                total += v;
            }
            if (b < p.B) prefix[b] = carry + wbase + incl - cnt;
            carry += total;
            __syncthreads();
        }
        if (tid == 0) prefix[p.B] = carry;
        any_empty = __syncthreads_or(any_empty);
    }
    const long long Ttot = (long long)Hkv * prefix[p.B];
    // (the weight and the weighted total are recomputed from the parameters
    // where they are used rather than held in registers across the kernel)
    auto unit_w = [&]() -> long long { return p.dense ? 0 : p.unit_weight; };
    auto weighted_total = [&]() -> long long { return (long long)Hkv * prefix[p.B] + unit_w() * (p.B * Hkv); };
    // first page of CTA cc's range: the first page whose weighted position
    // reaches V = cc*Vtot/C.  Sequence b's units end at weighted positions
    // base_b + (h+1)*step_b with base_b = Hkv*(prefix[b] + W0*b) and
    // step_b = cnt_b + W0, so: the first sequence whose last unit ends past V
    // (a search over the sequences), then the unit in it, then the page.
    auto range_start = [&](int cc) -> long long {
        const long long W0 = unit_w();
        if (cc >= C) return (long long)Hkv * prefix[p.B];
        const long long V = (long long)cc * weighted_total() / C;
        int lo = 0, hi = p.B;
        while (lo < hi) {   // first b with base_{b+1} > V
            const int mid = (lo + hi) >> 1;
            if ((long long)Hkv * (prefix[mid + 1] + W0 * (mid + 1)) > V) hi = mid; else lo = mid + 1;
        }
        if (lo >= p.B) return (long long)Hkv * prefix[p.B];
        const int cn = prefix[lo + 1] - prefix[lo];
        const long long base = (long long)Hkv * (prefix[lo] + W0 * lo), step = cn + W0;   // step > 0 here
        long long hh = (V - base) / step;   // units of b that end at or before V
        if (hh < 0) hh = 0;
        if (hh > Hkv - 1) hh = Hkv - 1;
        const long long us = (long long)Hkv * prefix[lo] + hh * cn;
        const long long g = V - W0 * ((long long)lo * Hkv + hh + 1);
        return g > us ? g : us;
    };
    for (int x = tid; x <= C; x += blockDim.x) rstart[x] = range_start(x);
    __syncthreads();
    const long long g0 = rstart[c], g1 = rstart[c + 1];

    // sequences with no pages: zero their outputs (unit u handled by CTA u % C)
    if (any_empty) {
        for (int b = 0; b < p.B; ++b) {
            if (prefix[b + 1] != prefix[b]) continue;
            for (int h = 0; h < Hkv; ++h) {
                if ((b * Hkv + h) % C != c) continue;
                MT *o = static_cast<MT *>(p.out) + ((size_t)b * p.Hq + (size_t)h * G) * D;
                for (int i = tid; i < G * D; i += blockDim.x) o[i] = elem<MT>::from_f(0.f);
                if constexpr (FUSED) {   // and no kept ids
                    int32_t *row = p.selected + ((size_t)b * Hkv + h) * p.max_budget;
                    for (int i = tid; i < p.max_budget; i += blockDim.x) row[i] = -1;
                }
            }
        }
    }

    // locate flattened index g: sequence b, KV head h, position j in the unit
    auto locate = [&](long long g, int &b, int &h, int &j, long long &ustart, int &cnt) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {   // largest b with Hkv * prefix[b] <= g
            const int mid = (lo + hi + 1) >> 1;
            if ((long long)Hkv * prefix[mid] <= g) lo = mid; else hi = mid - 1;
        }
        b = lo;
        cnt = prefix[b + 1] - prefix[b];
        const long long off = g - (long long)Hkv * prefix[b];
        h = (int)(off / cnt);
        j = (int)(off - (long long)h * cnt);
        ustart = (long long)Hkv * prefix[b] + (long long)h * cnt;
    };

    // The range is processed rotated: first [gL, g1), the part of the range's
    // last unit that lies in it, then [g0, gL).  Both partial units of a range
    // (its first and its last) are therefore done early, so every split unit's
    // ticket completes mid-kernel and the range ends on whole units.
    const long long n_loc = g1 - g0;
    long long gL = g0;
    if (n_loc > 0) {
        int b, h, j, cnt;
        long long us;
        locate(g1 - 1, b, h, j, us, cnt);
        if (us > g0) gL = us;
    }
    const long long nL = g1 - gL;
    auto rot = [&](long long pos) -> long long { return pos < nL ? gL + pos : g0 + (pos - nL); };
    auto run_end = [&](long long pos) -> long long { return pos < nL ? g1 : gL; };

    // Producer lookups (see the producer below).  Where the pages of its first
    // two batches sit in the flattened order depends only on this kernel's
    // inputs, so the producer works it out before waiting for the selection.
    struct Look { int page, phys, b, h, j, stage; bool active, ok; };
    const int WB = S < 32 ? S : 32;
    auto look_loc = [&](long long bb, Look &lk) {   // locate; the kept id is not read yet
        const long long pos = bb + lane;
        lk.active = lane < WB && pos < n_loc;
        lk.ok = false;
        lk.page = -1; lk.phys = -1; lk.b = 0; lk.h = 0; lk.j = 0;
        lk.stage = 2;
        if (lk.active) {
            int cnt;
            long long us;
            locate(rot(pos), lk.b, lk.h, lk.j, us, cnt);
            lk.stage = 0;
        }
    };
    Look la, lb, lc;
    if (warp == 0) {
        look_loc(0, la);
        look_loc(WB, lb);
    }

    if (tid == 0) trace_stamp(tr ? tr + 1 : nullptr);
    pdl_wait();   // selected ids and counters come from the preceding kernel
    if (tid == 0) trace_stamp(tr ? tr + 2 : nullptr);


    if constexpr (FUSED) {
        // -------------------------------------------------------- selectors
        // The selector warps score and select the units whose first kept page
        // lies in this CTA's range ("owned" units), in the order the range is
        // consumed: the range's last unit first (the rotation starts there; a
        // neighbour's range may start with it too), then the others ascending.
        // Each unit's kept ids are published with a device-scope release of
        // its ready flag, which the producers (here and in the neighbouring
        // CTA) acquire before reading them.
        if (warp > NW) {
            const SelGroup<kSelThreads, kSelBarrier> grp{tid - 32 * (NW + 1)};
            SelectParams sp;
            sp.bounds = p.bounds;
            sp.block_table = p.block_table;
            sp.seq_lens = p.seq_lens;
            sp.budget = p.budget;
            sp.q = p.q;
            sp.selected = p.selected;
            sp.scores_out = p.scores_out;
            sp.counters = p.counters;
            sp.B = p.B;
            sp.status = p.status;
            sp.num_phys = p.num_phys;
            sp.Hkv = Hkv;
            sp.P = P;
            sp.G = G;
            sp.Hq = p.Hq;
            sp.max_pages = p.max_pages;
            sp.max_budget = p.max_budget;
            sp.scales = p.scales;
            sp.trace = nullptr;
            BoxStage stage;
            stage.buf = sel_buf;
            stage.bar = sel_bar;
            stage.phys = sel_phys;
            stage.slots_per_warp = kSelSlotsPerWarp;
            stage.wait_limit_ns = p.drain_limit_ns;   // bulk copies of this CTA: drained, never abandoned
            uint32_t phase_bits = 0;    // parity of this warp's staging slots
            auto run_unit = [&](int u) {
                select_unit<T, D, MMA, GMAX>(grp, sp, u, sel_sc, *sel_x, MMA ? &stage : nullptr, &phase_bits);
                __threadfence();
                grp.sync();                      // every id of the row is stored
                if (grp.tid == 0) st_release_gpu(&p.ready[u], 1);
            };
            if (n_loc > 0) {
                int b, h, j, cnt;
                long long us;
                locate(g1 - 1, b, h, j, us, cnt);
                const int u_last = b * Hkv + h;
                if (us >= g0) run_unit(u_last);
                locate(g0, b, h, j, us, cnt);
                int u = b * Hkv + h + (us < g0 ? 1 : 0);   // skip a unit begun in an earlier range
                for (; u < u_last; ++u) {        // units strictly inside the range
                    const int ub = u / Hkv;
                    if (prefix[ub + 1] == prefix[ub]) continue;   // no pages: handled above
                    run_unit(u);
                }
            }
            return;
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Pages are handled in batches of WB <= min(32, S): the lanes resolve one
        // page each (kept id -> block table -> tile row), then every lane issues
        // its own page's two TMA boxes as soon as its stage is free, so up to 32
        // copies leave per warp instruction instead of one.
        uint32_t stage0 = 0, phase0 = 0;     // stage and phase of the batch's first page
        bool aborted = false;
        // Lookups are software-pipelined over batches: the kept-id load of batch
        // k+2 and the block-table load of batch k+1 are in flight while batch k
        // is issued, so their latency hides behind the ring instead of stalling it.
        // A lookup moves through stages: 0 located, kept id not read yet (the
        // single-launch kernel reads it only once the unit's selection is
        // published); 1 id read; 2 block-table entry read, or nothing to do.
        int seen_ready = -1;   // the last unit this lane saw published (acquired once)
        auto read_id = [&](Look &lk) {                   // stage 0 -> 1 when the id is available
            const size_t u = (size_t)lk.b * Hkv + lk.h;
            if (p.dense) {
                lk.page = lk.j;
            } else if constexpr (FUSED) {
                if ((int)u != seen_ready) {
                    if (ld_acquire_gpu(&p.ready[u]) == 0) return;
                    seen_ready = (int)u;
                }
                lk.page = __ldcg(&p.selected[u * p.max_budget + lk.j]);
            } else {
                lk.page = p.selected[u * p.max_budget + lk.j];
            }
            lk.stage = 1;
        };
        auto look_a = [&](long long bb, Look &lk) {      // locate; read the kept id
            look_loc(bb, lk);
            if (lk.stage == 0) read_id(lk);
        };
        auto look_b = [&](Look &lk) {                    // check the id; read the block-table entry
            if (lk.stage == 0) read_id(lk);
            if (lk.stage != 1) return;
            lk.stage = 2;
            const int N = (lens[lk.b] + P - 1) / P;
            if (lk.page < 0 || lk.page >= N) {
                if (p.status) atomicOr(p.status, QASA_DEVERR_SELECTED);
                return;
            }
            lk.ok = true;
            lk.phys = p.block_table[(size_t)lk.b * p.max_pages + lk.page];
        };
        // Complete a lookup that is about to be issued.  In the single-launch
        // kernel this waits (bounded) for the selection of every lane's unit.
        auto finish = [&](Look &lk) -> bool {
            if constexpr (FUSED) {
                uint64_t t_begin = 0;
                for (int spin = 0;; ++spin) {
                    if (lk.stage == 0) read_id(lk);
                    if (!__any_sync(0xffffffffu, lk.stage == 0)) break;
                    int stop = 0;
                    if (lane == 0 && (spin & 15) == 15) {
                        const uint64_t now = global_timer_ns();
                        if (t_begin == 0) t_begin = now;
                        else if (now - t_begin > p.wait_limit_ns || *abort_flag) stop = 1;
                    }
                    if (__shfl_sync(0xffffffffu, stop, 0)) {
                        if (lane == 0) {
                            if (p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                            *abort_flag = 1;
                        }
                        return false;
                    }
                    __nanosleep(128);
                }
            }
            look_b(lk);
            return true;
        };
        look_b(la);                                  // batches 0 and 1 were located before the wait
        if (lb.stage == 0) read_id(lb);
        for (long long base = 0; base < n_loc && !aborted; base += WB) {
            const int nb = (int)min((long long)WB, n_loc - base);
            if (!finish(la)) {
                aborted = true;
                break;
            }
            int nvalid = 0, row = 0;
            const int page = la.page;
            if (la.active && la.ok) {                    // check the physical page
                if (la.phys < 0 || la.phys >= p.num_phys) {
                    if (p.status) atomicOr(p.status, QASA_DEVERR_PAGE_ID);
                } else {
                    nvalid = min(P, lens[la.b] - page * P);
                    row = (int)(((long long)la.phys * Hkv + la.h) * P);
                }
            }
            // (the first batch is issued before the next lookups: nothing is in
            // flight yet, so their latency would only delay the first copies)
            if (base != 0) {
                look_b(lb);
                look_a(base + 2 * (long long)WB, lc);
            }
            uint32_t s_l = stage0 + lane, ph_l = phase0;
            if (s_l >= (uint32_t)S) { s_l -= S; ph_l ^= 1u; }
            bool pending = lane < nb;
            uint64_t t_begin = 0;
            for (int spin = 0;; ++spin) {
                const bool any = __any_sync(0xffffffffu, pending);
                int stop = 0;
                if (lane == 0 && any && (spin & 63) == 63) {
                    const uint64_t now = global_timer_ns();
                    if (t_begin == 0) t_begin = now;
                    else if (now - t_begin > p.wait_limit_ns || *abort_flag) stop = 1;
                }
                stop = __shfl_sync(0xffffffffu, stop, 0);
                if (!any) break;
                if (stop) {
                    if (lane == 0) {
                        if (p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    aborted = true;
                    break;
                }
                const bool ready = pending && mbar_test_wait(&empty_bar[s_l], ph_l ^ 1u);
                if (!__any_sync(0xffffffffu, ready)) {   // nothing free yet: back off
                    __nanosleep(64);
                    continue;
                }
                if (ready) {
                    if (tr && base == 0 && lane == 0) trace_stamp(tr + 3);
                    info[s_l].page = page;
                    info[s_l].nvalid = nvalid;
                    unsigned char *st = ring + (size_t)s_l * STAGE;
                    if (nvalid > 0) {
                        mbar_arrive_expect_tx(&full_bar[s_l], STAGE + (F8 ? 16 : 0));
                        if constexpr (F8) {
                            // the code tiles (one box for K and V when the pools allow),
                            // and the page's scales (16 bytes)
                            if (p.one_box == 2) {
                                tma_load_3d(st, &kmap, &full_bar[s_l], 0, row, 0);
                            } else {
                                tma_load_2d(st, &kmap, &full_bar[s_l], 0, row);
                                tma_load_2d(st + TILE, &vmap, &full_bar[s_l], 0, row);
                            }
                            bulk_load(&st_scale[s_l], p.scales + (size_t)(row / P) * 4, 16, &full_bar[s_l]);
                        } else if (p.one_box == 2) {
                            // K and V tiles of the page in one box (the V pool sits at a
                            // fixed offset from the K pool): one TMA operation per page
                            tma_load_4d(st, &kmap, &full_bar[s_l], 0, row, 0, 0);
                        } else if (p.one_box) {
                            tma_load_3d(st, &kmap, &full_bar[s_l], 0, row, 0);
                            tma_load_3d(st + TILE, &vmap, &full_bar[s_l], 0, row, 0);
                        } else {
#pragma unroll
                            for (int x = 0; x < NSUB; ++x) {
                                tma_load_2d(st + x * P * 128, &kmap, &full_bar[s_l], x * BOXW, row);
                                tma_load_2d(st + TILE + x * P * 128, &vmap, &full_bar[s_l], x * BOXW, row);
                            }
                        }
                        last_ph[s_l] = (int)ph_l;
                    } else {
                        mbar_arrive(&full_bar[s_l]);
                    }
                    pending = false;
                }
            }
            if (base == 0) {
                look_b(lb);
                look_a(2 * (long long)WB, lc);
            }
            stage0 += nb;
            if (stage0 >= (uint32_t)S) { stage0 -= S; phase0 ^= 1u; }
            la = lb;
            lb = lc;
        }
        if (lane == 0) trace_stamp(tr ? tr + 5 : nullptr);
        // drain: the copies this CTA issued must land before it exits (bounded)
        __syncwarp();
        for (int s = lane; s < S; s += 32) {
            const int ph = last_ph[s];
            if (ph >= 0 && !mbar_wait_bounded(&full_bar[s], (uint32_t)ph, p.drain_limit_ns) && p.status)
                atomicOr(p.status, QASA_DEVERR_TIMEOUT);
        }
        return;
    }

    // A working warp may overwrite the shared state slot for segment k once the
    // combiners have read segment k-1 (phase k-1 of the "free" barrier).
    auto wait_slot_free = [&](uint32_t k) -> bool {
        if (mbar_wait_bounded(&seg_bar[1], (k & 1u) ^ 1u, p.wait_limit_ns)) return true;
        if (lane == 0) {
            if (p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        return false;
    };

    // The combiners: for every segment of the CTA range, in order, merge the
    // working warps' (m, l, o) into registers, release the slot, then write the
    // output (whole unit) or this CTA's partial plus the unit's page ticket; the
    // CTA that completes a unit's ticket merges all its partials.
    //
    // The warps not working on pages (NC = NW - NWK >= 1 of them, index ci)
    // share this: a whole unit's heads are split between them (heads ci,
    // ci + NC, ...); a unit split with another CTA is done by warp 0 of them
    // alone (all heads, the partial, the ticket and the last merge) while the
    // others only release the slot.
    auto combine_segments = [&](int ci, int NC) {
        constexpr int JPH = D / 32;                    // elements per lane per head
        long long pos = 0;
        uint32_t kseg = 0;
        while (pos < n_loc) {
            const long long g = rot(pos);
            int b, h, j0, cnt;
            long long us;
            locate(g, b, h, j0, us, cnt);
            const long long ue = us + cnt;
            const long long s1 = min(run_end(pos), ue);
            pos += s1 - g;
            const int u = b * Hkv + h;
            if (pos >= n_loc && g == us && s1 == ue) return;   // merged by the working warps
            if (!mbar_wait_bounded(&seg_bar[0], kseg & 1u, p.wait_limit_ns)) {
                if (lane == 0) {
                    if (p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                return;
            }
            const bool whole = g == us && s1 == ue;    // the whole unit is in this CTA
            if (whole && NC > 1) {
                // heads ci, ci + NC, ... (at most KH of them) of a whole unit
                constexpr int KH = (GMAX + 1) / 2;
                float acc[KH][JPH], Mh[KH], Lh[KH];
#pragma unroll
                for (int k = 0; k < KH; ++k) {
                    Mh[k] = -INFINITY;
                    Lh[k] = 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) acc[k][jj] = 0.f;
                }
                for (int x = 0; x < NWK; ++x) {
#pragma unroll
                    for (int k = 0; k < KH; ++k) {
                        const int hh = ci + k * NC;
                        if (hh >= G) break;
                        float ox[JPH];
#pragma unroll
                        for (int jj = 0; jj < JPH; ++jj) ox[jj] = scr_o[(x * GMAX + hh) * D + jj * 32 + lane];
                        merge_state<JPH>(Mh[k], Lh[k], acc[k], scr_m[x * GMAX + hh], scr_l[x * GMAX + hh], ox);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&seg_bar[1]);   // the slot may be reused (once every combiner is here)
                ++kseg;
                MT *ob = static_cast<MT *>(p.out) + ((size_t)b * p.Hq + (size_t)h * G) * D;
#pragma unroll
                for (int k = 0; k < KH; ++k) {
                    const int hh = ci + k * NC;
                    if (hh >= G) break;
                    const float inv = Lh[k] > 0.f ? 1.f / Lh[k] : 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) ob[hh * D + jj * 32 + lane] = elem<MT>::from_f(acc[k][jj] * inv);
                }
                continue;
            }
            if (!whole && ci != 0) {                   // warp 0 of the combiners takes it
                __syncwarp();
                if (lane == 0) mbar_arrive(&seg_bar[1]);
                ++kseg;
                continue;
            }
            // every head (a whole unit with one combiner warp, or a split unit):
            // online merge over the working warps; one warp's loads are all
            // independent, so they overlap instead of forming a chain
            float acc[GMAX][JPH], Mh[GMAX], Lh[GMAX];
#pragma unroll
            for (int hh = 0; hh < GMAX; ++hh) {
                Mh[hh] = -INFINITY;
                Lh[hh] = 0.f;
#pragma unroll
                for (int jj = 0; jj < JPH; ++jj) acc[hh][jj] = 0.f;
            }
            for (int x = 0; x < NWK; ++x) {
                float mx[GMAX], lx[GMAX], ox[GMAX][JPH];
#pragma unroll
                for (int hh = 0; hh < GMAX; ++hh) {
                    const bool on = hh < G;
                    mx[hh] = on ? scr_m[x * GMAX + hh] : -INFINITY;
                    lx[hh] = on ? scr_l[x * GMAX + hh] : 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) ox[hh][jj] = on ? scr_o[(x * GMAX + hh) * D + jj * 32 + lane] : 0.f;
                }
#pragma unroll
                for (int hh = 0; hh < GMAX; ++hh) merge_state<JPH>(Mh[hh], Lh[hh], acc[hh], mx[hh], lx[hh], ox[hh]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&seg_bar[1]);   // the slot may be reused (once every combiner is here)
            ++kseg;

            MT *ob = static_cast<MT *>(p.out) + ((size_t)b * p.Hq + (size_t)h * G) * D;
            if (whole) {
#pragma unroll
                for (int hh = 0; hh < GMAX; ++hh) {
                    if (hh >= G) break;
                    const float inv = Lh[hh] > 0.f ? 1.f / Lh[hh] : 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) ob[hh * D + jj * 32 + lane] = elem<MT>::from_f(acc[hh][jj] * inv);
                }
                continue;
            }
            // partial: publish it, then take the unit's ticket.  __syncwarp orders
            // the lanes' stores before lane 0's acquire-release atomic, which
            // publishes them and makes the other CTAs' partials visible.  The ticket counts pages, so CTAs with an empty
            // range (grid larger than the kept-page count) cannot leave it short.
            const size_t slot = (size_t)u + c;
#pragma unroll
            for (int hh = 0; hh < GMAX; ++hh) {
                if (hh >= G) break;
#pragma unroll
                for (int jj = 0; jj < JPH; ++jj) p.part_o[(slot * G + hh) * D + jj * 32 + lane] = acc[hh][jj];
                if (lane == 0) {
                    p.part_ml[(slot * G + hh) * 2] = Mh[hh];
                    p.part_ml[(slot * G + hh) * 2 + 1] = Lh[hh];
                }
            }
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                const int npg = (int)(s1 - g);
                const int prev = atomic_add_acq_rel_gpu(&p.counters[u], npg);   // release ours, acquire theirs
                last = (prev + npg == cnt);
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();
            if (last) {
                const long long wu = unit_w() * (u + 1), vt = weighted_total();
                const int cf = cta_of_v(us + wu, C, vt), cl = cta_of_v(ue - 1 + wu, C, vt);
#pragma unroll
                for (int hh = 0; hh < GMAX; ++hh) {
                    Mh[hh] = -INFINITY;
                    Lh[hh] = 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) acc[hh][jj] = 0.f;
                }
                for (int x = cf; x <= cl; ++x) {
                    if (rstart[x] == rstart[x + 1]) continue;   // empty range
                    const size_t sb = (size_t)(u + x) * G;
                    float mx[GMAX], lx[GMAX], ox[GMAX][JPH];
#pragma unroll
                    for (int hh = 0; hh < GMAX; ++hh) {
                        const bool on = hh < G;
                        mx[hh] = on ? __ldcg(&p.part_ml[(sb + hh) * 2]) : -INFINITY;
                        lx[hh] = on ? __ldcg(&p.part_ml[(sb + hh) * 2 + 1]) : 0.f;
#pragma unroll
                        for (int jj = 0; jj < JPH; ++jj) ox[hh][jj] = on ? __ldcg(&p.part_o[(sb + hh) * D + jj * 32 + lane]) : 0.f;
                    }
#pragma unroll
                    for (int hh = 0; hh < GMAX; ++hh) merge_state<JPH>(Mh[hh], Lh[hh], acc[hh], mx[hh], lx[hh], ox[hh]);
                }
#pragma unroll
                for (int hh = 0; hh < GMAX; ++hh) {
                    if (hh >= G) break;
                    const float inv = Lh[hh] > 0.f ? 1.f / Lh[hh] : 0.f;
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) ob[hh * D + jj * 32 + lane] = elem<MT>::from_f(acc[hh][jj] * inv);
                }
                if (lane == 0) p.counters[u] = 0;
            }
        }
    };

    // ---------------------------------------------------------------- consumers
    // Warps 1..NWK take pages; the other warps are the combiners, which merge
    // the working warps' states at every unit boundary (segment) of the CTA
    // range while they move on.
    const int w = warp - 1;
    if (w >= NWK) {
        combine_segments(w - NWK, NW - NWK);
        if (w == NW - 1 && lane == 0) trace_stamp(tr ? tr + 7 : nullptr);
        return;
    }
    long long pos = 0;
    uint32_t kseg = 0;
    while (pos < n_loc) {
        const long long g = rot(pos);
        int b, h, j0, cnt;
        long long us;
        locate(g, b, h, j0, us, cnt);
        const long long ue = us + cnt;
        const long long s1 = min(run_end(pos), ue);
        const MT *qb = static_cast<const MT *>(p.q) + ((size_t)b * p.Hq + (size_t)h * G) * D;
        // FP8: turn a code tile into this warp's half copy (rows >= nvalid as zeros)
        unsigned char *my_k = f8_scr + (size_t)w * 2 * P * D * 2, *my_v = my_k + P * D * 2;
        auto f8_to_half = [&](const unsigned char *src, unsigned char *dst, int nvalid) {
            constexpr int CH = D / 16;               // 16-code chunks per row
            for (int idx = lane; idx < P * CH; idx += 32) {
                const int r = idx / CH, k = idx % CH;
                uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
                if (r < nvalid) e4m3x16_to_h(*reinterpret_cast<const uint4 *>(src + r * D + k * 16), lo, hi);
                *reinterpret_cast<uint4 *>(dst + swz128_offset<P>(r, 2 * k)) = lo;
                *reinterpret_cast<uint4 *>(dst + swz128_offset<P>(r, 2 * k + 1)) = hi;
            }
        };

        // Page i of the CTA range goes to consumer warp i % NWK and ring stage
        // i % S.  S is a multiple of NWK, so every stage always belongs to the
        // same warp, which consumes its rounds in order: a parity wait on a
        // stage can then never alias with a fill two phases behind (copies
        // complete out of order, so a stage shared by several warps could be
        // observed "full" while an older fill into it is still in flight).
        const int first = (int)pos;
        const int lastx = (int)(pos + (s1 - g));
        int i = first + ((w - first % NWK) % NWK + NWK) % NWK;
        int s = i % S;
        uint32_t ph = (uint32_t)((i / S) & 1);

        if constexpr (MMA) {
            const int cq = lane & 3, nq = lane >> 2;
            uint32_t qf[D / 16][2];
            if constexpr (F8MMA) {
                // FP8: the K fragments come from code bytes 4c..4c+3 of a row, which
                // feed MMA slots (2c, 2c+1) and (2c+8, 2c+9): q takes the same
                // channel order, channels 16ks + 4cq .. 16ks + 4cq + 3 per lane
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint2 r = make_uint2(0u, 0u);
                    if (nq < G) r = *reinterpret_cast<const uint2 *>(qb + (size_t)nq * D + ks * 16 + 4 * cq);
                    qf[ks][0] = r.x;
                    qf[ks][1] = r.y;
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    qf[ks][0] = 0u; qf[ks][1] = 0u;
                    if (nq < G) {
                        const MT *qr = qb + (size_t)nq * D + ks * 16 + 2 * cq;
                        qf[ks][0] = *reinterpret_cast<const uint32_t *>(qr);
                        qf[ks][1] = *reinterpret_cast<const uint32_t *>(qr + 8);
                    }
                }
            }
            float o[D / 16][4];
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

            for (; i < lastx; i += NWK, s += NWK) {
                while (s >= S) { s -= S; ph ^= 1u; }
                if (*abort_flag) break;
                if (!mbar_wait_bounded(&full_bar[s], ph, p.wait_limit_ns)) {
                    if (lane == 0 && p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (tr && i == w && lane == 0) trace_stamp(tr + 4);
                const int nvalid = info[s].nvalid;
                unsigned char *kst = ring + (size_t)s * STAGE;
                unsigned char *vst = kst + TILE;
                uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
                float zscale = p.scale_log2, vscale = 1.f;
                if constexpr (F8MMA) {
                    if (nvalid > 0) {
                        const float4 am = st_scale[s];
                        zscale = p.scale_log2 * fp8_scale(am.x);
                        vscale = fp8_scale(am.y);
                    }
                }
                if constexpr (F8CONV) {
                    if (nvalid > 0) {
                        const float4 am = st_scale[s];
                        zscale = p.scale_log2 * fp8_scale(am.x);
                        vscale = fp8_scale(am.y);
                        f8_to_half(kst, my_k, nvalid);
                        f8_to_half(vst, my_v, nvalid);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_bar[s]);   // the codes are copied out: free the stage
                    kbase = smem_u32(my_k);
                    vbase = smem_u32(my_v);
                } else if (nvalid > 0 && nvalid < P) {
                    // rows past the sequence end may hold anything: zero V there so that
                    // the masked (zero) weights cannot meet a NaN in the P.V product
                    const int rows = ((nvalid + 15) & ~15) - nvalid;
                    for (int e = lane; e < rows * NSUB * 8; e += 32) {
                        const int r = nvalid + e / (NSUB * 8), ch = e % (NSUB * 8);
                        *reinterpret_cast<uint4 *>(vst + swz128_offset<P>(r, ch)) = make_uint4(0, 0, 0, 0);
                    }
                    __syncwarp();
                }
#pragma unroll
                for (int sub = 0; sub < P / 16; ++sub) {
                    if (sub * 16 >= nvalid) break;
                    float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
                    if constexpr (F8MMA) {
                        // S^T = K q^T with K fragments converted in registers: ldmatrix
                        // on the (128-byte swizzled) code tile gives a lane the codes of
                        // channels 4c..4c+3 of rows g and g+8 of two 16-channel blocks
#pragma unroll
                        for (int kk = 0; kk < D / 32; ++kk) {
                            const int tok = sub * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                            uint32_t r[4];
                            ldmatrix_x4(kbase + swz128_offset<P>(tok, 2 * kk + (lane >> 4)), r[0], r[1], r[2], r[3]);
                            const uint32_t a0[4] = {e4m3x2_to_h2(r[0]), e4m3x2_to_h2(r[1]), e4m3x2_to_h2(r[0] >> 16),
                                                    e4m3x2_to_h2(r[1] >> 16)};
                            mma16816<MT>::run(sa, a0, qf[2 * kk][0], qf[2 * kk][1]);
                            const uint32_t a1[4] = {e4m3x2_to_h2(r[2]), e4m3x2_to_h2(r[3]), e4m3x2_to_h2(r[2] >> 16),
                                                    e4m3x2_to_h2(r[3] >> 16)};
                            mma16816<MT>::run(sb, a1, qf[2 * kk + 1][0], qf[2 * kk + 1][1]);
                        }
                    } else {
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const int tok = sub * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                            const int chn = 2 * ks + (lane >> 4);
                            uint32_t a[4];
                            ldmatrix_x4(kbase + swz128_offset<P>(tok, chn), a[0], a[1], a[2], a[3]);
                            if (ks & 1) mma16816<MT>::run(sb, a, qf[ks][0], qf[ks][1]);
                            else mma16816<MT>::run(sa, a, qf[ks][0], qf[ks][1]);
                        }
                    }
                    const int t0 = sub * 16 + (lane >> 2), t1 = t0 + 8;
                    const bool v0 = t0 < nvalid, v1 = t1 < nvalid;
                    const float z0 = v0 ? (sa[0] + sb[0]) * zscale : -INFINITY;
                    const float z1 = v0 ? (sa[1] + sb[1]) * zscale : -INFINITY;
                    const float z2 = v1 ? (sa[2] + sb[2]) * zscale : -INFINITY;
                    const float z3 = v1 ? (sa[3] + sb[3]) * zscale : -INFINITY;
                    float x0 = fmaxf(z0, z2), x1 = fmaxf(z1, z3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
                        x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
                    }
                    const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
                    const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
                    const float p0 = exp2f(z0 - n0), p1 = exp2f(z1 - n1);
                    const float p2 = exp2f(z2 - n0), p3 = exp2f(z3 - n1);
                    l0 = l0 * al0 + p0 + p2;
                    l1 = l1 * al1 + p1 + p3;
                    m0 = n0; m1 = n1;
                    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {   // the maximum moved
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
                        }
                    }
                    // FP8: the page's V scale rides on the weights (l keeps the plain sum)
                    const uint32_t pb0 = movmatrix_trans(mma16816<MT>::pack2(p0 * vscale, p1 * vscale));
                    const uint32_t pb1 = movmatrix_trans(mma16816<MT>::pack2(p2 * vscale, p3 * vscale));
                    if constexpr (F8MMA) {
                        // V^T fragments from the code tile: ldmatrix.trans hands a lane
                        // the codes of tokens (2cq, 2cq+1) x channels (2nq, 2nq+1) of a
                        // 16-channel chunk; byte permutes regroup them per channel and
                        // each pair converts to halves.  Row nq of M-tile j is channel
                        // 16j + 2nq, row nq + 8 is channel 16j + 2nq + 1.
#pragma unroll
                        for (int j = 0; j < D / 16; j += 2) {
                            const int tok = sub * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                            uint32_t r[4];
                            ldmatrix_x4_trans(vbase + swz128_offset<P>(tok, j + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const uint32_t X = __byte_perm(r[2 * hf], r[2 * hf + 1], 0x6420);
                                const uint32_t Y = __byte_perm(r[2 * hf], r[2 * hf + 1], 0x7531);
                                const uint32_t a[4] = {e4m3x2_to_h2(X), e4m3x2_to_h2(Y), e4m3x2_to_h2(X >> 16),
                                                       e4m3x2_to_h2(Y >> 16)};
                                mma16816<MT>::run(o[j + hf], a, pb0, pb1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int mt = 0; mt < D / 16; ++mt) {
                            const int tok = sub * 16 + (lane & 7) + (lane >> 4) * 8;
                            const int chn = 2 * mt + ((lane >> 3) & 1);
                            uint32_t a[4];
                            ldmatrix_x4_trans(vbase + swz128_offset<P>(tok, chn), a[0], a[1], a[2], a[3]);
                            mma16816<MT>::run(o[mt], a, pb0, pb1);
                        }
                    }
                }
                __syncwarp();
                if (!F8CONV && lane == 0) mbar_arrive(&empty_bar[s]);
            }
            // hand this warp's state to the combiners
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            if (!wait_slot_free(kseg)) break;
            const int h0 = 2 * cq, h1 = 2 * cq + 1;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                // accumulator rows nq / nq + 8 of M-tile mt: channels mt*16 + nq / + 8
                // (FP8 tensor-core path: mt*16 + 2nq / + 1)
                const int ch = F8MMA ? mt * 16 + 2 * nq : mt * 16 + nq;
                const int ch2 = F8MMA ? ch + 1 : ch + 8;
                if (h0 < G) {
                    scr_o[(w * GMAX + h0) * D + ch] = o[mt][0];
                    scr_o[(w * GMAX + h0) * D + ch2] = o[mt][2];
                }
                if (h1 < G) {
                    scr_o[(w * GMAX + h1) * D + ch] = o[mt][1];
                    scr_o[(w * GMAX + h1) * D + ch2] = o[mt][3];
                }
            }
            if (nq == 0) {
                if (h0 < G) { scr_m[w * GMAX + h0] = m0; scr_l[w * GMAX + h0] = l0; }
                if (h1 < G) { scr_m[w * GMAX + h1] = m1; scr_l[w * GMAX + h1] = l1; }
            }
        } else {
            // ---------------------------------------------- FFMA consumer
            constexpr int EPC = chunk16<MT>::n;
            constexpr int LPT = 32 / P;              // lanes per token
            constexpr int CPT = D / LPT;             // channels per lane for q.k
            constexpr int KCH = CPT / EPC;           // 16-byte chunks per lane for q.k
            constexpr int DPL = D / 32;              // channels per lane for p.v
            float *qs = ff_q + w * GMAX * D;
            float *ps = ff_p + w * GMAX * P;
            for (int e = lane; e < G * D; e += 32) qs[e] = elem<MT>::to_f(qb[e]);
            __syncwarp();
            float o[GMAX][DPL], m[GMAX], l[GMAX];
#pragma unroll
            for (int gg = 0; gg < GMAX; ++gg) {
                m[gg] = -INFINITY; l[gg] = 0.f;
#pragma unroll
                for (int x = 0; x < DPL; ++x) o[gg][x] = 0.f;
            }
            const int tk = lane / LPT, sl = lane % LPT;
            for (; i < lastx; i += NWK, s += NWK) {
                while (s >= S) { s -= S; ph ^= 1u; }
                if (*abort_flag) break;
                if (!mbar_wait_bounded(&full_bar[s], ph, p.wait_limit_ns)) {
                    if (lane == 0 && p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                const int nvalid = info[s].nvalid;
                const unsigned char *kst = ring + (size_t)s * STAGE;
                const unsigned char *vst = kst + TILE;
                float zscale = p.scale_log2, vscale = 1.f;
                if constexpr (F8CONV) {
                    if (nvalid > 0) {
                        const float4 am = st_scale[s];
                        zscale = p.scale_log2 * fp8_scale(am.x);
                        vscale = fp8_scale(am.y);
                        f8_to_half(kst, my_k, nvalid);
                        f8_to_half(vst, my_v, nvalid);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_bar[s]);   // the codes are copied out: free the stage
                    kst = my_k;
                    vst = my_v;
                }
                if (nvalid > 0) {
                    float acc[GMAX];
#pragma unroll
                    for (int gg = 0; gg < GMAX; ++gg) acc[gg] = 0.f;
#pragma unroll
                    for (int x = 0; x < KCH; ++x) {
                        const int chunk = sl * KCH + x;
                        float f[EPC];
                        chunk16<MT>::unpack(*reinterpret_cast<const uint4 *>(kst + swz128_offset<P>(tk, chunk)), f);
#pragma unroll
                        for (int gg = 0; gg < GMAX; ++gg)
#pragma unroll
                            for (int e = 0; e < EPC; ++e)
                                acc[gg] = fmaf(qs[gg * D + chunk * EPC + e], f[e], acc[gg]);
                    }
                    const bool valid = tk < nvalid;
#pragma unroll
                    for (int gg = 0; gg < GMAX; ++gg) {
                        if (gg >= G) break;
                        float a = acc[gg];
                        if (LPT == 2) a += __shfl_xor_sync(0xffffffffu, a, 1);
                        const float z = valid ? a * zscale : -INFINITY;
                        float mx = z;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                        const float nm = fmaxf(m[gg], mx);
                        const float al = exp2f(m[gg] - nm);
                        const float pz = exp2f(z - nm);
                        float sum = sl == 0 ? pz : 0.f;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                        l[gg] = l[gg] * al + sum;
                        m[gg] = nm;
#pragma unroll
                        for (int x = 0; x < DPL; ++x) o[gg][x] *= al;
                        if (sl == 0) ps[gg * P + tk] = pz * vscale;   // FP8: V scale on the weight
                    }
                    __syncwarp();
                    for (int t = 0; t < nvalid; ++t) {
                        const int byte = lane * DPL * MES;
                        const unsigned char *vp = vst + swz128_offset<P>(t, byte >> 4) + (byte & 15);
                        float v[DPL];
#pragma unroll
                        for (int x = 0; x < DPL; ++x) v[x] = elem<MT>::to_f(reinterpret_cast<const MT *>(vp)[x]);
#pragma unroll
                        for (int gg = 0; gg < GMAX; ++gg) {
                            if (gg >= G) break;
                            const float pw = ps[gg * P + t];
#pragma unroll
                            for (int x = 0; x < DPL; ++x) o[gg][x] = fmaf(pw, v[x], o[gg][x]);
                        }
                    }
                }
                __syncwarp();
                if (!F8CONV && lane == 0) mbar_arrive(&empty_bar[s]);
            }
            if (!wait_slot_free(kseg)) break;
#pragma unroll
            for (int gg = 0; gg < GMAX; ++gg) {
                if (gg >= G) break;
#pragma unroll
                for (int x = 0; x < DPL; ++x) scr_o[(w * GMAX + gg) * D + lane * DPL + x] = o[gg][x];
                if (lane == 0) { scr_m[w * GMAX + gg] = m[gg]; scr_l[w * GMAX + gg] = l[gg]; }
            }
        }
        __syncwarp();
        if (lastx >= n_loc && g == us && s1 == ue) {
            // The range's last segment is a whole unit: instead of handing it
            // to the combiners (a few warps), the working warps
            // merge it together, warp w taking heads w, w + NWK, ...
            if (lane == 0) mbar_arrive(&seg_bar[2]);
            if (!mbar_wait_bounded(&seg_bar[2], 0u, p.wait_limit_ns)) {
                if (lane == 0) {
                    if (p.status) atomicOr(p.status, QASA_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            if (w == 0 && lane == 0) trace_stamp(tr ? tr + 9 : nullptr);
            constexpr int JPH = D / 32;
            MT *ob = static_cast<MT *>(p.out) + ((size_t)b * p.Hq + (size_t)h * G) * D;
            for (int hh = w; hh < G; hh += NWK) {
                float M = -INFINITY, L = 0.f, acc[JPH];
#pragma unroll
                for (int jj = 0; jj < JPH; ++jj) acc[jj] = 0.f;
                for (int x = 0; x < NWK; ++x) {
                    float ox[JPH];
#pragma unroll
                    for (int jj = 0; jj < JPH; ++jj) ox[jj] = scr_o[(x * GMAX + hh) * D + jj * 32 + lane];
                    merge_state<JPH>(M, L, acc, scr_m[x * GMAX + hh], scr_l[x * GMAX + hh], ox);
                }
                const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
                for (int jj = 0; jj < JPH; ++jj) ob[hh * D + jj * 32 + lane] = elem<MT>::from_f(acc[jj] * inv);
            }
            if (w == 0 && lane == 0) trace_stamp(tr ? tr + 10 : nullptr);
            break;
        }
        if (lane == 0) mbar_arrive(&seg_bar[0]);
        ++kseg;
        pos = lastx;
    }
    if (lane == 0) trace_latest(tr ? tr + 6 : nullptr);
}

// ------------------------------------------------------------------ launch

template <typename T, int D, int P, bool MMA, int GMAX, bool FUSED>
static cudaError_t launch_attn_t(const CUtensorMap &km, const CUtensorMap &vm, const AttnParams &p0,
                                 int grid, size_t smem_budget, bool pdl, cudaStream_t stream) {
    // The single-launch kernel adds 4 selector warps; one consumer warp fewer
    // keeps its registers per thread at the two-kernel level.
    constexpr int NW = FUSED ? 7 : 8;
    constexpr bool F8 = is_fp8<T>::value;
    constexpr bool F8CONV = F8 && !(MMA && D == 128);   // FP8 tiles converted through shared memory
    constexpr int STAGE = 2 * P * D * (F8 ? 1 : (int)sizeof(T));
    AttnParams p = p0;
    // Pick the number of working consumer warps (up to NW-1) that allows the deepest ring
    // whose depth is a multiple of it (each stage owned by one consumer warp).
    const size_t per = (size_t)STAGE + 2 * sizeof(uint64_t) + sizeof(StageInfo) + sizeof(int) + (F8 ? 16 : 0);
    // ring depth cap: 64 stages or ~200 KB of tiles in flight, whichever is less
    // (16-bit pages reach the shared-memory limit first; FP8 pages are half the
    // bytes and need twice the stages for the same bytes in flight)
    constexpr int kMaxStages = (200 * 1024 / STAGE) < 64 ? (200 * 1024 / STAGE) : 64;
    int stages = 0, consumers = 0;
    // 16-bit KV: four working warps whenever the ring still holds at least four
    // pages per warp (fewer states per unit-boundary merge; the streaming rate
    // is the same from four warps up), six for pages of 4 KB or less, whose
    // rate is set by the per-page work rather than by the bytes
    if constexpr (!F8) {
        constexpr int kPreferred = STAGE <= 4096 ? 6 : 4;
        if (kPreferred <= NW - 1) {
            const size_t fixed = attn_smem_bytes(0, STAGE, kPreferred, GMAX, D, P, MMA, p.B, grid, FUSED, p.max_pages,
                                                 F8, F8CONV);
            int s = fixed < smem_budget ? (int)((smem_budget - fixed) / per) : 0;
            if (s > kMaxStages) s = kMaxStages;
            s = s / kPreferred * kPreferred;
            if (s >= 4 * kPreferred) { stages = s; consumers = kPreferred; }
        }
    }
    for (int nw = NW - 1; nw >= 1 && stages == 0; --nw) {   // at least one warp is left to combine
        const size_t fixed = attn_smem_bytes(0, STAGE, nw, GMAX, D, P, MMA, p.B, grid, FUSED, p.max_pages, F8, F8CONV);
        if (fixed >= smem_budget) continue;
        int s = (int)((smem_budget - fixed) / per);
        if (s > kMaxStages) s = kMaxStages;
        const int c = s < nw ? s : nw;
        if (c < 1) continue;
        s = s / c * c;
        if constexpr (F8) {
            // FP8 pages are half the bytes, so the ring is deep enough at any
            // count; the consumers' per-page work is what limits: take the most
            if (s >= 2 * c && c > consumers) { stages = s; consumers = c; }
            continue;
        }
        if (s > stages || (s == stages && c > consumers)) { stages = s; consumers = c; }
        if (nw <= 4 && stages >= 2) break;
    }
    if (const char *force = std::getenv("QASA_ATTN_CONSUMERS")) {   // diagnostic: fix the consumer warps
        const int want = std::atoi(force);
        if (want >= 1 && want <= NW - 1) {
            const size_t fixed = attn_smem_bytes(0, STAGE, want, GMAX, D, P, MMA, p.B, grid, FUSED, p.max_pages, F8, F8CONV);
            int s = fixed < smem_budget ? (int)((smem_budget - fixed) / per) : 0;
            if (s > kMaxStages) s = kMaxStages;
            s = s / want * want;
            if (s >= 2) { stages = s; consumers = want; }
        }
    }
    if (stages < 2) return cudaErrorInvalidConfiguration;
    p.stages = stages;
    p.consumers = consumers;
    const size_t smem = attn_smem_bytes(stages, STAGE, consumers, GMAX, D, P, MMA, p.B, grid, FUSED, p.max_pages, F8, F8CONV);
    auto kern = attn_kernel<T, D, P, MMA, GMAX, NW, FUSED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * (NW + 1) + (FUSED ? kSelThreads : 0));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (FUSED) {
        // CTAs wait (bounded) for selections made by other CTAs: ask for a
        // launch in which every CTA is resident at once
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    } else {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = (FUSED || pdl) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, km, vm, p);
}

template <typename T, int D, int P, bool FUSED>
static cudaError_t launch_attn_dp(const CUtensorMap &km, const CUtensorMap &vm, const AttnParams &p,
                                  int grid, size_t smem_budget, bool pdl, cudaStream_t stream) {
    if constexpr (is_fp8<T>::value || sizeof(T) == 2) {
        // tensor cores for every group size: with G < 8 the unused query heads
        // of the 8-wide MMA are zero (for G = 1, 1.25x faster than FFMA at
        // GPT2-345M shapes, the same selection)
        return launch_attn_t<T, D, P, true, 8, FUSED>(km, vm, p, grid, smem_budget, pdl, stream);
    } else {
        return launch_attn_t<T, D, P, false, 8, FUSED>(km, vm, p, grid, smem_budget, pdl, stream);
    }
}

template <typename T, bool FUSED>
static cudaError_t launch_attn_dt(int D, int P, const CUtensorMap &km, const CUtensorMap &vm,
                                  const AttnParams &p, int grid, size_t smem_budget, bool pdl,
                                  cudaStream_t stream) {
    if (D == 64)
        return P == 16 ? launch_attn_dp<T, 64, 16, FUSED>(km, vm, p, grid, smem_budget, pdl, stream)
                       : launch_attn_dp<T, 64, 32, FUSED>(km, vm, p, grid, smem_budget, pdl, stream);
    return P == 16 ? launch_attn_dp<T, 128, 16, FUSED>(km, vm, p, grid, smem_budget, pdl, stream)
                   : launch_attn_dp<T, 128, 32, FUSED>(km, vm, p, grid, smem_budget, pdl, stream);
}

cudaError_t launch_attention(qasa_dtype dt, int D, int P, const CUtensorMap &km,
                             const CUtensorMap &vm, const AttnParams &p, int grid,
                             size_t smem_budget, bool pdl, cudaStream_t stream) {
    switch (dt) {
    case QASA_DTYPE_E4M3: return launch_attn_dt<fp8e4m3, false>(D, P, km, vm, p, grid, smem_budget, pdl, stream);
    case QASA_DTYPE_F32: return launch_attn_dt<float, false>(D, P, km, vm, p, grid, smem_budget, pdl, stream);
    case QASA_DTYPE_F16: return launch_attn_dt<__half, false>(D, P, km, vm, p, grid, smem_budget, pdl, stream);
    default: return launch_attn_dt<__nv_bfloat16, false>(D, P, km, vm, p, grid, smem_budget, pdl, stream);
    }
}

cudaError_t launch_fused_decode(qasa_dtype dt, int D, int P, const CUtensorMap &km,
                                const CUtensorMap &vm, const AttnParams &p, int grid,
                                size_t smem_budget, cudaStream_t stream) {
    switch (dt) {
    case QASA_DTYPE_E4M3: return cudaErrorNotSupported;   // the selection is not fused for FP8 KV
    case QASA_DTYPE_F32: return launch_attn_dt<float, true>(D, P, km, vm, p, grid, smem_budget, false, stream);
    case QASA_DTYPE_F16: return launch_attn_dt<__half, true>(D, P, km, vm, p, grid, smem_budget, false, stream);
    default: return launch_attn_dt<__nv_bfloat16, true>(D, P, km, vm, p, grid, smem_budget, false, stream);
    }
}

}  // namespace qasa
